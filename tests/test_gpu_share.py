"""Decode steps with shared prefixes (pkv_pool_set_prefix_sharing) against the oracle.

The oracle attends every row over its whole table, prefix and all ("KV Cache Management",
PagedAttention model); the library attends each run of rows that share their first blocks
to those blocks once (the tcgen05 prefix kernel) and to each row's own blocks in the decode
kernel, merged with the online-softmax rule.  Every row of every step is compared; the
tests also check that the plan did form the groups, so the shared path is what ran.
"""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev, to_raw

pytestmark = pytest.mark.gpu


def _plan_header(meta, n, W_):
    off = (n * (W_ + 2) + 3) // 4 * 4
    return [int(x) for x in meta[off:off + 4]]


def _build(dtype, H_q, seed, members=(37, 5, 20), prefixes=(1000, 2050, 300), min_members=4):
    """Three parents forked into runs of branches (random suffixes), interleaved with
    unrelated sequences; returns the batch and the step's row order."""
    g = W.Geometry(L=1, H_q=H_q, H_kv=8, d_head=128, block_size=16, dtype=dtype, num_blocks=4096)
    b = PagedBatch(g, W.permutation(seed, "fo", g.num_blocks), seed=seed,
                   kv_scales=(0.5, 0.25) if dtype == "e4m3" else (1.0, 1.0))
    pkv.pkv_pool_set_prefix_sharing(b.lib, min_members, 1, 0)
    rng = W.substream(seed, "suffix")
    singles = b.new_seqs(4)
    b.append(singles, [700, 1, 0, 1500], "single")
    run = [singles[0]]
    for k, (m, p) in enumerate(zip(members, prefixes)):
        (parent,) = b.new_seqs(1)
        b.append([parent], [p], f"prefix{k}")
        kids = [b.fork(parent) for _ in range(m)]
        suffix = [int(x) for x in rng.integers(0, 100, m)]
        suffix[0] = 0  # one branch whose first write is this step's (a copy of the shared tail)
        b.append(kids, suffix, f"suffix{k}")
        run += kids + [singles[1 + k]] if k < 3 else kids
    return b, np.array(run, np.int32)


@pytest.mark.parametrize("dtype,H_q", [("bf16", 64), ("bf16", 128), ("f16", 64), ("e4m3", 64), ("e4m3", 128)])
def test_shared_prefix_steps_match_oracle(dtype, H_q):
    import torch

    b, run = _build(dtype, H_q, seed=71)
    g = b.g
    n, Wd = len(run), 160
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    assert mi > n * (Wd + 2)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    act = "bf16" if dtype == "e4m3" else dtype
    td = torch.bfloat16 if act == "bf16" else torch.float16
    for step in range(3):
        q = W.normal(71, f"q{step}", (n, g.H_q, g.d_head), act)
        kn = W.normal(71, f"k{step}", (n, g.H_kv, g.d_head), act)
        vn = W.normal(71, f"v{step}", (n, g.H_kv, g.d_head), act)
        out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=td, device="cuda")
        pkv.pkv_decode_step(b.lib, 0, run, Wd, to_dev(q, act), to_dev(kn, act), to_dev(vn, act), b.kp, b.vp, scale,
                            out, meta_host, meta_dev, ws)
        torch.cuda.synchronize()
        hdr = _plan_header(meta_host.numpy(), n, Wd)
        assert hdr[0] >= 3 and hdr[1] == 37, hdr  # three groups, the largest of 37 rows
        if H_q == 128:
            assert hdr[3] == 0  # groups of 16 heads: decode on every SM, then the prefix kernel
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        if len(ocows):
            oracle.copy_blocks(g, ocows, b.hk, b.hv)
        oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv, b.k_scale, b.v_scale)
        pkv.pkv_check_device_error()
        tables, lens = b.tables(run.tolist(), Wd)
        ref = b.decode_ref(q, tables, lens, scale)
        check_attention(out_f64(out, act), ref, act)
        b.check_state()
    b.check_pools_bitexact()


def test_shared_prefix_packed_launcher_matches_oracle():
    """The end-to-end form: inputs and metadata packed in one page-locked buffer."""
    import torch

    b, run = _build("bf16", 64, seed=72, members=(33, 8), prefixes=(777, 4100))
    g = b.g
    n, Wd = len(run), 300
    rq, rk = g.H_q * g.d_head * 2, g.H_kv * g.d_head * 2
    off_k, off_v, off_meta = n * rq, n * (rq + rk), n * (rq + 2 * rk)
    in_bytes = off_meta + 4 * pkv.pkv_step_meta_ints(b.lib, n, Wd)
    in_host = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    in_dev = torch.zeros(in_bytes, dtype=torch.uint8, device="cuda")
    out_dev = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    out_host = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    launch = pkv.PackedStepLauncher(b.lib, 0, in_dev, out_dev, b.kp, b.vp, scale, ws)
    meta_view = in_host[off_meta:].view(torch.int32)
    for step in range(2):
        q = W.normal(72, f"q{step}", (n, g.H_q, g.d_head), "bf16")
        kn = W.normal(72, f"k{step}", (n, g.H_kv, g.d_head), "bf16")
        vn = W.normal(72, f"v{step}", (n, g.H_kv, g.d_head), "bf16")
        for src, o in ((q, 0), (kn, off_k), (vn, off_v)):
            raw = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
            in_host[o:o + raw.size] = torch.from_numpy(raw)
        cows = pkv.pkv_step_plan(b.lib, run, Wd, meta_view)
        assert _plan_header(meta_view.numpy(), n, Wd)[0] >= 2
        launch(n, Wd, cows, in_host, off_k, off_v, in_bytes, out_host, off_meta=off_meta)
        torch.cuda.synchronize()
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        if len(ocows):
            oracle.copy_blocks(g, ocows, b.hk, b.hv)
        oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv)
        pkv.pkv_check_device_error()
        tables, lens = b.tables(run.tolist(), Wd)
        check_attention(out_host.double().numpy(), b.decode_ref(q, tables, lens, scale), "bf16")
    b.check_pools_bitexact()


def test_forked_workload_with_sharing_sampled():
    """The forked configuration (16,376-token prefix, 64 branches, U[0, 2048] suffixes) with
    sharing on, as the benchmark runs it: two steps, 16 sampled branches against the oracle."""
    import torch

    wl = W.forked()
    g = wl.geometry
    b = PagedBatch(g, wl.free_order, seed=wl.seed)
    pkv.pkv_pool_set_prefix_sharing(b.lib, 8, 1, 0)
    (parent,) = b.new_seqs(1)
    b.append([parent], [int(wl.lengths[0])], "prefix")
    kids = [b.fork(parent) for _ in range(wl.extra["n_branch"])]
    b.append(kids, [int(x) for x in wl.extra["suffix"]], "suffix")
    run = np.array(kids, np.int32)
    n, Wd = len(run), -(-(int(wl.lengths[0]) + 2048 + 4) // g.block_size)
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    sample = list(range(0, 64, 4))
    for step in range(2):
        q = W.normal(wl.seed, f"sq{step}", (n, g.H_q, g.d_head), g.dtype)
        kn = W.normal(wl.seed, f"sk{step}", (n, g.H_kv, g.d_head), g.dtype)
        vn = W.normal(wl.seed, f"sv{step}", (n, g.H_kv, g.d_head), g.dtype)
        out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.pkv_decode_step(b.lib, 0, run, Wd, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), b.kp, b.vp,
                            wl.scale, out, meta_host, meta_dev, ws)
        torch.cuda.synchronize()
        hdr = _plan_header(meta_host.numpy(), n, Wd)
        assert hdr[0] > 1 and hdr[1] == 64, hdr  # one group of all 64 branches, in several splits
        assert hdr[3] > 0, hdr  # the decode of the branches' own blocks beside the prefix kernel
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        if len(ocows):
            oracle.copy_blocks(g, ocows, b.hk, b.hv)
        oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv)
        pkv.pkv_check_device_error()
        tables, lens = b.tables(run.tolist(), Wd)
        got = out_f64(out, "bf16")
        assert np.all(np.isfinite(got))
        check_attention(got[sample], b.decode_ref(q[sample], tables[sample], lens[sample], wl.scale), "bf16")
    b.check_pools_bitexact()


@pytest.mark.parametrize("side_by_side", [True, False])
def test_both_schedules_give_the_oracle_result(side_by_side):
    """The same step with the decode beside the prefix kernel (header word 3 > 0, as planned)
    and with it forced to run on every SM first (word 3 = 0 written into the plan)."""
    import torch

    b, run = _build("bf16", 64, seed=74, members=(64,), prefixes=(3000,))
    g = b.g
    n, Wd = len(run), 320
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    q = W.normal(74, "q", (n, g.H_q, g.d_head), "bf16")
    kn = W.normal(74, "k", (n, g.H_kv, g.d_head), "bf16")
    vn = W.normal(74, "v", (n, g.H_kv, g.d_head), "bf16")
    cows = pkv.pkv_step_plan(b.lib, run, Wd, meta_host)
    off = (n * (Wd + 2) + 3) // 4 * 4
    assert int(meta_host[off + 3]) > 0  # planned side by side
    if not side_by_side:
        meta_host[off + 3] = 0
    out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_step_launch(b.lib, 0, n, Wd, cows, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), b.kp,
                        b.vp, scale, out, meta_host, meta_dev, ws)
    torch.cuda.synchronize()
    oslots, ocows = b.orc.append(run.tolist(), [1] * n)
    if len(ocows):
        oracle.copy_blocks(g, ocows, b.hk, b.hv)
    oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv)
    pkv.pkv_check_device_error()
    tables, lens = b.tables(run.tolist(), Wd)
    check_attention(out_f64(out, "bf16"), b.decode_ref(q, tables, lens, scale), "bf16")
    b.check_pools_bitexact()


def test_shared_prefix_beyond_the_in_kernel_plan():
    """4,500 rows in 450 runs of 10 branches (a 40-token prefix: 2 shared blocks each): past
    4,096 sequences the decode kernel follows the plan kernel, which also starts each row's
    tiles after its shared blocks; every row against the oracle."""
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=16384)
    b = PagedBatch(g, W.permutation(75, "fo", g.num_blocks), seed=75)
    pkv.pkv_pool_set_prefix_sharing(b.lib, 4, 1, 0)
    rng = W.substream(75, "suffix")
    parents = b.new_seqs(450)
    b.append(parents, [40] * 450, "prefix")
    run = []
    for p_ in parents:
        run += [b.fork(p_) for _ in range(10)]
    b.append(run, [int(x) for x in rng.integers(0, 30, len(run))], "suffix")
    run = np.array(run, np.int32)
    n, Wd = len(run), 8
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    q = W.normal(75, "q", (n, g.H_q, g.d_head), "bf16")
    kn = W.normal(75, "k", (n, g.H_kv, g.d_head), "bf16")
    vn = W.normal(75, "v", (n, g.H_kv, g.d_head), "bf16")
    out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_step(b.lib, 0, run, Wd, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), b.kp, b.vp,
                        scale, out, meta_host, meta_dev, ws)
    torch.cuda.synchronize()
    hdr = _plan_header(meta_host.numpy(), n, Wd)
    assert hdr[0] >= 450 and hdr[1] == 10, hdr  # every run is a group
    oslots, ocows = b.orc.append(run.tolist(), [1] * n)
    if len(ocows):
        oracle.copy_blocks(g, ocows, b.hk, b.hv)
    oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv)
    pkv.pkv_check_device_error()
    tables, lens = b.tables(run.tolist(), Wd)
    check_attention(out_f64(out, "bf16"), b.decode_ref(q, tables, lens, scale), "bf16")
    b.check_state()


def test_agents_over_a_shared_prompt_sampled():
    """Structured prefix sharing ("KV Cache Management", Step 5: a 24,576-token shared system
    prompt and repository index, 8,192 tokens of each agent's own): 48 agents forked from one
    parent, one decode step with sharing on (pkv_step_plan, then pkv_step_launch), the shape
    `bench.py --shared-prefix 24576` times.  Sampled agents against the oracle, which gets host
    copies of exactly their blocks from before the step plus the step's new tokens written on
    the host."""
    import torch

    wl = W.agent(48, 32768, spare_steps=32)
    g = wl.geometry
    kp = W.device_normal(wl.seed, "k_pool_shared", g.pool_shape(), g.dtype, "cuda")
    vp = W.device_normal(wl.seed, "v_pool_shared", g.pool_shape(), g.dtype, "cuda")
    b = PagedBatch(g, wl.free_order, seed=wl.seed, host_pool=False, fill_device=(kp, vp))
    pkv.pkv_pool_set_prefix_sharing(b.lib, 8, 1, 0)
    (parent,) = b.new_seqs(1)
    b.append([parent], [24576], "prompt", plan_only=True)
    kids = [b.fork(parent) for _ in range(48)]
    b.append(kids, [8192] * 48, "own", plan_only=True)
    run = np.array(kids, np.int32)
    n, Wd = len(run), 2050
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    cows = pkv.pkv_step_plan(b.lib, run, Wd, meta_host)
    oslots, ocows = b.orc.append(run.tolist(), [1] * n)
    assert np.array_equal(meta_host[:n].numpy(), oslots) and len(cows) == len(ocows) == 0
    assert _plan_header(meta_host.numpy(), n, Wd)[1] == 48  # one run of all 48 agents
    sample = [0, 23, 47]
    tables, lens = b.tables(run.tolist(), Wd)
    used = sorted({int(x) for r in sample for x in tables[r, : -(-int(lens[r]) // g.block_size)]})
    remap = {blk: j for j, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    hk = to_raw(kp.index_select(0, idx), g.dtype)  # before the step writes anything
    hv = to_raw(vp.index_select(0, idx), g.dtype)
    q = W.normal(wl.seed, "sq", (n, g.H_q, g.d_head), g.dtype)
    kn = W.normal(wl.seed, "sk", (n, g.H_kv, g.d_head), g.dtype)
    vn = W.normal(wl.seed, "sv", (n, g.H_kv, g.d_head), g.dtype)
    out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_step_launch(b.lib, 0, n, Wd, cows, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), kp, vp,
                        wl.scale, out, meta_host, meta_dev, ws)
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    got = out_f64(out, "bf16")
    assert np.all(np.isfinite(got))
    gc = W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, len(used))
    cslots = np.array([remap[int(oslots[r]) // g.block_size] * g.block_size + int(oslots[r]) % g.block_size
                       for r in sample], np.int32)
    oracle.write_slots(gc, 0, kn[sample], vn[sample], cslots, hk, hv)
    ct = np.zeros((len(sample), Wd), np.int32)
    for i, r in enumerate(sample):
        nb = -(-int(lens[r]) // g.block_size)
        ct[i, :nb] = [remap[int(x)] for x in tables[r, :nb]]
    ref = oracle.decode_attention(gc, 0, q[sample], hk, hv, ct, lens[sample], wl.scale)
    check_attention(got[sample], ref, "bf16")


def _one_step_against_oracle(b, run, Wd, seed):
    """One pkv_decode_step over `run`, every row against the oracle; returns the plan header."""
    import torch

    g = b.g
    n = len(run)
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    q = W.normal(seed, "q", (n, g.H_q, g.d_head), "bf16")
    kn = W.normal(seed, "k", (n, g.H_kv, g.d_head), "bf16")
    vn = W.normal(seed, "v", (n, g.H_kv, g.d_head), "bf16")
    out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_step(b.lib, 0, run, Wd, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), b.kp, b.vp,
                        scale, out, meta_host, meta_dev, ws)
    torch.cuda.synchronize()
    hdr = _plan_header(meta_host.numpy(), n, Wd)
    oslots, ocows = b.orc.append(run.tolist(), [1] * n)
    if len(ocows):
        oracle.copy_blocks(g, ocows, b.hk, b.hv)
    oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv)
    pkv.pkv_check_device_error()
    tables, lens = b.tables(run.tolist(), Wd)
    check_attention(out_f64(out, "bf16"), b.decode_ref(q, tables, lens, scale), "bf16")
    b.check_pools_bitexact()
    return hdr


def test_rows_with_a_single_token_of_their_own():
    """40 branches of a 4,096-token prefix (256 full blocks) with no suffix: after the step each
    row's only own token is the step's, in a block of its own."""
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=1024)
    b = PagedBatch(g, W.permutation(76, "fo", g.num_blocks), seed=76)
    pkv.pkv_pool_set_prefix_sharing(b.lib, 4, 1, 0)
    (parent,) = b.new_seqs(1)
    b.append([parent], [4096], "prefix")
    run = np.array([b.fork(parent) for _ in range(40)], np.int32)
    hdr = _one_step_against_oracle(b, run, 260, 76)
    assert hdr[0] >= 1 and hdr[1] == 40, hdr


def test_sharing_on_without_a_run_long_enough():
    """Sharing on, but no run reaches min_members: the plan is empty and the step is the plain
    decode (with the larger metadata)."""
    b, run = _build("bf16", 64, seed=77, members=(5, 6), prefixes=(700, 900), min_members=8)
    hdr = _one_step_against_oracle(b, run, 80, 77)
    assert hdr == [0, 0, 0, 0], hdr


def test_shared_prefix_step_on_the_second_layer():
    """A two-layer pool: the step runs on layer 1, so the prefix kernel, the decode and the
    append all address layer 1's slabs of every block."""
    import torch

    g = W.Geometry(L=2, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=512)
    b = PagedBatch(g, W.permutation(78, "fo", g.num_blocks), seed=78)
    pkv.pkv_pool_set_prefix_sharing(b.lib, 4, 1, 0)
    (parent,) = b.new_seqs(1)
    b.append([parent], [1500], "prefix", layer=-1)
    run = [b.fork(parent) for _ in range(12)]
    b.append(run, [int(x) for x in W.substream(78, "sfx").integers(0, 60, 12)], "suffix", layer=-1)
    run = np.array(run, np.int32)
    n, Wd = len(run), 100
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    q = W.normal(78, "q", (n, g.H_q, g.d_head), "bf16")
    kn = W.normal(78, "k", (n, g.H_kv, g.d_head), "bf16")
    vn = W.normal(78, "v", (n, g.H_kv, g.d_head), "bf16")
    out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_step(b.lib, 1, run, Wd, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), b.kp, b.vp,
                        scale, out, meta_host, meta_dev, ws)
    torch.cuda.synchronize()
    assert _plan_header(meta_host.numpy(), n, Wd)[1] == 12
    oslots, ocows = b.orc.append(run.tolist(), [1] * n)
    if len(ocows):
        oracle.copy_blocks(g, ocows, b.hk, b.hv)
    oracle.write_slots(g, 1, kn, vn, oslots, b.hk, b.hv)
    pkv.pkv_check_device_error()
    tables, lens = b.tables(run.tolist(), Wd)
    check_attention(out_f64(out, "bf16"), b.decode_ref(q, tables, lens, scale, layer=1), "bf16")
    b.check_pools_bitexact()


def test_corrupt_plan_header_is_rejected():
    import torch

    b, run = _build("bf16", 64, seed=73, members=(6,), prefixes=(500,))
    g = b.g
    n, Wd = len(run), 64
    mi = pkv.pkv_step_meta_ints(b.lib, n, Wd)
    meta_host = torch.zeros(mi, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(mi, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    cows = pkv.pkv_step_plan(b.lib, run, Wd, meta_host)
    off = (n * (Wd + 2) + 3) // 4 * 4
    meta_host[off] = 1 << 30  # more work items than the plan holds
    x = torch.zeros((n, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((n, g.H_kv, g.d_head), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_step_launch(b.lib, 0, n, Wd, cows, x, kv, kv, b.kp, b.vp, 0.1, x, meta_host, meta_dev, ws)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
