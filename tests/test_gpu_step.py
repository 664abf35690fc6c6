"""pkv_decode_step (plan + CoW copy + append + attend in one call) against the oracle."""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev, to_raw, torch_dtype

pytestmark = pytest.mark.gpu


def test_decode_step_matches_oracle_with_forks():
    import torch

    g = W.Geometry(L=2, H_q=32, H_kv=4, d_head=128, block_size=16, dtype="bf16", num_blocks=512)
    b = PagedBatch(g, W.permutation(41, "fo", g.num_blocks), seed=41)
    ids = b.new_seqs(6)
    b.append(ids, [1, 16, 40, 300, 0, 77], "prompt", layer=-1)
    kids = [b.fork(ids[2]), b.fork(ids[3])]  # the first step copies their shared tail blocks
    run = np.array(ids[:4] + kids + [ids[5]], np.int32)
    n, Wd = len(run), 24
    meta_host = torch.zeros(n * (Wd + 2), dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    for step in range(3):
        for layer in (0, 1):
            q = W.normal(41, f"q{step}{layer}", (n, g.H_q, g.d_head), "bf16")
            kn = W.normal(41, f"k{step}{layer}", (n, g.H_kv, g.d_head), "bf16")
            vn = W.normal(41, f"v{step}{layer}", (n, g.H_kv, g.d_head), "bf16")
            out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
            if layer == 0:
                pkv.pkv_decode_step(b.lib, 0, run, Wd, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"),
                                    b.kp, b.vp, scale, out, meta_host, meta_dev, ws)
                oslots, ocows = b.orc.append(run.tolist(), [1] * n)
                if len(ocows):
                    oracle.copy_blocks(g, ocows, b.hk, b.hv)
                assert np.array_equal(meta_host[:n].numpy(), oslots)
            else:
                # a second layer of the same step: the slots are already planned
                pkv.pkv_append_kv(b.lib, 1, to_dev(kn, "bf16"), to_dev(vn, "bf16"), meta_dev[:n], b.kp, b.vp)
                tables = meta_dev[n:n + n * Wd].view(n, Wd)
                lens = meta_dev[n + n * Wd:n + n * Wd + n]
                pkv.pkv_decode_attention(b.lib, 1, to_dev(q, "bf16"), b.kp, b.vp, tables, lens, scale, out, ws)
            oracle.write_slots(g, layer, kn, vn, oslots, b.hk, b.hv)
            pkv.pkv_check_device_error()
            tables, lens = b.tables(run.tolist(), Wd)
            ref = b.decode_ref(q, tables, lens, scale, layer=layer)
            check_attention(out_f64(out, "bf16"), ref, "bf16")
        b.check_state()
    b.check_pools_bitexact()


def test_decode_step_rejects_a_narrow_table_without_change():
    import torch

    g = W.Geometry(L=1, H_q=8, H_kv=2, d_head=64, block_size=16, dtype="bf16", num_blocks=64)
    b = PagedBatch(g, None, seed=42)
    ids = b.new_seqs(2)
    b.append(ids, [32, 3], "p")
    before = (pkv.pkv_refcounts(b.lib).copy(), pkv.pkv_free_list(b.lib).copy())
    meta_host = torch.zeros(2 * 4, dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(2 * 4, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, 2), dtype=torch.uint8, device="cuda")
    x = torch.zeros((2, 8, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:  # W = 2 cannot hold 33 tokens
        pkv.pkv_decode_step(b.lib, 0, ids, 2, x, kv, kv, b.kp, b.vp, 0.1, x, meta_host, meta_dev, ws)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert np.array_equal(before[0], pkv.pkv_refcounts(b.lib)) and np.array_equal(before[1], pkv.pkv_free_list(b.lib))
    assert pkv.pkv_seq_len(b.lib, ids[0]) == 32


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_decode_step_host_buffers_match_oracle(dtype):
    """pkv_decode_step_host: inputs in page-locked host memory, result copied back by the call."""
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype=dtype, num_blocks=256)
    b = PagedBatch(g, W.permutation(43, "fo", g.num_blocks), seed=43,
                   kv_scales=(0.5, 0.25) if dtype == "e4m3" else (1.0, 1.0))
    ids = b.new_seqs(5)
    b.append(ids, [15, 16, 100, 0, 333], "prompt")
    kid = b.fork(ids[2])
    run = np.array(ids + [kid], np.int32)
    n, Wd = len(run), 24
    meta_host = torch.zeros(n * (Wd + 2), dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    q_dev = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    k_dev = torch.empty((n, g.H_kv, g.d_head), dtype=torch.bfloat16, device="cuda")
    v_dev = torch.empty_like(k_dev)
    o_dev = torch.empty_like(q_dev)
    scale = 1.0 / math.sqrt(g.d_head)
    for step in range(3):
        q = W.normal(43, f"q{step}", (n, g.H_q, g.d_head), "bf16")
        kn = W.normal(43, f"k{step}", (n, g.H_kv, g.d_head), "bf16")
        vn = W.normal(43, f"v{step}", (n, g.H_kv, g.d_head), "bf16")
        pin = lambda x: torch.from_numpy(x.copy()).pin_memory()
        out_host = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16).pin_memory()
        pkv.pkv_decode_step_host(b.lib, 0, run, Wd, pin(q).view(torch.bfloat16), pin(kn).view(torch.bfloat16),
                                 pin(vn).view(torch.bfloat16), out_host, q_dev, k_dev, v_dev, o_dev, b.kp, b.vp, scale,
                                 meta_host, meta_dev, ws)
        torch.cuda.synchronize()
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        if len(ocows):
            oracle.copy_blocks(g, ocows, b.hk, b.hv)
        oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv, b.k_scale, b.v_scale)
        pkv.pkv_check_device_error()
        tables, lens = b.tables(run.tolist(), Wd)
        ref = b.decode_ref(q, tables, lens, scale)
        check_attention(out_host.double().numpy(), ref, "bf16")
        b.check_state()
    b.check_pools_bitexact()


@pytest.mark.parametrize("dtype,api", [("bf16", "function"), ("e4m3", "function"), ("bf16", "launcher"),
                                       ("bf16", "packed"), ("e4m3", "packed_early_meta"),
                                       ("bf16", "packed_meta_inside")])
def test_step_plan_ahead_then_launch_host_match_oracle(dtype, api):
    """pkv_step_plan of step t + 1 runs while step t (pkv_step_launch_host, a StepLauncher with
    the fixed buffers bound once, or a PackedStepLauncher: one packed input copy, the metadata
    copied by the call or queued by the caller right after the plan) is on the GPU, as a serving
    loop's scheduler would; every step's result matches the oracle and the pools and
    control-plane state stay identical to the oracle's."""
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype=dtype, num_blocks=256)
    b = PagedBatch(g, W.permutation(44, "fo", g.num_blocks), seed=44,
                   kv_scales=(0.5, 0.25) if dtype == "e4m3" else (1.0, 1.0))
    ids = b.new_seqs(4)
    b.append(ids, [16, 31, 200, 1], "prompt")
    kids = [b.fork(ids[1]), b.fork(ids[2])]  # the first step copies their shared tail blocks
    run = np.array(ids + kids, np.int32)
    n, Wd, steps = len(run), 24, 5
    metas = [torch.zeros(n * (Wd + 2), dtype=torch.int32).pin_memory() for _ in range(2)]
    mdev = [torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda") for _ in range(2)]
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    q_dev = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    k_dev = torch.empty((n, g.H_kv, g.d_head), dtype=torch.bfloat16, device="cuda")
    v_dev = torch.empty_like(k_dev)
    o_dev = torch.empty_like(q_dev)
    out_host = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16).pin_memory()
    scale = 1.0 / math.sqrt(g.d_head)
    pin = lambda x: torch.from_numpy(x.copy()).pin_memory().view(torch.bfloat16)
    plans = {}
    launcher = pkv.StepLauncher(b.lib, 0, q_dev, k_dev, v_dev, o_dev, b.kp, b.vp, scale, ws)
    rq, rk = g.H_q * g.d_head * 2, g.H_kv * g.d_head * 2
    off_k, off_v = n * rq + 48, n * rq + 48 + n * rk + 16  # any 16-byte multiples that keep the parts apart
    in_bytes = off_v + n * rk
    off_meta = in_bytes + 32  # the metadata packed after the inputs (the "packed_meta_inside" calls)
    in_dev = torch.empty(off_meta + 4 * n * (Wd + 2) + 64, dtype=torch.uint8, device="cuda")
    packed = pkv.PackedStepLauncher(b.lib, 0, in_dev, o_dev, b.kp, b.vp, scale, ws)

    def plan(t):
        m = metas[t % 2]
        cows = pkv.pkv_step_plan(b.lib, run, Wd, m)
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        mn = m.numpy()
        assert np.array_equal(mn[:n], oslots) and np.array_equal(cows, ocows)
        plans[t] = (cows, oslots, mn[n:n + n * Wd].reshape(n, Wd).copy(), mn[n + n * Wd:n + n * Wd + n].copy())

    plan(0)
    for t in range(steps):
        q = W.normal(44, f"q{t}", (n, g.H_q, g.d_head), "bf16")
        kn = W.normal(44, f"k{t}", (n, g.H_kv, g.d_head), "bf16")
        vn = W.normal(44, f"v{t}", (n, g.H_kv, g.d_head), "bf16")
        cows, oslots, tab, lens = plans[t]
        out_host.fill_(float("nan"))
        if api == "launcher":
            launcher(n, Wd, cows, pin(q), pin(kn), pin(vn), out_host, metas[t % 2], mdev[t % 2])
        elif api.startswith("packed"):
            in_host = torch.zeros(off_meta + 4 * n * (Wd + 2), dtype=torch.uint8).pin_memory()
            for x, o in ((q, 0), (kn, off_k), (vn, off_v)):
                in_host[o:o + x.nbytes].copy_(torch.from_numpy(x.reshape(-1).view(np.uint8)))
            if api == "packed_meta_inside":
                in_host[off_meta:].view(torch.int32).copy_(metas[t % 2][:n * (Wd + 2)])
                packed(n, Wd, cows, in_host, off_k, off_v, off_meta + 4 * n * (Wd + 2), out_host, off_meta=off_meta)
            elif api == "packed_early_meta":
                mdev[t % 2].copy_(metas[t % 2], non_blocking=True)
                packed(n, Wd, cows, in_host, off_k, off_v, in_bytes, out_host, mdev[t % 2])
            else:
                packed(n, Wd, cows, in_host, off_k, off_v, in_bytes, out_host, mdev[t % 2], meta_host=metas[t % 2])
        else:
            pkv.pkv_step_launch_host(b.lib, 0, n, Wd, cows, pin(q), pin(kn), pin(vn), out_host, q_dev, k_dev, v_dev,
                                     o_dev, b.kp, b.vp, scale, metas[t % 2], mdev[t % 2], ws)
        if len(cows):
            oracle.copy_blocks(g, cows, b.hk, b.hv)
        oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv, b.k_scale, b.v_scale)
        if t + 1 < steps:
            plan(t + 1)  # the host half of the next step while this one runs
        torch.cuda.synchronize()
        pkv.pkv_check_device_error()
        ref = b.decode_ref(q, tab, lens, scale)
        check_attention(out_host.double().numpy(), ref, "bf16")
    b.check_state()
    b.check_pools_bitexact()


def test_step_launcher_keeps_its_pool_and_checks_host_buffers():
    """A StepLauncher holds the pool it was built on (dropping the caller's last reference
    does not destroy it under the launcher) and rejects host buffers shorter than the step
    copies, before any copy is issued."""
    import gc

    import torch

    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks)
    ids = np.array([pkv.pkv_seq_create(pool) for _ in range(2)], np.int32)
    pkv.pkv_plan_append(pool, ids, [10, 40])
    kp = torch.zeros(g.pool_shape(), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    n, Wd = 2, 4
    ws = torch.empty(pkv.pkv_decode_workspace_size(pool, n), dtype=torch.uint8, device="cuda")
    q_dev = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    k_dev = torch.empty((n, g.H_kv, g.d_head), dtype=torch.bfloat16, device="cuda")
    launcher = pkv.StepLauncher(pool, 0, q_dev, k_dev, k_dev.clone(), q_dev.clone(), kp, vp, 0.1, ws)
    del pool
    gc.collect()
    meta_host = torch.zeros(n * (Wd + 2), dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda")
    pool = launcher._pool
    cows = pkv.pkv_step_plan(pool, ids, Wd, meta_host)
    qh = torch.zeros((n, g.H_q, g.d_head), dtype=torch.bfloat16).pin_memory()
    kh = torch.zeros((n, g.H_kv, g.d_head), dtype=torch.bfloat16).pin_memory()
    oh = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError, match="out_host"):
        launcher(n, Wd, cows, qh, kh, kh, oh[:1], meta_host, meta_dev)
    with pytest.raises(ValueError, match="meta_dev"):
        launcher(n, Wd, cows, qh, kh, kh, oh, meta_host, meta_dev[:-1])
    with pytest.raises(ValueError, match="exceeds"):
        launcher(n + 1, Wd, cows, qh, kh, kh, oh, meta_host, meta_dev)
    launcher(n, Wd, cows, qh, kh, kh, oh, meta_host, meta_dev)  # zero q and keys: outputs are means of zero V
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    assert torch.all(oh == 0)


@pytest.mark.parametrize("H_q,H_kv,d,B,dtype", [
    (64, 8, 128, 16, "bf16"),
    (48, 4, 64, 16, "f16"),     # G = 12 (two head blocks), d 64
    (32, 2, 128, 32, "bf16"),   # G = 16, 32-token blocks
    (64, 8, 128, 16, "e4m3"),   # FP8 pool: the kernel quantises the new token
    (12, 12, 64, 16, "f32"),    # CUDA-core path: the append kernel runs first
    (16, 2, 96, 16, "bf16"),    # d 96: CUDA-core path
])
def test_decode_step_appends_inside_the_attention_launch(H_q, H_kv, d, B, dtype):
    """On the tensor-core path pkv_decode_step writes each new token from inside the
    attention kernel (one launch for append and attention); elsewhere the append kernel
    runs first.  Either way the pools stay bit-exact with the oracle's and every output
    matches the oracle, over steps whose new tokens open blocks, fill them and copy
    shared tails."""
    import torch

    g = W.Geometry(L=2, H_q=H_q, H_kv=H_kv, d_head=d, block_size=B, dtype=dtype, num_blocks=400)
    b = PagedBatch(g, W.permutation(45, "fo", g.num_blocks), seed=45,
                   kv_scales=(0.75, 1.5) if dtype == "e4m3" else (1.0, 1.0))
    ids = b.new_seqs(5)
    b.append(ids, [B - 1, B, 3 * B + 5, 1, 700], "prompt", layer=-1)
    kids = [b.fork(ids[2]), b.fork(ids[4])]
    run = np.array(ids + kids, np.int32)
    n, Wd = len(run), 64
    act = "bf16" if dtype == "e4m3" else dtype
    td = torch_dtype(act)
    meta_host = torch.zeros(n * (Wd + 2), dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(d)
    for step in range(3):
        layer = step % 2
        q = W.normal(45, f"q{step}", (n, H_q, d), act)
        kn = W.normal(45, f"k{step}", (n, H_kv, d), act)
        vn = W.normal(45, f"v{step}", (n, H_kv, d), act)
        out = torch.full((n, H_q, d), float("nan"), dtype=td, device="cuda")
        pkv.pkv_decode_step(b.lib, layer, run, Wd, to_dev(q, act), to_dev(kn, act), to_dev(vn, act), b.kp, b.vp,
                            scale, out, meta_host, meta_dev, ws)
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        assert np.array_equal(meta_host[:n].numpy(), oslots)
        if len(ocows):
            oracle.copy_blocks(g, ocows, b.hk, b.hv)
        oracle.write_slots(g, layer, kn, vn, oslots, b.hk, b.hv, b.k_scale, b.v_scale)
        pkv.pkv_check_device_error()
        tables, lens = b.tables(run.tolist(), Wd)
        check_attention(out_f64(out, act), b.decode_ref(q, tables, lens, scale, layer=layer), act)
        b.check_state()
        b.check_pools_bitexact()


def test_packed_step_rejects_a_layout_that_does_not_hold_the_rows():
    """pkv_step_launch_packed checks its packed layout (parts in order, 16-byte offsets, each
    holding n rows, in_bytes covering the last part) before any copy or launch: a bad layout
    is INVALID_ARG and the pools stay as they were."""
    import torch

    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    b = PagedBatch(g, None, seed=46)
    ids = b.new_seqs(2)
    b.append(ids, [10, 40], "p")
    n, Wd = 2, 4
    rq, rk = g.H_q * g.d_head * 2, g.H_kv * g.d_head * 2
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    out_dev = torch.empty((n, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    in_dev = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    in_host = torch.zeros(1 << 16, dtype=torch.uint8).pin_memory()
    out_host = torch.zeros((n, g.H_q, g.d_head), dtype=torch.bfloat16).pin_memory()
    meta_dev = torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda")
    launcher = pkv.PackedStepLauncher(b.lib, 0, in_dev, out_dev, b.kp, b.vp, 0.1, ws)
    kp0, vp0 = b.kp.clone(), b.vp.clone()
    ok_k, ok_v = n * rq, n * rq + n * rk
    bad = [
        (ok_k - 16, ok_v, ok_v + n * rk, 0),            # q rows overrun k_new
        (ok_k, ok_k, ok_v + n * rk, 0),                 # k_new rows overrun v_new
        (ok_k, ok_v, ok_v + n * rk - 16, 0),            # in_bytes short of the v_new rows
        (ok_k + 8, ok_v + 16, ok_v + 16 + n * rk, 0),   # an offset not a multiple of 16
        (ok_k, ok_v, ok_v + n * rk + 64, ok_v + 16),    # metadata inside the v_new rows
    ]
    for off_k, off_v, in_bytes, off_meta in bad:
        with pytest.raises(pkv.PkvError) as e:
            launcher(n, Wd, np.zeros((0, 2), np.int32), in_host, off_k, off_v, in_bytes, out_host, meta_dev,
                     off_meta=off_meta)
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    torch.cuda.synchronize()
    assert torch.equal(b.kp, kp0) and torch.equal(b.vp, vp0)
    b.check_state()
