"""Paged decode attention on the GPU against the oracle (element by element)."""
import math

import numpy as np
import pytest

import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, to_dev

pytestmark = pytest.mark.gpu


def run_case(g, lens, seed, steps=1, free_order=None, W_extra=0, scale=None):
    b = PagedBatch(g, free_order if free_order is not None else W.permutation(seed, "fo", g.num_blocks), seed=seed)
    ids = b.new_seqs(len(lens))
    b.append(ids, lens, "prompt")
    scale = scale if scale is not None else 1.0 / math.sqrt(g.d_head)
    worst = 0.0
    for step in range(steps):
        b.append(ids, [1] * len(ids), f"step{step}")  # append, then attend over len + 1
        tables, lens_ = b.tables(ids)
        if W_extra:
            tables = np.concatenate([tables, np.full((len(ids), W_extra), 0, np.int32)], axis=1)
        q = W.normal(seed, f"q{step}", (len(ids), g.H_q, g.d_head), g.dtype)
        got, _, _ = b.decode_gpu(ids, q, scale, tables=tables, lens=lens_)
        ref = b.decode_ref(q, tables, lens_, scale)
        worst = max(worst, check_attention(got, ref, g.dtype))
    return b, worst


def test_tiny_gpt2_geometry_fp32():
    """12 heads = 12 KV heads, d_head 64, fp32, B = 16, 512-block seeded permutation,
    8 lengths uniform in [1, 512]; one append then one decode step."""
    wl = W.tiny()
    run_case(wl.geometry, [int(x) for x in wl.lengths], wl.seed, free_order=wl.free_order)


@pytest.mark.parametrize("lens", [
    [1, 15, 16, 17, 31, 32, 33],
    [100, 1000, 4097, 2, 64],
    [0, 5, 0, 300],
])
def test_gqa_bf16_ragged_lengths(lens):
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=1024)
    run_case(g, lens, 7, steps=2)


@pytest.mark.parametrize("H_q,H_kv,d,B,dtype", [
    (64, 8, 64, 16, "bf16"),
    (64, 8, 128, 16, "f16"),
    (32, 8, 128, 16, "bf16"),   # G = 4
    (8, 8, 128, 16, "bf16"),    # G = 1 on tensor cores
    (24, 4, 128, 32, "bf16"),   # G = 6, B = 32
    (64, 8, 128, 8, "bf16"),    # B = 8: CUDA-core path
    (16, 2, 96, 16, "bf16"),    # d = 96: CUDA-core path
    (12, 12, 64, 16, "f32"),
    (16, 4, 128, 16, "f32"),
    (32, 2, 128, 16, "bf16"),   # G = 16 on tensor cores (two 8-head blocks)
    (48, 4, 64, 16, "f16"),     # G = 12 on tensor cores
    (32, 2, 96, 16, "f16"),     # G = 16, d = 96: CUDA-core path
    (16, 1, 64, 16, "f32"),     # G = 16, fp32: CUDA-core path
])
def test_geometries(H_q, H_kv, d, B, dtype):
    g = W.Geometry(L=2, H_q=H_q, H_kv=H_kv, d_head=d, block_size=B, dtype=dtype, num_blocks=600)
    run_case(g, [3, 40, 129, 700, 1], 11, steps=1)


@pytest.mark.parametrize("H_q,H_kv,d,dtype,B", [
    (32, 2, 128, "bf16", 16),   # G = 16
    (72, 8, 128, "bf16", 16),   # G = 9: seven padded heads in the second block
    (48, 4, 64, "f16", 16),     # G = 12
    (128, 8, 128, "bf16", 16),  # G = 16 with 8 KV heads (a 128-query-head layer)
    (80, 8, 64, "bf16", 16),    # G = 10
    (32, 2, 128, "f16", 32),    # G = 16, 32-token blocks
])
def test_wide_groups_on_tensor_cores(H_q, H_kv, d, dtype, B):
    """9 to 16 query heads per KV head run on the tensor-core kernel with two 8-head
    column blocks (one launch per call: every CTA plans its own warps); the lengths make
    pairs that end inside one warp's range and pairs split across warps (merged
    partials), ragged tails and an empty sequence."""
    g = W.Geometry(L=2, H_q=H_q, H_kv=H_kv, d_head=d, block_size=B, dtype=dtype, num_blocks=1500)
    b = PagedBatch(g, W.permutation(61, f"fo{H_q}{d}", g.num_blocks), seed=61)
    lens = [3, 40, 129, 700, 1, 0, 4000, 17, 2049, 15, 16, 300]
    ids = b.new_seqs(len(lens))
    b.append(ids, lens, "p", layer=1)
    b.append(ids, [1] * len(ids), "t", layer=1)
    for step, scale in enumerate([1 / math.sqrt(d), 0.3]):
        q = W.normal(61, f"q{step}", (len(ids), g.H_q, g.d_head), dtype)
        before = pkv.pkv_launch_count()
        got, tables, sl = b.decode_gpu(ids, q, scale, layer=1)
        assert pkv.pkv_launch_count() - before == 1  # the tensor-core attention, planned in the kernel
        check_attention(got, b.decode_ref(q, tables, sl, scale, layer=1), dtype)


def test_long_single_sequence_split_across_many_warps():
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=1400)
    run_case(g, [20000], 13, steps=2)


def test_many_short_sequences():
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=2048)
    lens = [int(x) for x in W.uniform_int(14, "lens", 0, 40, 700)]
    run_case(g, lens, 14, steps=1)


def test_chat_mix_small():
    wl = W.chat(n_seq=48, num_blocks=2048)
    run_case(wl.geometry, [int(x) for x in wl.lengths], wl.seed, steps=3, free_order=wl.free_order)


def test_table_wider_than_needed_and_scale():
    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=256)
    run_case(g, [50, 90], 15, steps=1, W_extra=7, scale=0.02)


def test_bad_inputs_are_recorded_not_faulted():
    import torch

    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    b = PagedBatch(g, None, seed=16)
    ids = b.new_seqs(2)
    b.append(ids, [20, 40], "p")
    tables, lens = b.tables(ids)
    q = W.normal(16, "q", (2, 16, 128), "bf16")
    bad = tables.copy()
    bad[1, 1] = 9999  # block id out of range
    out = torch.empty((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, 2), dtype=torch.uint8, device="cuda")
    pkv.pkv_decode_attention(b.lib, 0, to_dev(q, "bf16"), b.kp, b.vp, torch.from_numpy(bad).cuda(),
                             torch.from_numpy(lens).cuda(), 0.1, out, ws)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_check_device_error()
    assert e.value.name == "PKV_ERR_DEVICE_CHECK"
    long = lens.copy()
    long[0] = 10_000  # beyond W * B
    pkv.pkv_decode_attention(b.lib, 0, to_dev(q, "bf16"), b.kp, b.vp, torch.from_numpy(tables).cuda(),
                             torch.from_numpy(long).cuda(), 0.1, out, ws)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_check_device_error()
    assert e.value.name == "PKV_ERR_DEVICE_CHECK"
    # the context is still usable
    got, t2, l2 = b.decode_gpu(ids, q, 0.1)
    check_attention(got, b.decode_ref(q, t2, l2, 0.1), "bf16")


def test_workspace_too_small_is_rejected():
    import torch

    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    b = PagedBatch(g, None, seed=17)
    ids = b.new_seqs(1)
    b.append(ids, [20], "p")
    tables, lens = b.tables(ids)
    out = torch.empty((1, 16, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention(b.lib, 0, out, b.kp, b.vp, torch.from_numpy(tables).cuda(),
                                 torch.from_numpy(lens).cuda(), 0.1, out, ws)
    assert e.value.name == "PKV_ERR_INVALID_ARG"


def test_plan_kernel_path_beyond_in_kernel_planning():
    """More than 4,096 sequences: a plan kernel computes the warps' first tiles and the
    attention kernel follows it as a programmatic dependent (two launches); lengths 0-40
    give many pairs split across warps and empty sequences."""
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=10000)
    b = PagedBatch(g, W.permutation(18, "fo", g.num_blocks), seed=18)
    lens = [int(x) for x in W.uniform_int(18, "lens", 0, 40, 4500)]
    ids = b.new_seqs(len(lens))
    b.append(ids, lens, "prompt")
    tables, sl = b.tables(ids)
    sl[::97] = 0  # a few empty sequences: zero output
    q = W.normal(18, "q", (len(ids), g.H_q, g.d_head), "bf16")
    before = pkv.pkv_launch_count()
    got, _, _ = b.decode_gpu(ids, q, 0.09, tables=tables, lens=sl)
    assert pkv.pkv_launch_count() - before == 2
    check_attention(got, b.decode_ref(q, tables, sl, 0.09), "bf16")
    assert np.all(got[::97] == 0)


def test_workspace_contents_do_not_matter():
    """The split-pair counters in the workspace carry each launch's tag, so a workspace
    holding anything -- random bytes, all ones, another batch's leftovers -- gives the
    same result without clearing: three calls on one workspace, two batches."""
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=3000)
    batches = []
    for seed, lens in ((19, [20000, 3, 700, 1]), (20, [5000, 5000, 0, 12000, 31])):
        b = PagedBatch(g, W.permutation(seed, "fo", g.num_blocks), seed=seed)
        ids = b.new_seqs(len(lens))
        b.append(ids, lens, "prompt")
        batches.append((b, ids))
    n_max = max(len(ids) for _, ids in batches)
    ws = torch.empty(pkv.pkv_decode_workspace_size(batches[0][0].lib, n_max), dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(21)
    fills = [lambda: ws.random_(0, 256, generator=gen), lambda: ws.fill_(255), lambda: None]
    for k, fill in enumerate(fills):
        b, ids = batches[k % 2]
        fill()
        tables, sl = b.tables(ids)
        q = W.normal(21, f"q{k}", (len(ids), g.H_q, g.d_head), "bf16")
        out = torch.full((len(ids), g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.pkv_decode_attention(b.lib, 0, to_dev(q, "bf16"), b.kp, b.vp, torch.from_numpy(tables).cuda(),
                                 torch.from_numpy(sl).cuda(), 0.088, out, ws)
        pkv.pkv_check_device_error()
        got = out.double().cpu().numpy()
        check_attention(got, b.decode_ref(q, tables, sl, 0.088), "bf16")


def test_two_streams_with_their_own_workspaces_at_once():
    """Two decode calls in flight at once on two streams, each with its own workspace (the
    split-pair counters live in the workspace, tagged per launch): both match the oracle, over
    several rounds of back-to-back launches."""
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=3000)
    b = PagedBatch(g, W.permutation(22, "fo", g.num_blocks), seed=22)
    lens = [20000, 7, 900, 1, 3000, 16, 17, 5000]
    ids = b.new_seqs(len(lens))
    b.append(ids, lens, "prompt")
    halves = [ids[0::2], ids[1::2]]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    work = []
    for k, part in enumerate(halves):
        tables, sl = b.tables(part)
        ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, len(part)), dtype=torch.uint8, device="cuda")
        work.append((part, tables, sl, torch.from_numpy(tables).cuda(), torch.from_numpy(sl).cuda(), ws))
    torch.cuda.synchronize()
    for rnd in range(3):
        outs, qs = [], []
        for k, (part, tables, sl, dt, dl, ws) in enumerate(work):
            q = W.normal(22, f"q{rnd}{k}", (len(part), g.H_q, g.d_head), "bf16")
            out = torch.full((len(part), g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
            qd = to_dev(q, "bf16")
            with torch.cuda.stream(streams[k]):
                pkv.pkv_decode_attention(b.lib, 0, qd, b.kp, b.vp, dt, dl, 0.0884, out, ws, stream=streams[k])
            outs.append((out, qd))
            qs.append(q)
        torch.cuda.synchronize()
        pkv.pkv_check_device_error()
        for k, (part, tables, sl, dt, dl, ws) in enumerate(work):
            check_attention(outs[k][0].double().cpu().numpy(), b.decode_ref(qs[k], tables, sl, 0.0884), "bf16")
