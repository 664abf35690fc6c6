"""FP8 (E4M3) KV storage on the GPU against the oracle.

"KV Cache Management" (cs249r vol. 3 ch. 5), PagedAttention model: b_elem = 1 byte
for FP8.  Appends quantise bf16 keys/values with the pool scales and must store the
same codes as the oracle (bit-exact); attention over the codes must match the
oracle's float64 attention over code * scale within the bf16 tolerance; copies and
swaps move the codes bit-exactly.
"""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev, to_raw

pytestmark = pytest.mark.gpu

SCALES = [(1.0, 1.0), (0.0173, 0.5), (2.5, 0.011)]


@pytest.mark.parametrize("d", [128, 64, 8])
@pytest.mark.parametrize("kv_scales", SCALES)
def test_quantised_append_bit_exact(d, kv_scales):
    g = W.Geometry(L=3, H_q=8, H_kv=4, d_head=d, block_size=16, dtype="e4m3", num_blocks=40)
    b = PagedBatch(g, W.permutation(51, "fo", g.num_blocks), seed=51, kv_scales=kv_scales)
    ids = b.new_seqs(5)
    b.append(ids, [1, 17, 33, 0, 100], "p0", layer=-1)
    b.append(ids[::-1], [3, 1, 16, 2, 1], "p1", layer=2)
    b.append(ids, [1] * 5, "p2", layer=0)
    b.check_pools_bitexact()
    b.check_state()


def test_quantised_append_saturates_and_keeps_signed_zero():
    """Values far beyond 448 * scale are stored as +-448; values below half the
    smallest subnormal round to a signed zero -- both sides agree on every code."""
    import torch

    g = W.Geometry(L=1, H_q=4, H_kv=2, d_head=128, block_size=16, dtype="e4m3", num_blocks=8)
    b = PagedBatch(g, None, seed=52, kv_scales=(0.5, 0.02))
    (s,) = b.new_seqs(1)
    slots, _ = b.append([s], [48], "plain")
    x = W.substream(52, "wide").standard_normal((48, 2, 128)).astype(np.float32)
    x *= np.float32(10.0) ** W.substream(52, "mag").integers(-6, 5, size=(48, 2, 128)).astype(np.float32)
    k = W.f32_to_bf16_bits(x)
    v = W.f32_to_bf16_bits(-x)
    pkv.pkv_append_kv(b.lib, 0, to_dev(k, "bf16"), to_dev(v, "bf16"), torch.from_numpy(slots).cuda(), b.kp, b.vp)
    oracle.write_slots(g, 0, k, v, slots, b.hk, b.hv, b.k_scale, b.v_scale)
    b.check_pools_bitexact()
    codes = to_raw(b.kp, "e4m3")
    assert (codes == 0x7E).any() and (codes == 0xFE).any() and (codes == 0x80).any() and (codes == 0x00).any()


@pytest.mark.parametrize("H_q,H_kv,d", [(64, 8, 128), (16, 16, 128), (32, 8, 128), (16, 4, 64), (24, 2, 64), (8, 2, 96),
                                        (32, 2, 128), (72, 8, 128), (48, 4, 64), (16, 1, 256)])
def test_fp8_decode_matches_oracle(H_q, H_kv, d):
    """Ragged lengths (0, 1, tails of 1..15 tokens, multi-block), permuted blocks.
    d 128 runs on tensor cores (G 16 and 9 as two 8-head blocks); the rest on CUDA
    cores (G 12 there; more than 8 heads with d_head 256 is refused)."""
    g = W.Geometry(L=2, H_q=H_q, H_kv=H_kv, d_head=d, block_size=16, dtype="e4m3", num_blocks=700)
    b = PagedBatch(g, W.permutation(53, f"fo{H_q}{d}", g.num_blocks), seed=53, kv_scales=(0.0173, 0.25))
    lens = [0, 1, 15, 16, 17, 31, 64, 100, 257, 1000, 2049, 3, 500, 0, 33, 4095]
    if H_q // H_kv > 8 and d != 128:
        lens = [n for n in lens if n < 1000]  # the CUDA-core path handles G > 8 only with small batches quickly
    ids = b.new_seqs(len(lens))
    b.append(ids, lens, "p", layer=1)
    b.append(ids, [1] * len(ids), "t", layer=1)
    q = W.normal(53, "q", (len(ids), g.H_q, g.d_head), "bf16")
    if H_q // H_kv > 8 and d > 128:
        with pytest.raises(pkv.PkvError) as e:
            b.decode_gpu(ids, q, 1 / math.sqrt(d), layer=1)
        assert e.value.name == "PKV_ERR_UNSUPPORTED"
        return
    got, tables, sl = b.decode_gpu(ids, q, 1 / math.sqrt(d), layer=1)
    check_attention(got, b.decode_ref(q, tables, sl, 1 / math.sqrt(d), layer=1), "bf16")


def test_fp8_decode_step_with_forks_and_copy_on_write():
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="e4m3", num_blocks=512)
    b = PagedBatch(g, W.permutation(54, "fo", g.num_blocks), seed=54, kv_scales=(0.05, 0.125))
    ids = b.new_seqs(5)
    b.append(ids, [40, 16, 300, 1, 77], "prompt")
    kids = [b.fork(ids[0]), b.fork(ids[2])]
    run = np.array(ids + kids, np.int32)
    n, Wd = len(run), 24
    meta_host = torch.zeros(n * (Wd + 2), dtype=torch.int32).pin_memory()
    meta_dev = torch.zeros(n * (Wd + 2), dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, n), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    for step in range(3):
        q = W.normal(54, f"q{step}", (n, g.H_q, g.d_head), "bf16")
        kn = W.normal(54, f"k{step}", (n, g.H_kv, g.d_head), "bf16")
        vn = W.normal(54, f"v{step}", (n, g.H_kv, g.d_head), "bf16")
        out = torch.full((n, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.pkv_decode_step(b.lib, 0, run, Wd, to_dev(q, "bf16"), to_dev(kn, "bf16"), to_dev(vn, "bf16"),
                            b.kp, b.vp, scale, out, meta_host, meta_dev, ws)
        oslots, ocows = b.orc.append(run.tolist(), [1] * n)
        if len(ocows):
            oracle.copy_blocks(g, ocows, b.hk, b.hv)
        oracle.write_slots(g, 0, kn, vn, oslots, b.hk, b.hv, b.k_scale, b.v_scale)
        pkv.pkv_check_device_error()
        tables, lens = b.tables(run.tolist(), Wd)
        check_attention(out_f64(out, "bf16"), b.decode_ref(q, tables, lens, scale), "bf16")
        b.check_state()
    b.check_pools_bitexact()


def test_fp8_noalloc_equals_workspace_call():
    import torch

    g = W.Geometry(L=1, H_q=32, H_kv=4, d_head=128, block_size=16, dtype="e4m3", num_blocks=900)
    b = PagedBatch(g, W.permutation(55, "fo", g.num_blocks), seed=55, kv_scales=(0.3, 0.7))
    ids = b.new_seqs(12)
    b.append(ids, [5, 900, 17, 1, 2000, 64, 0, 3000, 48, 700, 333, 1200], "p")
    q = W.normal(55, "q", (len(ids), g.H_q, g.d_head), "bf16")
    got, tables, lens = b.decode_gpu(ids, q, 0.09)
    out = torch.full((len(ids), g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_attention_noalloc(b.lib, 0, to_dev(q, "bf16"), b.kp, b.vp, torch.from_numpy(tables).cuda(),
                                     torch.from_numpy(lens).cuda(), 0.09, out)
    pkv.pkv_check_device_error()
    assert np.array_equal(out_f64(out, "bf16"), got)
    check_attention(got, b.decode_ref(q, tables, lens, 0.09), "bf16")


def _fp8_prefill(H_q, H_kv, d, history, chunks, seed, scales, num_blocks):
    import torch

    g = W.Geometry(L=1, H_q=H_q, H_kv=H_kv, d_head=d, block_size=16, dtype="e4m3", num_blocks=num_blocks)
    b = PagedBatch(g, W.permutation(seed, "fo", g.num_blocks), seed=seed, kv_scales=scales)
    ids = b.new_seqs(len(history))
    b.append(ids, history, "history")
    b.append(ids, chunks, "chunk")
    tables, lens = b.tables(ids)
    qo = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = W.normal(seed, "q", (int(qo[-1]), g.H_q, g.d_head), "bf16")
    out = torch.full((int(qo[-1]), g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / math.sqrt(d)
    pkv.pkv_prefill_attention(b.lib, 0, to_dev(q, "bf16"), torch.from_numpy(qo).cuda(), max(chunks), b.kp, b.vp,
                              torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), scale, out)
    pkv.pkv_check_device_error()
    ref = oracle.prefill_attention(g, 0, q, qo, b.hk, b.hv, tables, lens, scale, k_scale=b.k_scale,
                                   v_scale=b.v_scale)
    check_attention(out_f64(out, "bf16"), ref, "bf16")


@pytest.mark.parametrize("H_q,H_kv", [(64, 8), (16, 4), (48, 4), (8, 8), (128, 8)])
def test_fp8_prefill_tensor_cores(H_q, H_kv):
    # d_head 128: tcgen05 kernel on binary16 operands converted from the codes in shared memory;
    # ragged chunks (one query, a 16-query tile, 512), empty and long histories, ragged tails
    _fp8_prefill(H_q, H_kv, 128, [0, 5, 64, 1000, 37, 300, 3000], [17, 1, 100, 40, 130, 16, 512], 56, (0.1, 0.4), 400)


def test_fp8_prefill_history_longer_than_the_staged_table():
    _fp8_prefill(16, 2, 128, [66000, 100], [40, 200], 59, (0.1, 0.2), 4400)


def test_fp8_prefill_on_cuda_cores():
    # d_head 64 over an E4M3 pool runs on the CUDA-core kernel
    _fp8_prefill(16, 4, 64, [100, 0, 700], [37, 16, 5], 58, (0.2, 0.3), 200)


@pytest.mark.parametrize("engine", [0, 1])
def test_fp8_swap_round_trip_bit_exact(engine):
    import torch

    g = W.Geometry(L=4, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="e4m3", num_blocks=48)
    b = PagedBatch(g, W.permutation(57, "fo", g.num_blocks), seed=57, kv_scales=(0.2, 0.2))
    pkv.pkv_pool_set_swap_engine(b.lib, engine)
    ids = b.new_seqs(3)
    b.append(ids, [64, 20, 48], "fill", layer=-1)
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * 1  # M_block with b_elem = 1
    host = torch.zeros(16 * frame, dtype=torch.uint8).pin_memory()
    ohost = np.zeros(16 * frame, np.uint8)
    frames = {0: np.arange(0, 4), 2: np.arange(8, 11)[::-1].copy()}
    for s, fr in frames.items():
        got = pkv.pkv_swap_out(b.lib, s, b.kp, b.vp, host, 16, fr)
        exp = b.orc.swap_out(s, fr)
        assert np.array_equal(got, exp)
        oracle.swap_out_data(g, exp, fr, b.hk, b.hv, ohost)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), ohost)
    b.append([ids[1]], [40], "reuse", layer=-1)
    for s, fr in frames.items():
        got = pkv.pkv_swap_in(b.lib, s, host, 16, len(fr), b.kp, b.vp)
        exp, hs = b.orc.swap_in(s, len(fr))
        assert np.array_equal(got, exp)
        oracle.swap_in_data(g, exp, hs, ohost, b.hk, b.hv)
    b.check_pools_bitexact()
    b.check_state()


def test_fp8_agent_32k_sampled():
    """48 sequences x 32,768 tokens over a 3.2 GB FP8 pool (codes of N(0,1) draws) at
    permuted block ids; sampled sequences against the oracle over their own blocks."""
    import torch

    wl = W.agent(48, 32768, spare_steps=32)
    g0 = wl.geometry
    g = W.Geometry(g0.L, g0.H_q, g0.H_kv, g0.d_head, g0.block_size, "e4m3", g0.num_blocks)
    kp = W.device_normal(wl.seed, "k_pool_fp8", g.pool_shape(), "e4m3", "cuda")
    vp = W.device_normal(wl.seed, "v_pool_fp8", g.pool_shape(), "e4m3", "cuda")
    b = PagedBatch(g, wl.free_order, seed=wl.seed, host_pool=False, fill_device=(kp, vp), kv_scales=(0.5, 0.75))
    ids = b.new_seqs(48)
    b.append(ids, [32768] * 48, "prompt", plan_only=True)
    tables, lens = b.tables(ids)
    q = W.normal(wl.seed, "q_fp8", (48, g.H_q, g.d_head), "bf16")
    got, _, _ = b.decode_gpu(ids, q, wl.scale, tables=tables, lens=lens)
    assert np.all(np.isfinite(got))
    sample = [0, 29, 47]
    used = sorted({int(x) for r in sample for x in tables[r]})
    remap = {blk: j for j, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    hk = kp.index_select(0, idx).cpu().numpy()
    hv = vp.index_select(0, idx).cpu().numpy()
    gc = W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, "e4m3", len(used))
    ct = np.array([[remap[int(x)] for x in tables[r]] for r in sample], np.int32)
    ref = oracle.decode_attention(gc, 0, q[sample], hk, hv, ct, lens[sample], wl.scale, k_scale=b.k_scale,
                                  v_scale=b.v_scale)
    check_attention(got[sample], ref, "bf16")
