"""Chunked-prefill attention on the GPU against the oracle ("KV Cache Management",
"Chunked prefill mechanics": history in full, causal within the chunk)."""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev, to_raw, torch_dtype

pytestmark = pytest.mark.gpu


def run_prefill(g, history, chunks, seed, max_q=None, free_order=None):
    import torch

    b = PagedBatch(g, free_order if free_order is not None else W.permutation(seed, "fo", g.num_blocks), seed=seed)
    ids = b.new_seqs(len(history))
    b.append(ids, history, "hist")
    b.append(ids, chunks, "chunk")  # the chunk's keys/values are written first
    tables, lens = b.tables(ids)
    offs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    n_tok = int(offs[-1])
    q = W.normal(seed, "qchunk", (n_tok, g.H_q, g.d_head), g.dtype)
    out = torch.full((n_tok, g.H_q, g.d_head), float("nan"), dtype=torch_dtype(g.dtype), device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    pkv.pkv_prefill_attention(b.lib, 0, to_dev(q, g.dtype), torch.from_numpy(offs).cuda(),
                              max(chunks) if max_q is None else max_q, b.kp, b.vp, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), scale, out)
    pkv.pkv_check_device_error()
    ref = oracle.prefill_attention(g, 0, q, offs, b.hk, b.hv, tables, lens, scale)
    return check_attention(out_f64(out, g.dtype), ref, g.dtype)


@pytest.mark.parametrize("H_q,H_kv,d,B,dtype", [
    (64, 8, 128, 16, "bf16"),
    (64, 8, 64, 16, "bf16"),
    (64, 8, 128, 16, "f16"),
    (32, 8, 128, 16, "bf16"),   # G = 4
    (8, 8, 128, 32, "bf16"),    # G = 1, B = 32
    (48, 4, 128, 16, "bf16"),   # G = 12: rows of a warp span queries
    (128, 8, 128, 16, "bf16"),  # G = 16: 8 queries per 128-row tile
    (64, 1, 128, 16, "bf16"),   # G = 64 (one KV head): 2 queries per tile
    (12, 12, 64, 16, "f32"),    # CUDA-core path
    (16, 2, 96, 16, "bf16"),    # CUDA-core path
    (32, 2, 96, 16, "bf16"),    # CUDA-core path, G = 16
])
def test_prefill_geometries(H_q, H_kv, d, B, dtype):
    g = W.Geometry(L=1, H_q=H_q, H_kv=H_kv, d_head=d, block_size=B, dtype=dtype, num_blocks=800)
    run_prefill(g, [0, 5, 64, 1000, 37, 300], [17, 1, 100, 40, 130, 16], 81)


def test_prefill_ragged_chunks_and_empty_chunk():
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=1200)
    run_prefill(g, [3000, 0, 200, 15, 999], [512, 300, 0, 1, 33], 82)


def test_prefill_whole_prompt_is_causal_attention():
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=600)
    run_prefill(g, [0, 0], [1000, 257], 83)


def test_prefill_history_longer_than_the_staged_table():
    # 4,128 blocks of history: more than the 4,096 table entries the tensor-core kernel stages in
    # shared memory, so its producers read block ids from the table in global memory
    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=4400)
    run_prefill(g, [66000, 100], [40, 200], 85)


def test_prefill_chunk_longer_than_max_q_is_recorded():
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    b = PagedBatch(g, None, seed=84)
    ids = b.new_seqs(1)
    b.append(ids, [40], "c")
    tables, lens = b.tables(ids)
    q = torch.zeros((40, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    pkv.pkv_prefill_attention(b.lib, 0, q, torch.tensor([0, 40], dtype=torch.int32, device="cuda"), 16, b.kp, b.vp,
                              torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), 0.1, out)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_check_device_error()
    assert "code 6" in str(e.value)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_prefill_bench_size_sampled(dtype):
    """The prefill bench's workload -- 8 sequences of 16,384 cached tokens each take a 512-token
    chunk; 64 query / 8 KV heads, d 128; the tcgen05 kernel -- checked on sampled query rows.  A
    chunk row attends to exactly the keys up to its own position, so the oracle's decode attention
    over that prefix is its reference ("Chunked prefill mechanics": the chunked result equals a
    monolithic pass).  The oracle reads host copies of the sampled sequences' blocks taken from
    the seeded pool before any library kernel ran, with the chunk's keys/values written on the host."""
    import torch

    n, hist, C = 8, 16384, 512
    seed = 7101
    N = n * (hist + C) // 16 + 64
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype=dtype, num_blocks=N)
    kp = W.device_normal(seed, "pf_k_pool", g.pool_shape(), g.dtype, "cuda")
    vp = W.device_normal(seed, "pf_v_pool", g.pool_shape(), g.dtype, "cuda")
    b = PagedBatch(g, W.permutation(seed, "pf_fo", N), seed=seed, host_pool=False, fill_device=(kp, vp))
    ids = b.new_seqs(n)
    b.append(ids, [hist] * n, "hist", plan_only=True)  # the seeded pool holds the histories
    slots, cows = pkv.pkv_plan_append(b.lib, ids, [C] * n)
    oslots, ocows = b.orc.append(ids, [C] * n)
    assert np.array_equal(slots, oslots) and len(cows) == 0
    tables, lens = b.tables(ids)
    sample_seqs = [0, 3, 7]
    used = sorted({int(x) for s in sample_seqs for x in tables[s, : -(-int(lens[s]) // 16)]})
    remap = {blk: j for j, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    hk = to_raw(kp.index_select(0, idx), g.dtype)
    hv = to_raw(vp.index_select(0, idx), g.dtype)
    a = "bf16"  # q, out and the new keys/values (bf16 also around an E4M3 pool)
    kn = W.normal(seed, "pf_kn", (n * C, g.H_kv, g.d_head), a)
    vn = W.normal(seed, "pf_vn", (n * C, g.H_kv, g.d_head), a)
    pkv.pkv_append_kv(b.lib, 0, to_dev(kn, a), to_dev(vn, a), torch.from_numpy(slots).cuda(), kp, vp)
    q = W.normal(seed, "pf_q", (n * C, g.H_q, g.d_head), a)
    offs = np.arange(0, n * C + 1, C, dtype=np.int32)
    out = torch.full((n * C, g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / math.sqrt(g.d_head)
    pkv.pkv_prefill_attention(b.lib, 0, to_dev(q, a), torch.from_numpy(offs).cuda(), C, kp, vp,
                              torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), scale, out)
    pkv.pkv_check_device_error()
    got = out_f64(out, a)
    assert np.all(np.isfinite(got))
    gc = W.Geometry(1, g.H_q, g.H_kv, g.d_head, 16, g.dtype, len(used))
    rows = [s * C + i for s in sample_seqs for i in range(C)]
    cslots = np.array([remap[int(slots[r]) // 16] * 16 + int(slots[r]) % 16 for r in rows], np.int32)
    oracle.write_slots(gc, 0, kn[rows], vn[rows], cslots, hk, hv, b.k_scale, b.v_scale)
    samples = [(s, i) for s in sample_seqs for i in (0, 1, 17, 255, 256, 510, 511)]
    ct = np.zeros((len(samples), tables.shape[1]), np.int32)
    sl = np.zeros(len(samples), np.int32)
    for k, (s, i) in enumerate(samples):
        nb = -(-int(lens[s]) // 16)
        ct[k, :nb] = [remap[int(x)] for x in tables[s, :nb]]
        sl[k] = hist + i + 1
    picked = [s * C + i for s, i in samples]
    ref = oracle.decode_attention(gc, 0, q[picked], hk, hv, ct, sl, scale, k_scale=b.k_scale, v_scale=b.v_scale)
    check_attention(got[picked], ref, a)
