"""pkv_decode_attention_noalloc: decode attention for callers that cannot allocate
device memory (e.g. an engine whose KV block pool already fills the GPU, or a hot
loop that must not take cudaMalloc's implicit device synchronisation).

The entry point uses the library's static scratch array instead of a caller
workspace.  Its output must match pkv_decode_attention's (the entry point with a
caller workspace) within the attention tolerance, on two calls in a row (the
second call reuses whatever the first left in the shared array), and both must
match the oracle's attention over the same pool.  This file is collected last so
that a failure here does not hide the other tests' results.
"""
import math

import numpy as np
import pytest

import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev, torch_dtype

pytestmark = pytest.mark.gpu


def _batch(H_q=64):
    g = W.Geometry(L=1, H_q=H_q, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=4096)
    b = PagedBatch(g, W.permutation(31, "fo", g.num_blocks), seed=31)
    lens = [int(x) for x in W.uniform_int(31, "lens", 0, 700, 40)] + [20000, 1, 16, 17]
    ids = b.new_seqs(len(lens))
    b.append(ids, lens, "prompt")
    b.append(ids, [1] * len(ids), "step")
    return b, ids


@pytest.mark.parametrize("H_q", [64, 128])  # groups of 8, and of 16 (twice the partials)
def test_noalloc_matches_workspace_entry_point_twice(H_q):
    import torch

    b, ids = _batch(H_q)
    g = b.g
    tables, lens = b.tables(ids)
    d_tables = torch.from_numpy(tables).cuda()
    d_lens = torch.from_numpy(lens).cuda()
    q_raw = W.normal(31, "q", (len(ids), g.H_q, g.d_head), "bf16")
    q = to_dev(q_raw, "bf16")
    scale = 1.0 / math.sqrt(g.d_head)
    oracle_out = b.decode_ref(q_raw, tables, lens, scale)
    ref = torch.empty((len(ids), g.H_q, g.d_head), dtype=torch_dtype(g.dtype), device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_size(b.lib, len(ids)), dtype=torch.uint8, device="cuda")
    pkv.pkv_decode_attention(b.lib, 0, q, b.kp, b.vp, d_tables, d_lens, scale, ref, ws)
    pkv.pkv_check_device_error()
    ref64 = out_f64(ref, g.dtype)
    check_attention(ref64, oracle_out, g.dtype)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        pkv.pkv_decode_attention_noalloc(b.lib, 0, q, b.kp, b.vp, d_tables, d_lens, scale, out)
        pkv.pkv_check_device_error()
        got = out_f64(out, g.dtype)
        check_attention(got, ref64, g.dtype)  # against the entry point with a caller workspace
        check_attention(got, oracle_out, g.dtype)  # and against the oracle


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    import torch

    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    lib = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks)
    n = 2_000_000  # 8 bytes of scratch per sequence on top of ~10 MB of partials: beyond 24 MiB
    lens = torch.zeros(n, dtype=torch.int32, device="cuda")
    tables = torch.zeros((n, 1), dtype=torch.int32, device="cuda")
    pool_k = torch.zeros(g.pool_shape(), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, g.H_q, g.d_head), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_noalloc(lib, 0, q, pool_k, pool_k, tables, lens, 0.1, q)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert "scratch" in str(e.value)
