"""Swap-in overlapped with decode attention on two streams ("KV Cache Management",
"Asynchronous paged swapping": reloads stream in on an independent copy engine while
the accelerator keeps decoding).  The resident batch's results are unaffected by the
concurrent reload, and the restored sequence decodes correctly once its stream has
waited for the reload's event."""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("engine", [1, 0])
def test_swap_in_on_a_second_stream_while_decoding(engine):
    import torch

    g = W.Geometry(L=4, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=2048)
    b = PagedBatch(g, W.permutation(61, "fo", g.num_blocks), seed=61)
    pkv.pkv_pool_set_swap_engine(b.lib, engine)
    ids = b.new_seqs(9)
    lens = [1500, 2100, 700, 3000, 1999, 64, 1, 2600, 3000]
    b.append(ids, lens, "prompt", layer=-1)
    paused = ids[-1]
    resident = ids[:-1]
    n_frames = -(-3000 // 16)
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * 2
    host = torch.zeros(n_frames * frame, dtype=torch.uint8).pin_memory()
    ohost = np.zeros(n_frames * frame, np.uint8)
    frames = np.arange(n_frames)[::-1].copy()
    got = pkv.pkv_swap_out(b.lib, paused, b.kp, b.vp, host, n_frames, frames)
    oracle.swap_out_data(g, b.orc.swap_out(paused, frames), frames, b.hk, b.hv, ohost)
    torch.cuda.synchronize()
    assert pkv.pkv_seq_residency(b.lib, paused) == pkv.TIER_HOST

    s_swap, s_dec = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    # reload on its own stream ...
    new = pkv.pkv_swap_in(b.lib, paused, host, n_frames, len(frames), b.kp, b.vp, stream=s_swap)
    ev.record(s_swap)
    exp, hs = b.orc.swap_in(paused, len(frames))
    assert np.array_equal(new, exp)
    oracle.swap_in_data(g, exp, hs, ohost, b.hk, b.hv)
    assert pkv.pkv_seq_residency(b.lib, paused) == pkv.TIER_HBM
    scale = 1.0 / math.sqrt(g.d_head)
    # ... while the resident sequences decode every layer on another stream
    with torch.cuda.stream(s_dec):
        for layer in range(g.L):
            q = W.normal(61, f"q{layer}", (len(resident), g.H_q, g.d_head), "bf16")
            out, tables, lens_ = b.decode_gpu(resident, q, scale, layer=layer)
            check_attention(out, b.decode_ref(q, tables, lens_, scale, layer=layer), "bf16")
        # the restored sequence is decoded only after its reload
        s_dec.wait_event(ev)
        for layer in range(g.L):
            q = W.normal(61, f"qp{layer}", (1, g.H_q, g.d_head), "bf16")
            out, tables, lens_ = b.decode_gpu([paused], q, scale, layer=layer)
            check_attention(out, b.decode_ref(q, tables, lens_, scale, layer=layer), "bf16")
    torch.cuda.synchronize()
    b.check_state()
    b.check_pools_bitexact()
