"""Pipelined chunked reload behind chunked prefill ("KV Cache Management", "Asynchronous
paged swapping", "Pipelined Chunked Reload and Observation Prefill"): a paused sequence's
history streams back a range of layers at a time on its own stream while the observation's
chunked prefill runs on another; each layer's append and prefill attention wait only for the
event of the range that holds that layer.  Every chunk's output matches the oracle's
chunked-prefill attention, and the pools and control-plane state are bit-exact with the
oracle's after the interleaved schedule."""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev

pytestmark = pytest.mark.gpu


def _paused_batch(seed, engine, history=(3000, 700), L=4):
    import torch

    g = W.Geometry(L=L, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=2048)
    b = PagedBatch(g, W.permutation(seed, "fo", g.num_blocks), seed=seed)
    pkv.pkv_pool_set_swap_engine(b.lib, engine)
    ids = b.new_seqs(len(history))
    b.append(ids, list(history), "hist", layer=-1)
    paused = ids[0]
    nb = len(b.orc.table(paused))
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * 2
    host = torch.zeros(nb * frame, dtype=torch.uint8).pin_memory()
    ohost = np.zeros(nb * frame, np.uint8)
    frames = np.arange(nb)[::-1].copy()
    pkv.pkv_swap_out(b.lib, paused, b.kp, b.vp, host, nb, frames)
    oracle.swap_out_data(g, b.orc.swap_out(paused, frames), frames, b.hk, b.hv, ohost)
    torch.cuda.synchronize()
    return g, b, ids, host, ohost, nb


@pytest.mark.parametrize("engine,ranges", [
    (0, [(0, 1), (1, 2), (2, 4)]),  # SM copies, three ranges
    (1, [(0, 2), (2, 4)]),          # copy engines, two ranges
    (0, [(0, 4)]),                  # one range: the whole reload, as pkv_swap_in
])
def test_reload_by_layers_behind_chunked_prefill(engine, ranges):
    import torch

    g, b, ids, host, ohost, nb = _paused_batch(71, engine)
    paused, resident = ids[0], ids[1]
    s_copy, s_pre = torch.cuda.Stream(), torch.cuda.Stream()
    ev_of = {}
    for l0, l1 in ranges:  # the whole reload is queued at once on its own stream
        table = pkv.pkv_swap_in_layers(b.lib, paused, host, nb, nb, l0, l1, b.kp, b.vp, stream=s_copy)
        ev = torch.cuda.Event()
        ev.record(s_copy)
        for layer in range(l0, l1):
            ev_of[layer] = ev
        want = pkv.TIER_HBM if l1 == g.L else pkv.TIER_RELOADING
        assert pkv.pkv_seq_residency(b.lib, paused) == want
    exp, hs = b.orc.swap_in(paused, nb)
    assert np.array_equal(table, exp)
    oracle.swap_in_data(g, exp, hs, ohost, b.hk, b.hv)
    b.check_state()

    # the observation (and a resident sequence's chunk) prefilled in chunks on another stream
    scale = 1.0 / math.sqrt(g.d_head)
    chunks = [(256, 40), (256, 0), (188, 17)]
    waited = set()
    with torch.cuda.stream(s_pre):
        for c, (n_obs, n_res) in enumerate(chunks):
            run, n_new = [paused, resident], [n_obs, n_res]
            slots, _ = b.append(run, n_new, f"obs{c}", plan_only=True)
            tables, lens = b.tables(run)
            offs = np.array([0, n_obs, n_obs + n_res], np.int32)
            kv = {layer: (W.normal(71, f"k{c}_{layer}", (len(slots), g.H_kv, g.d_head), "bf16"),
                          W.normal(71, f"v{c}_{layer}", (len(slots), g.H_kv, g.d_head), "bf16")) for layer in range(g.L)}
            q = {layer: W.normal(71, f"q{c}_{layer}", (int(offs[-1]), g.H_q, g.d_head), "bf16") for layer in range(g.L)}
            d_slots = torch.from_numpy(slots).cuda()
            d_tables, d_lens, d_offs = (torch.from_numpy(x).cuda() for x in (tables, lens, offs))
            for layer in range(g.L):
                if ev_of[layer] not in waited:  # this layer's history has to be back first
                    s_pre.wait_event(ev_of[layer])
                    waited.add(ev_of[layer])
                k, v = kv[layer]
                pkv.pkv_append_kv(b.lib, layer, to_dev(k, "bf16"), to_dev(v, "bf16"), d_slots, b.kp, b.vp)
                oracle.write_slots(g, layer, k, v, slots, b.hk, b.hv)
                out = torch.full((int(offs[-1]), g.H_q, g.d_head), float("nan"), dtype=torch.bfloat16, device="cuda")
                pkv.pkv_prefill_attention(b.lib, layer, to_dev(q[layer], "bf16"), d_offs, 256, b.kp, b.vp, d_tables,
                                          d_lens, scale, out)
                ref = oracle.prefill_attention(g, layer, q[layer], offs, b.hk, b.hv, tables, lens, scale)
                check_attention(out_f64(out, "bf16"), ref, "bf16")
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    assert pkv.pkv_seq_residency(b.lib, paused) == pkv.TIER_HBM
    b.check_state()
    b.check_pools_bitexact()


def test_reload_by_layers_rejects_out_of_order_ranges_without_change():
    import torch

    g, b, ids, host, ohost, nb = _paused_batch(72, 0, history=(500,))
    paused = ids[0]
    state = lambda: (pkv.pkv_refcounts(b.lib).copy(), pkv.pkv_free_list(b.lib).copy())
    before = state()
    for l0, l1 in ((1, 2), (0, 0), (0, 5), (2, 1)):  # must start at 0; nonempty; within L
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_swap_in_layers(b.lib, paused, host, nb, nb, l0, l1, b.kp, b.vp)
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_swap_in_layers(b.lib, paused, host, nb, nb - 1, 0, 1, b.kp, b.vp)  # wrong count
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert all(np.array_equal(x, y) for x, y in zip(before, state()))
    assert pkv.pkv_seq_residency(b.lib, paused) == pkv.TIER_HOST
    pkv.pkv_swap_in_layers(b.lib, paused, host, nb, nb, 0, 1, b.kp, b.vp)
    exp, hs = b.orc.swap_in(paused, nb)
    oracle.swap_in_data(g, exp, hs, ohost, b.hk, b.hv)
    mid = state()
    for call in (lambda: pkv.pkv_swap_in_layers(b.lib, paused, host, nb, nb, 2, 4, b.kp, b.vp),  # gap
                 lambda: pkv.pkv_swap_in(b.lib, paused, host, nb, nb, b.kp, b.vp),  # not swapped out
                 lambda: pkv.pkv_swap_out(b.lib, paused, b.kp, b.vp, host, nb, np.arange(nb))):  # mid-reload
        with pytest.raises(pkv.PkvError) as e:
            call()
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert all(np.array_equal(x, y) for x, y in zip(mid, state()))
    assert np.array_equal(np.sort(pkv.pkv_seq_host_slots(b.lib, paused)), np.arange(nb))
    pkv.pkv_swap_in_layers(b.lib, paused, host, nb, nb, 1, 4, b.kp, b.vp)
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    b.check_state()
    b.check_pools_bitexact()
