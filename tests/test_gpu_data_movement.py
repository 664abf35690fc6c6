"""Append, copy-on-write copies and swaps on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, to_dev, to_raw

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64), ("bf16", 6)])
def test_append_per_layer_and_all_layers(dtype, d):
    g = W.Geometry(L=3, H_q=8, H_kv=4, d_head=d, block_size=16, dtype=dtype, num_blocks=40)
    b = PagedBatch(g, W.permutation(1, "fo", g.num_blocks), seed=1)
    ids = b.new_seqs(5)
    b.append(ids, [1, 17, 33, 0, 100], "p0", layer=-1)  # all layers at once
    b.append(ids[::-1], [3, 1, 16, 2, 1], "p1", layer=2)  # one layer
    b.append(ids, [1] * 5, "p2", layer=0)
    b.check_pools_bitexact()
    b.check_state()


def test_append_skips_bad_slots_and_reports_them():
    import torch

    g = W.Geometry(L=1, H_q=2, H_kv=2, d_head=8, block_size=4, dtype="bf16", num_blocks=4)
    b = PagedBatch(g, None, seed=2)
    k = W.normal(2, "k", (3, 2, 8), "bf16")
    slots = torch.tensor([1, 16, -3], dtype=torch.int32, device="cuda")
    pkv.pkv_append_kv(b.lib, 0, to_dev(k, "bf16"), to_dev(k, "bf16"), slots, b.kp, b.vp)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_check_device_error()
    assert e.value.name == "PKV_ERR_DEVICE_CHECK"
    oracle.write_slots(g, 0, k[:1], k[:1], np.array([1], np.int32), b.hk, b.hv)
    b.check_pools_bitexact()  # only the valid slot was written
    assert pkv.pkv_check_device_error() == (0, 0)  # cleared


@pytest.mark.parametrize("L,dtype", [(1, "bf16"), (4, "f32"), (80, "bf16")])
def test_copy_blocks_whole_blocks(L, dtype):
    g = W.Geometry(L=L, H_q=8, H_kv=8 if L < 80 else 8, d_head=128, block_size=16, dtype=dtype, num_blocks=24)
    b = PagedBatch(g, None, seed=3)
    raw_k = W.normal(3, "pk", g.pool_shape(), dtype)
    raw_v = W.normal(3, "pv", g.pool_shape(), dtype)
    b.kp.copy_(to_dev(raw_k, dtype))
    b.vp.copy_(to_dev(raw_v, dtype))
    b.hk[...] = raw_k
    b.hv[...] = raw_v
    pairs = np.array([[3, 7], [3, 8], [20, 0], [11, 23]], np.int32)
    pkv.pkv_copy_blocks(b.lib, pairs, b.kp, b.vp)
    oracle.copy_blocks(g, pairs, b.hk, b.hv)
    b.check_pools_bitexact()


def test_copy_blocks_rejects_bad_pairs_before_launch():
    g = W.Geometry(L=1, H_q=2, H_kv=2, d_head=8, block_size=4, dtype="bf16", num_blocks=4)
    b = PagedBatch(g, None)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_copy_blocks(b.lib, [[0, 4]], b.kp, b.vp)
    assert e.value.name == "PKV_ERR_BAD_BLOCK_ID"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_copy_blocks(b.lib, [[0, 1], [1, 2]], b.kp, b.vp)
    assert e.value.name == "PKV_ERR_INVALID_ARG"


def test_fork_then_append_copies_shared_tail():
    """A forked branch's first write copies the shared tail block (CoW) on the device."""
    g = W.Geometry(L=2, H_q=8, H_kv=2, d_head=64, block_size=16, dtype="bf16", num_blocks=32)
    b = PagedBatch(g, W.permutation(4, "fo", g.num_blocks), seed=4)
    (p,) = b.new_seqs(1)
    b.append([p], [40], "prefix", layer=-1)
    kids = [b.fork(p) for _ in range(3)]
    b.check_state()
    b.append(kids + [p], [1, 5, 0, 2], "div", layer=-1)
    assert b.n_cow == 3  # two branches and the parent write; the last owner writes in place
    b.check_pools_bitexact()
    b.check_state()


@pytest.mark.parametrize("engine", [0, 1])
def test_swap_round_trip_bit_exact(engine):
    import torch

    g = W.Geometry(L=4, H_q=8, H_kv=2, d_head=64, block_size=16, dtype="bf16", num_blocks=48)
    b = PagedBatch(g, W.permutation(5, "fo", g.num_blocks), seed=5)
    pkv.pkv_pool_set_swap_engine(b.lib, engine)
    ids = b.new_seqs(4)
    b.append(ids, [64, 20, 1, 48], "fill", layer=-1)
    frame_bytes = 2 * g.L * g.H_kv * g.block_size * g.d_head * 2
    host = torch.zeros(16 * frame_bytes, dtype=torch.uint8).pin_memory()
    ohost = np.zeros(16 * frame_bytes, np.uint8)
    before = {s: b.orc.table(s) for s in ids}
    order = [2, 0, 3]
    next_frame = 0
    for s in order:
        n = len(before[s])
        frames = np.arange(next_frame, next_frame + n)[::-1].copy()
        next_frame += n
        got = pkv.pkv_swap_out(b.lib, s, b.kp, b.vp, host, 16, frames)
        exp = b.orc.swap_out(s, frames)
        assert np.array_equal(got, exp)
        oracle.swap_out_data(g, exp, frames, b.hk, b.hv, ohost)
        assert np.array_equal(pkv.pkv_seq_host_slots(b.lib, s), frames)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), ohost)
    b.check_state()
    # the freed blocks are reused: append to the resident sequence
    b.append([ids[1]], [40], "reuse", layer=-1)
    for s in [3, 2]:
        n = len(before[s])
        front = pkv.pkv_free_list(b.lib)[:n].copy()
        got = pkv.pkv_swap_in(b.lib, s, host, 16, n, b.kp, b.vp)
        exp, hs = b.orc.swap_in(s, n)
        assert np.array_equal(got, exp)
        assert np.array_equal(got, front)  # the restored blocks are the FIFO's first n ids, in order
        oracle.swap_in_data(g, exp, hs, ohost, b.hk, b.hv)
    b.check_pools_bitexact()
    b.check_state()
    # images restored into the new blocks equal the originals
    for s in [3, 2]:
        assert b.orc.seq_len(s) == pkv.pkv_seq_len(b.lib, s)


def test_swap_errors_change_nothing():
    import torch

    g = W.Geometry(L=1, H_q=2, H_kv=2, d_head=8, block_size=4, dtype="bf16", num_blocks=8)
    b = PagedBatch(g, None)
    (s,) = b.new_seqs(1)
    b.append([s], [9], "x")
    host = torch.zeros(4 * 2 * 2 * 4 * 8 * 2, dtype=torch.uint8).pin_memory()
    state = (pkv.pkv_refcounts(b.lib).copy(), pkv.pkv_free_list(b.lib).copy())
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_swap_out(b.lib, s, b.kp, b.vp, host, 4, [0, 1, 4])  # frame 4 out of range
    assert e.value.name == "PKV_ERR_BAD_BLOCK_ID"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_swap_out(b.lib, s, b.kp, b.vp, host, 4, [0, 1, 1])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_swap_out(b.lib, s, b.kp, b.vp, host, 4, [0, 1])  # wrong count
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert np.array_equal(state[0], pkv.pkv_refcounts(b.lib))
    assert np.array_equal(state[1], pkv.pkv_free_list(b.lib))
    pkv.pkv_swap_out(b.lib, s, b.kp, b.vp, host, 4, [0, 1, 2])
    b.orc.swap_out(s, [0, 1, 2])
    # pool too full to swap back in
    t = b.new_seqs(1)
    b.append(t, [32], "fill")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_swap_in(b.lib, s, host, 4, 3, b.kp, b.vp)
    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
