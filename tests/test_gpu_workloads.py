"""Full-size workloads on the GPU against the oracle.

Control-plane state (slots, copy-on-write pairs, tables, reference counts, FIFO)
is compared exactly at every step.  Attention is compared element by element on
every sequence where the oracle is cheap (chat, forked samples) and on sampled
sequences where it is not (32K / 131K contexts): for those the oracle gets host
copies of exactly the sampled sequences' blocks, taken from the seeded pool before
any library kernel ran, plus the step's new tokens written on the host.
"""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention, out_f64, to_dev, to_raw, torch_dtype

pytestmark = pytest.mark.gpu


def test_chat_64_steps_full():
    """256 ragged sequences, 32,768-block pool in shuffled order, 64 decode steps with
    per-step appends; finished sequences release their blocks."""
    wl = W.chat()
    g = wl.geometry
    b = PagedBatch(g, wl.free_order, seed=wl.seed)
    ids = b.new_seqs(len(wl.lengths))
    b.append(ids, [int(x) for x in wl.lengths], "prompt")
    gen = wl.extra["generated"]
    live = list(ids)
    for k in range(wl.extra["steps"]):
        run = [s for s in live if gen[s] > k]
        if not run:
            break
        b.append(run, [1] * len(run), f"s{k}")
        tables, lens = b.tables(run)
        q = W.normal(wl.seed, f"q{k}", (len(run), g.H_q, g.d_head), g.dtype)
        got, _, _ = b.decode_gpu(run, q, wl.scale, tables=tables, lens=lens)
        check_attention(got, b.decode_ref(q, tables, lens, wl.scale), g.dtype)  # every step, every sequence
        for s in run:
            if gen[s] == k + 1:
                b.free(s)
                live.remove(s)
        b.check_state()
    b.check_pools_bitexact()
    for s in list(live):
        b.free(s)
    assert np.all(pkv.pkv_refcounts(b.lib) == 0)
    assert sorted(pkv.pkv_free_list(b.lib).tolist()) == list(range(g.num_blocks))


def _sampled_agent_step(n_seq, context, sample):
    import torch

    wl = W.agent(n_seq, context, spare_steps=32)
    g = wl.geometry
    kp = W.device_normal(wl.seed, f"k_pool_{n_seq}_{context}", g.pool_shape(), g.dtype, "cuda")
    vp = W.device_normal(wl.seed, f"v_pool_{n_seq}_{context}", g.pool_shape(), g.dtype, "cuda")
    b = PagedBatch(g, wl.free_order, seed=wl.seed, host_pool=False, fill_device=(kp, vp))
    ids = b.new_seqs(n_seq)
    b.append(ids, [context] * n_seq, "prompt", plan_only=True)  # the seeded pool holds the prompt
    # one decode step: plan the appended token, snapshot the sampled blocks, then run the step
    slots, cows = pkv.pkv_plan_append(b.lib, ids, [1] * n_seq)
    oslots, ocows = b.orc.append(ids, [1] * n_seq)
    assert np.array_equal(slots, oslots) and len(cows) == 0
    tables, lens = b.tables(ids)
    used = sorted({int(x) for r in sample for x in tables[r, : -(-int(lens[r]) // g.block_size)]})
    remap = {blk: j for j, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    hk = to_raw(kp.index_select(0, idx), g.dtype)
    hv = to_raw(vp.index_select(0, idx), g.dtype)
    kn = W.normal(wl.seed, "step_k", (n_seq, g.H_kv, g.d_head), g.dtype)
    vn = W.normal(wl.seed, "step_v", (n_seq, g.H_kv, g.d_head), g.dtype)
    pkv.pkv_append_kv(b.lib, 0, to_dev(kn, g.dtype), to_dev(vn, g.dtype), torch.from_numpy(slots).cuda(), kp, vp)
    q = W.normal(wl.seed, "step_q", (n_seq, g.H_q, g.d_head), g.dtype)
    got, _, _ = b.decode_gpu(ids, q, wl.scale, tables=tables, lens=lens)
    # oracle: the sampled sequences over their own blocks, new tokens written on the host
    gc = W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, len(used))
    cslots = np.array([remap[int(slots[r]) // g.block_size] * g.block_size + int(slots[r]) % g.block_size
                       for r in sample], np.int32)
    oracle.write_slots(gc, 0, kn[sample], vn[sample], cslots, hk, hv)
    ct = np.zeros((len(sample), tables.shape[1]), np.int32)
    for i, r in enumerate(sample):
        nb = -(-int(lens[r]) // g.block_size)
        ct[i, :nb] = [remap[int(x)] for x in tables[r, :nb]]
    ref = oracle.decode_attention(gc, 0, q[sample], hk, hv, ct, lens[sample], wl.scale)
    check_attention(got[sample], ref, g.dtype)
    assert np.all(np.isfinite(got))
    return got


@pytest.mark.parametrize("n_seq,context,sample", [
    (48, 32768, [0, 23, 47]),
    (192, 8192, [0, 100, 191]),
    (12, 131072, [0, 11]),
])
def test_agent_long_context_sampled(n_seq, context, sample):
    """6.4 GB of K/V at permuted block ids: 48 x 32K, and the fixed-footprint sweep."""
    _sampled_agent_step(n_seq, context, sample)


def test_forked_prefix_with_cow_full():
    """16,376-token prefix (1,023 full blocks + 8 tokens) forked into 64 branches:
    refcount 65 on the shared blocks; every branch's first write copies the shared
    tail block; decode steps with refcounts checked after each."""
    wl = W.forked()
    g = wl.geometry
    b = PagedBatch(g, wl.free_order, seed=wl.seed)
    (parent,) = b.new_seqs(1)
    b.append([parent], [int(wl.lengths[0])], "prefix")
    kids = [b.fork(parent) for _ in range(wl.extra["n_branch"])]
    ptable = b.orc.table(parent)
    assert len(ptable) == 1024
    assert set(pkv.pkv_refcounts(b.lib)[ptable].tolist()) == {65}
    suffix = [int(x) for x in wl.extra["suffix"]]
    _, cows = b.append(kids, suffix, "suffix")
    assert len(cows) == sum(1 for s in suffix if s > 0)
    assert all(c[0] == ptable[-1] for c in cows)  # every copy is of the shared tail block
    b.check_state()
    sample = list(range(0, 64, 4))
    for step in range(3):
        b.append(kids, [1] * len(kids), f"d{step}")
        b.check_state()
        tables, lens = b.tables(kids)
        q = W.normal(wl.seed, f"q{step}", (len(kids), g.H_q, g.d_head), g.dtype)
        got, _, _ = b.decode_gpu(kids, q, wl.scale, tables=tables, lens=lens)
        ref = b.decode_ref(q[sample], tables[sample], lens[sample], wl.scale)
        check_attention(got[sample], ref, g.dtype)
    # after every branch wrote, the shared prefix blocks are still owned by all 65
    assert set(pkv.pkv_refcounts(b.lib)[ptable[:-1]].tolist()) == {65}
    b.check_pools_bitexact()


def test_swap_full_size_every_image():
    """80-layer geometry (5 MiB blocks): 512 chunk sequences of 16 blocks (42.9 GB)
    evicted to pinned host frames in a seeded order, then a seeded half restored into
    different blocks.  Bookkeeping exact; every host frame and every restored block
    bit-exact against the pool's bytes from before the first eviction.

    The expected bytes are a copy of the seeded pool taken on the device before any
    library kernel ran (the pool and its copy fit in HBM; host copies of 43 GB would
    not fit a test's time budget); the comparisons are whole-tensor equality, chunk by
    chunk (16 frames, 80 MiB at a time)."""
    import torch

    wl = W.swap()
    g = wl.geometry
    cb = wl.extra["chunk_blocks"]
    nchunk = len(wl.lengths)
    kp = W.device_normal(wl.seed, "k_pool", g.pool_shape(), g.dtype, "cuda")
    vp = W.device_normal(wl.seed, "v_pool", g.pool_shape(), g.dtype, "cuda")
    kp0, vp0 = kp.clone(), vp.clone()  # the pool before any library kernel
    b = PagedBatch(g, wl.free_order, seed=wl.seed, host_pool=False, fill_device=(kp, vp))
    ids = b.new_seqs(nchunk)
    b.append(ids, [int(x) for x in wl.lengths], "chunks", plan_only=True)  # the seeded pool holds the data
    restore = [int(x) for x in wl.extra["restore"]]
    before = {s: b.orc.table(s).astype(np.int64) for s in ids}
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * g.elem_bytes
    assert frame == 16 * 327680
    host = torch.empty(nchunk * cb * frame, dtype=torch.uint8, pin_memory=True)
    order = [int(x) for x in wl.extra["evict_order"]]
    old_ids = set()
    for i, s in enumerate(order):
        frames = np.arange(i * cb, (i + 1) * cb, dtype=np.int64)
        got = pkv.pkv_swap_out(b.lib, s, kp, vp, host, nchunk * cb, frames)
        assert np.array_equal(got, b.orc.swap_out(s, frames))
        old_ids.update(got.tolist())
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    b.check_state()

    def image(pool, blocks):  # [n][L*H_kv*B*d] raw bytes of the given blocks
        return pool.index_select(0, blocks).view(len(blocks), -1).view(torch.uint8)

    # every host frame: [K image | V image] of the block it was evicted from
    hview = host.view(nchunk * cb, 2, -1)
    for i, s in enumerate(order):
        t = torch.from_numpy(before[s]).cuda()
        got = hview[i * cb:(i + 1) * cb].to("cuda", non_blocking=True)
        assert torch.equal(got[:, 0], image(kp0, t)), f"K frames of chunk {s}"
        assert torch.equal(got[:, 1], image(vp0, t)), f"V frames of chunk {s}"
    for s in restore:
        got = pkv.pkv_swap_in(b.lib, s, host, nchunk * cb, cb, kp, vp)
        exp, _ = b.orc.swap_in(s, cb)
        assert np.array_equal(got, exp)
        assert not set(got.tolist()) & old_ids  # different physical blocks
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    b.check_state()
    # every restored block equals the block its frame was evicted from
    for s in restore:
        new = torch.from_numpy(b.orc.table(s).astype(np.int64)).cuda()
        old = torch.from_numpy(before[s]).cuda()
        assert torch.equal(image(kp, new), image(kp0, old)), f"restored K of chunk {s}"
        assert torch.equal(image(vp, new), image(vp0, old)), f"restored V of chunk {s}"
