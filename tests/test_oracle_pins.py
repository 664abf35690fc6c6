"""Pins of the CPU oracle against facts the pages fix (no GPU).

Each test checks the oracle against something other than itself: a worked example
the pages print (fixtures in tests/golden/, each with its citation), a closed
form, an invariant, or a library routine (torch's scaled-dot-product attention in
float64) on the special case the paged definition reduces to.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def storage(dtype):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]


def empty_pools(g):
    return (np.zeros(g.pool_shape(), storage(g.dtype)), np.zeros(g.pool_shape(), storage(g.dtype)))


def build_case(g, lens, seed, free_order=None):
    """Allocate sequences of the given lengths through the oracle, write random K/V
    for every token, and return everything needed to check attention."""
    pool = oracle.Pool(g.num_blocks, g.block_size, free_order)
    kp, vp = empty_pools(g)
    ids = [pool.seq_create() for _ in lens]
    ks, vs = [], []
    for i, (sid, n) in enumerate(zip(ids, lens)):
        k = W.normal(seed, f"k{i}", (n, g.H_kv, g.d_head), g.dtype)
        v = W.normal(seed, f"v{i}", (n, g.H_kv, g.d_head), g.dtype)
        if n:
            slots, cows = pool.append([sid], [n])
            assert len(cows) == 0
            oracle.write_slots(g, 0, k, v, slots, kp, vp)
        ks.append(k)
        vs.append(v)
    q = W.normal(seed, "q", (len(lens), g.H_q, g.d_head), g.dtype)
    Wt = max([-(-n // g.block_size) for n in lens] + [1])
    tables, seq_lens = pool.tables(ids, Wt)
    return pool, ids, kp, vp, ks, vs, q, tables, seq_lens


def sdpa_reference(g, q, ks, vs, scale):
    """torch scaled_dot_product_attention in float64 on contiguous K/V, with KV head
    g serving query heads g*G .. g*G+G-1."""
    G = g.H_q // g.H_kv
    out = np.zeros((len(ks), g.H_q, g.d_head))
    for s, (k, v) in enumerate(zip(ks, vs)):
        if len(k) == 0:
            continue
        qt = torch.from_numpy(W.to_float64(q[s], g.dtype)).view(1, g.H_q, 1, g.d_head)
        kt = torch.from_numpy(W.to_float64(k, g.dtype)).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        vt = torch.from_numpy(W.to_float64(v, g.dtype)).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        out[s] = o[0, :, 0, :].numpy()
    return out


# ------------------------------------------------------------------ geometry


@pytest.mark.parametrize("case", golden("geometry.json")["cases"], ids=lambda c: c["name"])
def test_block_image_bytes_match_page_footprint(case):
    """A one-token block's host frame is exactly the page's bytes per token
    (2 * L * H_kv * d_head * b); a 16-token block is 16 times that."""
    B = case.get("block_size", 1)
    g = W.Geometry(L=case["L"], H_q=case["H_kv"], H_kv=case["H_kv"], d_head=case["d_head"], block_size=B,
                   dtype="bf16", num_blocks=2)
    kp = W.normal(1, "k", g.pool_shape(), "bf16")
    vp = W.normal(1, "v", g.pool_shape(), "bf16")
    frame = case["bytes_per_token"] * B
    host = np.full(3 * frame, 0xAB, np.uint8)
    oracle.swap_out_data(g, [1], [1], kp, vp, host)
    assert np.all(host[:frame] == 0xAB) and np.all(host[2 * frame:] == 0xAB)
    expect = np.concatenate([kp[1].view(np.uint8).ravel(), vp[1].view(np.uint8).ravel()])
    assert expect.size == frame
    assert np.array_equal(host[frame:2 * frame], expect)
    if "bytes_per_block" in case:
        assert frame == case["bytes_per_block"]
        assert case["pool_bytes"] // frame == case["pool_blocks"]


# ------------------------------------------------------------------ block tables


@pytest.mark.parametrize("case", golden("block_tables.json")["table_lengths"], ids=lambda c: str(c["tokens"]))
def test_table_lengths(case):
    B = case["block_size"]
    n = case["tokens"]
    pool = oracle.Pool(case["blocks"] + 3, B)
    s = pool.seq_create()
    slots, _ = pool.append([s], [n])
    table = pool.table(s)
    assert len(table) == case["blocks"]
    # slot of token t is T[t // B] * B + t % B
    t = np.arange(n)
    assert np.array_equal(slots, table[t // B] * B + t % B)
    if "tail_tokens" in case:
        assert n // B == case["full_blocks"] and n % B == case["tail_tokens"]
        tail = slots[case["full_blocks"] * B:]
        assert np.array_equal(tail % B, np.arange(case["tail_tokens"]))


def test_tail_waste_mean():
    """Allocated-but-unused slots averaged over lengths uniform mod B = (B-1)/2."""
    fx = golden("block_tables.json")["tail_waste"]
    B = fx["block_size"]
    waste = []
    for S in range(1, 10 * B + 1):
        pool = oracle.Pool(16, B)
        s = pool.seq_create()
        pool.append([s], [S])
        waste.append(len(pool.table(s)) * B - S)
    assert np.mean(waste) == pytest.approx(fx["expected_tokens"], abs=1e-12)


def _fig5_pool():
    fx = golden("block_tables.json")["figure5"]
    head = fx["free_order_head"]
    rest = [i for i in range(16) if i not in head]
    return fx, oracle.Pool(16, fx["block_size"], np.array(head + rest, np.int32))


def test_figure5_fork_then_copy_on_write():
    """Figure 5, read as: A holds 10 tokens in blocks 7, 3, 1; B forks and writes
    into logical block 2, which is shared, so B copies it into the next free block."""
    fx, pool = _fig5_pool()
    a = pool.seq_create()
    pool.append([a], [10])
    assert list(pool.table(a)) == fx["seq_a_table"]
    b = pool.seq_fork(a)
    ref = pool.refcounts()
    assert all(ref[p] == fx["shared_refcount"] for p in fx["seq_a_table"])
    slots, cows = pool.append([b], [1])
    assert [list(c) for c in cows] == [[1, 12]]
    assert list(pool.table(a)) == fx["seq_a_table"]
    assert list(pool.table(b)) == fx["seq_b_table"]
    ref = pool.refcounts()
    assert all(ref[p] == fx["shared_refcount"] for p in fx["shared_blocks"])
    assert ref[1] == 1 and ref[12] == 1
    assert slots[0] == 12 * fx["block_size"] + 2


def test_figure5_fork_at_block_boundary():
    """Figure 5, read as: A holds two full blocks 7, 3; B forks; each then writes a
    new logical block 2 (A first: block 1; B: block 12).  Same ids, no copy."""
    fx, pool = _fig5_pool()
    a = pool.seq_create()
    pool.append([a], [8])
    b = pool.seq_fork(a)
    _, cows = pool.append([a, b], [1, 1])
    assert len(cows) == 0
    assert list(pool.table(a)) == fx["seq_a_table"]
    assert list(pool.table(b)) == fx["seq_b_table"]
    ref = pool.refcounts()
    assert all(ref[p] == fx["shared_refcount"] for p in fx["shared_blocks"])


@pytest.mark.parametrize("one_call", [False, True])
def test_fork_40_tokens(one_call):
    fx = golden("block_tables.json")["fork_40"]
    B = fx["block_size"]
    pool = oracle.Pool(32, B)
    a = pool.seq_create()
    pool.append([a], [fx["prefix_tokens"]])
    in_use = lambda: int((pool.refcounts() > 0).sum())
    assert in_use() == fx["blocks_after_prefix"]
    b = pool.seq_fork(a)
    assert in_use() == fx["blocks_after_fork"]
    assert set(pool.refcounts()[pool.table(a)]) == {fx["refcount_after_fork"]}
    if one_call:
        # ascending id order: a writes first
        _, cows = pool.append([b, a], [1, 1])
        assert len(cows) == 1 and cows[0][0] == pool.table(b)[2]
        assert in_use() == fx["blocks_after_second_write"]
    else:
        _, cows = pool.append([b], [1])
        assert (len(cows) == 1) == fx["first_writer_copies"]
        assert in_use() == fx["blocks_after_first_write"]
        _, cows = pool.append([a], [1])
        assert (len(cows) == 1) == fx["second_writer_copies"]
        assert in_use() == fx["blocks_after_second_write"]
    # the two full prefix blocks stay shared
    assert list(pool.table(a)[:2]) == list(pool.table(b)[:2])
    assert set(pool.refcounts()[pool.table(a)[:2]]) == {2}


# ------------------------------------------------------------------ allocator invariants


def _check_invariants(pool, live):
    ref = pool.refcounts()
    free = pool.free_list()
    assert len(set(free.tolist())) == len(free)
    assert np.all(ref[free] == 0)
    owners = np.zeros_like(ref)
    for s in live:
        for p in pool.table(s):
            owners[p] += 1
    assert np.array_equal(owners, ref)
    assert len(free) + int((ref > 0).sum()) == pool.num_blocks


def test_random_ops_keep_counts_and_release_everything():
    rng = W.substream(11, "ops")
    for B in (1, 4, 16):
        pool = oracle.Pool(64, B, W.permutation(11, f"fo{B}", 64))
        live = []
        for step in range(400):
            op = rng.integers(0, 4)
            try:
                if op == 0 or not live:
                    live.append(pool.seq_create())
                elif op == 1:
                    k = int(rng.integers(1, min(len(live), 4) + 1))
                    sel = list(rng.choice(live, size=k, replace=False))
                    pool.append(sel, rng.integers(0, 2 * B + 1, size=k))
                elif op == 2:
                    live.append(pool.seq_fork(int(rng.choice(live))))
                else:
                    s = int(rng.choice(live))
                    pool.seq_free(s)
                    live.remove(s)
            except oracle.OracleError as e:
                assert e.status == "OUT_OF_BLOCKS"
            _check_invariants(pool, live)
        for s in list(live):
            pool.seq_free(s)
        assert np.all(pool.refcounts() == 0)
        assert sorted(pool.free_list().tolist()) == list(range(64))


def test_failed_reservation_changes_nothing():
    pool = oracle.Pool(6, 4, np.arange(6)[::-1].copy())
    a, b = pool.seq_create(), pool.seq_create()
    pool.append([a], [10])  # 3 blocks
    c = pool.seq_fork(a)
    before = (pool.refcounts(), pool.free_list(), pool.table(a), pool.table(c), pool.seq_len(a))
    with pytest.raises(oracle.OracleError) as e:
        # a: CoW + 1 new, b: 2 new, c: in place + 1 new -> 5 > 3 free
        pool.append([a, b, c], [3, 5, 3])
    assert e.value.status == "OUT_OF_BLOCKS"
    after = (pool.refcounts(), pool.free_list(), pool.table(a), pool.table(c), pool.seq_len(a))
    for x, y in zip(before, after):
        assert np.array_equal(x, y)
    assert pool.seq_len(b) == 0


def test_double_free_and_unknown_ids():
    pool = oracle.Pool(8, 4)
    a = pool.seq_create()
    pool.append([a], [5])
    pool.seq_free(a)
    with pytest.raises(oracle.OracleError) as e:
        pool.seq_free(a)
    assert e.value.status == "DOUBLE_FREE"
    with pytest.raises(oracle.OracleError) as e:
        pool.seq_free(99)
    assert e.value.status == "INVALID_ARG"
    with pytest.raises(oracle.OracleError) as e:
        pool.append([a], [1])
    assert e.value.status == "INVALID_ARG"


def test_out_of_blocks_exact_boundary():
    pool = oracle.Pool(4, 16)
    a = pool.seq_create()
    pool.append([a], [64])  # exactly fills the pool
    with pytest.raises(oracle.OracleError) as e:
        pool.append([a], [1])
    assert e.value.status == "OUT_OF_BLOCKS"
    assert pool.seq_len(a) == 64


# ------------------------------------------------------------------ data movement


def test_write_slots_places_each_token_at_block_and_offset():
    g = W.Geometry(L=3, H_q=4, H_kv=2, d_head=8, block_size=4, dtype="bf16", num_blocks=8)
    kp, vp = empty_pools(g)
    k = W.normal(3, "k", (g.L, 5, g.H_kv, g.d_head), "bf16")
    v = W.normal(3, "v", (g.L, 5, g.H_kv, g.d_head), "bf16")
    slots = np.array([0, 7, 13, 30, 21], np.int32)
    oracle.write_slots(g, -1, k, v, slots, kp, vp)
    for i, sl in enumerate(slots):
        p, o = divmod(int(sl), g.block_size)
        for l in range(g.L):
            assert np.array_equal(kp[p, l, :, o, :], k[l, i])
            assert np.array_equal(vp[p, l, :, o, :], v[l, i])
    # nothing else was touched
    mask = np.zeros(g.num_blocks * g.block_size, bool)
    mask[slots] = True
    untouched = kp.transpose(0, 3, 1, 2, 4).reshape(g.num_blocks * g.block_size, -1)[~mask]
    assert np.all(untouched == 0)
    # per-layer form writes only that layer
    kp2, vp2 = empty_pools(g)
    oracle.write_slots(g, 1, k[1], v[1], slots, kp2, vp2)
    assert np.all(kp2[:, [0, 2]] == 0) and np.array_equal(kp2[:, 1], kp[:, 1])


def test_copy_blocks_copies_every_slot_layer_and_tensor():
    g = W.Geometry(L=2, H_q=2, H_kv=2, d_head=8, block_size=4, dtype="f16", num_blocks=6)
    kp = W.normal(5, "k", g.pool_shape(), "f16")
    vp = W.normal(5, "v", g.pool_shape(), "f16")
    k0, v0 = kp.copy(), vp.copy()
    oracle.copy_blocks(g, np.array([[1, 4], [2, 0]]), kp, vp)
    for src, dst in ((1, 4), (2, 0)):
        assert np.array_equal(kp[dst], k0[src]) and np.array_equal(vp[dst], v0[src])
    for p in (1, 2, 3, 5):
        assert np.array_equal(kp[p], k0[p]) and np.array_equal(vp[p], v0[p])


def test_swap_round_trip_is_bit_exact_into_fresh_blocks():
    g = W.Geometry(L=2, H_q=4, H_kv=2, d_head=8, block_size=4, dtype="bf16", num_blocks=12)
    pool = oracle.Pool(g.num_blocks, g.block_size, W.permutation(7, "fo", g.num_blocks))
    kp = W.normal(7, "k", g.pool_shape(), "bf16")
    vp = W.normal(7, "v", g.pool_shape(), "bf16")
    a, b = pool.seq_create(), pool.seq_create()
    pool.append([a, b], [13, 6])  # 4 + 2 blocks
    old = pool.table(a)
    k_old, v_old = kp[old].copy(), vp[old].copy()
    host = np.zeros((8, 2) + g.pool_shape()[1:], np.uint16)
    slots = np.array([5, 0, 7, 2])
    ids = pool.swap_out(a, slots)
    assert np.array_equal(ids, old)
    oracle.swap_out_data(g, ids, slots, kp, vp, host)
    assert list(pool.free_list()[-4:]) == list(old)  # freed frames at the back of the FIFO
    kp[old] = 0
    vp[old] = 0
    new, hs = pool.swap_in(a, 4)
    assert np.array_equal(hs, slots)
    assert not set(new.tolist()) & set(old.tolist())
    oracle.swap_in_data(g, new, hs, host, kp, vp)
    assert np.array_equal(kp[new], k_old) and np.array_equal(vp[new], v_old)
    assert np.array_equal(pool.table(a), new) and pool.seq_len(a) == 13


# ------------------------------------------------------------------ attention


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("B", [1, 2, 4, 16])
def test_attention_matches_library_sdpa(dtype, B):
    """Paged attention equals torch's scaled-dot-product attention (float64) on the
    contiguous keys and values, for GQA groups of 4 and ragged lengths."""
    g = W.Geometry(L=1, H_q=8, H_kv=2, d_head=16, block_size=B, dtype=dtype, num_blocks=96)
    lens = [1, 2, 5, 8, 17, 0, 33][: 7 if B >= 4 else 5]
    fo = W.permutation(21, f"fo{B}", g.num_blocks)
    pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, lens, 21, fo)
    scale = 0.3
    out = oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, scale)
    ref = sdpa_reference(g, q, ks, vs, scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_attention_gpt2_geometry_matches_sdpa():
    wl = W.tiny(n_seq=3)
    g = wl.geometry
    pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, [int(x) for x in wl.lengths], wl.seed,
                                                                 wl.free_order)
    out = oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, wl.scale)
    np.testing.assert_allclose(out, sdpa_reference(g, q, ks, vs, wl.scale), rtol=1e-12, atol=1e-13)


def test_length_one_returns_v0_exactly():
    g = W.Geometry(L=1, H_q=6, H_kv=3, d_head=8, block_size=4, dtype="bf16", num_blocks=8)
    pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, [1, 1], 4)
    out = oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, 1.0)
    for s in range(2):
        for h in range(g.H_q):
            assert np.array_equal(out[s, h], W.to_float64(vs[s][0, h // 2], "bf16"))


def test_equal_keys_give_mean_of_values():
    g = W.Geometry(L=1, H_q=4, H_kv=1, d_head=8, block_size=4, dtype="f32", num_blocks=8)
    pool = oracle.Pool(8, 4)
    s = pool.seq_create()
    slots, _ = pool.append([s], [11])
    kp, vp = empty_pools(g)
    k = np.repeat(W.normal(2, "k", (1, 1, 8), "f32"), 11, axis=0)
    v = W.normal(2, "v", (11, 1, 8), "f32")
    oracle.write_slots(g, 0, k, v, slots, kp, vp)
    q = W.normal(2, "q", (1, 4, 8), "f32")
    tables, lens = pool.tables([s], 3)
    out = oracle.decode_attention(g, 0, q, kp, vp, tables, lens, 0.7)
    np.testing.assert_allclose(out[0], np.repeat(v.astype(np.float64).mean(axis=0), 4, axis=0), rtol=1e-13)


def test_output_invariant_under_physical_permutation():
    """Same logical contents under two different free orders: identical outputs."""
    g = W.Geometry(L=1, H_q=8, H_kv=2, d_head=16, block_size=4, dtype="bf16", num_blocks=40)
    lens = [3, 9, 16, 30]
    outs = []
    for fo in (np.arange(40, dtype=np.int32), W.permutation(8, "p", 40)):
        pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, lens, 8, fo)
        outs.append(oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, 0.25))
    assert np.array_equal(outs[0], outs[1])


def test_paged_equals_one_block_contiguous():
    """Block size 1 with scattered ids equals one block holding the whole sequence."""
    lens = [7, 12]
    res = []
    for B, nb, fo in ((1, 24, W.permutation(9, "p", 24)), (12, 2, None)):
        g = W.Geometry(L=1, H_q=4, H_kv=4, d_head=8, block_size=B, dtype="f32", num_blocks=nb)
        pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, lens, 9, fo)
        res.append(oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, 0.5))
    np.testing.assert_allclose(res[0], res[1], rtol=1e-13, atol=1e-15)


def test_fork_reads_parent_prefix_until_first_write():
    g = W.Geometry(L=1, H_q=4, H_kv=2, d_head=8, block_size=4, dtype="bf16", num_blocks=16)
    pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, [10], 12)
    a = ids[0]
    b = pool.seq_fork(a)
    t2, l2 = pool.tables([a, b], 4)
    q2 = np.concatenate([q, q])
    out = oracle.decode_attention(g, 0, q2, kp, vp, t2, l2, 0.5)
    assert np.array_equal(out[0], out[1])
    # b's first write copies the shared tail block; its first 10 tokens are unchanged
    slots, cows = pool.append([b], [1])
    oracle.copy_blocks(g, cows, kp, vp)
    knew = W.normal(12, "knew", (1, 2, 8), "bf16")
    oracle.write_slots(g, 0, knew, knew, slots, kp, vp)
    tb, lb = pool.tables([b], 4)
    lb_prefix = np.array([10], np.int32)
    out_b = oracle.decode_attention(g, 0, q, kp, vp, tb, lb_prefix, 0.5)
    assert np.array_equal(out_b[0], out[0])
    # and a still sees its own 10 tokens
    ta, la = pool.tables([a], 4)
    assert np.array_equal(oracle.decode_attention(g, 0, q, kp, vp, ta, la, 0.5)[0], out[0])


def test_reused_blocks_do_not_leak_old_values():
    """A block freed by one sequence and reused by another is read only up to the
    new owner's length."""
    g = W.Geometry(L=1, H_q=2, H_kv=1, d_head=8, block_size=8, dtype="f32", num_blocks=2)
    pool = oracle.Pool(2, 8)
    kp, vp = empty_pools(g)
    a = pool.seq_create()
    sa, _ = pool.append([a], [16])
    big = np.full((16, 1, 8), 50.0, np.float32)
    oracle.write_slots(g, 0, big, big, sa, kp, vp)
    pool.seq_free(a)
    b = pool.seq_create()
    sb, _ = pool.append([b], [3])
    k = W.normal(13, "k", (3, 1, 8), "f32")
    v = W.normal(13, "v", (3, 1, 8), "f32")
    oracle.write_slots(g, 0, k, v, sb, kp, vp)
    q = W.normal(13, "q", (1, 2, 8), "f32")
    tb, lb = pool.tables([b], 1)
    out = oracle.decode_attention(g, 0, q, kp, vp, tb, lb, 0.4)
    np.testing.assert_allclose(out, sdpa_reference(g, q, [k], [v], 0.4), rtol=1e-12)


def test_empty_sequence_gives_zero_and_bad_ids_are_rejected():
    g = W.Geometry(L=1, H_q=2, H_kv=1, d_head=8, block_size=4, dtype="f32", num_blocks=4)
    kp, vp = empty_pools(g)
    q = np.ones((1, 2, 8), np.float32)
    out = oracle.decode_attention(g, 0, q, kp, vp, np.zeros((1, 1), np.int32), np.zeros(1, np.int32), 1.0)
    assert np.all(out == 0)
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode_attention(g, 0, q, kp, vp, np.full((1, 1), 9, np.int32), np.ones(1, np.int32), 1.0)
    assert e.value.status == "BAD_BLOCK_ID"
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode_attention(g, 0, q, kp, vp, np.zeros((1, 1), np.int32), np.full(1, 5, np.int32), 1.0)
    assert e.value.status == "INVALID_ARG"


def test_threads_do_not_change_the_result():
    g = W.Geometry(L=1, H_q=8, H_kv=2, d_head=16, block_size=4, dtype="bf16", num_blocks=64)
    pool, ids, kp, vp, ks, vs, q, tables, seq_lens = build_case(g, [5, 40, 23, 64], 30)
    a = oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, 0.2, n_threads=1)
    b = oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, 0.2, n_threads=7)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ chunked prefill


def _sdpa_causal(g, q_rows, k, v, scale):
    """torch SDPA, float64, causal over a whole sequence (the monolithic forward pass)."""
    G = g.H_q // g.H_kv
    qt = torch.from_numpy(W.to_float64(q_rows, g.dtype)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(W.to_float64(k, g.dtype)).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(W.to_float64(v, g.dtype)).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("dtype,B", [("bf16", 16), ("f32", 4), ("f16", 1)])
def test_chunked_prefill_equals_monolithic_causal_attention(dtype, B):
    """"Chunked prefill mechanics": chunk k's queries attend to the cached history in
    full and causally within the chunk, which must equal one causal pass over the
    whole prompt.  Three sequences, each split into ragged chunks; every chunk of
    every sequence is computed in one oracle call per round."""
    g = W.Geometry(L=1, H_q=8, H_kv=2, d_head=16, block_size=B, dtype=dtype, num_blocks=200)
    lens = [37, 70, 5]
    cuts = [[0, 10, 11, 37], [0, 64, 70], [0, 5]]
    pool, ids, kp, vp, ks, vs, _, _, _ = build_case(g, lens, 71, W.permutation(71, "fo", g.num_blocks))
    qs = [W.normal(71, f"qp{i}", (n, g.H_q, g.d_head), dtype) for i, n in enumerate(lens)]
    scale = 0.25
    Wd = max(-(-n // B) for n in lens)
    tables, _ = pool.tables(ids, Wd)
    got = [np.zeros((n, g.H_q, g.d_head)) for n in lens]
    for rnd in range(max(len(c) - 1 for c in cuts)):
        rows, offs, cur = [], [0], []
        for i, c in enumerate(cuts):
            if rnd + 1 < len(c):
                a, b = c[rnd], c[rnd + 1]
                rows.append(qs[i][a:b])
                cur.append(b)
            else:
                cur.append(lens[i])  # empty chunk
            offs.append(offs[-1] + (len(rows[-1]) if rnd + 1 < len(c) else 0))
        q = np.concatenate(rows)
        out = oracle.prefill_attention(g, 0, q, np.array(offs), kp, vp, tables, np.array(cur, np.int32), scale)
        for i, c in enumerate(cuts):
            if rnd + 1 < len(c):
                got[i][c[rnd]:c[rnd + 1]] = out[offs[i]:offs[i + 1]]
    for i in range(len(lens)):
        ref = _sdpa_causal(g, qs[i], ks[i], vs[i], scale)
        np.testing.assert_allclose(got[i], ref, rtol=1e-12, atol=1e-13)


def test_prefill_last_query_is_the_decode_query_and_bad_chunks_are_rejected():
    g = W.Geometry(L=1, H_q=4, H_kv=1, d_head=8, block_size=4, dtype="f32", num_blocks=16)
    pool, ids, kp, vp, ks, vs, q, tables, lens = build_case(g, [13], 72)
    qrow = W.normal(72, "qq", (3, 4, 8), "f32")
    out = oracle.prefill_attention(g, 0, qrow, np.array([0, 3]), kp, vp, tables, lens, 0.5)
    # the chunk's last query sees every token: an ordinary decode query
    dec = oracle.decode_attention(g, 0, qrow[2:3], kp, vp, tables, lens, 0.5)
    np.testing.assert_allclose(out[2], dec[0], rtol=1e-13)
    # its first query sees all but the last two tokens
    dec2 = oracle.decode_attention(g, 0, qrow[0:1], kp, vp, tables, lens - 2, 0.5)
    np.testing.assert_allclose(out[0], dec2[0], rtol=1e-13)
    with pytest.raises(oracle.OracleError) as e:
        oracle.prefill_attention(g, 0, np.zeros((20, 4, 8), np.float32), np.array([0, 20]), kp, vp, tables, lens,
                                 0.5)
    assert e.value.status == "INVALID_ARG"


# ------------------------------------------------------------------ FP8 (E4M3) storage
#
# "KV Cache Management" (cs249r vol. 3 ch. 5), "The PagedAttention virtual memory
# model": M_block = 2 L H_kv B d_head b_elem with b_elem = 1 byte for FP8.  The
# format is OCP E4M3; torch's float8_e4m3fn is an independent implementation of it.


def _torch_e4m3_values(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e4m3_codes(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_values_match_torch_and_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = _torch_e4m3_values(codes)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert set(np.flatnonzero(np.isnan(mine)).tolist()) == {0x7F, 0xFF}
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok]) and np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))
    # closed forms of the format: bias 7, 3 fraction bits, largest finite 1.75 * 2^8
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x38] == 1.0 and mine[0xC0] == -2.0
    assert mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9 and mine[0x07] == 7 * 2.0 ** -9
    assert mine[0x00] == 0.0 and np.signbit(mine[0x80])


def test_e4m3_encode_round_trip_ties_to_even_and_saturation():
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(finite).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), finite)  # every value maps to its own code (-0 too)
    pos = np.arange(0, 0x7F, dtype=np.uint8)  # 0 .. 448 in increasing order
    pv = oracle.e4m3_decode(pos)
    assert np.all(np.diff(pv) > 0)
    mid = ((pv[:-1] + pv[1:]) / 2).astype(np.float32)  # exact: five significant bits
    assert np.array_equal(mid.astype(np.float64), (pv[:-1] + pv[1:]) / 2)
    even = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(oracle.e4m3_encode(mid), even)
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mid, np.float32(np.inf))), pos[1:])
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mid, np.float32(0))), pos[:-1])
    assert np.array_equal(oracle.e4m3_encode(-mid), even | 0x80)
    big = np.array([448, 460, 464, 1e4, 3e38, -500, -3e38], np.float32)
    assert oracle.e4m3_encode(big).tolist() == [0x7E] * 5 + [0xFE] * 2
    tiny = np.array([2.0 ** -10, 2.0 ** -10 * 1.001, -(2.0 ** -11), 2.0 ** -9 * 1.5], np.float32)
    assert oracle.e4m3_encode(tiny).tolist() == [0x00, 0x01, 0x80, 0x02]
    # against torch's conversion (round to nearest even) inside the finite range
    x = np.concatenate([W.substream(31, f"e4m3_{s}").standard_normal(20000).astype(np.float32) * s
                        for s in (1e-3, 0.05, 1.0, 30.0, 140.0)])
    x = x[np.abs(x) < 448]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3_codes(x))


def _fp8_case(g, lens, seed, k_scale, v_scale, free_order=None):
    """Sequences written into an FP8 pool through the oracle's quantised write; K/V
    drawn in bf16.  Returns the codes' values dequantised by torch."""
    pool = oracle.Pool(g.num_blocks, g.block_size, free_order)
    kp = np.zeros(g.pool_shape(), np.uint8)
    vp = np.zeros(g.pool_shape(), np.uint8)
    ids = [pool.seq_create() for _ in lens]
    kd, vd = [], []
    for i, (sid, n) in enumerate(zip(ids, lens)):
        k = W.normal(seed, f"k{i}", (n, g.H_kv, g.d_head), "bf16")
        v = W.normal(seed, f"v{i}", (n, g.H_kv, g.d_head), "bf16")
        if n:
            slots, _ = pool.append([sid], [n])
            oracle.write_slots(g, 0, k, v, slots, kp, vp, k_scale, v_scale)
            # the stored codes, read back through the table by plain indexing
            blk = np.array([pool.table(sid)[t // g.block_size] for t in range(n)])
            off = np.arange(n) % g.block_size
            kd.append(_torch_e4m3_values(kp[blk, 0, :, off, :]) * k_scale)
            vd.append(_torch_e4m3_values(vp[blk, 0, :, off, :]) * v_scale)
        else:
            kd.append(np.zeros((0, g.H_kv, g.d_head)))
            vd.append(np.zeros((0, g.H_kv, g.d_head)))
    Wt = max([-(-n // g.block_size) for n in lens] + [1])
    tables, seq_lens = pool.tables(ids, Wt)
    return pool, ids, kp, vp, kd, vd, tables, seq_lens


def test_quantised_write_stores_the_code_of_the_binary32_quotient():
    g = W.Geometry(L=2, H_q=4, H_kv=2, d_head=16, block_size=4, dtype="e4m3", num_blocks=8)
    k = W.normal(41, "k", (g.L, 6, g.H_kv, g.d_head), "bf16")
    v = W.normal(41, "v", (g.L, 6, g.H_kv, g.d_head), "bf16")
    v[0, 0, 0, :4] = W.f32_to_bf16_bits(np.array([900.0, -5000.0, 1e-4, -1e-4], np.float32))  # saturate / flush
    slots = np.array([0, 5, 6, 13, 31, 20], np.int32)
    for ks, vs in ((1.0, 1.0), (0.0173, 0.5), (3.0, 0.011)):
        kp = np.zeros(g.pool_shape(), np.uint8)
        vp = np.zeros(g.pool_shape(), np.uint8)
        oracle.write_slots(g, -1, k, v, slots, kp, vp, ks, vs)
        kq = W.bf16_bits_to_f32(k) / np.float32(ks)
        vq = W.bf16_bits_to_f32(v) / np.float32(vs)
        vq_codes = _torch_e4m3_codes(np.clip(vq, -448, 448))
        for i, sl in enumerate(slots):
            p, o = divmod(int(sl), g.block_size)
            for l in range(g.L):
                assert np.array_equal(kp[p, l, :, o, :], _torch_e4m3_codes(kq[l, i]))
                assert np.array_equal(vp[p, l, :, o, :], vq_codes[l, i])
        mask = np.zeros(g.num_blocks * g.block_size, bool)
        mask[slots] = True
        assert np.all(kp.transpose(0, 3, 1, 2, 4).reshape(g.num_blocks * g.block_size, -1)[~mask] == 0)
    # the page's byte count with b_elem = 1: one block of K plus V
    assert 2 * kp[0].nbytes == 2 * g.L * g.H_kv * g.block_size * g.d_head * 1


@pytest.mark.parametrize("B", [1, 4, 16])
def test_fp8_attention_matches_sdpa_on_dequantised_keys_and_values(B):
    """Attention over an FP8 pool equals torch's SDPA (float64) over the stored codes'
    values times the pool scales, with bf16 queries."""
    g = W.Geometry(L=1, H_q=8, H_kv=2, d_head=16, block_size=B, dtype="e4m3", num_blocks=96)
    lens = [1, 2, 5, 8, 17, 0, 33][: 7 if B >= 4 else 5]
    k_scale, v_scale = 0.0173, 0.25
    pool, ids, kp, vp, kd, vd, tables, seq_lens = _fp8_case(g, lens, 43, k_scale, v_scale,
                                                            W.permutation(43, f"fo{B}", g.num_blocks))
    q = W.normal(43, "q", (len(lens), g.H_q, g.d_head), "bf16")
    out = oracle.decode_attention(g, 0, q, kp, vp, tables, seq_lens, 0.3, k_scale=k_scale, v_scale=v_scale)
    G = g.H_q // g.H_kv
    for s in range(len(lens)):
        if lens[s] == 0:
            assert np.all(out[s] == 0)
            continue
        qt = torch.from_numpy(W.to_float64(q[s], "bf16")).view(1, g.H_q, 1, g.d_head)
        kt = torch.from_numpy(kd[s]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        vt = torch.from_numpy(vd[s]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.3)[0, :, 0, :].numpy()
        np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-13)
    # chunked prefill over the same pool: the last 5 tokens of sequence 4 as a chunk
    s = 4
    qs = W.normal(43, "qc", (5, g.H_q, g.d_head), "bf16")
    got = oracle.prefill_attention(g, 0, qs, np.array([0, 5], np.int32), kp, vp, tables[s:s + 1],
                                   seq_lens[s:s + 1], 0.3, k_scale=k_scale, v_scale=v_scale)
    P = lens[s] - 5
    for i in range(5):
        qt = torch.from_numpy(W.to_float64(qs[i], "bf16")).view(1, g.H_q, 1, g.d_head)
        kt = torch.from_numpy(kd[s][: P + i + 1]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        vt = torch.from_numpy(vd[s][: P + i + 1]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.3)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[i], ref, rtol=1e-12, atol=1e-13)
