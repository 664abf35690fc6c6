"""The library's host control plane against the oracle allocator (no GPU).

Block ids, slots, copy-on-write pairs, tables, reference counts, the FIFO and the
error statuses must agree exactly after every operation.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W

STATUS = {"PKV_ERR_INVALID_ARG": "INVALID_ARG", "PKV_ERR_OUT_OF_BLOCKS": "OUT_OF_BLOCKS",
          "PKV_ERR_DOUBLE_FREE": "DOUBLE_FREE", "PKV_ERR_BAD_BLOCK_ID": "BAD_BLOCK_ID"}


def both(f_lib, f_orc):
    """Run one operation on both sides; statuses and results must agree."""
    try:
        r1, e1 = f_lib(), None
    except pkv.PkvError as e:
        r1, e1 = None, STATUS[e.name]
    try:
        r2, e2 = f_orc(), None
    except oracle.OracleError as e:
        r2, e2 = None, e.status
    assert e1 == e2
    return r1, r2


def same_state(lib, orc, live):
    assert np.array_equal(pkv.pkv_refcounts(lib), orc.refcounts())
    assert np.array_equal(pkv.pkv_free_list(lib), orc.free_list())
    if live:
        Wd = max(len(orc.table(s)) for s in live) + 1
        t1, l1 = pkv.pkv_export_tables(lib, live, Wd)
        t2, l2 = orc.tables(live, Wd)
        assert np.array_equal(t1, t2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("B,N,seed", [(1, 48, 1), (4, 64, 2), (16, 96, 3), (16, 32, 4)])
def test_random_operation_sequences_agree(B, N, seed):
    fo = W.permutation(seed, "fo", N)
    lib = pkv.pkv_pool_create(1, 4, 2, 8, B, "bf16", N, fo)
    orc = oracle.Pool(N, B, fo)
    rng = W.substream(seed, "ops")
    live, dead = [], []
    for step in range(600):
        op = int(rng.integers(0, 6))
        if op == 0 or not live:
            a, b = both(lambda: pkv.pkv_seq_create(lib), lambda: orc.seq_create())
            assert a == b
            live.append(a)
        elif op in (1, 2):
            k = int(rng.integers(1, min(len(live), 5) + 1))
            sel = [int(x) for x in rng.choice(live, size=k, replace=False)]
            nn = [int(x) for x in rng.integers(0, 3 * B + 1, size=k)]
            r1, r2 = both(lambda: pkv.pkv_plan_append(lib, sel, nn), lambda: orc.append(sel, nn))
            if r1 is not None:
                assert np.array_equal(r1[0], r2[0]) and np.array_equal(r1[1], r2[1])
        elif op == 3:
            p = int(rng.choice(live))
            a, b = both(lambda: pkv.pkv_seq_fork(lib, p), lambda: orc.seq_fork(p))
            assert a == b
            live.append(a)
        elif op == 4:
            s = int(rng.choice(live))
            both(lambda: pkv.pkv_seq_free(lib, s), lambda: orc.seq_free(s))
            live.remove(s)
            dead.append(s)
        else:
            # error paths: double free, unknown id, append to a freed sequence
            s = int(rng.choice(dead)) if dead else 10_000
            both(lambda: pkv.pkv_seq_free(lib, s), lambda: orc.seq_free(s))
            both(lambda: pkv.pkv_plan_append(lib, [s], [1]), lambda: orc.append([s], [1]))
        same_state(lib, orc, live)
    for s in list(live):
        both(lambda: pkv.pkv_seq_free(lib, s), lambda: orc.seq_free(s))
    assert np.all(pkv.pkv_refcounts(lib) == 0)
    assert sorted(pkv.pkv_free_list(lib).tolist()) == list(range(N))


def test_workload_shapes_agree():
    """Chat-like prompts, a forked prefix and long contexts plan identically."""
    wl = W.chat(n_seq=64, num_blocks=4096)
    g = wl.geometry
    lib = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, wl.free_order)
    orc = oracle.Pool(g.num_blocks, g.block_size, wl.free_order)
    ids = [pkv.pkv_seq_create(lib) for _ in range(64)]
    assert ids == [orc.seq_create() for _ in range(64)]
    r1 = pkv.pkv_plan_append(lib, ids, wl.lengths)
    r2 = orc.append(ids, wl.lengths)
    assert np.array_equal(r1[0], r2[0])
    for step in range(8):
        r1 = pkv.pkv_plan_append(lib, ids[::-1], [1] * 64)
        r2 = orc.append(ids[::-1], [1] * 64)
        assert np.array_equal(r1[0], r2[0]) and len(r1[1]) == 0
    same_state(lib, orc, ids)


def test_forked_prefix_copy_on_write_matches():
    fx = W.forked(n_branch=8, prefix=200, max_suffix=40, num_blocks=256)
    g = fx.geometry
    lib = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, fx.free_order)
    orc = oracle.Pool(g.num_blocks, g.block_size, fx.free_order)
    p = pkv.pkv_seq_create(lib)
    orc.seq_create()
    pkv.pkv_plan_append(lib, [p], [200])
    orc.append([p], [200])
    kids = [pkv.pkv_seq_fork(lib, p) for _ in range(8)]
    assert kids == [orc.seq_fork(p) for _ in range(8)]
    assert set(pkv.pkv_refcounts(lib)[pkv.pkv_export_tables(lib, [p], 13)[0][0]].tolist()) == {9}
    suf = [int(x) for x in fx.extra["suffix"]]
    r1 = pkv.pkv_plan_append(lib, kids, suf)
    r2 = orc.append(kids, suf)
    assert np.array_equal(r1[0], r2[0]) and np.array_equal(r1[1], r2[1])
    # every branch with a non-empty suffix copied the shared tail block
    assert len(r1[1]) == sum(1 for s in suf if s > 0)
    same_state(lib, orc, [p] + kids)


def test_out_of_blocks_leaves_state_unchanged():
    lib = pkv.pkv_pool_create(1, 2, 2, 8, 4, "f16", 6)
    a = pkv.pkv_seq_create(lib)
    b = pkv.pkv_seq_create(lib)
    pkv.pkv_plan_append(lib, [a], [10])
    c = pkv.pkv_seq_fork(lib, a)
    before = (pkv.pkv_refcounts(lib).copy(), pkv.pkv_free_list(lib).copy(), pkv.pkv_export_tables(lib, [a, c], 4))
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_plan_append(lib, [a, b, c], [3, 5, 3])
    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
    after = (pkv.pkv_refcounts(lib), pkv.pkv_free_list(lib), pkv.pkv_export_tables(lib, [a, c], 4))
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    assert np.array_equal(before[2][0], after[2][0]) and np.array_equal(before[2][1], after[2][1])


def test_invalid_arguments_are_rejected_without_change():
    lib = pkv.pkv_pool_create(1, 2, 2, 8, 4, "f32", 8)
    a = pkv.pkv_seq_create(lib)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_plan_append(lib, [a, a], [1, 1])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_plan_append(lib, [a], [-1])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    pkv.pkv_plan_append(lib, [a], [9])
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_export_tables(lib, [a], 2)  # needs 3 entries
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    # swap-in of a resident sequence (raw C call: no device buffers are needed to reject it)
    host = np.zeros(8, np.uint8)
    rc = pkv._L().pkv_swap_in(lib.handle, a, host.ctypes.data, 1, 0, None, None, None, None)
    assert pkv._L().pkv_status_name(rc).decode() == "PKV_ERR_INVALID_ARG"
    assert pkv.pkv_seq_len(lib, a) == 9


def test_fp8_pool_scales_and_geometry_checks():
    p = pkv.pkv_pool_create(2, 8, 2, 128, 16, "e4m3", 64)
    assert pkv.pkv_pool_geometry(p).dtype == pkv.E4M3
    assert pkv.pkv_pool_kv_scales(p) == (1.0, 1.0)
    pkv.pkv_pool_set_kv_scales(p, 0.25, 0.5)
    assert pkv.pkv_pool_kv_scales(p) == (0.25, 0.5)
    for bad in [(0.0, 1.0), (1.0, -2.0), (float("inf"), 1.0), (1.0, float("nan"))]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_pool_set_kv_scales(p, *bad)
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert pkv.pkv_pool_kv_scales(p) == (0.25, 0.5)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_set_kv_scales(pkv.pkv_pool_create(1, 2, 2, 8, 4, "bf16", 4), 0.5, 0.5)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(1, 2, 2, 12, 4, "e4m3", 4)  # d_head not a multiple of 8
    assert e.value.name == "PKV_ERR_UNSUPPORTED"


def test_step_plan_matches_the_oracle_and_rejects_without_change():
    """pkv_step_plan (the host half of a decode step): one token per sequence, slot mapping,
    tables and lengths in the metadata buffer and the copy-on-write pairs, as the oracle plans
    them; a sequence whose table would overflow W is rejected with nothing changed."""
    import torch

    g = W.Geometry(L=2, H_q=8, H_kv=2, d_head=64, block_size=16, dtype="bf16", num_blocks=96)
    fo = W.permutation(91, "fo", g.num_blocks)
    lib = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, fo)
    orc = oracle.Pool(g.num_blocks, g.block_size, fo)
    ids = [pkv.pkv_seq_create(lib) for _ in range(4)]
    assert ids == [orc.seq_create() for _ in range(4)]
    pkv.pkv_plan_append(lib, ids, [15, 16, 40, 0])
    orc.append(ids, [15, 16, 40, 0])
    kids = [pkv.pkv_seq_fork(lib, ids[2]), pkv.pkv_seq_fork(lib, ids[0])]
    assert kids == [orc.seq_fork(ids[2]), orc.seq_fork(ids[0])]
    run = ids + kids
    n, Wd = len(run), 8
    meta = torch.zeros(n * (Wd + 2), dtype=torch.int32)
    for step in range(20):
        cows = pkv.pkv_step_plan(lib, run, Wd, meta)
        oslots, ocows = orc.append(run, [1] * n)
        t2, l2 = orc.tables(run, Wd)
        m = meta.numpy()
        assert np.array_equal(m[:n], oslots) and np.array_equal(cows, ocows)
        assert np.array_equal(m[n:n + n * Wd].reshape(n, Wd), t2) and np.array_equal(m[n + n * Wd:n + n * Wd + n], l2)
    same_state(lib, orc, run)
    before = (pkv.pkv_refcounts(lib).copy(), pkv.pkv_free_list(lib).copy())
    with pytest.raises(pkv.PkvError) as e:  # 40 + 20 tokens fit 4 blocks: W = 3 cannot hold the next one
        pkv.pkv_step_plan(lib, run, 3, meta)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    assert np.array_equal(before[0], pkv.pkv_refcounts(lib)) and np.array_equal(before[1], pkv.pkv_free_list(lib))
