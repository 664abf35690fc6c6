"""The shared-prefix plan that a decode step writes after its metadata (host logic, no GPU).

A run of consecutive batch rows whose tables begin with the same physical blocks (branches
forked from one parent: "KV Cache Management", "Zero-copy deliberation via copy-on-write
branching") is planned as one group; the checks here are what makes the device side correct:
every member's first kb table entries are the first member's, every member keeps at least one
token of its own after them, the work items cut [0, kb) into disjoint whole-block ranges, and
every (member, item) partial has its own slot within the workspace's capacity.
"""
import numpy as np
import pytest

import paged_kv_cache_80_gb300 as pkv


def _pool(dtype="bf16", H_q=64, H_kv=8, d_head=128, B=16, N=4096):
    return pkv.pkv_pool_create(1, H_q, H_kv, d_head, B, dtype, N)


def _parse(meta, n, W, sharing=True):
    """Split step metadata into (slots, tables, lens, header, rows, items)."""
    slots = meta[:n]
    tables = meta[n:n + n * W].reshape(n, W)
    lens = meta[n + n * W:n + n * W + n]
    if not sharing:
        return slots, tables, lens, None, None, None
    off = (n * (W + 2) + 3) // 4 * 4
    hdr = meta[off:off + 4]
    rows = meta[off + 4:off + 4 + 4 * n].reshape(n, 4)
    items = meta[off + 4 + 4 * n:].reshape(-1, 8)[:hdr[0]]
    return slots, tables, lens, hdr, rows, items


def _check_plan(n, B, tables, lens, hdr, rows, items, slot_cap, full=None):
    """Everything the device side relies on, from the plan alone.  `tables` are the step
    metadata's tables (a run's shared entries are written only in its first row); `full` are
    the pool's own tables of the same rows (pkv_export_tables), when given."""
    n_items, max_members, n_slots = int(hdr[0]), int(hdr[1]), int(hdr[2])
    assert len(items) == n_items
    used = np.zeros(n_slots, np.int32)
    groups = {}
    for it in items:
        rb, re, kb0, kb1, base = (int(x) for x in it[:5])
        assert 0 <= rb < re <= n and 0 <= kb0 < kb1 and base >= 0 and base + (re - rb) <= n_slots
        assert not it[5:].any()
        used[base:base + (re - rb)] += 1
        groups.setdefault((rb, re), []).append((kb0, kb1, base))
    assert np.all(used == 1), "every (member, item) partial has a slot of its own"
    assert n_slots <= slot_cap
    in_group = np.zeros(n, bool)
    for (rb, re), its in groups.items():
        its.sort()
        kb = int(rows[rb, 0])
        # the items cut [0, kb) into consecutive whole-block ranges, in slot order
        assert its[0][0] == 0 and its[-1][1] == kb
        assert all(its[i][1] == its[i + 1][0] for i in range(len(its) - 1))
        assert all(its[i][2] == its[0][2] + i * (re - rb) for i in range(len(its)))
        assert re - rb <= max_members
        for r in range(rb, re):
            assert not in_group[r]
            in_group[r] = True
            assert tuple(rows[r]) == (kb, len(its), its[0][2] + (r - rb), re - rb)
            assert kb * B < lens[r], "each member keeps a token of its own after the shared blocks"
            if full is not None:
                nb = -(-int(lens[r]) // B)
                assert np.array_equal(full[r, :kb], full[rb, :kb]), "the shared blocks are the first member's"
                assert np.array_equal(tables[r, kb:nb], full[r, kb:nb]), "the row's own entries are written"
                if r == rb:
                    assert np.array_equal(tables[r, :nb], full[r, :nb]), "the first row's table is whole"
    assert not rows[~in_group].any(), "rows outside groups have no prefix"
    return groups


def _full(pool, ids, W):
    return pkv.pkv_export_tables(pool, ids, W)[0]


def _forked_batch(pool, prefix, n_kids, suffixes):
    parent = pkv.pkv_seq_create(pool)
    pkv.pkv_plan_append(pool, [parent], [prefix])
    kids = [pkv.pkv_seq_fork(pool, parent) for _ in range(n_kids)]
    if any(suffixes):
        pkv.pkv_plan_append(pool, kids, suffixes)
    return parent, kids


def test_sharing_off_keeps_the_plain_metadata():
    pool = _pool()
    assert pkv.pkv_step_meta_ints(pool, 7, 10) == 7 * 12
    pkv.pkv_pool_set_prefix_sharing(pool, 4, 1, 152)
    assert pkv.pkv_step_meta_ints(pool, 7, 10) == (7 * 12 + 3) // 4 * 4 + 4 + 4 * 7 + 8 * (7 + 256)
    pkv.pkv_pool_set_prefix_sharing(pool, 0, 1, 152)
    assert pkv.pkv_step_meta_ints(pool, 7, 10) == 7 * 12


def test_two_groups_among_unrelated_rows():
    """[u0, 40 branches of P, u1, 10 branches of Q, u2]: two groups, the unrelated rows alone."""
    pool = _pool()
    pkv.pkv_pool_set_prefix_sharing(pool, 4, 1, 152)
    u = [pkv.pkv_seq_create(pool) for _ in range(3)]
    pkv.pkv_plan_append(pool, u, [500, 37, 2000])
    rng = np.random.default_rng(5)
    _, kp = _forked_batch(pool, 1000, 40, [int(x) for x in rng.integers(0, 300, 40)])
    _, kq = _forked_batch(pool, 4104, 10, [0] * 10)  # 256 full blocks + 8: every branch's step copies the tail
    ids = [u[0]] + kp + [u[1]] + kq + [u[2]]
    n, W = len(ids), 300
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    cows = pkv.pkv_step_plan(pool, ids, W, meta)
    assert len(cows) == 10 + sum(1 for k in range(40) if pkv.pkv_seq_len(pool, kp[k]) - 1 == 1000 and 1000 % 16)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    groups = _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, ids, W))
    assert set(groups) == {(1, 41), (42, 52)}
    assert rows[1, 0] == 1000 // 16  # 62 full blocks of P's prefix
    assert rows[42, 0] == 4104 // 16  # 256 full blocks of Q's (the tail block went to copies)
    # the prefix grid: (members / 32 rounded up) x 8 KV heads per split; with the decode beside it
    # on hdr[3] SMs (one CTA each) the two fit the 152 target together, else the grid alone comes
    # near it
    ctas = sum(((re - rb + 31) // 32) * 8 * len(v) for (rb, re), v in groups.items())
    if hdr[3]:
        assert 8 <= hdr[3] and ctas + hdr[3] <= 152
    else:
        assert 100 <= ctas <= 152


def test_small_runs_are_not_grouped_and_min_blocks_holds():
    pool = _pool()
    pkv.pkv_pool_set_prefix_sharing(pool, 4, 8, 152)
    _, k3 = _forked_batch(pool, 800, 3, [5, 5, 5])       # 3 branches: fewer than min_members
    _, k5 = _forked_batch(pool, 100, 5, [1, 2, 3, 4, 5])  # 6 shared blocks: fewer than min_blocks
    _, k6 = _forked_batch(pool, 130, 6, [20] * 6)         # 8 full blocks shared: a group
    ids = k3 + k5 + k6
    n, W = len(ids), 64
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    pkv.pkv_step_plan(pool, ids, W, meta)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    groups = _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, ids, W))
    assert set(groups) == {(8, 14)}
    assert rows[8, 0] == 8


def test_prefix_stops_before_each_rows_last_token():
    """Branches of a 64-token (4-block) prefix with no suffix: after the step each has 65
    tokens, so all 4 blocks are shared; branches of a 63-token prefix: 3 full blocks."""
    pool = _pool()
    pkv.pkv_pool_set_prefix_sharing(pool, 2, 1, 152)
    _, ka = _forked_batch(pool, 64, 4, [0] * 4)
    _, kb = _forked_batch(pool, 63, 4, [0] * 4)
    ids = ka + kb
    n, W = len(ids), 8
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    pkv.pkv_step_plan(pool, ids, W, meta)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, ids, W))
    assert list(rows[:4, 0]) == [4] * 4 and list(rows[4:, 0]) == [3] * 4


def test_caps_hold_with_a_huge_grid_target():
    """A target far beyond the SM count: splits stop at 256 keys and within the slot cap."""
    pool = _pool(N=16384)
    pkv.pkv_pool_set_prefix_sharing(pool, 2, 1, 1 << 20)
    batches = [_forked_batch(pool, 2000 + 37 * i, 3, [i, 0, 2 * i])[1] for i in range(20)]
    ids = [s for b in batches for s in b]
    n, W = len(ids), 200
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    pkv.pkv_step_plan(pool, ids, W, meta)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    groups = _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, ids, W))
    assert len(groups) == 20
    assert hdr[2] <= 2 * n + 1024 and hdr[0] <= n + 256
    for its in groups.values():
        assert all((k1 - k0) * 16 >= 256 or len(its) == 1 for k0, k1, _ in its[:-1])


def test_sixteen_head_groups_take_sixteen_members_per_cta():
    pool = _pool(H_q=128)
    pkv.pkv_pool_set_prefix_sharing(pool, 4, 1, 152)
    _, kids = _forked_batch(pool, 3000, 40, [3] * 40)
    n, W = len(kids), 200
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    pkv.pkv_step_plan(pool, kids, W, meta)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    groups = _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, kids, W))
    ((rb, re), its), = groups.items()
    assert (rb, re) == (0, 40)
    assert len(its) == 152 // (3 * 8)  # 40 members: 3 CTAs of 16 per KV head and split
    assert hdr[3] == 0  # groups of 16 heads: the decode runs on every SM, then the prefix kernel


def test_side_by_side_split_for_the_forked_shape():
    """64 branches over a 1,023-block prefix with suffixes of ~1,000 tokens: the decode of the
    branches' own blocks goes beside the prefix kernel (header word 3 = its SMs), and the two
    grids together fit the SM count."""
    pool = _pool(N=16384)
    pkv.pkv_pool_set_prefix_sharing(pool, 8, 1, 152)
    rng = np.random.default_rng(9)
    _, kids = _forked_batch(pool, 16376, 64, [int(x) for x in rng.integers(0, 2048, 64)])
    n, W = len(kids), 1200
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    pkv.pkv_step_plan(pool, kids, W, meta)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    groups = _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, kids, W))
    ((rb, re), its), = groups.items()
    assert (rb, re) == (0, 64) and rows[0, 0] == 1023
    ctas = 2 * 8 * len(its)
    assert 16 <= hdr[3] <= 152 - ctas


def test_fp8_pools_keep_the_decode_on_every_sm():
    pool = _pool(dtype="e4m3", N=16384)
    pkv.pkv_pool_set_prefix_sharing(pool, 8, 1, 152)
    _, kids = _forked_batch(pool, 16376, 64, [1000] * 64)
    n, W = len(kids), 1200
    meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
    pkv.pkv_step_plan(pool, kids, W, meta)
    _, tables, lens, hdr, rows, items = _parse(meta, n, W)
    _check_plan(n, 16, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, kids, W))
    assert hdr[3] == 0 and hdr[0] == 152 // 16


def test_option_validation():
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_set_prefix_sharing(_pool(), 1, 1, 152)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_set_prefix_sharing(_pool(), 4, 0, 152)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    for kw in ({"dtype": "f32"}, {"d_head": 64}, {"H_q": 136, "H_kv": 8}, {"B": 8}):
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_pool_set_prefix_sharing(_pool(**kw), 4, 1, 152)
        assert e.value.name == "PKV_ERR_UNSUPPORTED", kw


@pytest.mark.parametrize("seed", range(12))
def test_random_fork_trees_and_batch_orders(seed):
    """Seeded random pools: parents of random lengths, branches forked at random depths (some
    from branches), random suffixes, unrelated sequences, a random batch order and random
    option values; every plan must satisfy the invariants the kernels rely on."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.choice([16, 32]))
    H_q = int(rng.choice([64, 128]))
    pool = _pool(H_q=H_q, B=B, N=8192)
    pkv.pkv_pool_set_prefix_sharing(pool, int(rng.integers(2, 6)), int(rng.integers(1, 4)),
                                    int(rng.choice([64, 152, 300])))
    seqs = []
    for _ in range(int(rng.integers(1, 4))):  # fork trees
        root = pkv.pkv_seq_create(pool)
        pkv.pkv_plan_append(pool, [root], [int(rng.integers(1, 600))])
        nodes = [root]
        for _ in range(int(rng.integers(2, 20))):
            parent = nodes[int(rng.integers(0, len(nodes)))]
            kid = pkv.pkv_seq_fork(pool, parent)
            grow = int(rng.integers(0, 120))
            if grow:
                pkv.pkv_plan_append(pool, [kid], [grow])
            nodes.append(kid)
        seqs += nodes
    for _ in range(int(rng.integers(0, 6))):  # unrelated sequences
        s = pkv.pkv_seq_create(pool)
        pkv.pkv_plan_append(pool, [s], [int(rng.integers(0, 300))])
        seqs.append(s)
    ids = np.array(seqs, np.int32)
    if rng.random() < 0.5:
        ids = ids[rng.permutation(len(ids))]
    else:
        ids = np.sort(ids)  # branches of one tree next to each other
    n = len(ids)
    W = max(pkv.pkv_seq_len(pool, int(s)) for s in ids) // B + 2
    for step in range(2):
        meta = np.zeros(pkv.pkv_step_meta_ints(pool, n, W), np.int32)
        pkv.pkv_step_plan(pool, ids, W, meta)
        _, tables, lens, hdr, rows, items = _parse(meta, n, W)
        _check_plan(n, B, tables, lens, hdr, rows, items, 2 * n + 1024, _full(pool, ids, W))
        assert 0 <= hdr[3] <= 300
