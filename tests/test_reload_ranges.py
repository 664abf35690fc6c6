"""The reload-by-layer-ranges state machine (pkv_swap_in_layers) on the CPU: a swapped-out
sequence with no blocks needs no device memory, so the ordering rules and the residency
transitions are checked through the raw C calls without a GPU."""
import ctypes

import numpy as np

import paged_kv_cache_80_gb300 as pkv


def _empty_swapped(L=4):
    lib = pkv._L()
    pool = pkv.pkv_pool_create(L, 8, 2, 64, 16, "bf16", 32)
    s = pkv.pkv_seq_create(pool)  # no tokens, no blocks
    rc = lib.pkv_swap_out(pool.handle, s, None, None, None, 0, None, 0, None, None)
    assert rc == 0
    return lib, pool, s


def _reload(lib, pool, s, l0, l1):
    return lib.pkv_swap_in_layers(pool.handle, s, None, 0, 0, l0, l1, None, None, None, None)


def _name(lib, rc):
    return lib.pkv_status_name(rc).decode()


def test_ranges_must_start_at_zero_and_follow_each_other():
    lib, pool, s = _empty_swapped()
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_HOST
    for l0, l1 in ((1, 2), (0, 0), (0, 5), (3, 2), (-1, 1)):
        assert _name(lib, _reload(lib, pool, s, l0, l1)) == "PKV_ERR_INVALID_ARG"
        assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_HOST  # nothing changed
    assert _reload(lib, pool, s, 0, 1) == 0
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_RELOADING
    assert _name(lib, _reload(lib, pool, s, 2, 4)) == "PKV_ERR_INVALID_ARG"  # a gap
    assert _name(lib, _reload(lib, pool, s, 0, 1)) == "PKV_ERR_INVALID_ARG"  # again from 0
    # a whole-sequence swap-in or a swap-out is refused while the reload is under way
    assert _name(lib, lib.pkv_swap_in(pool.handle, s, None, 0, 0, None, None, None, None)) == "PKV_ERR_INVALID_ARG"
    assert _name(lib, lib.pkv_swap_out(pool.handle, s, None, None, None, 0, None, 0, None, None)) == \
        "PKV_ERR_INVALID_ARG"
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_RELOADING
    assert _reload(lib, pool, s, 1, 3) == 0
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_RELOADING
    assert _reload(lib, pool, s, 3, 4) == 0
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_HBM
    assert _name(lib, _reload(lib, pool, s, 0, 4)) == "PKV_ERR_INVALID_ARG"  # not swapped out any more


def test_one_range_is_a_whole_swap_in_and_the_sequence_can_swap_again():
    lib, pool, s = _empty_swapped(L=3)
    assert _reload(lib, pool, s, 0, 3) == 0
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_HBM
    assert lib.pkv_swap_out(pool.handle, s, None, None, None, 0, None, 0, None, None) == 0
    assert pkv.pkv_seq_residency(pool, s) == pkv.TIER_HOST


def test_a_freed_sequence_mid_reload_leaves_no_state():
    lib, pool, s = _empty_swapped()
    assert _reload(lib, pool, s, 0, 2) == 0
    pkv.pkv_seq_free(pool, s)
    assert _name(lib, _reload(lib, pool, s, 2, 4)) == "PKV_ERR_INVALID_ARG"  # a released sequence
    assert np.all(pkv.pkv_refcounts(pool) == 0)
