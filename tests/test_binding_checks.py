"""The binding's step calls reject undersized buffers before anything reaches the library.

The C calls copy fixed byte counts (n*(W+2) int32 of metadata, n rows of q / k_new /
v_new / out) and cannot see the caller's buffer sizes, so the binding checks them; a
too-small buffer must raise ValueError without changing the pool's state.  These
checks run before any device pointer is taken, so they are tested here on the CPU.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_80_gb300 as pkv


def _pool():
    lib = pkv.pkv_pool_create(1, 8, 2, 64, 16, "bf16", 64)
    ids = [pkv.pkv_seq_create(lib) for _ in range(3)]
    pkv.pkv_plan_append(lib, ids, [5, 16, 40])
    return lib, np.array(ids, np.int32)


def _buffers(n, W, short=None):
    """Host stand-ins of every step buffer, sized for n sequences; `short` names one to make a row short."""
    q = torch.zeros((n, 8, 64), dtype=torch.bfloat16)
    kv = torch.zeros((n, 2, 64), dtype=torch.bfloat16)
    bufs = {"meta_host": torch.zeros(n * (W + 2), dtype=torch.int32),
            "meta_dev": torch.zeros(n * (W + 2), dtype=torch.int32),
            "q": q.clone(), "k_new": kv.clone(), "v_new": kv.clone(), "out": q.clone()}
    if short is not None:
        t = bufs[short]
        bufs[short] = t.reshape(-1)[: t.numel() - 1].clone()
    return bufs


def _state(lib):
    return pkv.pkv_refcounts(lib).copy(), pkv.pkv_free_list(lib).copy(), [pkv.pkv_seq_len(lib, s) for s in range(3)]


@pytest.mark.parametrize("short", ["meta_host", "meta_dev", "q", "k_new", "v_new", "out"])
def test_step_calls_reject_short_buffers(short):
    lib, ids = _pool()
    n, W = len(ids), 4
    before = _state(lib)
    b = _buffers(n, W, short)
    ws = torch.zeros(16, dtype=torch.uint8)
    kp = torch.zeros(1, dtype=torch.bfloat16)
    calls = {
        "pkv_decode_step": lambda: pkv.pkv_decode_step(lib, 0, ids, W, b["q"], b["k_new"], b["v_new"], kp, kp, 0.1,
                                                       b["out"], b["meta_host"], b["meta_dev"], ws),
        "pkv_decode_step_host": lambda: pkv.pkv_decode_step_host(
            lib, 0, ids, W, b["q"], b["k_new"], b["v_new"], b["out"], b["q"], b["k_new"], b["v_new"], b["out"], kp,
            kp, 0.1, b["meta_host"], b["meta_dev"], ws),
        "pkv_step_launch": lambda: pkv.pkv_step_launch(lib, 0, n, W, np.zeros((0, 2), np.int32), b["q"], b["k_new"],
                                                       b["v_new"], kp, kp, 0.1, b["out"], b["meta_host"],
                                                       b["meta_dev"], ws),
        "pkv_step_launch_host": lambda: pkv.pkv_step_launch_host(
            lib, 0, n, W, np.zeros((0, 2), np.int32), b["q"], b["k_new"], b["v_new"], b["out"], b["q"], b["k_new"],
            b["v_new"], b["out"], kp, kp, 0.1, b["meta_host"], b["meta_dev"], ws),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="bytes; this step needs"):
            call()
    assert all(np.array_equal(x, y) for x, y in zip(before[:2], _state(lib)[:2]))
    assert before[2] == _state(lib)[2]


def test_step_plan_rejects_a_short_metadata_buffer():
    lib, ids = _pool()
    before = _state(lib)
    with pytest.raises(ValueError, match="meta_host"):
        pkv.pkv_step_plan(lib, ids, 4, torch.zeros(len(ids) * 6 - 1, dtype=torch.int32))
    assert before[2] == _state(lib)[2]
    assert np.array_equal(before[0], _state(lib)[0])


def test_full_size_buffers_pass_the_size_checks():
    """With every buffer large enough the calls get as far as taking device pointers
    (which host tensors are not): the size checks themselves do not reject them."""
    lib, ids = _pool()
    n, W = len(ids), 4
    b = _buffers(n, W)
    ws = torch.zeros(16, dtype=torch.uint8)
    kp = torch.zeros(1, dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="CUDA tensor"):
        pkv.pkv_step_launch(lib, 0, n, W, np.zeros((0, 2), np.int32), b["q"], b["k_new"], b["v_new"], kp, kp, 0.1,
                            b["out"], b["meta_host"], b["meta_dev"], ws)


def test_sharing_enlarges_the_metadata_the_binding_checks():
    """With prefix sharing on, a step's metadata holds the shared-prefix plan after the lengths:
    a buffer of the plain n*(W+2) int32 is now too small, for the planning call as for the
    launches, and is rejected before the library writes past it."""
    lib = pkv.pkv_pool_create(1, 16, 2, 128, 16, "bf16", 256)
    parent = pkv.pkv_seq_create(lib)
    pkv.pkv_plan_append(lib, [parent], [100])
    ids = np.array([pkv.pkv_seq_fork(lib, parent) for _ in range(5)], np.int32)
    n, W = len(ids), 12
    assert pkv.pkv_step_meta_ints(lib, n, W) == n * (W + 2)
    pkv.pkv_pool_set_prefix_sharing(lib, 4, 1, 152)
    need = pkv.pkv_step_meta_ints(lib, n, W)
    assert need > n * (W + 2)
    before = [pkv.pkv_seq_len(lib, s) for s in ids]
    with pytest.raises(ValueError, match="meta_host"):
        pkv.pkv_step_plan(lib, ids, W, torch.zeros(n * (W + 2), dtype=torch.int32))
    assert [pkv.pkv_seq_len(lib, s) for s in ids] == before  # nothing planned
    meta = torch.zeros(need, dtype=torch.int32)
    pkv.pkv_step_plan(lib, ids, W, meta)  # the right size plans: one group of the 5 branches
    off = (n * (W + 2) + 3) // 4 * 4
    assert int(meta[off]) >= 1 and int(meta[off + 1]) == 5
    q = torch.zeros((n, 16, 128), dtype=torch.bfloat16)
    kv = torch.zeros((n, 2, 128), dtype=torch.bfloat16)
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="meta_dev"):
        pkv.pkv_step_launch(lib, 0, n, W, np.zeros((0, 2), np.int32), q, kv, kv, q, q, 0.1, q, meta,
                            torch.zeros(n * (W + 2), dtype=torch.int32), ws)


def test_sharing_needs_the_host_metadata_in_a_packed_launch():
    """With sharing on, a packed launch whose metadata the caller queued itself (off_meta 0,
    meta_host NULL) is rejected before anything is queued: the call reads the step's plan from
    the host copy (and the plan leaves a run's shared entries only in its first row's table)."""
    import ctypes

    lib = pkv.pkv_pool_create(1, 16, 2, 128, 16, "bf16", 64)
    pkv.pkv_pool_set_prefix_sharing(lib, 4, 1, 152)
    n, W = 4, 8
    rq, rk = 16 * 128 * 2, 2 * 128 * 2
    off_k, off_v = n * rq, n * (rq + rk)
    in_bytes = n * (rq + 2 * rk)
    fake = ctypes.c_void_p(256)  # never dereferenced: the call fails on its arguments first
    rc = pkv._L().pkv_step_launch_packed(lib.handle, 0, n, W, None, 0, fake, fake, off_k, off_v, 0, in_bytes, fake,
                                          fake, fake, fake, 0.1, None, fake, fake, 1 << 20, None, None, None)
    assert pkv._L().pkv_status_name(rc).decode() == "PKV_ERR_INVALID_ARG"
    assert "sharing" in pkv._L().pkv_last_error_message().decode()
