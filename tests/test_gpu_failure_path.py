"""Failure detection on the GPU without a fault: a bounded wait runs out (nothing
completes the barrier), the kernel records a timeout and returns, the host reads
the status, and the context keeps working."""
import numpy as np
import pytest

import paged_kv_cache_80_gb300 as pkv
import workloads as W
from helpers import PagedBatch, check_attention

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    pkv.pkv_check_device_error()  # start clean
    pkv.pkv_selftest_bounded_wait(50_000_000)  # 50 ms
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_check_device_error()
    assert e.value.name == "PKV_ERR_DEVICE_CHECK"
    assert "code 5" in str(e.value)
    # the error word was cleared and the device still runs the hot path
    assert pkv.pkv_check_device_error() == (0, 0)
    g = W.Geometry(L=1, H_q=16, H_kv=2, d_head=128, block_size=16, dtype="bf16", num_blocks=64)
    b = PagedBatch(g, None, seed=51)
    ids = b.new_seqs(2)
    b.append(ids, [30, 70], "p")
    q = W.normal(51, "q", (2, 16, 128), "bf16")
    got, t, l = b.decode_gpu(ids, q, 0.1)
    check_attention(got, b.decode_ref(q, t, l, 0.1), "bf16")


def test_selftest_rejects_bad_timeouts():
    for bad in (0, -5, 20_000_000_000):
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_selftest_bounded_wait(bad)
        assert e.value.name == "PKV_ERR_INVALID_ARG"
