"""The library's admission simulator (pkv_sim_run, on the pool's own allocator) against the
oracle's (no GPU): identical step counts, preemptions and occupancy for every policy on
seeded workloads, and the argument checks."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W
from oracle.admission import simulate


@pytest.mark.parametrize("kind", ["chat", "long_prompt", "long_answer"])
@pytest.mark.parametrize("policy,watermark", [("reserve_max", 0.0), ("reserve_declared", 0.0), ("paged", 0.0),
                                              ("paged", 0.05), ("paged", 0.2)])
def test_library_simulator_matches_oracle(kind, policy, watermark):
    pr, an, de = W.admission(kind, 400)
    for blocks, B in ((256, 16), (700, 8)):
        lib = pkv.pkv_sim_run(pkv.pkv_pool_create(1, 2, 2, 8, B, "bf16", blocks), policy, pr, an, de,
                              watermark=watermark)
        orc = simulate(oracle.Pool(blocks, B), policy, pr, an, de, watermark=watermark)
        assert lib == orc


def test_simulator_leaves_the_pool_free_and_checks_arguments():
    p = pkv.pkv_pool_create(1, 2, 2, 8, 16, "bf16", 256)
    pr, an, de = W.admission("chat", 100)
    pkv.pkv_sim_run(p, "paged", pr, an, de, watermark=0.1)
    assert len(pkv.pkv_free_list(p)) == 256 and np.all(pkv.pkv_refcounts(p) == 0)
    for bad in [dict(prompt=[10], answer=[0]), dict(prompt=[1000], answer=[100]), dict(prompt=[5], answer=[9], declared=[3])]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_sim_run(p, "reserve_declared" if "declared" in bad else "paged", bad["prompt"], bad["answer"],
                            bad.get("declared", [9]))
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_sim_run(p, "paged", [4], [1], watermark=1.0)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:  # 8 blocks of 16 cannot hold a 1,024-token reservation
        pkv.pkv_sim_run(pkv.pkv_pool_create(1, 2, 2, 8, 16, "bf16", 8), "reserve_max", [4], [1])
    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
    s = pkv.pkv_seq_create(p)
    pkv.pkv_plan_append(p, [s], [3])
    with pytest.raises(pkv.PkvError) as e:  # the pool must start empty
        pkv.pkv_sim_run(p, "paged", [4], [1])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
