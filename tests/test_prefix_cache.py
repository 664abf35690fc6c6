"""The library's radix prefix cache against the oracle's (host control plane, no GPU).

Random request streams over a few shared "system prompts" (the agent workload of "KV Cache
Management", "Prefix Caching Across Turns": long invariant prefixes, short divergent turns)
drive both implementations in lockstep: attach (match, split, adopt, pin), append the rest
of the prompt and the generated tokens, insert, release, free, sequences that bypass the
cache, and evictions toward random targets.  After every operation the trees (preorder
export with reference counts, stamps and creation order), the block owner counts, the FIFO,
the match of random probes and the statistics must be identical.
"""
import random

import numpy as np
import pytest

import oracle
import paged_kv_cache_80_gb300 as pkv
from oracle.radix import RadixCache


class Pair:
    def __init__(self, num_blocks, B, seed):
        fo = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
        self.B = B
        self.lib = pkv.pkv_pool_create(1, 2, 2, 8, B, "bf16", num_blocks, fo)
        self.cache = pkv.pkv_prefix_cache_create(self.lib)
        self.orc = oracle.Pool(num_blocks, B, fo)
        self.ocache = RadixCache(self.orc, B)

    def check(self, probes=()):
        assert pkv.pkv_prefix_export(self.cache) == self.ocache.export()
        assert np.array_equal(pkv.pkv_refcounts(self.lib), self.orc.refcounts())
        assert np.array_equal(pkv.pkv_free_list(self.lib), self.orc.free_list())
        for p in probes:
            n1, b1 = pkv.pkv_prefix_match(self.cache, p)
            n2, b2 = self.ocache.match(p)
            assert n1 == n2 and list(b1) == list(b2)
        st = pkv.pkv_prefix_get_stats(self.cache)
        rows = self.ocache.export()
        parents = {r[0] for r in rows}
        assert st.nodes == len(rows) and st.blocks == sum(r[1] for r in rows)
        assert st.pinned_nodes == sum(1 for r in rows if r[2] > 0)
        assert st.dormant_leaves == sum(1 for i, r in enumerate(rows) if r[2] == 0 and i not in parents)
        assert (st.prompt_tokens, st.matched_tokens) == (self.ocache.prompt_tokens, self.ocache.matched_tokens)


@pytest.mark.parametrize("B,seed", [(2, 1), (4, 2), (16, 3), (1, 4)])
def test_random_request_streams_match_the_oracle(B, seed):
    rng = random.Random(seed)
    P = Pair(2048 if B >= 4 else 600, B, seed)
    alphabet = 3 if B <= 2 else 50
    systems = [[rng.randrange(alphabet) for _ in range(rng.randrange(0, 6 * B))] for _ in range(5)]

    def prompt():
        return rng.choice(systems) + [rng.randrange(alphabet) for _ in range(rng.randrange(0, 4 * B))]

    running = []  # (seq, tokens)
    for step in range(250):
        op = rng.random()
        if op < 0.45:
            pr, gen = prompt(), [rng.randrange(alphabet) for _ in range(rng.randrange(0, 3 * B))]
            s1, m1 = pkv.pkv_prefix_attach(P.cache, pr)
            s2, m2 = P.ocache.attach(pr)
            assert (s1, m1) == (s2, m2)
            n_new = len(pr) - m1 + len(gen)
            try:
                a, _ = pkv.pkv_plan_append(P.lib, [s1], [n_new])
            except pkv.PkvError as e:
                assert e.name == "PKV_ERR_OUT_OF_BLOCKS"
                with pytest.raises(oracle.OracleError):
                    P.orc.append([s2], [n_new])
                pkv.pkv_prefix_release(P.cache, s1)
                P.ocache.release(s2)
                pkv.pkv_seq_free(P.lib, s1)
                P.orc.seq_free(s2)
            else:
                b, _ = P.orc.append([s2], [n_new])
                assert np.array_equal(a, b)
                running.append((s1, pr + gen))
        elif op < 0.55:
            # a request that bypasses the cache, indexed when it finishes (its blocks duplicate cached content)
            pr = prompt()
            s1 = pkv.pkv_seq_create(P.lib)
            s2 = P.orc.seq_create()
            try:
                pkv.pkv_plan_append(P.lib, [s1], [len(pr)])
                P.orc.append([s2], [len(pr)])
                pkv.pkv_prefix_insert(P.cache, s1, pr)
                P.ocache.insert(s2, pr)
            except pkv.PkvError:
                with pytest.raises(oracle.OracleError):
                    P.orc.append([s2], [len(pr)])
            pkv.pkv_seq_free(P.lib, s1)
            P.orc.seq_free(s2)
        elif op < 0.85 and running:
            seq, toks = running.pop(rng.randrange(len(running)))
            keep = rng.random() < 0.2  # sometimes index only part of what it holds
            n = rng.randrange(len(toks) + 1) if keep else len(toks)
            pkv.pkv_prefix_insert(P.cache, seq, toks[:n])
            P.ocache.insert(seq, toks[:n])
            pkv.pkv_prefix_release(P.cache, seq)
            P.ocache.release(seq)
            pkv.pkv_seq_free(P.lib, seq)
            P.orc.seq_free(seq)
        else:
            target = len(P.orc.free_list()) + rng.randrange(0, 40)
            assert pkv.pkv_prefix_evict(P.cache, target) == P.ocache.evict(target)
        P.check([prompt() for _ in range(3)])
    # everything finishes; the cache still holds its blocks until evicted or destroyed
    for seq, toks in running:
        pkv.pkv_prefix_release(P.cache, seq)
        P.ocache.release(seq)
        pkv.pkv_seq_free(P.lib, seq)
        P.orc.seq_free(seq)
    P.check()
    assert pkv.pkv_prefix_get_stats(P.cache).pinned_nodes == 0
    assert pkv.pkv_prefix_evict(P.cache, 10 ** 9) == P.ocache.evict(10 ** 9)
    P.check()
    assert pkv.pkv_prefix_get_stats(P.cache).nodes == 0
    assert np.all(pkv.pkv_refcounts(P.lib) == 0)


def test_destroy_returns_the_blocks_and_errors_change_nothing():
    P = Pair(64, 4, 7)
    s = pkv.pkv_seq_create(P.lib)
    s2 = P.orc.seq_create()
    pkv.pkv_plan_append(P.lib, [s], [18])
    P.orc.append([s2], [18])
    toks = list(range(18))
    pkv.pkv_prefix_insert(P.cache, s, toks)
    P.ocache.insert(s2, toks)
    P.check()
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_prefix_insert(P.cache, s, toks + [1])  # more tokens than the sequence holds
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_prefix_release(P.cache, s)  # never attached
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_destroy(P.lib)  # a cache still holds references
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    P.check()
    pkv.pkv_seq_free(P.lib, s)
    P.orc.seq_free(s2)
    pkv.pkv_prefix_cache_destroy(P.cache)
    P.ocache.destroy()
    assert np.array_equal(pkv.pkv_refcounts(P.lib), P.orc.refcounts())
    assert np.array_equal(pkv.pkv_free_list(P.lib), P.orc.free_list())
    assert np.all(P.orc.refcounts() == 0)


def test_agent_turns_hit_rate():
    """Napkin Math 0.4 shape: agents sharing a 4,096-token system prompt (B 16), each turn
    appending a 32-token observation to its own history; every turn after an agent's first
    reuses its whole history in full blocks."""
    rng = random.Random(9)
    P = Pair(8192, 16, 9)
    system = [rng.randrange(32000) for _ in range(4096)]
    hist = {a: list(system) for a in range(8)}
    for turn in range(6):
        for a in range(8):
            obs = [rng.randrange(32000) for _ in range(32)]
            pr = hist[a] + obs
            s1, m1 = pkv.pkv_prefix_attach(P.cache, pr)
            s2, m2 = P.ocache.attach(pr)
            assert (s1, m1) == (s2, m2)
            assert m1 == (len(hist[a]) // 16) * 16 if (turn > 0 or a > 0) else m1 == 0
            gen = [rng.randrange(32000) for _ in range(24)]
            pkv.pkv_plan_append(P.lib, [s1], [len(pr) - m1 + len(gen)])
            P.orc.append([s2], [len(pr) - m2 + len(gen)])
            hist[a] = pr + gen
            pkv.pkv_prefix_insert(P.cache, s1, hist[a])
            P.ocache.insert(s2, hist[a])
            pkv.pkv_prefix_release(P.cache, s1)
            P.ocache.release(s2)
            pkv.pkv_seq_free(P.lib, s1)
            P.orc.seq_free(s2)
        P.check()
    st = pkv.pkv_prefix_get_stats(P.cache)
    assert st.matched_tokens / st.prompt_tokens == pytest.approx(P.ocache.hit_rate())
    assert st.matched_tokens / st.prompt_tokens > 0.95
