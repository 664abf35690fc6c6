"""Pins of the radix prefix cache oracle (oracle/radix.py) against the pages (no GPU).

"KV Cache Management" (cs249r vol. 3 ch. 5), "Prefix Caching Across Turns": the worked
numbers of "Longest prefix matching" (100 matched tokens at B = 16 -> 6 full blocks, 96
usable) and Napkin Math 0.4 (a 4,096-token prefix of 256 blocks, 32 novel tokens), Figure 6
(pinned nodes survive, dormant leaves go least recently used first), the cascading
eligibility rule of "Dynamic radix eviction", Eq. 2 (hit rate), plus brute-force checks of
the longest whole-block match against every cached path and of the block owner counts.
Each pin takes the cache class as an argument so that the planted mistakes at the end can
be run through the same checks.
"""
import importlib.util
import os
import random
import sys
import types

import numpy as np
import pytest

import oracle
from oracle.radix import RadixCache

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def new_cache(cls, num_blocks, B, free_order=None):
    pool = oracle.Pool(num_blocks, B, free_order)
    return pool, cls(pool, B)


def run_request(pool, cache, prompt, generated, finish=True):
    """Serve a prompt from the cache, append the rest of the prompt and the generated
    tokens, and (if finish) index the sequence, release its pins and free it."""
    seq, matched = cache.attach(prompt)
    pool.append([seq], [len(prompt) - matched + len(generated)])
    if finish:
        cache.insert(seq, list(prompt) + list(generated))
        cache.release(seq)
        pool.seq_free(seq)
    return seq, matched


# ------------------------------------------------------------------ pins


def pin_truncation_100_tokens(cls):
    pool, c = new_cache(cls, 64, 16)
    base = list(range(1000, 1112))  # 7 full blocks
    seq, _ = run_request(pool, c, base, [], finish=False)
    c.insert(seq, base)
    prompt = base[:100] + [1, 2, 3, 4, 5]
    n, blocks = c.match(prompt)
    assert n == 96 and len(blocks) == 6  # floor(100 / 16) = 6 full blocks, tail of 4 recomputed
    assert list(blocks) == [int(x) for x in pool.table(seq)[:6]]
    assert c.match(base[:100])[0] == 96
    assert c.match(base[:15])[0] == 0


def pin_napkin_04(cls):
    pool, c = new_cache(cls, 600, 16)
    system = list(range(5000, 5000 + 4096))
    s0, m0 = run_request(pool, c, system, [7] * 20)
    assert m0 == 0
    seq, matched = c.attach(system + list(range(32)))
    assert matched == 4096 and pool.seq_len(seq) == 4096 and len(pool.table(seq)) == 256
    free_before = len(pool.free_list())
    pool.append([seq], [32])
    assert len(pool.table(seq)) == 258 and free_before - len(pool.free_list()) == 2  # 32 novel tokens
    assert c.hit_rate() == pytest.approx(4096 / (4096 + 4128))


def _figure6(cls):
    """Node 1: system prompt; children 2 (python), 3 (bash), 4 (git)."""
    pool, c = new_cache(cls, 80, 4)
    sysp = [9] * 8
    branch = {name: [t] * 8 for name, t in (("python", 1), ("bash", 2), ("git", 3))}
    run_request(pool, c, sysp + branch["bash"], [2] * 4)       # finishes first (oldest)
    run_request(pool, c, sysp + branch["git"], [3] * 4)        # finishes second
    run_request(pool, c, sysp + branch["python"], [])          # indexes the python scratchpad
    # an active request reading through the system prompt and the scratchpad pins both
    py, matched = run_request(pool, c, sysp + branch["python"] + [4] * 4, [], finish=False)
    assert matched == 16
    rows = c.export()
    return pool, c, py, rows


def pin_figure6_leaf_first_lru(cls):
    pool, c, py, rows = _figure6(cls)
    # nodes: the system prompt (shared, pinned through the running python request), its three branches
    first_tokens = {tuple(r[5][:4]): r for r in rows}
    assert first_tokens[(9, 9, 9, 9)][2] == 1 and first_tokens[(1, 1, 1, 1)][2] == 1  # pinned
    assert first_tokens[(2, 2, 2, 2)][2] == 0 and first_tokens[(3, 3, 3, 3)][2] == 0  # dormant leaves
    free0 = len(pool.free_list())
    c.evict(free0 + 1)  # the least recently used dormant leaf goes first: bash
    left = {tuple(r[5][:4]) for r in c.export()}
    assert (2, 2, 2, 2) not in left and (3, 3, 3, 3) in left and (1, 1, 1, 1) in left
    c.evict(10 ** 6)  # everything evictable: git too, never the pinned path
    left = {tuple(r[5][:4]) for r in c.export()}
    assert left == {(9, 9, 9, 9), (1, 1, 1, 1)}
    c.release(py)
    pool.seq_free(py)
    c.evict(10 ** 6)  # python becomes a dormant leaf, then its parent (cascade)
    assert c.export() == []
    assert len(pool.free_list()) == 80


def pin_cascade_only_after_children(cls):
    pool, c = new_cache(cls, 40, 2)
    run_request(pool, c, [1, 1, 2, 2], [])
    run_request(pool, c, [1, 1, 3, 3], [])
    run_request(pool, c, [1, 1], [])  # the shared parent is stamped last: youngest
    rows = c.export()
    assert len(rows) == 3 and rows[0][1] == 1  # parent [1,1] with two children
    free0 = len(pool.free_list())
    c.evict(free0 + 1)  # one block short: the oldest child leaf goes, not the younger parent
    assert {tuple(r[5]) for r in c.export()} == {(1, 1), (3, 3)}
    c.evict(free0 + 3)
    assert c.export() == []


def pin_brute_force_match_and_owner_counts(cls, seed=0, steps=120):
    rng = random.Random(seed)
    B = 2
    pool, c = new_cache(cls, 400, B, np.random.default_rng(seed).permutation(400).astype(np.int32))
    running = []
    bases = [[rng.randrange(3) for _ in range(rng.randrange(0, 7))] for _ in range(4)]
    for _ in range(steps):
        op = rng.random()
        if op < 0.55:
            prompt = rng.choice(bases) + [rng.randrange(3) for _ in range(rng.randrange(0, 7))]
            gen = [rng.randrange(3) for _ in range(rng.randrange(0, 4))]
            seq, matched = c.attach(prompt)
            pool.append([seq], [len(prompt) - matched + len(gen)])
            running.append((seq, prompt + gen, prompt[:matched]))
        elif op < 0.85 and running:
            seq, toks, _ = running.pop(rng.randrange(len(running)))
            c.insert(seq, toks)
            c.release(seq)
            pool.seq_free(seq)
        else:
            target = len(pool.free_list()) + rng.randrange(0, 12)
            c.evict(target)
            rows = c.export()
            parents = {r[0] for r in rows}
            dormant = [i for i, r in enumerate(rows) if r[2] == 0 and i not in parents]
            assert len(pool.free_list()) >= target or not dormant
        # brute force: every cached path, and the longest whole-block prefix of random probes
        rows = c.export()
        paths = []
        for i, r in enumerate(rows):
            toks, blks, j = [], [], i
            while j != -1:
                toks = rows[j][5] + toks
                blks = rows[j][6] + blks
                j = rows[j][0]
            paths.append((toks, blks))
        for _ in range(3):
            probe = rng.choice(bases) + [rng.randrange(3) for _ in range(rng.randrange(0, 7))]
            best, best_blocks = 0, []
            for toks, blks in paths:
                k = 0
                while (k + 1) * B <= min(len(toks), len(probe)) and toks[k * B:(k + 1) * B] == probe[k * B:(k + 1) * B]:
                    k += 1
                if k > best // B:
                    best, best_blocks = k * B, blks[:k]
            n, blocks = c.match(probe)
            assert n == best and list(blocks) == list(best_blocks)
        # owners: each live sequence's blocks plus one per block indexed by the cache
        # pins: a node is referenced once per running request whose matched prefix holds its whole path
        for (toks, _), r in zip(paths, rows):
            want_ref = sum(1 for _, _, m in running if len(toks) <= len(m) and m[:len(toks)] == toks)
            assert r[2] == want_ref
        want = np.zeros(400, np.int64)
        for seq, _, _ in running:
            for p in pool.table(seq):
                want[p] += 1
        for r in rows:
            for p in r[6]:
                want[p] += 1
        assert np.array_equal(pool.refcounts(), want)
        pinned = sum(1 for r in rows if r[2] > 0)
        assert pinned <= len(rows)
    # Eq. 2 bookkeeping
    assert 0.0 <= c.hit_rate() <= 1.0


PINS = [pin_truncation_100_tokens, pin_napkin_04, pin_figure6_leaf_first_lru, pin_cascade_only_after_children,
        pin_brute_force_match_and_owner_counts]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_radix_oracle_pin(pin):
    pin(RadixCache)


# ------------------------------------------------------------------ planted mistakes

RADIX_MUTANTS = {
    "lru_picks_newest": ("leaf = min(queue, key=lambda n: (n.last_access, n.serial))",
                         "leaf = max(queue, key=lambda n: (n.last_access, n.serial))"),
    "no_cascade": ("                queue.append(parent)", "                pass"),
    "release_only_deepest": ("        n = deepest\n        while n is not self.root:\n            n.ref_count -= 1\n            n.last_access = self.clock\n            n = n.parent",
                             "        deepest.ref_count -= 1\n        deepest.last_access = self.clock"),
    "split_drops_pins": ("        upper.ref_count = node.ref_count", "        upper.ref_count = 0"),
    "insert_takes_no_reference": ("                    self.pool.block_retain(p)", "                    pass"),
    "partial_block_shared": ("        return [tuple(tokens[i * B:(i + 1) * B]) for i in range(len(tokens) // B)]",
                             "        return [tuple(tokens[i * B:(i + 1) * B]) for i in range(-(-len(tokens) // B))]"),
    # pinned leaves become candidates and are not skipped
    "evicts_pinned": ("        queue = [n for n in self._nodes() if n.ref_count == 0 and not n.children]",
                      "        queue = [n for n in self._nodes() if not n.children]",
                      "            if leaf.ref_count > 0:\n                continue\n", ""),
}


def _load_mutant(name, *edits):
    src = open(os.path.join(ROOT, "oracle", "radix.py")).read()
    for old, new in zip(edits[::2], edits[1::2]):
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    mod = types.ModuleType(f"radix_mutant_{name}")
    exec(compile(src, f"radix_mutant_{name}", "exec"), mod.__dict__)
    return mod.RadixCache


@pytest.mark.parametrize("name", sorted(RADIX_MUTANTS))
def test_every_planted_radix_mistake_fails_a_pin(name):
    cls = _load_mutant(name, *RADIX_MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin(cls)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
