"""Admission-policy simulator, the oracle's version (test infrastructure only).

A plain restatement of "PagedAttention" (programmer.ie Inference ch. 14), "The policy is
where it succeeds or fails", on the oracle's block pool: a saturated queue of requests, a
decode loop in which every running sequence emits one token per step (prefill ignored),
three admission rules (reserve the maximum, reserve the declared limit, paged with a
watermark: admit only if, after the request's blocks are taken, the stated fraction of the
pool would still be free), preemption of the newest running sequence when a growing one
needs a block and none is free, and a flat recomputation charge per preemption.

Readings where the page is silent (the library's header states the same): the queue is
served head first; a preempted request goes back to the head of the queue and, when
readmitted, holds blocks for its prompt and the tokens it had already generated; within a
step sequences are processed oldest first and a finished one frees its blocks at once;
charged steps = steps + recompute_steps x preemptions.

Tokens that stay inside an already allocated block change no allocator state, so a paged
sequence's tokens are handed to the pool when one opens a block (all pending tokens at
once: exactly one new block), which leaves every allocation, free and FIFO order as a
token-by-token append would.
"""
from __future__ import annotations

import math
from collections import deque


def simulate(pool, policy: str, prompt, answer, declared=None, max_context: int = 1024, watermark: float = 0.0,
             recompute_steps: int = 4) -> dict:
    """Run the queue to completion on `pool` (an oracle.Pool with every block free)."""
    B, N = pool.block_size, pool.num_blocks
    assert pool.free_count() == N
    n = len(prompt)
    generated = [0] * n
    seq_of = [None] * n
    in_pool = [0] * n  # tokens of request i handed to the pool so far

    def tokens_on_admission(i):
        if policy == "reserve_max":
            return max_context
        if policy == "reserve_declared":
            return min(max_context, int(prompt[i]) + int(declared[i]))
        return int(prompt[i]) + generated[i]  # paged: the prompt, plus what it had generated if recomputed

    queue = deque(range(n))
    running = []  # oldest first
    steps = preemptions = completed = max_running = running_sum = 0
    while completed < n:
        # admit from the head of the queue while the rule allows
        while queue:
            i = queue[0]
            need = math.ceil(tokens_on_admission(i) / B)
            free = pool.free_count()
            if policy == "paged":
                admit = need <= free and (free - need) >= watermark * N
            else:
                admit = need <= free
            if not admit:
                break
            queue.popleft()
            s = pool.seq_create()
            if tokens_on_admission(i) > 0:
                pool.append([s], [tokens_on_admission(i)])
            seq_of[i] = s
            in_pool[i] = tokens_on_admission(i)
            running.append(i)
        if not running:
            raise RuntimeError("a request does not fit in the empty pool")
        # one decode step
        steps += 1
        running_sum += len(running)
        max_running = max(max_running, len(running))
        k = 0
        while k < len(running):
            i = running[k]
            pos = int(prompt[i]) + generated[i]  # position of the new token
            if policy == "paged" and pos % B == 0:
                # the new token opens a block: take a free one, or preempt the newest sequence
                preempted_self = False
                while pool.free_count() == 0:
                    victim = running.pop()
                    pool.seq_free(seq_of[victim])
                    seq_of[victim] = None
                    queue.appendleft(victim)
                    preemptions += 1
                    if victim == i:
                        preempted_self = True
                        break
                if preempted_self:
                    continue
            if policy == "paged" and pos % B == 0:
                pool.append([seq_of[i]], [pos + 1 - in_pool[i]])  # opens the block of `pos`
                in_pool[i] = pos + 1
            generated[i] += 1
            if generated[i] == int(answer[i]):
                pool.seq_free(seq_of[i])
                seq_of[i] = None
                running.pop(k)
                completed += 1
                continue
            k += 1
    return {"steps": steps, "charged_steps": steps + recompute_steps * preemptions, "preemptions": preemptions,
            "completed": completed, "max_running": max_running,
            "mean_running": running_sum / steps if steps else 0.0}
