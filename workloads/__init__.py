"""Seeded synthetic inputs for the paged KV cache hot path.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It only draws random numbers and shapes workloads (lengths, free-list
orders, tensor contents); it holds none of the paged-cache arithmetic (no block
tables, slots, softmax or copies).

Workload shapes follow the pages' workloads:

* ``tiny``      -- GPT-2-small geometry (12 heads, d_head 64, fp32), the geometry of
  the GPT-2 cache in "PagedAttention" (programmer.ie Inference ch. 14, "The real cache").
* ``chat``      -- 70B GQA layer (64 query / 8 KV heads, d_head 128, bf16), the
  chat-like length mix of "PagedAttention" ("Where contiguous allocation wastes
  memory": mean prompt 217, mean output 154, maximum context 1,024, lognormal).
* ``agent32k``  -- 48 sequences of 32,768 tokens: "KV Cache Management"
  (cs249r vol. 3 ch. 5), Napkin Math 0.1 (8,192 / 32,768 / 131,072-token contexts).
* ``forked``    -- one shared prefix forked into 64 branches ("KV Cache Management",
  "Zero-copy deliberation via copy-on-write branching").
* ``swap``      -- 80-layer 70B geometry (327,680 bytes per token), 256-token chunks
  ("KV Cache Management", "Asynchronous paged swapping").

Every generator takes an explicit seed; ``substream(seed, tag)`` derives an
independent PCG64 stream per named array so that any array can be regenerated
without the others.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional

import numpy as np

# dtype names used throughout (element bytes in parentheses)
DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}

# seed = workload index * 1000 + 7
SEEDS = {"tiny": 1007, "chat": 2007, "agent32k": 3007, "forked": 4007, "swap": 5007, "admission": 6007}


def substream(seed: int, tag: str) -> np.random.Generator:
    """Independent PCG64 stream for (seed, tag)."""
    h = int.from_bytes(hashlib.sha256(tag.encode()).digest()[:8], "little")
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, h])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the
    16-bit patterns as uint16.  Inputs are finite (normal draws)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(seed: int, tag: str, shape, dtype: str) -> np.ndarray:
    """N(0,1) draws in float32, stored in ``dtype``.

    Returns raw element storage: uint16 bit patterns for bf16, float16 for f16,
    float32 for f32.
    """
    g = substream(seed, tag)
    x = g.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def to_float64(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw element storage (as returned by :func:`normal`) to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(raw).astype(np.float64)
    return np.asarray(raw).astype(np.float64)


def device_normal(seed: int, tag: str, shape, dtype: str, device):
    """N(0,1) draws made on a torch device (for pools too large to draw on the host).

    The values come from torch's seeded generator on ``device``; they are the input
    for both sides (the oracle reads back the blocks it needs).
    """
    import torch

    h = int.from_bytes(hashlib.sha256(tag.encode()).digest()[:6], "little")
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1_000_003 + h) % (2**63 - 1))
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}[dtype]
    # FP8 draws are returned as their uint8 codes (the pool's storage)
    out = torch.empty(shape, dtype=torch.uint8 if dtype == "e4m3" else tdt, device=device)
    # fill in slabs to bound the float32 temporary
    flat = out.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        x = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(tdt)
        flat[i : i + n] = x.view(torch.uint8) if dtype == "e4m3" else x
    return out


def permutation(seed: int, tag: str, n: int) -> np.ndarray:
    return substream(seed, tag).permutation(n).astype(np.int32)


def uniform_int(seed: int, tag: str, lo: int, hi: int, size) -> np.ndarray:
    """Integers uniform on [lo, hi] inclusive."""
    return substream(seed, tag).integers(lo, hi + 1, size=size).astype(np.int64)


def lognormal_lengths(seed: int, tag: str, mean: float, size, sigma: float = 1.0) -> np.ndarray:
    """Lognormal draws with the given mean: mu = ln(mean) - sigma^2/2, rounded to ints."""
    mu = math.log(mean) - sigma * sigma / 2.0
    x = substream(seed, tag).lognormal(mu, sigma, size=size)
    return np.rint(x).astype(np.int64)


@dataclasses.dataclass(frozen=True)
class Geometry:
    L: int
    H_q: int
    H_kv: int
    d_head: int
    block_size: int
    dtype: str
    num_blocks: int

    @property
    def elem_bytes(self) -> int:
        return DTYPE_BYTES[self.dtype]

    def pool_shape(self):
        """Pool layout: [num_blocks][L][H_kv][block_size][d_head]."""
        return (self.num_blocks, self.L, self.H_kv, self.block_size, self.d_head)


@dataclasses.dataclass
class Workload:
    name: str
    geometry: Geometry
    seed: int
    free_order: np.ndarray  # initial FIFO order of block ids
    lengths: np.ndarray  # starting lengths of the sequences (after prompt / prefix)
    extra: dict

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.geometry.d_head)


def tiny(n_seq: int = 8) -> Workload:
    """12 query = 12 KV heads, d_head 64, fp32, B=16, 512-block pool in a seeded
    random order; lengths uniform in [1, 512]."""
    s = SEEDS["tiny"]
    g = Geometry(L=1, H_q=12, H_kv=12, d_head=64, block_size=16, dtype="f32", num_blocks=512)
    return Workload("tiny", g, s, permutation(s, "free_order", 512), uniform_int(s, "lengths", 1, 512, n_seq), {})


def chat(n_seq: int = 256, num_blocks: int = 32768, steps: int = 64) -> Workload:
    """Chat-like ragged batch: prompt lengths lognormal (mean 217), generated lengths
    lognormal (mean 154), sigma 1; prompt clipped to [1, 1024 - steps], generated
    clipped to [1, 1024 - prompt]."""
    s = SEEDS["chat"]
    g = Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=num_blocks)
    prompt = np.clip(lognormal_lengths(s, "prompt", 217.0, n_seq), 1, 1024 - steps)
    gen = lognormal_lengths(s, "generated", 154.0, n_seq)
    gen = np.clip(gen, 1, 1024 - prompt)
    return Workload("chat", g, s, permutation(s, "free_order", num_blocks), prompt,
                    {"generated": gen, "steps": steps})


def agent(n_seq: int = 48, context: int = 32768, spare_steps: int = 256) -> Workload:
    """Long-context agent batch: n_seq sequences of ``context`` tokens, block ids a
    seeded random permutation of a pool sized for the contexts plus ``spare_steps``
    decode steps."""
    s = SEEDS["agent32k"]
    B = 16
    nb = n_seq * (-(-context // B)) + n_seq * (-(-spare_steps // B) + 1)
    g = Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=B, dtype="bf16", num_blocks=nb)
    return Workload(f"agent{context}", g, s, permutation(s, f"free_order_{n_seq}_{context}", nb),
                    np.full(n_seq, context, dtype=np.int64), {})


def forked(n_branch: int = 64, prefix: int = 16376, max_suffix: int = 2048, num_blocks: int = 16384) -> Workload:
    """One parent prefix of ``prefix`` tokens (ends mid-block: 16,376 = 1,023 full
    16-token blocks + 8), forked into ``n_branch`` branches, each appending a suffix
    uniform in [0, max_suffix]."""
    s = SEEDS["forked"]
    g = Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=num_blocks)
    return Workload("forked", g, s, permutation(s, "free_order", num_blocks),
                    np.array([prefix], dtype=np.int64),
                    {"suffix": uniform_int(s, "suffix", 0, max_suffix, n_branch), "n_branch": n_branch})


def swap(n_chunks: int = 512, chunk_blocks: int = 16, num_blocks: int = 12288, L: int = 80) -> Workload:
    """80-layer 70B geometry; ``n_chunks`` sequences of one 256-token chunk each are
    evicted to the host tier in a seeded random order, then a seeded random half is
    restored."""
    s = SEEDS["swap"]
    g = Geometry(L=L, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=num_blocks)
    evict_order = permutation(s, "evict_order", n_chunks)
    restore = substream(s, "restore").choice(n_chunks, size=n_chunks // 2, replace=False).astype(np.int32)
    return Workload("swap", g, s, permutation(s, "free_order", num_blocks),
                    np.full(n_chunks, chunk_blocks * 16, dtype=np.int64),
                    {"evict_order": evict_order, "restore": restore, "chunk_blocks": chunk_blocks})


# (mean prompt, mean answer) of the admission-simulator workloads: "chat-like" is the chat
# length mix above; "long prompt" and "long answer" are not parameterised on the page.
ADMISSION_KINDS = {"chat": (217.0, 154.0), "long_prompt": (600.0, 60.0), "long_answer": (40.0, 500.0)}


def admission(kind: str = "chat", n: int = 3000, max_context: int = 1024):
    """Request lengths for the admission simulator: lognormal prompt and answer (sigma 1,
    the given means), prompt clipped to [1, max_context - 1], answer to [1, max_context -
    prompt]; each request declares an output limit of twice its answer, capped by the
    context.  Returns int32 arrays (prompt, answer, declared)."""
    s = SEEDS["admission"]
    mp, ma = ADMISSION_KINDS[kind]
    prompt = np.clip(lognormal_lengths(s, f"{kind}_prompt", mp, n), 1, max_context - 1)
    answer = np.clip(lognormal_lengths(s, f"{kind}_answer", ma, n), 1, max_context - prompt)
    declared = np.minimum(max_context - prompt, 2 * answer)
    return prompt.astype(np.int32), answer.astype(np.int32), declared.astype(np.int32)
