"""CPU oracle for the paged KV cache hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline arm
import this package.  The product library never does, and the oracle imports
nothing from the product package.  It wraps ``pkv_oracle.cpp`` (plain C++17,
double-precision attention, FIFO reference-counted allocator) through ctypes and
takes numpy arrays.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against facts the pages fix (worked examples, closed forms, invariants, library
routines on special cases).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "OUT_OF_BLOCKS", 3: "DOUBLE_FREE", 4: "BAD_BLOCK_ID"}
DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}

_lib = None


def lib():
    global _lib
    if _lib is None:
        # PKV_ORACLE_LIB points the tests at a deliberately broken copy (mutation tests)
        path = os.environ.get("PKV_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        P32 = ctypes.POINTER(ctypes.c_int32)
        P64 = ctypes.POINTER(ctypes.c_int64)
        L.orc_pool_new.restype = vp
        L.orc_pool_new.argtypes = [i64, i64, P32]
        L.orc_pool_delete.argtypes = [vp]
        L.orc_seq_create.argtypes = [vp, P32]
        L.orc_seq_fork.argtypes = [vp, i32, P32]
        L.orc_seq_free.argtypes = [vp, i32]
        L.orc_append.argtypes = [vp, P32, P32, ctypes.c_int, P32, P32, P32]
        L.orc_seq_len.restype = i64
        L.orc_seq_len.argtypes = [vp, i32]
        L.orc_seq_table.restype = i64
        L.orc_seq_table.argtypes = [vp, i32, P32, i64]
        L.orc_refcounts.argtypes = [vp, P32]
        L.orc_free_list.restype = i64
        L.orc_free_list.argtypes = [vp, P32]
        L.orc_seq_adopt.argtypes = [vp, P32, i64, i64, P32]
        L.orc_free_count.restype = i64
        L.orc_free_count.argtypes = [vp]
        L.orc_block_retain.argtypes = [vp, i32]
        L.orc_block_release.argtypes = [vp, i32]
        L.orc_swap_out.argtypes = [vp, i32, P64, P32]
        L.orc_swap_in.argtypes = [vp, i32, P32, P64]
        geo = [ctypes.c_int] * 5 + [i64]
        L.orc_write_slots.argtypes = geo + [ctypes.c_int, vp, vp, P32, i64, vp, vp]
        L.orc_copy_blocks.argtypes = geo + [P32, i64, vp, vp]
        L.orc_swap_out_data.argtypes = geo + [P32, P64, i64, vp, vp, vp]
        L.orc_swap_in_data.argtypes = geo + [P32, P64, i64, vp, vp, vp]
        L.orc_write_slots_e4m3.argtypes = [ctypes.c_int] * 4 + [i64, ctypes.c_int, vp, vp, P32, i64,
                                                                 ctypes.c_float, ctypes.c_float, vp, vp]
        L.orc_e4m3_encode.argtypes = [vp, i64, vp]
        L.orc_e4m3_decode.argtypes = [vp, i64, vp]
        L.orc_decode_attention.argtypes = [ctypes.c_int] * 6 + [i64, ctypes.c_int, vp, ctypes.c_int, vp, vp, dbl,
                                                                 dbl, P32, ctypes.c_int, P32, ctypes.c_int, dbl,
                                                                 ctypes.POINTER(dbl), ctypes.c_int]
        L.orc_prefill_attention.argtypes = [ctypes.c_int] * 6 + [i64, ctypes.c_int, vp, ctypes.c_int, P32, vp, vp,
                                                                  dbl, dbl, P32, ctypes.c_int, P32, ctypes.c_int, dbl,
                                                                  ctypes.POINTER(dbl), ctypes.c_int]
        L.orc_hardware_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _p64(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _vp(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.status = STATUS.get(code, str(code))


def _check(code: int, what: str):
    if code != 0:
        raise OracleError(code, what)


class Pool:
    """Reference-counted FIFO block allocator with per-sequence block tables."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[np.ndarray] = None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        fo = None
        if free_order is not None:
            self._fo = np.ascontiguousarray(free_order, dtype=np.int32)
            fo = _p32(self._fo)
        self._h = lib().orc_pool_new(self.num_blocks, self.block_size, fo)
        if not self._h:
            raise ValueError("bad pool arguments")

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_pool_delete(self._h)
            self._h = None

    def seq_create(self) -> int:
        out = np.zeros(1, np.int32)
        _check(lib().orc_seq_create(self._h, _p32(out)), "seq_create")
        return int(out[0])

    def seq_fork(self, parent: int) -> int:
        out = np.zeros(1, np.int32)
        _check(lib().orc_seq_fork(self._h, parent, _p32(out)), "seq_fork")
        return int(out[0])

    def seq_free(self, seq: int) -> None:
        _check(lib().orc_seq_free(self._h, seq), "seq_free")

    def seq_adopt(self, blocks: Sequence[int], length: int) -> int:
        """New sequence over the given (allocated) blocks, each gaining an owner."""
        b = np.ascontiguousarray(blocks, dtype=np.int32)
        out = np.zeros(1, np.int32)
        _check(lib().orc_seq_adopt(self._h, _p32(b) if len(b) else None, len(b), int(length), _p32(out)),
               "seq_adopt")
        return int(out[0])

    def block_retain(self, p: int) -> None:
        _check(lib().orc_block_retain(self._h, int(p)), "block_retain")

    def block_release(self, p: int) -> None:
        _check(lib().orc_block_release(self._h, int(p)), "block_release")

    def append(self, seq_ids: Sequence[int], n_new: Sequence[int]):
        """Returns (slot_mapping int32[sum n_new], cow_pairs int32[n_cow, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        nn = np.ascontiguousarray(n_new, dtype=np.int32)
        total = int(nn.sum()) if len(nn) else 0
        slots = np.zeros(max(total, 1), np.int32)
        pairs = np.zeros((max(len(ids), 1), 2), np.int32)
        ncow = np.zeros(1, np.int32)
        _check(lib().orc_append(self._h, _p32(ids), _p32(nn), len(ids), _p32(slots), _p32(pairs), _p32(ncow)),
               "append")
        return slots[:total].copy(), pairs[: int(ncow[0])].copy()

    def seq_len(self, seq: int) -> int:
        return int(lib().orc_seq_len(self._h, seq))

    def table(self, seq: int) -> np.ndarray:
        n = lib().orc_seq_table(self._h, seq, None, 0)
        if n < 0:
            raise OracleError(1, "table")
        out = np.zeros(max(n, 1), np.int32)
        lib().orc_seq_table(self._h, seq, _p32(out), n)
        return out[:n].copy()

    def refcounts(self) -> np.ndarray:
        out = np.zeros(self.num_blocks, np.int32)
        lib().orc_refcounts(self._h, _p32(out))
        return out

    def free_count(self) -> int:
        return int(lib().orc_free_count(self._h))

    def free_list(self) -> np.ndarray:
        out = np.zeros(self.num_blocks, np.int32)
        n = lib().orc_free_list(self._h, _p32(out))
        return out[:n].copy()

    def swap_out(self, seq: int, host_slots: Sequence[int]) -> np.ndarray:
        """Bookkeeping of a swap-out; returns the block ids copied (table order)."""
        hs = np.ascontiguousarray(host_slots, dtype=np.int64)
        ids = np.zeros(max(len(hs), 1), np.int32)
        _check(lib().orc_swap_out(self._h, seq, _p64(hs), _p32(ids)), "swap_out")
        return ids[: len(hs)].copy()

    def swap_in(self, seq: int, n: int):
        """Bookkeeping of a swap-in; returns (new block ids, host slots)."""
        ids = np.zeros(max(n, 1), np.int32)
        hs = np.zeros(max(n, 1), np.int64)
        _check(lib().orc_swap_in(self._h, seq, _p32(ids), _p64(hs)), "swap_in")
        return ids[:n].copy(), hs[:n].copy()

    def tables(self, seq_ids: Sequence[int], W: int):
        """Padded [n, W] int32 tables (pad 0) and int32 lengths."""
        t = np.zeros((len(seq_ids), W), np.int32)
        lens = np.zeros(len(seq_ids), np.int32)
        for i, s in enumerate(seq_ids):
            tb = self.table(s)
            t[i, : len(tb)] = tb
            lens[i] = self.seq_len(s)
        return t, lens


def _geo(g):
    return (g.L, g.H_kv, g.d_head, g.block_size, DTYPE_CODE[g.dtype], g.num_blocks)


def q_dtype(g) -> str:
    """Element type of the activations (q, out, new keys/values) around a pool:
    bfloat16 for an FP8 pool, the pool's own type otherwise."""
    return "bf16" if g.dtype == "e4m3" else g.dtype


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at 448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode(_vp(x), x.size, _vp(out))
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of E4M3 codes."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode(_vp(c), c.size, _vp(out))
    return out


def write_slots(g, layer: int, k_new: np.ndarray, v_new: np.ndarray, slot_mapping: np.ndarray,
                k_pool: np.ndarray, v_pool: np.ndarray, k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """Write new keys/values at their slots.  For an FP8 pool k_new/v_new are bf16
    (uint16 storage) and are quantised with the pool scales; otherwise bytes move."""
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    if g.dtype == "e4m3":
        _check(lib().orc_write_slots_e4m3(g.L, g.H_kv, g.d_head, g.block_size, g.num_blocks, layer, _vp(k_new),
                                          _vp(v_new), _p32(sm), len(sm), float(k_scale), float(v_scale),
                                          _vp(k_pool), _vp(v_pool)), "write_slots_e4m3")
        return
    _check(lib().orc_write_slots(*_geo(g), layer, _vp(k_new), _vp(v_new), _p32(sm), len(sm), _vp(k_pool),
                                 _vp(v_pool)), "write_slots")


def copy_blocks(g, pairs: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray) -> None:
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    _check(lib().orc_copy_blocks(*_geo(g), _p32(pr), len(pr), _vp(k_pool), _vp(v_pool)), "copy_blocks")


def swap_out_data(g, block_ids, host_slots, k_pool, v_pool, host) -> None:
    ids = np.ascontiguousarray(block_ids, dtype=np.int32)
    hs = np.ascontiguousarray(host_slots, dtype=np.int64)
    _check(lib().orc_swap_out_data(*_geo(g), _p32(ids), _p64(hs), len(ids), _vp(k_pool), _vp(v_pool), _vp(host)),
           "swap_out_data")


def swap_in_data(g, new_ids, host_slots, host, k_pool, v_pool) -> None:
    ids = np.ascontiguousarray(new_ids, dtype=np.int32)
    hs = np.ascontiguousarray(host_slots, dtype=np.int64)
    _check(lib().orc_swap_in_data(*_geo(g), _p32(ids), _p64(hs), len(ids), _vp(host), _vp(k_pool), _vp(v_pool)),
           "swap_in_data")


def decode_attention(g, layer: int, q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, tables: np.ndarray,
                     seq_lens: np.ndarray, scale: float, n_threads: int = 0, k_scale: float = 1.0,
                     v_scale: float = 1.0) -> np.ndarray:
    """Plain softmax attention in float64; q is [n_seq][H_q][d] raw storage of
    ``q_dtype(g)``; stored keys/values are read as scale * element."""
    q = np.ascontiguousarray(q)
    tb = np.ascontiguousarray(tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    n_seq = len(sl)
    W = tb.shape[1] if tb.ndim == 2 else 0
    out = np.zeros((n_seq, g.H_q, g.d_head), np.float64)
    code = lib().orc_decode_attention(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, DTYPE_CODE[g.dtype],
                                      g.num_blocks, layer, _vp(q), DTYPE_CODE[q_dtype(g)], _vp(k_pool),
                                      _vp(v_pool), float(k_scale), float(v_scale), _p32(tb), W,
                                      _p32(sl), n_seq, float(scale),
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(n_threads))
    _check(code, "decode_attention")
    return out


def prefill_attention(g, layer: int, q: np.ndarray, q_offsets: np.ndarray, k_pool: np.ndarray,
                      v_pool: np.ndarray, tables: np.ndarray, seq_lens: np.ndarray, scale: float,
                      n_threads: int = 0, k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Chunked-prefill attention in float64; q is [n_tok][H_q][d] raw storage, the
    chunk of sequence s is rows q_offsets[s]..q_offsets[s+1] (its last tokens)."""
    q = np.ascontiguousarray(q)
    qo = np.ascontiguousarray(q_offsets, dtype=np.int32)
    tb = np.ascontiguousarray(tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    n_seq = len(sl)
    W = tb.shape[1] if tb.ndim == 2 else 0
    out = np.zeros((int(qo[-1]), g.H_q, g.d_head), np.float64)
    code = lib().orc_prefill_attention(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, DTYPE_CODE[g.dtype],
                                       g.num_blocks, layer, _vp(q), DTYPE_CODE[q_dtype(g)], _p32(qo), _vp(k_pool),
                                       _vp(v_pool), float(k_scale), float(v_scale), _p32(tb), W,
                                       _p32(sl), n_seq, float(scale),
                                       out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(n_threads))
    _check(code, "prefill_attention")
    return out


def hardware_threads() -> int:
    return int(lib().orc_hardware_threads())
