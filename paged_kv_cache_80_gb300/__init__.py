"""Python binding of libpkv (the paged KV cache hot path for GB300).

Argument marshalling only: every function below calls the C entry point of the
same name in ``libpkv.so`` (declared in ``include/pkv.h``).  Device buffers are
torch CUDA tensors (their data pointers are passed), host control-plane arrays
are numpy arrays, and streams default to torch's current stream.  There is no
fallback: if the library is not built, or a buffer is on the wrong device, the
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Union

import numpy as np

__all__ = [
    "PkvError", "Geometry", "Pool", "library_path", "F32", "F16", "BF16",
    "pkv_version", "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_geometry", "pkv_seq_create", "pkv_seq_fork",
    "pkv_seq_free", "pkv_seq_len", "pkv_plan_append", "pkv_export_tables", "pkv_refcounts", "pkv_free_list",
    "pkv_append_kv", "pkv_decode_workspace_size", "pkv_decode_attention", "pkv_decode_attention_noalloc",
    "pkv_decode_step", "pkv_decode_step_host", "pkv_step_plan", "pkv_step_launch", "pkv_step_launch_host",
    "StepLauncher", "PackedStepLauncher",
    "pkv_prefill_attention",
    "pkv_copy_blocks", "pkv_swap_out",
    "pkv_swap_in", "pkv_swap_in_layers", "pkv_seq_host_slots", "pkv_seq_residency", "TIER_HBM", "TIER_HOST", "TIER_RELOADING", "pkv_pool_set_swap_engine", "pkv_pool_set_prefix_sharing", "pkv_step_meta_ints", "pkv_check_device_error", "pkv_launch_count",
    "pkv_selftest_bounded_wait", "pkv_device_code_version", "pkv_pool_set_kv_scales", "pkv_pool_kv_scales",
    "PrefixStats", "pkv_prefix_cache_create", "pkv_prefix_cache_destroy", "pkv_prefix_match", "pkv_prefix_attach",
    "pkv_prefix_insert", "pkv_prefix_release", "pkv_prefix_evict", "pkv_prefix_get_stats", "pkv_prefix_export",
    "SimConfig", "SimResult", "SIM_POLICIES", "pkv_sim_run",
]

F32, F16, BF16, E4M3 = 0, 1, 2, 3
DTYPES = {"f32": F32, "f16": F16, "bf16": BF16, "e4m3": E4M3}
_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "libpkv.so")


class PkvError(RuntimeError):
    def __init__(self, status: int, name: str, message: str, where: str):
        super().__init__(f"{where}: {name}: {message}")
        self.status = status
        self.name = name


class Geometry(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("d_head", ctypes.c_int32), ("block_size", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64)]


class PrefixStats(ctypes.Structure):
    _fields_ = [("nodes", ctypes.c_int64), ("blocks", ctypes.c_int64), ("pinned_nodes", ctypes.c_int64),
                ("dormant_leaves", ctypes.c_int64), ("prompt_tokens", ctypes.c_int64),
                ("matched_tokens", ctypes.c_int64)]


class SimConfig(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("max_context", ctypes.c_int32), ("watermark", ctypes.c_double),
                ("recompute_steps", ctypes.c_int32)]


class SimResult(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("charged_steps", ctypes.c_int64), ("preemptions", ctypes.c_int64),
                ("completed", ctypes.c_int64), ("max_running", ctypes.c_int64), ("mean_running", ctypes.c_double)]


SIM_POLICIES = {"reserve_max": 0, "reserve_declared": 1, "paged": 2}

_lib = None


def _L():
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        P32, P64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
        sig = {
            "pkv_version": ([], ctypes.c_int),
            "pkv_last_error_message": ([], ctypes.c_char_p),
            "pkv_status_name": ([ctypes.c_int], ctypes.c_char_p),
            "pkv_pool_create": ([ctypes.POINTER(Geometry), P32, ctypes.POINTER(vp)], ctypes.c_int),
            "pkv_pool_destroy": ([vp], ctypes.c_int),
            "pkv_pool_geometry": ([vp, ctypes.POINTER(Geometry)], ctypes.c_int),
            "pkv_seq_create": ([vp, P32], ctypes.c_int),
            "pkv_seq_fork": ([vp, i32, P32], ctypes.c_int),
            "pkv_seq_free": ([vp, i32], ctypes.c_int),
            "pkv_seq_len": ([vp, i32, P64], ctypes.c_int),
            "pkv_plan_append": ([vp, P32, P32, i32, P32, P32, P32], ctypes.c_int),
            "pkv_export_tables": ([vp, P32, i32, P32, i32, P32], ctypes.c_int),
            "pkv_refcounts": ([vp, P32], ctypes.c_int),
            "pkv_free_list": ([vp, P32, P64], ctypes.c_int),
            "pkv_append_kv": ([vp, i32, vp, vp, vp, i32, vp, vp, vp], ctypes.c_int),
            "pkv_decode_workspace_size": ([vp, i32, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
            "pkv_decode_attention": ([vp, i32, vp, vp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp, ctypes.c_size_t,
                                      vp], ctypes.c_int),
            "pkv_decode_attention_noalloc": ([vp, i32, vp, vp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp],
                                             ctypes.c_int),
            "pkv_copy_blocks": ([vp, P32, i32, vp, vp, vp], ctypes.c_int),
            "pkv_prefill_attention": ([vp, i32, vp, vp, i32, i32, vp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp],
                                      ctypes.c_int),
            "pkv_decode_step": ([vp, i32, vp, i32, i32, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp,
                                 ctypes.c_size_t, vp, vp, vp], ctypes.c_int),
            "pkv_decode_step_host": ([vp, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                      vp, vp, vp, ctypes.c_size_t, vp, vp, vp], ctypes.c_int),
            "pkv_step_plan": ([vp, vp, i32, i32, vp, vp, P32], ctypes.c_int),
            "pkv_step_launch": ([vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp,
                                 ctypes.c_size_t, vp, vp, vp], ctypes.c_int),
            "pkv_step_launch_host": ([vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp, vp, vp], ctypes.c_int),
            "pkv_step_launch_packed": ([vp, i32, i32, i32, vp, i32, vp, vp, ctypes.c_size_t, ctypes.c_size_t,
                                        ctypes.c_size_t, ctypes.c_size_t, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp,
                                        ctypes.c_size_t, vp, vp, vp], ctypes.c_int),
            "pkv_swap_out": ([vp, i32, vp, vp, vp, i64, P64, i32, P32, vp], ctypes.c_int),
            "pkv_swap_in": ([vp, i32, vp, i64, i32, vp, vp, P32, vp], ctypes.c_int),
            "pkv_seq_host_slots": ([vp, i32, P64, i32, P32], ctypes.c_int),
            "pkv_seq_residency": ([vp, i32, P32], ctypes.c_int),
            "pkv_swap_in_layers": ([vp, i32, vp, i64, i32, i32, i32, vp, vp, P32, vp], ctypes.c_int),
            "pkv_pool_set_swap_engine": ([vp, i32], ctypes.c_int),
            "pkv_pool_set_prefix_sharing": ([vp, i32, i32, i32], ctypes.c_int),
            "pkv_step_meta_ints": ([vp, i32, i32, P64], ctypes.c_int),
            "pkv_pool_set_kv_scales": ([vp, ctypes.c_float, ctypes.c_float], ctypes.c_int),
            "pkv_pool_kv_scales": ([vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)], ctypes.c_int),
            "pkv_check_device_error": ([vp, P32, P64], ctypes.c_int),
            "pkv_launch_count": ([], ctypes.c_uint64),
            "pkv_device_code_version": ([P32, P32], ctypes.c_int),
            "pkv_selftest_bounded_wait": ([i64, vp], ctypes.c_int),
            "pkv_prefix_cache_create": ([vp, ctypes.POINTER(vp)], ctypes.c_int),
            "pkv_prefix_cache_destroy": ([vp], ctypes.c_int),
            "pkv_prefix_match": ([vp, P32, i64, P64, P32], ctypes.c_int),
            "pkv_prefix_attach": ([vp, P32, i64, P32, P64], ctypes.c_int),
            "pkv_prefix_insert": ([vp, i32, P32, i64], ctypes.c_int),
            "pkv_prefix_release": ([vp, i32], ctypes.c_int),
            "pkv_prefix_evict": ([vp, i64, P64], ctypes.c_int),
            "pkv_prefix_get_stats": ([vp, ctypes.POINTER(PrefixStats)], ctypes.c_int),
            "pkv_prefix_export": ([vp, P64, P32, P32, i64, i64], ctypes.c_int),
            "pkv_sim_run": ([vp, ctypes.POINTER(SimConfig), P32, P32, P32, i32, ctypes.POINTER(SimResult)],
                            ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        L = _L()
        raise PkvError(rc, L.pkv_status_name(rc).decode(), L.pkv_last_error_message().decode(), where)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _p64(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _a(a: np.ndarray) -> int:
    """Address of a contiguous numpy array, for parameters declared as void pointers (the
    per-step calls: cheaper than building a typed ctypes pointer)."""
    return a.ctypes.data


def _dev(t, what: str) -> int:
    """Device pointer of a CUDA tensor (raises for anything else)."""
    if not hasattr(t, "is_cuda") or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _host_ptr(t, what: str) -> int:
    """Address of a host buffer: a CPU torch tensor (pinned for kernel access) or numpy array."""
    if isinstance(t, np.ndarray):
        if not t.flags.c_contiguous:
            raise ValueError(f"{what} must be contiguous")
        return t.ctypes.data
    if hasattr(t, "is_cuda") and not t.is_cuda:
        if not t.is_contiguous():
            raise ValueError(f"{what} must be contiguous")
        return t.data_ptr()
    raise TypeError(f"{what} must be a host buffer")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Pool:
    """Owner of a pkv_pool handle (destroyed with the object)."""

    def __init__(self, handle: ctypes.c_void_p, geometry: Geometry):
        self.handle = handle
        self.geometry = geometry
        self._meta_ints = {}  # (n, W) -> step metadata int32 count (cleared when sharing changes)

    @property
    def _as_parameter_(self):
        return self.handle

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.pkv_pool_destroy(h)
            self.handle = None


PoolLike = Union[Pool, ctypes.c_void_p]


def _h(pool: PoolLike):
    return pool.handle if isinstance(pool, Pool) else pool


def _nbytes(t) -> int:
    """Size in bytes of a numpy array or torch tensor."""
    return int(t.nbytes) if isinstance(t, np.ndarray) else t.numel() * t.element_size()


def pkv_step_meta_ints(pool: PoolLike, n: int, W: int) -> int:
    """int32 count of one decode step's metadata (n*(W+2) with prefix sharing off)."""
    if isinstance(pool, Pool):
        v = pool._meta_ints.get((n, W))
        if v is not None:
            return v
    out = ctypes.c_int64()
    _check(_L().pkv_step_meta_ints(_h(pool), int(n), int(W), ctypes.byref(out)), "pkv_step_meta_ints")
    if isinstance(pool, Pool):
        pool._meta_ints[(n, W)] = out.value
    return out.value


def pkv_pool_set_prefix_sharing(pool: PoolLike, min_members: int, min_blocks: int = 1, target_ctas: int = 0) -> None:
    """Decode steps attend to blocks shared by runs of batch rows once per run (0 turns it off)."""
    _check(_L().pkv_pool_set_prefix_sharing(_h(pool), int(min_members), int(min_blocks), int(target_ctas)),
           "pkv_pool_set_prefix_sharing")
    if isinstance(pool, Pool):
        pool._meta_ints.clear()


def _step_bytes(pool: PoolLike, n: int, W: int):
    """Bytes a decode step of n sequences reads or writes in each buffer: metadata
    (pkv_step_meta_ints int32), q / out rows (n*H_q*d_head activations), k_new / v_new rows
    (n*H_kv*d_head activations; activations are bf16 around an FP8 pool)."""
    g = pool.geometry if isinstance(pool, Pool) else pkv_pool_geometry(pool)
    ab = {F32: 4, F16: 2, BF16: 2, E4M3: 2}[g.dtype]
    return 4 * pkv_step_meta_ints(pool, n, W), ab * n * g.H_q * g.d_head, ab * n * g.H_kv * g.d_head


def _require_bytes(*bufs):
    """Raise ValueError for the first (buffer, bytes needed, name) whose buffer is smaller:
    the library copies fixed byte counts into and out of these buffers and cannot see
    their sizes."""
    for t, need, what in bufs:
        have = _nbytes(t)
        if have < need:
            raise ValueError(f"{what} holds {have} bytes; this step needs {need}")


# ------------------------------------------------------------------ library


def pkv_version() -> int:
    return _L().pkv_version()


# ------------------------------------------------------------------ control plane


def pkv_pool_create(L: int, H_q: int, H_kv: int, d_head: int, block_size: int, dtype: Union[str, int],
                    num_blocks: int, initial_free_order: Optional[np.ndarray] = None) -> Pool:
    g = Geometry(L, H_q, H_kv, d_head, block_size, DTYPES.get(dtype, dtype), num_blocks)
    fo = None
    if initial_free_order is not None:
        fo_arr = _i32(initial_free_order)
        if fo_arr.size != num_blocks:
            raise ValueError("initial_free_order must have num_blocks entries")
        fo = _p32(fo_arr)
    h = ctypes.c_void_p()
    _check(_L().pkv_pool_create(ctypes.byref(g), fo, ctypes.byref(h)), "pkv_pool_create")
    return Pool(h, g)


def pkv_pool_destroy(pool: Pool) -> None:
    _check(_L().pkv_pool_destroy(_h(pool)), "pkv_pool_destroy")
    if isinstance(pool, Pool):
        pool.handle = None


def pkv_pool_geometry(pool: PoolLike) -> Geometry:
    g = Geometry()
    _check(_L().pkv_pool_geometry(_h(pool), ctypes.byref(g)), "pkv_pool_geometry")
    return g


def pkv_seq_create(pool: PoolLike) -> int:
    out = ctypes.c_int32()
    _check(_L().pkv_seq_create(_h(pool), ctypes.byref(out)), "pkv_seq_create")
    return out.value


def pkv_seq_fork(pool: PoolLike, parent: int) -> int:
    out = ctypes.c_int32()
    _check(_L().pkv_seq_fork(_h(pool), parent, ctypes.byref(out)), "pkv_seq_fork")
    return out.value


def pkv_seq_free(pool: PoolLike, seq: int) -> None:
    _check(_L().pkv_seq_free(_h(pool), seq), "pkv_seq_free")


def pkv_seq_len(pool: PoolLike, seq: int) -> int:
    out = ctypes.c_int64()
    _check(_L().pkv_seq_len(_h(pool), seq, ctypes.byref(out)), "pkv_seq_len")
    return out.value


def pkv_plan_append(pool: PoolLike, seq_ids: Sequence[int], n_new: Sequence[int]):
    """Returns (slot_mapping int32[sum n_new], cow_pairs int32[n_cow, 2])."""
    ids, nn = _i32(seq_ids), _i32(n_new)
    if ids.shape != nn.shape:
        raise ValueError("seq_ids and n_new differ in length")
    total = int(nn.sum()) if nn.size else 0
    slots = np.zeros(max(total, 1), np.int32)
    pairs = np.zeros((max(ids.size, 1), 2), np.int32)
    ncow = ctypes.c_int32()
    _check(_L().pkv_plan_append(_h(pool), _p32(ids), _p32(nn), ids.size, _p32(slots), _p32(pairs),
                                ctypes.byref(ncow)), "pkv_plan_append")
    return slots[:total], pairs[: ncow.value]


def pkv_export_tables(pool: PoolLike, seq_ids: Sequence[int], W: int, tables: Optional[np.ndarray] = None,
                      seq_lens: Optional[np.ndarray] = None):
    """Returns (tables int32[n, W], seq_lens int32[n]); fills the given arrays if passed."""
    ids = _i32(seq_ids)
    if tables is None:
        tables = np.zeros((ids.size, max(W, 1)), np.int32)
    if seq_lens is None:
        seq_lens = np.zeros(max(ids.size, 1), np.int32)
    _check(_L().pkv_export_tables(_h(pool), _p32(ids), ids.size, _p32(tables), W, _p32(seq_lens)),
           "pkv_export_tables")
    return tables[: ids.size, :W], seq_lens[: ids.size]


def pkv_refcounts(pool: PoolLike) -> np.ndarray:
    g = pkv_pool_geometry(pool)
    out = np.zeros(g.num_blocks, np.int32)
    _check(_L().pkv_refcounts(_h(pool), _p32(out)), "pkv_refcounts")
    return out


def pkv_free_list(pool: PoolLike) -> np.ndarray:
    g = pkv_pool_geometry(pool)
    out = np.zeros(g.num_blocks, np.int32)
    n = ctypes.c_int64()
    _check(_L().pkv_free_list(_h(pool), _p32(out), ctypes.byref(n)), "pkv_free_list")
    return out[: n.value]


def pkv_pool_set_swap_engine(pool: PoolLike, engine: int) -> None:
    _check(_L().pkv_pool_set_swap_engine(_h(pool), engine), "pkv_pool_set_swap_engine")


def pkv_pool_set_kv_scales(pool: PoolLike, k_scale: float, v_scale: float) -> None:
    """FP8 pools: stored keys read as code * k_scale, values as code * v_scale."""
    _check(_L().pkv_pool_set_kv_scales(_h(pool), k_scale, v_scale), "pkv_pool_set_kv_scales")


def pkv_pool_kv_scales(pool: PoolLike):
    k, v = ctypes.c_float(), ctypes.c_float()
    _check(_L().pkv_pool_kv_scales(_h(pool), ctypes.byref(k), ctypes.byref(v)), "pkv_pool_kv_scales")
    return k.value, v.value


TIER_HBM, TIER_HOST, TIER_RELOADING = 0, 1, 2


def pkv_seq_residency(pool: PoolLike, seq: int) -> int:
    out = ctypes.c_int32()
    _check(_L().pkv_seq_residency(_h(pool), seq, ctypes.byref(out)), "pkv_seq_residency")
    return out.value


def pkv_seq_host_slots(pool: PoolLike, seq: int) -> np.ndarray:
    n = ctypes.c_int32()
    _check(_L().pkv_seq_host_slots(_h(pool), seq, None, 0, ctypes.byref(n)), "pkv_seq_host_slots")
    out = np.zeros(max(n.value, 1), np.int64)
    _check(_L().pkv_seq_host_slots(_h(pool), seq, _p64(out), n.value, ctypes.byref(n)), "pkv_seq_host_slots")
    return out[: n.value]


# ------------------------------------------------------------------ data plane


def pkv_append_kv(pool: PoolLike, layer: int, k_new, v_new, slot_mapping, k_pool, v_pool, stream=None) -> None:
    n_tok = int(slot_mapping.numel())
    _check(_L().pkv_append_kv(_h(pool), layer, _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                              _dev(slot_mapping, "slot_mapping"), n_tok, _dev(k_pool, "k_pool"),
                              _dev(v_pool, "v_pool"), _stream(stream)), "pkv_append_kv")


def pkv_decode_workspace_size(pool: PoolLike, n_seq: int) -> int:
    out = ctypes.c_size_t()
    _check(_L().pkv_decode_workspace_size(_h(pool), n_seq, ctypes.byref(out)), "pkv_decode_workspace_size")
    return out.value


def pkv_decode_attention(pool: PoolLike, layer: int, q, k_pool, v_pool, block_tables, seq_lens, scale: float, out,
                         workspace, stream=None) -> None:
    n_seq = int(seq_lens.numel())
    W = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    _check(_L().pkv_decode_attention(_h(pool), layer, _dev(q, "q"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                                     _dev(block_tables, "block_tables"), W, _dev(seq_lens, "seq_lens"), n_seq,
                                     float(scale), _dev(out, "out"), _dev(workspace, "workspace"),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "pkv_decode_attention")


def pkv_decode_attention_noalloc(pool: PoolLike, layer: int, q, k_pool, v_pool, block_tables, seq_lens,
                                 scale: float, out, stream=None) -> None:
    """Decode attention without a workspace: for callers that cannot allocate device
    memory (the library's own static 24 MiB scratch is used instead)."""
    n_seq = int(seq_lens.numel())
    W = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    _check(_L().pkv_decode_attention_noalloc(_h(pool), layer, _dev(q, "q"), _dev(k_pool, "k_pool"),
                                             _dev(v_pool, "v_pool"), _dev(block_tables, "block_tables"), W,
                                             _dev(seq_lens, "seq_lens"), n_seq, float(scale), _dev(out, "out"),
                                             _stream(stream)), "pkv_decode_attention_noalloc")


def pkv_decode_step(pool: PoolLike, layer: int, seq_ids, W: int, q, k_new, v_new, k_pool, v_pool, scale: float,
                    out, meta_host, meta_dev, workspace, attn_events=None, stream=None) -> None:
    """One decode step (plan, CoW copy, append, attend) for the sequences seq_ids.
    meta_host: pinned CPU int32 tensor, meta_dev: CUDA int32 tensor, each >= n*(W+2)."""
    ids = _i32(seq_ids)
    n = ids.size
    mb, qb, kb = _step_bytes(pool, n, W)
    _require_bytes((meta_host, mb, "meta_host"), (meta_dev, mb, "meta_dev"), (q, qb, "q"), (k_new, kb, "k_new"),
                   (v_new, kb, "v_new"), (out, qb, "out"))
    ev0, ev1 = _events(attn_events)
    _check(_L().pkv_decode_step(_h(pool), layer, _a(ids), n, W, _dev(q, "q"), _dev(k_new, "k_new"),
                                _dev(v_new, "v_new"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), float(scale),
                                _dev(out, "out"), _host_ptr(meta_host, "meta_host"), _dev(meta_dev, "meta_dev"),
                                _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), ev0, ev1,
                                _stream(stream)), "pkv_decode_step")


def pkv_decode_step_host(pool: PoolLike, layer: int, seq_ids, W: int, q_host, k_new_host, v_new_host, out_host,
                         q_dev, k_new_dev, v_new_dev, out_dev, k_pool, v_pool, scale: float, meta_host, meta_dev,
                         workspace, attn_events=None, stream=None) -> None:
    """pkv_decode_step with q / k_new / v_new read from, and out written to, host
    tensors (page-locked for asynchronous copies) through the *_dev staging tensors;
    synchronise the stream before reading out_host."""
    ids = _i32(seq_ids)
    n = ids.size
    mb, qb, kb = _step_bytes(pool, n, W)
    _require_bytes((meta_host, mb, "meta_host"), (meta_dev, mb, "meta_dev"), (q_host, qb, "q_host"),
                   (k_new_host, kb, "k_new_host"), (v_new_host, kb, "v_new_host"), (out_host, qb, "out_host"),
                   (q_dev, qb, "q_dev"), (k_new_dev, kb, "k_new_dev"), (v_new_dev, kb, "v_new_dev"),
                   (out_dev, qb, "out_dev"))
    ev0, ev1 = _events(attn_events)
    _check(_L().pkv_decode_step_host(_h(pool), layer, _a(ids), n, W, _host_ptr(q_host, "q_host"),
                                     _host_ptr(k_new_host, "k_new_host"), _host_ptr(v_new_host, "v_new_host"),
                                     _host_ptr(out_host, "out_host"), _dev(q_dev, "q_dev"), _dev(k_new_dev, "k_new_dev"),
                                     _dev(v_new_dev, "v_new_dev"), _dev(out_dev, "out_dev"), _dev(k_pool, "k_pool"),
                                     _dev(v_pool, "v_pool"), float(scale), _host_ptr(meta_host, "meta_host"),
                                     _dev(meta_dev, "meta_dev"), _dev(workspace, "workspace"),
                                     workspace.numel() * workspace.element_size(), ev0, ev1, _stream(stream)),
           "pkv_decode_step_host")


def pkv_step_plan(pool: PoolLike, seq_ids, W: int, meta_host) -> np.ndarray:
    """The host half of a decode step: plan one token per sequence into meta_host
    (pinned int32, >= n*(W+2)); returns the copy-on-write pairs [n_cow][2]."""
    ids = _i32(seq_ids)
    n = ids.size
    _require_bytes((meta_host, 4 * pkv_step_meta_ints(pool, n, W), "meta_host"))
    cows = np.zeros(max(2 * n, 2), np.int32)
    n_cow = ctypes.c_int32(0)
    _check(_L().pkv_step_plan(_h(pool), _a(ids), n, W, _host_ptr(meta_host, "meta_host"), _a(cows),
                              ctypes.byref(n_cow)), "pkv_step_plan")
    return cows[: 2 * n_cow.value].reshape(-1, 2)


def _events(attn_events):
    if attn_events is None:
        return None, None
    for ev in attn_events:
        if not ev.cuda_event:  # torch creates its CUDA event at the first record
            ev.record()
    return attn_events[0].cuda_event, attn_events[1].cuda_event


def pkv_step_launch(pool: PoolLike, layer: int, n: int, W: int, cow_pairs, q, k_new, v_new, k_pool, v_pool,
                    scale: float, out, meta_host, meta_dev, workspace, attn_events=None, stream=None) -> None:
    """The device half of a decode step planned by pkv_step_plan (device q / k_new / v_new / out)."""
    mb, qb, kb = _step_bytes(pool, n, W)
    _require_bytes((meta_host, mb, "meta_host"), (meta_dev, mb, "meta_dev"), (q, qb, "q"), (k_new, kb, "k_new"),
                   (v_new, kb, "v_new"), (out, qb, "out"))
    cp = _i32(cow_pairs).reshape(-1)
    ev0, ev1 = _events(attn_events)
    _check(_L().pkv_step_launch(_h(pool), layer, n, W, _a(cp), cp.size // 2, _dev(q, "q"), _dev(k_new, "k_new"),
                                _dev(v_new, "v_new"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), float(scale),
                                _dev(out, "out"), _host_ptr(meta_host, "meta_host"), _dev(meta_dev, "meta_dev"),
                                _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), ev0, ev1,
                                _stream(stream)), "pkv_step_launch")


def pkv_step_launch_host(pool: PoolLike, layer: int, n: int, W: int, cow_pairs, q_host, k_new_host, v_new_host,
                         out_host, q_dev, k_new_dev, v_new_dev, out_dev, k_pool, v_pool, scale: float, meta_host,
                         meta_dev, workspace, attn_events=None, stream=None) -> None:
    """pkv_step_launch with host input and result tensors (page-locked) copied inside the call."""
    mb, qb, kb = _step_bytes(pool, n, W)
    _require_bytes((meta_host, mb, "meta_host"), (meta_dev, mb, "meta_dev"), (q_host, qb, "q_host"),
                   (k_new_host, kb, "k_new_host"), (v_new_host, kb, "v_new_host"), (out_host, qb, "out_host"),
                   (q_dev, qb, "q_dev"), (k_new_dev, kb, "k_new_dev"), (v_new_dev, kb, "v_new_dev"),
                   (out_dev, qb, "out_dev"))
    cp = _i32(cow_pairs).reshape(-1)
    ev0, ev1 = _events(attn_events)
    _check(_L().pkv_step_launch_host(_h(pool), layer, n, W, _a(cp), cp.size // 2, _host_ptr(q_host, "q_host"),
                                     _host_ptr(k_new_host, "k_new_host"), _host_ptr(v_new_host, "v_new_host"),
                                     _host_ptr(out_host, "out_host"), _dev(q_dev, "q_dev"), _dev(k_new_dev, "k_new_dev"),
                                     _dev(v_new_dev, "v_new_dev"), _dev(out_dev, "out_dev"), _dev(k_pool, "k_pool"),
                                     _dev(v_pool, "v_pool"), float(scale), _host_ptr(meta_host, "meta_host"),
                                     _dev(meta_dev, "meta_dev"), _dev(workspace, "workspace"),
                                     workspace.numel() * workspace.element_size(), ev0, ev1, _stream(stream)),
           "pkv_step_launch_host")


class StepLauncher:
    """pkv_step_launch_host with the buffers that stay the same from step to step bound once:
    the device staging tensors (q, k_new, v_new, out: their leading rows are used), the pools,
    the workspace, the scale and the stream.  The stream is fixed at construction (torch's
    current stream then, when None): calls made later under another torch stream still
    launch on it.  Each call then takes only what changes per step, so a serving loop's host
    side is shorter; the result is the same as pkv_step_launch_host's.  The launcher holds
    references to the pool and every bound buffer, so none is freed while it lives, and each
    call checks that its host and metadata buffers hold what the step copies."""

    def __init__(self, pool: PoolLike, layer: int, q_dev, k_new_dev, v_new_dev, out_dev, k_pool, v_pool,
                 scale: float, workspace, stream=None):
        self._pool = pool
        self._layer = int(layer)
        g = pool.geometry if isinstance(pool, Pool) else pkv_pool_geometry(pool)
        ab = {F32: 4, F16: 2, BF16: 2, E4M3: 2}[g.dtype]
        self._row_q, self._row_k = ab * g.H_q * g.d_head, ab * g.H_kv * g.d_head
        # rows that every bound device buffer can take
        self._rows = min(_nbytes(q_dev) // self._row_q, _nbytes(k_new_dev) // self._row_k,
                         _nbytes(v_new_dev) // self._row_k, _nbytes(out_dev) // self._row_q)
        self._dev = (_dev(q_dev, "q_dev"), _dev(k_new_dev, "k_new_dev"), _dev(v_new_dev, "v_new_dev"),
                     _dev(out_dev, "out_dev"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"))
        self._scale = float(scale)
        self._ws = (_dev(workspace, "workspace"), workspace.numel() * workspace.element_size())
        self._stream = _stream(stream)
        self._f = _L().pkv_step_launch_host
        self._keep = (pool, q_dev, k_new_dev, v_new_dev, out_dev, k_pool, v_pool, workspace)  # keep them alive

    @property
    def stream(self) -> int:
        """The CUDA stream (as an integer handle) every call launches on."""
        return self._stream

    def __call__(self, n: int, W: int, cow_pairs, q_host, k_new_host, v_new_host, out_host, meta_host, meta_dev,
                 attn_events=None) -> None:
        if n > self._rows:
            raise ValueError(f"n = {n} exceeds the {self._rows} rows of the bound device buffers")
        mb, qb, kb = 4 * pkv_step_meta_ints(self._pool, n, W), n * self._row_q, n * self._row_k
        _require_bytes((meta_host, mb, "meta_host"), (meta_dev, mb, "meta_dev"), (q_host, qb, "q_host"),
                       (k_new_host, kb, "k_new_host"), (v_new_host, kb, "v_new_host"), (out_host, qb, "out_host"))
        cp = _i32(cow_pairs).reshape(-1)
        ev0, ev1 = _events(attn_events)
        q, k, v, o, kp, vp = self._dev
        _check(self._f(_h(self._pool), self._layer, n, W, _a(cp), cp.size // 2, _host_ptr(q_host, "q_host"),
                       _host_ptr(k_new_host, "k_new_host"), _host_ptr(v_new_host, "v_new_host"),
                       _host_ptr(out_host, "out_host"), q, k, v, o, kp, vp, self._scale,
                       _host_ptr(meta_host, "meta_host"), _dev(meta_dev, "meta_dev"), self._ws[0], self._ws[1], ev0,
                       ev1, self._stream), "pkv_step_launch_host")


class PackedStepLauncher:
    """pkv_step_launch_packed with the buffers that stay the same from step to step bound once:
    the device input staging `in_dev` (q, k_new, v_new at the offsets each call gives, one
    copy per step), the device result rows `out_dev`, the pools, the scale, the workspace
    and the stream (fixed at construction: torch's current stream then, when None).  Each call
    takes the page-locked host input buffer of the step (q at byte 0, k_new at off_k, v_new at
    off_v; `in_bytes` of it are copied), the host result buffer, the device metadata buffer
    and, unless the caller already queued the metadata copy, the host metadata.  The launcher
    holds references to the pool and every bound buffer."""

    def __init__(self, pool: PoolLike, layer: int, in_dev, out_dev, k_pool, v_pool, scale: float, workspace,
                 stream=None):
        self._pool = pool
        self._layer = int(layer)
        g = pool.geometry if isinstance(pool, Pool) else pkv_pool_geometry(pool)
        ab = {F32: 4, F16: 2, BF16: 2, E4M3: 2}[g.dtype]
        self._row_q, self._row_k = ab * g.H_q * g.d_head, ab * g.H_kv * g.d_head
        self._in_bytes = _nbytes(in_dev)
        self._rows = _nbytes(out_dev) // self._row_q
        self._dev = (_dev(in_dev, "in_dev"), _dev(out_dev, "out_dev"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"))
        self._scale = float(scale)
        self._ws = (_dev(workspace, "workspace"), workspace.numel() * workspace.element_size())
        self._stream = _stream(stream)
        self._f = _L().pkv_step_launch_packed
        self._keep = (pool, in_dev, out_dev, k_pool, v_pool, workspace)

    @property
    def stream(self) -> int:
        return self._stream

    def __call__(self, n: int, W: int, cow_pairs, in_host, off_k: int, off_v: int, in_bytes: int, out_host,
                 meta_dev=None, meta_host=None, off_meta: int = 0, attn_events=None) -> None:
        """One step; the metadata is either packed in in_host at off_meta (written there by
        pkv_step_plan; meta_dev and meta_host unused), or copied from meta_host to meta_dev by
        the call, or (meta_host None) already queued into meta_dev by the caller."""
        if n > self._rows:
            raise ValueError(f"n = {n} exceeds the {self._rows} rows of the bound out_dev")
        mb = 4 * pkv_step_meta_ints(self._pool, n, W)
        _require_bytes((in_host, in_bytes, "in_host"), (out_host, n * self._row_q, "out_host"))
        if in_bytes > self._in_bytes:
            raise ValueError(f"in_bytes = {in_bytes} exceeds the {self._in_bytes} bytes of the bound in_dev")
        if not off_meta:
            if meta_dev is None:
                raise ValueError("meta_dev is needed unless the metadata is packed (off_meta)")
            _require_bytes((meta_dev, mb, "meta_dev"))
            if meta_host is not None:
                _require_bytes((meta_host, mb, "meta_host"))
        cp = _i32(cow_pairs).reshape(-1)
        ev0, ev1 = _events(attn_events)
        ind, outd, kp, vp = self._dev
        _check(self._f(_h(self._pool), self._layer, n, W, _a(cp), cp.size // 2, _host_ptr(in_host, "in_host"), ind,
                       int(off_k), int(off_v), int(off_meta), int(in_bytes), _host_ptr(out_host, "out_host"), outd,
                       kp, vp, self._scale,
                       None if (off_meta or meta_host is None) else _host_ptr(meta_host, "meta_host"),
                       None if off_meta else _dev(meta_dev, "meta_dev"), self._ws[0], self._ws[1], ev0, ev1,
                       self._stream), "pkv_step_launch_packed")


def pkv_prefill_attention(pool: PoolLike, layer: int, q, q_offsets, max_q: int, k_pool, v_pool, block_tables,
                          seq_lens, scale: float, out, stream=None) -> None:
    """Chunked-prefill attention; q/out are [n_tok][H_q][d], q_offsets device int32 [n_seq+1]."""
    n_seq = int(seq_lens.numel())
    W = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    _check(_L().pkv_prefill_attention(_h(pool), layer, _dev(q, "q"), _dev(q_offsets, "q_offsets"), int(q.shape[0]),
                                      int(max_q), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                                      _dev(block_tables, "block_tables"), W, _dev(seq_lens, "seq_lens"), n_seq,
                                      float(scale), _dev(out, "out"), _stream(stream)), "pkv_prefill_attention")


def pkv_copy_blocks(pool: PoolLike, pairs, k_pool, v_pool, stream=None) -> None:
    pr = _i32(pairs).reshape(-1, 2)
    _check(_L().pkv_copy_blocks(_h(pool), _p32(pr), pr.shape[0], _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                                _stream(stream)), "pkv_copy_blocks")


def pkv_swap_out(pool: PoolLike, seq: int, k_pool, v_pool, host, host_frames: int, host_slots,
                 stream=None) -> np.ndarray:
    hs = _i64(host_slots)
    ids = np.zeros(max(hs.size, 1), np.int32)
    _check(_L().pkv_swap_out(_h(pool), seq, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), _host_ptr(host, "host"),
                             host_frames, _p64(hs), hs.size, _p32(ids), _stream(stream)), "pkv_swap_out")
    return ids[: hs.size]


def pkv_swap_in(pool: PoolLike, seq: int, host, host_frames: int, n: int, k_pool, v_pool,
                stream=None) -> np.ndarray:
    ids = np.zeros(max(n, 1), np.int32)
    _check(_L().pkv_swap_in(_h(pool), seq, _host_ptr(host, "host"), host_frames, n, _dev(k_pool, "k_pool"),
                            _dev(v_pool, "v_pool"), _p32(ids), _stream(stream)), "pkv_swap_in")
    return ids[:n]


def pkv_swap_in_layers(pool: PoolLike, seq: int, host, host_frames: int, n: int, layer_begin: int, layer_end: int,
                       k_pool, v_pool, stream=None) -> np.ndarray:
    """Reload layers [layer_begin, layer_end) of a swapped-out sequence (the first call, at layer
    0, allocates and remaps); returns the sequence's table."""
    ids = np.zeros(max(n, 1), np.int32)
    _check(_L().pkv_swap_in_layers(_h(pool), seq, _host_ptr(host, "host"), host_frames, n, layer_begin, layer_end,
                                   _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), _p32(ids), _stream(stream)),
           "pkv_swap_in_layers")
    return ids[:n]


def pkv_selftest_bounded_wait(timeout_ns: int, stream=None) -> None:
    _check(_L().pkv_selftest_bounded_wait(int(timeout_ns), _stream(stream)), "pkv_selftest_bounded_wait")


def pkv_launch_count() -> int:
    return int(_L().pkv_launch_count())


def pkv_device_code_version():
    """(binaryVersion, ptxVersion) of the library's device code as loaded on the current
    device (needs a GPU)."""
    b, p = ctypes.c_int32(), ctypes.c_int32()
    _check(_L().pkv_device_code_version(ctypes.byref(b), ctypes.byref(p)), "pkv_device_code_version")
    return b.value, p.value


def pkv_check_device_error(stream=None):
    """Synchronise the stream and read/clear the device error word.  Returns
    (code, detail); raises PkvError(DEVICE_CHECK) if a kernel recorded one."""
    code = ctypes.c_int32()
    detail = ctypes.c_int64()
    rc = _L().pkv_check_device_error(_stream(stream), ctypes.byref(code), ctypes.byref(detail))
    _check(rc, "pkv_check_device_error")
    return code.value, detail.value


# ------------------------------------------------------------------ radix prefix cache (host)


class PrefixCache:
    """Owner of a pkv_prefix_cache handle; keeps its pool alive and is destroyed first."""

    def __init__(self, handle: ctypes.c_void_p, pool: PoolLike):
        self.handle = handle
        self.pool = pool

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.pkv_prefix_cache_destroy(h)
            self.handle = None


def _c(cache) -> ctypes.c_void_p:
    return cache.handle if isinstance(cache, PrefixCache) else cache


def pkv_prefix_cache_create(pool: PoolLike) -> PrefixCache:
    h = ctypes.c_void_p()
    _check(_L().pkv_prefix_cache_create(_h(pool), ctypes.byref(h)), "pkv_prefix_cache_create")
    return PrefixCache(h, pool)


def pkv_prefix_cache_destroy(cache: PrefixCache) -> None:
    _check(_L().pkv_prefix_cache_destroy(_c(cache)), "pkv_prefix_cache_destroy")
    cache.handle = None


def pkv_prefix_match(cache, tokens):
    """(matched tokens, their blocks) for a prompt; changes nothing."""
    t = _i32(tokens)
    n = ctypes.c_int64()
    out = np.zeros(max(len(t), 1), np.int32)
    _check(_L().pkv_prefix_match(_c(cache), _p32(t), len(t), ctypes.byref(n), _p32(out)), "pkv_prefix_match")
    B = _pool_block_size(cache)
    return n.value, out[: n.value // B].copy()


def _pool_block_size(cache) -> int:
    return pkv_pool_geometry(cache.pool).block_size


def pkv_prefix_attach(cache, tokens):
    """Serve a prompt from the cache: (new sequence id, matched tokens)."""
    t = _i32(tokens)
    seq = ctypes.c_int32()
    n = ctypes.c_int64()
    _check(_L().pkv_prefix_attach(_c(cache), _p32(t), len(t), ctypes.byref(seq), ctypes.byref(n)),
           "pkv_prefix_attach")
    return seq.value, n.value


def pkv_prefix_insert(cache, seq: int, tokens) -> None:
    t = _i32(tokens)
    _check(_L().pkv_prefix_insert(_c(cache), seq, _p32(t), len(t)), "pkv_prefix_insert")


def pkv_prefix_release(cache, seq: int) -> None:
    _check(_L().pkv_prefix_release(_c(cache), seq), "pkv_prefix_release")


def pkv_prefix_evict(cache, target_free: int) -> int:
    n = ctypes.c_int64()
    _check(_L().pkv_prefix_evict(_c(cache), int(target_free), ctypes.byref(n)), "pkv_prefix_evict")
    return n.value


def pkv_prefix_get_stats(cache) -> PrefixStats:
    st = PrefixStats()
    _check(_L().pkv_prefix_get_stats(_c(cache), ctypes.byref(st)), "pkv_prefix_get_stats")
    return st


def pkv_prefix_export(cache):
    """Preorder rows (parent row, blocks, ref, last_access, serial, tokens, block ids)."""
    st = pkv_prefix_get_stats(cache)
    B = _pool_block_size(cache)
    nodes = np.zeros((max(st.nodes, 1), 5), np.int64)
    toks = np.zeros(max(st.blocks * B, 1), np.int32)
    blks = np.zeros(max(st.blocks, 1), np.int32)
    _check(_L().pkv_prefix_export(_c(cache), nodes.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _p32(toks),
                                  _p32(blks), st.nodes, st.blocks), "pkv_prefix_export")
    rows, off = [], 0
    for r in range(st.nodes):
        parent, nb, ref, last, serial = (int(x) for x in nodes[r])
        rows.append((parent, nb, ref, last, serial, toks[off * B:(off + nb) * B].tolist(), blks[off:off + nb].tolist()))
        off += nb
    return rows


# ------------------------------------------------------------------ admission simulator (host)


def pkv_sim_run(pool: PoolLike, policy: str, prompt, answer, declared=None, max_context: int = 1024,
                watermark: float = 0.0, recompute_steps: int = 4) -> dict:
    """Steps to serve a saturated queue under an admission policy (see pkv.h)."""
    cfg = SimConfig(SIM_POLICIES[policy], max_context, watermark, recompute_steps)
    p, a = _i32(prompt), _i32(answer)
    d = _i32(declared) if declared is not None else None
    res = SimResult()
    _check(_L().pkv_sim_run(_h(pool), ctypes.byref(cfg), _p32(p), _p32(a), _p32(d) if d is not None else None, len(p),
                            ctypes.byref(res)), "pkv_sim_run")
    return {k: getattr(res, k) for k, _ in SimResult._fields_}
