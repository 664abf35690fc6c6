"""Helpers shared by the GPU parity tests: one paged batch driven in lockstep
through the library (device) and the oracle (host)."""
from __future__ import annotations

import numpy as np

import oracle
import paged_kv_cache_80_gb300 as pkv
import workloads as W

NP_STORE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "e4m3": np.uint8}


def torch_dtype(dtype):
    import torch

    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8}[dtype]


def act(g) -> str:
    """Element type of q, out and new keys/values around the pool (bf16 for FP8)."""
    return oracle.q_dtype(g)


def to_dev(raw: np.ndarray, dtype: str, device="cuda"):
    import torch

    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(raw).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(raw)).to(device)


def to_raw(t, dtype: str) -> np.ndarray:
    import torch

    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_f64(t, dtype: str) -> np.ndarray:
    return W.to_float64(to_raw(t, dtype), dtype)


def check_attention(got: np.ndarray, ref: np.ndarray, dtype: str):
    """bf16/f16 storage: max-abs <= 2e-2 and mean-abs <= 2e-3; fp32: the largest
    error of each output vector <= 1e-5 of that vector's largest magnitude."""
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    if dtype == "f32":
        scale = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
        rel = err.max(axis=-1) / scale
        assert rel.max() <= 1e-5, f"relative error {rel.max():.3e}"
        return rel.max()
    assert err.max() <= 2e-2, f"max abs error {err.max():.3e}"
    assert err.mean() <= 2e-3, f"mean abs error {err.mean():.3e}"
    return err.max()


class PagedBatch:
    """A library pool on the device and an oracle pool on the host, advanced together."""

    def __init__(self, g: W.Geometry, free_order=None, seed: int = 0, host_pool: bool = True, device="cuda",
                 fill_device=None, kv_scales=(1.0, 1.0)):
        import torch

        self.g, self.seed, self.device = g, seed, device
        self.lib = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, free_order)
        self.k_scale, self.v_scale = (float(np.float32(kv_scales[0])), float(np.float32(kv_scales[1])))
        if g.dtype == "e4m3":
            pkv.pkv_pool_set_kv_scales(self.lib, self.k_scale, self.v_scale)
        self.orc = oracle.Pool(g.num_blocks, g.block_size, free_order)
        td = torch_dtype(g.dtype)
        if fill_device is None:
            self.kp = torch.zeros(g.pool_shape(), dtype=td, device=device)
            self.vp = torch.zeros(g.pool_shape(), dtype=td, device=device)
        else:
            self.kp, self.vp = fill_device
        self.hk = np.zeros(g.pool_shape(), NP_STORE[g.dtype]) if host_pool else None
        self.hv = np.zeros(g.pool_shape(), NP_STORE[g.dtype]) if host_pool else None
        self.ids = []
        self.n_cow = 0

    def new_seqs(self, n):
        a = [pkv.pkv_seq_create(self.lib) for _ in range(n)]
        b = [self.orc.seq_create() for _ in range(n)]
        assert a == b
        self.ids += a
        return a

    def fork(self, parent):
        a = pkv.pkv_seq_fork(self.lib, parent)
        assert a == self.orc.seq_fork(parent)
        self.ids.append(a)
        return a

    def free(self, seq):
        pkv.pkv_seq_free(self.lib, seq)
        self.orc.seq_free(seq)
        self.ids.remove(seq)

    def append(self, seq_ids, n_new, tag, layer=0, write_host=True, plan_only=False):
        """Plan on both sides (slots and CoW pairs must match), copy CoW blocks,
        then write fresh N(0,1) keys/values for the new tokens (unless plan_only:
        the pool's existing contents then stand for the tokens)."""
        import torch

        g = self.g
        slots, cows = pkv.pkv_plan_append(self.lib, seq_ids, n_new)
        oslots, ocows = self.orc.append(seq_ids, n_new)
        assert np.array_equal(slots, oslots) and np.array_equal(cows, ocows)
        if plan_only:
            assert len(cows) == 0
            return slots, cows
        if len(cows):
            pkv.pkv_copy_blocks(self.lib, cows, self.kp, self.vp)
            if write_host and self.hk is not None:
                oracle.copy_blocks(g, cows, self.hk, self.hv)
            self.n_cow += len(cows)
        if len(slots) == 0:
            return slots, cows
        lay = g.L if layer < 0 else 1
        shape = (lay, len(slots), g.H_kv, g.d_head) if layer < 0 else (len(slots), g.H_kv, g.d_head)
        a = act(g)
        k = W.normal(self.seed, f"k_{tag}", shape, a)
        v = W.normal(self.seed, f"v_{tag}", shape, a)
        pkv.pkv_append_kv(self.lib, layer, to_dev(k, a, self.device), to_dev(v, a, self.device),
                          torch.from_numpy(slots).to(self.device), self.kp, self.vp)
        if write_host and self.hk is not None:
            oracle.write_slots(g, layer, k, v, slots, self.hk, self.hv, self.k_scale, self.v_scale)
        return slots, cows

    def tables(self, seq_ids, W_=None):
        if W_ is None:
            W_ = max([len(self.orc.table(s)) for s in seq_ids] + [1])
        t1, l1 = pkv.pkv_export_tables(self.lib, seq_ids, W_)
        t2, l2 = self.orc.tables(seq_ids, W_)
        assert np.array_equal(t1, t2) and np.array_equal(l1, l2)
        return t1.copy(), l1.copy()

    def check_state(self):
        assert np.array_equal(pkv.pkv_refcounts(self.lib), self.orc.refcounts())
        assert np.array_equal(pkv.pkv_free_list(self.lib), self.orc.free_list())

    def check_pools_bitexact(self):
        assert np.array_equal(to_raw(self.kp, self.g.dtype), self.hk)
        assert np.array_equal(to_raw(self.vp, self.g.dtype), self.hv)

    def decode_gpu(self, seq_ids, q_raw, scale, layer=0, W_=None, tables=None, lens=None):
        import torch

        g = self.g
        if tables is None:
            tables, lens = self.tables(seq_ids, W_)
        out = torch.full((len(seq_ids), g.H_q, g.d_head), float("nan"), dtype=torch_dtype(act(g)),
                         device=self.device)
        ws = torch.empty(pkv.pkv_decode_workspace_size(self.lib, len(seq_ids)), dtype=torch.uint8,
                         device=self.device)
        pkv.pkv_decode_attention(self.lib, layer, to_dev(q_raw, act(g), self.device), self.kp, self.vp,
                                 torch.from_numpy(np.ascontiguousarray(tables)).to(self.device),
                                 torch.from_numpy(np.ascontiguousarray(lens)).to(self.device), scale, out, ws)
        pkv.pkv_check_device_error()
        return out_f64(out, act(g)), tables, lens

    def decode_ref(self, q_raw, tables, lens, scale, layer=0):
        return oracle.decode_attention(self.g, layer, q_raw, self.hk, self.hv, tables, lens, scale,
                                       k_scale=self.k_scale, v_scale=self.v_scale)
