#!/usr/bin/env python3
"""Benchmark of the paged KV cache hot path on one GB300 (or N replicas).

One step = one pass of the hot path over the batch: plan the step's appends on
the host control plane (slots, copy-on-write pairs, block tables), copy the
control-plane output to the device, copy shared blocks (CoW), write the new
tokens' K/V at their slots, run paged decode attention over len + 1 tokens, and
release finished sequences.  Workloads (synthetic, seeded):

  agent32k (default): 48 sequences x 32,768 tokens, 70B GQA layer (64 query /
      8 KV heads, d_head 128, bf16, 16-token blocks), block ids a seeded random
      permutation of the pool; 6.4 GB of K/V read per step.
  chat:     256 sequences, lognormal prompt (mean 217) + generated (mean 154)
      lengths clipped to 1,024, 32,768-block pool in a shuffled order; a step is
      one decode step of the 64-step schedule (finished sequences are released).
  forked:   a 16,376-token prefix forked into 64 branches with U[0, 2048] suffixes
      (first append of each branch copies the shared tail block).
  swap:     80-layer 70B geometry (5 MiB blocks); a step evicts 512 chunks of 16
      blocks to a pinned host tier and restores all of them into new blocks.
  tiny:     GPT-2-small geometry, fp32, 8 sequences.

Prints one JSON line.  `--impl reference` times the CPU oracle instead (on a
bounded sample of the same workload, on the host cores).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s & tokens/s (% of 8 TB/s HBM); swap GB/s vs host link"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per algorithmic byte
# of one decode launch, per (stored K/V type, query heads per KV head), from ncu
# captures (summary in profiles/) of the kernels built from the sources with this
# digest: bf16 with 8-head groups at agent 48 x 16,384 (a long batch, so the same
# 120/152 grid as agent 48 x 32,768), the others at 48 x 4,096.  Reported only while
# the sources hash to TRAFFIC_SOURCES_SHA256.
TRAFFIC_SOURCES_SHA256 = "36bcf71d49f183fe0dfe3b9c95aed9fe2351b59eb608f07a9d81cfedce7d1441"
TRAFFIC_RECORD = {
    ("bf16", 8): 1.0018,   # 3,227.3 + 2.9 MB DRAM for 3,224.4 MB algorithmic (mean of 2 launches)
    ("e4m3", 8): 1.0117,   # 406.9 + 2.9 MB for 405.1 MB
    ("bf16", 16): 1.0113,  # 814.4 + 4.6 MB for 809.9 MB
}


def decode_sources_digest() -> str:
    """SHA-256 of the decode kernel's sources with comments and blank space removed (a
    comment-only edit leaves the recorded traffic valid; any code change voids it)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in ("pkv_decode.cu", "pkv_attn.cuh", "pkv_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_80_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()
NOMINAL_HBM_GBS = 8000.0


# ------------------------------------------------------------------ environment


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def mark(self):
        """Per-step marks need NVML's timestamps; nvidia-smi's 200 ms samples have none."""

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class NvmlSampler:
    """Read-only NVML queries (SM clock, max SM clock, clock-event reasons) every
    millisecond from a thread while the timed region runs, each stamped with the host
    clock; mark() stamps a timed step, and each step is given the sample nearest to it."""

    INTERVAL_S = 0.001

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, dev):
        import ctypes
        import threading

        self.ctypes, self.threading = ctypes, threading
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
            ok = self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok and self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.reason_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.marks = []
        self.stop_flag = False

    def _sample(self):
        c = self.ctypes
        mhz, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz))  # NVML_CLOCK_SM
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, c.byref(mx))
        self.reason_fn(self.h, c.byref(rs))
        self.samples.append((mhz.value, mx.value, rs.value, time.perf_counter()))

    def _loop(self):
        while not self.stop_flag:
            self._sample()
            time.sleep(self.INTERVAL_S)

    def mark(self):
        self.marks.append(time.perf_counter())

    def start(self):
        self.thread = self.threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag = True
        self.thread.join()
        if not self.samples:
            self._sample()
        sm = [s[0] for s in self.samples]
        reasons = sorted({name for s in self.samples for bit, name in self.REASONS.items() if s[2] & bit})
        ts_all = [s[3] for s in self.samples]
        gap = (ts_all[-1] - ts_all[0]) / (len(ts_all) - 1) * 1e3 if len(ts_all) > 1 else None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[1] for s in self.samples),
               "reasons": reasons, "samples": len(self.samples),
               "source": "NVML, back to back with a 1 ms pause" + (f" (one sample every {gap:.1f} ms)" if gap else "")}
        if self.marks:
            ts = np.array([s[3] for s in self.samples])
            near = [self.samples[int(np.abs(ts - m).argmin())][0] for m in self.marks]
            out["per_step"] = {"steps": len(near), "sm_mhz_min": min(near), "sm_mhz_median": statistics.median(near),
                               "sm_mhz_max": max(near),
                               "note": "the sample nearest each timed step's launch (host clock)"}
        return out


def clock_sampler(torch, dev):
    try:
        return NvmlSampler(torch, dev)
    except Exception:
        return ClockSampler(torch.cuda.current_device())


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------------ our arm: workloads


class Staging:
    """Ring of pinned host / device buffers for the control plane's per-step output
    (slot mapping, block tables, lengths), copied to the device in one transfer."""

    def __init__(self, torch, dev, n_ints: int, depth: int = 4):
        self.torch = torch
        self.host = [torch.empty(n_ints, dtype=torch.int32, pin_memory=True) for _ in range(depth)]
        self.dev = [torch.empty(n_ints, dtype=torch.int32, device=dev) for _ in range(depth)]
        self.host_np = [h.numpy() for h in self.host]
        self.events = [torch.cuda.Event() for _ in range(depth)]
        for e in self.events:
            e.record()
        self.i = 0

    def next(self):
        k = self.i % len(self.host)
        self.i += 1
        self.events[k].synchronize()
        return k, self.host_np[k], self.host[k], self.dev[k]

    def mark(self, k, n_ints: int):
        """Record that slot k's host buffer is in use by work enqueued so far."""
        self.events[k].record()
        return n_ints * 4


class DecodeRunner:
    """Decode steps over a paged batch: plan -> CoW copy -> append -> attend -> release."""

    name = "decode"

    def __init__(self, torch, pkv, dev, total_steps: int):
        self.torch, self.pkv, self.dev = torch, pkv, dev
        self.total_steps = total_steps
        self.decode_ms = []  # per timed step (CUDA events around the attention call)
        self.kv_bytes = []
        self.alg_bytes = []
        self.tokens = []
        self.h2d_meta = 0
        self.e2e_in_bytes = 0
        self.e2e_out_bytes = 0
        self.l2_flush = None  # a device buffer larger than L2, rewritten after every step when set

    def enable_l2_flush(self):
        """Write 256 MB (twice the L2) after every step, so that no step finds the previous
        step's K/V in L2.  The write runs inside the whole-step time; the decode call's own
        CUDA events do not include it."""
        self.l2_flush = self.torch.empty(64 << 20, dtype=self.torch.int32, device=self.dev)
        self.config["l2"] = ("flushed: 256 MB written after every step (inside the whole-step time, outside "
                             "the decode call's events); " + self.config.get("l2", ""))

    def flush_l2(self, t):
        if self.l2_flush is not None:
            self.l2_flush.fill_(t)

    # subclasses set: g, pool, ids (live batch in order), kp, vp, Wd, scale,
    # q/kn/vn device tensors [steps][n_max][...], and implement running(t)

    def _set_geometry(self, g, kv_scales=(1.0, 1.0)):
        """g.dtype is the stored K/V type; q, out and new keys/values are bf16 around
        an FP8 pool."""
        self.g = g
        self.act = "bf16" if g.dtype == "e4m3" else g.dtype
        self.act_bytes = W.DTYPE_BYTES[self.act]
        self.kv_scales = kv_scales

    def _new_pool(self, free_order):
        g, pkv = self.g, self.pkv
        pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, free_order)
        if g.dtype == "e4m3":
            pkv.pkv_pool_set_kv_scales(pool, *self.kv_scales)
        return pool

    def _alloc_common(self, n_max: int):
        torch, g = self.torch, self.g
        td = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[self.act]
        self.td = td
        self.out = torch.empty((n_max, g.H_q, g.d_head), dtype=td, device=self.dev)
        self.ws = torch.empty(self.pkv.pkv_decode_workspace_size(self.pool, n_max), dtype=torch.uint8,
                              device=self.dev)
        self.staging = Staging(torch, self.dev, self.pkv.pkv_step_meta_ints(self.pool, n_max, self.Wd))
        self.stream = torch.cuda.current_stream().cuda_stream
        self._fast_pool = self.pool
        self._prepare_fast()

    def _prepare_fast(self):
        """Addresses and events for the timed loop, made once: the loop then calls
        pkv_decode_step through a raw ctypes prototype with plain integers."""
        import ctypes

        torch = self.torch
        vp_, i32 = ctypes.c_void_p, ctypes.c_int32
        f = self.pkv._L()["pkv_decode_step"]  # a separate function object (argtypes below)
        f.argtypes = [vp_, i32, vp_, i32, i32, vp_, vp_, vp_, vp_, vp_, ctypes.c_float, vp_, vp_, vp_, vp_,
                      ctypes.c_size_t, vp_, vp_, vp_]
        f.restype = ctypes.c_int
        self.raw_step = f
        es = lambda x: x.element_size() * x[0].numel()
        self.q_base, self.q_stride = self.q.data_ptr(), es(self.q)
        self.k_base, self.k_stride = self.kn.data_ptr(), es(self.kn)
        self.v_base, self.v_stride = self.vn.data_ptr(), es(self.vn)
        self.ptrs = (self.kp.data_ptr(), self.vp.data_ptr(), self.out.data_ptr(), self.ws.data_ptr(),
                     self.ws.numel())
        self.handle = self.pool.handle.value if hasattr(self.pool.handle, "value") else self.pool.handle

    def make_events(self, n):
        """n pairs of timing events, created up front (torch creates a CUDA event at its first record)."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            a.record()
            b.record()
        return evs

    def step(self, t: int, timed: bool = False, events=None):
        """Plan, CoW copy, append and attend through one pkv_decode_step call (device inputs)."""
        torch, pkv, g = self.torch, self.pkv, self.g
        ids = self.running(t)
        n = len(ids)
        if n == 0:
            return
        self.last_ids = ids
        k, hnp, hbuf, dmeta = self.staging.next()
        kp, vp, outp, wsp, wsb = self.ptrs
        h = self.handle if self.pool is self._fast_pool else self._refresh_handle()
        rc = self.raw_step(h, 0, ids.ctypes.data, n, self.Wd, self.q_base + t * self.q_stride,
                           self.k_base + t * self.k_stride, self.v_base + t * self.v_stride, kp, vp,
                           self.scale, outp, hbuf.data_ptr(), dmeta.data_ptr(), wsp, wsb,
                           events[0].cuda_event if events else None, events[1].cuda_event if events else None,
                           self.stream)
        if rc:
            pkv._check(rc, "pkv_decode_step")
        self.flush_l2(t)
        nbytes = self.staging.mark(k, pkv.pkv_step_meta_ints(self.pool, n, self.Wd))
        if timed:
            self.decode_ms.append(events)
            lens = hnp[n + n * self.Wd:n + n * self.Wd + n]
            tok = int(lens.sum(dtype=np.int64))
            kvb = tok * g.H_kv * g.d_head * g.elem_bytes * 2
            self.kv_bytes.append(kvb)
            qo = 2 * n * g.H_q * g.d_head * self.act_bytes
            app = 2 * n * g.H_kv * g.d_head * (self.act_bytes + g.elem_bytes)  # new keys/values in, slots out
            self.alg_bytes.append(kvb + qo + app + n * self.Wd * 4 + n * 4)
            self.tokens.append(n)
            self.h2d_meta += nbytes
        self.after_step(t, ids)

    def e2e_steps(self, host, t0: int, steps: int, events=None, timed: bool = False):
        """End to end through the public host-buffer calls: each step's inputs come from pinned
        host memory and its result is read on the host before the next step's inputs are
        sent.  The host half of step t + 1 (pkv_step_plan: slots, tables, CoW pairs -- it needs
        no result of step t) runs while step t is on the GPU, as a serving loop's scheduler
        does, and writes its metadata into step t + 1's packed input buffer; the device half
        (pkv_step_launch_packed through a PackedStepLauncher, which binds the buffers that stay
        the same from step to step) copies the packed inputs and metadata in with one copy,
        runs the step and copies the result out."""
        torch, pkv, g = self.torch, self.pkv, self.g

        rows, metas, metas_np = self._e2e_views

        def plan(t):
            ids = self.running(t)
            if len(ids) == 0:
                return None
            cows = pkv.pkv_step_plan(self.pool, ids, self.Wd, metas[t])
            return ids, self.pool, metas_np[t], cows

        nxt = plan(t0)
        for i in range(steps):
            t = t0 + i
            cur, nxt = nxt, None
            if cur is not None:
                ids, pool, mnp, cows = cur
                n = len(ids)
                in_bytes = self.off_meta + 4 * pkv.pkv_step_meta_ints(pool, n, self.Wd)
                self.launcher_for(pool)(n, self.Wd, cows, rows[t], self.off_k, self.off_v, in_bytes, self.out_host,
                                        off_meta=self.off_meta, attn_events=events[i] if events else None)
                self.flush_l2(t)
                self.pool = pool
                self.after_step(t, ids)
            if i + 1 < steps:
                nxt = plan(t + 1)  # the next step's host half, while this step runs
            torch.cuda.current_stream().synchronize()  # the step's result is read on the host
            if cur is None:
                continue
            self.last_ids = ids
            if timed:
                if events:
                    self.decode_ms.append(events[i])
                lens = mnp[n + n * self.Wd:n + n * self.Wd + n]
                kvb = int(lens.sum(dtype=np.int64)) * g.H_kv * g.d_head * g.elem_bytes * 2
                self.kv_bytes.append(kvb)
                self.alg_bytes.append(kvb + 2 * n * g.H_q * g.d_head * self.act_bytes + n * self.Wd * 4 + n * 4 +
                                      2 * n * g.H_kv * g.d_head * (self.act_bytes + g.elem_bytes))
                self.tokens.append(n)
            self.e2e_in_bytes += in_bytes
            self.e2e_out_bytes += n * g.H_q * g.d_head * self.act_bytes

    def launcher_for(self, pool):
        """pkv_step_launch_packed with this runner's device staging, pools, scale and workspace
        bound once: a PackedStepLauncher per (control-plane state, stream).  The key holds the
        Pool object itself (it stays alive while cached) and the stream the launcher is fixed
        to, torch's current stream; the previous step's launcher is reused while the state is
        the same (the end-to-end loop runs on one stream)."""
        last = getattr(self, "_last_launcher", None)
        if last is not None and last[0] is pool:  # the common case: the same state as the step before
            return last[1]
        if not hasattr(self, "_launchers"):
            self._launchers = {}
        stream = self.torch.cuda.current_stream().cuda_stream
        key = (pool, stream)
        if key not in self._launchers:
            self._launchers[key] = self.pkv.PackedStepLauncher(pool, 0, self.in_e2e, self.out, self.kp, self.vp,
                                                               self.scale, self.ws, stream=stream)
        self._last_launcher = (pool, self._launchers[key])
        return self._launchers[key]

    def _refresh_handle(self):
        self._fast_pool = self.pool
        self.handle = self.pool.handle.value if hasattr(self.pool.handle, "value") else self.pool.handle
        return self.handle

    def after_step(self, t, ids):
        pass

    def prepare_e2e(self):
        """Each step's inputs packed in one pinned host buffer: q, k_new and v_new (n_max rows
        each), then the step's metadata, which pkv_step_plan writes there; a step of n
        sequences copies the three input parts whole and the metadata of its n rows (the layout
        does not depend on n)."""
        torch, g = self.torch, self.g
        n = self.n_max
        rq, rk = g.H_q * g.d_head * self.act_bytes, g.H_kv * g.d_head * self.act_bytes
        self.off_k, self.off_v = n * rq, n * (rq + rk)
        self.off_meta = n * (rq + 2 * rk)
        step_bytes = self.off_meta + 4 * self.pkv.pkv_step_meta_ints(self.pool, n, self.Wd)
        host = torch.empty((self.total_steps, step_bytes), dtype=torch.uint8, pin_memory=True)
        for t in range(self.total_steps):
            for src, o0, o1 in ((self.q, 0, self.off_k), (self.kn, self.off_k, self.off_v),
                                (self.vn, self.off_v, self.off_meta)):
                host[t, o0:o1].view(self.td).copy_(src[t].reshape(-1))
        self.in_e2e = torch.empty(step_bytes, dtype=torch.uint8, device=self.dev)
        self.out_host = torch.empty(self.out.shape, dtype=self.td, pin_memory=True)
        # per step: the packed row, its metadata part as int32 (pkv_step_plan writes there) and a
        # numpy view of it, made once so that the loop does no tensor slicing
        rows = [host[t] for t in range(self.total_steps)]
        metas = [r[self.off_meta:].view(torch.int32) for r in rows]
        self._e2e_views = (rows, metas, [m.numpy() for m in metas])
        return host

    def inputs_for_steps(self, tag):
        torch, g = self.torch, self.g
        n = self.n_max
        a = self.act
        self.q = W.device_normal(self.seed, f"{tag}_q", (self.total_steps, n, g.H_q, g.d_head), a, self.dev)
        self.kn = W.device_normal(self.seed, f"{tag}_k", (self.total_steps, n, g.H_kv, g.d_head), a, self.dev)
        self.vn = W.device_normal(self.seed, f"{tag}_v", (self.total_steps, n, g.H_kv, g.d_head), a, self.dev)


class AgentRunner(DecodeRunner):
    name = "agent32k"

    def __init__(self, torch, pkv, dev, total_steps, n_seq=48, context=32768, kv_dtype="bf16", q_heads=0,
                 shared=0, share=8):
        super().__init__(torch, pkv, dev, total_steps)
        wl = W.agent(n_seq, context, spare_steps=total_steps + 16)
        self.wl, self.seed = wl, wl.seed
        g0 = with_kv_dtype(wl.geometry, kv_dtype)
        if q_heads:  # another query-head count over the same 8 KV heads (group size q_heads / 8)
            g0 = W.Geometry(g0.L, q_heads, g0.H_kv, g0.d_head, g0.block_size, g0.dtype, g0.num_blocks)
        self._set_geometry(g0)
        g = self.g
        self.n_max = n_seq
        self.scale = wl.scale
        self.pool = self._new_pool(wl.free_order)
        if shared:
            # "KV Cache Management", structured prefix sharing: every agent's context begins with the
            # same `shared` tokens (one parent's, forked: the same physical blocks), then its own
            if share:
                pkv.pkv_pool_set_prefix_sharing(self.pool, share, 1, 0)
            parent = pkv.pkv_seq_create(self.pool)
            pkv.pkv_plan_append(self.pool, [parent], [shared])
            self.ids = [pkv.pkv_seq_fork(self.pool, parent) for _ in range(n_seq)]
            pkv.pkv_plan_append(self.pool, self.ids, [context - shared] * n_seq)
            self.unique_tokens = shared + n_seq * (context - shared)  # grows by one token per agent per step
            self.share_desc = (f"on: runs of >= {share} rows sharing their first blocks attend to them once per step "
                               "(pkv_pool_set_prefix_sharing)" if share else "off: every agent reads the prefix")
        else:
            self.ids = [pkv.pkv_seq_create(self.pool) for _ in range(n_seq)]
            pkv.pkv_plan_append(self.pool, self.ids, [context] * n_seq)
        self.ids_np = np.array(self.ids, np.int32)
        # the pool's contents are the prompt keys/values: N(0,1) drawn on the device
        self.kp = W.device_normal(self.seed, "k_pool", g.pool_shape(), g.dtype, dev)
        self.vp = W.device_normal(self.seed, "v_pool", g.pool_shape(), g.dtype, dev)
        self.Wd = -(-(context + total_steps + 1) // g.block_size)
        self.inputs_for_steps("agent")
        self._alloc_common(n_seq)
        self.config = dict(workload_config("agent32k", g, n_seq, context), pool_blocks=g.num_blocks)
        if shared:
            self.config["workload"] += (f"; the first {shared:,} tokens shared by all (one parent's prefix, forked: "
                                        "structured prefix sharing)")
            self.config["shared_prefix_tokens"] = shared

    def running(self, t):
        return self.ids_np

    def after_step(self, t, ids):
        if hasattr(self, "unique_tokens"):
            self.unique_tokens += len(ids)


class ChatRunner(DecodeRunner):
    name = "chat"

    def __init__(self, torch, pkv, dev, total_steps, n_seq=256, kv_dtype="bf16"):
        super().__init__(torch, pkv, dev, total_steps)
        wl = W.chat(n_seq=n_seq)
        self.wl, self.seed = wl, wl.seed
        self._set_geometry(with_kv_dtype(wl.geometry, kv_dtype))
        g = self.g
        self.n_max = n_seq
        self.scale = wl.scale
        self.sched_steps = wl.extra["steps"]
        self.gen = wl.extra["generated"]
        self.gen_np = np.asarray(self.gen)
        self.all_ids = np.arange(n_seq, dtype=np.int32)
        self.prompt = wl.lengths
        self.kp = W.device_normal(self.seed, "k_pool", g.pool_shape(), g.dtype, dev)
        self.vp = W.device_normal(self.seed, "v_pool", g.pool_shape(), g.dtype, dev)
        self.Wd = -(-1024 // g.block_size) + 1
        # one control-plane state per pass of the 64-step schedule, made up front
        n_pass = -(-total_steps // self.sched_steps) + 1
        self.states = [self._fresh_state() for _ in range(n_pass)]
        self.pool = self.states[0][0]
        self.inputs_for_steps("chat")
        self._alloc_common(n_seq)
        self.config = dict(workload_config("chat", g, n_seq), pool_blocks=g.num_blocks)

    def _fresh_state(self):
        pkv = self.pkv
        pool = self._new_pool(self.wl.free_order)
        ids = [pkv.pkv_seq_create(pool) for _ in range(self.n_max if hasattr(self, "n_max") else 256)]
        pkv.pkv_plan_append(pool, ids, self.prompt)
        return (pool, ids)

    def running(self, t):
        k = t % self.sched_steps
        self.pool, ids = self.states[t // self.sched_steps]
        if not hasattr(self, "_run_by_k"):  # the schedule's running sets and releases, made once
            self._run_by_k = [self.all_ids[self.gen_np > j] for j in range(self.sched_steps)]
            self._done_by_k = [[int(x) for x in self.all_ids[self.gen_np == j + 1]] for j in range(self.sched_steps)]
        return self._run_by_k[k]

    def after_step(self, t, ids):
        for s in self._done_by_k[t % self.sched_steps]:  # generated budget reached: release
            self.pkv.pkv_seq_free(self.pool, s)


class ForkedRunner(DecodeRunner):
    name = "forked"

    def __init__(self, torch, pkv, dev, total_steps, n_branch=64, kv_dtype="bf16", share=8):
        super().__init__(torch, pkv, dev, total_steps)
        wl = W.forked(n_branch=n_branch)
        self.wl, self.seed = wl, wl.seed
        self._set_geometry(with_kv_dtype(wl.geometry, kv_dtype))
        g = self.g
        self.n_max = n_branch
        self.scale = wl.scale
        self.pool = self._new_pool(wl.free_order)
        self.share = share
        if share:  # the branches' shared prefix attended once per step (before the workspace is sized)
            pkv.pkv_pool_set_prefix_sharing(self.pool, share, 1, 0)
        self.kp = W.device_normal(self.seed, "k_pool", g.pool_shape(), g.dtype, dev)
        self.vp = W.device_normal(self.seed, "v_pool", g.pool_shape(), g.dtype, dev)
        parent = pkv.pkv_seq_create(self.pool)
        pkv.pkv_plan_append(self.pool, [parent], [int(wl.lengths[0])])
        self.ids = [pkv.pkv_seq_fork(self.pool, parent) for _ in range(n_branch)]
        suffix = [int(x) for x in wl.extra["suffix"]]
        slots, cows = pkv.pkv_plan_append(self.pool, self.ids, suffix)
        pkv.pkv_copy_blocks(self.pool, cows, self.kp, self.vp)
        if len(slots):
            kn = W.device_normal(self.seed, "suffix_k", (len(slots), g.H_kv, g.d_head), self.act, dev)
            vn = W.device_normal(self.seed, "suffix_v", (len(slots), g.H_kv, g.d_head), self.act, dev)
            pkv.pkv_append_kv(self.pool, 0, kn, vn, torch.from_numpy(slots).to(dev), self.kp, self.vp)
        self.unique_tokens = int(wl.lengths[0]) + sum(suffix)  # grows by one token per branch per step
        self.ids_np = np.array(self.ids, np.int32)
        self.Wd = -(-(int(wl.lengths[0]) + 2048 + total_steps + 1) // g.block_size)
        self.inputs_for_steps("forked")
        self._alloc_common(n_branch)
        self.config = workload_config("forked", g, n_branch, prefix=int(wl.lengths[0]))
        self.share_desc = (f"on: runs of >= {share} rows sharing their first blocks attend to them once per step "
                           "(pkv_pool_set_prefix_sharing)" if share else "off: every branch reads the prefix")

    def running(self, t):
        return self.ids_np

    def after_step(self, t, ids):
        self.unique_tokens += len(ids)


class TinyRunner(DecodeRunner):
    name = "tiny"

    def __init__(self, torch, pkv, dev, total_steps):
        super().__init__(torch, pkv, dev, total_steps)
        wl = W.tiny()
        self.wl, self.seed = wl, wl.seed
        self._set_geometry(wl.geometry)
        g = self.g
        self.n_max = len(wl.lengths)
        self.scale = wl.scale
        self.pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks,
                                        wl.free_order)
        self.ids = [pkv.pkv_seq_create(self.pool) for _ in range(self.n_max)]
        self.ids_np = np.array(self.ids, np.int32)
        pkv.pkv_plan_append(self.pool, self.ids, wl.lengths)
        self.kp = W.device_normal(self.seed, "k_pool", g.pool_shape(), g.dtype, dev)
        self.vp = W.device_normal(self.seed, "v_pool", g.pool_shape(), g.dtype, dev)
        self.Wd = -(-(512 + total_steps + 1) // g.block_size)
        self.inputs_for_steps("tiny")
        self._alloc_common(self.n_max)
        self.config = workload_config("tiny", self.g, self.n_max)

    def running(self, t):
        return self.ids_np


def with_kv_dtype(g, kv_dtype):
    return W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, kv_dtype, g.num_blocks)


def kv_desc(g):
    return "FP8 E4M3 K/V (bf16 q/out)" if g.dtype == "e4m3" else g.dtype


def workload_config(name, g, n_seq, context=0, prefix=0):
    """The bench line's config for a decode workload (both arms print the same one)."""
    rep = "replicas (no collectives)"
    if name == "agent32k":
        return {"workload": f"agent{context // 1024}k: {n_seq} sequences x {context} tokens, {g.H_q} query / "
                            f"{g.H_kv} KV heads, d_head 128, {kv_desc(g)}, 16-token blocks, permuted block ids",
                "n_seq": n_seq, "context": context, "H_q": g.H_q, "H_kv": g.H_kv, "d_head": g.d_head,
                "block_size": g.block_size,
                "l2": f"inputs larger than L2 ({n_seq * context * 2048 * g.elem_bytes / 1e9:.2f} GB of K/V per step)",
                "parallelism": rep}
    if name == "chat":
        return {"workload": "chat: 256 sequences, lognormal prompt (mean 217) + generated (mean 154) "
                            f"lengths <= 1024, 64 query / 8 KV heads, d_head 128, {kv_desc(g)}, 16-token blocks, "
                            "32,768-block pool in shuffled order, 64-step schedule",
                "n_seq": n_seq, "H_q": g.H_q, "H_kv": g.H_kv, "d_head": g.d_head, "block_size": g.block_size,
                "l2": "inputs larger than L2 (0.2-0.3 GB of K/V per step)", "parallelism": rep}
    if name == "forked":
        return {"workload": "forked: 16,376-token prefix forked into 64 branches (refcount 65) with "
                            f"U[0,2048] suffixes, 64 query / 8 KV heads, d_head 128, {kv_desc(g)}, 16-token blocks",
                "n_seq": n_seq, "prefix": prefix, "H_q": g.H_q, "H_kv": g.H_kv, "d_head": g.d_head,
                "block_size": g.block_size,
                "l2": "logical K/V per step 4.5 GB > L2; the 67 MB shared prefix is re-read by every branch",
                "parallelism": rep}
    return {"workload": "tiny: GPT-2-small geometry (12 heads, d_head 64, fp32), 8 sequences of "
                        "U[1,512] tokens, 512-block permuted pool",
            "n_seq": n_seq, "l2": "inputs smaller than L2 (launch-bound case)", "parallelism": rep}


RUNNERS = {"agent32k": AgentRunner, "chat": ChatRunner, "forked": ForkedRunner, "tiny": TinyRunner}


def run_decode(args, torch, pkv, dev, world, rank):
    total = args.warmup + args.steps + 2 + args.steps  # timed region, then e2e warm-up + e2e steps
    kw = {} if args.workload == "tiny" else {"kv_dtype": args.kv_dtype}
    if args.workload == "forked":
        kw["share"] = args.share
    if args.workload == "agent32k" and (args.context or args.n_seq or args.q_heads or args.shared_prefix):
        r = AgentRunner(torch, pkv, dev, total, n_seq=args.n_seq or 48, context=args.context or 32768,
                        q_heads=args.q_heads, shared=args.shared_prefix, share=args.share, **kw)
    else:
        r = RUNNERS[args.workload](torch, pkv, dev, total, **kw)
    if args.l2_flush:
        r.enable_l2_flush()
    g = r.g
    launches0 = None
    for t in range(args.warmup):
        r.step(t)
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    barrier(world)
    clocks = clock_sampler(torch, dev)
    clocks.start()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    evs = r.make_events(args.steps)
    launches0 = pkv.pkv_launch_count()
    u0 = getattr(r, "unique_tokens", None)
    e_start.record()
    for i, t in enumerate(range(args.warmup, args.warmup + args.steps)):
        r.step(t, timed=True, events=evs[i])
        clocks.mark()
    e_end.record()
    torch.cuda.synchronize()
    launches = pkv.pkv_launch_count() - launches0
    barrier(world)
    clk = clocks.stop()
    ms = e_start.elapsed_time(e_end)
    ms_max = reduce_max(torch, world, ms)
    pkv.pkv_check_device_error()
    dec_ms = [a.elapsed_time(b) for a, b in r.decode_ms]
    kv_total = sum(r.kv_bytes)
    alg_avg = sum(r.alg_bytes) / len(r.alg_bytes)
    dec_avg = sum(dec_ms) / len(dec_ms)

    # end to end: inputs from pinned host memory each step, result read back each step
    host = r.prepare_e2e()
    t0 = args.warmup + args.steps
    r.e2e_steps(host, t0, 2)
    r.e2e_in_bytes = r.e2e_out_bytes = 0
    kv_before = len(r.kv_bytes)
    barrier(world)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    r.e2e_steps(host, t0 + 2, args.steps, timed=True)  # no timing events inside the end-to-end loop
    torch.cuda.synchronize()
    e2e_s = reduce_max(torch, world, (time.perf_counter() - h0) * 1e3) / 1e3
    e2e_kv = sum(r.kv_bytes[kv_before:])

    peak, peak_kind = load_peaks()
    value = world * kv_total / (ms_max / 1e3) / 1e9
    traffic = args.traffic
    ratio = TRAFFIC_RECORD.get((g.dtype, g.H_q // g.H_kv))
    if traffic is None and ratio and TRAFFIC_SOURCES_SHA256 == decode_sources_digest():
        traffic = round(ratio * alg_avg)
    achieved = alg_avg / (dec_avg / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": g.dtype, "data": "synthetic", "config": r.config,
        "tokens_per_s": round(world * sum(r.tokens[:args.steps]) / (ms_max / 1e3), 1),
        "hbm_frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "decode step device work: append (programmatic primary) + stream-K attention planned in-kernel + merge",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "alg_bytes_per_launch": int(alg_avg), "avg_launch_ms": round(dec_avg, 4),
                     "note": "the peak is a read + write copy (torch copy_, MEASURED_PEAKS.json); this call's "
                             "bytes are >99.9 % reads, and a read stream runs a little faster than a copy, so "
                             "frac can exceed 1; hbm_frac_of_8tbs is the same rate against the nominal 8 TB/s"},
        "e2e": {"value": round(world * e2e_kv / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(r.e2e_in_bytes / args.steps),
                "d2h_bytes_per_step": int(r.e2e_out_bytes / args.steps)},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if u0 is not None:  # forked: the distinct K/V a step reads (prefix once, every branch's own tokens)
        n = len(r.ids_np)
        per_tok = g.H_kv * g.d_head * g.elem_bytes * 2
        ub = (u0 + n * (args.steps + 1) / 2) * per_tok
        line["shared_prefix"] = r.share_desc
        line["unique"] = {"kv_bytes_per_step": int(ub), "gb_per_s_decode_call": round(ub / (dec_avg / 1e3) / 1e9, 1),
                          "frac": round(ub / (dec_avg / 1e3) / 1e9 / peak, 4),
                          "note": "distinct K/V bytes (the shared prefix counted once) / decode-call time, "
                                  "against the same HBM peak; value counts every branch's logical bytes"}
        # the roofline of this step: the bytes it must move from HBM (the prefix once), not the
        # branches' logical bytes, which L2 reuse or prefix sharing serve without HBM traffic
        other = alg_avg - sum(r.kv_bytes[:args.steps]) / args.steps  # q, out, tables, new keys/values
        alg_u = ub + other
        logical = line["roofline"]["achieved"]
        line["roofline"].update({
            "achieved": round(alg_u / (dec_avg / 1e3) / 1e9, 1), "frac": round(alg_u / (dec_avg / 1e3) / 1e9 / peak, 4),
            "alg_bytes_per_launch": int(alg_u), "traffic": None, "logical_achieved": logical,
            "note": "forked: algorithmic bytes count the shared prefix once (what the step must read from HBM) plus "
                    "each branch's own K/V, q, out, tables and new keys/values; logical_achieved counts every "
                    "branch's whole context"})
    return line, r


def config_records(args, torch, pkv, dev, world, rank, steps: int = 20):
    """Bounded runs of the other decode configurations (tiny, chat, forked, and the agents over a
    shared 24,576-token prompt of "KV Cache Management", Step 5) for the default line: the same
    measurement as `--workload <name>` (`--workload agent32k --shared-prefix 24576`) at `steps`
    timed steps, reduced to its key figures."""
    recs = {}
    for name in ("tiny", "chat", "forked", "agent_shared_prompt"):
        sub = argparse.Namespace(**vars(args))
        sub.workload, sub.steps, sub.warmup = name, steps, 3
        sub.l2_flush, sub.kv_dtype, sub.q_heads, sub.context, sub.n_seq, sub.traffic = False, "bf16", 0, 0, 0, None
        sub.shared_prefix = 0
        if name == "agent_shared_prompt":
            sub.workload, sub.shared_prefix, sub.share = "agent32k", 24576, 8
        ln, r = run_decode(sub, torch, pkv, dev, world, rank)
        recs[name] = {"workload": ln["config"]["workload"], "value": ln["value"], "unit": ln["unit"],
                      "ms_per_step": ln["ms_per_step"], "tokens_per_s": ln["tokens_per_s"],
                      "decode_call": {k: ln["roofline"][k] for k in ("achieved", "frac", "avg_launch_ms",
                                                                      "logical_achieved") if k in ln["roofline"]},
                      "e2e": ln["e2e"]["value"], "gpu_launches": ln["gpu_launches"],
                      "sm_mhz": ln["clocks"]["sm_mhz"] if ln["clocks"] else None, "steps": steps}
        if "unique" in ln:
            recs[name]["unique"] = {k: ln["unique"][k] for k in ("kv_bytes_per_step", "gb_per_s_decode_call", "frac")}
            recs[name]["shared_prefix"] = ln["shared_prefix"]
        del r
        torch.cuda.empty_cache()
    return recs


def measure_link(torch, dev, nbytes: int = 1 << 30, reps: int = 3):
    """Copy-engine ceiling of the host link: pinned cudaMemcpyAsync of nbytes per direction
    (2 untimed, then `reps` timed back to back), in GB/s."""
    probe_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    probe_h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    link = {}
    for name, (dst, src) in (("d2h", (probe_h, probe_d)), ("h2d", (probe_d, probe_h))):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        link[name] = reps * nbytes / (a.elapsed_time(b) / 1e3) / 1e9
    del probe_d, probe_h
    return link


def rated_link_gbs(torch, dev):
    """Rated per-direction bandwidth of this GPU's host link: the sum of its NVLink-C2C links'
    speeds as `nvidia-smi c2c -s` reports them (a read-only query), or None."""
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        out = subprocess.run(["nvidia-smi", "c2c", "-s"], capture_output=True, text=True, timeout=20).stdout
    except Exception:
        return None
    total, mine = 0.0, False
    for line in out.splitlines():
        if line.startswith("GPU "):
            mine = uuid in line
        elif mine and "C2C Link" in line and "GB/s" in line:
            try:
                total += float(line.split(":")[1].split()[0])
            except (IndexError, ValueError):
                pass
    return round(total, 1) if total > 0 else None


def swap_record(torch, pkv, dev, n_chunks: int = 64):
    """A bounded swap measurement for the decode lines: n_chunks 80-layer chunks of 16 blocks
    (5 MiB each) evicted to pinned host frames and restored into fresh blocks, twice, with
    the SM copy kernel; GB/s per direction against the link measured in the same run."""
    wl = W.swap(n_chunks=n_chunks, num_blocks=n_chunks * 16 * 3 // 2)
    g = wl.geometry
    cb = wl.extra["chunk_blocks"]
    pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, wl.free_order)
    ids = [pkv.pkv_seq_create(pool) for _ in range(n_chunks)]
    pkv.pkv_plan_append(pool, ids, wl.lengths)
    kp = W.device_normal(wl.seed, "k_pool", g.pool_shape(), g.dtype, dev)
    vp = W.device_normal(wl.seed, "v_pool", g.pool_shape(), g.dtype, dev)
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * g.elem_bytes
    host = torch.empty(n_chunks * cb * frame, dtype=torch.uint8, pin_memory=True)
    order = [int(x) for x in wl.extra["evict_order"]]
    frames = [np.arange(i * cb, (i + 1) * cb, dtype=np.int64) for i in range(n_chunks)]
    t_out, t_in = [], []
    for rnd in range(3):  # one untimed round, two timed
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        for i, s in enumerate(order):
            pkv.pkv_swap_out(pool, ids[s], kp, vp, host, n_chunks * cb, frames[i])
        e[1].record()
        for s in order[::-1]:
            pkv.pkv_swap_in(pool, ids[s], host, n_chunks * cb, cb, kp, vp)
        e[2].record()
        torch.cuda.synchronize()
        if rnd:
            t_out.append(e[0].elapsed_time(e[1]) / 1e3)
            t_in.append(e[1].elapsed_time(e[2]) / 1e3)
    pkv.pkv_check_device_error()
    del kp, vp, host
    link = measure_link(torch, dev)
    rated = rated_link_gbs(torch, dev)
    nbytes = n_chunks * cb * frame
    out_gbs, in_gbs = nbytes / statistics.mean(t_out) / 1e9, nbytes / statistics.mean(t_in) / 1e9
    rec = {"workload": f"{n_chunks} chunks x 16 blocks of the 80-layer 70B geometry ({nbytes / 1e9:.2f} GB) out to "
                       "pinned host frames and back into fresh blocks, SM copy kernel, mean of 2 rounds",
           "out_gbs": round(out_gbs, 1), "in_gbs": round(in_gbs, 1),
           "link_gbs": {k: round(v, 1) for k, v in link.items()},
           "link_source": "1 GiB pinned cudaMemcpyAsync per direction, this run",
           "frac": round(min(out_gbs / link["d2h"], in_gbs / link["h2d"]), 4)}
    if rated:
        rec["rated_link_gbs"] = rated
        rec["rated_source"] = "sum of this GPU's NVLink-C2C link speeds (nvidia-smi c2c -s), per direction"
        rec["frac_of_rated"] = round(min(out_gbs, in_gbs) / rated, 4)
    return rec


def run_swap(args, torch, pkv, dev, world, rank):
    wl = W.swap() if args.swap_chunks == 512 else W.swap(n_chunks=args.swap_chunks,
                                                         num_blocks=args.swap_chunks * 16 * 3 // 2)
    g = wl.geometry
    nchunk = len(wl.lengths)
    cb = wl.extra["chunk_blocks"]
    pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, g.num_blocks, wl.free_order)
    if args.swap_engine:
        pkv.pkv_pool_set_swap_engine(pool, 1)
    ids = [pkv.pkv_seq_create(pool) for _ in range(nchunk)]
    pkv.pkv_plan_append(pool, ids, wl.lengths)
    kp = W.device_normal(wl.seed, "k_pool", g.pool_shape(), g.dtype, dev)
    vp = W.device_normal(wl.seed, "v_pool", g.pool_shape(), g.dtype, dev)
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * g.elem_bytes
    n_frames = nchunk * cb
    host = torch.empty(n_frames * frame, dtype=torch.uint8, pin_memory=True)
    order = [int(x) for x in wl.extra["evict_order"]]
    frames_of = {s: np.arange(i * cb, (i + 1) * cb, dtype=np.int64) for i, s in enumerate(ids)}

    # host-link roofline: one 1 GiB pinned copy each way on the copy engines
    link = measure_link(torch, dev)
    rated = rated_link_gbs(torch, dev)

    out_ms, in_ms = [], []

    def one_step(timed):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        for s in order:
            pkv.pkv_swap_out(pool, ids[s], kp, vp, host, n_frames, frames_of[ids[s]])
        e[1].record()
        for s in order[::-1]:
            pkv.pkv_swap_in(pool, ids[s], host, n_frames, cb, kp, vp)
        e[2].record()
        if timed:
            out_ms.append((e[0], e[1]))
            in_ms.append((e[1], e[2]))

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    barrier(world)
    clocks = clock_sampler(torch, dev)
    clocks.start()
    l0 = pkv.pkv_launch_count()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record()
    for _ in range(args.steps):
        one_step(True)
    ee.record()
    torch.cuda.synchronize()
    launches = pkv.pkv_launch_count() - l0
    clk = clocks.stop()
    ms = reduce_max(torch, world, es.elapsed_time(ee))
    pkv.pkv_check_device_error()
    bytes_dir = nchunk * cb * frame
    t_out = statistics.mean(a.elapsed_time(b) for a, b in out_ms) / 1e3
    t_in = statistics.mean(a.elapsed_time(b) for a, b in in_ms) / 1e3
    out_gbs, in_gbs = bytes_dir / t_out / 1e9, bytes_dir / t_in / 1e9
    value = world * 2 * bytes_dir * args.steps / (ms / 1e3) / 1e9
    peak = min(link["d2h"], link["h2d"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": g.dtype, "data": "synthetic",
        "config": {"workload": f"swap: 80-layer 70B GQA geometry (327,680 B/token), {nchunk} chunks x 16 blocks "
                               f"({nchunk * cb * frame / 1e9:.1f} GB) evicted to pinned host memory and restored "
                               "into new blocks",
                   "engine": "copy engines" if args.swap_engine else "SM kernel",
                   "l2": f"inputs larger than L2 ({nchunk * cb * frame / 1e9:.1f} GB per direction)" if nchunk * cb * frame > (256 << 20) else "inputs smaller than L2 (diagnostic size)", "parallelism": "replicas (no collectives)"},
        "swap_out_gbs": round(out_gbs, 1), "swap_in_gbs": round(in_gbs, 1),
        "host_link_gbs": {k: round(v, 1) for k, v in link.items()},
        "rated_link_gbs": rated, "frac_of_rated": round(min(out_gbs, in_gbs) / rated, 4) if rated else None,
        "roofline": {"bound": "host-link", "achieved": round(min(out_gbs, in_gbs), 1), "peak": round(peak, 1),
                     "unit": "GB/s", "frac": round(min(out_gbs / link["d2h"], in_gbs / link["h2d"]), 4),
                     "traffic": None, "kernel": "pkv_swap_out / pkv_swap_in",
                     "peak_source": "measured in this run: 1 GiB pinned cudaMemcpyAsync per direction"},
        "e2e": {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": bytes_dir,
                "d2h_bytes_per_step": bytes_dir},
        "gpu_launches": int(launches), "clocks": clk,
    }
    return line, None


def run_overlap(args, torch, pkv, dev, world, rank):
    """Reload of paused sequences (copy engines, own stream) overlapped with decode
    attention of a resident batch (another stream).  Phases: decode alone, reload
    alone, both at once; hidden = (T_dec + T_swap - T_both) / T_swap."""
    L, n_res, ctx, n_paused, plen = 8, 32, 8192, 64, 1024
    seed = W.SEEDS["swap"] + 1
    blocks_res, blocks_p = n_res * ctx // 16, n_paused * plen // 16
    N = blocks_res + 2 * blocks_p + 64
    g = W.Geometry(L=L, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=N)
    pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, N,
                               W.permutation(seed, "overlap_fo", N))
    pkv.pkv_pool_set_swap_engine(pool, args.swap_engine)
    res = [pkv.pkv_seq_create(pool) for _ in range(n_res)]
    pkv.pkv_plan_append(pool, res, [ctx] * n_res)
    paused = [pkv.pkv_seq_create(pool) for _ in range(n_paused)]
    pkv.pkv_plan_append(pool, paused, [plen] * n_paused)
    kp = W.device_normal(seed, "k_pool", g.pool_shape(), g.dtype, dev)
    vp = W.device_normal(seed, "v_pool", g.pool_shape(), g.dtype, dev)
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * g.elem_bytes
    per = plen // 16
    host = torch.empty(blocks_p * frame, dtype=torch.uint8, pin_memory=True)
    frames = {s: np.arange(i * per, (i + 1) * per, dtype=np.int64) for i, s in enumerate(paused)}
    Wd = ctx // 16
    tables, lens = pkv.pkv_export_tables(pool, res, Wd)
    d_tables, d_lens = torch.from_numpy(tables.copy()).to(dev), torch.from_numpy(lens.copy()).to(dev)
    q = W.device_normal(seed, "q", (g.L, n_res, g.H_q, g.d_head), g.dtype, dev)
    out = torch.empty((n_res, g.H_q, g.d_head), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pkv.pkv_decode_workspace_size(pool, n_res), dtype=torch.uint8, device=dev)
    s_dec, s_swap = torch.cuda.Stream(), torch.cuda.Stream()
    scale = 1.0 / math.sqrt(g.d_head)

    def evict():
        for s_ in paused:
            pkv.pkv_swap_out(pool, s_, kp, vp, host, blocks_p, frames[s_], stream=s_swap)
        torch.cuda.synchronize()

    def decode_steps(k):
        for _ in range(k):
            for layer in range(g.L):
                pkv.pkv_decode_attention(pool, layer, q[layer], kp, vp, d_tables, d_lens, scale, out, ws,
                                         stream=s_dec)

    def reload():
        for s_ in paused:
            pkv.pkv_swap_in(pool, s_, host, blocks_p, per, kp, vp, stream=s_swap)

    def timed(fn_dec, fn_swap):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        torch.cuda.synchronize()
        ev[0].record(s_dec)
        s_swap.wait_event(ev[0])
        if fn_dec:
            fn_dec()
        ev[1].record(s_dec)
        if fn_swap:
            fn_swap()
        ev[2].record(s_swap)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / 1e3, ev[0].elapsed_time(ev[2]) / 1e3

    evict()
    k = args.steps
    decode_steps(args.warmup)
    reload()
    evict()
    clocks = clock_sampler(torch, dev)
    clocks.start()
    l0 = pkv.pkv_launch_count()
    t_dec, _ = timed(lambda: decode_steps(k), None)
    _, t_swap = timed(None, reload)
    evict()
    t_dec_b, t_swap_b = timed(lambda: decode_steps(k), reload)
    launches = pkv.pkv_launch_count() - l0
    clk = clocks.stop()
    pkv.pkv_check_device_error()
    t_both = max(t_dec_b, t_swap_b)
    kv = int(lens.astype(np.int64).sum()) * g.H_kv * g.d_head * 2 * 2 * g.L * k
    sw = blocks_p * frame
    peak, _ = load_peaks()
    hidden = (t_dec + t_swap - t_both) / t_swap
    return {
        "metric": METRIC, "value": round(kv / t_dec_b / 1e9, 2), "unit": "GB/s", "n_gpus": world, "steps": k,
        "warmup": args.warmup, "ms_per_step": round(t_both / k * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "overlap: decode of 32 x 8,192-token sequences over 8 layers on one stream while 64 "
                               "paused 1,024-token sequences (2.1 GB) reload from pinned host memory on another",
                   "engine": "copy engines" if args.swap_engine else "SM kernel",
                   "l2": "inputs larger than L2", "parallelism": "replicas (no collectives)"},
        "decode_gbs_alone": round(kv / t_dec / 1e9, 1), "decode_gbs_overlapped": round(kv / t_dec_b / 1e9, 1),
        "swap_in_gbs_alone": round(sw / t_swap / 1e9, 1), "swap_in_gbs_overlapped": round(sw / t_swap_b / 1e9, 1),
        "hidden_reload_fraction": round(hidden, 3),
        "ms": {"decode_alone": round(t_dec * 1e3, 3), "reload_alone": round(t_swap * 1e3, 3),
               "both": round(t_both * 1e3, 3)},
        "roofline": {"bound": "hbm", "achieved": round(kv / t_dec_b / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(kv / t_dec_b / 1e9 / peak, 4), "traffic": None,
                     "kernel": "pkv_decode_attention while a reload runs"},
        "e2e": {"value": round(kv / t_dec_b / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": int(sw / k),
                "d2h_bytes_per_step": 0},
        "gpu_launches": int(launches), "clocks": clk,
    }, None


def run_reload_prefill(args, torch, pkv, dev, world, rank):
    """Pipelined chunked reload behind the observation's chunked prefill ("KV Cache Management",
    "Asynchronous paged swapping"): a paused 80-layer sequence's history (16,384 tokens, 5.4 GB)
    returns from pinned host frames a range of layers at a time on one stream while a 2,048-token
    observation is prefilled in 512-token chunks on another (per layer: append, then prefill
    attention over the history and the chunk); layer l of the first chunk waits only for the
    range holding l.  Phases: reload alone, prefill alone, serial (whole reload, then prefill),
    pipelined; hidden = (T_reload + T_prefill - T_pipelined) / T_reload."""
    L, hist, obs, C, per_range = 80, args.context or 16384, 2048, 512, args.reload_layers
    seed = W.SEEDS["swap"] + 2
    nb_hist, nb_obs = -(-hist // 16), -(-(hist + obs) // 16) - hist // 16
    N = nb_hist + nb_obs + 64
    g = W.Geometry(L=L, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=N)
    fo = W.permutation(seed, "reload_fo", N)
    kp = W.device_normal(seed, "k_pool", g.pool_shape(), g.dtype, dev)
    vp = W.device_normal(seed, "v_pool", g.pool_shape(), g.dtype, dev)
    frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * g.elem_bytes
    host = torch.empty(nb_hist * frame, dtype=torch.uint8, pin_memory=True)
    frames = np.arange(nb_hist, dtype=np.int64)
    k_new = W.device_normal(seed, "k_obs", (L, obs, g.H_kv, g.d_head), g.dtype, dev)
    v_new = W.device_normal(seed, "v_obs", (L, obs, g.H_kv, g.d_head), g.dtype, dev)
    q = W.device_normal(seed, "q_obs", (L, obs, g.H_q, g.d_head), g.dtype, dev)
    out = torch.empty((C, g.H_q, g.d_head), dtype=torch.bfloat16, device=dev)
    offs = torch.tensor([0, C], dtype=torch.int32, device=dev)
    ranges = [(l0, min(L, l0 + per_range)) for l0 in range(0, L, per_range)]
    s_copy, s_pre = torch.cuda.Stream(), torch.cuda.Stream()
    scale = 1.0 / math.sqrt(g.d_head)

    def paused_state():
        """A fresh control plane whose one sequence holds the history, evicted to the host frames."""
        pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, N, fo)
        pkv.pkv_pool_set_swap_engine(pool, args.swap_engine)
        seq = pkv.pkv_seq_create(pool)
        pkv.pkv_plan_append(pool, [seq], [hist])
        pkv.pkv_swap_out(pool, seq, kp, vp, host, nb_hist, frames, stream=s_copy)
        torch.cuda.synchronize()
        return pool, seq

    def reload(pool, seq, by_range, stream):
        evs = {}
        for l0, l1 in (ranges if by_range else [(0, L)]):
            pkv.pkv_swap_in_layers(pool, seq, host, nb_hist, nb_hist, l0, l1, kp, vp, stream=stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            for layer in range(l0, l1):
                evs[layer] = ev
        return evs

    def prefill(pool, seq, stream, evs=None):
        slots, _ = pkv.pkv_plan_append(pool, [seq], [obs])
        W_ = -(-(hist + obs) // 16)
        tables, _ = pkv.pkv_export_tables(pool, [seq], W_)
        d_slots = torch.from_numpy(slots.copy()).to(dev, non_blocking=True)
        d_tables = torch.from_numpy(tables.copy()).to(dev, non_blocking=True)
        d_lens = [torch.tensor([hist + (c + 1) * C], dtype=torch.int32).to(dev, non_blocking=True)
                  for c in range(obs // C)]
        waited = set()
        for c in range(obs // C):
            for layer in range(L):
                if evs is not None and evs[layer] not in waited:
                    stream.wait_event(evs[layer])
                    waited.add(evs[layer])
                pkv.pkv_append_kv(pool, layer, k_new[layer, c * C:(c + 1) * C], v_new[layer, c * C:(c + 1) * C],
                                  d_slots[c * C:(c + 1) * C], kp, vp, stream=stream)
                pkv.pkv_prefill_attention(pool, layer, q[layer, c * C:(c + 1) * C], offs, C, kp, vp, d_tables,
                                          d_lens[c], scale, out, stream=stream)

    def timed(fn):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_pre)
        s_copy.wait_event(a)
        fn()
        e_copy = torch.cuda.Event()
        e_copy.record(s_copy)
        s_pre.wait_event(e_copy)
        b.record(s_pre)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3

    def run(mode):
        pool, seq = paused_state()
        if mode == "reload":
            return timed(lambda: reload(pool, seq, True, s_copy))
        if mode == "prefill":
            reload(pool, seq, False, s_copy)
            torch.cuda.synchronize()
            return timed(lambda: prefill(pool, seq, s_pre))
        if mode == "serial":
            return timed(lambda: (reload(pool, seq, False, s_pre), prefill(pool, seq, s_pre)))
        return timed(lambda: prefill(pool, seq, s_pre, reload(pool, seq, True, s_copy)))

    for mode in ("reload", "prefill", "pipelined"):  # warm-up
        run(mode)
    clocks = clock_sampler(torch, dev)
    clocks.start()
    l0 = pkv.pkv_launch_count()
    reps = max(1, args.steps)
    t = {m: statistics.median(run(m) for _ in range(reps)) for m in ("reload", "prefill", "serial", "pipelined")}
    launches = pkv.pkv_launch_count() - l0
    clk = clocks.stop()
    pkv.pkv_check_device_error()
    rb = nb_hist * frame
    flop = L * sum(4.0 * g.H_q * g.d_head * (hist + c * C + i + 1) for c in range(obs // C) for i in range(C))
    hidden = (t["reload"] + t["prefill"] - t["pipelined"]) / t["reload"]
    peak, _ = load_peaks()
    tflops = flop / t["pipelined"] / 1e12
    return {
        "metric": METRIC, "value": round(rb / t["pipelined"] / 1e9, 2), "unit": "GB/s", "n_gpus": world,
        "steps": reps, "warmup": 1, "ms_per_step": round(t["pipelined"] * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"reload_prefill: an 80-layer 70B GQA sequence's {hist}-token history "
                               f"({rb / 1e9:.2f} GB) reloaded from pinned host frames {per_range} layers at a time "
                               f"while a {obs}-token observation is prefilled in {C}-token chunks",
                   "engine": "copy engines" if args.swap_engine else "SM kernel",
                   "l2": "inputs larger than L2", "parallelism": "replicas (no collectives)"},
        "hidden_reload_fraction": round(hidden, 3),
        "exposed_reload_ms": round((t["pipelined"] - t["prefill"]) * 1e3, 3),
        "ms": {k: round(v * 1e3, 3) for k, v in t.items()},
        "reload_gbs_alone": round(rb / t["reload"] / 1e9, 1),
        "prefill_tflops_alone": round(flop / t["prefill"] / 1e12, 1), "prefill_tflops_pipelined": round(tflops, 1),
        "roofline": {"bound": "host-link", "achieved": round(rb / t["reload"] / 1e9, 1), "peak": None,
                     "unit": "GB/s", "frac": None, "traffic": None,
                     "kernel": "pkv_swap_in_layers (reload alone); see the swap workload for the link's peak"},
        "e2e": {"value": round(rb / t["pipelined"] / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": rb,
                "d2h_bytes_per_step": 0},
        "gpu_launches": int(launches), "clocks": clk,
    }, None


def run_prefill(args, torch, pkv, dev, world, rank):
    """Chunked prefill: 8 sequences with 16,384 cached tokens each take a 512-token chunk.
    Each step forks the 8 histories (no data moves), plans and writes the chunks'
    keys/values, and runs chunked-prefill attention (history in full, causal within
    the chunk)."""
    n, hist, C = 8, args.context or 16384, 512
    seed = W.SEEDS["agent32k"] + 11
    total = args.warmup + args.steps
    N = n * hist // 16 + total * n * (C // 16) + 64
    kvd = getattr(args, "kv_dtype", "bf16") or "bf16"
    g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype=kvd, num_blocks=N)
    pool = pkv.pkv_pool_create(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, N,
                               W.permutation(seed, "prefill_fo", N))
    base = [pkv.pkv_seq_create(pool) for _ in range(n)]
    pkv.pkv_plan_append(pool, base, [hist] * n)
    kp = W.device_normal(seed, "k_pool", g.pool_shape(), g.dtype, dev)
    vp = W.device_normal(seed, "v_pool", g.pool_shape(), g.dtype, dev)
    act = "bf16" if kvd == "e4m3" else g.dtype  # q, out and new keys/values around an E4M3 pool: bf16
    q = W.device_normal(seed, "q", (total, n * C, g.H_q, g.d_head), act, dev)
    kn = W.device_normal(seed, "kn", (total, n * C, g.H_kv, g.d_head), act, dev)
    vn = W.device_normal(seed, "vn", (total, n * C, g.H_kv, g.d_head), act, dev)
    out = torch.empty((n * C, g.H_q, g.d_head), dtype=torch.bfloat16, device=dev)
    offs = torch.arange(0, n * C + 1, C, dtype=torch.int32, device=dev)
    Wd = (hist + C) // 16
    scale = 1.0 / math.sqrt(g.d_head)
    ev = []

    def step(t, timed):
        kids = [pkv.pkv_seq_fork(pool, b) for b in base]
        slots, cows = pkv.pkv_plan_append(pool, kids, [C] * n)
        tables, lens = pkv.pkv_export_tables(pool, kids, Wd)
        d_slots = torch.from_numpy(slots).to(dev, non_blocking=True)
        d_tab = torch.from_numpy(tables.copy()).to(dev, non_blocking=True)
        d_len = torch.from_numpy(lens.copy()).to(dev, non_blocking=True)
        if len(cows):
            pkv.pkv_copy_blocks(pool, cows, kp, vp)
        pkv.pkv_append_kv(pool, 0, kn[t], vn[t], d_slots, kp, vp)
        e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) if timed else None
        if e:
            e[0].record()
        pkv.pkv_prefill_attention(pool, 0, q[t], offs, C, kp, vp, d_tab, d_len, scale, out)
        if e:
            e[1].record()
            ev.append(e)
        return kids

    for t in range(args.warmup):
        step(t, False)
    torch.cuda.synchronize()
    pkv.pkv_check_device_error()
    clocks = clock_sampler(torch, dev)
    clocks.start()
    l0 = pkv.pkv_launch_count()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record()
    for t in range(args.warmup, total):
        step(t, True)
    ee.record()
    torch.cuda.synchronize()
    launches = pkv.pkv_launch_count() - l0
    clk = clocks.stop()
    pkv.pkv_check_device_error()
    ms = es.elapsed_time(ee) / args.steps
    att = statistics.mean(a.elapsed_time(b) for a, b in ev)
    flop = sum(4.0 * g.H_q * g.d_head * (hist + i + 1) for i in range(C)) * n
    kvb = n * (hist + C) * g.H_kv * g.d_head * W.DTYPE_BYTES[g.dtype] * 2
    tflops = flop / (att / 1e3) / 1e12
    peak = 1916.4
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    return {
        "metric": METRIC, "value": round(flop / (ms / 1e3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 (E4M3 K/V)" if kvd == "e4m3" else "bf16",
        "data": "synthetic",
        "config": {"workload": f"prefill: {n} sequences x {hist:,} cached tokens, a {C}-token chunk each (forked "
                               f"histories), 64 query / 8 KV heads, d_head 128, {kv_desc(g)}, 16-token blocks",
                   "l2": (f"inputs larger than L2 ({kvb / 1e9:.2f} GB of K/V per step)" if kvb > 129e6 else
                          f"K/V smaller than L2 ({kvb / 1e9:.2f} GB per step), not flushed: a diagnostic size"),
                   "parallelism": "replicas (no collectives)"},
        "tokens_per_s": round(n * C / (ms / 1e3), 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4), "traffic": None,
                     "kernel": "pkv_prefill_attention (" + ("mma.sync m16n8k16" if os.environ.get("PKV_PREFILL_MMA_SYNC")
                                                           else "tcgen05.mma kind::f16, TMEM accumulators") + ")",
                     "avg_launch_ms": round(att, 4),
                     "kv_bytes_per_launch": kvb},
        "e2e": {"value": round(flop / (ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(n * Wd * 4 + n * C * 4), "d2h_bytes_per_step": 0},
        "gpu_launches": int(launches), "clocks": clk,
    }, None


# ------------------------------------------------------------------ CPU baseline (the oracle)


def oracle_sample_decode(runner, n_sample: int, reps: int = 1):
    """Time the oracle's attention on n_sample sequences of the runner's batch, on
    host copies of exactly their blocks.  Returns (GB/s, seconds, description)."""
    import torch
    import oracle

    g = runner.g
    pool = runner.pool
    ids = []
    for s in (int(x) for x in runner.last_ids):  # sequences still resident after the last step
        try:
            runner.pkv.pkv_seq_len(pool, s)
            ids.append(s)
        except runner.pkv.PkvError:
            pass
    ids = ids[:n_sample]
    Wd = runner.Wd
    tables, lens = runner.pkv.pkv_export_tables(pool, ids, Wd)
    used = sorted({int(b) for i in range(len(ids)) for b in tables[i, : -(-int(lens[i]) // g.block_size)]})
    remap = {b: j for j, b in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=runner.kp.device)
    store = {"bf16": np.uint16, "f16": np.float16, "f32": np.float32}[runner.act]

    def host_copy(t):
        x = t.index_select(0, idx).cpu().contiguous()
        if g.dtype == "bf16":
            return x.view(torch.int16).numpy().view(np.uint16)
        return x.numpy()

    hk, hv = host_copy(runner.kp), host_copy(runner.vp)
    gc = W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, len(used))
    ct = np.zeros_like(tables)
    for i in range(len(ids)):
        nb = -(-int(lens[i]) // g.block_size)
        ct[i, :nb] = [remap[int(b)] for b in tables[i, :nb]]
    q = W.normal(runner.seed, "oracle_q", (len(ids), g.H_q, g.d_head), runner.act).astype(store)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.decode_attention(gc, 0, q, hk, hv, ct, lens, runner.scale, k_scale=runner.kv_scales[0],
                                v_scale=runner.kv_scales[1])
    dt = (time.perf_counter() - t0) / reps
    kvb = int(lens.astype(np.int64).sum()) * g.H_kv * g.d_head * g.elem_bytes * 2
    return kvb / dt / 1e9, dt, f"oracle attention over {len(ids)} of the batch's sequences " \
                               f"({int(lens.sum())} tokens), {oracle.hardware_threads()} threads"


# ------------------------------------------------------------------ reference arm (the oracle alone)


def reference_arm(args, world, rank):
    import oracle

    if rank != 0:
        return None
    cores = oracle.hardware_threads()
    if args.workload == "prefill":
        hist, C = 16384, 32
        g = W.Geometry(L=1, H_q=64, H_kv=8, d_head=128, block_size=16, dtype="bf16", num_blocks=(hist + C) // 16)
        kp = W.normal(1, "ref_k", g.pool_shape(), "bf16")
        vp = W.normal(1, "ref_v", g.pool_shape(), "bf16")
        tables = W.permutation(1, "ref_perm", g.num_blocks).reshape(1, -1)
        q = W.normal(1, "ref_q", (C, g.H_q, g.d_head), "bf16")
        lens = np.array([hist + C], np.int32)
        times = []
        for step in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.prefill_attention(g, 0, q, np.array([0, C], np.int32), kp, vp, tables, lens, 1 / math.sqrt(128))
            if step >= args.warmup:
                times.append(time.perf_counter() - t0)
        flop = sum(4.0 * g.H_q * g.d_head * (hist + i + 1) for i in range(C))
        t_step = statistics.mean(times)
        value = flop / t_step / 1e12
        return {
            "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prefill (sampled: one sequence, 32 chunk queries over 16,384 cached tokens)"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "oracle chunked-prefill attention, 1 sequence x 32 queries x 16,416 keys"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    if args.workload in ("swap", "overlap", "reload_prefill"):
        wl = W.swap(n_chunks=16)
        g = wl.geometry
        nb = 64
        gs = W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, nb)
        kp = W.normal(wl.seed, "k_pool", gs.pool_shape(), "bf16")
        vp = W.normal(wl.seed, "v_pool", gs.pool_shape(), "bf16")
        frame = 2 * g.L * g.H_kv * g.block_size * g.d_head * 2
        host = np.zeros(nb * frame, np.uint8)
        ids = np.arange(nb, dtype=np.int32)
        slots = np.arange(nb, dtype=np.int64)[::-1].copy()
        times = []
        for step in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.swap_out_data(gs, ids, slots, kp, vp, host)
            oracle.swap_in_data(gs, ids, slots, host, kp, vp)
            if step >= args.warmup:
                times.append(time.perf_counter() - t0)
        bytes_step = 2 * nb * frame
        value = bytes_step / statistics.mean(times) / 1e9
        desc = f"oracle memcpy swap-out + swap-in of {nb} 5 MiB blocks per step"
        config = {"workload": "swap: 80-layer 70B GQA geometry, 5 MiB blocks (sampled)"}
        dtype = "bf16"
    else:
        spec = {"agent32k": (lambda: W.agent(args.n_seq or 48, args.context or 32768, 256), 2),
                "chat": (lambda: W.chat(), 64),
                "forked": (lambda: W.forked(), 4),
                "tiny": (lambda: W.tiny(), 8)}[args.workload]
        wl, n_s = spec[0](), spec[1]
        g = wl.geometry if args.workload == "tiny" else with_kv_dtype(wl.geometry, args.kv_dtype)
        act = oracle.q_dtype(g)
        lens = np.array([int(x) for x in wl.lengths[:n_s]], np.int32) if args.workload != "forked" else \
            np.array([int(wl.lengths[0]) + int(s) for s in wl.extra["suffix"][:n_s]], np.int32)
        if args.workload == "chat":
            lens = np.array([int(wl.lengths[i]) + 1 for i in range(n_s)], np.int32)
        nblk = [-(-int(x) // g.block_size) for x in lens]
        gs = W.Geometry(g.L, g.H_q, g.H_kv, g.d_head, g.block_size, g.dtype, sum(nblk))
        if g.dtype == "e4m3":  # codes of N(0,1) draws
            kp = oracle.e4m3_encode(W.normal(wl.seed, "ref_k", gs.pool_shape(), "f32"))
            vp = oracle.e4m3_encode(W.normal(wl.seed, "ref_v", gs.pool_shape(), "f32"))
        else:
            kp = W.normal(wl.seed, "ref_k", gs.pool_shape(), g.dtype)
            vp = W.normal(wl.seed, "ref_v", gs.pool_shape(), g.dtype)
        perm = W.permutation(wl.seed, "ref_perm", sum(nblk))
        Wd = max(nblk)
        tables = np.zeros((n_s, Wd), np.int32)
        o = 0
        for i, nb in enumerate(nblk):
            tables[i, :nb] = perm[o:o + nb]
            o += nb
        q = W.normal(wl.seed, "ref_q", (n_s, g.H_q, g.d_head), act)
        times = []
        for step in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.decode_attention(gs, 0, q, kp, vp, tables, lens, wl.scale)
            if step >= args.warmup:
                times.append(time.perf_counter() - t0)
        bytes_step = int(lens.astype(np.int64).sum()) * g.H_kv * g.d_head * g.elem_bytes * 2
        value = bytes_step / statistics.mean(times) / 1e9
        desc = f"oracle attention over {n_s} sequences ({int(lens.sum())} tokens) of the {args.workload} workload"
        # the same config as this workload's line from the library arm, plus the sample size
        n_full = {"agent32k": args.n_seq or 48, "chat": 256, "forked": 64, "tiny": 8}[args.workload]
        config = dict(workload_config(args.workload, g, n_full, context=args.context or 32768,
                                      prefix=int(wl.lengths[0]) if args.workload == "forked" else 0),
                      sampled_sequences=n_s)
        dtype = g.dtype
    t_step = statistics.mean(times)
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": config,
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ plumbing


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(torch, world, x: float) -> float:
    """Max over ranks (timing only; the data path has no collective)."""
    if world <= 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 100; swap 4)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 10; swap 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["agent32k", "chat", "forked", "swap", "tiny", "overlap", "prefill",
                                           "reload_prefill"],
                    default="agent32k")
    ap.add_argument("--swap-engine", type=int, default=0, help="swap workload: 0 SM kernel, 1 copy engines")
    ap.add_argument("--reload-layers", type=int, default=1,
                    help="reload_prefill workload: layers per reload range (default 1)")
    ap.add_argument("--swap-chunks", type=int, default=512,
                    help="swap workload: chunks evicted and restored (default 512, 42.9 GB; fewer for small captures)")
    ap.add_argument("--share", type=int, default=8,
                    help="forked / --shared-prefix: prefix sharing, the least rows of a run that shares its first "
                         "blocks (0: off)")
    ap.add_argument("--shared-prefix", type=int, default=0,
                    help="agent32k: the first S tokens of every context are one parent's prefix, forked (structured "
                         "prefix sharing, e.g. 24576 with --context 32768)")
    ap.add_argument("--no-config-records", action="store_true",
                    help="default line: skip the bounded tiny / chat / forked / shared-prompt agent runs added to it")
    ap.add_argument("--no-swap-record", action="store_true",
                    help="decode workloads: skip the bounded swap measurement added to the line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--context", type=int, default=0, help="agent workload: tokens per sequence (default 32768)")
    ap.add_argument("--n-seq", type=int, default=0, help="agent workload: sequences (default 48)")
    ap.add_argument("--l2-flush", action="store_true",
                    help="decode workloads: overwrite a 256 MB buffer after every step (forked: the prefix "
                         "then comes from HBM at each step's first read)")
    ap.add_argument("--q-heads", type=int, default=0,
                    help="agent workload: query heads over its 8 KV heads (default 64; 128 = groups of 16)")
    ap.add_argument("--kv-dtype", choices=["bf16", "e4m3"], default="bf16",
                    help="decode workloads: stored K/V type (e4m3 = FP8 pool, bf16 q/out)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per decode launch, if captured for this kernel version")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {"swap": 4, "overlap": 8, "prefill": 20, "reload_prefill": 3}.get(args.workload, 100)
    if args.warmup is None:
        args.warmup = 3 if args.workload == "swap" else 10
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()

    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group("gloo")
        line = reference_arm(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch

    import paged_kv_cache_80_gb300 as pkv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if args.workload == "swap":
        line, runner = run_swap(args, torch, pkv, dev, world, rank)
    elif args.workload == "overlap":
        line, runner = run_overlap(args, torch, pkv, dev, world, rank)
    elif args.workload == "prefill":
        line, runner = run_prefill(args, torch, pkv, dev, world, rank)
    elif args.workload == "reload_prefill":
        line, runner = run_reload_prefill(args, torch, pkv, dev, world, rank)
    else:
        line, runner = run_decode(args, torch, pkv, dev, world, rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if runner is not None:
            n_sample = {"agent32k": 16, "chat": 256, "forked": 16, "tiny": 8}[args.workload]
            v, dt, desc = oracle_sample_decode(runner, n_sample)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": __import__("oracle").hardware_threads(),
                                    "kind": "oracle", "sample": desc + f", {dt:.2f} s"}
        elif args.workload == "prefill":
            ref = reference_arm(argparse.Namespace(workload="prefill", steps=1, warmup=0), 1, 0)
            line["cpu_baseline"] = dict(ref["cpu_baseline"])
        else:
            ref = reference_arm(argparse.Namespace(workload="swap", steps=2, warmup=1), 1, 0)
            line["cpu_baseline"] = dict(ref["cpu_baseline"])
            line["cpu_baseline"]["sample"] += " (host-tier copy baseline)"
    if world == 1 and runner is not None and not args.no_swap_record and args.workload != "tiny":
        # the second target of the metric (swap GB/s against the host link), bounded, after the decode
        # measurement; the decode pools are released first
        runner.kp = runner.vp = None
        runner._launchers = {}
        runner._last_launcher = None
        torch.cuda.empty_cache()
        line["swap"] = swap_record(torch, pkv, dev)
    if (world == 1 and args.workload == "agent32k" and not (args.context or args.n_seq or args.q_heads
                                                            or args.shared_prefix)
            and args.kv_dtype == "bf16" and not args.no_config_records):
        # driver-observed figures for the other decode configurations, bounded
        runner = None
        line["other_configs"] = config_records(args, torch, pkv, dev, world, rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
