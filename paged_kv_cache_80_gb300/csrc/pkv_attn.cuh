// Declarations shared by the attention translation units (decode and chunked prefill):
// the launch-argument block, the element types and conversions, the CUDA-core
// attention routine, and the host helpers for tensor maps and arguments.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct E4M3 {  // one stored OCP FP8 E4M3 element
  uint8_t bits;
};

constexpr int TILE = 16;   // tokens per tile (the mma M dimension)
constexpr int GPAD = 8;    // query heads per mma N dimension
constexpr int SIMT_GMAX = 16;  // query heads per KV head on the CUDA-core kernels (16 only for d_head <= 128)
constexpr uint64_t kWaitNs = 2000000000ull;  // a tile load that takes 2 s is a fault: give up

struct DecodeArgs {
  const void* q;
  void* out;
  const int32_t* tables;
  const int32_t* seq_lens;
  int32_t* tile_prefix;  // [n_seq + 1]: tiles of sequences before s (per KV head)
  int32_t* lens_c;       // [n_seq]: lengths clamped to [0, W*B]
  int32_t* hdr;          // [0] = total tiles over all pairs
  // [total_warps]: arrivals at the split pair whose first tile lies in warp w's range, as
  // (epoch << 16) | count; a word carrying another launch's epoch counts as zero, so the
  // array needs no clearing between launches
  unsigned long long* counters;
  int4* wstart;          // [total_warps]: (sequence, KV head, tile, tiles of pair) at each warp's first tile
  float* partials;
  int* err;
  int64_t num_blocks;
  int32_t n_seq, W, H_q, H_kv, G, L, layer, B;
  int32_t D, elem;   // head dimension, bytes per activation element (q, out)
  float scale_log2;  // scale * log2(e) (* k_scale for an FP8 pool)
  float v_mul;       // 1, or v_scale for an FP8 pool
  int32_t total_warps;
  int32_t self_plan;           // 1: every CTA plans its own warps from seq_lens (no plan kernel)
  unsigned long long epoch;    // 48-bit tag of this launch (nonzero, unique in the process)
  // Shared prefixes (all null without one).  share[s] = {kb, items, slot0, stride}: the first kb
  // table blocks of sequence s are a prefix it shares with other rows of the batch, attended by
  // the prefix kernel, whose `items` partials for s sit in slots slot0 + i * stride; the decode
  // kernel attends to the rest and leaves its partial of such a row in sfx_ml / sfx_o (row s)
  // instead of writing out; the combine kernel merges the two into out.  share_items: the
  // prefix kernel's work items, 8 ints each {row_begin, row_end, kb0, kb1, slot_base, 0, 0, 0}.
  // Partials: per (slot or row, query head) the running max m (base 2) and sum l, and O
  // relative to 2^m.
  const int4* share;
  const int32_t* share_items;
  float* prior_ml;
  float* prior_o;
  int64_t prior_slots;  // slots prior_ml / prior_o hold
  float* sfx_ml;
  float* sfx_o;
};

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }


template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f<E4M3>(E4M3 x) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(x.bits, __NV_E4M3)));
}

template <typename T>
__device__ __forceinline__ T f_to(float x);
template <>
__device__ __forceinline__ float f_to<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half f_to<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 f_to<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

constexpr int SIMT_WARPS = 8;

// One CTA per (sequence, KV head).  Lane j holds elements j, j+32, ... of the head
// vector.  Warp w takes chunks of TOK consecutive tokens (w*TOK, w*TOK + 8*TOK, ...):
// it loads all TOK keys and values first (independent loads in flight), then
// scores them for every query head of the group (warp reductions) and folds them
// into the running (m, l, O) of each head with one rescale per chunk.  The warps
// are merged in shared memory at the end.
// Attention of the G query rows at q (contiguous, d apart) over the first len tokens
// of sequence s, KV head g; writes G rows at out.  Run by the whole CTA.  TS is the
// stored K/V element, TA the q / out element; HP >= G is the head capacity (8, or 16
// for wider groups).
template <typename TS, typename TA, int NPL, int HP = GPAD>
__device__ __forceinline__ void simt_attend(const DecodeArgs& a, const TS* __restrict__ kp,
                                            const TS* __restrict__ vp, int d, int s, int g, int len, const TA* q,
                                            TA* out) {
  constexpr int TOK = NPL >= 8 ? 2 : (NPL >= 4 ? 4 : 8);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = a.G;
  float qv[HP][NPL], o[HP][NPL], m[HP], l[HP];
#pragma unroll
  for (int h = 0; h < HP; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + 32 * j;
      qv[h][j] = (h < G && e < d) ? to_f(q[h * d + e]) * a.scale_log2 : 0.f;
      o[h][j] = 0.f;
    }
  }
  for (int t0 = warp * TOK; t0 < len; t0 += SIMT_WARPS * TOK) {
    float k[TOK][NPL], v[TOK][NPL];
    bool ok[TOK];
#pragma unroll
    for (int u = 0; u < TOK; ++u) {
      const int t = t0 + u;
      ok[u] = t < len;
      int64_t base = 0;
      if (ok[u]) {
        int blk = a.tables[static_cast<int64_t>(s) * a.W + t / a.B];
        if (blk < 0 || blk >= a.num_blocks) {
          if (lane == 0) record_error(a.err, DERR_DECODE_BLOCK, blk);
          ok[u] = false;
        } else {
          base = (((static_cast<int64_t>(blk) * a.L + a.layer) * a.H_kv + g) * a.B + t % a.B) * d;
        }
      }
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int e = lane + 32 * j;
        k[u][j] = (ok[u] && e < d) ? to_f(kp[base + e]) : 0.f;
        v[u][j] = (ok[u] && e < d) ? to_f(vp[base + e]) : 0.f;
      }
    }
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      if (h >= G) break;
      float sc[TOK];
#pragma unroll
      for (int u = 0; u < TOK; ++u) {
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < NPL; ++j) dot = fmaf(qv[h][j], k[u][j], dot);
        sc[u] = dot;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < TOK; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
      float mx = m[h];
#pragma unroll
      for (int u = 0; u < TOK; ++u)
        if (ok[u]) mx = fmaxf(mx, sc[u]);
      const float corr = exp2f(m[h] - mx);
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < NPL; ++j) o[h][j] *= corr;
#pragma unroll
      for (int u = 0; u < TOK; ++u) {
        const float p = ok[u] ? exp2f(sc[u] - mx) : 0.f;
        psum += p;
#pragma unroll
        for (int j = 0; j < NPL; ++j) o[h][j] = fmaf(p, v[u][j], o[h][j]);
      }
      l[h] = l[h] * corr + psum;
      m[h] = mx;
    }
  }
  // merge the warps: smem [warp][head] (m, l) and [warp][head][d]
  extern __shared__ float sm[];
  float* sml = sm;                          // SIMT_WARPS * G * 2
  float* so = sm + SIMT_WARPS * G * 2;      // SIMT_WARPS * G * d
#pragma unroll
  for (int h = 0; h < HP; ++h) {
    if (h >= G) break;
    if (lane == 0) {
      sml[(warp * G + h) * 2] = m[h];
      sml[(warp * G + h) * 2 + 1] = l[h];
    }
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + 32 * j;
      if (e < d) so[(warp * G + h) * d + e] = o[h][j];
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < G * d; k += blockDim.x) {
    const int h = k / d, e = k - h * d;
    float M = -INFINITY;
    for (int w = 0; w < SIMT_WARPS; ++w) M = fmaxf(M, sml[(w * G + h) * 2]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < SIMT_WARPS; ++w) {
        const float mw = sml[(w * G + h) * 2];
        if (mw == -INFINITY) continue;
        const float e2 = exp2f(mw - M);
        L += sml[(w * G + h) * 2 + 1] * e2;
        acc += so[(w * G + h) * d + e] * e2;
      }
    }
    out[h * d + e] = f_to<TA>(L > 0.f ? acc / L * a.v_mul : 0.f);
  }
}

// ---------------------------------------------------------------- host helpers (pkv_decode.cu)

// cuTensorMapEncodeTiled through the runtime's driver entry point (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
// Cached TMA descriptors of the K and V pools ({d_head, rows}, 16-token boxes, 128-byte swizzle).
int get_tensor_maps(Pool& P, const void* k, const void* v, CUtensorMap* tk, CUtensorMap* tv);
// Fields of DecodeArgs shared by every attention launch.
int fill_args(const Pool& P, int32_t layer, const void* q, void* out, const int32_t* tables, int32_t W,
              const int32_t* seq_lens, int32_t n_seq, float scale, DecodeArgs* a);
// The prefix kernel of a decode step with shared prefixes (pkv_prefill.cu): one CTA per (pair
// of 128-row tiles of the item's rows, KV head, work item); a carries share_items and prior_*.
// Launched as the programmatic dependent of the decode kernel just before it (it reads nothing
// that kernel writes, and waits for that grid only before it completes).
int launch_prefix_share(Pool& P, const DecodeArgs& a, const void* q, const void* k_pool, const void* v_pool,
                        int32_t n_items, int32_t max_members, cudaStream_t st);

}  // namespace pkv
