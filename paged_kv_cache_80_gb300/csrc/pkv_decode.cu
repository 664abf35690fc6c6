// Paged decode attention for one layer of a ragged batch.
//
// What it computes ("KV Cache Management", cs249r vol. 3 ch. 5, "The PagedAttention
// virtual memory model"; "PagedAttention", programmer.ie ch. 14, "It is the same
// function"): for sequence s and query head h (KV head g = floor(h / G)),
//   out[s][h] = sum_{t < len_s} softmax_t(scale * q[s][h] . K_s[t]) V_s[t],
//   K_s[t] = k_pool[T_s[floor(t / B)]][layer][g][t mod B].
// The kernel takes the block table and walks the sequence's logical blocks,
// fetching each physical block where it lies.
//
// Tensor-core path (bf16/f16, d_head 64 or 128, G <= 16, B a multiple of 16):
//   * One launch per call for up to 4,096 sequences: every CTA plans its own warps from
//     the lengths (tiles per sequence, their prefix, each warp's first tile); larger
//     batches launch a one-CTA plan kernel first, which the attention kernel follows
//     as its programmatic dependent.
//   * Work unit = a 16-token tile of one (sequence, KV head) pair: the K and V
//     slabs of 16 x d_head elements, contiguous in the pool.  All tiles of the
//     batch are laid end to end (sequence-major, then KV head) and cut into equal
//     contiguous ranges, one per warp of a persistent grid sized to the SM count
//     (stream-K style), so every warp reads the same number of bytes whatever the
//     length mix.
//   * Each warp runs its own S-stage pipeline: lane 0 issues TMA tensor loads of
//     the K and V tiles (128-byte swizzled boxes) and, at the first tile of a pair,
//     a bulk copy of the G query rows, completing on a per-stage mbarrier.
//   * One KV read serves all G query heads of the group: S^T = K q^T is one
//     m16n8k16 mma per 16 columns of d_head (M = 16 tokens, N = 8 heads), and
//     O^T += V^T P^T is one mma per 16 rows of d_head, with P^T moved from the
//     accumulator layout into the operand layout by movmatrix.
//   * Online softmax across tiles: running max m and normaliser l per head, the
//     accumulator rescaled by exp(m_prev - m_new) ("Chunked prefill mechanics":
//     m_new = max(m_prev, m_blk), l_new = l_prev e^{m_prev-m_new} + l_blk e^{m_blk-m_new},
//     O_new likewise), in base 2 with log2(e) folded into the scale.
//   * A pair fully inside one warp's range is normalised and written directly; a
//     pair split across warps leaves (m, l, O) partials.  At the end of its range a
//     warp publishes its partials and counts them (an epoch-tagged counter per split
//     pair, so the workspace needs no clearing); the warp that completes a pair's count
//     merges its partials with the same rule.
//   * Groups of 9 to 16 query heads run as two 8-head column blocks: every K / V
//     fragment feeds two mma.
// FP8 pools (E4M3 codes, "KV Cache Management" b_elem = 1): the same kernel with
//   16 x 128-byte tiles (one TMA box each); every lane reads its operand bytes with
//   16-byte shared loads and converts code pairs to binary16 (exact), so the mma
//   runs on f16 operands (q rounded to f16 once per pair).  The contraction index of
//   q K^T is permuted so that a lane's K bytes are contiguous (lane c of a quad owns
//   d = 32c .. 32c+31), and the d rows of V^T so that a lane's V bytes are (quad row
//   g owns d = 16g .. 16g+15); the k_scale is folded into the softmax scale and the
//   v_scale into the final normalisation.
// CUDA-core path (fp32, or other geometries): one CTA per (sequence, KV head),
// warps stride over tokens with an online softmax per head, then merge in smem.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pkv_attn.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kHdrBytes = 256;
constexpr int kPlanSmemInts = 8192;  // prefix entries the plan kernel keeps in shared memory
// --------------------------------------------------------------------------- plan

__device__ __forceinline__ int run_total_from(const DecodeArgs& a) { return *const_cast<volatile int32_t*>(a.hdr); }

// The keys of sequence s that this kernel attends to: `len` tokens from table block `kb` on.
// kb is the shared prefix's block count (share[s].x) when one is given and leaves at least one
// token, else 0 (an out-of-range value is recorded and ignored); len is the length clamped to
// the table's capacity [0, W*B], minus the prefix.  `record` reports bad values.
struct Span {
  int32_t len, kb;
};
__device__ __forceinline__ Span seq_span(const DecodeArgs& a, int s, bool record) {
  int32_t len = a.seq_lens[s];
  const int64_t maxlen = static_cast<int64_t>(a.W) * a.B;
  if (len < 0 || len > maxlen) {
    if (record) record_error(a.err, DERR_DECODE_LEN, s);
    len = len < 0 ? 0 : static_cast<int32_t>(maxlen);
  }
  int32_t kb = 0;
  if (a.share) {
    kb = a.share[s].x;
    if (kb < 0 || static_cast<int64_t>(kb) * a.B >= len) {
      if (record && kb != 0) record_error(a.err, DERR_SHARE, s);
      kb = 0;
    }
  }
  return Span{len - kb * a.B, kb};
}
__device__ __forceinline__ int32_t clamped_len(const DecodeArgs& a, int s, bool record) {
  return seq_span(a, s, record).len;
}

// One CTA: clamp lengths, tiles per sequence, exclusive prefix, total tile count.
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeArgs a) {
  // let the attention kernel launch now; it waits for this grid before reading its outputs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int32_t warp_sums[32];
  const int tid = threadIdx.x;
  const int per = (a.n_seq + blockDim.x - 1) / blockDim.x;
  const int s0 = min(a.n_seq, tid * per), s1 = min(a.n_seq, s0 + per);
  int32_t local = 0;
  for (int s = s0; s < s1; ++s) {
    const int32_t len = seq_span(a, s, true).len;
    a.lens_c[s] = len;
    local += (len + TILE - 1) / TILE;
  }
  // block-wide exclusive scan of `local`
  const int lane = tid & 31, warp = tid >> 5;
  int32_t incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < (blockDim.x >> 5) ? warp_sums[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int32_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int32_t run = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - local;
  for (int s = s0; s < s1; ++s) {
    a.tile_prefix[s] = run;
    run += (a.lens_c[s] + TILE - 1) / TILE;
  }
  if (tid == blockDim.x - 1) {
    a.tile_prefix[a.n_seq] = run;
    a.hdr[0] = run * a.H_kv;
  }
  // an empty sequence attends to nothing: zero output (16-byte stores; H_q*D*b is a multiple of 16)
  const int row16 = a.H_q * a.D * a.elem / 16;
  for (int s = s0; s < s1; ++s)
    if (a.lens_c[s] == 0)
      for (int k = 0; k < row16; ++k)
        reinterpret_cast<int4*>(static_cast<char*>(a.out) + static_cast<int64_t>(s) * row16 * 16)[k] =
            make_int4(0, 0, 0, 0);
  __syncthreads();  // the prefix array is complete (global writes of this block are visible)
  // the prefix in shared memory for the searches below, when it fits
  extern __shared__ int32_t q_smem[];
  const bool in_smem = a.n_seq + 1 <= kPlanSmemInts;
  if (in_smem)
    for (int k = tid; k <= a.n_seq; k += blockDim.x) q_smem[k] = a.tile_prefix[k];
  __syncthreads();
  const int32_t* Qp = in_smem ? q_smem : a.tile_prefix;
  // each warp's first tile: sequence s (largest with H_kv*Q[s] <= start), KV head, tile, tiles of pair
  const int total = run_total_from(a);
  const int R = (total + a.total_warps - 1) / a.total_warps;
  for (int w = tid; w < a.total_warps; w += blockDim.x) {
    const int start = w * R;
    if (start >= total) {
      a.wstart[w] = make_int4(-1, 0, 0, 0);
      continue;
    }
    int lo = 0, hi = a.n_seq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.H_kv * Qp[mid] <= start) lo = mid; else hi = mid - 1;
    }
    const int nt = Qp[lo + 1] - Qp[lo];
    const int within = start - a.H_kv * Qp[lo];
    a.wstart[w] = make_int4(lo, within / nt, within - (within / nt) * nt, nt);
  }
}

// --------------------------------------------------------------------------- in-kernel plan

// Sequences up to which every CTA of the attention kernel plans its own warps (no plan kernel).
constexpr int kSelfPlanMaxSeqs = 4096;


// The plan kernel's work for this CTA's NW warps only, from the lengths: tiles per
// sequence, their block-wide exclusive prefix, the total, and each warp's first tile
// (sequence, KV head, tile, tiles of the pair) with the prefix of its sequence.  Every
// CTA reads all n_seq lengths (n_seq <= kSelfPlanMaxSeqs) and gets the same total; the
// thread whose chunk of sequences holds a warp's start finds it.  CTA 0 records bad
// lengths; CTA (s mod grid) zeroes the output of an empty sequence s.  Ends with a CTA
// barrier, so it is called by every thread before any warp leaves.
template <int NW>
__device__ void self_plan(const DecodeArgs& a, int4* s_start, int32_t* s_q, int32_t* s_total) {
  __shared__ int32_t wsum[NW];
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.n_seq + NT - 1) / NT;
  const int s0 = min(a.n_seq, tid * per), s1 = min(a.n_seq, s0 + per);
  const int row16 = a.H_q * a.D * a.elem / 16;
  int32_t local = 0;
  for (int s = s0; s < s1; ++s) {
    const int32_t len = clamped_len(a, s, blockIdx.x == 0);
    local += (len + TILE - 1) / TILE;
    if (len == 0 && s % gridDim.x == blockIdx.x)  // an empty sequence attends to nothing: zero output
      for (int k = 0; k < row16; ++k)
        reinterpret_cast<int4*>(static_cast<char*>(a.out) + static_cast<int64_t>(s) * row16 * 16)[k] =
            make_int4(0, 0, 0, 0);
  }
  int32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    before += w < warp ? wsum[w] : 0;
    tot += wsum[w];
  }
  const int32_t excl = before + incl - local;
  const int total = tot * a.H_kv;
  const int R = (total + a.total_warps - 1) / a.total_warps;
#pragma unroll 1
  for (int w = 0; w < NW; ++w) {
    const int start = (blockIdx.x * NW + w) * R;
    if (start >= total) {
      if (tid == 0) s_start[w] = make_int4(-1, 0, 0, 0);
    } else if (local > 0 && a.H_kv * excl <= start && start < a.H_kv * (excl + local)) {
      int32_t q = excl;
      for (int s = s0; s < s1; ++s) {
        const int nt = (clamped_len(a, s, false) + TILE - 1) / TILE;
        if (a.H_kv * (q + nt) > start) {
          const int within = start - a.H_kv * q;
          s_start[w] = make_int4(s, within / nt, within - (within / nt) * nt, nt);
          s_q[w] = q;
          break;
        }
        q += nt;
      }
    }
  }
  if (tid == 0) *s_total = total;
  __syncthreads();
}

// --------------------------------------------------------------------------- tensor-core path

// EB: bytes per stored K/V element; NB: 8-head column blocks of the mma N dimension (1 for
// G <= 8, 2 for 9 <= G <= 16: every K/V fragment loaded from shared memory feeds NB mmas).
template <int D, int EB = 2, int NB = 1>
struct TcCfg {
  static constexpr int GP = GPAD * NB;                     // query rows held per group (padded)
  static constexpr int KV_TILE_BYTES = TILE * D * EB;     // one 16 x D tile of K (or V)
  static constexpr int Q_BYTES = GP * D * 2;               // up to GP query rows (16-bit)
  static constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES + Q_BYTES;
  static constexpr int NBOX = D * EB / 128;                // 128-byte TMA boxes per tile row
  static constexpr int BOX_ELEMS = 128 / EB;
  static constexpr int NKC = D / 16;                       // 16-wide chunks of d_head
  static constexpr int OFL = NKC * 32 * 4;                 // floats of one head block's O^T fragments
  // floats per partial slot: the O^T fragments of each head block, then m[GP], then l[GP]
  static constexpr int PSTRIDE = NB * OFL + 2 * GP;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment for the swizzle");
};

template <int D, int EB, int S, int NW, int NB = 1>
struct TcSmem {
  static constexpr int WARP_BYTES = S * TcCfg<D, EB, NB>::STAGE_BYTES + 64 * 16 + S * 8 + 8;
  static constexpr int WARP_STRIDE = (WARP_BYTES + 1023) / 1024 * 1024;
  static constexpr int TOTAL = NW * WARP_STRIDE + 1024;  // + alignment slack
};

// Four E4M3 codes (bytes 0..3 of w) to binary16 pairs (exact): lo = (b0, b1), hi = (b2, b3),
// the first of each pair in the low half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two bfloat16 values (low half first) to two binary16 values (round to nearest).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Write the G output rows of one (sequence, KV head) pair from a lane's accumulator
// fragment acc[c] (the O^T fragment of d-chunk c), scaled by i0 (head h0) and i1
// (head h0 + 1).  16-bit pools: chunk c, quad row r holds d = 16c + r (x, y) and
// d + 8 (z, w).  FP8 pools: quad row r holds d = 16r + 2c (x, y) and d + 1 (z, w),
// so a lane has 16 consecutive d of its two heads (two 16-byte stores per head).
template <typename TO, int D, bool F8>
__device__ __forceinline__ void store_group(TO* out, const float4 (&acc)[D / 16], float i0, float i1, int lane,
                                            int G) {
  const int h0 = 2 * (lane & 3), trow = lane >> 2;
  if constexpr (F8) {
    static_assert(D == 128, "FP8 tiles are 128 bytes wide");
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (h0 + hh >= G) continue;
      const float sc = hh ? i1 : i0;
      uint32_t w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        __nv_bfloat162 v = __floats2bfloat162_rn((hh ? acc[c].y : acc[c].x) * sc, (hh ? acc[c].w : acc[c].z) * sc);
        w[c] = *reinterpret_cast<uint32_t*>(&v);
      }
      uint4* dst = reinterpret_cast<uint4*>(out + (h0 + hh) * D + 16 * trow);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const int dd = 16 * c + trow;
      if (h0 < G) {
        out[h0 * D + dd] = from_float<TO>(acc[c].x * i0);
        out[h0 * D + dd + 8] = from_float<TO>(acc[c].z * i0);
      }
      if (h0 + 1 < G) {
        out[(h0 + 1) * D + dd] = from_float<TO>(acc[c].y * i1);
        out[(h0 + 1) * D + dd + 8] = from_float<TO>(acc[c].w * i1);
      }
    }
  }
}

// A row with a shared prefix (share[s].x blocks attended by the prefix kernel): the decode
// kernel's part of its attention, head block nb of KV head g, is left as a partial for the
// combine kernel -- acc (O^T fragments in store_group's element layout, relative to 2^M) and
// (M, L) per head of the lane (M0, L0: head h0; M1, L1: h0 + 1).  Returns false, writing
// nothing, for a row without one.
template <int D, bool F8>
__device__ __forceinline__ bool leave_partial(const DecodeArgs& a, int s, int g, int nb, int lane,
                                              const float4 (&acc)[D / 16], float M0, float M1, float L0, float L1) {
  if (!a.share || seq_span(a, s, false).kb == 0) return false;
  const int h0 = 2 * (lane & 3), trow = lane >> 2;
  const int hl = GPAD * nb + h0;  // the lane's first head within the group
  const bool live0 = hl < a.G, live1 = hl + 1 < a.G;
  const int64_t row = static_cast<int64_t>(s) * a.H_q + static_cast<int64_t>(g) * a.G + hl;
  float* o0 = a.sfx_o + row * D;
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    // 16-bit pools: d = 16c + trow (x, y) and + 8 (z, w); FP8 pools: d = 16 trow + 2c (x, y) and
    // + 1 (z, w); x, z head h0 and y, w head h0 + 1
    const int da = F8 ? 16 * trow + 2 * c : 16 * c + trow;
    const int db = F8 ? da + 1 : da + 8;
    if (live0) {
      o0[da] = acc[c].x;
      o0[db] = acc[c].z;
    }
    if (live1) {
      o0[D + da] = acc[c].y;
      o0[D + db] = acc[c].w;
    }
  }
  if (trow == 0) {
    if (live0) *reinterpret_cast<float2*>(a.sfx_ml + 2 * row) = make_float2(M0, L0);
    if (live1) *reinterpret_cast<float2*>(a.sfx_ml + 2 * row + 2) = make_float2(M1, L1);
  }
  return true;
}

// Merge the partials of one split pair (contributing warps wa..wb) and write its
// G output rows.  Run by one whole warp; lane l owns float4 l of every d-chunk of
// each head block, merged one block at a time.  Partials are read through L2
// (ld.global.cg): other SMs wrote them.
template <typename TO, int D, bool F8, int NB>
__device__ __forceinline__ void merge_pair(const DecodeArgs& a, int s, int g, int pbeg, int wa, int wb, int R,
                                           int lane) {
  using C = TcCfg<D, 2, NB>;
  const int h0 = 2 * (lane & 3);
  TO* out = static_cast<TO*>(a.out) + (static_cast<int64_t>(s) * a.H_q + g * a.G) * D;
#pragma unroll 1
  for (int nb = 0; nb < NB; ++nb) {
    if (GPAD * nb >= a.G) break;
    const int hm = NB * C::OFL + GPAD * nb + h0;  // m of heads h0, h0 + 1 of this block; l is GP further
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float4 acc[C::NKC];
#pragma unroll
    for (int c = 0; c < C::NKC; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    // two contributors per round: all their loads are issued before any use
    for (int w = wa; w <= wb; w += 2) {
      const bool two = w + 1 <= wb;
      const float* p0 =
          a.partials + static_cast<int64_t>(w * 2 + ((w == wa && pbeg != wa * R) ? 1 : 0)) * C::PSTRIDE;
      const float* p1 = two ? a.partials + static_cast<int64_t>((w + 1) * 2) * C::PSTRIDE : p0;
      const float ma0 = __ldcg(p0 + hm), ma1 = __ldcg(p0 + hm + 1);
      const float la0 = __ldcg(p0 + hm + C::GP), la1 = __ldcg(p0 + hm + C::GP + 1);
      float mb0 = __ldcg(p1 + hm), mb1 = __ldcg(p1 + hm + 1);
      const float lb0 = __ldcg(p1 + hm + C::GP), lb1 = __ldcg(p1 + hm + C::GP + 1);
      float4 va[C::NKC], vb[C::NKC];
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        va[c] = __ldcg(reinterpret_cast<const float4*>(p0 + nb * C::OFL) + c * 32 + lane);
        vb[c] = __ldcg(reinterpret_cast<const float4*>(p1 + nb * C::OFL) + c * 32 + lane);
      }
      if (!two) mb0 = mb1 = -INFINITY;
      const float n0 = fmaxf(M0, fmaxf(ma0, mb0)), n1 = fmaxf(M1, fmaxf(ma1, mb1));
      const float r0 = exp2f(M0 - n0), r1 = exp2f(M1 - n1);
      const float ea0 = exp2f(ma0 - n0), ea1 = exp2f(ma1 - n1);
      const float eb0 = two ? exp2f(mb0 - n0) : 0.f, eb1 = two ? exp2f(mb1 - n1) : 0.f;
      L0 = L0 * r0 + la0 * ea0 + lb0 * eb0;
      L1 = L1 * r1 + la1 * ea1 + lb1 * eb1;
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        acc[c].x = acc[c].x * r0 + va[c].x * ea0 + vb[c].x * eb0;
        acc[c].y = acc[c].y * r1 + va[c].y * ea1 + vb[c].y * eb1;
        acc[c].z = acc[c].z * r0 + va[c].z * ea0 + vb[c].z * eb0;
        acc[c].w = acc[c].w * r1 + va[c].w * ea1 + vb[c].w * eb1;
      }
      M0 = n0;
      M1 = n1;
    }
    if (leave_partial<D, F8>(a, s, g, nb, lane, acc, M0, M1, L0, L1)) continue;
    const float i0 = a.v_mul / L0, i1 = a.v_mul / L1;
    store_group<TO, D, F8>(out + GPAD * nb * D, acc, i0, i1, lane, a.G - GPAD * nb);
  }
}

// The combine kernel of a decode step with shared prefixes: one warp per (row, query head) of
// the rows that have one, lane l holding d = 4l .. 4l + 3 (d_head 128).  It merges the decode
// kernel's partial of the row (its own blocks) with the prefix kernel's partials of the row (the
// splits of the shared blocks) by the online-softmax rule ("Chunked prefill mechanics": m the
// largest, each l and O scaled by 2^(m_part - m)) and writes O / l (times v_scale for an FP8 pool).
template <typename TO>
__global__ void __launch_bounds__(256) share_combine_kernel(const DecodeArgs a) {
  constexpr int D = 128;
  // launched as the programmatic dependent of the prefix kernel, which completes only after the
  // decode kernel has: it waits here until both grids' partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // (row, head)
  if (p >= static_cast<int64_t>(a.n_seq) * a.H_q) return;
  const int s = static_cast<int>(p / a.H_q);
  if (seq_span(a, s, false).kb == 0) return;  // written by the decode kernel
  const int4 sh = a.share[s];
  if (sh.y < 1 || sh.z < 0 || sh.w < 0 ||
      static_cast<int64_t>(sh.z) + static_cast<int64_t>(sh.y - 1) * sh.w >= a.prior_slots) {
    if (lane == 0 && p % a.H_q == 0) record_error(a.err, DERR_SHARE, s);
    return;
  }
  const int64_t hq = p % a.H_q;
  const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.sfx_ml) + p);
  float m = ml.x, l = ml.y;
  float4 o = __ldcg(reinterpret_cast<const float4*>(a.sfx_o + p * D) + lane);
  constexpr int K = 12;  // partials whose loads are in flight at once (a step's splits are usually fewer)
  for (int i0 = 0; i0 < sh.y; i0 += K) {
    float2 pm[K];
    float4 po[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (i0 + k < sh.y) {
        const int64_t row = (static_cast<int64_t>(sh.z) + static_cast<int64_t>(i0 + k) * sh.w) * a.H_q + hq;
        pm[k] = __ldcg(reinterpret_cast<const float2*>(a.prior_ml) + row);
        po[k] = __ldcg(reinterpret_cast<const float4*>(a.prior_o + row * D) + lane);
      } else {
        pm[k] = make_float2(-INFINITY, 0.f);
        po[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float mn = m;
#pragma unroll
    for (int k = 0; k < K; ++k) mn = fmaxf(mn, pm[k].x);
    const float r = exp2f(m - mn);
    l *= r;
    o.x *= r;
    o.y *= r;
    o.z *= r;
    o.w *= r;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float e = exp2f(pm[k].x - mn);  // 0 for the padding entries
      l += pm[k].y * e;
      o.x += po[k].x * e;
      o.y += po[k].y * e;
      o.z += po[k].z * e;
      o.w += po[k].w * e;
    }
    m = mn;
  }
  const float inv = a.v_mul / l;
  TO* out = static_cast<TO*>(a.out) + p * D + 4 * lane;
  *reinterpret_cast<uint2*>(out) = make_uint2(pack2<TO>(o.x * inv, o.y * inv), pack2<TO>(o.z * inv, o.w * inv));
}

// Descriptor of one tile, built by the warp a batch at a time:
//   x = TMA row coordinate of the slab, y = pair id (s * H_kv + g),
//   z = valid tokens | first-of-pair << 8 | last-of-pair << 9 | new-pair-in-range << 10,
//   w = tiles of the sequences before s (the pair's place in the batch's tile order).
constexpr int F_FIRST = 1 << 8, F_LAST = 1 << 9, F_NEWPAIR = 1 << 10;

template <typename T, int D, int S, int NW, int NB>
__global__ void __launch_bounds__(NW * 32) decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                                                            const __grid_constant__ CUtensorMap tmv,
                                                            const DecodeArgs a) {
  // T = stored K/V element; TA = q / out element; TM = mma operand type
  constexpr bool F8 = std::is_same<T, E4M3>::value;
  using TA = typename std::conditional<F8, __nv_bfloat16, T>::type;
  using TM = typename std::conditional<F8, __half, T>::type;
  constexpr bool BF16 = std::is_same<TM, __nv_bfloat16>::value;
  constexpr int EB = F8 ? 1 : 2;
  using C = TcCfg<D, EB, NB>;
  using SM = TcSmem<D, EB, S, NW, NB>;
  extern __shared__ uint8_t smem_raw[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * NW + warp;
  // a programmatic dependent launched after this grid (the prefix kernel of a step with shared
  // prefixes) may become resident now; it reads nothing this grid writes, and waits for this
  // grid before it completes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* region = base + warp * SM::WARP_STRIDE;
  int4* desc = reinterpret_cast<int4*>(region + S * C::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(region + S * C::STAGE_BYTES + 64 * 16);
  const uint32_t stage0 = smem_u32(region);

  auto init_barriers = [&] {
    if (lane == 0) {
      for (int st = 0; st < S; ++st) mbar_init(bar0 + 8 * st, 1);
      fence_barrier_init();
    }
    __syncwarp();
  };

  // ---- this warp's range of the batch's tiles and its first tile: planned here by every CTA
  // (small batches), or read from the plan kernel, which this kernel then follows as a
  // programmatic dependent (everything above overlaps it).  A self-planning launch may itself
  // follow a decode step's append kernel as a programmatic dependent: it reads only lengths and
  // tables before its first tile load, and waits for the append's grid just before that load.
  __shared__ int4 s_start[NW];
  __shared__ int32_t s_q[NW];
  __shared__ int32_t s_total;
  int total, cq;
  int4 w0;
  if (a.self_plan) {
    self_plan<NW>(a, s_start, s_q, &s_total);
    init_barriers();  // after the plan's loads, which need no barrier
    total = s_total;
    w0 = s_start[warp];
    cq = s_q[warp];
  } else {
    init_barriers();  // while the plan kernel runs
    asm volatile("griddepcontrol.wait;" ::: "memory");
    total = a.hdr[0];
    w0 = a.wstart[gw];
    cq = w0.x >= 0 ? a.tile_prefix[w0.x] : 0;
  }
  const int R = (total + a.total_warps - 1) / a.total_warps;
  const int my_start = gw * R;
  const int my_end = min(total, my_start + R);
  if (my_start >= my_end) return;  // the whole warp leaves; no block-level barriers follow
  const int n_my = my_end - my_start;

  // ---- tile walk state: (sequence, KV head, tile within pair, tiles of the pair, tiles before
  // the sequence)
  int cs = w0.x, ch = w0.y, cj = w0.z, cn = w0.w;
  auto tiles_of = [&](int s) { return (clamped_len(a, s, false) + TILE - 1) / TILE; };

  // Fill descriptors for range tiles [t0, t0 + 32) into ring slots (t & 63).
  auto fill = [&](int t0) {
    int ss = cs, hh = ch, jj = cj + lane, nn = cn, qq = cq;
    while (jj >= nn && ss < a.n_seq) {
      jj -= nn;
      if (++hh == a.H_kv) {
        hh = 0;
        qq += nn;
        ++ss;
        nn = ss < a.n_seq ? tiles_of(ss) : 0;
      }
    }
    const int t = t0 + lane;
    if (t < n_my) {
      const int tok0 = jj * TILE;
      const int lb = tok0 / a.B;
      const int sub = tok0 - lb * a.B;
      const Span sp = seq_span(a, ss, false);
      int blk = a.tables[static_cast<int64_t>(ss) * a.W + sp.kb + lb];
      if (blk < 0 || blk >= a.num_blocks) {
        record_error(a.err, DERR_DECODE_BLOCK, blk);
        blk = 0;
      }
      const int valid = min(TILE, sp.len - tok0);
      int flags = valid;
      if (jj == 0) flags |= F_FIRST;
      if (jj == nn - 1) flags |= F_LAST;
      if (jj == 0 || t == 0) flags |= F_NEWPAIR;
      const int row = ((blk * a.L + a.layer) * a.H_kv + hh) * a.B + sub;
      desc[t & 63] = make_int4(row, ss * a.H_kv + hh, flags, qq);
    }
    // carry = position of tile t0 + 32 (one past lane 31's tile)
    int ns = __shfl_sync(0xffffffffu, ss, 31), nh = __shfl_sync(0xffffffffu, hh, 31);
    int nj = __shfl_sync(0xffffffffu, jj, 31) + 1, nnn = __shfl_sync(0xffffffffu, nn, 31);
    int nq = __shfl_sync(0xffffffffu, qq, 31);
    while (nj >= nnn && ns < a.n_seq) {
      nj -= nnn;
      if (++nh == a.H_kv) {
        nh = 0;
        nq += nnn;
        ++ns;
        nnn = ns < a.n_seq ? tiles_of(ns) : 0;
      }
    }
    cs = ns; ch = nh; cj = nj; cn = nnn; cq = nq;
    __syncwarp();
  };

  auto issue = [&](int t) {  // lane 0 only
    const int4 d = desc[t & 63];
    const int st = t % S;
    const uint32_t bar = bar0 + 8 * st;
    const uint32_t sk = stage0 + st * C::STAGE_BYTES;
    const uint32_t sv = sk + C::KV_TILE_BYTES;
    const bool newpair = d.z & F_NEWPAIR;
    fence_proxy_async();
    mbar_arrive_expect_tx(bar, 2 * C::KV_TILE_BYTES + (newpair ? a.G * D * 2 : 0));
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) {
      tma_load_2d(sk + b * (TILE * 128), &tmk, b * C::BOX_ELEMS, d.x, bar);
      tma_load_2d(sv + b * (TILE * 128), &tmv, b * C::BOX_ELEMS, d.x, bar);
    }
    if (newpair) {
      const int s = d.y / a.H_kv, g = d.y - (d.y / a.H_kv) * a.H_kv;
      const TA* qsrc = static_cast<const TA*>(a.q) + (static_cast<int64_t>(s) * a.H_q + g * a.G) * D;
      bulk_load(sk + 2 * C::KV_TILE_BYTES, qsrc, a.G * D * 2, bar);
    }
  };

  fill(0);
  if (n_my > 32) fill(32);
  if (a.self_plan) asm volatile("griddepcontrol.wait;" ::: "memory");  // the append's K/V are written
  if (lane == 0)
    for (int t = 0; t < S && t < n_my; ++t) issue(t);

  // per-lane ldmatrix geometry (128-byte swizzle: chunk c of row r sits at c ^ (r & 7))
  const int r8 = lane & 7, mi = lane >> 3;
  const int k_row = r8 + 8 * (mi & 1), k_add = mi >> 1;  // QK: A = K tile (t x d)
  const int v_row = r8 + 8 * (mi >> 1), v_add = mi & 1;  // PV: A = V^T via .trans
  const int h0 = 2 * (lane & 3);                         // heads of this lane's columns
  const int trow = lane >> 2;                            // token row of c0/c1 (c2/c3: +8)
  const int c4 = lane & 3;

  // per head block nb: O^T fragments, q fragments, running max and sum of heads 8nb + h0, 8nb + h0 + 1
  float o[NB][C::NKC][4];
  uint32_t qf[NB][C::NKC][2];
  float m[NB][2], l[NB][2];
  int cur_pair = -1;
  bool cur_started = false, cur_first_in_range = false;
  // split pairs whose partial this warp wrote: one that ended inside the range, one at its end
  int pend_pair = -1, pend_pbeg = 0, pend_nt = 0, end_pair = -1, end_pbeg = 0, end_nt = 0;

  for (int i = 0; i < n_my; ++i) {
    if (i >= 32 && (i & 31) == 0 && i + 32 < n_my) fill(i + 32);
    const int4 d = desc[i & 63];
    const int st = i % S;
    const uint32_t sk = stage0 + st * C::STAGE_BYTES;
    const uint32_t sv = sk + C::KV_TILE_BYTES;
    if (!mbar_wait_bounded(bar0 + 8 * st, (i / S) & 1, kWaitNs)) {
      if (lane == 0) record_error(a.err, DERR_DECODE_TIMEOUT, i);
      // drain the other stages' loads (bounded) before leaving
      for (int k = 1; k < S && i + k < n_my; ++k)
        mbar_wait_bounded(bar0 + 8 * ((i + k) % S), ((i + k) / S) & 1, kWaitNs);
      return;
    }

    if (d.z & F_NEWPAIR) {
      cur_pair = d.y;
      cur_started = d.z & F_FIRST;
      cur_first_in_range = (i == 0);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        m[nb][0] = m[nb][1] = -INFINITY;
        l[nb][0] = l[nb][1] = 0.f;
#pragma unroll
        for (int c = 0; c < C::NKC; ++c) o[nb][c][0] = o[nb][c][1] = o[nb][c][2] = o[nb][c][3] = 0.f;
        const uint8_t* qs = region + st * C::STAGE_BYTES + 2 * C::KV_TILE_BYTES;
        const int hq = trow + GPAD * nb;  // this lane's query row (B-operand column) in block nb
        const bool live = hq < a.G;
        if constexpr (F8) {
          // step c of q K^T covers d = 32 c4 + 4c .. +3: (b0, b1) the first two, (b2, b3) the last two
#pragma unroll
          for (int c = 0; c < C::NKC; ++c) {
            const uint2 w = *reinterpret_cast<const uint2*>(qs + (hq * D + (D / 4) * c4 + 4 * c) * 2);
            qf[nb][c][0] = live ? bf16x2_to_f16x2(w.x) : 0u;
            qf[nb][c][1] = live ? bf16x2_to_f16x2(w.y) : 0u;
          }
        } else {
#pragma unroll
          for (int c = 0; c < C::NKC; ++c) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(qs + hq * D * 2 + (16 * c + h0) * 2);
            qf[nb][c][0] = live ? p[0] : 0u;
            qf[nb][c][1] = live ? p[4] : 0u;
          }
        }
      }
    }

    // ---- S^T = K q^T  (16 tokens x 8 heads per block), two accumulation chains per block
    float sa[NB][4], sb[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int r = 0; r < 4; ++r) sa[nb][r] = sb[nb][r] = 0.f;
    if constexpr (F8) {
      // K rows trow and trow + 8, bytes 32 c4 .. 32 c4 + 31 (16-byte chunks 2c4, 2c4 + 1; swizzle
      // XOR = row & 7 = trow); step c takes bytes 4c .. 4c + 3 of each row
      const uint4 ka0 = lds128(sk + trow * 128 + (((2 * c4) ^ trow) << 4));
      const uint4 ka1 = lds128(sk + trow * 128 + (((2 * c4 + 1) ^ trow) << 4));
      const uint4 kb0 = lds128(sk + (trow + 8) * 128 + (((2 * c4) ^ trow) << 4));
      const uint4 kb1 = lds128(sk + (trow + 8) * 128 + (((2 * c4 + 1) ^ trow) << 4));
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        const uint32_t wa = word_of(c < 4 ? ka0 : ka1, c & 3), wb = word_of(c < 4 ? kb0 : kb1, c & 3);
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(wa, a0, a2);
        e4m3x4_to_f16x2x2(wb, a1, a3);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          if (c & 1) mma_16816<BF16>(sb[nb], a0, a1, a2, a3, qf[nb][c][0], qf[nb][c][1]);
          else mma_16816<BF16>(sa[nb], a0, a1, a2, a3, qf[nb][c][0], qf[nb][c][1]);
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        const int chunk = 2 * (c & 3) + k_add;
        const uint32_t addr = sk + (c >> 2) * (TILE * 128) + k_row * 128 + ((chunk ^ r8) << 4);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          if (c & 1) mma_16816<BF16>(sb[nb], a0, a1, a2, a3, qf[nb][c][0], qf[nb][c][1]);
          else mma_16816<BF16>(sa[nb], a0, a1, a2, a3, qf[nb][c][0], qf[nb][c][1]);
        }
      }
    }
    float sc[NB][4];  // scores (base-2 logits): c0, c1 token trow, heads h0, h0 + 1; c2, c3 token trow + 8
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int r = 0; r < 4; ++r) sc[nb][r] = (sa[nb][r] + sb[nb][r]) * a.scale_log2;
    const int valid = d.z & 0xff;
    if (valid < TILE) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if (trow >= valid) sc[nb][0] = sc[nb][1] = -INFINITY;
        if (trow + 8 >= valid) sc[nb][2] = sc[nb][3] = -INFINITY;
      }
      // zero the V rows past the end so that 0 * (stale value) cannot make NaN
      uint8_t* vrows = region + st * C::STAGE_BYTES + C::KV_TILE_BYTES;
      for (int k = lane; k < (TILE - valid) * 8 * C::NBOX; k += 32) {
        const int b = k / ((TILE - valid) * 8);
        const int rem = k - b * (TILE - valid) * 8;
        const int r = valid + rem / 8, c16 = rem & 7;
        *reinterpret_cast<int4*>(vrows + b * (TILE * 128) + r * 128 + c16 * 16) = make_int4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // ---- online softmax over this tile (per head: columns h0, h0 + 1 of each block)
    uint32_t pb[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float x0 = fmaxf(sc[nb][0], sc[nb][2]), x1 = fmaxf(sc[nb][1], sc[nb][3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      const float n0 = fmaxf(m[nb][0], x0), n1 = fmaxf(m[nb][1], x1);
      const float c0 = exp2f(m[nb][0] - n0), c1 = exp2f(m[nb][1] - n1);
      m[nb][0] = n0;
      m[nb][1] = n1;
      const float p0 = exp2f(sc[nb][0] - n0), p2 = exp2f(sc[nb][2] - n0);
      const float p1 = exp2f(sc[nb][1] - n1), p3 = exp2f(sc[nb][3] - n1);
      l[nb][0] = l[nb][0] * c0 + (p0 + p2);
      l[nb][1] = l[nb][1] * c1 + (p1 + p3);
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        o[nb][c][0] *= c0;
        o[nb][c][1] *= c1;
        o[nb][c][2] *= c0;
        o[nb][c][3] *= c1;
      }
      // P^T (16 tokens x 8 heads) from the accumulator layout into the B-operand layout
      pb[nb][0] = movmatrix_trans(pack2<TM>(p0, p1));
      pb[nb][1] = movmatrix_trans(pack2<TM>(p2, p3));
    }

    // ---- O^T += V^T P^T  (d_head x 8 heads per block)
    if constexpr (F8) {
      // token rows 2c4, 2c4 + 1, 2c4 + 8, 2c4 + 9, bytes 16 trow .. 16 trow + 15 of each (chunk trow;
      // swizzle XOR = row & 7); step c takes d = 16 trow + 2c (A rows trow) and + 1 (rows trow + 8)
      const int r0 = 2 * c4;
      const uint4 v0 = lds128(sv + r0 * 128 + ((trow ^ r0) << 4));
      const uint4 v1 = lds128(sv + (r0 + 1) * 128 + ((trow ^ (r0 + 1)) << 4));
      const uint4 v2 = lds128(sv + (r0 + 8) * 128 + ((trow ^ r0) << 4));
      const uint4 v3 = lds128(sv + (r0 + 9) * 128 + ((trow ^ (r0 + 1)) << 4));
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        // bytes 2c, 2c + 1 of the 16: word c / 2, byte 2 (c & 1); interleave tokens (2c4, 2c4 + 1)
        const unsigned sel = (c & 1) ? 0x7362u : 0x5140u;
        const uint32_t x = __byte_perm(word_of(v0, c >> 1), word_of(v1, c >> 1), sel);
        const uint32_t y = __byte_perm(word_of(v2, c >> 1), word_of(v3, c >> 1), sel);
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(x, a0, a1);
        e4m3x4_to_f16x2x2(y, a2, a3);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_16816<BF16>(o[nb][c], a0, a1, a2, a3, pb[nb][0], pb[nb][1]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < C::NKC; ++c) {
        const int chunk = 2 * (c & 3) + v_add;
        const uint32_t addr = sv + (c >> 2) * (TILE * 128) + v_row * 128 + ((chunk ^ r8) << 4);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_16816<BF16>(o[nb][c], a0, a1, a2, a3, pb[nb][0], pb[nb][1]);
      }
    }

    __syncwarp();  // every lane is done with this stage
    if (lane == 0 && i + S < n_my) issue(i + S);

    // ---- end of this pair within the range: write the result or a partial
    if ((d.z & F_LAST) || i == n_my - 1) {
      float Ls[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        float L0 = l[nb][0], L1 = l[nb][1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          L0 += __shfl_xor_sync(0xffffffffu, L0, off);
          L1 += __shfl_xor_sync(0xffffffffu, L1, off);
        }
        Ls[nb][0] = L0;
        Ls[nb][1] = L1;
      }
      const int s = cur_pair / a.H_kv, g = cur_pair - (cur_pair / a.H_kv) * a.H_kv;
      if (cur_started && (d.z & F_LAST)) {
        TA* out = static_cast<TA*>(a.out) + (static_cast<int64_t>(s) * a.H_q + g * a.G) * D;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          if (GPAD * nb >= a.G) break;
          float4 acc4[C::NKC];
#pragma unroll
          for (int c = 0; c < C::NKC; ++c) acc4[c] = make_float4(o[nb][c][0], o[nb][c][1], o[nb][c][2], o[nb][c][3]);
          if (leave_partial<D, F8>(a, s, g, nb, lane, acc4, m[nb][0], m[nb][1], Ls[nb][0], Ls[nb][1])) continue;
          const float i0 = a.v_mul / Ls[nb][0], i1 = a.v_mul / Ls[nb][1];
          store_group<TA, D, F8>(out + GPAD * nb * D, acc4, i0, i1, lane, a.G - GPAD * nb);
        }
      } else {
        const int slot = cur_first_in_range ? 0 : 1;
        float* ps = a.partials + static_cast<int64_t>(gw * 2 + slot) * C::PSTRIDE;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
          for (int c = 0; c < C::NKC; ++c)
            reinterpret_cast<float4*>(ps + nb * C::OFL)[c * 32 + lane] =
                make_float4(o[nb][c][0], o[nb][c][1], o[nb][c][2], o[nb][c][3]);
          if (lane < 4) {
            const int hm = NB * C::OFL + GPAD * nb + h0;
            ps[hm] = m[nb][0];
            ps[hm + 1] = m[nb][1];
            ps[hm + C::GP] = Ls[nb][0];
            ps[hm + C::GP + 1] = Ls[nb][1];
          }
        }
        // this warp's share of a split pair: arrive at the pair's counter once the range is done
        // (a pair that ends before the range does waits there, so no fence stalls the tiles)
        const int nt = tiles_of(s);
        const int pbeg = a.H_kv * d.w + g * nt;
        if (i != n_my - 1) {
          pend_pair = cur_pair;
          pend_pbeg = pbeg;
          pend_nt = nt;
        } else {
          end_pair = cur_pair;
          end_pbeg = pbeg;
          end_nt = nt;
        }
      }
    }
  }

  // ---- end of the range: publish this warp's partials, count them, merge what is complete.
  // The warp that writes a split pair's last partial merges it ("Chunked prefill mechanics"
  // rule): publish (the warp barrier orders every lane's writes before lane 0's cumulative
  // fence), count, and let the last arrival read everyone's.  The pair's counter is that of
  // the first warp of its range (a warp's range ends with at most one split pair), tagged
  // with this launch's epoch: a word left by an earlier launch (or never written) counts as
  // no arrival.
  if (pend_pair >= 0 || end_pair >= 0) {
    __syncwarp();
    if (lane < 2) __threadfence();
    // lane 0 counts the pair that ended inside the range, lane 1 the one at its end, at once
    const int pair = lane == 0 ? pend_pair : end_pair;
    const int pbeg = lane == 0 ? pend_pbeg : end_pbeg, nt = lane == 0 ? pend_nt : end_nt;
    int last = 0;
    if (lane < 2 && pair >= 0) {
      const int wa = pbeg / R, wb = (pbeg + nt - 1) / R;
      unsigned long long* c = a.counters + wa;
      // first guess: every other contributor is in (right for the last one, which merges, so its
      // count takes one atomic); a wrong guess returns the word and the loop goes on from it
      unsigned long long cur = (a.epoch << 16) | static_cast<unsigned long long>(wb - wa);
      for (;;) {
        const bool ours = (cur >> 16) == a.epoch;
        const unsigned long long prev = atomicCAS(c, cur, ours ? cur + 1 : ((a.epoch << 16) | 1ull));
        if (prev == cur) {
          last = (ours ? static_cast<int>(cur & 0xffffull) : 0) == wb - wa;
          break;
        }
        cur = prev;
      }
    }
    const unsigned lasts = __ballot_sync(0xffffffffu, last);
    if (lasts) __threadfence();
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
      if (!(lasts & (1u << k))) continue;
      const int p = k == 0 ? pend_pair : end_pair;
      const int pb = k == 0 ? pend_pbeg : end_pbeg, n_t = k == 0 ? pend_nt : end_nt;
      const int s = p / a.H_kv, g = p - (p / a.H_kv) * a.H_kv;
      merge_pair<TA, D, F8, NB>(a, s, g, pb, pb / R, (pb + n_t - 1) / R, R, lane);
    }
  }
}

// --------------------------------------------------------------------------- CUDA-core path

template <typename TS, typename TA, int NPL, int HP>
__global__ void __launch_bounds__(SIMT_WARPS * 32) decode_simt_kernel(const DecodeArgs a, const TS* __restrict__ kp,
                                                                        const TS* __restrict__ vp, int d) {
  const int pair = blockIdx.x;
  const int s = pair / a.H_kv, g = pair - (pair / a.H_kv) * a.H_kv;
  int len = a.seq_lens[s];
  const int64_t maxlen = static_cast<int64_t>(a.W) * a.B;
  if (len < 0 || len > maxlen) {
    if (threadIdx.x == 0 && g == 0) record_error(a.err, DERR_DECODE_LEN, s);
    len = len < 0 ? 0 : static_cast<int>(maxlen);
  }
  const int64_t row = (static_cast<int64_t>(s) * a.H_q + g * a.G) * d;
  simt_attend<TS, TA, NPL, HP>(a, kp, vp, d, s, g, len, static_cast<const TA*>(a.q) + row,
                               static_cast<TA*>(a.out) + row);
}

// --------------------------------------------------------------------------- host side

struct TcVariant {
  int stages, warps;
};

// Pipeline depth and warps per CTA; PKV_TC_VARIANT selects another for tuning.  An
// FP8 tile carries half the bytes of a 16-bit one and more instructions per byte, so
// its default CTAs are small: 2 stages x 2 warps, 7 CTAs (14 warps) per SM at 146
// registers (agent 48 x 32,768: 1.014 of the copy peak against 0.996 for 4 x 2 and 1.010
// for 2 x 4; 12 x 131,072: 1.018 against 0.999; chat's attention 36.7 against 38.8 us).
// Groups of 9 to 16 query heads (two head blocks) hold twice the accumulators: every pool
// type takes 2 stages x 4 warps there (FP8 with 16-head groups: 0.906 against 0.745 for
// 3 x 2); FP8 is built in 3 x 2 as well.
TcVariant tc_variant(const Pool& P) {
  static const TcVariant table[] = {{2, 4}, {3, 4}, {4, 4}, {2, 8}, {3, 2}, {6, 4}, {2, 2}, {4, 2}, {3, 1}};
  const bool fp8 = P.geo.dtype == PKV_E4M3, wide = P.geo.H_q / P.geo.H_kv > GPAD;
  int idx = fp8 && !wide ? 6 : 0;
  if (const char* e = std::getenv("PKV_TC_VARIANT")) {
    // only variants built for this pool type: 0-4 for 16-bit pools, 0-8 for FP8; 0 (and 4
    // for FP8) with groups of 9 to 16 heads (pick_tc builds no others)
    const int v = std::max(0, std::min(8, std::atoi(e)));
    if (wide ? (fp8 && (v == 0 || v == 4)) : (fp8 || v <= 4)) idx = v;
  }
  return table[idx];
}

bool tc_eligible(const Pool& P) {
  const auto& g = P.geo;
  const int G = g.H_q / g.H_kv;
  const int64_t rows = g.num_blocks * g.L * g.H_kv * g.block_size;
  const bool dt = ((g.dtype == PKV_BF16 || g.dtype == PKV_F16) && (g.d_head == 64 || g.d_head == 128)) ||
                  (g.dtype == PKV_E4M3 && g.d_head == 128);
  return dt && G <= 2 * GPAD && g.block_size % TILE == 0 && rows < (int64_t(1) << 31) && encode_fn() != nullptr;
}

int device_sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("device query: ") + cudaGetErrorString(e));
  return PKV_OK;
}

template <typename T, int D, int S, int NW, int NB = 1>
const void* tc_kernel_ptr() {
  return reinterpret_cast<const void*>(&decode_tc_kernel<T, D, S, NW, NB>);
}

using KernelPtr = const void*;

template <typename T, int D>
KernelPtr pick_tc(const TcVariant& v, int G, int* smem) {
  constexpr int EB = std::is_same<T, E4M3>::value ? 1 : 2;
  if (G > GPAD) {  // two head blocks (the variants tc_variant allows for them)
    if constexpr (EB == 1) {
      if (v.stages == 3 && v.warps == 2) {
        *smem = TcSmem<D, EB, 3, 2, 2>::TOTAL;
        return tc_kernel_ptr<T, D, 3, 2, 2>();
      }
    }
    *smem = TcSmem<D, EB, 2, 4, 2>::TOTAL;
    return tc_kernel_ptr<T, D, 2, 4, 2>();
  }
#define PKV_TC_CASE(S_, NW_)                           \
  if (v.stages == S_ && v.warps == NW_) {              \
    *smem = TcSmem<D, EB, S_, NW_>::TOTAL;             \
    return tc_kernel_ptr<T, D, S_, NW_>();             \
  }
  PKV_TC_CASE(2, 4)
  PKV_TC_CASE(3, 4)
  PKV_TC_CASE(4, 4)
  PKV_TC_CASE(2, 8)
  PKV_TC_CASE(3, 2)
  if constexpr (EB == 1) {
    PKV_TC_CASE(6, 4)
    PKV_TC_CASE(2, 2)
    PKV_TC_CASE(4, 2)
    PKV_TC_CASE(3, 1)
  }
#undef PKV_TC_CASE
  *smem = TcSmem<D, EB, 2, 4>::TOTAL;
  return tc_kernel_ptr<T, D, 2, 4>();
}

KernelPtr tc_kernel_with(const Pool& P, const TcVariant& v, int* smem) {
  const int G = P.geo.H_q / P.geo.H_kv;
  if (P.geo.dtype == PKV_E4M3) return pick_tc<E4M3, 128>(v, G, smem);
  const bool bf = P.geo.dtype == PKV_BF16;
  if (P.geo.d_head == 128) return bf ? pick_tc<__nv_bfloat16, 128>(v, G, smem) : pick_tc<__half, 128>(v, G, smem);
  return bf ? pick_tc<__nv_bfloat16, 64>(v, G, smem) : pick_tc<__half, 64>(v, G, smem);
}

KernelPtr tc_kernel_for(const Pool& P, int* smem) { return tc_kernel_with(P, tc_variant(P), smem); }

// Persistent grid for the tensor-core kernel: resident CTAs per SM x SM count.
int tc_grid(const Pool& P, int* grid, int* warps, int* smem) {
  KernelPtr k = tc_kernel_for(P, smem);
  int dev = 0;
  cudaGetDevice(&dev);
  struct Known {
    int dev;
    KernelPtr k;
    int grid;
  };
  static std::mutex mu;
  static std::vector<Known> known;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const auto& kn : known)
      if (kn.dev == dev && kn.k == k) {
        *grid = kn.grid;
        *warps = tc_variant(P).warps;
        return PKV_OK;
      }
  }
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, *smem);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  int per_sm = 0;
  const int nw = tc_variant(P).warps;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, nw * 32, *smem);
  if (e != cudaSuccess || per_sm < 1)
    return fail(PKV_ERR_CUDA, std::string("occupancy query: ") + cudaGetErrorString(e));
  int sms = 0;
  if (int rc = device_sm_count(&sms)) return rc;
  *grid = per_sm * sms;
  *warps = nw;
  std::lock_guard<std::mutex> lk(mu);
  known.push_back({dev, k, *grid});
  return PKV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t prefix, lens, counters, wstart, partials, prior_ml, prior_o, sfx_ml, sfx_o, total;
};

// n_prior > 0: room for that many shared-prefix partial slots (m, l and O per query head) at the
// end, and for the decode kernel's partial of every row.
WsLayout ws_layout(int n_seq, int H_kv, int64_t total_warps, int D, int G, int64_t n_prior = 0) {
  WsLayout w;
  w.prefix = kHdrBytes;
  w.lens = w.prefix + align256(sizeof(int32_t) * (n_seq + 1));
  w.counters = w.lens + align256(sizeof(int32_t) * n_seq);
  w.wstart = w.counters + align256(sizeof(unsigned long long) * total_warps);
  w.partials = w.wstart + align256(sizeof(int4) * total_warps);
  const int nb = G > GPAD ? 2 : 1;  // head blocks (the kernel's TcCfg::PSTRIDE)
  const int pstride = nb * (D / 16) * 32 * 4 + 2 * GPAD * nb;
  w.prior_ml = w.partials + align256(sizeof(float) * total_warps * 2 * pstride);
  const int64_t n_sfx = n_prior > 0 ? n_seq : 0;
  w.prior_o = w.prior_ml + align256(sizeof(float) * 2 * n_prior * H_kv * G);
  w.sfx_ml = w.prior_o + align256(sizeof(float) * static_cast<size_t>(D) * n_prior * H_kv * G);
  w.sfx_o = w.sfx_ml + align256(sizeof(float) * 2 * n_sfx * H_kv * G);
  w.total = w.sfx_o + align256(sizeof(float) * static_cast<size_t>(D) * n_sfx * H_kv * G);
  return w;
}

// The CUDA-core decode kernel for the pool's element types: one CTA per (sequence, KV head).
template <typename TS, typename TA>
void simt_decode_t(const DecodeArgs& a, const void* kp, const void* vp, int grid, size_t smem, cudaStream_t st) {
  const int d = a.D;
#define PKV_SIMT(NPL, HP)                                                                            \
  {                                                                                                  \
    auto kern = decode_simt_kernel<TS, TA, NPL, HP>;                                                 \
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)); \
    kern<<<grid, SIMT_WARPS * 32, smem, st>>>(a, static_cast<const TS*>(kp), static_cast<const TS*>(vp), d); \
  }
  if (a.G > GPAD) {  // 9 .. 16 query heads per KV head, d_head <= 128
    switch ((d + 31) / 32) {
      case 1: PKV_SIMT(1, SIMT_GMAX) break;
      case 2: PKV_SIMT(2, SIMT_GMAX) break;
      default: PKV_SIMT(4, SIMT_GMAX) break;
    }
  } else {
    switch ((d + 31) / 32) {
      case 1: PKV_SIMT(1, GPAD) break;
      case 2: PKV_SIMT(2, GPAD) break;
      case 3: case 4: PKV_SIMT(4, GPAD) break;
      default: PKV_SIMT(8, GPAD) break;
    }
  }
#undef PKV_SIMT
}

int launch_simt_decode(const Pool& P, const DecodeArgs& a, const void* kp, const void* vp, cudaStream_t st) {
  const auto& g = P.geo;
  const size_t smem = sizeof(float) * (SIMT_WARPS * a.G * 2 + SIMT_WARPS * a.G * static_cast<size_t>(g.d_head));
  const int pairs = a.n_seq * g.H_kv;
  switch (g.dtype) {
    case PKV_F32: simt_decode_t<float, float>(a, kp, vp, pairs, smem, st); break;
    case PKV_F16: simt_decode_t<__half, __half>(a, kp, vp, pairs, smem, st); break;
    case PKV_BF16: simt_decode_t<__nv_bfloat16, __nv_bfloat16>(a, kp, vp, pairs, smem, st); break;
    default: simt_decode_t<E4M3, __nv_bfloat16>(a, kp, vp, pairs, smem, st); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("decode launch: ") + cudaGetErrorString(e));
  count_launch();
  return PKV_OK;
}

// TMA descriptors of the K and V pools as 2-D arrays {d_head, all rows}: 16-token
// boxes 128 bytes wide (64 16-bit or 128 FP8 elements), 128-byte swizzle.
int encode_kv_maps(const pkv_geometry& g, const void* k, const void* v, CUtensorMap* tk, CUtensorMap* tv) {
  if ((reinterpret_cast<uintptr_t>(k) & 15) || (reinterpret_cast<uintptr_t>(v) & 15))
    return fail(PKV_ERR_INVALID_ARG, "k_pool and v_pool must be 16-byte aligned");
  const int eb = static_cast<int>(elem_size(g.dtype));
  const CUtensorMapDataType dt = g.dtype == PKV_E4M3  ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : g.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.d_head),
                        static_cast<cuuint64_t>(g.num_blocks) * g.L * g.H_kv * g.block_size};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(g.d_head) * eb};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), TILE};
  cuuint32_t estr[2] = {1, 1};
  auto fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  for (int which = 0; which < 2; ++which) {
    CUresult r = fn(which ? tv : tk, dt, 2, const_cast<void*>(which ? v : k), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string(r));
  }
  return PKV_OK;
}

// A 48-bit tag for one attention launch, unique within the process (never 0): the
// split-pair counters it leaves behind carry it, so the next launch needs no clearing pass.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> ctr{[] {
    // start at an arbitrary point so that leftovers of another process are unlikely to match
    unsigned long long z = static_cast<unsigned long long>(
        std::chrono::steady_clock::now().time_since_epoch().count()) ^
        (static_cast<unsigned long long>(getpid()) << 24);
    z += 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
  }()};
  for (;;) {
    const unsigned long long e = ctr.fetch_add(1, std::memory_order_relaxed) & ((1ull << 48) - 1);
    if (e != 0) return e;
  }
}

// The attention launch.  Up to kSelfPlanMaxSeqs sequences, every CTA plans its own warps
// (one launch; after_append: as the programmatic dependent of the decode step's append
// kernel launched just before, which lets it start).  Beyond that, plan_kernel first and the
// attention kernel as its programmatic dependent: its CTAs become resident and initialise
// their barriers while the plan kernel runs, and wait (griddepcontrol.wait) before reading
// the plan's outputs.
int launch_tc_sequence(DecodeArgs& a, CUtensorMap* maps, KernelPtr k, int grid, int nw, int smem,
                       cudaStream_t st, bool after_append = false) {
  a.epoch = next_epoch();
  a.self_plan = a.n_seq <= kSelfPlanMaxSeqs ? 1 : 0;
  cudaError_t e;
  if (!a.self_plan) {
    const size_t plan_smem = a.n_seq + 1 <= kPlanSmemInts ? sizeof(int32_t) * (a.n_seq + 1) : 0;
    plan_kernel<<<1, 1024, plan_smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("plan launch: ") + cudaGetErrorString(e));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(nw * 32);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (a.self_plan && !after_append) ? 0 : 1;
  void* args[] = {&maps[0], &maps[1], &a};
  e = cudaLaunchKernelExC(&cfg, k, args);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("decode launch: ") + cudaGetErrorString(e));
  count_launch(a.self_plan ? 1 : 2);
  return PKV_OK;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  }
  return fn;
}

// Fields of DecodeArgs shared by every attention launch.  For an FP8 pool the key
// scale is folded into the softmax scale and the value scale into the final
// normalisation (stored code * scale is the element's value).
int fill_args(const Pool& P, int32_t layer, const void* q, void* out, const int32_t* tables, int32_t W,
              const int32_t* seq_lens, int32_t n_seq, float scale, DecodeArgs* a) {
  const auto& g = P.geo;
  void* err = nullptr;
  if (int rc = device_error_word(&err)) return rc;
  *a = DecodeArgs{};
  a->q = q;
  a->out = out;
  a->tables = tables;
  a->seq_lens = seq_lens;
  a->err = static_cast<int*>(err);
  a->num_blocks = g.num_blocks;
  a->n_seq = n_seq;
  a->W = W;
  a->H_q = g.H_q;
  a->H_kv = g.H_kv;
  a->G = g.H_q / g.H_kv;
  a->L = g.L;
  a->layer = layer;
  a->B = g.block_size;
  a->D = g.d_head;
  a->elem = static_cast<int32_t>(act_size(g.dtype));
  const bool fp8 = g.dtype == PKV_E4M3;
  a->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 * (fp8 ? P.k_scale : 1.0));
  a->v_mul = fp8 ? P.v_scale : 1.f;
  return PKV_OK;
}

struct TensorMaps {
  struct Entry {
    int device;
    const void* k;
    const void* v;
    CUtensorMap tk, tv;
  };
  std::vector<Entry> entries;  // most recent last, at most 8
};

void destroy_tensor_maps(Pool& P) {
  delete P.tmaps;
  P.tmaps = nullptr;
}

int get_tensor_maps(Pool& P, const void* k, const void* v, CUtensorMap* tk, CUtensorMap* tv) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(P.tmap_mu);
  if (!P.tmaps) P.tmaps = new TensorMaps();
  auto& es = P.tmaps->entries;
  for (auto& e : es)
    if (e.device == dev && e.k == k && e.v == v) {
      *tk = e.tk;
      *tv = e.tv;
      return PKV_OK;
    }
  TensorMaps::Entry ent;
  ent.device = dev;
  ent.k = k;
  ent.v = v;
  if (int rc = encode_kv_maps(P.geo, k, v, &ent.tk, &ent.tv)) return rc;
  if (es.size() >= 8) es.erase(es.begin());
  es.push_back(ent);
  *tk = ent.tk;
  *tv = ent.tv;
  return PKV_OK;
}

// Shared-prefix partial slots a workspace holds for n_seq sequences (0 with sharing off).
int64_t share_slots(const Pool& P, int32_t n_seq) {
  return share_on(P) && share_geometry_ok(P.geo) ? share_slot_cap(n_seq) : 0;
}

int decode_workspace_bytes(const Pool& P, int32_t n_seq, size_t* bytes) {
  int64_t warps_total = 0;
  if (tc_eligible(P)) {
    int grid = 0, nw = 0, smem = 0;
    if (int rc = tc_grid(P, &grid, &nw, &smem)) return rc;
    warps_total = static_cast<int64_t>(grid) * nw;
  }
  *bytes = ws_layout(n_seq, P.geo.H_kv, warps_total, P.geo.d_head, P.geo.H_q / P.geo.H_kv, share_slots(P, n_seq))
               .total;
  return PKV_OK;
}

int launch_decode(Pool& P, int32_t layer, const void* q, const void* k_pool, const void* v_pool,
                  const int32_t* tables, int32_t W, const int32_t* seq_lens, int32_t n_seq, float scale, void* out,
                  void* ws, size_t ws_bytes, void* stream, const AppendFuse* fuse, const ShareLaunch* share,
                  bool long_batch) {
  const auto& g = P.geo;
  const int G = g.H_q / g.H_kv;
  if (G > SIMT_GMAX || (G > GPAD && g.d_head > 128))
    return fail(PKV_ERR_UNSUPPORTED, "more than 16 query heads per KV head, or more than 8 with d_head > 128");
  if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (static_cast<int64_t>(n_seq) * g.H_kv * ((static_cast<int64_t>(W) * g.block_size + TILE - 1) / TILE) >=
      (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "batch too large (tile count must stay below 2^31)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DecodeArgs a;
  if (int rc = fill_args(P, layer, q, out, tables, W, seq_lens, n_seq, scale, &a)) return rc;

  if (tc_eligible(P)) {
    int grid = 0, nw = 0, smem = 0;
    if (int rc = tc_grid(P, &grid, &nw, &smem)) return rc;
    const bool shared = share && share->n_items > 0;
    KernelPtr kern = tc_kernel_for(P, &smem);
    if (shared && share->decode_sms > 0 && G <= GPAD) {
      // beside the prefix kernel: one 8-warp CTA on each of decode_sms SMs, its dynamic shared
      // memory raised so that no SM takes two (the prefix kernel's CTAs take the other SMs)
      kern = tc_kernel_with(P, TcVariant{2, 8}, &smem);
      smem = std::max(smem, 116 * 1024);
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
      int sms = 0;
      if (int rc = device_sm_count(&sms)) return rc;
      grid = std::min(share->decode_sms, sms);
      nw = 8;
    } else if (long_batch && g.dtype != PKV_E4M3 && G <= GPAD && !shared) {
      // long sequences, 16-bit tiles: the default 2 CTAs an SM on 120 of 152 SMs' worth of CTAs
      // stream faster than on all (48 x 32,768: 1.059 against 1.036 of the copy peak; 12 x 131,072:
      // 1.062 against 1.035; 192 x 8,192 the same) -- fewer concurrent streams over the same HBM;
      // FP8 tiles carry half the bytes and want every SM
      grid = std::max(1, grid * 120 / 152);
    }
    const WsLayout L =
        ws_layout(n_seq, g.H_kv, static_cast<int64_t>(grid) * nw, g.d_head, G, shared ? share_slot_cap(n_seq) : 0);
    if (ws_bytes < L.total) return fail(PKV_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(L.total));
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
      return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    CUtensorMap tk, tv;
    if (int rc = get_tensor_maps(P, k_pool, v_pool, &tk, &tv)) return rc;
    char* w = static_cast<char*>(ws);
    a.hdr = reinterpret_cast<int32_t*>(w);
    a.tile_prefix = reinterpret_cast<int32_t*>(w + L.prefix);
    a.lens_c = reinterpret_cast<int32_t*>(w + L.lens);
    a.counters = reinterpret_cast<unsigned long long*>(w + L.counters);
    a.wstart = reinterpret_cast<int4*>(w + L.wstart);
    a.partials = reinterpret_cast<float*>(w + L.partials);
    a.total_warps = grid * nw;
    CUtensorMap maps[2] = {tk, tv};
    if (shared) {  // the plan's rows and work items, and the partials' room in the workspace
      if (reinterpret_cast<uintptr_t>(share->plan_dev) & 15)
        return fail(PKV_ERR_INVALID_ARG, "the shared-prefix plan must be 16-byte aligned");
      a.share = reinterpret_cast<const int4*>(share->plan_dev + 4);
      a.share_items = share->plan_dev + 4 + 4 * static_cast<int64_t>(n_seq);
      a.prior_ml = reinterpret_cast<float*>(w + L.prior_ml);
      a.prior_o = reinterpret_cast<float*>(w + L.prior_o);
      a.prior_slots = share_slot_cap(n_seq);
      a.sfx_ml = reinterpret_cast<float*>(w + L.sfx_ml);
      a.sfx_o = reinterpret_cast<float*>(w + L.sfx_o);
    }
    bool after_append = false;
    if (fuse) {  // the step's append kernel first, letting the attention launch start under it
      after_append = n_seq <= kSelfPlanMaxSeqs;
      if (int rc = launch_append(P, layer, fuse->k_new, fuse->v_new, fuse->slots, n_seq, fuse->k_pool, fuse->v_pool,
                                 stream, after_append))
        return rc;
    }
    if (int rc = launch_tc_sequence(a, maps, kern, grid, nw, smem, st, after_append)) return rc;
    if (shared) {
      // the shared blocks once per run of rows: the prefix kernel takes SMs as the decode grid
      // leaves them, and its partials are still in L2 for the combine kernel
      if (int rc = launch_prefix_share(P, a, q, k_pool, v_pool, share->n_items, share->max_members, st)) return rc;
      // the rows with a shared prefix: their two partials merged into out
      const int64_t warps = static_cast<int64_t>(n_seq) * g.H_q;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
      cfg.blockDim = dim3(256);
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const void* k = g.dtype == PKV_F16 ? reinterpret_cast<const void*>(&share_combine_kernel<__half>)
                                         : reinterpret_cast<const void*>(&share_combine_kernel<__nv_bfloat16>);
      void* args[] = {&a};
      const cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
      if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("combine launch: ") + cudaGetErrorString(e));
      count_launch();
    }
    return PKV_OK;
  }

  if (share && share->n_items > 0)
    return fail(PKV_ERR_UNSUPPORTED, "shared prefixes need the tensor-core decode path");
  if (fuse)
    if (int rc = launch_append(P, layer, fuse->k_new, fuse->v_new, fuse->slots, n_seq, fuse->k_pool, fuse->v_pool,
                               stream))
      return rc;
  return launch_simt_decode(P, a, k_pool, v_pool, st);
}

}  // namespace pkv


// ============================================================================ no-allocation entry point
//
// pkv_decode_attention_noalloc: the same decode attention, for callers that cannot
// allocate device memory (for example a serving engine that sized its KV block pool
// to fill the device at start-up, or code that must not pay cudaMalloc's implicit
// device synchronisation).  Its scratch is the file-scope array below instead of a
// caller-provided workspace; nothing here allocates device or host memory.
namespace pkv {
namespace {

// 24 MiB: the stream-K partials of one persistent grid (on a 152-SM GB300 about 10 MB
// for 16-bit pools with groups of up to 8 query heads, 18 MB for FP8 pools -- more,
// smaller CTAs -- and 20 MB for groups of 9 to 16) plus per-sequence prefix and
// length arrays.  Held by every GPU that loads the library
// until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(24) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (host code cannot use the symbol itself: it is a host-side stand-in).
int noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_CUDA, "device index out of range");
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return fail(PKV_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    addr[dev] = p;
  }
  *out = addr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_decode_attention_noalloc(const pkv_pool* pool, int32_t layer, const void* q, const void* k_pool,
                                            const void* v_pool, const int32_t* block_tables, int32_t W,
                                            const int32_t* seq_lens, int32_t n_seq, float scale, void* out,
                                            pkv_stream_t stream) {
  using namespace pkv;
  clear_error();
  if (!pool || n_seq < 0 || W < 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_decode_attention_noalloc");
  const Pool& P = *reinterpret_cast<const Pool*>(pool);
  const auto& g = P.geo;
  if (layer < 0 || layer >= g.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  if (n_seq == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  const int G = g.H_q / g.H_kv;
  if (G > SIMT_GMAX || (G > GPAD && g.d_head > 128))
    return fail(PKV_ERR_UNSUPPORTED, "more than 16 query heads per KV head, or more than 8 with d_head > 128");
  if (static_cast<int64_t>(n_seq) * g.H_kv * ((static_cast<int64_t>(W) * g.block_size + TILE - 1) / TILE) >=
      (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "batch too large (tile count must stay below 2^31)");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DecodeArgs a;
  if (int rc = fill_args(P, layer, q, out, block_tables, W, seq_lens, n_seq, scale, &a)) return rc;

  if (!tc_eligible(P)) {
    // the CUDA-core kernel needs no scratch at all
    return launch_simt_decode(P, a, k_pool, v_pool, st);
  }

  // persistent grid, computed here without any cache
  int smem = 0;
  KernelPtr k = tc_kernel_for(P, &smem);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  int per_sm = 0, sms = 0, dev = 0;
  const int nw = tc_variant(P).warps;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, nw * 32, smem);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || per_sm < 1) return fail(PKV_ERR_CUDA, std::string("grid query: ") + cudaGetErrorString(e));
  const int grid = per_sm * sms;
  const WsLayout L = ws_layout(n_seq, g.H_kv, static_cast<int64_t>(grid) * nw, g.d_head, G);
  if (L.total > kNoallocScratchBytes)
    return fail(PKV_ERR_INVALID_ARG, "pkv_decode_attention_noalloc: this batch needs " + std::to_string(L.total) +
                                         " bytes of scratch, more than the static " +
                                         std::to_string(kNoallocScratchBytes) +
                                         "; use pkv_decode_attention with a caller workspace");
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  void* ws = nullptr;
  if (int rc = noalloc_scratch(&ws)) return rc;

  // tensor maps encoded on the stack (no cache)
  CUtensorMap maps[2];
  if (int rc = encode_kv_maps(g, k_pool, v_pool, &maps[0], &maps[1])) return rc;
  // every field the kernels read is written earlier in the same call (the plan kernel's
  // header, prefix, clamped lengths and warp starts; each partial before it is counted),
  // except the split-pair counters, whose words carry the launch's epoch: a word left by an
  // earlier call counts as zero
  char* w = static_cast<char*>(ws);
  a.hdr = reinterpret_cast<int32_t*>(w);
  a.tile_prefix = reinterpret_cast<int32_t*>(w + L.prefix);
  a.lens_c = reinterpret_cast<int32_t*>(w + L.lens);
  a.counters = reinterpret_cast<unsigned long long*>(w + L.counters);
  a.wstart = reinterpret_cast<int4*>(w + L.wstart);
  a.partials = reinterpret_cast<float*>(w + L.partials);
  a.total_warps = grid * nw;
  return launch_tc_sequence(a, maps, k, grid, nw, smem, st);
}
