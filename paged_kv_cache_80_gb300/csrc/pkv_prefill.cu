// Chunked-prefill paged attention for one layer ("KV Cache Management", cs249r vol. 3
// ch. 5, "Chunked prefill mechanics"): the queries of a chunk attend to the cached keys of
// earlier chunks in full and to their own chunk causally.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <string>

#include "pkv_attn.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// --------------------------------------------------------------------------- chunked prefill (tensor cores)
//
// "KV Cache Management", "Chunked prefill mechanics": the queries of a chunk attend to
// the cached keys of earlier chunks in full and to their own chunk causally,
// O_k = Softmax(Q_k K_<=k^T / sqrt(d) + M_k) V_<=k; the chunk's keys/values are already
// in the pool, so query i of sequence s (position P_s + i, P_s = len_s - C_s) sees the
// paged keys 0 .. P_s + i.
// One CTA per (query block, KV head, sequence): 8 warps x 16 rows = 128 rows, a row
// being one (query, head of the group) pair, so every K/V tile staged in shared memory
// serves all of them.  Keys stream in tiles of 64 (four 16-token slabs, each from its
// own pool block, TMA with 128-byte swizzle, two stages).  S = Q K^T and O += P V are
// mma.sync m16n8k16 with the accumulator of S reused as the A operand of P V.

constexpr int PF_WARPS = 8;
constexpr int PF_ROWS = PF_WARPS * 16;
constexpr int PF_KEYS = 64;
constexpr int PF_SLABS = PF_KEYS / TILE;

template <int D>
struct PfCfg {
  static constexpr int SLAB = TILE * D * 2;          // one 16-token slab of K (or V)
  static constexpr int STAGE = 2 * PF_SLABS * SLAB;  // K slabs then V slabs
  static constexpr int NKC = D / 16;                 // 16-wide chunks of d
  static constexpr int NDG = D / 8;                  // 8-wide groups of d (PV n8 tiles)
  static constexpr int NBOX = D / 64;
};

template <typename T, int D>
__global__ void __launch_bounds__(PF_WARPS * 32, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                       const __grid_constant__ CUtensorMap tmv,
                                                                       const DecodeArgs a, const int32_t* q_off,
                                                                       int blk_cap) {
  using C = PfCfg<D>;
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  const int qb = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G;
  const int QB = PF_ROWS / G;  // queries per CTA
  const int qbeg = q_off[s];
  const int Cs = q_off[s + 1] - qbeg;
  const int i0 = qb * QB;
  if (qb == gridDim.x - 1 && tid == 0 && g == 0 && Cs > i0 + QB) record_error(a.err, DERR_PREFILL_CHUNK, s);
  if (i0 >= Cs) return;  // uniform over the CTA
  const int i1 = min(Cs, i0 + QB);
  const int len = a.seq_lens[s];
  if (Cs < 0 || len < Cs || len > static_cast<int64_t>(a.W) * a.B) {
    if (tid == 0 && qb == 0 && g == 0) record_error(a.err, DERR_DECODE_LEN, s);
    return;
  }
  const int P = len - Cs;
  const int pmin = P + i0, pmax = P + i1 - 1;
  const int nkeys = pmax + 1;
  const int ntiles = (nkeys + PF_KEYS - 1) / PF_KEYS;
  const int nblk = (nkeys + a.B - 1) / a.B;
  if (nblk > blk_cap) {  // the host sizes blk_cap from W: cannot happen for valid lengths
    if (tid == 0) record_error(a.err, DERR_DECODE_LEN, s);
    return;
  }

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage0 = smem_u32(base);
  int32_t* blks = reinterpret_cast<int32_t*>(base + 2 * C::STAGE);
  const uint32_t bar0 = smem_u32(base + 2 * C::STAGE + ((blk_cap * 4 + 15) / 16) * 16);

  for (int k = tid; k < nblk; k += blockDim.x) {
    int b = a.tables[static_cast<int64_t>(s) * a.W + k];
    if (b < 0 || b >= a.num_blocks) {
      record_error(a.err, DERR_DECODE_BLOCK, b);
      b = 0;
    }
    blks[k] = b;
  }
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int kt) {  // thread 0 only
    const int st = kt & 1;
    const uint32_t bar = bar0 + 8 * st;
    const uint32_t sk = stage0 + st * C::STAGE;
    int n = 0;
    for (int j = 0; j < PF_SLABS; ++j) n += (kt * PF_KEYS + j * TILE < nkeys) ? 1 : 0;
    fence_proxy_async();
    mbar_arrive_expect_tx(bar, 2 * n * C::SLAB);
    for (int j = 0; j < n; ++j) {
      const int t0 = kt * PF_KEYS + j * TILE;
      const int lb = t0 / a.B;
      const int row = ((blks[lb] * a.L + a.layer) * a.H_kv + g) * a.B + (t0 - lb * a.B);
#pragma unroll
      for (int b = 0; b < C::NBOX; ++b) {
        tma_load_2d(sk + j * C::SLAB + b * (TILE * 128), &tmk, b * 64, row, bar);
        tma_load_2d(sk + (PF_SLABS + j) * C::SLAB + b * (TILE * 128), &tmv, b * 64, row, bar);
      }
    }
  };
  if (tid == 0) {
    issue(0);
    if (ntiles > 1) issue(1);
  }

  // this warp's rows: r0 = warp*16 + lane/4, r1 = r0 + 8; row r = (query r / G, head r % G)
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  const int qi0 = i0 + r0 / G, qi1 = i0 + r1 / G;
  const bool v0 = r0 < QB * G && qi0 < i1, v1 = r1 < QB * G && qi1 < i1;
  const int p0 = v0 ? P + qi0 : pmax, p1 = v1 ? P + qi1 : pmax;  // last visible key
  const int64_t qrow0 = (static_cast<int64_t>(qbeg + qi0) * a.H_q + g * G + r0 % G) * D;
  const int64_t qrow1 = (static_cast<int64_t>(qbeg + qi1) * a.H_q + g * G + r1 % G) * D;
  const int c2 = 2 * (lane & 3);
  uint32_t qa[C::NKC][4];
  {
    const T* q = static_cast<const T*>(a.q);
#pragma unroll
    for (int c = 0; c < C::NKC; ++c) {
      qa[c][0] = v0 ? *reinterpret_cast<const uint32_t*>(q + qrow0 + 16 * c + c2) : 0u;
      qa[c][1] = v1 ? *reinterpret_cast<const uint32_t*>(q + qrow1 + 16 * c + c2) : 0u;
      qa[c][2] = v0 ? *reinterpret_cast<const uint32_t*>(q + qrow0 + 16 * c + 8 + c2) : 0u;
      qa[c][3] = v1 ? *reinterpret_cast<const uint32_t*>(q + qrow1 + 16 * c + 8 + c2) : 0u;
    }
  }
  float o[C::NDG][4];
#pragma unroll
  for (int n = 0; n < C::NDG; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int r8 = lane & 7, mi = lane >> 3;

  for (int kt = 0; kt < ntiles; ++kt) {
    const int st = kt & 1;
    const uint32_t sk = stage0 + st * C::STAGE;
    const uint32_t sv = sk + PF_SLABS * C::SLAB;
    if (!mbar_wait_bounded(bar0 + 8 * st, (kt >> 1) & 1, kWaitNs)) {
      if (lane == 0) record_error(a.err, DERR_DECODE_TIMEOUT, kt);
      if (tid == 0 && kt + 1 < ntiles) mbar_wait_bounded(bar0 + 8 * ((kt + 1) & 1), ((kt + 1) >> 1) & 1, kWaitNs);
      return;
    }
    const int kbase = kt * PF_KEYS;
    const int nvalid = min(PF_KEYS, nkeys - kbase);  // keys of this tile that exist
    if (nvalid < PF_KEYS && (nvalid & (TILE - 1))) {
      // zero the V rows past the last key of the last loaded slab (0 * stale could be NaN)
      const int js = nvalid / TILE, r_from = nvalid - js * TILE;
      uint8_t* vrows = base + st * C::STAGE + (PF_SLABS + js) * C::SLAB;
      for (int k = tid; k < (TILE - r_from) * 8 * C::NBOX; k += blockDim.x) {
        const int b = k / ((TILE - r_from) * 8);
        const int rem = k - b * (TILE - r_from) * 8;
        *reinterpret_cast<int4*>(vrows + b * (TILE * 128) + (r_from + rem / 8) * 128 + (rem & 7) * 16) =
            make_int4(0, 0, 0, 0);
      }
      __syncthreads();
    }
    // ---- S = Q K^T over the tile's 64 keys: 8 groups of 8 keys
    float sf[PF_KEYS / 8][4];
#pragma unroll
    for (int grp = 0; grp < PF_KEYS / 8; ++grp) {
      sf[grp][0] = sf[grp][1] = sf[grp][2] = sf[grp][3] = 0.f;
      if (grp * 8 >= nvalid) continue;
      const int slab = grp >> 1, krow = (grp & 1) * 8 + r8;
#pragma unroll
      for (int c = 0; c < C::NKC; c += 2) {
        const int doff = 16 * c + 8 * mi;
        const int chunk = (doff & 63) >> 3;
        const uint32_t addr = sk + slab * C::SLAB + (doff >> 6) * (TILE * 128) + krow * 128 + ((chunk ^ r8) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        mma_16816<BF16>(sf[grp], qa[c][0], qa[c][1], qa[c][2], qa[c][3], b0, b1);
        mma_16816<BF16>(sf[grp], qa[c + 1][0], qa[c + 1][1], qa[c + 1][2], qa[c + 1][3], b2, b3);
      }
    }
    // ---- scale, causal mask, online softmax (rows r0: c0/c1, r1: c2/c3)
    const bool need_mask = kbase + PF_KEYS - 1 > pmin;
    float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
    for (int grp = 0; grp < PF_KEYS / 8; ++grp) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sf[grp][e] * a.scale_log2;
        if (need_mask) {
          const int t = kbase + grp * 8 + c2 + (e & 1);
          if (t > ((e < 2) ? p0 : p1)) v = -INFINITY;
        }
        sf[grp][e] = v;
      }
      x0 = fmaxf(x0, fmaxf(sf[grp][0], sf[grp][1]));
      x1 = fmaxf(x1, fmaxf(sf[grp][2], sf[grp][3]));
    }
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);  // finite: key 0 is visible to every row
    const float cr0 = exp2f(m0 - n0), cr1 = exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int grp = 0; grp < PF_KEYS / 8; ++grp) {
      sf[grp][0] = exp2f(sf[grp][0] - n0);
      sf[grp][1] = exp2f(sf[grp][1] - n0);
      sf[grp][2] = exp2f(sf[grp][2] - n1);
      sf[grp][3] = exp2f(sf[grp][3] - n1);
      ps0 += sf[grp][0] + sf[grp][1];
      ps1 += sf[grp][2] + sf[grp][3];
    }
    l0 = l0 * cr0 + ps0;
    l1 = l1 * cr1 + ps1;
#pragma unroll
    for (int n = 0; n < C::NDG; ++n) {
      o[n][0] *= cr0;
      o[n][1] *= cr0;
      o[n][2] *= cr1;
      o[n][3] *= cr1;
    }
    // ---- O += P V: one k16 step per slab; P's accumulator layout is the A operand
#pragma unroll
    for (int j = 0; j < PF_SLABS; ++j) {
      if (j * TILE >= nvalid) continue;
      const uint32_t pa0 = pack2<T>(sf[2 * j][0], sf[2 * j][1]);
      const uint32_t pa1 = pack2<T>(sf[2 * j][2], sf[2 * j][3]);
      const uint32_t pa2 = pack2<T>(sf[2 * j + 1][0], sf[2 * j + 1][1]);
      const uint32_t pa3 = pack2<T>(sf[2 * j + 1][2], sf[2 * j + 1][3]);
      const int vrow = 8 * (mi & 1) + r8;
#pragma unroll
      for (int n = 0; n < C::NDG; n += 2) {
        const int doff = 8 * (n + (mi >> 1));
        const int chunk = (doff & 63) >> 3;
        const uint32_t addr = sv + j * C::SLAB + (doff >> 6) * (TILE * 128) + vrow * 128 + ((chunk ^ r8) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
        mma_16816<BF16>(o[n], pa0, pa1, pa2, pa3, b0, b1);
        mma_16816<BF16>(o[n + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
    __syncthreads();  // every warp is done with this stage
    if (tid == 0 && kt + 2 < ntiles) issue(kt + 2);
  }

  // ---- normalise and write the valid rows
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  T* out = static_cast<T*>(a.out);
#pragma unroll
  for (int n = 0; n < C::NDG; ++n) {
    const int dd = 8 * n + c2;
    if (v0) *reinterpret_cast<uint32_t*>(out + qrow0 + dd) = pack2<T>(o[n][0] * inv0, o[n][1] * inv0);
    if (v1) *reinterpret_cast<uint32_t*>(out + qrow1 + dd) = pack2<T>(o[n][2] * inv1, o[n][3] * inv1);
  }
}

// --------------------------------------------------------------------------- chunked prefill (tcgen05)
//
// One CTA per (pair of query blocks, KV head, sequence).  Its rows are two M = 128 tiles of
// (query, head) pairs, A and B (row r = query r / G, head r % G; B holds the 128 / G queries
// after A's), and both tiles use every K and V tile the CTA loads: against one tile per CTA
// this halves the L2-to-SM bytes and the TMA copies per multiply-add, and it gives the tensor
// cores a second chain of products to run while one tile's softmax is on the CUDA cores.
//   * warps 0-3 (softmax of A) and 4-7 (softmax of B): one thread per row, which is also its
//     TMEM lane; reads S with tcgen05.ld, keeps the row's running max m and sum l, writes P
//     (16-bit) back over S, and at the end reads O, divides by l and stores the row;
//   * warps 8 and 10 (producers; warp 8 owns TMEM): TMA loads of Q (3-D boxes whose rows land
//     as (query, head)) and of the 64-key K (warp 8) and V (warp 10) tiles, 4 slabs of 16
//     tokens, each from its own pool block, into rings of 4.  Lane i copies K slab i as two
//     boxes, one per 64-wide d chunk, at 2 KB stride so that the 8-row groups are uniformly
//     1 KB apart, or V slab i as one 4 KB box of both chunks.  Warp 10 zeroes the V rows past
//     the sequence end in the last tile so that P = 0 never meets a non-finite value;
//   * warps 9 and 11 (one thread each): the tensor-core issuers of A and of B: S = Q K^T
//     (tcgen05.mma kind::f16, both K-major, 128-byte swizzle, M = 128, N = 64, 8 x K = 16)
//     and O += P V (4 x K = 16) with P read from TMEM and V as an MN-major operand (N = d).
// TMEM (512 columns): tile X has two 64-column S buffers at [128 X, 128 X + 128) and O at
// [256 + 128 X, 384 + 128 X).  The softmax writes P (16-bit pairs) over the first 32 columns
// of the S it read; S = Q K^T of key tile j + 1 goes into the other buffer, so it runs on the
// tensor cores while the softmax of key tile j runs, and a buffer is reused once the P V that
// read it is complete.  The two softmaxes take turns (A of key tile j, then B of j, then A of
// j + 1), so that each has the CUDA cores of the SM to itself while the other tile's products
// run.
// The online softmax ("Chunked prefill mechanics": m_new = max(m, m_blk), l and O scaled by
// e^{m - m_new}) rescales O in TMEM only when a row's max grows by more than 2^8; otherwise
// the old max stays the reference, which is exact because P and l use the same reference.
// E4M3 pools ("KV Cache Management", b_elem = 1): the producers copy 2 KB slabs of codes into
// 2-deep staging rings instead, warps 8 and 10 round their tile's q to binary16 in place, and
// the softmax warpgroups convert each staged tile into the binary16 operand rings (3 deep)
// during the other group's turn; the products run on binary16 operands, k_scale folds into the
// softmax scale and v_scale into the final 1 / l.

// mbarrier wait that suspends the thread until the phase completes or `hint_ns` passes, so
// that waiting warps leave the issue slots of their SM sub-partition to the softmax warps
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// non-blocking test of an mbarrier phase
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr int UM_KEYS = 64;  // keys per tile: S of both tiles, double-buffered, fits in TMEM
constexpr int UM_SLABS = UM_KEYS / TILE;
constexpr int UM_THREADS = 384;  // softmax 2 x 4 warps; K producer, issuer A, V producer, issuer B
// Registers: launched at 65,536 / 384 = 168 a thread (12 warps, 3 per SM sub-partition); the
// producer warpgroup gives back down to 56 and the softmax warpgroups take 208:
// 4 x 32 x 56 + 8 x 32 x 208 = 60,416 <= 384 x 168 = 64,512.
constexpr int UM_REGS_LOW = 56, UM_REGS_HIGH = 208;
static_assert(4 * 32 * UM_REGS_LOW + 8 * 32 * UM_REGS_HIGH <= UM_THREADS * 168, "register split");
constexpr int UM_TILE_BYTES = 128 * 128 * 2;     // one Q tile (128 rows x d 128, 16-bit)
constexpr int UM_KV_BYTES = UM_KEYS * 128 * 2;   // one K or V tile (16-bit operands)
constexpr int UM_STG_BYTES = UM_KEYS * 128;      // one E4M3 K or V tile as stored (1 byte per element)
constexpr int UM_FS = 2;                         // E4M3 staging ring depth
// K and V operand rings: 4 deep for 16-bit pools, 3 for E4M3 pools (whose staging needs the rest)
__host__ __device__ constexpr int um_ks(bool kv8) { return kv8 ? 3 : 4; }
// barriers: q; the K and V rings (at most 4 deep); (S, P, O) per tile and S buffer; vz; two drains;
// turn per tile; the E4M3 staging rings (full, free); Q converted
constexpr int UM_BARS = 1 + 4 * 4 + 3 * 4 + 1 + 2 + 2 + 4 * UM_FS + 1;
constexpr int UM_TBL = 4096;  // block-table entries staged in shared memory (65,536 tokens at B = 16)
constexpr int um_smem(bool kv8) {
  return 1024 + 2 * UM_TILE_BYTES + 2 * um_ks(kv8) * UM_KV_BYTES + (kv8 ? 2 * UM_FS * UM_STG_BYTES : 0) + UM_BARS * 8 +
         16 + UM_TBL * 4;
}
static_assert(um_smem(false) <= 232448 && um_smem(true) <= 232448, "shared memory per CTA");

// two E4M3 codes per 16-bit half of w to two binary16 pairs (exact), the first of each pair low
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// two bfloat16 values (low half first) rounded to binary16
__device__ __forceinline__ uint32_t bf16x2_rn_f16x2(uint32_t w) {
  __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<uint32_t*>(&h);
}

// T: the type of q and out; KV8: an E4M3 pool, whose products run on binary16 operands (the
// codes convert exactly; q is rounded to binary16 as on the FP8 decode path).
// SH: the shared-prefix form for decode.  CTA z takes work item z of a.share_items: the decode
// queries of batch rows [rb, re) (rows that share their first table blocks), every one of them
// against all keys of blocks [kb0, kb1) of row rb's table (no causal edge: the prefix precedes
// every query); the epilogue leaves the partial (m, l, unnormalised O) of each (row, head) in
// slot slot_base + (row - rb) of a.prior_ml / a.prior_o for the combine kernel.
template <typename T, bool KV8, bool SH = false>
__global__ void __launch_bounds__(UM_THREADS, 1) prefill_umma_kernel(const __grid_constant__ CUtensorMap tmq,
                                                                      const __grid_constant__ CUtensorMap tmk,
                                                                      const __grid_constant__ CUtensorMap tmv3,
                                                                      const DecodeArgs a, const int32_t* q_off) {
  constexpr int D = 128;
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value && !KV8;  // operand type of the products
  using TP = typename std::conditional<BF16, __nv_bfloat16, __half>::type;  // type of P
  constexpr int KS = um_ks(KV8);
  extern __shared__ uint8_t smem_raw[];
  const int qb = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G;
  const int QB = 128 / G;  // queries per tile
  const int32_t* item = SH ? a.share_items + 8 * static_cast<int64_t>(s) : nullptr;
  const int qbeg = SH ? item[0] : q_off[s];
  const int Cs = SH ? item[1] - item[0] : q_off[s + 1] - qbeg;
  const int i0 = qb * 2 * QB;  // first query of tile A
  if (qb == gridDim.x - 1 && tid == 0 && g == 0 && Cs > i0 + 2 * QB) record_error(a.err, DERR_PREFILL_CHUNK, s);
  if (i0 >= Cs) {  // uniform over the CTA, before any barrier or TMEM use
    if constexpr (SH)
      if (tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  int nkeys, P = 0;
  int64_t trow0;  // the first table entry of the keys
  if constexpr (SH) {
    const int kb0 = item[2], kb1 = item[3];
    if (qbeg < 0 || item[1] > a.n_seq || kb0 < 0 || kb1 <= kb0 || kb1 > a.W || item[4] < 0 ||
        static_cast<int64_t>(item[4]) + Cs > a.prior_slots) {
      if (tid == 0 && qb == 0 && g == 0) record_error(a.err, DERR_SHARE, s);
      if (tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      return;
    }
    nkeys = (kb1 - kb0) * a.B;
    trow0 = static_cast<int64_t>(qbeg) * a.W + kb0;
  } else {
    const int len = a.seq_lens[s];
    if (Cs < 0 || len < Cs || len > static_cast<int64_t>(a.W) * a.B) {
      if (tid == 0 && qb == 0 && g == 0) record_error(a.err, DERR_DECODE_LEN, s);
      return;
    }
    P = len - Cs;
    nkeys = P + min(Cs, i0 + (i0 + QB < Cs ? 2 : 1) * QB);  // the last query's position + 1
    trow0 = static_cast<int64_t>(s) * a.W;
  }
  const int nq = i0 + QB < Cs ? 2 : 1;  // tiles with rows in the chunk
  const int i1 = min(Cs, i0 + nq * QB);
  const int pmax = nkeys - 1;
  const int nt = (nkeys + UM_KEYS - 1) / UM_KEYS;
  const bool tail = nkeys < nt * UM_KEYS;  // the last tile has keys past the sequence end

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t qs = smem_u32(base);
  const uint32_t ks0 = qs + 2 * UM_TILE_BYTES, vs0 = ks0 + KS * UM_KV_BYTES;
  const int stg_off = 2 * UM_TILE_BYTES + 2 * KS * UM_KV_BYTES;  // E4M3 staging: K ring, then V ring
  uint8_t* bar_p = base + stg_off + (KV8 ? 2 * UM_FS * UM_STG_BYTES : 0);
  const uint32_t bars = smem_u32(bar_p);
  const uint32_t q_full = bars;
  const uint32_t k_full = bars + 8, k_empty = k_full + 8 * KS;
  const uint32_t v_full = k_empty + 8 * KS, v_empty = v_full + 8 * KS;
  // S, P and O barriers are indexed by 2 X + b: tile X, S buffer b
  const uint32_t s_full = v_empty + 8 * KS, p_full = s_full + 32, o_done = p_full + 32, vz = o_done + 32;
  const uint32_t drain = vz + 8;  // two barriers: the issuers' last commits after an abort
  const uint32_t turn = drain + 16;  // per tile: its softmax of the current key tile is done
  const uint32_t sk_full = turn + 16, sv_full = sk_full + 8 * UM_FS;  // E4M3 staging landed
  const uint32_t sk_free = sv_full + 8 * UM_FS, sv_free = sk_free + 8 * UM_FS;  // staging read
  const uint32_t q_ready = sv_free + 8 * UM_FS;                                  // E4M3: q in binary16
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_p + UM_BARS * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_p + UM_BARS * 8 + 4);
  int32_t* tbl = reinterpret_cast<int32_t*>(bar_p + UM_BARS * 8 + 16);
  const int nblk = (nkeys + a.B - 1) / a.B;
  const bool tbl_in_smem = nblk <= UM_TBL;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int k = 0; k < KS; ++k) {
      mbar_init(k_full + 8 * k, KV8 ? 128 : 1);  // E4M3: the 128 threads of the converting warpgroup
      mbar_init(k_empty + 8 * k, nq);            // released by every tile's QK^T
      mbar_init(v_full + 8 * k, KV8 ? 128 : 1);
      mbar_init(v_empty + 8 * k, nq);
    }
    for (int f = 0; f < UM_FS; ++f) {
      mbar_init(sk_full + 8 * f, 1);
      mbar_init(sv_full + 8 * f, 1);
      mbar_init(sk_free + 8 * f, 128);
      mbar_init(sv_free + 8 * f, 128);
    }
    mbar_init(q_ready, nq);
    for (int i = 0; i < 4; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(p_full + 8 * i, 128);
      mbar_init(o_done + 8 * i, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(drain + 8 * x, 1);
      mbar_init(turn + 8 * x, 4);  // one arrival per softmax warp
    }
    mbar_init(vz, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // bounded wait that also gives up once another role has given up
  auto wait = [&](uint32_t bar, uint32_t parity, int where) -> bool {
    if (mbar_try_wait(bar, parity)) return true;  // fast path: no timer read
    const uint64_t t0 = global_ns();
    for (;;) {
      if (mbar_wait_suspend(bar, parity, 20000)) return true;
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitNs) {
        *abort_flag = 1;
        record_error(a.err, DERR_DECODE_TIMEOUT, where);
        return false;
      }
    }
  };
  // after an abort: bounded wait for work this thread already started (copies or MMAs)
  auto settle = [&](uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity) && global_ns() - t0 < kWaitNs) {
    }
  };

  if (warp >= 8) {
    // each warpgroup sets its register count once, before its warps go their own ways
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(UM_REGS_LOW));
    if (warp == 8 || warp == 10) {
      // ------------------------------------------------------------ producers: warp 8 Q and K, warp 10 V
      const bool kw = warp == 8;
      if (kw && lane == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(q_full, nq * 2 * 64 * G * QB * 2);  // G * QB rows per tile (126 for G = 3)
        for (int x = 0; x < nq; ++x) {
          tma_load_3d(qs + x * UM_TILE_BYTES, &tmq, 0, g * G, qbeg + i0 + x * QB, q_full);
          tma_load_3d(qs + x * UM_TILE_BYTES + 16384, &tmq, 64, g * G, qbeg + i0 + x * QB, q_full);
        }
      }
      auto block_at = [&](int lb) -> int {
        int blk = a.tables[trow0 + lb];
        if (blk < 0 || blk >= a.num_blocks) {
          record_error(a.err, DERR_DECODE_BLOCK, blk);
          blk = 0;
        }
        return blk;
      };
      if (tbl_in_smem) {  // the sequence's table slice, once (both warps write the same values)
        for (int k = lane; k < nblk; k += 32) tbl[k] = block_at(k);
        __syncwarp();
      }
      const uint32_t full0 = kw ? k_full : v_full, empty0 = kw ? k_empty : v_empty;
      if constexpr (KV8) {
        // E4M3 pool: lane i < 4 copies slab i of a 64-key tile of codes (one 2 KB box, 128-byte
        // swizzle) into a staging ring; a softmax warpgroup converts it (see there)
        const uint32_t sfull0 = kw ? sk_full : sv_full, sfree0 = kw ? sk_free : sv_free;
        const int stg = stg_off + (kw ? 0 : UM_FS * UM_STG_BYTES);
        const CUtensorMap* map = kw ? &tmk : &tmv3;
        bool ok = true;
        // q of this warp's tile (warp 8: A, warp 10: B) to binary16 in place once it has landed
        const int xq = kw ? 0 : 1;
        if (xq < nq) {
          if (lane == 0) ok = wait(q_full, 0, 1);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (ok) {
            uint4* qt = reinterpret_cast<uint4*>(base + xq * UM_TILE_BYTES);
            for (int k = lane; k < UM_TILE_BYTES / 16; k += 32) {
              uint4 w = qt[k];
              w = make_uint4(bf16x2_rn_f16x2(w.x), bf16x2_rn_f16x2(w.y), bf16x2_rn_f16x2(w.z), bf16x2_rn_f16x2(w.w));
              qt[k] = w;
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
          }
        }
        int issued = 0;
        for (int j = 0; j < nt && ok; ++j) {
          int row = 0;
          const int t0 = j * UM_KEYS + lane * TILE;
          if (lane < UM_SLABS && t0 < nkeys) {
            const int lb = t0 / a.B;
            const int blk = tbl_in_smem ? tbl[lb] : block_at(lb);
            row = ((blk * a.L + a.layer) * a.H_kv + g) * a.B + (t0 - lb * a.B);
          }
          const int nv = min(UM_SLABS, (nkeys - j * UM_KEYS + TILE - 1) / TILE);
          const int f = j % UM_FS;
          if (lane == 0) {
            if (j >= UM_FS) ok = wait(sfree0 + 8 * f, ((j / UM_FS) - 1) & 1, 110 + j);
            if (ok) mbar_arrive_expect_tx(sfull0 + 8 * f, nv * TILE * 128);
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;  // also orders the expect_tx before the copies
          if (!ok) break;
          ++issued;
          if (lane < nv) tma_load_2d(qs + stg + f * UM_STG_BYTES + lane * TILE * 128, map, 0, row, sfull0 + 8 * f);
        }
        if (*abort_flag && lane == 0) {  // copies into the staging ring may still be landing
          for (int jj = max(0, issued - UM_FS); jj < issued; ++jj) settle(sfull0 + 8 * (jj % UM_FS), (jj / UM_FS) & 1);
        }
      } else {
        bool ok = true;
        int issued = 0;
        for (int j = 0; j < nt && ok; ++j) {
          int row = 0;
          const int t0 = j * UM_KEYS + lane * TILE;
          if (lane < UM_SLABS && t0 < nkeys) {
            const int lb = t0 / a.B;
            const int blk = tbl_in_smem ? tbl[lb] : block_at(lb);
            row = ((blk * a.L + a.layer) * a.H_kv + g) * a.B + (t0 - lb * a.B);
          }
          const int nv = min(UM_SLABS, (nkeys - j * UM_KEYS + TILE - 1) / TILE);
          const int slot = j % KS;
          if (lane == 0) {
            if (j >= KS) ok = wait(empty0 + 8 * slot, ((j / KS) - 1) & 1, 100 + j);
            if (ok) mbar_arrive_expect_tx(full0 + 8 * slot, nv * 2 * TILE * 128);
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;  // also orders the expect_tx before the copies
          if (!ok) break;
          issued += 1;
          if (lane < nv) {
            if (kw) {  // K slab i: two 2 KB boxes, one per d chunk ([chunk][64 keys][128 B])
              const uint32_t dst = ks0 + slot * UM_KV_BYTES + lane * TILE * 128;
              tma_load_2d(dst, &tmk, 0, row, k_full + 8 * slot);
              tma_load_2d(dst + UM_KEYS * 128, &tmk, 64, row, k_full + 8 * slot);
            } else {  // V slab i: one 4 KB box of both d chunks ([slab][chunk][16 keys][128 B])
              tma_load_3d(vs0 + slot * UM_KV_BYTES + lane * 2 * TILE * 128, &tmv3, 0, row, 0, v_full + 8 * slot);
            }
          }
          if (!kw && tail && j == nt - 1) {
            // zero the V rows past the sequence end once the tile has landed
            bool landed = true;
            if (lane == 0) landed = wait(v_full + 8 * slot, (j / KS) & 1, 200);
            landed = __shfl_sync(0xffffffffu, landed ? 1 : 0, 0) != 0;
            if (landed) {
              uint8_t* vt = base + 2 * UM_TILE_BYTES + (KS + slot) * UM_KV_BYTES;
              const int r0 = nkeys - j * UM_KEYS;
              for (int k = lane; k < (UM_KEYS - r0) * 16; k += 32) {  // 16-byte pieces, both d chunks
                const int r = r0 + k / 16, c = k % 16;
                *reinterpret_cast<int4*>(vt + (r / TILE) * 4096 + (c / 8) * 2048 + (r % TILE) * 128 + (c % 8) * 16) =
                    make_int4(0, 0, 0, 0);
              }
              fence_proxy_async();
              __syncwarp();
              if (lane == 0) mbar_arrive(vz);
            }
          }
        }
        if (*abort_flag && lane == 0) {  // the last ring's copies may still be landing
          for (int jj = max(0, issued - KS); jj < issued; ++jj) settle(full0 + 8 * (jj % KS), (jj / KS) & 1);
        }
      }
    } else {
      // ------------------------------------------------------------ tensor-core issuer of tile X (warp 9 A, warp 11 B)
      const int X = warp == 9 ? 0 : 1;
      if (lane == 0 && X < nq) {
        const uint32_t idesc_s = umma_idesc_f16(BF16, 128, UM_KEYS, false);
        const uint32_t idesc_o = umma_idesc_f16(BF16, 128, D, true);
        const uint32_t qx = qs + X * UM_TILE_BYTES;
        const uint32_t sx = tmem + 128 * X, ox = tmem + 256 + 128 * X;
        // S = Q K^T of key tile i into S buffer i & 1 (which held P(i - 2) until its P V was
        // complete) and O += P V of key tile j are two in-order streams with their own inputs;
        // the thread starts whichever is ready, so neither waits behind the other.
        auto qk = [&](int i) {
          const uint32_t kb = ks0 + (i % KS) * UM_KV_BYTES;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t kin = (k & 3) * 32;  // 16 elements = 32 bytes along the swizzled 128-byte row
            umma_ss(sx + UM_KEYS * (i & 1), umma_desc_sw128(qx + (k >> 2) * 16384 + kin, 16, 1024),
                    umma_desc_sw128(kb + (k >> 2) * (UM_KEYS * 128) + kin, 16, 1024), idesc_s, k > 0);
          }
          umma_commit(s_full + 8 * (2 * X + (i & 1)));
          umma_commit(k_empty + 8 * (i % KS));
        };
        auto pv = [&](int j) {
          const uint32_t vb = vs0 + (j % KS) * UM_KV_BYTES;
#pragma unroll
          for (int k = 0; k < UM_KEYS / 16; ++k)
            umma_ts(ox, sx + UM_KEYS * (j & 1) + 8 * k, umma_desc_sw128(vb + k * 4096, 2048, 1024), idesc_o,
                    (j > 0 || k > 0) ? 1u : 0u);
          umma_commit(o_done + 8 * (2 * X + (j & 1)));
          umma_commit(v_empty + 8 * (j % KS));
        };
        bool ok = wait(KV8 ? q_ready : q_full, 0, 1);
        int i = 0, j = 0;  // next S = Q K^T, next P V
        uint64_t t_last = global_ns();
        while (ok && j < nt) {
          bool progressed = false;
          if (i < nt && i <= j + 1 && (i < 2 || mbar_test(o_done + 8 * (2 * X + (i & 1)), ((i - 2) >> 1) & 1)) &&
              mbar_test(k_full + 8 * (i % KS), (i / KS) & 1)) {
            tc_fence_after();
            qk(i++);
            progressed = true;
          }
          if (j < i && mbar_test(p_full + 8 * (2 * X + (j & 1)), (j >> 1) & 1) &&
              mbar_test(v_full + 8 * (j % KS), (j / KS) & 1) && (KV8 || !tail || j < nt - 1 || mbar_test(vz, 0))) {
            tc_fence_after();
            pv(j++);
            progressed = true;
          }
          if (progressed) {
            t_last = global_ns();
          } else if (*abort_flag) {
            ok = false;
          } else if (global_ns() - t_last > kWaitNs) {
            *abort_flag = 1;
            record_error(a.err, DERR_DECODE_TIMEOUT, 400 + j);
            ok = false;
          }
        }
        if (*abort_flag) {
          umma_commit(drain + 8 * X);
          settle(drain + 8 * X, 0);
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(UM_REGS_HIGH));
    if (warp / 4 < nq) {
      // ---------------------------------------------------------- softmax and epilogue of tile X (warps 4X .. 4X + 3)
      const int X = warp / 4;
      const int r = tid & 127;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      const uint32_t o_addr = lane_addr + 256 + 128 * X;
      const int qi = i0 + X * QB + r / G, h = r % G;
      const bool valid = r < QB * G && qi < i1;
      const int lim = (valid && !SH) ? P + qi : pmax;  // last visible key
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      // E4M3 pools: this warpgroup converts a staged tile of codes (K or V of key tile c) into
      // the binary16 operand ring while the other warpgroup has its softmax turn.  Staging row r
      // of slab i holds d = 16 u .. 16 u + 15 in 16-byte unit u ^ (r & 7); the operand rows hold
      // d in two 64-wide chunks of eight 16-byte units, unit t at t ^ (row & 7).  V rows past the
      // sequence end are written as zeros.
      auto convert = [&](int c, bool is_k) -> bool {
        const int f = c % UM_FS, slot = c % KS;
        bool ok2 = wait((is_k ? sk_full : sv_full) + 8 * f, (c / UM_FS) & 1, 130 + c);
        if (ok2 && c >= KS) ok2 = wait((is_k ? k_empty : v_empty) + 8 * slot, ((c / KS) - 1) & 1, 140 + c);
        if (!__all_sync(0xffffffffu, ok2)) return false;
        const uint8_t* src = base + stg_off + ((is_k ? 0 : UM_FS) + f) * UM_STG_BYTES;
        uint8_t* dst = base + 2 * UM_TILE_BYTES + ((is_k ? 0 : KS) + slot) * UM_KV_BYTES;
        const int r0 = nkeys - c * UM_KEYS;  // tile rows at or past r0 are past the sequence end
#pragma unroll
        for (int k = 0; k < UM_STG_BYTES / 16 / 128; ++k) {
          const int idx = r + 128 * k;
          const int i = idx >> 7, rr = (idx >> 3) & 15, u = idx & 7, R = TILE * i + rr;
          const uint4 w = *reinterpret_cast<const uint4*>(src + i * (TILE * 128) + rr * 128 + ((u ^ (rr & 7)) << 4));
          uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
          if (is_k || R < r0) {
            e4m3x4_to_f16x4(w.x, o0.x, o0.y);
            e4m3x4_to_f16x4(w.y, o0.z, o0.w);
            e4m3x4_to_f16x4(w.z, o1.x, o1.y);
            e4m3x4_to_f16x4(w.w, o1.z, o1.w);
          }
          const int cc = u >> 2, t = (u & 3) * 2, sw = R & 7;
          // K: [chunk][64 keys][128 B]; V: [slab][chunk][16 keys][128 B]
          uint8_t* rowp = is_k ? dst + cc * (UM_KEYS * 128) + R * 128 : dst + i * 4096 + cc * 2048 + rr * 128;
          *reinterpret_cast<uint4*>(rowp + ((t ^ sw) << 4)) = o0;
          *reinterpret_cast<uint4*>(rowp + (((t + 1) ^ sw) << 4)) = o1;
        }
        fence_proxy_async();  // the generic-proxy writes and reads, before the async proxy's use
        mbar_arrive((is_k ? k_full : v_full) + 8 * slot);
        mbar_arrive((is_k ? sk_free : sv_free) + 8 * f);
        return true;
      };
      // A converts K, B converts V (A both when the CTA has one tile): K(0 .. 2) and V(0, 1)
      // first, then after its softmax of key tile j, K(j + 3) in the slot that QK^T(j) freed
      // and V(j + 2) in the slot that P V(j - 1) freed.
      const bool conv_k = KV8 && X == 0, conv_v = KV8 && (X == 1 || nq == 1);
      for (int c = 0; c < min(nt, KS) && ok && conv_k; ++c) ok = convert(c, true);
      for (int c = 0; c < min(nt, 2) && ok && conv_v; ++c) ok = convert(c, false);
      // tcgen05.ld / st are warp-collective: every decision below is uniform over the warp
      for (int j = 0; j < nt && ok; ++j) {
        const int b = j & 1;
        const uint32_t s_addr = lane_addr + 128 * X + UM_KEYS * b;
        ok = __all_sync(0xffffffffu, wait(s_full + 8 * (2 * X + b), (j >> 1) & 1, 700 + j));
        // the two tiles' softmaxes alternate (A of key tile j, B of j, A of j + 1, ...), so that
        // one tile's products run on the tensor cores while the other's exponentials run
        if (ok && X == 0 && nq == 2 && j > 0) ok = __all_sync(0xffffffffu, wait(turn + 8, (j - 1) & 1, 900 + j));
        if (ok && X == 1) ok = __all_sync(0xffffffffu, wait(turn, j & 1, 900 + j));
        if (!ok) break;
        tc_fence_after();
        constexpr int NC = UM_KEYS / 32;
        uint32_t sv[NC][32];
#pragma unroll
        for (int c = 0; c < NC; ++c) tmem_ld32(s_addr + 32 * c, sv[c]);
        tmem_ld_wait();
        const int k0 = j * UM_KEYS;
        // mask only tiles where some row of the warp meets the causal edge or the sequence end
        if (__any_sync(0xffffffffu, k0 + UM_KEYS - 1 > lim)) {
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (k0 + 32 * c + e > lim) sv[c][e] = __float_as_uint(-INFINITY);
        }
        // row max on the raw scores (the scale is positive), 8 independent chains
        float mx8[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx8[t] = -INFINITY;
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sv[c][e]));
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float sl = a.scale_log2;
        const float m_new = fmaxf(m, mx * sl);
        if (__any_sync(0xffffffffu, m_new > m + 8.f)) {  // the reference max moves: rescale l and O so far
          const float alpha = fast_exp2(m - m_new);
          if (j > 0) {
            ok = __all_sync(0xffffffffu, wait(o_done + 8 * (2 * X + ((j - 1) & 1)), ((j - 1) >> 1) & 1, 800 + j));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(o_addr + 32 * c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(o_addr + 32 * c, o);
            }
          }
          l *= alpha;
          m = m_new;
        }
        // P = 2^(scale * s - m), 16-bit, two keys per TMEM column, written over the S just
        // read (this lane's row only: its S is in registers); 8 partial sums
        const float neg_m = -m;
        float ls8[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) ls8[t] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {  // 32 keys -> 16 columns
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = fast_exp2(fmaf(__uint_as_float(sv[c][2 * e]), sl, neg_m));
            const float p1 = fast_exp2(fmaf(__uint_as_float(sv[c][2 * e + 1]), sl, neg_m));
            ls8[e & 7] += p0 + p1;
            pw[e] = pack2<TP>(p0, p1);
          }
          tmem_st16(s_addr + 16 * c, pw);
          // the other tile's turn starts halfway through these exponentials, so that its S load
          // and row max (no special-function work) overlap the second half (16-bit pools; with
          // E4M3 pools, whose softmax warpgroups also convert, at the end of the exponentials)
          if (!KV8 && c == NC / 2 - 1 && lane == 0) mbar_arrive(turn + 8 * X);
        }
        if (KV8 && lane == 0) mbar_arrive(turn + 8 * X);
        l += ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + 8 * (2 * X + b));
        if (conv_k && j + KS < nt) ok = convert(j + KS, true);
        if (ok && conv_v && j + 2 < nt) ok = convert(j + 2, false);
      }
      if (ok) ok = __all_sync(0xffffffffu, wait(o_done + 8 * (2 * X + ((nt - 1) & 1)), ((nt - 1) >> 1) & 1, 1000));
      if (ok && SH) {
        // the partial of (row qbeg + qi, head g G + h): m, l and O relative to 2^m, unscaled
        tc_fence_after();
        const int64_t row = (static_cast<int64_t>(item[4]) + qi) * a.H_q + g * G + h;
        float4* dst = reinterpret_cast<float4*>(a.prior_o + row * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + 32 * c, o);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[8 * c + v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                           __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
          }
        }
        if (valid) *reinterpret_cast<float2*>(a.prior_ml + 2 * row) = make_float2(m, l);
      } else if (ok) {
        tc_fence_after();
        const float inv = a.v_mul / l;  // v_scale of an E4M3 pool, else 1
        T* out = static_cast<T*>(a.out) + (static_cast<int64_t>(qbeg + qi) * a.H_q + g * G + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + 32 * c, o);
          tmem_ld_wait();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pack2<T>(__uint_as_float(o[8 * v]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                                  pack2<T>(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                                  pack2<T>(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                                  pack2<T>(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) tmem_dealloc(tmem, 512);
  // the shared-prefix form runs as the decode kernel's programmatic dependent; it completes only
  // after that grid has, so that the combine kernel, which waits for this grid, sees both
  if constexpr (SH)
    if (tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Chunked prefill on CUDA cores: one CTA per (query row, KV head).  The row's
// sequence s is found in q_off; its position is len_s - C_s + (row - q_off[s]) and it
// attends to every token up to and including that position.
template <typename TS, typename TA, int NPL, int HP>
__global__ void __launch_bounds__(SIMT_WARPS * 32) prefill_simt_kernel(const DecodeArgs a, const int32_t* q_off,
                                                                         const TS* __restrict__ kp,
                                                                         const TS* __restrict__ vp, int d) {
  const int row = blockIdx.x, g = blockIdx.y;
  int lo = 0, hi = a.n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (q_off[mid] <= row) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int C = q_off[s + 1] - q_off[s];
  const int len = a.seq_lens[s];
  const int64_t base = (static_cast<int64_t>(row) * a.H_q + g * a.G) * d;
  if (C < 0 || len < C || len > static_cast<int64_t>(a.W) * a.B) {
    if (threadIdx.x == 0 && g == 0 && row == q_off[s]) record_error(a.err, DERR_DECODE_LEN, s);
    for (int k = threadIdx.x; k < a.G * d; k += blockDim.x) static_cast<TA*>(a.out)[base + k] = f_to<TA>(0.f);
    return;
  }
  const int pos = len - C + (row - q_off[s]);
  simt_attend<TS, TA, NPL, HP>(a, kp, vp, d, s, g, pos + 1, static_cast<const TA*>(a.q) + base,
                               static_cast<TA*>(a.out) + base);
}

// The CUDA-core prefill kernel for the pool's element types: one CTA per (query row, KV head).
template <typename TS, typename TA>
void simt_prefill_t(const DecodeArgs& a, const int32_t* q_off, const void* kp, const void* vp, dim3 grid, size_t smem,
                    cudaStream_t st) {
  const int d = a.D;
#define PKV_PF_SIMT(NPL, HP)                                                                         \
  {                                                                                                  \
    auto kern = prefill_simt_kernel<TS, TA, NPL, HP>;                                                \
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)); \
    kern<<<grid, SIMT_WARPS * 32, smem, st>>>(a, q_off, static_cast<const TS*>(kp), static_cast<const TS*>(vp), d); \
  }
  if (a.G > GPAD) {  // 9 .. 16 query heads per KV head, d_head <= 128
    switch ((d + 31) / 32) {
      case 1: PKV_PF_SIMT(1, SIMT_GMAX) break;
      case 2: PKV_PF_SIMT(2, SIMT_GMAX) break;
      default: PKV_PF_SIMT(4, SIMT_GMAX) break;
    }
  } else {
    switch ((d + 31) / 32) {
      case 1: PKV_PF_SIMT(1, GPAD) break;
      case 2: PKV_PF_SIMT(2, GPAD) break;
      case 3: case 4: PKV_PF_SIMT(4, GPAD) break;
      default: PKV_PF_SIMT(8, GPAD) break;
    }
  }
#undef PKV_PF_SIMT
}

// TMA descriptors of the tcgen05 kernel: q as {d, H_q, n_tok} (a box of {64, G, 128 / G} lands as
// 128 (query, head) rows of 128 bytes), K as the decode kernel's 16-token slabs, V as
// {64, rows, 2 d chunks} (a {64, 16, 2} box is one 16-token slab of both chunks, 4 KB; E4M3
// pools copy slabs of codes with the 2-D map and convert them in the kernel).
int umma_maps(Pool& P, const void* q, int32_t n_tok, const void* k_pool, const void* v_pool, bool kv8,
              CUtensorMap* maps) {
  const auto& g = P.geo;
  const int G = g.H_q / g.H_kv;
  if (int rc = get_tensor_maps(P, k_pool, v_pool, &maps[1], &maps[2])) return rc;
  if (!kv8) {
    cuuint64_t vd[3] = {64, static_cast<cuuint64_t>(g.num_blocks) * g.L * g.H_kv * g.block_size, 2};
    cuuint64_t vs[2] = {256, 128};
    cuuint32_t vb[3] = {64, TILE, 2};
    cuuint32_t ve[3] = {1, 1, 1};
    const CUtensorMapDataType vt =
        g.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = encode_fn()(&maps[2], vt, 3, const_cast<void*>(v_pool), vd, vs, vb, ve, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (v slabs) failed: " + std::to_string(r));
  }
  const int QB = 128 / G;
  const CUtensorMapDataType dt =
      g.dtype == PKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;  // q: bf16 for E4M3
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(g.H_q), static_cast<cuuint64_t>(std::max(n_tok, 1))};
  cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(g.H_q) * 256};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(QB)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode_fn()(&maps[0], dt, 3, const_cast<void*>(q), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed: " + std::to_string(r));
  return PKV_OK;
}

}  // namespace

int launch_prefix_share(Pool& P, const DecodeArgs& a, const void* q, const void* k_pool, const void* v_pool,
                        int32_t n_items, int32_t max_members, cudaStream_t st) {
  const auto& g = P.geo;
  const int G = g.H_q / g.H_kv;
  if (n_items <= 0) return PKV_OK;
  if (!share_geometry_ok(g) || !encode_fn())
    return fail(PKV_ERR_UNSUPPORTED, "shared prefixes need a tensor-core pool with d_head 128");
  const bool kv8 = g.dtype == PKV_E4M3;
  CUtensorMap maps[3];
  if (int rc = umma_maps(P, q, a.n_seq, k_pool, v_pool, kv8, maps)) return rc;
  const void* k = kv8 ? reinterpret_cast<const void*>(&prefill_umma_kernel<__nv_bfloat16, true, true>)
                  : g.dtype == PKV_BF16 ? reinterpret_cast<const void*>(&prefill_umma_kernel<__nv_bfloat16, false, true>)
                                        : reinterpret_cast<const void*>(&prefill_umma_kernel<__half, false, true>);
  const int smem = um_smem(kv8);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  const int QB = 128 / G;
  dim3 grid((max_members + 2 * QB - 1) / (2 * QB), g.H_kv, n_items);
  DecodeArgs args_copy = a;
  const int32_t* no_off = nullptr;
  void* args[] = {&maps[0], &maps[1], &maps[2], &args_copy, const_cast<int32_t**>(&no_off)};
  // the decode kernel's programmatic dependent: its CTAs take the SMs that decode CTAs leave
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(UM_THREADS);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelExC(&cfg, k, args);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("shared-prefix launch: ") + cudaGetErrorString(e));
  count_launch();
  return PKV_OK;
}

int launch_prefill(Pool& P, int32_t layer, const void* q, const int32_t* q_off, int32_t n_tok, int32_t max_q,
                   const void* k_pool, const void* v_pool, const int32_t* tables, int32_t W, const int32_t* seq_lens,
                   int32_t n_seq, float scale, void* out, void* stream) {
  const auto& g = P.geo;
  const int G = g.H_q / g.H_kv;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DecodeArgs a;
  if (int rc = fill_args(P, layer, q, out, tables, W, seq_lens, n_seq, scale, &a)) return rc;
  cudaError_t e = cudaSuccess;
  const int64_t rows = g.num_blocks * g.L * g.H_kv * g.block_size;
  const bool tc = (g.dtype == PKV_BF16 || g.dtype == PKV_F16) && (g.d_head == 64 || g.d_head == 128) &&
                  G <= PF_ROWS && g.block_size % TILE == 0 && rows < (int64_t(1) << 31) && encode_fn() != nullptr;
  static const bool force_mma_sync = std::getenv("PKV_PREFILL_MMA_SYNC") != nullptr;
  // E4M3 pools with d_head 128: the same tcgen05 kernel on binary16 operands converted in shared memory
  const bool tc8 = g.dtype == PKV_E4M3 && g.d_head == 128 && G <= PF_ROWS && g.block_size % TILE == 0 &&
                   rows < (int64_t(1) << 31) && encode_fn() != nullptr;
  if ((tc && g.d_head == 128 && !force_mma_sync) || tc8) {
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
      return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    CUtensorMap maps[3];
    if (int rc = umma_maps(P, q, n_tok, k_pool, v_pool, tc8, maps)) return rc;
    const void* k = tc8 ? reinterpret_cast<const void*>(&prefill_umma_kernel<__nv_bfloat16, true>)
                    : g.dtype == PKV_BF16 ? reinterpret_cast<const void*>(&prefill_umma_kernel<__nv_bfloat16, false>)
                                          : reinterpret_cast<const void*>(&prefill_umma_kernel<__half, false>);
    const int smem = um_smem(tc8);
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    const int QB = 128 / G;
    dim3 grid((max_q + 2 * QB - 1) / (2 * QB), g.H_kv, n_seq);
    void* args[] = {&maps[0], &maps[1], &maps[2], &a, const_cast<int32_t**>(&q_off)};
    e = cudaLaunchKernel(k, grid, dim3(UM_THREADS), args, smem, st);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("prefill launch: ") + cudaGetErrorString(e));
    count_launch();
    return PKV_OK;
  }
  if (!tc && !tc8 && (G > SIMT_GMAX || (G > GPAD && g.d_head > 128)))
    return fail(PKV_ERR_UNSUPPORTED, "on the CUDA-core path: more than 16 query heads per KV head, or more than 8 with d_head > 128");
  if (tc) {
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
      return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    CUtensorMap maps[2];
    if (int rc = get_tensor_maps(P, k_pool, v_pool, &maps[0], &maps[1])) return rc;
    const int stage = 2 * PF_SLABS * TILE * g.d_head * 2;
    const int blk_cap = W;
    const size_t smem = 1024 + 2 * static_cast<size_t>(stage) + ((blk_cap * 4 + 15) / 16) * 16 + 16;
    if (smem > 227 * 1024) return fail(PKV_ERR_UNSUPPORTED, "block table too wide for the prefill kernel");
    const int QB = PF_ROWS / G;
    dim3 grid((max_q + QB - 1) / QB, g.H_kv, n_seq);
    const bool bf = g.dtype == PKV_BF16;
    const void* k = g.d_head == 128 ? (bf ? reinterpret_cast<const void*>(&prefill_tc_kernel<__nv_bfloat16, 128>)
                                          : reinterpret_cast<const void*>(&prefill_tc_kernel<__half, 128>))
                                    : (bf ? reinterpret_cast<const void*>(&prefill_tc_kernel<__nv_bfloat16, 64>)
                                          : reinterpret_cast<const void*>(&prefill_tc_kernel<__half, 64>));
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    int cap = blk_cap;
    void* args[] = {&maps[0], &maps[1], &a, const_cast<int32_t**>(&q_off), &cap};
    e = cudaLaunchKernel(k, grid, dim3(PF_WARPS * 32), args, smem, st);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("prefill launch: ") + cudaGetErrorString(e));
    count_launch();
    return PKV_OK;
  }
  const size_t smem = sizeof(float) * (SIMT_WARPS * G * 2 + SIMT_WARPS * G * static_cast<size_t>(g.d_head));
  const dim3 grid(n_tok, g.H_kv);
  switch (g.dtype) {
    case PKV_F32: simt_prefill_t<float, float>(a, q_off, k_pool, v_pool, grid, smem, st); break;
    case PKV_F16: simt_prefill_t<__half, __half>(a, q_off, k_pool, v_pool, grid, smem, st); break;
    case PKV_BF16: simt_prefill_t<__nv_bfloat16, __nv_bfloat16>(a, q_off, k_pool, v_pool, grid, smem, st); break;
    default: simt_prefill_t<E4M3, __nv_bfloat16>(a, q_off, k_pool, v_pool, grid, smem, st); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("prefill launch: ") + cudaGetErrorString(e));
  count_launch();
  return PKV_OK;
}


}  // namespace pkv
