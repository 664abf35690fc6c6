// Data-movement kernels: append (write new keys/values at their slots) and the
// image copier used for copy-on-write block copies and for swapping blocks
// between the HBM pool and the host tier.  Also the per-device error word.
//
// Sources: "PagedAttention" (programmer.ie Inference ch. 14), "The real cache"
// (each new key and value is written at its block and offset); "KV Cache
// Management" (cs249r vol. 3 ch. 5), "Zero-copy deliberation via copy-on-write
// branching" (a CoW copies the shared block's B tokens into a fresh block) and
// "Asynchronous paged swapping" (block frames move between HBM and pinned host
// DRAM).  All of these are pure byte streams: the kernels use 16-byte vector
// loads and stores with several transactions in flight per thread.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// ------------------------------------------------------------------ launch counter

static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

// ------------------------------------------------------------------ error word

__device__ __align__(16) int g_error_word[4];

int device_error_word(void** out) {
  static void* cache[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_CUDA, "device index out of range");
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    cache[dev] = p;
  }
  *out = cache[dev];
  return PKV_OK;
}

// ------------------------------------------------------------------ append

struct AppendArgs {
  const char* k_new;
  const char* v_new;
  const int32_t* slots;
  char* k_pool;
  char* v_pool;
  int* err;
  int64_t total;        // vectors to move (per K or V)
  int64_t n_slots;      // num_blocks * B
  int32_t n_tok, H_kv, B, L, layer;  // layer < 0: all layers
  int32_t vec_per_row;  // row bytes / VEC
  int32_t lets_dependents;  // let a programmatic dependent launched next start now
};

template <int VEC>
struct VecT;
template <>
struct VecT<16> { using T = int4; };
template <>
struct VecT<8> { using T = int2; };
template <>
struct VecT<4> { using T = int; };
template <>
struct VecT<2> { using T = short; };

// One thread per VEC-byte piece of a (layer, token, head) row; consecutive
// threads cover consecutive bytes of a row, so loads and stores are coalesced.
template <int VEC>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  using V = typename VecT<VEC>::T;
  if (a.lets_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < a.total; idx += stride) {
    int64_t r = idx / a.vec_per_row;
    const int c = static_cast<int>(idx - r * a.vec_per_row);
    const int h = static_cast<int>(r % a.H_kv);
    r /= a.H_kv;
    const int i = static_cast<int>(r % a.n_tok);
    const int l = static_cast<int>(r / a.n_tok);  // source layer index (0 unless all layers)
    const int32_t slot = a.slots[i];
    if (slot < 0 || slot >= a.n_slots) {
      if (c == 0 && h == 0 && l == 0) record_error(a.err, DERR_APPEND_SLOT, slot);
      continue;
    }
    const int layer = a.layer < 0 ? l : a.layer;
    const int64_t blk = slot / a.B, off = slot - blk * a.B;
    const int64_t src = ((static_cast<int64_t>(l) * a.n_tok + i) * a.H_kv + h) * a.vec_per_row + c;
    const int64_t dst = (((blk * a.L + layer) * a.H_kv + h) * a.B + off) * a.vec_per_row + c;
    reinterpret_cast<V*>(a.k_pool)[dst] = reinterpret_cast<const V*>(a.k_new)[src];
    reinterpret_cast<V*>(a.v_pool)[dst] = reinterpret_cast<const V*>(a.v_new)[src];
  }
}

// Append into an FP8 pool ("KV Cache Management", PagedAttention model: b_elem = 1
// for FP8): one thread per 8 elements of a (layer, token, head) row -- 16 bytes of
// bf16 in, 8 bytes of E4M3 codes out (quant4_e4m3: the code nearest x / scale).
__global__ void __launch_bounds__(256) append_e4m3_kernel(const AppendArgs a, float k_scale, float v_scale) {
  if (a.lets_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < a.total; idx += stride) {
    int64_t r = idx / a.vec_per_row;
    const int c = static_cast<int>(idx - r * a.vec_per_row);
    const int h = static_cast<int>(r % a.H_kv);
    r /= a.H_kv;
    const int i = static_cast<int>(r % a.n_tok);
    const int l = static_cast<int>(r / a.n_tok);
    const int32_t slot = a.slots[i];
    if (slot < 0 || slot >= a.n_slots) {
      if (c == 0 && h == 0 && l == 0) record_error(a.err, DERR_APPEND_SLOT, slot);
      continue;
    }
    const int layer = a.layer < 0 ? l : a.layer;
    const int64_t blk = slot / a.B, off = slot - blk * a.B;
    const int64_t src = ((static_cast<int64_t>(l) * a.n_tok + i) * a.H_kv + h) * a.vec_per_row + c;
    const int64_t dst = (((blk * a.L + layer) * a.H_kv + h) * a.B + off) * a.vec_per_row + c;
    const uint4 k = reinterpret_cast<const uint4*>(a.k_new)[src];
    const uint4 v = reinterpret_cast<const uint4*>(a.v_new)[src];
    reinterpret_cast<uint2*>(a.k_pool)[dst] = make_uint2(quant4_e4m3(k.x, k.y, k_scale), quant4_e4m3(k.z, k.w, k_scale));
    reinterpret_cast<uint2*>(a.v_pool)[dst] = make_uint2(quant4_e4m3(v.x, v.y, v_scale), quant4_e4m3(v.z, v.w, v_scale));
  }
}

static int vec_width(int64_t row_bytes, const void* const* ptrs, int n) {
  uintptr_t m = static_cast<uintptr_t>(row_bytes);
  for (int i = 0; i < n; ++i) m |= reinterpret_cast<uintptr_t>(ptrs[i]);
  for (int v : {16, 8, 4, 2})
    if ((m & (v - 1)) == 0) return v;
  return 1;
}

static int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 132;
  }
  return cache[dev];
}

int launch_append(const Pool& P, int32_t layer, const void* k_new, const void* v_new, const int32_t* slots,
                  int32_t n_tok, void* k_pool, void* v_pool, void* stream, bool lets_dependents) {
  if (n_tok == 0) return PKV_OK;
  void* err = nullptr;
  if (int rc = device_error_word(&err)) return rc;
  const auto& g = P.geo;
  const bool fp8 = g.dtype == PKV_E4M3;
  const int64_t row = static_cast<int64_t>(g.d_head) * elem_size(g.dtype);
  const void* ptrs[4] = {k_new, v_new, k_pool, v_pool};
  const int vec = vec_width(row, ptrs, 4);
  if (vec < 2) return fail(PKV_ERR_INVALID_ARG, "append: buffers must be 2-byte aligned");
  if (fp8 && ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15 ||
              (reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 7))
    return fail(PKV_ERR_INVALID_ARG, "append to an FP8 pool: k_new/v_new must be 16-byte and the pools 8-byte aligned");
  AppendArgs a;
  a.k_new = static_cast<const char*>(k_new);
  a.v_new = static_cast<const char*>(v_new);
  a.slots = slots;
  a.k_pool = static_cast<char*>(k_pool);
  a.v_pool = static_cast<char*>(v_pool);
  a.err = static_cast<int*>(err);
  a.n_tok = n_tok;
  a.H_kv = g.H_kv;
  a.B = g.block_size;
  a.L = g.L;
  a.layer = layer;
  a.vec_per_row = fp8 ? g.d_head / 8 : static_cast<int32_t>(row / vec);
  a.n_slots = g.num_blocks * g.block_size;
  a.lets_dependents = lets_dependents ? 1 : 0;
  const int layers = layer < 0 ? g.L : 1;
  a.total = static_cast<int64_t>(layers) * n_tok * g.H_kv * a.vec_per_row;
  const int threads = 256;
  const int64_t want = (a.total + threads - 1) / threads;
  const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sm_count()) * 16));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fp8) append_e4m3_kernel<<<blocks, threads, 0, s>>>(a, P.k_scale, P.v_scale);
  else switch (vec) {
    case 16: append_kernel<16><<<blocks, threads, 0, s>>>(a); break;
    case 8: append_kernel<8><<<blocks, threads, 0, s>>>(a); break;
    case 4: append_kernel<4><<<blocks, threads, 0, s>>>(a); break;
    default: append_kernel<2><<<blocks, threads, 0, s>>>(a); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("append launch: ") + cudaGetErrorString(e));
  count_launch();
  return PKV_OK;
}

// ------------------------------------------------------------------ image copies

constexpr int kCopyBatch = 1024;     // images per launch (passed by value)
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;       // 16-byte vectors in flight per thread
constexpr int64_t kCopySeg = static_cast<int64_t>(kCopyThreads) * kCopyUnroll * 16 * 8;  // 128 KiB per CTA

struct CopyBatch {
  const char* src[kCopyBatch];
  char* dst[kCopyBatch];
  int64_t bytes;  // per image (a multiple of 16)
  int32_t n;
};

// grid.y = image, grid.x = 128 KiB segment of the image.  Each thread keeps
// kCopyUnroll independent 16-byte loads in flight before storing them.
__global__ void __launch_bounds__(kCopyThreads) copy_images_kernel(const __grid_constant__ CopyBatch b) {
  const int img = blockIdx.y;
  const int4* __restrict__ src = reinterpret_cast<const int4*>(b.src[img]);
  int4* __restrict__ dst = reinterpret_cast<int4*>(b.dst[img]);
  const int64_t nvec = b.bytes >> 4;
  const int64_t seg_vec = kCopySeg >> 4;
  const int64_t beg = static_cast<int64_t>(blockIdx.x) * seg_vec;
  const int64_t end = min(nvec, beg + seg_vec);
  constexpr int64_t step = static_cast<int64_t>(kCopyThreads) * kCopyUnroll;
  for (int64_t base = beg + threadIdx.x; base < end; base += step) {
    int4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t k = base + static_cast<int64_t>(u) * kCopyThreads;
      if (k < end) v[u] = __ldcs(src + k);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t k = base + static_cast<int64_t>(u) * kCopyThreads;
      if (k < end) __stcs(dst + k, v[u]);
    }
  }
}

// The same copies from a fixed number of CTAs, each looping over (image, 128 KiB segment)
// items: a transfer that shares the GPU with compute (a reload behind prefill) takes only the
// SMs the host link needs, not one CTA per segment.
__global__ void __launch_bounds__(kCopyThreads) copy_images_few_kernel(const __grid_constant__ CopyBatch b,
                                                                       int32_t segs) {
  const int64_t nvec = b.bytes >> 4;
  const int64_t seg_vec = kCopySeg >> 4;
  constexpr int64_t step = static_cast<int64_t>(kCopyThreads) * kCopyUnroll;
  for (int64_t w = blockIdx.x; w < static_cast<int64_t>(b.n) * segs; w += gridDim.x) {
    const int img = static_cast<int>(w / segs);
    const int4* __restrict__ src = reinterpret_cast<const int4*>(b.src[img]);
    int4* __restrict__ dst = reinterpret_cast<int4*>(b.dst[img]);
    const int64_t beg = (w - static_cast<int64_t>(img) * segs) * seg_vec;
    const int64_t end = min(nvec, beg + seg_vec);
    for (int64_t base = beg + threadIdx.x; base < end; base += step) {
      int4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t k = base + static_cast<int64_t>(u) * kCopyThreads;
        if (k < end) v[u] = __ldcs(src + k);
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t k = base + static_cast<int64_t>(u) * kCopyThreads;
        if (k < end) __stcs(dst + k, v[u]);
      }
    }
  }
}

int launch_copy_images(const void* src_base, void* dst_base, const CopyItem* items, int64_t n, int64_t bytes,
                       void* stream, int max_ctas) {
  if (n == 0 || bytes == 0) return PKV_OK;
  if ((bytes & 15) || (reinterpret_cast<uintptr_t>(src_base) & 15) || (reinterpret_cast<uintptr_t>(dst_base) & 15))
    return fail(PKV_ERR_INVALID_ARG, "copy: images and bases must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static thread_local CopyBatch b;  // 16 KiB: kept off the stack
  b.bytes = bytes;
  const int64_t segs = (bytes + kCopySeg - 1) / kCopySeg;
  if (segs > 0x7fffffff) return fail(PKV_ERR_INVALID_ARG, "copy: image too large");
  for (int64_t i0 = 0; i0 < n; i0 += kCopyBatch) {
    const int m = static_cast<int>(std::min<int64_t>(kCopyBatch, n - i0));
    for (int j = 0; j < m; ++j) {
      b.src[j] = static_cast<const char*>(src_base) + items[i0 + j].src_off;
      b.dst[j] = static_cast<char*>(dst_base) + items[i0 + j].dst_off;
    }
    b.n = m;
    if (max_ctas > 0) {
      const int64_t items_n = static_cast<int64_t>(m) * segs;
      copy_images_few_kernel<<<static_cast<unsigned>(std::min<int64_t>(items_n, max_ctas)), kCopyThreads, 0, s>>>(
          b, static_cast<int32_t>(segs));
    } else {
      dim3 grid(static_cast<unsigned>(segs), static_cast<unsigned>(m));
      copy_images_kernel<<<grid, kCopyThreads, 0, s>>>(b);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("copy launch: ") + cudaGetErrorString(e));
    count_launch();
  }
  return PKV_OK;
}

}  // namespace pkv

// ------------------------------------------------------------------ C ABI: device error check

// ------------------------------------------------------------------ failure-path self-test

namespace pkv {
// One warp waits on an mbarrier that nothing will complete, with the same bounded
// wait the decode kernel uses; when the bound runs out it records a timeout and
// returns, leaving the context usable.
__global__ void selftest_wait_kernel(int* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const uint64_t t0 = global_ns();
  const bool done = mbar_wait_bounded(b, 0, timeout_ns);
  if (!done && threadIdx.x == 0) record_error(err, DERR_SELFTEST_TIMEOUT, static_cast<long long>(global_ns() - t0));
}
}  // namespace pkv

extern "C" int pkv_selftest_bounded_wait(int64_t timeout_ns, pkv_stream_t stream) {
  pkv::clear_error();
  if (timeout_ns <= 0 || timeout_ns > 10000000000ll) return pkv::fail(PKV_ERR_INVALID_ARG, "timeout must be in (0, 10 s]");
  void* w = nullptr;
  if (int rc = pkv::device_error_word(&w)) return rc;
  pkv::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int*>(w),
                                                                                   static_cast<uint64_t>(timeout_ns));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, std::string("self-test launch: ") + cudaGetErrorString(e));
  pkv::count_launch();
  return PKV_OK;
}

extern "C" uint64_t pkv_launch_count(void) { return pkv::g_launches.load(std::memory_order_relaxed); }

extern "C" int pkv_device_code_version(int32_t* binary_version, int32_t* ptx_version) {
  pkv::clear_error();
  cudaFuncAttributes attr{};
  const cudaError_t e = cudaFuncGetAttributes(&attr, pkv::append_kernel<4>);
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, std::string("cudaFuncGetAttributes: ") + cudaGetErrorString(e));
  if (binary_version) *binary_version = attr.binaryVersion;
  if (ptx_version) *ptx_version = attr.ptxVersion;
  return PKV_OK;
}

extern "C" int pkv_check_device_error(pkv_stream_t stream, int32_t* code, int64_t* detail) {
  pkv::clear_error();
  if (code) *code = 0;
  if (detail) *detail = 0;
  void* w = nullptr;
  if (int rc = pkv::device_error_word(&w)) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  int host[4] = {0, 0, 0, 0};
  e = cudaMemcpy(host, w, sizeof(host), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, std::string("read error word: ") + cudaGetErrorString(e));
  if (host[0] == 0) return PKV_OK;
  int zero[4] = {0, 0, 0, 0};
  e = cudaMemcpy(w, zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, std::string("clear error word: ") + cudaGetErrorString(e));
  int64_t det;
  std::memcpy(&det, &host[2], 8);
  if (code) *code = host[0];
  if (detail) *detail = det;
  return pkv::fail(PKV_ERR_DEVICE_CHECK, "a kernel recorded a bad index: code " + std::to_string(host[0]) +
                                              ", value " + std::to_string(det));
}
