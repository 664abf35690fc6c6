// Host control plane and C ABI entry points.
//
// The control plane follows "KV Cache Management" (cs249r vol. 3 ch. 5), "The
// PagedAttention virtual memory model" (block table T: l -> p with l = floor(t/B),
// o = t mod B; allocation from a free-list ring buffer when o == 0) and "Zero-copy
// deliberation via copy-on-write branching" (fork = table duplication plus a
// reference-count increment; a write into a block with more than one owner first
// copies it into a fresh block; release walks the table and returns blocks that
// reach zero owners to the free list), and "PagedAttention" (programmer.ie ch. 14),
// "Inference Lab increment" (out-of-blocks and double-free errors; a failed
// reservation leaks nothing).
//
// All-or-nothing reservation is done with a dry run that counts the blocks an
// append needs (new blocks plus copy-on-write copies, with the owner counts the
// earlier sequences of the same call leave behind) before anything is changed.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

static thread_local std::string g_msg;

int fail(int status, const std::string& msg) {
  g_msg = msg;
  return status;
}

void clear_error() { g_msg.clear(); }

// ------------------------------------------------------------------ free ring

void FreeRing::reset(const std::vector<int32_t>& order) {
  ring_ = order;
  cap_ = static_cast<int64_t>(order.size());
  head_ = 0;
  count_ = cap_;
}

int32_t FreeRing::pop_front() {
  int32_t p = ring_[head_];
  head_ = (head_ + 1) % cap_;
  --count_;
  return p;
}

void FreeRing::push_back(int32_t p) {
  ring_[(head_ + count_) % cap_] = p;
  ++count_;
}

}  // namespace pkv

using pkv::fail;
using pkv::Pool;
using pkv::SeqState;

namespace {

Pool* as_pool(pkv_pool* p) { return reinterpret_cast<Pool*>(p); }
const Pool* as_pool(const pkv_pool* p) { return reinterpret_cast<const Pool*>(p); }

int check_geometry(const pkv_geometry* g) {
  if (!g) return fail(PKV_ERR_INVALID_ARG, "geometry is NULL");
  if (g->L <= 0 || g->H_kv <= 0 || g->H_q <= 0 || g->d_head <= 0 || g->block_size <= 0 || g->num_blocks <= 0)
    return fail(PKV_ERR_INVALID_ARG, "geometry fields must be positive");
  if (g->H_q % g->H_kv) return fail(PKV_ERR_INVALID_ARG, "H_q must be a multiple of H_kv");
  if (g->d_head % 2 || g->d_head > 256) return fail(PKV_ERR_INVALID_ARG, "d_head must be even and <= 256");
  if (g->dtype != PKV_F32 && g->dtype != PKV_F16 && g->dtype != PKV_BF16 && g->dtype != PKV_E4M3)
    return fail(PKV_ERR_UNSUPPORTED, "dtype must be PKV_F32, PKV_F16, PKV_BF16 or PKV_E4M3");
  if (g->dtype == PKV_E4M3 && g->d_head % 8)
    return fail(PKV_ERR_UNSUPPORTED, "an FP8 pool needs d_head a multiple of 8");
  if (g->num_blocks >= (int64_t(1) << 31)) return fail(PKV_ERR_INVALID_ARG, "num_blocks must be < 2^31");
  if (g->num_blocks * g->block_size >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_blocks * block_size must be < 2^31 (int32 slots)");
  return PKV_OK;
}

SeqState* find_seq(Pool& P, int32_t id) {
  if (id < 0 || id >= P.next_id || P.seqs[id].state != 0) return nullptr;
  return &P.seqs[id];
}

const SeqState* find_seq(const Pool& P, int32_t id) {
  if (id < 0 || id >= P.next_id || P.seqs[id].state != 0) return nullptr;
  return &P.seqs[id];
}

// Releasing a released sequence is a double free; any other use of it, or of an
// id never created, is an invalid argument.
int unknown_seq(const Pool& P, int32_t id, bool releasing = false) {
  if (releasing && id >= 0 && id < P.next_id && P.seqs[id].state == 1)
    return fail(PKV_ERR_DOUBLE_FREE, "sequence " + std::to_string(id) + " was already released");
  return fail(PKV_ERR_INVALID_ARG, "unknown or released sequence " + std::to_string(id));
}

// Token t's logical block t / B and offset t mod B: a shift and a mask when B is a power of two
// (a 64-bit division costs tens of cycles, and a decode step takes several per sequence).
struct BlockIdx {
  int64_t B;
  int sh;
  explicit BlockIdx(int64_t b)
      : B(b), sh((b & (b - 1)) == 0 ? __builtin_ctzll(static_cast<unsigned long long>(b)) : -1) {}
  int64_t blk(int64_t t) const { return sh >= 0 ? t >> sh : t / B; }
  int64_t off(int64_t t) const { return sh >= 0 ? t & (B - 1) : t % B; }
  int64_t blocks(int64_t tokens) const { return blk(tokens + B - 1); }  // ceil(tokens / B)
};

// Drop one owner of block p; at zero it goes to the back of the FIFO.
void drop_owner(Pool& P, int32_t p) {
  if (--P.ref[p] == 0) P.free.push_back(p);
}

// Device-accessible address of a host-tier buffer, or nullptr.
void* device_view_of_host(void* host) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, host) == cudaSuccess) {
    if (attr.type == cudaMemoryTypeHost && attr.devicePointer) return attr.devicePointer;
    if (attr.type == cudaMemoryTypeManaged) return host;
  }
  cudaGetLastError();
  int dev = 0, pageable = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) == cudaSuccess && pageable)
    return host;
  cudaGetLastError();
  return nullptr;
}

// CTAs of the SM copier for swaps: 32 keep the host link at its copy rate (out 188 / in 205 GB/s,
// as with one CTA per 128 KiB of every image) and leave the other SMs to whatever runs beside the
// swap (a reload behind decode: 86 % hidden instead of 75 %).  PKV_SWAP_CTAS overrides it for tuning
// (0: one CTA per 128 KiB).
int swap_ctas() {
  if (const char* e = std::getenv("PKV_SWAP_CTAS")) return std::max(0, std::atoi(e));
  return 32;
}

// Copy n images of `bytes` with the copy engines.
int copy_engine(const void* src_base, void* dst_base, const pkv::CopyItem* items, int64_t n, int64_t bytes,
                cudaStream_t s) {
  for (int64_t i = 0; i < n; ++i) {
    cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dst_base) + items[i].dst_off,
                                    static_cast<const char*>(src_base) + items[i].src_off, bytes, cudaMemcpyDefault, s);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_version(void) { return PKV_VERSION; }

const char* pkv_last_error_message(void) { return pkv::g_msg.c_str(); }

const char* pkv_status_name(int s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
    case PKV_ERR_DOUBLE_FREE: return "PKV_ERR_DOUBLE_FREE";
    case PKV_ERR_BAD_BLOCK_ID: return "PKV_ERR_BAD_BLOCK_ID";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    default: return "PKV_ERR_UNKNOWN";
  }
}

int pkv_pool_create(const pkv_geometry* geometry, const int32_t* initial_free_order, pkv_pool** out) {
  pkv::clear_error();
  if (!out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
  if (int rc = check_geometry(geometry)) return rc;
  const int64_t N = geometry->num_blocks;
  std::vector<int32_t> order(N);
  if (initial_free_order) {
    std::vector<uint8_t> seen(N, 0);
    for (int64_t i = 0; i < N; ++i) {
      int32_t p = initial_free_order[i];
      if (p < 0 || p >= N || seen[p]) return fail(PKV_ERR_INVALID_ARG, "initial_free_order is not a permutation");
      seen[p] = 1;
      order[i] = p;
    }
  } else {
    for (int64_t i = 0; i < N; ++i) order[i] = static_cast<int32_t>(i);
  }
  Pool* P = new Pool();
  P->geo = *geometry;
  P->slab_elems = static_cast<int64_t>(geometry->block_size) * geometry->d_head;
  P->block_elems = static_cast<int64_t>(geometry->L) * geometry->H_kv * P->slab_elems;
  P->block_bytes = P->block_elems * pkv::elem_size(geometry->dtype);
  P->free.reset(order);
  P->ref.assign(N, 0);
  P->dropped.assign(N, 0);
  *out = reinterpret_cast<pkv_pool*>(P);
  return PKV_OK;
}

int pkv_pool_destroy(pkv_pool* pool) {
  pkv::clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  Pool* P = as_pool(pool);
  if (P->n_prefix_caches > 0) return fail(PKV_ERR_INVALID_ARG, "destroy the pool's prefix caches first");
  pkv::destroy_tensor_maps(*P);
  delete P;
  return PKV_OK;
}

int pkv_pool_geometry(const pkv_pool* pool, pkv_geometry* out) {
  pkv::clear_error();
  if (!pool || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  *out = as_pool(pool)->geo;
  return PKV_OK;
}

int pkv_seq_create(pkv_pool* pool, int32_t* seq_id) {
  pkv::clear_error();
  if (!pool || !seq_id) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  Pool& P = *as_pool(pool);
  if (P.next_id == INT32_MAX) return fail(PKV_ERR_INVALID_ARG, "sequence ids exhausted");
  P.seqs.emplace_back();
  *seq_id = P.next_id++;
  return PKV_OK;
}

int pkv_seq_fork(pkv_pool* pool, int32_t parent, int32_t* child) {
  pkv::clear_error();
  if (!pool || !child) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  Pool& P = *as_pool(pool);
  const SeqState* par = find_seq(P, parent);
  if (!par) return unknown_seq(P, parent);
  if (par->swapped) return fail(PKV_ERR_INVALID_ARG, "cannot fork a swapped-out sequence");
  if (P.next_id == INT32_MAX) return fail(PKV_ERR_INVALID_ARG, "sequence ids exhausted");
  SeqState c;
  c.table = par->table;  // table duplication
  c.len = par->len;      // S_child = S_prefix
  for (int32_t p : c.table) ++P.ref[p];  // one more owner per shared block
  P.seqs.push_back(std::move(c));  // may move the parent's state: `par` is not used after this
  *child = P.next_id++;
  return PKV_OK;
}

int pkv_seq_free(pkv_pool* pool, int32_t seq) {
  pkv::clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  Pool& P = *as_pool(pool);
  SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq, true);
  for (int32_t p : s->table)
    if (P.ref[p] <= 0) return fail(PKV_ERR_DOUBLE_FREE, "block " + std::to_string(p) + " has no owner");
  for (int32_t p : s->table) drop_owner(P, p);
  *s = SeqState();
  s->state = 1;
  return PKV_OK;
}

int pkv_seq_len(const pkv_pool* pool, int32_t seq, int64_t* len) {
  pkv::clear_error();
  if (!pool || !len) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  const Pool& P = *as_pool(pool);
  const SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq);
  *len = s->len;
  return PKV_OK;
}

int pkv_plan_append(pkv_pool* pool, const int32_t* seq_ids, const int32_t* n_new, int32_t n, int32_t* slot_mapping,
                    int32_t* cow_pairs, int32_t* n_cow) {
  pkv::clear_error();
  if (!pool || n < 0 || (n > 0 && (!seq_ids || !n_new || !slot_mapping || !cow_pairs)) || !n_cow)
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_plan_append");
  Pool& P = *as_pool(pool);
  const int64_t B = P.geo.block_size;

  // validate, and order the requests by ascending sequence id
  std::vector<int32_t>& order = P.order;
  order.resize(n);
  bool ascending = true;
  int64_t total_tok = 0;
  for (int32_t i = 0; i < n; ++i) {
    const SeqState* s = find_seq(P, seq_ids[i]);
    if (!s) return unknown_seq(P, seq_ids[i]);
    if (s->swapped) return fail(PKV_ERR_INVALID_ARG, "sequence " + std::to_string(seq_ids[i]) + " is swapped out");
    if (n_new[i] < 0) return fail(PKV_ERR_INVALID_ARG, "n_new must be >= 0");
    if (s->len + n_new[i] > (int64_t(1) << 31) - 1) return fail(PKV_ERR_INVALID_ARG, "sequence too long");
    order[i] = i;
    if (i > 0 && seq_ids[i] <= seq_ids[i - 1]) ascending = false;
    total_tok += n_new[i];
  }
  if (total_tok > INT32_MAX) return fail(PKV_ERR_INVALID_ARG, "too many tokens in one append");
  if (!ascending) {
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return seq_ids[a] < seq_ids[b]; });
    for (int32_t k = 1; k < n; ++k)
      if (seq_ids[order[k]] == seq_ids[order[k - 1]]) return fail(PKV_ERR_INVALID_ARG, "duplicate sequence id");
  }

  // dry run: blocks needed, with owner counts as earlier copies in this call leave them
  const BlockIdx bi(B);
  int64_t needed = 0;
  for (int32_t i : order) {
    if (n_new[i] == 0) continue;
    const SeqState& s = P.seqs[seq_ids[i]];
    const int64_t len = s.len;
    if (bi.off(len) != 0) {
      const int32_t tail = s.table[bi.blk(len)];
      if (P.ref[tail] - P.dropped[tail] > 1) {
        ++needed;
        ++P.dropped[tail];
      }
    }
    needed += bi.blocks(len + n_new[i]) - bi.blocks(len);  // positions with o == 0
  }
  for (int32_t i : order) {  // reset the scratch counts
    const SeqState& s = P.seqs[seq_ids[i]];
    if (n_new[i] != 0 && bi.off(s.len) != 0) P.dropped[s.table[bi.blk(s.len)]] = 0;
  }
  if (needed > P.free.size())
    return fail(PKV_ERR_OUT_OF_BLOCKS, "append needs " + std::to_string(needed) + " blocks, " +
                                           std::to_string(P.free.size()) + " free");

  // commit; sequence i's tokens start at the caller's offset sum_{j<i} n_new[j]
  std::vector<int64_t>& first_tok = P.first_tok;
  first_tok.resize(n + 1);
  first_tok[0] = 0;
  for (int32_t i = 0; i < n; ++i) first_tok[i + 1] = first_tok[i] + n_new[i];
  int32_t cows = 0;
  for (int32_t i : order) {
    SeqState& s = P.seqs[seq_ids[i]];
    int32_t* out = slot_mapping + first_tok[i];
    for (int32_t k = 0; k < n_new[i]; ++k) {
      const int64_t t = s.len;
      const int64_t l = bi.blk(t), o = bi.off(t);
      if (o == 0) {
        s.table.push_back(P.free.pop_front());
        P.ref[s.table.back()] = 1;
      } else if (P.ref[s.table[l]] > 1) {
        const int32_t old = s.table[l];
        const int32_t fresh = P.free.pop_front();
        P.ref[fresh] = 1;
        cow_pairs[2 * cows] = old;
        cow_pairs[2 * cows + 1] = fresh;
        ++cows;
        drop_owner(P, old);
        s.table[l] = fresh;
      }
      out[k] = static_cast<int32_t>(s.table[l] * B + o);
      ++s.len;
    }
  }
  *n_cow = cows;
  return PKV_OK;
}

int pkv_export_tables(const pkv_pool* pool, const int32_t* seq_ids, int32_t n, int32_t* tables, int32_t W,
                      int32_t* seq_lens) {
  pkv::clear_error();
  if (!pool || n < 0 || W < 0 || (n > 0 && (!seq_ids || (W > 0 && !tables) || !seq_lens)))
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_export_tables");
  const Pool& P = *as_pool(pool);
  for (int32_t i = 0; i < n; ++i) {
    const SeqState* s = find_seq(P, seq_ids[i]);
    if (!s) return unknown_seq(P, seq_ids[i]);
    if (s->swapped) return fail(PKV_ERR_INVALID_ARG, "sequence " + std::to_string(seq_ids[i]) + " is swapped out");
    if (static_cast<int64_t>(s->table.size()) > W)
      return fail(PKV_ERR_INVALID_ARG, "W = " + std::to_string(W) + " is smaller than a table of " +
                                           std::to_string(s->table.size()) + " blocks");
  }
  for (int32_t i = 0; i < n; ++i) {
    const SeqState& s = *find_seq(P, seq_ids[i]);
    int32_t* row = tables + static_cast<int64_t>(i) * W;
    std::copy(s.table.begin(), s.table.end(), row);
    std::fill(row + s.table.size(), row + W, 0);
    seq_lens[i] = static_cast<int32_t>(s.len);
  }
  return PKV_OK;
}

int pkv_refcounts(const pkv_pool* pool, int32_t* out) {
  pkv::clear_error();
  if (!pool || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  const Pool& P = *as_pool(pool);
  std::copy(P.ref.begin(), P.ref.end(), out);
  return PKV_OK;
}

int pkv_free_list(const pkv_pool* pool, int32_t* out, int64_t* n) {
  pkv::clear_error();
  if (!pool || !out || !n) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  const Pool& P = *as_pool(pool);
  for (int64_t i = 0; i < P.free.size(); ++i) out[i] = P.free.front_at(i);
  *n = P.free.size();
  return PKV_OK;
}

int pkv_pool_set_kv_scales(pkv_pool* pool, float k_scale, float v_scale) {
  pkv::clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  Pool& P = *as_pool(pool);
  if (P.geo.dtype != PKV_E4M3) return fail(PKV_ERR_UNSUPPORTED, "scales apply to FP8 (PKV_E4M3) pools only");
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return fail(PKV_ERR_INVALID_ARG, "scales must be finite and > 0");
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  return PKV_OK;
}

int pkv_pool_kv_scales(const pkv_pool* pool, float* k_scale, float* v_scale) {
  pkv::clear_error();
  if (!pool || !k_scale || !v_scale) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  *k_scale = as_pool(pool)->k_scale;
  *v_scale = as_pool(pool)->v_scale;
  return PKV_OK;
}

int pkv_pool_set_swap_engine(pkv_pool* pool, int32_t engine) {
  pkv::clear_error();
  if (!pool || (engine != 0 && engine != 1)) return fail(PKV_ERR_INVALID_ARG, "engine must be 0 or 1");
  as_pool(pool)->swap_engine = engine;
  return PKV_OK;
}

// ------------------------------------------------------------------ data plane

int pkv_pool_set_prefix_sharing(pkv_pool* pool, int32_t min_members, int32_t min_blocks, int32_t target_ctas) {
  pkv::clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  Pool& P = *as_pool(pool);
  if (min_members == 0) {
    P.share_min_members = 0;
    return PKV_OK;
  }
  if (min_members < 2 || min_blocks < 1)
    return fail(PKV_ERR_INVALID_ARG, "min_members must be 0 (off) or >= 2, and min_blocks >= 1");
  if (!pkv::share_geometry_ok(P.geo))
    return fail(PKV_ERR_UNSUPPORTED, "shared prefixes need a bf16, f16 or E4M3 pool with d_head 128, at most 16 "
                                     "query heads per KV head and a block size that is a multiple of 16");
  if (target_ctas <= 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms <= 0) {
      cudaGetLastError();
      return fail(PKV_ERR_CUDA, "no device to size the prefix kernel's grid from: give target_ctas");
    }
    target_ctas = sms;
  }
  P.share_min_members = min_members;
  P.share_min_blocks = min_blocks;
  P.share_ctas = target_ctas;
  return PKV_OK;
}

int pkv_step_meta_ints(const pkv_pool* pool, int32_t n, int32_t W, int64_t* ints) {
  pkv::clear_error();
  if (!pool || n < 0 || W <= 0 || !ints) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_step_meta_ints");
  *ints = pkv::step_meta_ints(*as_pool(pool), n, W);
  return PKV_OK;
}

int pkv_append_kv(const pkv_pool* pool, int32_t layer, const void* k_new, const void* v_new,
                  const int32_t* slot_mapping, int32_t n_tok, void* k_pool, void* v_pool, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n_tok < 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_append_kv");
  const Pool& P = *as_pool(pool);
  if (layer < -1 || layer >= P.geo.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  if (n_tok > 0 && (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool))
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  return pkv::launch_append(P, layer, k_new, v_new, slot_mapping, n_tok, k_pool, v_pool, stream);
}

int pkv_decode_workspace_size(const pkv_pool* pool, int32_t n_seq, size_t* bytes) {
  pkv::clear_error();
  if (!pool || !bytes || n_seq < 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
  return pkv::decode_workspace_bytes(*as_pool(pool), n_seq, bytes);
}

int pkv_decode_attention(const pkv_pool* pool, int32_t layer, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, int32_t W, const int32_t* seq_lens, int32_t n_seq, float scale,
                         void* out, void* workspace, size_t ws_bytes, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n_seq < 0 || W < 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_decode_attention");
  const Pool& P = *as_pool(pool);
  if (layer < 0 || layer >= P.geo.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  if (n_seq == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out || !workspace)
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  return pkv::launch_decode(const_cast<Pool&>(P), layer, q, k_pool, v_pool, block_tables, W, seq_lens, n_seq, scale,
                            out, workspace, ws_bytes, stream);
}

int pkv_prefill_attention(const pkv_pool* pool, int32_t layer, const void* q, const int32_t* q_offsets, int32_t n_tok,
                          int32_t max_q, const void* k_pool, const void* v_pool, const int32_t* block_tables, int32_t W,
                          const int32_t* seq_lens, int32_t n_seq, float scale, void* out, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n_seq < 0 || W < 0 || n_tok < 0 || max_q < 0)
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_prefill_attention");
  const Pool& P = *as_pool(pool);
  if (layer < 0 || layer >= P.geo.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  if (n_seq == 0 || n_tok == 0) return PKV_OK;
  if (n_seq > 65535) return fail(PKV_ERR_INVALID_ARG, "at most 65535 sequences per call");
  if (!q || !q_offsets || !k_pool || !v_pool || !block_tables || !seq_lens || !out)
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  if (P.geo.H_q / P.geo.H_kv > 128) return fail(PKV_ERR_UNSUPPORTED, "more than 128 query heads per KV head");
  return pkv::launch_prefill(const_cast<Pool&>(P), layer, q, q_offsets, n_tok, max_q, k_pool, v_pool, block_tables,
                             W, seq_lens, n_seq, scale, out, stream);
}

int pkv_copy_blocks(const pkv_pool* pool, const int32_t* pairs, int32_t n, void* k_pool, void* v_pool,
                    pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || (n > 0 && (!pairs || !k_pool || !v_pool)))
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_copy_blocks");
  const Pool& P = *as_pool(pool);
  std::vector<uint8_t> is_dst(P.geo.num_blocks, 0), is_src(P.geo.num_blocks, 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = pairs[2 * i], d = pairs[2 * i + 1];
    if (s < 0 || s >= P.geo.num_blocks || d < 0 || d >= P.geo.num_blocks)
      return fail(PKV_ERR_BAD_BLOCK_ID, "copy pair (" + std::to_string(s) + ", " + std::to_string(d) + ") out of range");
    if (is_dst[d]) return fail(PKV_ERR_INVALID_ARG, "a destination block appears twice");
    is_dst[d] = 1;
    is_src[s] = 1;
  }
  for (int32_t i = 0; i < n; ++i)
    if (is_src[pairs[2 * i + 1]] && pairs[2 * i] != pairs[2 * i + 1])
      return fail(PKV_ERR_INVALID_ARG, "a destination block is also a source");
  std::vector<pkv::CopyItem> items(n);
  for (int32_t i = 0; i < n; ++i)
    items[i] = {pairs[2 * i] * P.block_bytes, pairs[2 * i + 1] * P.block_bytes};
  if (int rc = pkv::launch_copy_images(k_pool, k_pool, items.data(), n, P.block_bytes, stream)) return rc;
  return pkv::launch_copy_images(v_pool, v_pool, items.data(), n, P.block_bytes, stream);
}

int pkv_swap_out(pkv_pool* pool, int32_t seq, const void* k_pool, const void* v_pool, void* host, int64_t host_frames,
                 const int64_t* host_slots, int32_t n, int32_t* block_ids_out, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || host_frames < 0 || (n > 0 && (!k_pool || !v_pool || !host || !host_slots)))
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_swap_out");
  Pool& P = *as_pool(pool);
  SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq);
  if (s->swapped) return fail(PKV_ERR_INVALID_ARG, "sequence is already swapped out");
  if (s->reload_next >= 0) return fail(PKV_ERR_INVALID_ARG, "sequence is still being reloaded");
  if (static_cast<int64_t>(s->table.size()) != n)
    return fail(PKV_ERR_INVALID_ARG, "n must equal the sequence's block count (" + std::to_string(s->table.size()) + ")");
  std::unordered_map<int64_t, int> seen;
  for (int32_t j = 0; j < n; ++j) {
    if (host_slots[j] < 0 || host_slots[j] >= host_frames)
      return fail(PKV_ERR_BAD_BLOCK_ID, "host frame " + std::to_string(host_slots[j]) + " out of range");
    if (seen[host_slots[j]]++) return fail(PKV_ERR_INVALID_ARG, "a host frame appears twice");
  }
  for (int32_t p : s->table)
    if (P.ref[p] <= 0) return fail(PKV_ERR_DOUBLE_FREE, "block " + std::to_string(p) + " has no owner");
  if (n > 0) {
    void* dhost = host;
    if (P.swap_engine == 0 && !(dhost = device_view_of_host(host)))
      return fail(PKV_ERR_INVALID_ARG, "host tier is not device-accessible (use page-locked memory)");
    std::vector<pkv::CopyItem> kit(n), vit(n);
    for (int32_t j = 0; j < n; ++j) {
      const int64_t frame = host_slots[j] * 2 * P.block_bytes;
      kit[j] = {s->table[j] * P.block_bytes, frame};
      vit[j] = {s->table[j] * P.block_bytes, frame + P.block_bytes};
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int ctas = swap_ctas();
    int rc = P.swap_engine == 0 ? pkv::launch_copy_images(k_pool, dhost, kit.data(), n, P.block_bytes, st, ctas)
                                : copy_engine(k_pool, dhost, kit.data(), n, P.block_bytes, st);
    if (rc == PKV_OK)
      rc = P.swap_engine == 0 ? pkv::launch_copy_images(v_pool, dhost, vit.data(), n, P.block_bytes, st, ctas)
                              : copy_engine(v_pool, dhost, vit.data(), n, P.block_bytes, st);
    if (rc != PKV_OK) return rc;
  }
  // remap: the frames now hold the blocks; the GPU blocks lose this owner
  if (block_ids_out) std::copy(s->table.begin(), s->table.end(), block_ids_out);
  s->host_frames.assign(host_slots, host_slots + n);
  for (int32_t p : s->table) drop_owner(P, p);
  s->table.clear();
  s->swapped = true;
  return PKV_OK;
}

int pkv_swap_in(pkv_pool* pool, int32_t seq, const void* host, int64_t host_frames, int32_t n, void* k_pool,
                void* v_pool, int32_t* new_block_ids, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || (n > 0 && (!k_pool || !v_pool || !host)))
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_swap_in");
  Pool& P = *as_pool(pool);
  SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq);
  if (!s->swapped) return fail(PKV_ERR_INVALID_ARG, "sequence is not swapped out");
  if (static_cast<int64_t>(s->host_frames.size()) != n)
    return fail(PKV_ERR_INVALID_ARG, "n must equal the sequence's swapped block count (" +
                                         std::to_string(s->host_frames.size()) + ")");
  for (int64_t f : s->host_frames)
    if (f >= host_frames) return fail(PKV_ERR_BAD_BLOCK_ID, "recorded host frame beyond host_frames");
  if (P.free.size() < n)
    return fail(PKV_ERR_OUT_OF_BLOCKS, "swap-in needs " + std::to_string(n) + " blocks, " +
                                           std::to_string(P.free.size()) + " free");
  if (n > 0) {
    void* dhost = const_cast<void*>(host);
    if (P.swap_engine == 0 && !(dhost = device_view_of_host(dhost)))
      return fail(PKV_ERR_INVALID_ARG, "host tier is not device-accessible (use page-locked memory)");
    std::vector<pkv::CopyItem> kit(n), vit(n);
    for (int32_t j = 0; j < n; ++j) {
      const int64_t frame = s->host_frames[j] * 2 * P.block_bytes;
      const int64_t blk = P.free.front_at(j) * P.block_bytes;  // the blocks that will be popped
      kit[j] = {frame, blk};
      vit[j] = {frame + P.block_bytes, blk};
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int ctas = swap_ctas();
    int rc = P.swap_engine == 0 ? pkv::launch_copy_images(dhost, k_pool, kit.data(), n, P.block_bytes, st, ctas)
                                : copy_engine(dhost, k_pool, kit.data(), n, P.block_bytes, st);
    if (rc == PKV_OK)
      rc = P.swap_engine == 0 ? pkv::launch_copy_images(dhost, v_pool, vit.data(), n, P.block_bytes, st, ctas)
                              : copy_engine(dhost, v_pool, vit.data(), n, P.block_bytes, st);
    if (rc != PKV_OK) return rc;
  }
  for (int32_t j = 0; j < n; ++j) {
    const int32_t p = P.free.pop_front();
    P.ref[p] = 1;
    s->table.push_back(p);
    if (new_block_ids) new_block_ids[j] = p;
  }
  s->host_frames.clear();
  s->swapped = false;
  return PKV_OK;
}

// CTAs of the SM copier in a reload by layers: 32 keep the host link at its copy rate (~205 GB/s
// alone) and leave the other SMs to the prefill the reload runs behind (16 reach ~175 GB/s; 128
// slow the prefill).  PKV_RELOAD_CTAS overrides it for tuning.
static int reload_ctas() {
  if (const char* e = std::getenv("PKV_RELOAD_CTAS")) return std::max(1, std::atoi(e));
  return 32;
}

int pkv_swap_in_layers(pkv_pool* pool, int32_t seq, const void* host, int64_t host_frames, int32_t n,
                       int32_t layer_begin, int32_t layer_end, void* k_pool, void* v_pool, int32_t* new_block_ids,
                       pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || (n > 0 && (!k_pool || !v_pool || !host)))
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_swap_in_layers");
  Pool& P = *as_pool(pool);
  SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq);
  const int32_t L = P.geo.L;
  if (layer_begin < 0 || layer_end <= layer_begin || layer_end > L)
    return fail(PKV_ERR_INVALID_ARG, "layer range must satisfy 0 <= layer_begin < layer_end <= L");
  const bool first = s->swapped;
  if (first) {
    if (layer_begin != 0) return fail(PKV_ERR_INVALID_ARG, "a reload starts at layer 0");
  } else {
    if (s->reload_next < 0) return fail(PKV_ERR_INVALID_ARG, "sequence is neither swapped out nor being reloaded");
    if (layer_begin != s->reload_next)
      return fail(PKV_ERR_INVALID_ARG, "layer ranges must follow each other: the next one starts at layer " +
                                           std::to_string(s->reload_next));
  }
  if (static_cast<int64_t>(s->host_frames.size()) != n)
    return fail(PKV_ERR_INVALID_ARG, "n must equal the sequence's swapped block count (" +
                                         std::to_string(s->host_frames.size()) + ")");
  for (int64_t f : s->host_frames)
    if (f >= host_frames) return fail(PKV_ERR_BAD_BLOCK_ID, "recorded host frame beyond host_frames");
  if (first && P.free.size() < n)
    return fail(PKV_ERR_OUT_OF_BLOCKS, "swap-in needs " + std::to_string(n) + " blocks, " +
                                           std::to_string(P.free.size()) + " free");
  if (n > 0) {
    const int kReloadCtas = reload_ctas();
    void* dhost = const_cast<void*>(host);
    if (P.swap_engine == 0 && !(dhost = device_view_of_host(dhost)))
      return fail(PKV_ERR_INVALID_ARG, "host tier is not device-accessible (use page-locked memory)");
    // a block image and a frame half are [L][H_kv][B][d]: the layer range is one contiguous piece of each
    const int64_t layer_bytes = P.block_bytes / L;
    const int64_t off = layer_begin * layer_bytes, bytes = (layer_end - layer_begin) * layer_bytes;
    std::vector<pkv::CopyItem> kit(n), vit(n);
    for (int32_t j = 0; j < n; ++j) {
      const int64_t frame = s->host_frames[j] * 2 * P.block_bytes;
      const int64_t blk = static_cast<int64_t>(first ? P.free.front_at(j) : s->table[j]) * P.block_bytes;
      kit[j] = {frame + off, blk + off};
      vit[j] = {frame + P.block_bytes + off, blk + off};
    }
    // a reload shares the GPU with the prefill it runs behind: the SM copier takes a few SMs only
    // (kReloadCtas CTAs keep the host link busy), not one CTA per 128 KiB
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = P.swap_engine == 0 ? pkv::launch_copy_images(dhost, k_pool, kit.data(), n, bytes, st, kReloadCtas)
                                : copy_engine(dhost, k_pool, kit.data(), n, bytes, st);
    if (rc == PKV_OK)
      rc = P.swap_engine == 0 ? pkv::launch_copy_images(dhost, v_pool, vit.data(), n, bytes, st, kReloadCtas)
                              : copy_engine(dhost, v_pool, vit.data(), n, bytes, st);
    if (rc != PKV_OK) return rc;
  }
  if (first) {  // allocate and remap exactly as pkv_swap_in does
    for (int32_t j = 0; j < n; ++j) {
      const int32_t p = P.free.pop_front();
      P.ref[p] = 1;
      s->table.push_back(p);
    }
    s->swapped = false;
  }
  if (new_block_ids) std::copy(s->table.begin(), s->table.end(), new_block_ids);
  s->reload_next = layer_end;
  if (layer_end == L) {  // every layer is back
    s->host_frames.clear();
    s->reload_next = -1;
  }
  return PKV_OK;
}

int pkv_seq_residency(const pkv_pool* pool, int32_t seq, int32_t* tier) {
  pkv::clear_error();
  if (!pool || !tier) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  const Pool& P = *as_pool(pool);
  const SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq);
  *tier = s->swapped ? PKV_TIER_HOST : (s->reload_next >= 0 ? PKV_TIER_RELOADING : PKV_TIER_HBM);
  return PKV_OK;
}

int pkv_seq_host_slots(const pkv_pool* pool, int32_t seq, int64_t* out, int32_t capacity, int32_t* n) {
  pkv::clear_error();
  if (!pool || !n || capacity < 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
  const Pool& P = *as_pool(pool);
  const SeqState* s = find_seq(P, seq);
  if (!s) return unknown_seq(P, seq);
  if (!s->swapped && s->reload_next < 0) return fail(PKV_ERR_INVALID_ARG, "sequence is not swapped out");
  *n = static_cast<int32_t>(s->host_frames.size());
  if (out)
    for (int32_t j = 0; j < *n && j < capacity; ++j) out[j] = s->host_frames[j];
  return PKV_OK;
}

// The checks pkv_decode_step makes before anything changes: resident, unswapped sequences whose
// tables still fit W after one more token.
static int step_check(pkv_pool* pool, const int32_t* seq_ids, int32_t n, int32_t W) {
  const Pool& CP = *as_pool(pool);
  const BlockIdx bi(CP.geo.block_size);
  for (int32_t i = 0; i < n; ++i) {
    const SeqState* s = find_seq(CP, seq_ids[i]);
    if (!s) return unknown_seq(CP, seq_ids[i]);
    if (s->swapped) return fail(PKV_ERR_INVALID_ARG, "sequence " + std::to_string(seq_ids[i]) + " is swapped out");
    if (bi.blocks(s->len + 1) > W)
      return fail(PKV_ERR_INVALID_ARG, "W = " + std::to_string(W) + " cannot hold sequence " +
                                           std::to_string(seq_ids[i]) + " after the step");
  }
  return PKV_OK;
}

static int step_workspace_check(pkv_pool* pool, int32_t n, size_t ws_bytes) {
  size_t need = 0;
  if (int rc = pkv::decode_workspace_bytes(*as_pool(pool), n, &need)) return rc;
  if (ws_bytes < need) return fail(PKV_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(need));
  return PKV_OK;
}

// The shared-prefix plan of a step's batch (layout in pkv_internal.h), from the tables after the
// step's append.  A run of consecutive rows is a group when every row after the first shares at
// least min_blocks leading blocks with the first (the same physical blocks: a fork's prefix)
// and at least half of what the rows before it share; the group's prefix is the blocks all of
// them share, cut so that every row keeps at least one token of its own (so no row's shared
// blocks are written in this step).  Groups of fewer than min_members rows are dropped.  Each
// group's prefix is cut into splits of whole blocks so that the prefix kernel's grid (CTAs =
// member pairs of 128-row tiles x KV heads x splits, over all groups) comes near a target,
// splits of at least 256 keys, within the plan's item and slot caps.
//
// The target: the prefix kernel is bound by the tensor cores and the decode of the rows' own
// blocks by HBM, which on this GPU needs only ~96 SMs for its full rate.  With 16-bit pools and
// groups of up to 8 query heads the step can run the two side by side: the decode on S SMs (one
// 8-warp CTA on each, header word 3 = S) and the prefix kernel's CTAs, one per SM, on the others.
// S and the target come from a time model of the two kernels measured on GB300 -- decode: 10 us +
// own K/V bytes / min(6.95 TB/s, S x 70 GB/s) (a CTA's shared memory caps its bytes in flight;
// 70 GB/s an SM is what the forked shape's short pairs reach); prefix: 12 us + (keys of a split) x
// (128-row tiles of a CTA) x 8.6 ns -- taking the S that minimises the larger of the two, unless
// running them one after the other on all share_ctas SMs (header word 3 = 0) is estimated faster.
// (FP8 pools move half the bytes per tile in flight, so their decode keeps every SM.)  The model
// only places work; any choice gives the same results.
static void plan_sharing(Pool& P, const int32_t* ids, int32_t n, int32_t* plan) {
  const int64_t B = P.geo.block_size;
  int32_t* rows = plan + 4;
  int32_t* items = plan + 4 + 4 * static_cast<int64_t>(n);
  std::fill(plan, plan + 4 + 4 * static_cast<int64_t>(n), 0);
  std::vector<int32_t>& grp = P.share_scratch;  // (row_begin, row_end, blocks, splits) per group
  grp.clear();
  for (int32_t i = 0; i < n;) {
    const SeqState& a = P.seqs[ids[i]];
    int64_t c = (a.len - 1) / B;  // blocks that leave row i a token of its own
    int32_t j = i + 1;
    while (j < n && c >= P.share_min_blocks) {
      const SeqState& b = P.seqs[ids[j]];
      const int64_t cb = std::min<int64_t>(c, (b.len - 1) / B);
      int64_t k = 0;  // the common leading entries: 64 at a time while they match, then one by one
      while (k + 64 <= cb && std::memcmp(a.table.data() + k, b.table.data() + k, 64 * sizeof(int32_t)) == 0)
        k += 64;
      while (k < cb && a.table[k] == b.table[k]) ++k;
      if (k < P.share_min_blocks || 2 * k < c) break;
      c = k;
      ++j;
    }
    if (j - i >= P.share_min_members && c >= P.share_min_blocks) {
      grp.insert(grp.end(), {i, j, static_cast<int32_t>(c), 1});
      i = j;
    } else {
      ++i;
    }
  }
  const int64_t ng = static_cast<int64_t>(grp.size()) / 4;
  if (ng == 0) return;
  const int64_t G = P.geo.H_q / P.geo.H_kv, QB = 128 / G, per_cta = 2 * QB;
  auto ctas_of = [&](int64_t gi) { return (grp[4 * gi + 1] - grp[4 * gi] + per_cta - 1) / per_cta * P.geo.H_kv; };
  double total = 0.0;
  for (int64_t gi = 0; gi < ng; ++gi) total += static_cast<double>(ctas_of(gi)) * grp[4 * gi + 2];
  // splits of every group for a grid target; returns (CTAs, the longest CTA's keys x tiles)
  auto assign = [&](double target, int64_t* ctas, double* longest) {
    *ctas = 0;
    *longest = 0.0;
    for (int64_t gi = 0; gi < ng; ++gi) {
      const int64_t ct = ctas_of(gi), kb = grp[4 * gi + 2], m = grp[4 * gi + 1] - grp[4 * gi];
      const double want = target * (static_cast<double>(ct) * kb / total) / ct;
      const int64_t most = std::max<int64_t>(1, kb * B / 256);
      const int64_t sp = std::max<int64_t>(1, std::min<int64_t>(most, static_cast<int64_t>(want)));
      grp[4 * gi + 3] = static_cast<int32_t>(sp);
      const int64_t bps = (kb + sp - 1) / sp;
      *ctas += ct * ((kb + bps - 1) / bps);
      *longest = std::max(*longest, static_cast<double>(bps * B) * (m > QB ? 2 : 1));
    }
  };
  int32_t decode_sms = 0;
  {
    // the decode's own bytes: every row's tokens after its shared blocks
    double own = 0.0;
    for (int32_t r = 0, gi = 0; r < n; ++r) {
      while (gi < ng && grp[4 * gi + 1] <= r) ++gi;
      const int64_t kb = (gi < ng && grp[4 * gi] <= r) ? grp[4 * gi + 2] : 0;
      own += static_cast<double>(P.seqs[ids[r]].len - kb * B);
    }
    own *= static_cast<double>(P.geo.H_kv) * P.geo.d_head * pkv::elem_size(P.geo.dtype) * 2;
    auto t_decode = [&](double sms) { return 10e-6 + own / std::min(6.95e12, sms * 70e9); };
    auto t_prefix = [&](double longest) { return 12e-6 + longest * 8.6e-9; };
    int64_t ctas = 0;
    double longest = 0.0;
    assign(P.share_ctas, &ctas, &longest);
    double best = t_decode(P.share_ctas) + t_prefix(longest), best_target = P.share_ctas;
    if (G <= 8 && P.geo.dtype != PKV_E4M3)
      for (int32_t target = 8; target <= P.share_ctas - 8; target += 4) {
        assign(target, &ctas, &longest);
        const int64_t sms = P.share_ctas - ctas;
        if (sms < 8) continue;
        const double t = std::max(t_decode(static_cast<double>(sms)), t_prefix(longest));
        if (t < best) {
          best = t;
          best_target = target;
          decode_sms = static_cast<int32_t>(sms);
        }
      }
    assign(best_target, &ctas, &longest);
  }
  int64_t n_items = 0, n_slots = 0;
  for (int64_t gi = 0; gi < ng; ++gi) {
    n_items += grp[4 * gi + 3];
    n_slots += static_cast<int64_t>(grp[4 * gi + 3]) * (grp[4 * gi + 1] - grp[4 * gi]);
  }
  // within the caps: fewer splits where there are most, then fewer groups
  while (n_items > pkv::share_item_cap(n) || n_slots > pkv::share_slot_cap(n)) {
    int64_t best = -1;
    for (int64_t gi = 0; gi < ng; ++gi)
      if (grp[4 * gi + 3] > 1 && (best < 0 || grp[4 * gi + 3] > grp[4 * best + 3])) best = gi;
    if (best < 0) break;
    --grp[4 * best + 3];
    --n_items;
    n_slots -= grp[4 * best + 1] - grp[4 * best];
  }
  int64_t kept = ng;
  while (kept > 0 && (n_items > pkv::share_item_cap(n) || n_slots > pkv::share_slot_cap(n))) {
    --kept;
    n_items -= grp[4 * kept + 3];
    n_slots -= static_cast<int64_t>(grp[4 * kept + 3]) * (grp[4 * kept + 1] - grp[4 * kept]);
  }
  int32_t it = 0, slot = 0, max_members = 0;
  for (int64_t gi = 0; gi < kept; ++gi) {
    const int32_t rb = grp[4 * gi], re = grp[4 * gi + 1], kb = grp[4 * gi + 2], m = re - rb;
    const int32_t bps = (kb + grp[4 * gi + 3] - 1) / grp[4 * gi + 3];
    const int32_t splits = (kb + bps - 1) / bps;
    for (int32_t k = 0; k < splits; ++k, ++it) {
      int32_t* e = items + 8 * static_cast<int64_t>(it);
      e[0] = rb;
      e[1] = re;
      e[2] = k * bps;
      e[3] = std::min(kb, (k + 1) * bps);
      e[4] = slot + k * m;
      e[5] = e[6] = e[7] = 0;
    }
    for (int32_t r = rb; r < re; ++r) {
      int32_t* w = rows + 4 * static_cast<int64_t>(r);
      w[0] = kb;
      w[1] = splits;
      w[2] = slot + (r - rb);
      w[3] = m;
    }
    slot += splits * m;
    max_members = std::max(max_members, m);
  }
  plan[0] = it;
  plan[1] = max_members;
  plan[2] = slot;
  plan[3] = it > 0 ? decode_sms : 0;
}

int pkv_step_plan(pkv_pool* pool, const int32_t* seq_ids, int32_t n, int32_t W, int32_t* meta_host,
                  int32_t* cow_pairs, int32_t* n_cow) {
  pkv::clear_error();
  if (!pool || n < 0 || W <= 0 || !n_cow) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_step_plan");
  *n_cow = 0;
  if (n == 0) return PKV_OK;
  if (!seq_ids || !meta_host || !cow_pairs) return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  if (int rc = step_check(pool, seq_ids, n, W)) return rc;
  static thread_local std::vector<int32_t> ones;
  if (static_cast<int32_t>(ones.size()) < n) ones.assign(n, 1);
  int32_t* slots = meta_host;
  int32_t* tables = meta_host + n;
  int32_t* lens = meta_host + n + static_cast<int64_t>(n) * W;
  if (int rc = pkv_plan_append(pool, seq_ids, ones.data(), n, slots, cow_pairs, n_cow)) return rc;
  Pool& P = *as_pool(pool);
  // with sharing on, the plan first: a run's shared blocks are read only from its first row's
  // table (the prefix kernel), so the other rows' copies of them need not be written
  const int32_t* share_rows = nullptr;
  std::vector<uint8_t>& first = P.share_first;
  if (pkv::share_on(P)) {
    int32_t* plan = meta_host + pkv::share_plan_offset(n, W);
    std::fill(meta_host + static_cast<int64_t>(n) * (W + 2), plan, 0);  // the alignment gap
    plan_sharing(P, seq_ids, n, plan);
    share_rows = plan + 4;
    first.assign(n, 0);
    const int32_t* items = plan + 4 + 4 * static_cast<int64_t>(n);
    for (int32_t it = 0; it < plan[0]; ++it) first[items[8 * it]] = 1;
  }
  // the tables and lengths after the append (the sequences were checked above); entries past a
  // table's end, and a run's shared entries in its rows after the first, are left as they were:
  // no kernel reads them
  for (int32_t i = 0; i < n; ++i) {
    const SeqState& s = P.seqs[seq_ids[i]];
    const int64_t from = (share_rows && !first[i]) ? share_rows[4 * static_cast<int64_t>(i)] : 0;
    std::copy(s.table.begin() + from, s.table.end(), tables + static_cast<int64_t>(i) * W + from);
    lens[i] = static_cast<int32_t>(s.len);
  }
  return PKV_OK;
}

// The device half of a decode step; meta_host NULL: meta_dev already holds the plan, whose host
// copy is at plan_host (read for the shared-prefix header).
static int step_launch(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs, int32_t n_cow,
                       const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool, float scale,
                       void* out, const int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes,
                       pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream,
                       const int32_t* plan_host = nullptr) {
  if (!pool || n < 0 || W <= 0 || n_cow < 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to the step launch");
  if (n == 0) return PKV_OK;
  if (!q || !k_new || !v_new || !k_pool || !v_pool || !out || !meta_dev || !workspace || (n_cow > 0 && !cow_pairs))
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  if (layer < 0 || layer >= as_pool(pool)->geo.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  if (int rc = step_workspace_check(pool, n, ws_bytes)) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Pool& P = *as_pool(pool);
  if (meta_host) {
    const size_t meta_bytes = sizeof(int32_t) * static_cast<size_t>(pkv::step_meta_ints(P, n, W));
    cudaError_t e = cudaMemcpyAsync(meta_dev, meta_host, meta_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
      return fail(PKV_ERR_CUDA, std::string("cudaMemcpyAsync (step metadata): ") + cudaGetErrorString(e));
    plan_host = meta_host;
  }
  if (pkv::share_on(P) && !plan_host)
    return fail(PKV_ERR_INVALID_ARG, "with prefix sharing on, the launch needs the step's host metadata");
  pkv::ShareLaunch share{nullptr, 0, 0, 0};
  bool long_batch = false;
  if (plan_host) {  // the lengths after the append: tiles per (sequence, KV head) pair on average
    const int32_t* lens = plan_host + n + static_cast<int64_t>(n) * W;
    int64_t tiles = 0;
    for (int32_t i = 0; i < n; ++i) tiles += (static_cast<int64_t>(lens[i]) + 15) / 16;
    long_batch = tiles >= 1024ll * n;
  }
  if (pkv::share_on(P) && plan_host) {
    const int64_t off = pkv::share_plan_offset(n, W);
    const int32_t* hdr = plan_host + off;
    if (hdr[0] < 0 || hdr[0] > pkv::share_item_cap(n) || hdr[1] < 0 || hdr[1] > n || hdr[2] < 0 ||
        hdr[2] > pkv::share_slot_cap(n) || hdr[3] < 0 || hdr[3] > P.share_ctas)
      return fail(PKV_ERR_INVALID_ARG, "the step metadata's shared-prefix plan is corrupt");
    share = pkv::ShareLaunch{meta_dev + off, hdr[0], hdr[1], hdr[3]};
  }
  if (n_cow > 0)
    if (int rc = pkv_copy_blocks(pool, cow_pairs, n_cow, k_pool, v_pool, stream)) return rc;
  // append and attention in one launch on the tensor-core path (the kernel writes each new
  // token before it loads the tile that holds it); the append kernel first otherwise
  if (attn_begin) cudaEventRecord(reinterpret_cast<cudaEvent_t>(attn_begin), st);
  const pkv::AppendFuse fuse{k_new, v_new, meta_dev, k_pool, v_pool};
  if (int rc = pkv::launch_decode(*as_pool(pool), layer, q, k_pool, v_pool, meta_dev + n, W,
                                  meta_dev + n + static_cast<int64_t>(n) * W, n, scale, out, workspace, ws_bytes,
                                  stream, &fuse, &share, long_batch))
    return rc;
  if (attn_end) cudaEventRecord(reinterpret_cast<cudaEvent_t>(attn_end), st);
  return PKV_OK;
}

int pkv_step_launch(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs, int32_t n_cow,
                    const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool, float scale,
                    void* out, const int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes,
                    pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream) {
  pkv::clear_error();
  if (n > 0 && !meta_host) return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  return step_launch(pool, layer, n, W, cow_pairs, n_cow, q, k_new, v_new, k_pool, v_pool, scale, out, meta_host,
                     meta_dev, workspace, ws_bytes, attn_begin, attn_end, stream);
}

int pkv_step_launch_packed(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs,
                           int32_t n_cow, const void* in_host, void* in_dev, size_t off_k, size_t off_v,
                           size_t off_meta, size_t in_bytes, void* out_host, void* out_dev, void* k_pool,
                           void* v_pool, float scale, const int32_t* meta_host, int32_t* meta_dev, void* workspace,
                           size_t ws_bytes, pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || W <= 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_step_launch_packed");
  if (n == 0) return PKV_OK;
  if (!in_host || !in_dev || !out_host || !out_dev) return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  const pkv_geometry& g = as_pool(pool)->geo;
  const size_t ab = static_cast<size_t>(pkv::act_size(g.dtype));
  const size_t qb = ab * n * g.H_q * g.d_head, kb = ab * n * g.H_kv * g.d_head;
  const size_t mb = sizeof(int32_t) * static_cast<size_t>(pkv::step_meta_ints(*as_pool(pool), n, W));
  if ((off_k | off_v | off_meta) & 15) return fail(PKV_ERR_INVALID_ARG, "offsets must be multiples of 16");
  if (off_k < qb || off_v < off_k + kb || in_bytes < off_v + kb || (off_meta && (off_meta < off_v + kb ||
                                                                                 in_bytes < off_meta + mb)))
    return fail(PKV_ERR_INVALID_ARG, "packed input: q, k_new, v_new (and the metadata) of n rows must fit before "
                                     "off_k, off_v, off_meta and in_bytes");
  if (pkv::share_on(*as_pool(pool)) && !off_meta && !meta_host)
    return fail(PKV_ERR_INVALID_ARG, "with prefix sharing on, the launch reads the step's plan from the host "
                                     "metadata: pass meta_host or pack the metadata (off_meta)");
  const int32_t* plan_host = meta_host;
  if (off_meta) {  // the metadata travels with the inputs
    plan_host = reinterpret_cast<const int32_t*>(static_cast<const char*>(in_host) + off_meta);
    meta_host = nullptr;
    meta_dev = reinterpret_cast<int32_t*>(static_cast<char*>(in_dev) + off_meta);
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(in_dev, in_host, in_bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaMemcpyAsync (step input): ") + cudaGetErrorString(e));
  char* d = static_cast<char*>(in_dev);
  if (int rc = step_launch(pool, layer, n, W, cow_pairs, n_cow, d, d + off_k, d + off_v, k_pool, v_pool, scale,
                           out_dev, meta_host, meta_dev, workspace, ws_bytes, attn_begin, attn_end, stream, plan_host))
    return rc;
  e = cudaMemcpyAsync(out_host, out_dev, qb, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaMemcpyAsync (step result): ") + cudaGetErrorString(e));
  return PKV_OK;
}

int pkv_step_launch_host(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs,
                         int32_t n_cow, const void* q_host, const void* k_new_host, const void* v_new_host,
                         void* out_host, void* q_dev, void* k_new_dev, void* v_new_dev, void* out_dev, void* k_pool,
                         void* v_pool, float scale, const int32_t* meta_host, int32_t* meta_dev, void* workspace,
                         size_t ws_bytes, pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || W <= 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_step_launch_host");
  if (n == 0) return PKV_OK;
  if (!q_host || !k_new_host || !v_new_host || !out_host || !q_dev || !k_new_dev || !v_new_dev || !out_dev)
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  const pkv_geometry& g = as_pool(pool)->geo;
  const size_t ab = static_cast<size_t>(pkv::act_size(g.dtype));
  const size_t qb = ab * n * g.H_q * g.d_head, kb = ab * n * g.H_kv * g.d_head;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const struct {
    void* dst;
    const void* src;
    size_t bytes;
  } in[3] = {{q_dev, q_host, qb}, {k_new_dev, k_new_host, kb}, {v_new_dev, v_new_host, kb}};
  for (const auto& c : in) {
    const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaMemcpyAsync (step input): ") + cudaGetErrorString(e));
  }
  if (int rc = pkv_step_launch(pool, layer, n, W, cow_pairs, n_cow, q_dev, k_new_dev, v_new_dev, k_pool, v_pool, scale,
                               out_dev, meta_host, meta_dev, workspace, ws_bytes, attn_begin, attn_end, stream))
    return rc;
  const cudaError_t e = cudaMemcpyAsync(out_host, out_dev, qb, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, std::string("cudaMemcpyAsync (step result): ") + cudaGetErrorString(e));
  return PKV_OK;
}

int pkv_decode_step(pkv_pool* pool, int32_t layer, const int32_t* seq_ids, int32_t n, int32_t W, const void* q,
                    const void* k_new, const void* v_new, void* k_pool, void* v_pool, float scale, void* out,
                    int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes, pkv_event_t attn_begin,
                    pkv_event_t attn_end, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || W <= 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_decode_step");
  if (n == 0) return PKV_OK;
  if (!seq_ids || !q || !k_new || !v_new || !k_pool || !v_pool || !out || !meta_host || !meta_dev || !workspace)
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  if (layer < 0 || layer >= as_pool(pool)->geo.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  // everything is validated before the plan changes any state
  if (int rc = step_check(pool, seq_ids, n, W)) return rc;
  if (int rc = step_workspace_check(pool, n, ws_bytes)) return rc;
  static thread_local std::vector<int32_t> cows;
  if (static_cast<int32_t>(cows.size()) < 2 * n) cows.resize(2 * n);
  int32_t n_cow = 0;
  if (int rc = pkv_step_plan(pool, seq_ids, n, W, meta_host, cows.data(), &n_cow)) return rc;
  return pkv_step_launch(pool, layer, n, W, cows.data(), n_cow, q, k_new, v_new, k_pool, v_pool, scale, out,
                         meta_host, meta_dev, workspace, ws_bytes, attn_begin, attn_end, stream);
}

int pkv_decode_step_host(pkv_pool* pool, int32_t layer, const int32_t* seq_ids, int32_t n, int32_t W,
                         const void* q_host, const void* k_new_host, const void* v_new_host, void* out_host,
                         void* q_dev, void* k_new_dev, void* v_new_dev, void* out_dev, void* k_pool, void* v_pool,
                         float scale, int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes,
                         pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream) {
  pkv::clear_error();
  if (!pool || n < 0 || W <= 0) return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_decode_step_host");
  if (n == 0) return PKV_OK;
  if (!seq_ids || !q_host || !k_new_host || !v_new_host || !out_host || !q_dev || !k_new_dev || !v_new_dev ||
      !out_dev || !k_pool || !v_pool || !meta_host || !meta_dev || !workspace)
    return fail(PKV_ERR_INVALID_ARG, "NULL buffer");
  if (layer < 0 || layer >= as_pool(pool)->geo.L) return fail(PKV_ERR_INVALID_ARG, "layer out of range");
  if (int rc = step_check(pool, seq_ids, n, W)) return rc;
  if (int rc = step_workspace_check(pool, n, ws_bytes)) return rc;
  static thread_local std::vector<int32_t> cows;
  if (static_cast<int32_t>(cows.size()) < 2 * n) cows.resize(2 * n);
  int32_t n_cow = 0;
  if (int rc = pkv_step_plan(pool, seq_ids, n, W, meta_host, cows.data(), &n_cow)) return rc;
  return pkv_step_launch_host(pool, layer, n, W, cows.data(), n_cow, q_host, k_new_host, v_new_host, out_host, q_dev,
                              k_new_dev, v_new_dev, out_dev, k_pool, v_pool, scale, meta_host, meta_dev, workspace,
                              ws_bytes, attn_begin, attn_end, stream);
}

}  // extern "C"
