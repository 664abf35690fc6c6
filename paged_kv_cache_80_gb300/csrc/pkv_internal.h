// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace pkv {

// ------------------------------------------------------------------ errors

// Set the thread-local message and return the status (for `return fail(...)`).
int fail(int status, const std::string& msg);
void clear_error();

// ------------------------------------------------------------------ control plane

// FIFO of free block ids kept in a fixed ring of capacity num_blocks
// ("free-list ring buffer", KV Cache Management, PagedAttention model).
class FreeRing {
 public:
  void reset(const std::vector<int32_t>& order);
  int64_t size() const { return count_; }
  int32_t front_at(int64_t i) const { return ring_[(head_ + i) % cap_]; }
  int32_t pop_front();
  void push_back(int32_t p);

 private:
  std::vector<int32_t> ring_;
  int64_t cap_ = 0, head_ = 0, count_ = 0;
};

struct SeqState {
  std::vector<int32_t> table;       // logical block -> physical block
  int64_t len = 0;                  // tokens written
  uint8_t state = 0;                // 0 live, 1 released
  bool swapped = false;             // blocks live in host frames
  std::vector<int64_t> host_frames; // frames holding the blocks while swapped (or being reloaded)
  int32_t reload_next = -1;         // a reload by layer ranges: layers [reload_next, L) still to copy
};

struct TensorMaps;  // cached TMA descriptors (defined in pkv_decode.cu)

struct Pool {
  pkv_geometry geo{};
  int64_t slab_elems = 0;   // B * d: one (block, layer, head) slab
  int64_t block_elems = 0;  // L * H_kv * B * d: one block of K (or V), all layers
  int64_t block_bytes = 0;  // block_elems * element size
  FreeRing free;
  std::vector<int32_t> ref;
  // Sequence ids are 0, 1, 2, ... and never reused, so states are indexed by id;
  // a released sequence keeps an empty state marked released.
  std::vector<SeqState> seqs;
  std::vector<int32_t> dropped;  // per block: owners given up by earlier CoWs of one append (dry run)
  std::vector<int32_t> order;    // scratch: request order of one append
  std::vector<int64_t> first_tok;  // scratch: caller offsets of one append
  int32_t next_id = 0;
  int32_t swap_engine = 0;  // 0 SM kernel, 1 copy engine
  float k_scale = 1.f, v_scale = 1.f;  // FP8 pools: stored code * scale
  int32_t n_prefix_caches = 0;         // live radix prefix caches holding references
  // shared prefixes in decode steps (pkv_pool_set_prefix_sharing): off while share_min_members == 0;
  // share_ctas: the SMs a step may use
  int32_t share_min_members = 0, share_min_blocks = 1, share_ctas = 0;
  std::vector<int32_t> share_scratch;  // planner scratch
  std::vector<uint8_t> share_first;    // planner scratch: rows that begin a run

  std::mutex tmap_mu;
  TensorMaps* tmaps = nullptr;
};

// Bytes of one stored pool element.
inline int64_t elem_size(int32_t dtype) { return dtype == PKV_F32 ? 4 : (dtype == PKV_E4M3 ? 1 : 2); }
// Bytes of one activation element (q, out, new keys/values): bf16 around an FP8 pool.
inline int64_t act_size(int32_t dtype) { return dtype == PKV_E4M3 ? 2 : elem_size(dtype); }

// ------------------------------------------------------------------ shared prefixes
//
// A decode step whose batch holds runs of rows that share their first table blocks (branches
// forked from one parent: "Zero-copy deliberation via copy-on-write branching") attends to the
// shared blocks once for the whole run, in the prefix kernel, and to each row's own blocks in the
// decode kernel; the combine kernel merges the two.  The plan (int32), made on the host with the
// step's metadata and copied with it: a header {n_items, max_members, n_slots, decode SMs}; per
// batch row {kb, items, slot0, stride} (the row's first kb blocks are shared; its prefix partials
// sit in slots slot0 + i * stride, i < items); then up to share_item_cap(n) work items of 8 ints
// {row_begin, row_end, kb0, kb1, slot_base, 0, 0, 0}: the rows, the range of row_begin's table
// blocks, and the slot of row_begin's partial.
inline int64_t share_item_cap(int64_t n) { return n + 256; }
inline int64_t share_slot_cap(int64_t n) { return 2 * n + 1024; }
inline int64_t share_plan_ints(int64_t n) { return 4 + 4 * n + 8 * share_item_cap(n); }
// The geometry the prefix kernel takes (tcgen05, d_head 128, up to 16 query heads per KV head).
inline bool share_geometry_ok(const pkv_geometry& g) {
  const int64_t G = g.H_q / g.H_kv;
  return (g.dtype == PKV_BF16 || g.dtype == PKV_F16 || g.dtype == PKV_E4M3) && g.d_head == 128 && G <= 16 &&
         g.block_size % 16 == 0 && g.num_blocks * g.L * g.H_kv * g.block_size < (int64_t(1) << 31);
}
inline bool share_on(const Pool& P) { return P.share_min_members > 0; }
// Step metadata: slots [n], tables [n][W], lens [n], then (sharing on) the plan from a 16-byte boundary.
inline int64_t share_plan_offset(int64_t n, int64_t W) { return (n * (W + 2) + 3) / 4 * 4; }
inline int64_t step_meta_ints(const Pool& P, int64_t n, int64_t W) {
  return share_on(P) ? share_plan_offset(n, W) + share_plan_ints(n) : n * (W + 2);
}
// The shared-prefix part of a decode launch: the plan on the device and its header's counts;
// decode_sms > 0: the decode kernel runs as one 8-warp CTA on each of that many SMs, beside the
// prefix kernel on the others (0: on every SM, then the prefix kernel).
struct ShareLaunch {
  const int32_t* plan_dev;
  int32_t n_items, max_members, decode_sms;
};

// ------------------------------------------------------------------ device side

// Count one kernel launch (reported by pkv_launch_count).
void count_launch(int n = 1);

// Address of the current device's error word: int32 code, int32 pad, int64 detail.
int device_error_word(void** out);

// Kernel launchers (return PKV_OK or a failure with the message set).
struct CopyItem {
  int64_t src_off;  // byte offsets
  int64_t dst_off;
};

// lets_dependents: the kernel lets a programmatic dependent launched right after it start
// before it completes (the decode step's attention, which waits for it before loading K/V).
int launch_append(const Pool& P, int32_t layer, const void* k_new, const void* v_new, const int32_t* slots,
                  int32_t n_tok, void* k_pool, void* v_pool, void* stream, bool lets_dependents = false);

// Copy `n` contiguous images of `bytes` bytes each, image i from src_base +
// items[i].src_off to dst_base + items[i].dst_off (device-accessible pointers).  max_ctas > 0:
// from at most that many CTAs (a copy that runs beside compute), else one CTA per 128 KiB.
int launch_copy_images(const void* src_base, void* dst_base, const CopyItem* items, int64_t n, int64_t bytes,
                       void* stream, int max_ctas = 0);

int decode_workspace_bytes(const Pool& P, int32_t n_seq, size_t* bytes);
// The new token of each sequence of a decode step (k_new / v_new rows [n_seq][H_kv][d], slot
// slots[s]), written by the append kernel launched first; on the tensor-core path the
// attention kernel follows it as a programmatic dependent (its start overlaps the append).
struct AppendFuse {
  const void* k_new;
  const void* v_new;
  const int32_t* slots;
  void* k_pool;
  void* v_pool;
};
// long_batch: the caller knows (from the lengths on the host) that the batch averages at least
// 1,024 tiles per (sequence, KV head) pair; such a batch streams faster from a smaller grid.
int launch_decode(Pool& P, int32_t layer, const void* q, const void* k_pool, const void* v_pool,
                  const int32_t* tables, int32_t W, const int32_t* seq_lens, int32_t n_seq, float scale, void* out,
                  void* ws, size_t ws_bytes, void* stream, const AppendFuse* fuse = nullptr,
                  const ShareLaunch* share = nullptr, bool long_batch = false);
int launch_prefill(Pool& P, int32_t layer, const void* q, const int32_t* q_off, int32_t n_tok, int32_t max_q,
                   const void* k_pool, const void* v_pool, const int32_t* tables, int32_t W, const int32_t* seq_lens,
                   int32_t n_seq, float scale, void* out, void* stream);
void destroy_tensor_maps(Pool& P);

// Device error codes recorded by kernels (the `code` of pkv_check_device_error).
enum DeviceErr : int32_t {
  DERR_NONE = 0,
  DERR_APPEND_SLOT = 1,     // slot out of range in append
  DERR_DECODE_LEN = 2,      // seq_len < 0 or > W * B
  DERR_DECODE_BLOCK = 3,    // block id out of range in a table
  DERR_DECODE_TIMEOUT = 4,  // a bounded mbarrier wait gave up
  DERR_SELFTEST_TIMEOUT = 5,  // the self-test's wait gave up (expected)
  DERR_PREFILL_CHUNK = 6,     // a chunk longer than max_q
  DERR_SHARE = 7,             // a shared-prefix plan entry out of range
};

}  // namespace pkv
