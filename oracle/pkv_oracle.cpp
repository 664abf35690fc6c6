// CPU oracle for the paged KV cache hot path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
// this file: only the tests, the package's smoke check and the benchmark's CPU
// baseline arm use it.  It shares no code, header, table or constant with the
// CUDA library; the two meet only through the seeded input generators.
//
// It is written to be read against the pages, step by step, and is deliberately
// slow: a reference-counted FIFO block allocator, per-sequence block tables with
// fork and copy-on-write, byte copies for the data movement, and textbook softmax
// attention in double precision over keys and values reassembled into contiguous
// arrays.
//
// Sources (page title, then section):
//   [KVM]  "KV Cache Management" (cs249r book, vol. 3 ch. 5)
//          - "The PagedAttention virtual memory model", Definition 0.1 and Table 3:
//            l = floor(t/B), o = t mod B, T: l -> p, free-list ring buffer / FIFO,
//            allocate on o == 0.
//          - "Zero-copy deliberation via copy-on-write branching": fork (table
//            duplication, reference-count increment, S_child = S_prefix), CoW on a
//            write to a block whose count is > 1, release walk.
//          - "Chunked prefill mechanics": online-softmax statistics (used by the
//            GPU path; the oracle computes the plain softmax it is equivalent to).
//          - "Asynchronous paged swapping": swap-out copies blocks to pinned host
//            frames and pushes the freed GPU frames to the FIFO; swap-in reloads
//            them into freshly allocated frames.
//   [PA]   "PagedAttention" (programmer.ie Inference book, ch. 14)
//          - "Paging": blocks hold block_size consecutive positions of every layer;
//            shared blocks are read-only; writing needs a private copy first.
//          - "The real cache": decode writes each new key and value at its block
//            and offset, then gathers each sequence's blocks and attends.
//          - "Sharing and copy-on-write": the first writer copies, the last owner
//            writes in place.
//          - "Inference Lab increment": out-of-blocks and double-free errors, a
//            failed multi-block reservation leaks nothing.
//
// Readings where the pages are silent (all stated in the design notes):
//   * the free list is a FIFO (pop front, push back), initial order given;
//   * sequences in one append call are processed in ascending id order, each
//     sequence's tokens in position order;
//   * CoW copies the whole block (every slot, every layer, K and V);
//   * query head h reads KV head floor(h / G), G = H_q / H_kv;
//   * a sequence of length 0 attends to nothing and yields a zero output;
//   * FP8 storage ([KVM] b_elem = 1 "for FP8") is the OCP E4M3 format with one
//     scale per pool for K and one for V: a value x is stored as the E4M3 code
//     nearest to x / scale (binary32 quotient, ties to an even fraction, values
//     beyond the largest finite 448 stored as 448) and read back as code * scale;
//     the activations around such a pool (new keys/values, queries, outputs) are
//     bfloat16.
//
// Pool data layout (both K and V): [num_blocks][L][H_kv][B][d_head] elements.
// Host tier layout: [slot][2 (K, V)][L][H_kv][B][d_head] elements.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <deque>
#include <map>
#include <set>
#include <thread>
#include <vector>

namespace {

// status codes of the oracle (its own numbering; the tests compare names)
enum {
  ORC_OK = 0,
  ORC_INVALID_ARG = 1,
  ORC_OUT_OF_BLOCKS = 2,
  ORC_DOUBLE_FREE = 3,
  ORC_BAD_BLOCK_ID = 4,
};

struct Sequence {
  std::vector<int32_t> table;  // T: logical block l -> physical block p
  int64_t len = 0;             // tokens written
  bool on_host = false;        // swapped out: table is empty, host_slots hold the images
  std::vector<int64_t> host_slots;
};

struct Pool {
  int64_t num_blocks = 0;
  int64_t B = 0;
  std::deque<int32_t> free_fifo;      // free physical block ids, front = next to allocate
  std::vector<int32_t> ref;           // ref_count[p]
  std::map<int32_t, Sequence> seqs;   // live sequences, iterated in ascending id
  std::set<int32_t> released;         // ids that were freed (for double-free detection)
  int32_t next_id = 0;
};

// Pop the front of the FIFO and give the block one owner.
bool allocate_block(Pool& P, int32_t* out) {
  if (P.free_fifo.empty()) return false;
  int32_t p = P.free_fifo.front();
  P.free_fifo.pop_front();
  P.ref[p] = 1;
  *out = p;
  return true;
}

// Drop one owner of block p; at zero it goes to the back of the FIFO.
int release_block(Pool& P, int32_t p) {
  if (P.ref[p] <= 0) return ORC_DOUBLE_FREE;
  P.ref[p] -= 1;
  if (P.ref[p] == 0) P.free_fifo.push_back(p);
  return ORC_OK;
}

// 0 f32, 1 f16, 2 bf16, 3 FP8 E4M3
size_t elem_bytes(int dtype) { return dtype == 0 ? 4 : (dtype == 3 ? 1 : 2); }

// Value of an FP8 E4M3 code (OCP 8-bit floating point, "E4M3"): 1 sign bit, 4
// exponent bits with bias 7, 3 fraction bits; exponent 0 is subnormal
// (frac/8 * 2^-6); there are no infinities and only S.1111.111 is NaN, so the
// largest finite magnitude is 1.75 * 2^8 = 448.
double e4m3_value(uint8_t c) {
  int sign = c >> 7;
  int expo = (c >> 3) & 0xf;
  int frac = c & 7;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -9);  // frac/8 * 2^(1-7)
  } else if (expo == 15 && frac == 7) {
    v = NAN;
  } else {
    v = std::ldexp(1.0 + frac / 8.0, expo - 7);
  }
  return sign ? -v : v;
}

// The E4M3 code nearest to x: every finite non-negative code is tried in increasing
// order of value; on a tie the code with the even fraction wins (round to nearest,
// ties to even); magnitudes beyond 448 get 448 (saturation to the largest finite
// value).  The sign is kept, so a negative value that rounds to zero is -0.
uint8_t e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7f;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(x));
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    const double err = std::fabs(e4m3_value(static_cast<uint8_t>(c)) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return static_cast<uint8_t>(sign | best);
}

// Exact decode of one stored element to double.
double decode(const void* base, int64_t index, int dtype) {
  if (dtype == 3) return e4m3_value(static_cast<const uint8_t*>(base)[index]);
  if (dtype == 0) {
    float f;
    std::memcpy(&f, static_cast<const char*>(base) + index * 4, 4);
    return static_cast<double>(f);
  }
  uint16_t h;
  std::memcpy(&h, static_cast<const char*>(base) + index * 2, 2);
  if (dtype == 2) {  // bfloat16: the upper half of an IEEE binary32
    uint32_t bits = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return static_cast<double>(f);
  }
  // IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -24);  // subnormal: frac * 2^-14 * 2^-10
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = std::ldexp(1.0 + frac / 1024.0, expo - 15);
  }
  return sign ? -v : v;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- control plane

void* orc_pool_new(int64_t num_blocks, int64_t block_size, const int32_t* free_order) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  Pool* P = new Pool();
  P->num_blocks = num_blocks;
  P->B = block_size;
  P->ref.assign(num_blocks, 0);
  std::vector<char> seen(num_blocks, 0);
  for (int64_t i = 0; i < num_blocks; ++i) {
    int32_t p = free_order ? free_order[i] : static_cast<int32_t>(i);
    if (p < 0 || p >= num_blocks || seen[p]) {
      delete P;
      return nullptr;
    }
    seen[p] = 1;
    P->free_fifo.push_back(p);
  }
  return P;
}

void orc_pool_delete(void* h) { delete static_cast<Pool*>(h); }

int orc_seq_create(void* h, int32_t* seq_id) {
  Pool& P = *static_cast<Pool*>(h);
  int32_t id = P.next_id++;
  P.seqs[id] = Sequence();
  *seq_id = id;
  return ORC_OK;
}

// Fork [KVM, copy-on-write branching]: table duplication, reference-count
// increment for every shared block, child length = parent length.  No data moves.
int orc_seq_fork(void* h, int32_t parent, int32_t* child) {
  Pool& P = *static_cast<Pool*>(h);
  auto it = P.seqs.find(parent);
  if (it == P.seqs.end() || it->second.on_host) return ORC_INVALID_ARG;
  Sequence c;
  c.table = it->second.table;
  c.len = it->second.len;
  for (int32_t p : c.table) P.ref[p] += 1;
  int32_t id = P.next_id++;
  P.seqs[id] = c;
  *child = id;
  return ORC_OK;
}

// A new sequence whose table is the given blocks, each gaining one owner, with length
// len: a request served from the prefix cache starts as the cached blocks it matched
// [KVM, "Prefix Caching Across Turns": matched blocks are re-attached to the request].
int orc_seq_adopt(void* h, const int32_t* blocks, int64_t n, int64_t len, int32_t* seq_id) {
  Pool& P = *static_cast<Pool*>(h);
  for (int64_t i = 0; i < n; ++i)
    if (blocks[i] < 0 || blocks[i] >= P.num_blocks || P.ref[blocks[i]] <= 0) return ORC_BAD_BLOCK_ID;
  Sequence s;
  s.table.assign(blocks, blocks + n);
  s.len = len;
  for (int32_t p : s.table) P.ref[p] += 1;
  int32_t id = P.next_id++;
  P.seqs[id] = s;
  *seq_id = id;
  return ORC_OK;
}

// Number of blocks on the free list.
int64_t orc_free_count(void* h) { return static_cast<int64_t>(static_cast<Pool*>(h)->free_fifo.size()); }

// One more owner of an allocated block (the prefix cache holding it).
int orc_block_retain(void* h, int32_t p) {
  Pool& P = *static_cast<Pool*>(h);
  if (p < 0 || p >= P.num_blocks || P.ref[p] <= 0) return ORC_BAD_BLOCK_ID;
  P.ref[p] += 1;
  return ORC_OK;
}

// One owner fewer (the prefix cache evicting it); at zero the block goes to the FIFO back.
int orc_block_release(void* h, int32_t p) {
  Pool& P = *static_cast<Pool*>(h);
  if (p < 0 || p >= P.num_blocks || P.ref[p] <= 0) return ORC_BAD_BLOCK_ID;
  return release_block(P, p);
}

// Release [KVM, release_sequence_blocks]: walk the table in order, drop one owner
// of each block, push blocks that reach zero to the FIFO, clear the table.
int orc_seq_free(void* h, int32_t seq) {
  Pool& P = *static_cast<Pool*>(h);
  auto it = P.seqs.find(seq);
  if (it == P.seqs.end()) return P.released.count(seq) ? ORC_DOUBLE_FREE : ORC_INVALID_ARG;
  for (int32_t p : it->second.table)
    if (P.ref[p] <= 0) return ORC_DOUBLE_FREE;  // checked before any change
  for (int32_t p : it->second.table) release_block(P, p);
  P.seqs.erase(it);
  P.released.insert(seq);
  return ORC_OK;
}

// Append n_new[i] tokens to sequence seq_ids[i], for all i.
//
// For every token t of a sequence [KVM, PagedAttention model; Definition 0.1]:
//   l = t / B, o = t mod B;
//   o == 0           -> pop a free block, T[l] = p_new;
//   else ref[T[l]]>1 -> copy-on-write: pop p_new, record (T[l] -> p_new) for a
//                       whole-block copy, drop one owner of the old block,
//                       T[l] = p_new                    [KVM, CoW branching];
//   slot = T[l] * B + o.
// slot_mapping is written at the caller's token positions (sequence i's tokens
// start at sum_{j<i} n_new[j]); allocation runs in ascending sequence id.
// All or nothing [PA, Inference Lab increment]: the work is done on a copy of the
// pool state, which replaces the live state only if every allocation succeeded.
int orc_append(void* h, const int32_t* seq_ids, const int32_t* n_new, int n, int32_t* slot_mapping,
               int32_t* cow_pairs, int32_t* n_cow) {
  Pool& live = *static_cast<Pool*>(h);
  if (n < 0) return ORC_INVALID_ARG;
  std::vector<int64_t> start(n + 1, 0);
  std::set<int32_t> ids;
  for (int i = 0; i < n; ++i) {
    auto it = live.seqs.find(seq_ids[i]);
    if (it == live.seqs.end() || it->second.on_host || n_new[i] < 0) return ORC_INVALID_ARG;
    if (!ids.insert(seq_ids[i]).second) return ORC_INVALID_ARG;  // duplicate id
    start[i + 1] = start[i] + n_new[i];
  }
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int a, int b) { return seq_ids[a] < seq_ids[b]; });

  Pool P = live;  // work on a copy
  int32_t cows = 0;
  for (int i : order) {
    Sequence& s = P.seqs[seq_ids[i]];
    for (int32_t k = 0; k < n_new[i]; ++k) {
      int64_t t = s.len;
      int64_t l = t / P.B;
      int64_t o = t % P.B;
      if (o == 0) {
        int32_t p;
        if (!allocate_block(P, &p)) return ORC_OUT_OF_BLOCKS;
        s.table.push_back(p);
      } else if (P.ref[s.table[l]] > 1) {
        int32_t p;
        if (!allocate_block(P, &p)) return ORC_OUT_OF_BLOCKS;
        int32_t old = s.table[l];
        cow_pairs[2 * cows] = old;
        cow_pairs[2 * cows + 1] = p;
        ++cows;
        release_block(P, old);  // count was > 1, so the block stays allocated
        s.table[l] = p;
      }
      slot_mapping[start[i] + k] = static_cast<int32_t>(s.table[l] * P.B + o);
      s.len += 1;
    }
  }
  live = P;
  *n_cow = cows;
  return ORC_OK;
}

int64_t orc_seq_len(void* h, int32_t seq) {
  Pool& P = *static_cast<Pool*>(h);
  auto it = P.seqs.find(seq);
  return it == P.seqs.end() ? -1 : it->second.len;
}

// Copy the block table of seq into out (capacity cap); returns its length or -1.
int64_t orc_seq_table(void* h, int32_t seq, int32_t* out, int64_t cap) {
  Pool& P = *static_cast<Pool*>(h);
  auto it = P.seqs.find(seq);
  if (it == P.seqs.end()) return -1;
  const auto& t = it->second.table;
  for (size_t i = 0; i < t.size() && static_cast<int64_t>(i) < cap; ++i) out[i] = t[i];
  return static_cast<int64_t>(t.size());
}

void orc_refcounts(void* h, int32_t* out) {
  Pool& P = *static_cast<Pool*>(h);
  for (int64_t p = 0; p < P.num_blocks; ++p) out[p] = P.ref[p];
}

// FIFO contents front to back; returns the count.
int64_t orc_free_list(void* h, int32_t* out) {
  Pool& P = *static_cast<Pool*>(h);
  int64_t i = 0;
  for (int32_t p : P.free_fifo) out[i++] = p;
  return i;
}

// Swap-out bookkeeping [KVM, asynchronous paged swapping]: the sequence's blocks,
// in table order, are assigned the given host frames; then each GPU frame loses
// one owner and frames reaching zero go to the back of the FIFO.  Writes the
// block ids that were copied (table order) to block_ids_out.
int orc_swap_out(void* h, int32_t seq, const int64_t* host_slots, int32_t* block_ids_out) {
  Pool& P = *static_cast<Pool*>(h);
  auto it = P.seqs.find(seq);
  if (it == P.seqs.end() || it->second.on_host) return ORC_INVALID_ARG;
  Sequence& s = it->second;
  for (int32_t p : s.table)
    if (P.ref[p] <= 0) return ORC_DOUBLE_FREE;
  s.host_slots.assign(host_slots, host_slots + s.table.size());
  for (size_t i = 0; i < s.table.size(); ++i) block_ids_out[i] = s.table[i];
  for (int32_t p : s.table) release_block(P, p);
  s.table.clear();
  s.on_host = true;
  return ORC_OK;
}

// Swap-in bookkeeping: allocate one fresh frame per host image (FIFO, all or
// nothing) and point the table at them in order.
int orc_swap_in(void* h, int32_t seq, int32_t* new_ids_out, int64_t* host_slots_out) {
  Pool& P = *static_cast<Pool*>(h);
  auto it = P.seqs.find(seq);
  if (it == P.seqs.end() || !it->second.on_host) return ORC_INVALID_ARG;
  Sequence& s = it->second;
  size_t n = s.host_slots.size();
  if (P.free_fifo.size() < n) return ORC_OUT_OF_BLOCKS;
  for (size_t i = 0; i < n; ++i) {
    int32_t p;
    allocate_block(P, &p);
    s.table.push_back(p);
    new_ids_out[i] = p;
    host_slots_out[i] = s.host_slots[i];
  }
  s.host_slots.clear();
  s.on_host = false;
  return ORC_OK;
}

// ---------------------------------------------------------------- data movement
//
// Byte copies on host-resident pools.  Geometry: L layers, H_kv KV heads, B
// slots per block, d elements per head vector, e bytes per element.

// Write token i's key and value for every KV head at slot_mapping[i]
// [PA, "The real cache"]: block = slot / B, offset = slot mod B.
// layer >= 0: k_new, v_new are [n_tok][H_kv][d] for that layer;
// layer == -1: they are [L][n_tok][H_kv][d] and every layer is written.
int orc_write_slots(int L, int H_kv, int d, int B, int dtype, int64_t num_blocks, int layer,
                    const void* k_new, const void* v_new, const int32_t* slot_mapping, int64_t n_tok,
                    void* k_pool, void* v_pool) {
  const size_t e = elem_bytes(dtype);
  const size_t row = static_cast<size_t>(d) * e;
  for (int64_t i = 0; i < n_tok; ++i)
    if (slot_mapping[i] < 0 || slot_mapping[i] >= num_blocks * B) return ORC_BAD_BLOCK_ID;
  int l0 = layer < 0 ? 0 : layer;
  int l1 = layer < 0 ? L : layer + 1;
  for (int l = l0; l < l1; ++l) {
    int64_t src_layer = layer < 0 ? l : 0;
    for (int64_t i = 0; i < n_tok; ++i) {
      int64_t p = slot_mapping[i] / B;
      int64_t o = slot_mapping[i] % B;
      for (int h = 0; h < H_kv; ++h) {
        int64_t src = ((src_layer * n_tok + i) * H_kv + h) * row;
        int64_t dst = (((p * L + l) * H_kv + h) * B + o) * row;
        std::memcpy(static_cast<char*>(k_pool) + dst, static_cast<const char*>(k_new) + src, row);
        std::memcpy(static_cast<char*>(v_pool) + dst, static_cast<const char*>(v_new) + src, row);
      }
    }
  }
  return ORC_OK;
}

// The E4M3 codes of n binary32 values (test access to the encoder above).
void orc_e4m3_encode(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

// Value of each of n E4M3 codes.
void orc_e4m3_decode(const uint8_t* codes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

// Write into an FP8 pool ([KVM] M_block with b_elem = 1): as orc_write_slots, but
// k_new and v_new hold bfloat16 values and each element x of a key is stored as
// the E4M3 code of the binary32 quotient x / k_scale (x / v_scale for a value).
int orc_write_slots_e4m3(int L, int H_kv, int d, int B, int64_t num_blocks, int layer, const void* k_new,
                         const void* v_new, const int32_t* slot_mapping, int64_t n_tok, float k_scale, float v_scale,
                         void* k_pool, void* v_pool) {
  for (int64_t i = 0; i < n_tok; ++i)
    if (slot_mapping[i] < 0 || slot_mapping[i] >= num_blocks * B) return ORC_BAD_BLOCK_ID;
  auto bf16_at = [](const void* base, int64_t idx) {
    uint16_t h;
    std::memcpy(&h, static_cast<const char*>(base) + idx * 2, 2);
    uint32_t bits = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return f;
  };
  int l0 = layer < 0 ? 0 : layer;
  int l1 = layer < 0 ? L : layer + 1;
  for (int l = l0; l < l1; ++l) {
    int64_t src_layer = layer < 0 ? l : 0;
    for (int64_t i = 0; i < n_tok; ++i) {
      int64_t p = slot_mapping[i] / B;
      int64_t o = slot_mapping[i] % B;
      for (int h = 0; h < H_kv; ++h) {
        int64_t src = ((src_layer * n_tok + i) * H_kv + h) * d;
        int64_t dst = (((p * L + l) * H_kv + h) * B + o) * d;
        for (int e = 0; e < d; ++e) {
          const float kq = bf16_at(k_new, src + e) / k_scale;
          const float vq = bf16_at(v_new, src + e) / v_scale;
          static_cast<uint8_t*>(k_pool)[dst + e] = e4m3_encode(kq);
          static_cast<uint8_t*>(v_pool)[dst + e] = e4m3_encode(vq);
        }
      }
    }
  }
  return ORC_OK;
}

// Copy-on-write data step [KVM, CoW branching]: copy every slot of every layer of
// block src into block dst, for K and for V, for each (src, dst) pair in order.
int orc_copy_blocks(int L, int H_kv, int d, int B, int dtype, int64_t num_blocks, const int32_t* pairs,
                    int64_t n, void* k_pool, void* v_pool) {
  const size_t blk = static_cast<size_t>(L) * H_kv * B * d * elem_bytes(dtype);
  for (int64_t i = 0; i < n; ++i) {
    int32_t s = pairs[2 * i], t = pairs[2 * i + 1];
    if (s < 0 || s >= num_blocks || t < 0 || t >= num_blocks) return ORC_BAD_BLOCK_ID;
    std::memcpy(static_cast<char*>(k_pool) + t * blk, static_cast<char*>(k_pool) + s * blk, blk);
    std::memcpy(static_cast<char*>(v_pool) + t * blk, static_cast<char*>(v_pool) + s * blk, blk);
  }
  return ORC_OK;
}

// Swap-out data step: the image of block_ids[i] (K then V, all layers) goes to
// host frame host_slots[i].
int orc_swap_out_data(int L, int H_kv, int d, int B, int dtype, int64_t num_blocks, const int32_t* block_ids,
                      const int64_t* host_slots, int64_t n, const void* k_pool, const void* v_pool, void* host) {
  const size_t blk = static_cast<size_t>(L) * H_kv * B * d * elem_bytes(dtype);
  for (int64_t i = 0; i < n; ++i) {
    int32_t p = block_ids[i];
    if (p < 0 || p >= num_blocks || host_slots[i] < 0) return ORC_BAD_BLOCK_ID;
    char* frame = static_cast<char*>(host) + host_slots[i] * 2 * blk;
    std::memcpy(frame, static_cast<const char*>(k_pool) + p * blk, blk);
    std::memcpy(frame + blk, static_cast<const char*>(v_pool) + p * blk, blk);
  }
  return ORC_OK;
}

// Swap-in data step: host frame host_slots[i] goes to block new_ids[i].
int orc_swap_in_data(int L, int H_kv, int d, int B, int dtype, int64_t num_blocks, const int32_t* new_ids,
                     const int64_t* host_slots, int64_t n, const void* host, void* k_pool, void* v_pool) {
  const size_t blk = static_cast<size_t>(L) * H_kv * B * d * elem_bytes(dtype);
  for (int64_t i = 0; i < n; ++i) {
    int32_t p = new_ids[i];
    if (p < 0 || p >= num_blocks || host_slots[i] < 0) return ORC_BAD_BLOCK_ID;
    const char* frame = static_cast<const char*>(host) + host_slots[i] * 2 * blk;
    std::memcpy(static_cast<char*>(k_pool) + p * blk, frame, blk);
    std::memcpy(static_cast<char*>(v_pool) + p * blk, frame + blk, blk);
  }
  return ORC_OK;
}

// ---------------------------------------------------------------- attention
//
// Decode attention, the plain definition [KVM, PagedAttention model; PA, "The real
// cache" and "It is the same function"].  For sequence s and query head h, with
// G = H_q / H_kv and g = floor(h / G):
//   K_s[t] = k_pool[T_s[floor(t/B)]][layer][g][t mod B][:]     for t < len_s
//   z_t    = scale * sum_i q[s][h][i] * K_s[t][i]
//   w_t    = exp(z_t - max_u z_u) / sum_u exp(z_u - max_u z_u)
//   out[s][h][:] = sum_t w_t * V_s[t][:]
// computed in double precision from the exact stored input values.  A sequence
// with len_s == 0 gives out = 0.  q is [n_seq][H_q][d] of q_dtype; tables are
// [n_seq][W].  Stored keys are read as k_scale * element, values as v_scale *
// element (1 and 1 for 16/32-bit pools; the pool scales for an FP8 pool).
// Work is split over (s, g) pairs across n_threads threads (0 = all cores).
int orc_decode_attention(int L, int H_q, int H_kv, int d, int B, int dtype, int64_t num_blocks, int layer,
                         const void* q, int q_dtype, const void* k_pool, const void* v_pool, double k_scale,
                         double v_scale, const int32_t* tables, int W, const int32_t* seq_lens, int n_seq,
                         double scale, double* out, int n_threads) {
  if (H_kv <= 0 || H_q % H_kv != 0 || layer < 0 || layer >= L) return ORC_INVALID_ARG;
  const int G = H_q / H_kv;
  for (int s = 0; s < n_seq; ++s) {
    if (seq_lens[s] < 0 || static_cast<int64_t>(seq_lens[s]) > static_cast<int64_t>(W) * B) return ORC_INVALID_ARG;
    for (int64_t l = 0; l * B < seq_lens[s]; ++l) {
      int32_t p = tables[static_cast<int64_t>(s) * W + l];
      if (p < 0 || p >= num_blocks) return ORC_BAD_BLOCK_ID;
    }
  }

  auto one_pair = [&](int s, int g) {
    const int64_t len = seq_lens[s];
    // reassemble the contiguous K_s, V_s of KV head g
    std::vector<double> K(len * d), V(len * d);
    for (int64_t t = 0; t < len; ++t) {
      int64_t p = tables[static_cast<int64_t>(s) * W + t / B];
      int64_t base = (((p * L + layer) * H_kv + g) * B + t % B) * d;
      for (int i = 0; i < d; ++i) {
        K[t * d + i] = k_scale * decode(k_pool, base + i, dtype);
        V[t * d + i] = v_scale * decode(v_pool, base + i, dtype);
      }
    }
    std::vector<double> z(len);
    for (int hh = 0; hh < G; ++hh) {
      const int h = g * G + hh;
      double* o = out + (static_cast<int64_t>(s) * H_q + h) * d;
      for (int i = 0; i < d; ++i) o[i] = 0.0;
      if (len == 0) continue;
      std::vector<double> qv(d);
      for (int i = 0; i < d; ++i) qv[i] = decode(q, (static_cast<int64_t>(s) * H_q + h) * d + i, q_dtype);
      double zmax = -INFINITY;
      for (int64_t t = 0; t < len; ++t) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += qv[i] * K[t * d + i];
        z[t] = scale * acc;
        zmax = std::max(zmax, z[t]);
      }
      double denom = 0.0;
      for (int64_t t = 0; t < len; ++t) denom += std::exp(z[t] - zmax);
      for (int64_t t = 0; t < len; ++t) {
        double w = std::exp(z[t] - zmax) / denom;
        for (int i = 0; i < d; ++i) o[i] += w * V[t * d + i];
      }
    }
  };

  const int64_t n_pairs = static_cast<int64_t>(n_seq) * H_kv;
  int nt = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (nt > n_pairs) nt = static_cast<int>(std::max<int64_t>(n_pairs, 1));
  std::atomic<int64_t> next(0);
  auto worker = [&]() {
    for (int64_t k = next.fetch_add(1); k < n_pairs; k = next.fetch_add(1))
      one_pair(static_cast<int>(k / H_kv), static_cast<int>(k % H_kv));
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return ORC_OK;
}

// Chunked-prefill attention [KVM, "Chunked prefill mechanics"]: the queries of
// chunk k attend to the cached keys of earlier chunks in full and to the keys of
// their own chunk causally:  O_k = Softmax(Q_k K_<=k^T / sqrt(d) + M_k) V_<=k.
// Here the chunk of sequence s is its last C_s = q_offsets[s+1] - q_offsets[s]
// tokens (already written to the pool, so seq_lens[s] counts them); query i of the
// chunk sits at position P_s + i with P_s = seq_lens[s] - C_s and sees positions
// t <= P_s + i.  q (of q_dtype) and out are [n_tok][H_q][d], row q_offsets[s] + i;
// keys and values are read as in orc_decode_attention.
int orc_prefill_attention(int L, int H_q, int H_kv, int d, int B, int dtype, int64_t num_blocks, int layer,
                          const void* q, int q_dtype, const int32_t* q_offsets, const void* k_pool,
                          const void* v_pool, double k_scale, double v_scale, const int32_t* tables, int W,
                          const int32_t* seq_lens, int n_seq, double scale, double* out, int n_threads) {
  if (H_kv <= 0 || H_q % H_kv != 0 || layer < 0 || layer >= L) return ORC_INVALID_ARG;
  const int G = H_q / H_kv;
  for (int s = 0; s < n_seq; ++s) {
    const int64_t C = q_offsets[s + 1] - q_offsets[s];
    if (C < 0 || seq_lens[s] < C || static_cast<int64_t>(seq_lens[s]) > static_cast<int64_t>(W) * B)
      return ORC_INVALID_ARG;
    for (int64_t l = 0; l * B < seq_lens[s]; ++l) {
      int32_t p = tables[static_cast<int64_t>(s) * W + l];
      if (p < 0 || p >= num_blocks) return ORC_BAD_BLOCK_ID;
    }
  }
  auto one_pair = [&](int s, int g) {
    const int64_t len = seq_lens[s];
    const int64_t C = q_offsets[s + 1] - q_offsets[s];
    const int64_t P = len - C;
    std::vector<double> K(len * d), V(len * d);
    for (int64_t t = 0; t < len; ++t) {
      int64_t p = tables[static_cast<int64_t>(s) * W + t / B];
      int64_t base = (((p * L + layer) * H_kv + g) * B + t % B) * d;
      for (int i = 0; i < d; ++i) {
        K[t * d + i] = k_scale * decode(k_pool, base + i, dtype);
        V[t * d + i] = v_scale * decode(v_pool, base + i, dtype);
      }
    }
    std::vector<double> z(len), qv(d);
    for (int64_t qi = 0; qi < C; ++qi) {
      const int64_t visible = P + qi + 1;  // mask M_k: history in full, own chunk causally
      const int64_t row = q_offsets[s] + qi;
      for (int hh = 0; hh < G; ++hh) {
        const int h = g * G + hh;
        double* o = out + (row * H_q + h) * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int i = 0; i < d; ++i) qv[i] = decode(q, (row * H_q + h) * d + i, q_dtype);
        double zmax = -INFINITY;
        for (int64_t t = 0; t < visible; ++t) {
          double acc = 0.0;
          for (int i = 0; i < d; ++i) acc += qv[i] * K[t * d + i];
          z[t] = scale * acc;
          zmax = std::max(zmax, z[t]);
        }
        double denom = 0.0;
        for (int64_t t = 0; t < visible; ++t) denom += std::exp(z[t] - zmax);
        for (int64_t t = 0; t < visible; ++t) {
          double w = std::exp(z[t] - zmax) / denom;
          for (int i = 0; i < d; ++i) o[i] += w * V[t * d + i];
        }
      }
    }
  };
  const int64_t n_pairs = static_cast<int64_t>(n_seq) * H_kv;
  int nt = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (nt > n_pairs) nt = static_cast<int>(std::max<int64_t>(n_pairs, 1));
  std::atomic<int64_t> next(0);
  auto worker = [&]() {
    for (int64_t k = next.fetch_add(1); k < n_pairs; k = next.fetch_add(1))
      one_pair(static_cast<int>(k / H_kv), static_cast<int>(k % H_kv));
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return ORC_OK;
}

int orc_hardware_threads() { return static_cast<int>(std::thread::hardware_concurrency()); }

}  // extern "C"
