/*
 * pkv.h -- C ABI of the paged KV cache hot path (GB300 / sm_103a).
 *
 * A pool of fixed-size KV blocks, per-sequence block tables with fork and
 * copy-on-write, and four device operations on the block pool: writing new
 * tokens' keys/values at their slots, ragged-batch GQA decode attention read
 * through the block tables, whole-block copies for copy-on-write, and swapping
 * blocks between the HBM pool and a page-locked host tier.
 *
 * Sources (page title, section):
 *   [KVM] "KV Cache Management" (cs249r book, vol. 3 ch. 5):
 *         "The PagedAttention virtual memory model" (Definition 0.1, Table 3,
 *         M_block), "Zero-copy deliberation via copy-on-write branching",
 *         "Chunked prefill mechanics" (online-softmax merge),
 *         "Asynchronous paged swapping".
 *   [PA]  "PagedAttention" (programmer.ie Inference book, ch. 14): "Paging",
 *         "The real cache", "Sharing and copy-on-write", "Inference Lab increment".
 *
 * Conventions
 *   - Every call returns an int status (enum pkv_status).  On failure the call
 *     changes no host state (all or nothing, [PA] "Inference Lab increment") and
 *     pkv_last_error_message() gives a thread-local description.
 *   - No C++ exception crosses the ABI.
 *   - A pool's control plane is not thread-safe: serialise calls on one pool.
 *   - Device operations are asynchronous on the given stream (a cudaStream_t;
 *     NULL = the legacy default stream).  They never allocate device memory.
 *   - Ownership: the caller owns every device buffer (pools, q, out, workspace,
 *     slot mappings, tables) and the page-locked host tier.  The library owns
 *     only the host control-plane state behind the opaque pkv_pool handle.
 *   - Device-side argument checks (block ids, slots, lengths) never trap: a
 *     kernel that meets a bad value records it in a per-device error word, skips
 *     or clamps the access, and finishes; pkv_check_device_error() reports it.
 *
 * Data layouts (row-major, element type = geometry.dtype)
 *   k_pool, v_pool : [num_blocks][L][H_kv][block_size][d_head]
 *                    A (block, layer, head) slab is block_size*d_head contiguous
 *                    elements; a block over all layers is contiguous, so one
 *                    physical block of K plus V is M_block = 2*L*H_kv*B*d*b bytes
 *                    ([KVM] M_block).  Slot s = block * block_size + offset.
 *   host tier      : frames of M_block bytes: [frame][2 (K, V)][L][H_kv][B][d].
 *   q, out         : [n_seq][H_q][d_head]
 *   block_tables   : int32 [n_seq][W]; entry l is the physical block of logical
 *                    block l = floor(t / block_size) ([KVM] Definition 0.1).
 *   Query head h reads KV head floor(h / G), G = H_q / H_kv.
 *
 * FP8 pools (dtype PKV_E4M3; [KVM] PagedAttention model: b_elem = 1 byte for FP8)
 *   K and V are stored as OCP FP8 E4M3 bytes (1 sign, 4 exponent bits with bias 7,
 *   3 fraction bits, largest finite 448) and read as code * k_scale (keys) or
 *   code * v_scale (values), one scale of each per pool (pkv_pool_set_kv_scales).
 *   Everything around such a pool is bfloat16: k_new / v_new of pkv_append_kv and
 *   pkv_decode_step, q and out.  An append stores the E4M3 code nearest to the
 *   binary32 quotient x / scale (ties to even; magnitudes beyond 448 stored as 448;
 *   a negative value that rounds to zero is stored as -0).  d_head must be a
 *   multiple of 8.  The tensor-core attention path computes q K^T and P V with
 *   binary16 operands, so |q| must stay below 65504 there; the codes convert to
 *   binary16 exactly.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_VERSION 1

typedef struct CUstream_st* pkv_stream_t; /* identical to cudaStream_t */
typedef struct pkv_pool pkv_pool;         /* opaque host control-plane state */

enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* bad argument, unknown or swapped-out sequence */
  PKV_ERR_OUT_OF_BLOCKS = 2, /* the free list cannot satisfy the request */
  PKV_ERR_DOUBLE_FREE = 3,   /* a sequence (or block) released twice */
  PKV_ERR_BAD_BLOCK_ID = 4,  /* a block id, slot or host frame out of range */
  PKV_ERR_CUDA = 5,          /* a CUDA runtime call failed (message has the name) */
  PKV_ERR_DEVICE_CHECK = 6,  /* a kernel recorded a bad index (pkv_check_device_error) */
  PKV_ERR_TIMEOUT = 7,       /* a bounded device wait gave up */
  PKV_ERR_UNSUPPORTED = 8    /* geometry or dtype this build does not handle */
};

enum pkv_dtype { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2, PKV_E4M3 = 3 };

/* Pool geometry ([KVM] Eq. 1: m_token = 2 * L * H_kv * d_head * b). */
typedef struct pkv_geometry {
  int32_t L;          /* layers held per block */
  int32_t H_q;        /* query heads (multiple of H_kv) */
  int32_t H_kv;       /* key/value heads */
  int32_t d_head;     /* head dimension (even, <= 256) */
  int32_t block_size; /* B, tokens per block */
  int32_t dtype;      /* enum pkv_dtype */
  int64_t num_blocks; /* N, physical blocks in the pool (< 2^31) */
} pkv_geometry;

/* ---------------------------------------------------------------- library */

int pkv_version(void);
/* Thread-local text of the last failure on this thread ("" if none). */
const char* pkv_last_error_message(void);
const char* pkv_status_name(int status);

/* ---------------------------------------------------------------- control plane (host only)
 *
 * The free list is a FIFO of block ids ([KVM] "free-list ring buffer", Table 3
 * "free-list stack / FIFO"): allocation pops the front, release pushes the back.
 * Sequence ids are assigned 0, 1, 2, ... and never reused.
 */

/* Create a pool.  initial_free_order: a permutation of [0, num_blocks) giving the
 * FIFO's initial order, or NULL for 0, 1, 2, ...  Errors: INVALID_ARG (geometry,
 * not a permutation), UNSUPPORTED (dtype). */
int pkv_pool_create(const pkv_geometry* geometry, const int32_t* initial_free_order, pkv_pool** out);
int pkv_pool_destroy(pkv_pool* pool);
int pkv_pool_geometry(const pkv_pool* pool, pkv_geometry* out);

/* Scales of an FP8 pool (see "FP8 pools" above): stored keys read as code * k_scale,
 * values as code * v_scale; both start at 1.  Later appends and attention calls use
 * the new values; codes already stored are not rewritten.  Errors: INVALID_ARG (a
 * scale that is not finite and > 0), UNSUPPORTED (a 16/32-bit pool). */
int pkv_pool_set_kv_scales(pkv_pool* pool, float k_scale, float v_scale);
int pkv_pool_kv_scales(const pkv_pool* pool, float* k_scale, float* v_scale);

/* New empty sequence. */
int pkv_seq_create(pkv_pool* pool, int32_t* seq_id);

/* Fork ([KVM] "Zero-copy deliberation via copy-on-write branching"): the child
 * gets a copy of the parent's table, every shared block gains one owner, and the
 * child's length is the parent's.  No data moves.  Errors: INVALID_ARG. */
int pkv_seq_fork(pkv_pool* pool, int32_t parent, int32_t* child);

/* Release ([KVM] release_sequence_blocks): walk the table in order, drop one
 * owner per block, push blocks that reach zero owners to the FIFO back.
 * Errors: DOUBLE_FREE (already released), INVALID_ARG (never created). */
int pkv_seq_free(pkv_pool* pool, int32_t seq);

int pkv_seq_len(const pkv_pool* pool, int32_t seq, int64_t* len);

/* Plan an append of n_new[i] tokens to sequence seq_ids[i], i < n (distinct ids,
 * resident).  Sequences are processed in ascending id; for each token t:
 * l = t / B, o = t mod B; o == 0 allocates a block for T[l]; otherwise if T[l]
 * has more than one owner it is copied first (copy-on-write: a fresh block is
 * allocated, the pair (old, new) is emitted, the old block loses one owner and
 * T[l] = new); the token's slot is T[l] * B + o ([KVM] PagedAttention model and
 * CoW branching; [PA] "Sharing and copy-on-write").
 *   slot_mapping : host int32 [sum n_new], sequence i's tokens start at
 *                  sum_{j<i} n_new[j] (the caller's order).
 *   cow_pairs    : host int32 [capacity n][2] (src, dst), at most one per sequence;
 *                  *n_cow receives the count.  The caller copies them with
 *                  pkv_copy_blocks BEFORE writing the new tokens.
 * All or nothing: OUT_OF_BLOCKS leaves every table, count and the FIFO unchanged
 * ([PA] "a failed multi-block reservation leaks no blocks"). */
int pkv_plan_append(pkv_pool* pool, const int32_t* seq_ids, const int32_t* n_new, int32_t n,
                    int32_t* slot_mapping, int32_t* cow_pairs, int32_t* n_cow);

/* Host copy of the tables of n resident sequences: tables is int32 [n][W], row i
 * holds seq_ids[i]'s blocks then zeros; seq_lens is int32 [n].
 * Errors: INVALID_ARG (unknown / swapped-out id, W too small). */
int pkv_export_tables(const pkv_pool* pool, const int32_t* seq_ids, int32_t n, int32_t* tables, int32_t W,
                      int32_t* seq_lens);

/* Reference count of every block: int32 [num_blocks]. */
int pkv_refcounts(const pkv_pool* pool, int32_t* out);

/* FIFO contents, front to back, into out (capacity num_blocks); *n = count. */
int pkv_free_list(const pkv_pool* pool, int32_t* out, int64_t* n);

/* ---------------------------------------------------------------- data plane (device, async)
 *
 * k_pool / v_pool are device pointers to the caller's pools (layout above,
 * 16-byte aligned).  Every kernel checks its indices against the geometry.
 */

/* Write new keys/values at their slots ([PA] "The real cache"; [KVM] Table 3):
 * K_pool[slot / B][layer][h][slot mod B][:] = k_new[i][h][:], same for V.
 *   layer >= 0 : k_new, v_new are device [n_tok][H_kv][d_head] for that layer.
 *   layer == -1: they are device [L][n_tok][H_kv][d_head], all layers written.
 *   slot_mapping: device int32 [n_tok]; a slot outside [0, N*B) is skipped and
 *   recorded in the device error word. */
int pkv_append_kv(const pkv_pool* pool, int32_t layer, const void* k_new, const void* v_new,
                  const int32_t* slot_mapping, int32_t n_tok, void* k_pool, void* v_pool, pkv_stream_t stream);

/* Bytes of device workspace pkv_decode_attention needs for n_seq sequences on
 * the current device (with prefix sharing on, also room for the shared-prefix
 * partials of a decode step of n_seq sequences). */
int pkv_decode_workspace_size(const pkv_pool* pool, int32_t n_seq, size_t* bytes);

/* Decode attention over the block tables ([KVM] PagedAttention model: the kernel
 * takes the block table and walks logical blocks 0 .. floor((S-1)/B); [PA] "It is
 * the same function"):
 *   out[s][h][:] = sum_{t < len_s} softmax_t(scale * q[s][h] . K_s[t]) V_s[t],
 *   K_s[t] = k_pool[T_s[floor(t/B)]][layer][floor(h/G)][t mod B].
 * The context is split into 16-token tiles shared evenly across all warps of a
 * persistent grid; partial (m, l, O) statistics of a sequence split across warps
 * are merged with the online-softmax rule of [KVM] "Chunked prefill mechanics".
 *   q, out      : device [n_seq][H_q][d_head], dtype = geometry dtype.
 *   block_tables: device int32 [n_seq][W];  seq_lens: device int32 [n_seq]
 *                 (0 <= len <= W*B; len 0 gives a zero output).
 *   workspace   : device, >= pkv_decode_workspace_size bytes, 256-byte aligned;
 *                 its contents need no initialisation and no state survives
 *                 between calls (the split-pair counters carry a tag unique to
 *                 each launch, so whatever a word held before counts as zero).
 * Calls on one workspace must not overlap on the GPU.  On the tensor-core path a
 * call is one kernel launch for up to 4,096 sequences (every CTA plans its own
 * warps from seq_lens); larger batches launch a plan kernel first.
 * bf16/f16 with d_head 64 or 128, and FP8 with d_head 128, with G <= 16 and B a
 * multiple of 16 run on the tensor-core path (TMA-staged tiles, mma.sync; groups
 * of 9 to 16 query heads as two 8-head column blocks); other geometries on CUDA
 * cores (G <= 16; G <= 8 when d_head > 128; wider groups return
 * PKV_ERR_UNSUPPORTED). */
int pkv_decode_attention(const pkv_pool* pool, int32_t layer, const void* q, const void* k_pool,
                         const void* v_pool, const int32_t* block_tables, int32_t W, const int32_t* seq_lens,
                         int32_t n_seq, float scale, void* out, void* workspace, size_t ws_bytes,
                         pkv_stream_t stream);

/* One decode step for n resident sequences, in one call: plan one new token per
 * sequence (pkv_plan_append), copy shared tail blocks (pkv_copy_blocks), write
 * the new keys/values (pkv_append_kv) and attend over len + 1 tokens
 * (pkv_decode_attention) -- [PA] "The real cache": write each new key and value
 * at its block and offset, then attend.
 *   seq_ids : HOST int32 [n], distinct resident sequences; row i of q, k_new,
 *             v_new and out belongs to seq_ids[i].
 *   q, out  : device [n][H_q][d_head];  k_new, v_new: device [n][H_kv][d_head].
 *   W       : table width; every sequence needs ceil((len + 1) / B) <= W.
 *   meta_host: page-locked host int32 [pkv_step_meta_ints(pool, n, W)] (n * (W + 2)
 *             with prefix sharing off): the step writes its slot mapping, tables
 *             (entries past each table's end are left as they were) and lengths
 *             there (and, with sharing on, its shared-prefix plan) and
 *             copies them to meta_dev (device int32, same size, 16-byte aligned) on
 *             the stream; do not reuse meta_host until that copy has run (e.g. a
 *             ring of buffers and events).
 *   workspace: as for pkv_decode_attention (pkv_decode_workspace_size(pool, n)).
 *   attn_begin, attn_end: optional cudaEvent_t (NULL = none) recorded on the
 *             stream just before the append and just after the attention (on the
 *             tensor-core path the attention kernel is the append kernel's
 *             programmatic dependent: it starts, plans its warps and reads its first
 *             table entries while the new tokens are written, and waits for the append
 *             before loading any K/V; the append kernel lets only this launch start
 *             early -- pkv_append_kv called on its own does not).
 * Arguments are validated before anything changes; after the plan is applied,
 * only a CUDA launch failure (PKV_ERR_CUDA) can still fail the call. */
typedef struct CUevent_st* pkv_event_t; /* identical to cudaEvent_t */

/* Shared prefixes in decode steps.  (The pages share a forked prefix's blocks in
 * memory -- [KVM] "Zero-copy deliberation via copy-on-write branching": the parent
 * and every branch map the same physical blocks -- and every branch still reads
 * them in attention; this option reads them once per step for all branches.)
 * With sharing on, a decode step (pkv_decode_step, pkv_step_plan + a launch call)
 * finds runs of consecutive batch rows whose tables begin with the same physical
 * blocks -- at least min_blocks of them, in at least min_members rows; every row
 * after the first shares at least half of what the rows before it share; the run's
 * prefix stops before the block of each row's last token -- and attends to those
 * blocks once for the whole run (a tcgen05 kernel, all the run's queries of a KV
 * head as 128-row tiles against each key tile, in splits of whole blocks sized so
 * that its grid comes near target_ctas CTAs) and to each row's own blocks in the
 * decode kernel; a combine kernel merges the two with the online-softmax rule ([KVM]
 * "Chunked prefill mechanics").  With 16-bit pools and up to 8 query heads per KV head
 * the step may run the decode on part of the SMs beside the prefix kernel on the
 * others (the split comes from a time model of the two kernels).  The result is the
 * same attention (within rounding).
 * Change the option only between steps: a step planned (pkv_step_plan) with one setting
 * must be launched with the same, since the setting decides the metadata's layout.
 *   min_members: 0 turns sharing off (the default); else >= 2.
 *   min_blocks : >= 1.
 *   target_ctas: <= 0 takes the current device's SM count (PKV_ERR_CUDA without one).
 * Needs a bf16, f16 or E4M3 pool with d_head 128, at most 16 query heads per KV head
 * and B a multiple of 16 (else PKV_ERR_UNSUPPORTED).  While it is on, the step
 * metadata is pkv_step_meta_ints(pool, n, W) int32 (the plan follows the lengths
 * from a 16-byte boundary) and pkv_decode_workspace_size includes room for the
 * prefix kernel's partials (2 n + 1024 slots of H_q x (d_head + 2) floats). */
int pkv_pool_set_prefix_sharing(pkv_pool* pool, int32_t min_members, int32_t min_blocks, int32_t target_ctas);
/* int32 count of one step's metadata for n sequences and table width W. */
int pkv_step_meta_ints(const pkv_pool* pool, int32_t n, int32_t W, int64_t* ints);
int pkv_decode_step(pkv_pool* pool, int32_t layer, const int32_t* seq_ids, int32_t n, int32_t W, const void* q,
                    const void* k_new, const void* v_new, void* k_pool, void* v_pool, float scale, void* out,
                    int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes, pkv_event_t attn_begin,
                    pkv_event_t attn_end, pkv_stream_t stream);

/* pkv_decode_step in two halves, so that a caller can plan step t + 1 on the host
 * while step t runs on the GPU (the plan of a step needs no result of the previous
 * one).  (The pages have no counterpart of these calls.)
 * pkv_step_plan: the host half -- checks the sequences as pkv_decode_step does, then
 *   plans one new token per sequence (pkv_plan_append) and writes the slot mapping,
 *   tables and lengths into meta_host (host int32 [pkv_step_meta_ints(pool, n, W)],
 *   as for pkv_decode_step) and the copy-on-write pairs into cow_pairs (host int32 [2 n];
 *   their count in *n_cow).  On failure nothing changes.
 * pkv_step_launch: the device half, on the stream: copies meta_host to meta_dev,
 *   copies the shared blocks, appends k_new / v_new at the planned slots and attends
 *   (arguments as for pkv_decode_step; n, W, cow_pairs and meta_host from the plan,
 *   meta_host page-locked and untouched until the copy has run).  Its argument
 *   errors do not undo the plan.
 * pkv_step_launch_host: pkv_step_launch with q / k_new / v_new read from, and out
 *   written to, host memory through the caller's device staging buffers, as for
 *   pkv_decode_step_host. */
int pkv_step_plan(pkv_pool* pool, const int32_t* seq_ids, int32_t n, int32_t W, int32_t* meta_host,
                  int32_t* cow_pairs, int32_t* n_cow);
int pkv_step_launch(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs, int32_t n_cow,
                    const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool, float scale,
                    void* out, const int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes,
                    pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream);
int pkv_step_launch_host(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs,
                         int32_t n_cow, const void* q_host, const void* k_new_host, const void* v_new_host,
                         void* out_host, void* q_dev, void* k_new_dev, void* v_new_dev, void* out_dev, void* k_pool,
                         void* v_pool, float scale, const int32_t* meta_host, int32_t* meta_dev, void* workspace,
                         size_t ws_bytes, pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream);

/* The device half of a decode step with the step's inputs packed in one page-locked
 * host buffer.  (The pages have no counterpart of this call; it is the step for callers
 * whose inputs arrive in host memory, with the fewest copies per step.)  On the stream:
 * ONE cudaMemcpyAsync of in_bytes from in_host to in_dev (device, same layout), the
 * metadata copy if the metadata is elsewhere (see below), the shared-block copies, the
 * append and the attention, and ONE copy of the n result rows from out_dev to out_host.
 *   in_host / in_dev: q [n][H_q][d_head] at byte 0, k_new [n][H_kv][d_head] at off_k,
 *                     v_new [n][H_kv][d_head] at off_v (activation type), and, when off_meta
 *                     is not 0, the step's metadata [pkv_step_meta_ints] int32 at off_meta (where
 *                     pkv_step_plan wrote it into in_host; meta_host and meta_dev are then
 *                     ignored and may be NULL).  Offsets are multiples of 16, each part
 *                     before the next, in_bytes covers the last part.
 *   off_meta 0: meta_host as in pkv_step_launch (copied to meta_dev by the call), or NULL
 *               when the caller has already queued meta_dev's contents on the stream
 *               (not with prefix sharing on: the call reads the plan from the host copy,
 *               PKV_ERR_INVALID_ARG before anything is queued).
 *   out_host [n][H_q][d_head] page-locked; out_dev device.
 * Every other argument is as for pkv_step_launch.  Errors: INVALID_ARG for a layout that
 * does not hold n rows; otherwise as pkv_step_launch. */
int pkv_step_launch_packed(pkv_pool* pool, int32_t layer, int32_t n, int32_t W, const int32_t* cow_pairs,
                           int32_t n_cow, const void* in_host, void* in_dev, size_t off_k, size_t off_v,
                           size_t off_meta, size_t in_bytes, void* out_host, void* out_dev, void* k_pool,
                           void* v_pool, float scale, const int32_t* meta_host, int32_t* meta_dev, void* workspace,
                           size_t ws_bytes, pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream);

/* pkv_decode_step with the step's inputs and result in HOST memory.  (The pages
 * have no counterpart of this call; it is the step for callers whose per-step
 * inputs arrive in, and whose result is read from, host memory.)  On the stream:
 * copies q_host, k_new_host and v_new_host into the caller's device staging
 * buffers q_dev, k_new_dev, v_new_dev (one cudaMemcpyAsync each), runs
 * pkv_decode_step on them with out_dev as its output, then copies out_dev to
 * out_host.  The caller synchronises the stream before reading out_host.
 *   q_host, out_host         : host [n][H_q][d_head];
 *   k_new_host, v_new_host   : host [n][H_kv][d_head] (the activation type: bf16
 *                              for an E4M3 pool); page-locked for the copies to
 *                              be asynchronous;
 *   q_dev, k_new_dev, v_new_dev, out_dev: device buffers of at least those sizes.
 * Every other argument is as for pkv_decode_step.  If the step's validation fails,
 * the staging copies may already be queued (caller-owned scratch); no pool state
 * changes. */
int pkv_decode_step_host(pkv_pool* pool, int32_t layer, const int32_t* seq_ids, int32_t n, int32_t W,
                         const void* q_host, const void* k_new_host, const void* v_new_host, void* out_host,
                         void* q_dev, void* k_new_dev, void* v_new_dev, void* out_dev, void* k_pool, void* v_pool,
                         float scale, int32_t* meta_host, int32_t* meta_dev, void* workspace, size_t ws_bytes,
                         pkv_event_t attn_begin, pkv_event_t attn_end, pkv_stream_t stream);

/* Decode attention that allocates nothing.  (The pages have no counterpart of
 * this call; it exists for callers of this library.)
 * Same arguments and result as pkv_decode_attention, minus the workspace: the
 * scratch is a 24 MiB array compiled into the library (a static __device__
 * variable, held by every GPU that loads the library until the process exits).
 * It is for callers that cannot call cudaMalloc: e.g. a serving engine that sized
 * its KV block pool to fill the device at start-up, so a later allocation would
 * fail, or code that must not take cudaMalloc's implicit device synchronisation.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - A batch that needs more scratch than 24 MiB is rejected with
 *     PKV_ERR_INVALID_ARG (the partials of one persistent grid on a 152-SM GB300
 *     take about 10 MB for 16-bit pools with groups of up to 8 query heads, 18 MB
 *     for FP8 pools and 20 MB for groups of 9 to 16; each sequence adds 8 bytes).
 *   - Every call on a device shares the one array and leaves its contents behind;
 *     nothing in it needs to start at zero.  Calls whose GPU work overlaps (two
 *     streams, or two threads) race on it: order them on one stream.
 * No cudaMalloc, cudaFree or other allocating routine is called. */
int pkv_decode_attention_noalloc(const pkv_pool* pool, int32_t layer, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables, int32_t W, const int32_t* seq_lens,
                                 int32_t n_seq, float scale, void* out, pkv_stream_t stream);

/* Chunked-prefill attention ([KVM] "Chunked prefill mechanics"): the queries of a
 * chunk attend to the cached history in full and to their own chunk causally,
 *   O_k = Softmax(Q_k K_<=k^T * scale + M_k) V_<=k.
 * The chunk of sequence s is its last C_s = q_offsets[s+1] - q_offsets[s] tokens,
 * already written to the pool (pkv_plan_append + pkv_append_kv), so seq_lens[s]
 * counts them: query i sits at position seq_lens[s] - C_s + i and sees positions
 * 0 .. that position.  Decode is the case C_s = 1.
 *   q, out     : device [n_tok][H_q][d_head], row q_offsets[s] + i (16-byte aligned).
 *   q_offsets  : device int32 [n_seq + 1], q_offsets[0] = 0, q_offsets[n_seq] = n_tok.
 *   max_q      : host int, >= every C_s (a longer chunk records code 6 in the device
 *                error word and its extra rows are not computed).
 *   block_tables, W, seq_lens: as for pkv_decode_attention (C_s <= len_s <= W*B).
 * bf16/f16 and FP8 (E4M3) pools with d_head 128 and B a multiple of 16 run on the
 * 5th-generation tensor cores (tcgen05, TMEM accumulators; one CTA per 2 x 128
 * (query, head) rows, 64-key tiles staged by TMA; E4M3 codes are converted to
 * binary16 in shared memory and q is rounded to binary16); bf16/f16 with d_head 64 on
 * mma.sync tensor cores; other geometries on CUDA cores.  No workspace. */
int pkv_prefill_attention(const pkv_pool* pool, int32_t layer, const void* q, const int32_t* q_offsets, int32_t n_tok,
                          int32_t max_q, const void* k_pool, const void* v_pool, const int32_t* block_tables, int32_t W,
                          const int32_t* seq_lens, int32_t n_seq, float scale, void* out, pkv_stream_t stream);

/* Copy-on-write data step ([KVM] "copies the B tokens from the shared block into
 * p_new"): for each (src, dst) in pairs (HOST int32 [n][2]), copy every slot of
 * every layer of block src into block dst, for K and V.  Pairs are passed to the
 * kernel by value.  Errors: BAD_BLOCK_ID. */
int pkv_copy_blocks(const pkv_pool* pool, const int32_t* pairs, int32_t n, void* k_pool, void* v_pool,
                    pkv_stream_t stream);

/* Swap a resident sequence out to the host tier ([KVM] "Asynchronous paged
 * swapping", swap_out_trajectory): block j of its table (j < n, n = its block
 * count) is copied to host frame host_slots[j] (HOST int64 [n], each in
 * [0, host_frames)); then, on the host, each GPU block loses one owner and blocks
 * reaching zero go to the FIFO back; the sequence keeps its length and is marked
 * swapped out.  Freed blocks may be reallocated at once: later writes to them
 * must be ordered after this call's stream work (same stream, or an event).
 *   host: page-locked (cudaHostAlloc / cudaHostRegister) or device-accessible
 *         host memory of host_frames * M_block bytes.
 *   block_ids_out: optional HOST int32 [n], the blocks copied (table order).
 * The copy runs as an SM kernel, or on the copy engines after
 * pkv_pool_set_swap_engine(pool, 1). */
int pkv_swap_out(pkv_pool* pool, int32_t seq, const void* k_pool, const void* v_pool, void* host,
                 int64_t host_frames, const int64_t* host_slots, int32_t n, int32_t* block_ids_out,
                 pkv_stream_t stream);

/* Swap a swapped-out sequence back in: allocate n fresh blocks from the FIFO
 * front (all or nothing), copy the host frames recorded at swap-out into them in
 * table order, and point the table at them.  new_block_ids: optional HOST int32 [n]. */
int pkv_swap_in(pkv_pool* pool, int32_t seq, const void* host, int64_t host_frames, int32_t n, void* k_pool,
                void* v_pool, int32_t* new_block_ids, pkv_stream_t stream);

/* Residency of a sequence's blocks (the dual-residency table of [KVM] "Asynchronous
 * paged swapping"): PKV_TIER_HBM while its blocks are in the pool, PKV_TIER_HOST
 * after pkv_swap_out until pkv_swap_in.  A swap-in may run on its own stream (with
 * the copy engines, pkv_pool_set_swap_engine(pool, 1), so the SMs stay with
 * attention) while other sequences decode; record an event after it and make the
 * stream that decodes the restored sequence wait on that event. */
enum pkv_tier { PKV_TIER_HBM = 0, PKV_TIER_HOST = 1, PKV_TIER_RELOADING = 2 };
int pkv_seq_residency(const pkv_pool* pool, int32_t seq, int32_t* tier);

/* Reload a swapped-out sequence a range of layers at a time ([KVM] "Asynchronous paged
 * swapping", "Pipelined Chunked Reload and Observation Prefill": the history streams in over
 * the copy path while the observation's own prefill runs, instead of a stall for the whole
 * transfer).  The first call (layer_begin 0) allocates the n fresh blocks from the FIFO front
 * (all or nothing) and points the table at them, as pkv_swap_in does; every call copies layers
 * [layer_begin, layer_end) of every block from the host frames recorded at swap-out (one
 * contiguous piece of each block image and frame half, both [L][H_kv][B][d]).  Ranges must
 * follow each other from layer 0 to L; until the last one the sequence's residency is
 * PKV_TIER_RELOADING and its recorded frames are kept (pkv_seq_host_slots).  Asynchronous on
 * `stream`: record an event after each range and make the stream that appends to or attends
 * over layer l of this sequence wait for the event of the range holding l -- the copy writes
 * whole block images of those layers, including slots a later append fills.
 * new_block_ids: optional HOST int32 [n], the table after the call.  Errors: INVALID_ARG (not
 * swapped out and not being reloaded, a range out of order or beyond L, n not the swapped block
 * count), BAD_BLOCK_ID (a recorded frame beyond host_frames), OUT_OF_BLOCKS (first call only);
 * a failed call changes nothing. */
int pkv_swap_in_layers(pkv_pool* pool, int32_t seq, const void* host, int64_t host_frames, int32_t n,
                       int32_t layer_begin, int32_t layer_end, void* k_pool, void* v_pool, int32_t* new_block_ids,
                       pkv_stream_t stream);

/* Host frames recorded for a swapped-out sequence: HOST int64 [capacity], *n = count. */
int pkv_seq_host_slots(const pkv_pool* pool, int32_t seq, int64_t* out, int32_t capacity, int32_t* n);

/* 0 = swap with SM kernels (default), 1 = with cudaMemcpyAsync on the copy engines. */
int pkv_pool_set_swap_engine(pkv_pool* pool, int32_t engine);

/* ---------------------------------------------------------------- radix prefix cache (host only)
 *
 * [KVM] "Prefix Caching Across Turns": a radix tree over the pool that indexes physical
 * blocks by the tokens they hold (Table 4, Definition 0.2), so that a new request whose
 * prompt starts with cached tokens reuses those blocks instead of recomputing them.
 *   - Only whole blocks are shared ("Longest prefix matching": block-aligned truncation,
 *     S_usable = floor(S_match / B) * B); the tree's edges hold whole blocks and a node's
 *     children are keyed by the B tokens of their first block.
 *   - The cache holds one owner reference on every block it indexes, so the blocks of a
 *     finished request stay resident ("dormant") after pkv_seq_free.
 *   - A node's reference count is the number of attached requests whose matched path runs
 *     through it (ref >= 1: pinned, never evicted).  Every operation advances a clock and
 *     stamps the nodes it traverses (last_access).
 *   - pkv_prefix_evict removes dormant leaves (ref 0, no children), least recently used
 *     first (ties: the older node), releasing all of a leaf's blocks; a parent left with no
 *     children and ref 0 becomes a candidate ("Dynamic radix eviction", leaf-first LRU).
 * Destroy every cache of a pool before the pool (pkv_pool_destroy refuses otherwise).
 * Not thread-safe: serialise calls with the pool's other control-plane calls. */
typedef struct pkv_prefix_cache pkv_prefix_cache;
typedef struct pkv_prefix_stats {
  int64_t nodes;           /* nodes other than the root */
  int64_t blocks;          /* blocks indexed (one owner reference each) */
  int64_t pinned_nodes;    /* reference count >= 1 */
  int64_t dormant_leaves;  /* reference count 0 and no children: eviction candidates */
  int64_t prompt_tokens;   /* sum of the prompt lengths given to pkv_prefix_attach */
  int64_t matched_tokens;  /* sum of the whole-block matches it served ([KVM] Eq. 2 hit rate =
                              matched_tokens / prompt_tokens) */
} pkv_prefix_stats;

int pkv_prefix_cache_create(pkv_pool* pool, pkv_prefix_cache** out);
/* Drops the cache's reference on every indexed block (blocks left with no owner go to the
 * FIFO back, tree preorder). */
int pkv_prefix_cache_destroy(pkv_prefix_cache* cache);

/* Longest cached whole-block prefix of tokens[0, n): *n_matched tokens (a multiple of B),
 * and, if block_ids is not NULL, its blocks (capacity n / B) in order.  Changes nothing. */
int pkv_prefix_match(const pkv_prefix_cache* cache, const int32_t* tokens, int64_t n, int64_t* n_matched,
                     int32_t* block_ids);

/* Serve a new request with prompt tokens[0, n): match as above, split a node matched only in
 * part at the match end, create a sequence (*seq) whose table is the matched blocks (each
 * gains one owner) and whose length is *n_matched, and pin the matched path (every node from
 * the deepest matched one to the root gains a reference and is stamped).  The caller appends
 * the remaining n - *n_matched prompt tokens with pkv_plan_append (a fresh block: the last
 * matched block is full). */
int pkv_prefix_attach(pkv_prefix_cache* cache, const int32_t* tokens, int64_t n, int32_t* seq, int64_t* n_matched);

/* Index the whole blocks of resident sequence seq under its tokens[0, n) (n <= its length;
 * floor(n / B) blocks): blocks whose token path is already cached are not adopted (the
 * sequence keeps its own); the rest become a new leaf, each block gaining the cache as an
 * owner.  A node that diverges (or ends) inside an edge is split at that block boundary.
 * Errors: INVALID_ARG (unknown, released or swapped-out sequence, n > length). */
int pkv_prefix_insert(pkv_prefix_cache* cache, int32_t seq, const int32_t* tokens, int64_t n);

/* Drop the pins pkv_prefix_attach took for seq (each node from its deepest matched node to
 * the root loses a reference and is stamped).  Call before or after pkv_seq_free; the cache
 * keeps the blocks.  Errors: INVALID_ARG (seq holds no pins). */
int pkv_prefix_release(pkv_prefix_cache* cache, int32_t seq);

/* Evict dormant leaves, least recently used first, while the pool's free list holds fewer
 * than target_free blocks and a candidate is left.  *n_released = blocks whose cache
 * reference was dropped (a block also owned by a live sequence stays allocated). */
int pkv_prefix_evict(pkv_prefix_cache* cache, int64_t target_free, int64_t* n_released);

int pkv_prefix_get_stats(const pkv_prefix_cache* cache, pkv_prefix_stats* out);

/* The tree in preorder, children in ascending order of their first block's tokens:
 * nodes int64 [stats.nodes][5] = (parent row or -1 for the root, blocks, ref, last_access,
 * creation serial); blocks int32 [stats.blocks] and tokens int32 [stats.blocks * B], node
 * after node. */
int pkv_prefix_export(const pkv_prefix_cache* cache, int64_t* nodes, int32_t* tokens, int32_t* blocks,
                      int64_t cap_nodes, int64_t cap_blocks);

/* ---------------------------------------------------------------- admission simulator (host only)
 *
 * [PA] "The policy is where it succeeds or fails": how many steps a decode loop needs to
 * finish a saturated queue of requests under an admission policy, using this pool's own
 * allocator (reservations and paged growth are pkv_seq_create / pkv_plan_append /
 * pkv_seq_free calls).  Every step, each running sequence emits one token (prefill is
 * free).  Requests are admitted from the queue head while the policy allows:
 *   PKV_SIM_RESERVE_MAX      reserve max_context tokens per sequence;
 *   PKV_SIM_RESERVE_DECLARED reserve prompt + declared[i] tokens;
 *   PKV_SIM_PAGED            allocate the prompt's blocks if, after they are taken, at least
 *                            watermark * num_blocks blocks are still free; a token that opens
 *                            a block with none free preempts the newest running sequence (its
 *                            blocks are freed, it returns to the queue head and is readmitted
 *                            with blocks for its prompt and the tokens it had generated).
 * Sequences are processed oldest first within a step; a finished one frees its blocks at once.
 * charged_steps = steps + recompute_steps * preemptions.  The pool must have every block
 * free; it is left that way.  Errors: INVALID_ARG (lengths: answer >= 1, prompt + answer <=
 * max_context, declared >= answer), OUT_OF_BLOCKS (a request cannot be admitted into the empty
 * pool: its blocks, plus the watermark for PKV_SIM_PAGED, exceed the pool). */
enum pkv_sim_policy { PKV_SIM_RESERVE_MAX = 0, PKV_SIM_RESERVE_DECLARED = 1, PKV_SIM_PAGED = 2 };
typedef struct pkv_sim_config {
  int32_t policy;          /* enum pkv_sim_policy */
  int32_t max_context;     /* tokens */
  double watermark;        /* PKV_SIM_PAGED: free fraction kept after an admission, in [0, 1) */
  int32_t recompute_steps; /* charged per preemption */
} pkv_sim_config;
typedef struct pkv_sim_result {
  int64_t steps, charged_steps, preemptions, completed, max_running;
  double mean_running;     /* running sequences per step, averaged over steps */
} pkv_sim_result;
int pkv_sim_run(pkv_pool* pool, const pkv_sim_config* cfg, const int32_t* prompt, const int32_t* answer,
                const int32_t* declared, int32_t n_req, pkv_sim_result* out);

/* Failure-path self-test: launch one warp that waits on an mbarrier nothing will
 * complete, bounded by timeout_ns (<= 10 s) of the GPU's global timer -- the same
 * bounded wait the decode kernel uses for its tile loads.  When the bound runs out
 * the kernel records code 5 (detail = nanoseconds waited) in the device error word
 * and returns; pkv_check_device_error then reports PKV_ERR_DEVICE_CHECK and the
 * context stays usable.  No fault, trap or hang is involved. */
int pkv_selftest_bounded_wait(int64_t timeout_ns, pkv_stream_t stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t pkv_launch_count(void);

/* Device code of this library as the runtime loaded it on the current device:
 * *binary_version and *ptx_version are cudaFuncAttributes' binaryVersion and ptxVersion
 * (major * 10 + minor) of the append kernel, e.g. 103 for sm_103a machine code.  Either
 * output pointer may be NULL.  Needs a CUDA device (PKV_ERR_CUDA otherwise). */
int pkv_device_code_version(int32_t* binary_version, int32_t* ptx_version);

/* Synchronize the stream, then read and clear the current device's error word.
 * Returns DEVICE_CHECK if a kernel recorded a bad index since the last check;
 * *code and *detail (the offending value) describe it: 1 a slot out of range (append),
 * 2 a sequence length < 0 or > W * B, 3 a block id out of range in a table, 4 a bounded
 * wait that gave up (detail: where), 6 a prefill chunk longer than max_q, 7 a
 * shared-prefix plan entry out of range (detail: the sequence or work item).
 * Either output pointer may be NULL. */
int pkv_check_device_error(pkv_stream_t stream, int32_t* code, int64_t* detail);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
