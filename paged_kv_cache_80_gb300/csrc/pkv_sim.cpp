// Admission-policy simulator over the pool's own allocator (host control plane).
//
// "PagedAttention" (programmer.ie Inference ch. 14), "The policy is where it succeeds or
// fails": a saturated queue of requests is served by a decode loop in which every running
// sequence emits one token per step (prefill is free).  Three admission policies:
//   0 reserve the maximum context for every sequence,
//   1 reserve the request's declared limit (prompt + declared output),
//   2 paged: admit when the request's blocks fit and, after they are taken, at least
//     `watermark` of the pool is still free; on a shortage, preempt the newest running
//     sequence (its blocks are freed and it is recomputed later: it returns to the front
//     of the queue and, readmitted, needs blocks for its prompt and the tokens it had
//     generated).
// Each preemption is charged `recompute_steps` extra steps.  The reservations and the
// paged allocations are real calls on the pool (create / append / free), so the test bed
// exercises the same allocator the cache uses.
#include <algorithm>
#include <deque>
#include <string>
#include <vector>

#include "pkv_internal.h"

extern "C" {
int pkv_seq_create(pkv_pool* pool, int32_t* seq_id);
int pkv_seq_free(pkv_pool* pool, int32_t seq);
int pkv_plan_append(pkv_pool* pool, const int32_t* seq_ids, const int32_t* n_new, int32_t n, int32_t* slot_mapping,
                    int32_t* cow_pairs, int32_t* n_cow);
}

using pkv::fail;

namespace {

struct Req {
  int32_t prompt, answer, declared;
  int32_t generated = 0;
  int32_t seq = -1;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Append n tokens to seq (allocating blocks as the pool's rule says).
int grow(pkv_pool* pool, int32_t seq, int32_t n, std::vector<int32_t>& slots) {
  if (n <= 0) return PKV_OK;
  slots.resize(static_cast<size_t>(n));
  int32_t cow[2], n_cow = 0;
  return pkv_plan_append(pool, &seq, &n, 1, slots.data(), cow, &n_cow);
}

}  // namespace

extern "C" int pkv_sim_run(pkv_pool* pool, const pkv_sim_config* cfg, const int32_t* prompt, const int32_t* answer,
                           const int32_t* declared, int32_t n_req, pkv_sim_result* out) {
  pkv::clear_error();
  if (!pool || !cfg || !out || n_req < 0 || (n_req > 0 && (!prompt || !answer)))
    return fail(PKV_ERR_INVALID_ARG, "bad arguments to pkv_sim_run");
  if (cfg->policy < 0 || cfg->policy > 2 || cfg->max_context <= 0 || cfg->watermark < 0 || cfg->watermark >= 1 ||
      cfg->recompute_steps < 0)
    return fail(PKV_ERR_INVALID_ARG, "bad simulator configuration");
  if (cfg->policy == 1 && !declared) return fail(PKV_ERR_INVALID_ARG, "policy 1 needs declared limits");
  pkv::Pool& P = *reinterpret_cast<pkv::Pool*>(pool);
  const int64_t N = P.geo.num_blocks, B = P.geo.block_size;
  if (P.free.size() != N) return fail(PKV_ERR_INVALID_ARG, "the simulator needs a pool with every block free");
  std::vector<Req> req(static_cast<size_t>(n_req));
  for (int32_t i = 0; i < n_req; ++i) {
    req[i].prompt = prompt[i];
    req[i].answer = answer[i];
    req[i].declared = declared ? declared[i] : 0;
    if (prompt[i] < 0 || answer[i] < 1 || (declared && declared[i] < answer[i]) ||
        prompt[i] + answer[i] > cfg->max_context)
      return fail(PKV_ERR_INVALID_ARG, "request " + std::to_string(i) + " has bad lengths");
  }
  // tokens a request holds in the pool when (re)admitted, per policy
  auto admit_tokens = [&](const Req& r) -> int64_t {
    if (cfg->policy == 0) return cfg->max_context;
    if (cfg->policy == 1) return std::min<int64_t>(cfg->max_context, int64_t(r.prompt) + r.declared);
    return int64_t(r.prompt) + r.generated;
  };

  std::deque<int32_t> queue;
  for (int32_t i = 0; i < n_req; ++i) queue.push_back(i);
  std::vector<int32_t> running;  // admission order, oldest first
  std::vector<int32_t> slots;
  pkv_sim_result r{};
  int64_t completed = 0, running_sum = 0;
  while (completed < n_req) {
    // admission, head of the queue first
    while (!queue.empty()) {
      Req& q = req[queue.front()];
      const int64_t need = ceil_div(admit_tokens(q), B);
      const int64_t free_now = P.free.size();
      const bool ok = cfg->policy == 2
                          ? (need <= free_now && static_cast<double>(free_now - need) >= cfg->watermark * static_cast<double>(N))
                          : need <= free_now;
      if (!ok) break;
      int32_t seq = 0;
      pkv_seq_create(pool, &seq);
      if (int rc = grow(pool, seq, static_cast<int32_t>(admit_tokens(q)), slots)) return rc;
      q.seq = seq;
      running.push_back(queue.front());
      queue.pop_front();
    }
    if (running.empty()) return fail(PKV_ERR_OUT_OF_BLOCKS, "a request cannot be admitted into the empty pool under this policy");
    // one decode step, oldest first; a paged sequence whose next token opens a block
    // takes a free block or preempts the newest running sequence
    r.steps += 1;
    running_sum += static_cast<int64_t>(running.size());
    r.max_running = std::max<int64_t>(r.max_running, static_cast<int64_t>(running.size()));
    for (size_t k = 0; k < running.size();) {
      const int32_t id = running[k];
      Req& q = req[id];
      bool preempted_self = false;
      if (cfg->policy == 2) {
        const int64_t pos = int64_t(q.prompt) + q.generated;  // position of the new token
        if (pos % B == 0) {
          while (P.free.size() == 0) {
            const int32_t victim = running.back();
            running.pop_back();
            pkv_seq_free(pool, req[victim].seq);
            req[victim].seq = -1;
            queue.push_front(victim);
            r.preemptions += 1;
            if (victim == id) {
              preempted_self = true;
              break;
            }
          }
        }
        if (preempted_self) continue;  // running[k] is gone and k already points past the end
        if (int rc = grow(pool, q.seq, 1, slots)) return rc;
      }
      q.generated += 1;
      if (q.generated == q.answer) {
        pkv_seq_free(pool, q.seq);
        q.seq = -1;
        running.erase(running.begin() + static_cast<std::ptrdiff_t>(k));
        completed += 1;
        continue;
      }
      ++k;
    }
  }
  r.completed = completed;
  r.charged_steps = r.steps + r.preemptions * cfg->recompute_steps;
  r.mean_running = r.steps ? static_cast<double>(running_sum) / static_cast<double>(r.steps) : 0.0;
  *out = r;
  return PKV_OK;
}
