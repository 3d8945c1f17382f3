// Serving runtime around the stack step ("NanoFlow: Towards Optimal LLM
// Serving Throughput", "The NanoFlow Runtime System").
//
// Batch formation: every iteration carries a constant token budget B_dense.
// Requests that are decoding get one token each first (their latency is on
// every request's critical path); prompts are cut into chunks, first-come
// first-served, that fill the rest of the budget exactly while there is
// prefill work.  Asynchronous scheduling: iteration i+1 is formed and enqueued
// while iteration i runs; the tokens iteration i produced are read back when
// iteration i+2 is formed, so a request that emitted its end token in
// iteration i still runs in iteration i+1 (one wasted token) — the pages'
// one-iteration deferral.  The token a decode row consumes is its request's
// previous output, kept on the device, so no iteration waits for the host.
// KV pages come from a free list and go back to it when a request finishes.
//
// Re-planning: the pages' pipeline is searched once and kept static, which
// they name as a limitation when the prefill/decode mix shifts.  Here the plan
// search (host only, fast) runs again whenever the decode share of the batch
// moved by more than a threshold since the last plan, or the token count
// changed; the new split is applied with nf_plan_set_batch.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <string>
#include <vector>

#include "../../include/nanoflow.h"
#include "common.cuh"
#include "internal.h"

namespace {

nf_status rfail(nf_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return nf::set_last_error(code, buf);
}

#define RT_TRY(expr)            \
  do {                          \
    nf_status s_ = (expr);      \
    if (s_ != NF_OK) return s_; \
  } while (0)

// ------------------------------------------------------------------ host
struct Request {
  int id = 0;
  std::vector<int> prompt;
  int max_new = 0;
  int slot = -1;            // device token slot while admitted
  int prompt_done = 0;      // prompt tokens scheduled
  int kv_len = 0;           // KV length after the last scheduled step
  int scheduled_gen = 0;    // output tokens whose rows were scheduled
  bool admitted = false;
  bool finished = false;    // as of the results applied so far
  std::vector<int> pages;
  std::vector<int> generated;
};

struct IterRecord {
  int iteration = -1;
  std::vector<int> row_request, row_pos, row_token, row_emit, row_slot;
  std::vector<int> seq_lens, block_table, prefill_q;
  int n_decode = 0, n_prefill = 0;
  bool applied = false;
};

struct Scheduler {
  int b_dense = 0, max_requests = 0, max_pages = 0, page = 16, eos = -1;
  std::vector<Request> reqs;          // by id
  std::deque<int> waiting;            // ids not yet admitted, in arrival order
  std::vector<int> active;            // admitted ids, in admission order
  std::vector<int> free_pages, free_slots;
  int iteration = 0;

  void init(int b, int maxr, int maxp, int num_pages, int page_size, int eos_token) {
    b_dense = b;
    max_requests = maxr;
    max_pages = maxp;
    page = page_size;
    eos = eos_token;
    free_pages.clear();
    for (int p = num_pages - 1; p >= 0; --p) free_pages.push_back(p);  // page 0 handed out first
    free_slots.clear();
    for (int s = maxr - 1; s >= 0; --s) free_slots.push_back(s);
  }

  // Pages so that `len` positions are covered; false if the pool is empty.
  bool cover(Request& r, int len) {
    const int need = (len + page - 1) / page;
    if (need > max_pages) return false;
    while ((int)r.pages.size() < need) {
      if (free_pages.empty()) return false;
      r.pages.push_back(free_pages.back());
      free_pages.pop_back();
    }
    return true;
  }

  void release(Request& r) {
    for (int p : r.pages) free_pages.push_back(p);
    r.pages.clear();
    if (r.slot >= 0) free_slots.push_back(r.slot);
    r.slot = -1;
  }

  // The next iteration's batch; rec.row_* empty when there is nothing to run.
  nf_status form(IterRecord& rec) {
    rec = IterRecord{};
    rec.iteration = iteration;
    std::vector<int> dec, pre, pre_len;
    // 1. one token for every decoding request, in admission order
    for (int id : active) {
      Request& r = reqs[id];
      if (r.finished || r.prompt_done < (int)r.prompt.size()) continue;
      if (r.scheduled_gen < 1 || r.scheduled_gen >= r.max_new) continue;
      if ((int)dec.size() >= b_dense) break;
      if (!cover(r, r.kv_len + 1)) return NF_ERR_OOM;
      dec.push_back(id);
    }
    // 2. prompt chunks fill the rest: requests already prefilling, then new ones
    int cap = b_dense - (int)dec.size();
    auto take_chunk = [&](Request& r) {
      int chunk = std::min<int>((int)r.prompt.size() - r.prompt_done, cap);
      while (chunk > 0 && !cover(r, r.prompt_done + chunk)) --chunk;  // what the pool allows
      if (chunk > 0) {
        pre.push_back(r.id);
        pre_len.push_back(chunk);
        cap -= chunk;
      }
      return chunk;
    };
    for (int id : active) {
      if (cap == 0) break;
      Request& r = reqs[id];
      if (!r.finished && r.prompt_done < (int)r.prompt.size()) take_chunk(r);
    }
    while (cap > 0 && !waiting.empty() && !free_slots.empty()) {
      Request& r = reqs[waiting.front()];
      if (take_chunk(r) == 0) break;  // no page left for a new prompt
      waiting.pop_front();
      r.admitted = true;
      r.slot = free_slots.back();
      free_slots.pop_back();
      active.push_back(r.id);
    }
    // 3. the rows: decode sequences first, then the prefill chunks
    const int n_seq = (int)(dec.size() + pre.size());
    rec.n_decode = (int)dec.size();
    rec.n_prefill = (int)pre.size();
    rec.block_table.assign((size_t)n_seq * max_pages, -1);
    int si = 0;
    auto emit_row = [&](Request& r, int pos, int tok, int emit) {
      rec.row_request.push_back(r.id);
      rec.row_pos.push_back(pos);
      rec.row_token.push_back(tok);
      rec.row_emit.push_back(emit);
      rec.row_slot.push_back(r.slot);
    };
    for (int id : dec) {
      Request& r = reqs[id];
      emit_row(r, r.kv_len, -1, 1);
      r.kv_len += 1;
      r.scheduled_gen += 1;
      rec.seq_lens.push_back(r.kv_len);
      std::copy(r.pages.begin(), r.pages.end(), rec.block_table.begin() + (size_t)si * max_pages);
      ++si;
    }
    for (size_t j = 0; j < pre.size(); ++j) {
      Request& r = reqs[pre[j]];
      const int chunk = pre_len[j];
      const bool last = r.prompt_done + chunk == (int)r.prompt.size();
      for (int c = 0; c < chunk; ++c) {
        const int pos = r.prompt_done + c;
        emit_row(r, pos, r.prompt[pos], last && c == chunk - 1);
      }
      r.prompt_done += chunk;
      r.kv_len = r.prompt_done;
      if (last) r.scheduled_gen = 1;
      rec.seq_lens.push_back(r.kv_len);
      rec.prefill_q.push_back(chunk);
      std::copy(r.pages.begin(), r.pages.end(), rec.block_table.begin() + (size_t)si * max_pages);
      ++si;
    }
    ++iteration;
    return NF_OK;
  }

  // Tokens an iteration produced (sampled[t] for rows with row_emit).
  void apply(IterRecord& rec, const int* sampled) {
    if (rec.applied) return;
    rec.applied = true;
    for (size_t t = 0; t < rec.row_request.size(); ++t) {
      if (!rec.row_emit[t]) continue;
      Request& r = reqs[rec.row_request[t]];
      if (r.finished) continue;  // a row scheduled before the end was known
      r.generated.push_back(sampled[t]);
      if (sampled[t] == eos || (int)r.generated.size() >= r.max_new) {
        r.finished = true;
        release(r);
        active.erase(std::find(active.begin(), active.end(), r.id));
      }
    }
  }
};

// ---------------------------------------------------------------- device
__global__ void compose_tokens_kernel(const int* row_token, const int* row_slot, const int* next_tok,
                                      int* tokens, int n) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n) tokens[t] = row_token[t] >= 0 ? row_token[t] : next_tok[row_slot[t]];
}

// Greedy sampling of the emitting rows: block i takes logits row i, which
// belongs to token row rows[i]; the index of the largest logit, the lowest
// index on ties, goes to the request's token slot and to sampled[rows[i]]
// (rows that emit nothing hold -1, set before).
__global__ void __launch_bounds__(256) sample_kernel(const __nv_bfloat16* logits, const int* rows,
                                                     const int* row_slot, int* next_tok, int* sampled,
                                                     int vocab) {
  const int t = rows[blockIdx.x];
  const __nv_bfloat16* row = logits + (size_t)blockIdx.x * vocab;
  float best = -INFINITY;
  int bi = vocab;
  for (int v = threadIdx.x; v < vocab; v += blockDim.x) {
    const float x = __bfloat162float(row[v]);
    if (x > best || (x == best && v < bi)) {
      best = x;
      bi = v;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  __shared__ float sb[8];
  __shared__ int si[8];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sb[w] = best;
    si[w] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < 8; ++k)
      if (sb[k] > best || (sb[k] == best && si[k] < bi)) {
        best = sb[k];
        bi = si[k];
      }
    if (bi >= vocab) bi = 0;  // every logit NaN
    sampled[t] = bi;
    next_tok[row_slot[t]] = bi;
  }
}

}  // namespace

struct nf_runtime_s {
  nf_model_shape shape{};
  nf_runtime_opts opts{};
  Scheduler sched;
  IterRecord recs[2];            // the iterations in flight (by parity)
  IterRecord last;               // the last formed batch (host-only mode)
  nf_plan plan = nullptr;
  double planned_share = -1.0;
  int planned_T = -1;
  // device
  int *d_next = nullptr, *d_tokens = nullptr, *d_sampled = nullptr, *d_rows = nullptr;
  int *d_bt = nullptr, *d_sl = nullptr;
  __nv_bfloat16* d_logits = nullptr;
  int* h_in[2] = {nullptr, nullptr};    // pinned: rows (token, slot, emit), block table, lengths
  int* h_out[2] = {nullptr, nullptr};   // pinned: sampled tokens
  cudaEvent_t done[2] = {nullptr, nullptr};
  cudaStream_t last_stream = nullptr;
  int launched = 0;
  int last_emit = 0;  // emitting rows of the last launched iteration (its logits rows)
};

namespace {

size_t in_ints(const nf_runtime_s* rt) {
  const size_t T = rt->opts.b_dense;
  return 4 * T + T * rt->opts.max_pages_per_seq + T;
}

void free_rt(nf_runtime rt) {
  if (!rt) return;
  if (rt->plan) nf_plan_destroy(rt->plan);
  void* dev[] = {rt->d_next, rt->d_tokens, rt->d_sampled, rt->d_rows, rt->d_bt, rt->d_sl, rt->d_logits};
  for (void* b : dev)
    if (b) cudaFree(b);
  for (int i = 0; i < 2; ++i) {
    if (rt->h_in[i]) cudaFreeHost(rt->h_in[i]);
    if (rt->h_out[i]) cudaFreeHost(rt->h_out[i]);
    if (rt->done[i]) cudaEventDestroy(rt->done[i]);
  }
  delete rt;
}

}  // namespace

extern "C" {

nf_status nf_runtime_create(const nf_model_shape* shape, const nf_runtime_opts* o, nf_runtime* out) {
  if (!shape || !o || !out) return rfail(NF_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (o->b_dense < 1 || o->max_requests < 1 || o->max_pages_per_seq < 1 || o->num_pages < 1 ||
      o->vocab < 8 || o->vocab % 8)
    return rfail(NF_ERR_INVALID_ARG,
                              "b_dense, max_requests, max_pages_per_seq, num_pages must be >= 1 and "
                              "vocab a positive multiple of 8");
  nf_runtime rt = new nf_runtime_s();
  rt->shape = *shape;
  rt->opts = *o;
  rt->sched.init(o->b_dense, o->max_requests, o->max_pages_per_seq, o->num_pages, shape->page_size,
                 o->eos_token);
  if (o->host_only) {
    *out = rt;
    return NF_OK;
  }
  // a plan with room for b_dense sequences of one token (the largest structure)
  std::vector<int32_t> none(1, 1);
  nf_batch_desc b{};
  b.n_decode = o->b_dense;
  b.n_prefill = 0;
  b.prefill_q_lens = none.data();
  b.max_pages_per_seq = o->max_pages_per_seq;
  b.num_pages = o->num_pages;
  nf_plan_opts po{};
  po.n_attn = po.n_ffn = 1;
  po.attn_bounds[1] = po.ffn_bounds[1] = o->b_dense;
  po.executor = NF_EXEC_SEQUENTIAL;
  po.kv_chunk = 1024;
  nf_status s = nf_plan_create(shape, &b, &po, &rt->plan);
  auto dalloc = [&](void** p, size_t n) { return cudaMalloc(p, n) == cudaSuccess; };
  const size_t T = o->b_dense;
  bool ok = s == NF_OK && dalloc((void**)&rt->d_next, (size_t)o->max_requests * 4) &&
            dalloc((void**)&rt->d_tokens, T * 4) && dalloc((void**)&rt->d_sampled, T * 4) &&
            dalloc((void**)&rt->d_rows, 4 * T * 4) &&
            dalloc((void**)&rt->d_bt, T * o->max_pages_per_seq * 4) &&
            dalloc((void**)&rt->d_sl, T * 4) &&
            dalloc((void**)&rt->d_logits, T * (size_t)o->vocab * 2);
  for (int i = 0; ok && i < 2; ++i)
    ok = cudaHostAlloc((void**)&rt->h_in[i], in_ints(rt) * 4, cudaHostAllocDefault) == cudaSuccess &&
         cudaHostAlloc((void**)&rt->h_out[i], T * 4, cudaHostAllocDefault) == cudaSuccess &&
         cudaEventCreateWithFlags(&rt->done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    free_rt(rt);
    return s != NF_OK ? s : rfail(NF_ERR_OOM, "runtime buffers could not be allocated");
  }
  *out = rt;
  return NF_OK;
}

void nf_runtime_destroy(nf_runtime rt) {
  if (rt && rt->launched && rt->last_stream) cudaStreamSynchronize(rt->last_stream);
  free_rt(rt);
}

nf_status nf_runtime_submit(nf_runtime rt, const int32_t* prompt, int32_t prompt_len,
                            int32_t max_new_tokens, int32_t* id) {
  if (!rt || !prompt || !id) return rfail(NF_ERR_INVALID_ARG, "NULL argument");
  if (prompt_len < 1 || max_new_tokens < 1)
    return rfail(NF_ERR_INVALID_ARG, "prompt_len and max_new_tokens must be >= 1");
  if ((int64_t)prompt_len + max_new_tokens >
      (int64_t)rt->opts.max_pages_per_seq * rt->shape.page_size)
    return rfail(NF_ERR_INVALID_ARG, "prompt + output exceed max_pages_per_seq pages");
  for (int i = 0; i < prompt_len; ++i)
    if (prompt[i] < 0 || prompt[i] >= rt->opts.vocab)
      return rfail(NF_ERR_INVALID_ARG, "prompt token %d out of range", i);
  Request r;
  r.id = (int)rt->sched.reqs.size();
  r.prompt.assign(prompt, prompt + prompt_len);
  r.max_new = max_new_tokens;
  rt->sched.reqs.push_back(r);
  rt->sched.waiting.push_back(r.id);
  *id = r.id;
  return NF_OK;
}

static void fill_view(const IterRecord& rec, nf_runtime_batch* out) {
  out->iteration = rec.iteration;
  out->n_tokens = (int32_t)rec.row_request.size();
  out->n_decode = rec.n_decode;
  out->n_prefill = rec.n_prefill;
  out->row_request = rec.row_request.data();
  out->row_pos = rec.row_pos.data();
  out->row_token = rec.row_token.data();
  out->row_emit = rec.row_emit.data();
  out->seq_lens = rec.seq_lens.data();
  out->block_table = rec.block_table.data();
  out->prefill_q_lens = rec.prefill_q.data();
}

nf_status nf_runtime_form(nf_runtime rt, nf_runtime_batch* out) {
  if (!rt || !out) return rfail(NF_ERR_INVALID_ARG, "NULL argument");
  if (!rt->opts.host_only)
    return rfail(NF_ERR_INVALID_ARG, "nf_runtime_form is for host-only runtimes");
  std::memset(out, 0, sizeof(*out));
  const IterRecord& old = rt->recs[rt->sched.iteration & 1];
  if (old.iteration >= 0 && !old.applied && !old.row_request.empty())
    return rfail(NF_ERR_INVALID_ARG, "apply iteration %d before forming iteration %d",
                 old.iteration, rt->sched.iteration);
  const nf_status s = rt->sched.form(rt->recs[rt->sched.iteration & 1]);
  if (s != NF_OK) return rfail(s, "the page pool cannot hold the decoding requests");
  const IterRecord& rec = rt->recs[(rt->sched.iteration - 1) & 1];
  fill_view(rec, out);
  out->free_pages = (int32_t)rt->sched.free_pages.size();
  return NF_OK;
}

nf_status nf_runtime_apply(nf_runtime rt, int32_t iteration, const int32_t* sampled) {
  if (!rt || !sampled) return rfail(NF_ERR_INVALID_ARG, "NULL argument");
  IterRecord& rec = rt->recs[iteration & 1];
  if (rec.iteration != iteration || rec.applied)
    return rfail(NF_ERR_INVALID_ARG, "iteration %d is not awaiting results", iteration);
  rt->sched.apply(rec, sampled);
  return NF_OK;
}

// Apply the results of the iteration held in slot `k` once the GPU is done with it.
static nf_status finish_iteration(nf_runtime rt, int k) {
  IterRecord& rec = rt->recs[k];
  if (rec.iteration < 0 || rec.applied || rec.row_request.empty()) return NF_OK;
  if (cudaEventSynchronize(rt->done[k]) != cudaSuccess)
    return rfail(NF_ERR_CUDA, "runtime iteration failed: %s",
                              cudaGetErrorString(cudaGetLastError()));
  rt->sched.apply(rec, rt->h_out[k]);
  return NF_OK;
}

nf_status nf_runtime_step(nf_runtime rt, const nf_stack_weights* w, void* const* k_pools,
                          void* const* v_pools, void* stream, nf_runtime_batch* out) {
  if (!rt || !w || !k_pools || !v_pools) return rfail(NF_ERR_INVALID_ARG, "NULL argument");
  if (rt->opts.host_only)
    return rfail(NF_ERR_INVALID_ARG, "a host-only runtime cannot launch steps");
  if (w->vocab != rt->opts.vocab)
    return rfail(NF_ERR_INVALID_ARG, "the LM head's vocab differs from the runtime's");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int k = rt->sched.iteration & 1;
  // the iteration two back used this slot's buffers: its tokens are in by now
  RT_TRY(finish_iteration(rt, k));
  IterRecord& rec = rt->recs[k];
  nf_status s = rt->sched.form(rec);
  if (s != NF_OK) return rfail(s, "the page pool cannot hold the decoding requests");
  if (out) {
    std::memset(out, 0, sizeof(*out));
    fill_view(rec, out);
    out->free_pages = (int32_t)rt->sched.free_pages.size();
  }
  const int T = (int)rec.row_request.size();
  if (T == 0) return NF_OK;  // nothing to run: every request finished (or waits for pages)
  // inputs of the iteration, staged in pinned memory and copied on the stream
  const int n_seq = rec.n_decode + rec.n_prefill, MP = rt->opts.max_pages_per_seq;
  int* h = rt->h_in[k];
  std::copy(rec.row_token.begin(), rec.row_token.end(), h);
  std::copy(rec.row_slot.begin(), rec.row_slot.end(), h + T);
  std::copy(rec.row_emit.begin(), rec.row_emit.end(), h + 2 * T);
  // emitting rows, in row order (the LM head runs on these only)
  int* hrows = h + 3 * (size_t)T;
  int n_emit = 0;
  for (int t = 0; t < T; ++t)
    if (rec.row_emit[t]) hrows[n_emit++] = t;
  int* hbt = h + 4 * (size_t)rt->opts.b_dense;
  std::copy(rec.block_table.begin(), rec.block_table.end(), hbt);
  int* hsl = hbt + (size_t)rt->opts.b_dense * MP;
  std::copy(rec.seq_lens.begin(), rec.seq_lens.end(), hsl);
  // the rows' arrays go to d_rows as [token | slot | emit | emitting rows]
  if (cudaMemcpyAsync(rt->d_rows, h, (3 * (size_t)T + n_emit) * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(rt->d_bt, hbt, (size_t)n_seq * MP * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(rt->d_sl, hsl, (size_t)n_seq * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return rfail(NF_ERR_CUDA, "runtime input copies failed");
  // the plan follows the batch; the search runs again when the mix moved
  nf_batch_desc b{};
  b.n_decode = rec.n_decode;
  b.n_prefill = rec.n_prefill;
  b.prefill_q_lens = rec.prefill_q.empty() ? rec.seq_lens.data() : rec.prefill_q.data();
  b.seq_lens_hint = rec.seq_lens.data();
  b.max_pages_per_seq = MP;
  b.num_pages = rt->opts.num_pages;
  const double share = (double)rec.n_decode / T;
  const bool replan = rt->opts.replan_threshold >= 0.f &&
                      (T != rt->planned_T || std::fabs(share - rt->planned_share) > rt->opts.replan_threshold);
  if (replan) {
    nf_plan_opts po{};
    double pred = 0;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    RT_TRY(nf_plan_search(&rt->shape, &b, nullptr, sms, &po, &pred));
    po.kv_chunk = 0;  // kept as created
    po.attn_warps = 0;
    po.attn_impl = NF_ATTN_AUTO;
    RT_TRY(nf_plan_set_batch(rt->plan, &b, &po, st));
    rt->planned_share = share;
    rt->planned_T = T;
    if (out) out->replanned = 1;
  } else {
    RT_TRY(nf_plan_set_batch(rt->plan, &b, nullptr, st));
  }
  const int* d_tok = rt->d_rows;
  const int* d_slot = rt->d_rows + T;
  const int* d_sel = rt->d_rows + 3 * T;
  compose_tokens_kernel<<<(T + 255) / 256, 256, 0, st>>>(d_tok, d_slot, rt->d_next, rt->d_tokens, T);
  if (cudaGetLastError() != cudaSuccess) return rfail(NF_ERR_CUDA, "token compose failed");
  // logits for the emitting rows only, then one sampling block per such row
  RT_TRY(nf_stack_step_rows(rt->plan, w, rt->d_tokens, k_pools, v_pools, rt->d_bt, rt->d_sl, d_sel,
                            n_emit, rt->d_logits, stream));
  if (cudaMemsetAsync(rt->d_sampled, 0xFF, (size_t)T * 4, st) != cudaSuccess)  // -1: no token
    return rfail(NF_ERR_CUDA, "runtime sampling failed");
  if (n_emit > 0)
    sample_kernel<<<n_emit, 256, 0, st>>>(rt->d_logits, d_sel, d_slot, rt->d_next, rt->d_sampled,
                                          rt->opts.vocab);
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyAsync(rt->h_out[k], rt->d_sampled, (size_t)T * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaEventRecord(rt->done[k], st) != cudaSuccess)
    return rfail(NF_ERR_CUDA, "runtime sampling failed");
  rt->last_stream = st;
  rt->last_emit = n_emit;
  ++rt->launched;
  return NF_OK;
}

nf_status nf_runtime_logits(nf_runtime rt, void* dst, int32_t cap_rows, int32_t* n_rows) {
  if (!rt || !n_rows) return rfail(NF_ERR_INVALID_ARG, "NULL argument");
  if (rt->opts.host_only) return rfail(NF_ERR_INVALID_ARG, "a host-only runtime has no logits");
  *n_rows = rt->launched ? rt->last_emit : 0;
  if (*n_rows == 0 || !dst) return NF_OK;
  if (cap_rows < *n_rows)
    return rfail(NF_ERR_INVALID_ARG, "the last iteration has %d logits rows, more than cap_rows %d",
                 *n_rows, cap_rows);
  if (cudaStreamSynchronize(rt->last_stream) != cudaSuccess ||
      cudaMemcpy(dst, rt->d_logits, (size_t)*n_rows * rt->opts.vocab * 2, cudaMemcpyDefault) !=
          cudaSuccess)
    return rfail(NF_ERR_CUDA, "reading the logits failed");
  return NF_OK;
}

nf_status nf_runtime_sync(nf_runtime rt) {
  if (!rt) return rfail(NF_ERR_INVALID_ARG, "runtime is NULL");
  if (rt->opts.host_only) return NF_OK;
  const int it = rt->sched.iteration;  // apply in launch order: older slot first
  RT_TRY(finish_iteration(rt, it & 1));
  RT_TRY(finish_iteration(rt, (it + 1) & 1));
  return nf_plan_poll(rt->plan, 0);
}

nf_status nf_runtime_result(nf_runtime rt, int32_t id, int32_t* finished, int32_t* n_tokens,
                            int32_t* tokens, int32_t cap) {
  if (!rt || id < 0 || id >= (int)rt->sched.reqs.size())
    return rfail(NF_ERR_INVALID_ARG, "unknown request");
  const Request& r = rt->sched.reqs[id];
  if (finished) *finished = r.finished ? 1 : 0;
  if (n_tokens) *n_tokens = (int32_t)r.generated.size();
  if (tokens)
    for (int i = 0; i < cap && i < (int)r.generated.size(); ++i) tokens[i] = r.generated[i];
  return NF_OK;
}

nf_status nf_runtime_counts(nf_runtime rt, int32_t* waiting, int32_t* active, int32_t* free_pages) {
  if (!rt) return rfail(NF_ERR_INVALID_ARG, "runtime is NULL");
  if (waiting) *waiting = (int32_t)rt->sched.waiting.size();
  if (active) *active = (int32_t)rt->sched.active.size();
  if (free_pages) *free_pages = (int32_t)rt->sched.free_pages.size();
  return NF_OK;
}

}  // extern "C"
