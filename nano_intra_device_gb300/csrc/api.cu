// C ABI of the nano-batched decoder-layer step: plans, executors, single-step
// entry points.  Host code; every arithmetic step runs in the kernels.
#include <algorithm>
#include <cmath>
#include <utility>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/nanoflow.h"
#include "common.cuh"
#include "kernels.h"
#include "internal.h"
#include "schedule.h"

using nf::GemmArgs;

namespace {

thread_local std::string g_err;

nf_status fail(nf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

#define NF_CUDA(call)                                                                   \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(NF_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));         \
  } while (0)

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

struct GlobalSplitWs {
  float* part = nullptr;
  int* cnt = nullptr;
};

// Split-K workspace of nf_gemm (no plan): allocated on first use.
GlobalSplitWs* global_split_ws();

// Status word for entry points that run without a plan (nf_gemm, nf_rmsnorm),
// one per device (device memory belongs to the device current when allocated).
constexpr int kMaxDevices = 64;
std::mutex g_global_mu;

uint32_t* global_status() {
  static uint32_t* p[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_global_mu);
  if (!p[dev] && cudaMalloc(&p[dev], sizeof(uint32_t)) == cudaSuccess)
    cudaMemset(p[dev], 0, sizeof(uint32_t));
  return p[dev];
}

constexpr int64_t kDefaultTimeoutNs = 2000000000LL;

// Split-K: used when a GEMM has fewer output tiles than half the SMs (small
// decode batches), so that every SM still works.  Each split keeps at least 4
// K-blocks; tiles x splits never exceeds the SM count, which bounds the
// workspace of fp32 partial tiles (128 x 256 each).
constexpr int kSplitMaxTiles = 256;
constexpr int kSplitMaxUnits = 256;
constexpr size_t kSplitPartBytes = (size_t)kSplitMaxUnits * 128 * 256 * 4;

// nf_gemm's split-K workspace on the current device, allocated on first use
// there (fields stay NULL when the allocation failed).
GlobalSplitWs* global_split_ws() {
  static GlobalSplitWs ws[kMaxDevices];
  static GlobalSplitWs none;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return &none;
  std::lock_guard<std::mutex> lk(g_global_mu);
  GlobalSplitWs& w = ws[dev];
  if (!w.part) {
    if (cudaMalloc(&w.part, kSplitPartBytes) != cudaSuccess ||
        cudaMalloc(&w.cnt, kSplitMaxTiles * 4) != cudaSuccess ||
        cudaMemset(w.cnt, 0, kSplitMaxTiles * 4) != cudaSuccess) {
      if (w.part) cudaFree(w.part);
      if (w.cnt) cudaFree(w.cnt);
      w.part = nullptr;
      w.cnt = nullptr;
      cudaGetLastError();
    }
  }
  return &w;
}

int choose_splits(int tiles, int K, int sms) {
  if (tiles <= 0 || tiles * 2 > sms || tiles > kSplitMaxTiles) return 1;
  const int nk = (K + 63) / 64;
  int s = sms / tiles;
  s = s < nk / 4 ? s : nk / 4;
  s = s < 16 ? s : 16;
  if (tiles * s > kSplitMaxUnits) s = kSplitMaxUnits / tiles;
  return s > 1 ? s : 1;
}

}  // namespace

struct nf_plan_s {
  nf_model_shape shape{};
  int n_decode = 0, n_prefill = 0;
  std::vector<int> prefill_q, seq_hint;
  int max_pages = 0, num_pages = 0;
  int n_seq = 0, T = 0;         // the current batch (nf_plan_set_batch may change it)
  int seq_cap = 0, T_cap = 0;   // what the workspace was allocated for
  int* set_stage = nullptr;     // pinned host staging of nf_plan_set_batch (two halves)
  float2* rope_cs = nullptr;    // RoPE (cos, sin) table [max_pages * page_size][head_dim / 2]
  int set_flip = 0;
  // set_ev[h]: recorded after the copies out of staging half h; a later call
  // waits for it before writing that half again
  cudaEvent_t set_ev[2] = {nullptr, nullptr};
  bool set_ev_live[2] = {false, false};
  std::vector<int> q_lens, tok_begin;
  nf_plan_opts opts{};
  int num_sms = 0;
  int max_chunks = 0, item_capacity = 0;
  // device workspace
  int *d_q_lens = nullptr, *d_tok_begin = nullptr, *d_seg_bounds = nullptr;
  int *tok_seq = nullptr, *tok_pos = nullptr, *tok_slot = nullptr, *tok_nchunks = nullptr;
  int *items = nullptr, *seg_items = nullptr, *fetch = nullptr, *row_done = nullptr;
  float* partials = nullptr;
  uint32_t* status = nullptr;
  __nv_bfloat16 *n1 = nullptr, *q = nullptr, *o = nullptr, *h = nullptr, *n2 = nullptr,
                *a = nullptr;
  // host-API staging
  __nv_bfloat16 *x_stage = nullptr, *y_stage = nullptr;
  int *bt_stage = nullptr, *sl_stage = nullptr;
  // executor
  cudaStream_t s_gemm = nullptr, s_attn = nullptr;
  std::vector<cudaEvent_t> ev;
  // tensor maps over plan buffers (A operands)
  CUtensorMap tm_n1{}, tm_o{}, tm_n2{}, tm_a{};
  // the same buffers with 64- and 128-row boxes: token tiles of the weight-row
  // GEMM, indexed as XM_N1 ... XM_A
  CUtensorMap tm_x64[4]{}, tm_x128[4]{};
  // tensor maps over the weights in use, and a cache of every weight set seen
  // (a stack reuses one plan for all its layers)
  const void* wkey[4] = {nullptr, nullptr, nullptr, nullptr};
  CUtensorMap tm_wqkv{}, tm_wo{}, tm_wg{}, tm_wu{}, tm_wd{};
  CUtensorMap tm_wo224{}, tm_wd224{};  // the same with 224-row boxes (224-column tiles)
  // weight-row GEMM: QKV with head_dim / 2-row boxes, O and down with 128-row boxes
  CUtensorMap tm_wqkv_h{}, tm_wo128{}, tm_wd128{};
  struct WeightMaps {
    const void* key[4];
    CUtensorMap qkv, o, g, u, d;  // a MoE layer keeps its expert maps in g (gate/up) and d
    CUtensorMap o224, d224;
    CUtensorMap qkv_h, o128, d128;
  };
  std::vector<WeightMaps> wcache;
  // mixture of experts: routing, grouped rows and the expert weight maps
  int *moe_off = nullptr, *moe_perm = nullptr, *moe_pair_row = nullptr;
  float *moe_pair_w = nullptr, *moe_out = nullptr;
  __nv_bfloat16 *moe_a = nullptr, *moe_act = nullptr;
  CUtensorMap tm_moe_a{}, tm_moe_act{}, tm_egu{}, tm_edn{};
  // attention: which kernel, and TMA maps over every (K pool, V pool) pair seen
  bool attn_mma = false;
  struct PoolMaps {
    const void *k, *v;
    CUtensorMap tk, tv;    // 8-row-group boxes (prefill kernel)
    CUtensorMap dk, dv;    // whole-page boxes (decode kernel)
  };
  std::vector<PoolMaps> pcache;
  // prefill-chunk attention: tiles of rows (first, end, sequence, 0) of every
  // attention nano-batch, nano-batch i's from pf_seg[i]; pinned staging for
  // nf_plan_set_batch (two halves)
  int4* pf_tiles = nullptr;
  int4* pf_stage = nullptr;
  int pf_seg[NF_MAX_NANO + 1] = {};
  // split-K GEMM workspace: fp32 partial tiles and per-tile arrival counters
  float* gemm_part = nullptr;
  int* gemm_cnt = nullptr;
  // split-KV counters: one set per layer of a stack step (zeroed by the metadata kernel)
  int counter_sets = 1, cur_set = 0;
  // stack: activations between layers, and the LM head's tensor map
  __nv_bfloat16 *xa = nullptr, *xb = nullptr;
  const void* lm_key = nullptr;
  int lm_vocab = 0;
  CUtensorMap tm_lm{}, tm_lm128{};
  // tracing
  struct TraceRec {
    int op, nano, step;
    cudaEvent_t b, e, s0;
  };
  int trace_left = 0, trace_step = 0;
  uint32_t trace_ops = ~0u;  // bit NF_OP_x: record that operation
  cudaEvent_t trace_s0 = nullptr;
  std::vector<TraceRec> trace;
  std::vector<cudaEvent_t> ev_pool;
  // host-buffer step: a CUDA graph of the copies in, the step and the copy out,
  // per set of pointers (seen once directly first), replayed on a plan-owned
  // stream; batch_version invalidates them when nf_plan_set_batch runs
  struct HostGraph {
    const void* key[16];
    uint64_t version;
    cudaGraphExec_t exec;  // nullptr: seen once, not captured yet
  };
  std::vector<HostGraph> hgraphs;
  uint64_t batch_version = 0;
  cudaStream_t s_host = nullptr;
  cudaEvent_t ev_host = nullptr;
  // pipelined host-buffer steps: two staging slots, a stream for the copies in
  // and one for the copies out; per slot: inputs landed, step done, y copied out
  struct HostPipe {
    __nv_bfloat16 *x[2] = {nullptr, nullptr}, *y[2] = {nullptr, nullptr};
    int *bt[2] = {nullptr, nullptr}, *sl[2] = {nullptr, nullptr};
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t in_done[2] = {}, step_done[2] = {}, out_done[2] = {};
    int next = 0;
  } pipe;
};

namespace {

size_t buf_bytes(nf_plan p, int which) {
  const size_t T = p->T, H = p->shape.hidden, QD = (size_t)p->shape.n_q_heads * p->shape.head_dim;
  switch (which) {
    case NF_BUF_TOK_SEQ:
    case NF_BUF_TOK_POS:
    case NF_BUF_TOK_SLOT: return T * 4;
    case NF_BUF_ITEMS: return (size_t)p->item_capacity * 2 * 4;
    case NF_BUF_ITEM_SEG: return (size_t)(p->opts.n_attn + 1) * 4;
    case NF_BUF_N1:
    case NF_BUF_H:
    case NF_BUF_N2: return T * H * 2;
    case NF_BUF_Q:
    case NF_BUF_O: return T * QD * 2;
    case NF_BUF_A: return T * (size_t)p->shape.ffn * 2;
    case NF_BUF_MOE_OFF: return p->moe_off ? (size_t)(p->shape.n_experts + 1) * 4 : 0;
    case NF_BUF_MOE_PERM:
    case NF_BUF_MOE_PAIR_ROW:
    case NF_BUF_MOE_PAIR_W: return p->moe_off ? T * p->shape.top_k * 4 : 0;
    default: return 0;
  }
}

const void* buf_ptr(nf_plan p, int which) {
  switch (which) {
    case NF_BUF_TOK_SEQ: return p->tok_seq;
    case NF_BUF_TOK_POS: return p->tok_pos;
    case NF_BUF_TOK_SLOT: return p->tok_slot;
    case NF_BUF_ITEMS: return p->items;
    case NF_BUF_ITEM_SEG: return p->seg_items;
    case NF_BUF_N1: return p->n1;
    case NF_BUF_Q: return p->q;
    case NF_BUF_O: return p->o;
    case NF_BUF_H: return p->h;
    case NF_BUF_N2: return p->n2;
    case NF_BUF_A: return p->a;
    case NF_BUF_MOE_OFF: return p->moe_off;
    case NF_BUF_MOE_PERM: return p->moe_perm;
    case NF_BUF_MOE_PAIR_ROW: return p->moe_pair_row;
    case NF_BUF_MOE_PAIR_W: return p->moe_pair_w;
    default: return nullptr;
  }
}

nf_status check_shape(const nf_model_shape* s) {
  if (!s) return fail(NF_ERR_INVALID_ARG, "shape is NULL");
  if (s->hidden <= 0 || s->hidden % 16)
    return fail(NF_ERR_INVALID_ARG, "hidden must be a positive multiple of 16 (got %d)", s->hidden);
  if (s->ffn <= 0 || s->ffn % 16)
    return fail(NF_ERR_INVALID_ARG, "ffn must be a positive multiple of 16 (got %d)", s->ffn);
  if (s->head_dim != 64 && s->head_dim != 128)
    return fail(NF_ERR_INVALID_ARG, "head_dim must be 64 or 128 (got %d)", s->head_dim);
  if (s->n_kv_heads <= 0 || s->n_q_heads <= 0 || s->n_q_heads % s->n_kv_heads)
    return fail(NF_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  const int grp = s->n_q_heads / s->n_kv_heads;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 8)
    return fail(NF_ERR_INVALID_ARG, "n_q_heads / n_kv_heads must be 1, 2, 4 or 8 (got %d)", grp);
  if (s->page_size != 16) return fail(NF_ERR_INVALID_ARG, "page_size must be 16 (got %d)", s->page_size);
  if (!(s->rms_eps >= 0.f) || !(s->rope_theta > 0.f))
    return fail(NF_ERR_INVALID_ARG, "rms_eps must be >= 0 and rope_theta > 0");
  if (s->n_experts < 0 || s->n_experts > nf::GEMM_MAX_GROUPS)
    return fail(NF_ERR_INVALID_ARG, "n_experts must be in [0, %d] (got %d)", nf::GEMM_MAX_GROUPS,
                s->n_experts);
  if (s->n_experts > 0 && (s->top_k < 1 || s->top_k > 2 || s->top_k > s->n_experts))
    return fail(NF_ERR_UNSUPPORTED, "top_k must be 1 or 2 and at most n_experts (got %d)",
                s->top_k);
  return NF_OK;
}

nf_status check_opts(const nf_plan_opts* o, int T, int num_sms) {
  for (int grp = 0; grp < 2; ++grp) {
    const int n = grp ? o->n_ffn : o->n_attn;
    const int32_t* b = grp ? o->ffn_bounds : o->attn_bounds;
    if (n < 1 || n > NF_MAX_NANO)
      return fail(NF_ERR_INVALID_ARG, "nano-batch count must be 1..%d (got %d)", NF_MAX_NANO, n);
    if (b[0] != 0 || b[n] != T)
      return fail(NF_ERR_INVALID_ARG, "nano-batch bounds must run from 0 to T=%d", T);
    for (int i = 0; i < n; ++i)
      if (b[i + 1] <= b[i]) return fail(NF_ERR_INVALID_ARG, "nano-batch bounds must increase");
  }
  if (o->executor != NF_EXEC_SEQUENTIAL && o->executor != NF_EXEC_STREAMS)
    return fail(NF_ERR_INVALID_ARG, "unknown executor %d", o->executor);
  if (o->kv_chunk < 16 || o->kv_chunk > 2048 || o->kv_chunk % 16)
    return fail(NF_ERR_INVALID_ARG, "kv_chunk must be a multiple of 16 in [16, 2048]");
  if (o->attn_sms < 0 || o->attn_sms > num_sms || o->gemm_sms < 0 || o->gemm_sms > num_sms)
    return fail(NF_ERR_INVALID_ARG, "SM shares must lie in [0, %d]", num_sms);
  if (o->timeout_ns <= 0) return fail(NF_ERR_INVALID_ARG, "timeout_ns must be positive");
  const int aw = o->attn_warps;
  if (aw < 4 || (aw > 8 && aw != 10 && aw != 12 && aw != 14))
    return fail(NF_ERR_INVALID_ARG, "attn_warps must be 4 ... 8, 10, 12 or 14");
  if (o->gemm_stages < 2 || o->gemm_stages > 4)
    return fail(NF_ERR_INVALID_ARG, "gemm_stages must be 2, 3 or 4");
  if (o->gemm_split_k < 0 || o->gemm_split_k > 2)
    return fail(NF_ERR_INVALID_ARG,
                "gemm_split_k must be 0 (automatic), 1 (never) or 2 (token-row tiles only)");
  if (o->attn_impl != NF_ATTN_AUTO && o->attn_impl != NF_ATTN_MMA)
    return fail(NF_ERR_INVALID_ARG, "attn_impl must be 0 (automatic) or 2 (tensor cores)");
  return NF_OK;
}

void free_plan(nf_plan p) {
  if (!p) return;
  void* bufs[] = {p->d_q_lens, p->d_tok_begin, p->d_seg_bounds, p->tok_seq, p->tok_pos,
                  p->tok_slot, p->tok_nchunks, p->items, p->seg_items, p->fetch, p->row_done,
                  p->partials, p->status, p->n1, p->q, p->o, p->h, p->n2, p->a, p->x_stage,
                  p->y_stage, p->bt_stage, p->sl_stage, p->xa, p->xb, p->gemm_part,
                  p->gemm_cnt, p->moe_off, p->moe_perm, p->moe_pair_row, p->moe_pair_w,
                  p->moe_a, p->moe_act, p->moe_out, p->rope_cs, p->pf_tiles};
  for (void* b : bufs)
    if (b) cudaFree(b);
  if (p->set_stage) cudaFreeHost(p->set_stage);
  if (p->pf_stage) cudaFreeHost(p->pf_stage);
  for (cudaEvent_t e : p->set_ev)
    if (e) cudaEventDestroy(e);
  for (auto& h : p->hgraphs)
    if (h.exec) cudaGraphExecDestroy(h.exec);
  if (p->s_host) cudaStreamDestroy(p->s_host);
  if (p->ev_host) cudaEventDestroy(p->ev_host);
  for (int i = 0; i < 2; ++i) {
    void* pb[] = {p->pipe.x[i], p->pipe.y[i], p->pipe.bt[i], p->pipe.sl[i]};
    for (void* b : pb)
      if (b) cudaFree(b);
    cudaEvent_t pe[] = {p->pipe.in_done[i], p->pipe.step_done[i], p->pipe.out_done[i]};
    for (cudaEvent_t e : pe)
      if (e) cudaEventDestroy(e);
  }
  if (p->pipe.s_in) cudaStreamDestroy(p->pipe.s_in);
  if (p->pipe.s_out) cudaStreamDestroy(p->pipe.s_out);
  for (cudaEvent_t e : p->ev) cudaEventDestroy(e);
  for (auto& r : p->trace) {
    cudaEventDestroy(r.b);
    cudaEventDestroy(r.e);
  }
  std::vector<cudaEvent_t> s0s;
  for (auto& r : p->trace)
    if (std::find(s0s.begin(), s0s.end(), r.s0) == s0s.end()) s0s.push_back(r.s0);
  for (cudaEvent_t e : s0s) cudaEventDestroy(e);
  for (cudaEvent_t e : p->ev_pool) cudaEventDestroy(e);
  if (p->s_gemm) cudaStreamDestroy(p->s_gemm);
  if (p->s_attn) cudaStreamDestroy(p->s_attn);
  delete p;
}

template <typename T>
nf_status dalloc(T** ptr, size_t bytes) {
  if (bytes == 0) bytes = 16;
  if (cudaMalloc(reinterpret_cast<void**>(ptr), bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(NF_ERR_OOM, "cudaMalloc of %zu bytes failed", bytes);
  }
  return NF_OK;
}

#define NF_TRY(expr)                \
  do {                              \
    nf_status s_ = (expr);          \
    if (s_ != NF_OK) return s_;     \
  } while (0)

// Tiles of prefill-chunk rows for the prefill attention kernel, attention
// nano-batch by nano-batch (rows of a chunk inside the nano-batch, at most
// prefill_tile_rows of them a tile); seg[i] = first tile of nano-batch i.
// At most T tiles: they are disjoint runs of rows.
void build_prefill_tiles(const nf_plan_s* p, int n_decode, int n_seq, const std::vector<int>& tok_begin,
                         const nf_plan_opts& o, std::vector<int4>& tiles, int* seg) {
  tiles.clear();
  const int qp = nf::prefill_tile_rows(p->shape.n_q_heads, p->shape.n_kv_heads);
  for (int i = 0; i < o.n_attn; ++i) {
    seg[i] = (int)tiles.size();
    const int a = o.attn_bounds[i], b = o.attn_bounds[i + 1];
    for (int j = n_decode; j < n_seq; ++j) {
      const int lo = std::max(a, tok_begin[j]), hi = std::min(b, tok_begin[j + 1]);
      for (int r = lo; r < hi; r += qp) tiles.push_back(make_int4(r, std::min(r + qp, hi), j, 0));
    }
  }
  seg[o.n_attn] = (int)tiles.size();
}

nf_status alloc_plan(nf_plan p) {
  p->T_cap = p->T;
  p->seq_cap = p->n_seq;
  const size_t T = p->T_cap, H = p->shape.hidden, F = p->shape.ffn;
  const size_t QD = (size_t)p->shape.n_q_heads * p->shape.head_dim;
  p->max_chunks = (p->max_pages * p->shape.page_size + p->opts.kv_chunk - 1) / p->opts.kv_chunk;
  p->item_capacity = p->T_cap * p->max_chunks;
  const size_t rec = nf::attn_partial_floats(p->shape.n_q_heads, p->shape.n_kv_heads,
                                             p->shape.head_dim);
  NF_TRY(dalloc(&p->d_q_lens, p->seq_cap * 4));
  NF_TRY(dalloc(&p->d_tok_begin, (p->seq_cap + 1) * 4));
  NF_TRY(dalloc(&p->d_seg_bounds, (NF_MAX_NANO + 1) * 4));
  NF_TRY(dalloc(&p->tok_seq, T * 4));
  NF_TRY(dalloc(&p->tok_pos, T * 4));
  NF_TRY(dalloc(&p->tok_slot, T * 4));
  NF_TRY(dalloc(&p->tok_nchunks, T * 4));
  NF_TRY(dalloc(&p->items, (size_t)p->item_capacity * 8));
  NF_TRY(dalloc(&p->seg_items, (NF_MAX_NANO + 1) * 4));
  NF_TRY(dalloc(&p->fetch, NF_MAX_NANO * 4));
  NF_TRY(dalloc(&p->row_done, T * p->shape.n_kv_heads * 4));
  NF_TRY(dalloc(&p->partials, T * p->max_chunks * p->shape.n_kv_heads * rec * 4));
  NF_TRY(dalloc(&p->status, 4));
  NF_TRY(dalloc(&p->n1, T * H * 2));
  NF_TRY(dalloc(&p->q, T * QD * 2));
  NF_TRY(dalloc(&p->o, T * QD * 2));
  NF_TRY(dalloc(&p->h, T * H * 2));
  NF_TRY(dalloc(&p->n2, T * H * 2));
  NF_TRY(dalloc(&p->a, T * F * 2));
  if (p->shape.n_experts > 0) {
    const size_t R = T * p->shape.top_k;  // grouped rows: one per (token, choice)
    NF_TRY(dalloc(&p->moe_off, (nf::GEMM_MAX_GROUPS + 1) * 4));
    NF_TRY(dalloc(&p->moe_perm, R * 4));
    NF_TRY(dalloc(&p->moe_pair_row, R * 4));
    NF_TRY(dalloc(&p->moe_pair_w, R * 4));
    NF_TRY(dalloc(&p->moe_a, R * H * 2));
    NF_TRY(dalloc(&p->moe_act, R * F * 2));
    NF_TRY(dalloc(&p->moe_out, R * H * 4));
    if (!nf::make_tmap_bf16(&p->tm_moe_a, p->moe_a, R, H, 128) ||
        !nf::make_tmap_bf16(&p->tm_moe_act, p->moe_act, R, F, 128))
      return fail(NF_ERR_CUDA, "tensor map creation failed");
  }
  {  // RoPE table for every position a sequence can reach, in double precision
    const int npos = p->max_pages * p->shape.page_size, half = p->shape.head_dim / 2;
    std::vector<float> cs((size_t)npos * half * 2);
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow((double)p->shape.rope_theta, -2.0 * i / p->shape.head_dim);
      for (int pos = 0; pos < npos; ++pos) {
        const double ang = pos * inv;
        cs[((size_t)pos * half + i) * 2] = (float)std::cos(ang);
        cs[((size_t)pos * half + i) * 2 + 1] = (float)std::sin(ang);
      }
    }
    NF_TRY(dalloc(&p->rope_cs, cs.size() * 4));
    NF_CUDA(cudaMemcpy(p->rope_cs, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
  }
  NF_TRY(dalloc(&p->gemm_part, kSplitPartBytes));
  NF_TRY(dalloc(&p->gemm_cnt, kSplitMaxTiles * 4));
  NF_CUDA(cudaMemset(p->gemm_cnt, 0, kSplitMaxTiles * 4));
  NF_CUDA(cudaMemset(p->status, 0, 4));
  NF_CUDA(cudaMemcpy(p->d_q_lens, p->q_lens.data(), p->n_seq * 4, cudaMemcpyHostToDevice));
  NF_CUDA(cudaMemcpy(p->d_tok_begin, p->tok_begin.data(), (p->n_seq + 1) * 4,
                     cudaMemcpyHostToDevice));
  NF_CUDA(cudaMemcpy(p->d_seg_bounds, p->opts.attn_bounds, (p->opts.n_attn + 1) * 4,
                     cudaMemcpyHostToDevice));
  NF_TRY(dalloc(&p->pf_tiles, T * sizeof(int4)));
  {
    std::vector<int4> tiles;
    build_prefill_tiles(p, p->n_decode, p->n_seq, p->tok_begin, p->opts, tiles, p->pf_seg);
    if (!tiles.empty())
      NF_CUDA(cudaMemcpy(p->pf_tiles, tiles.data(), tiles.size() * sizeof(int4),
                         cudaMemcpyHostToDevice));
  }
  NF_CUDA(cudaStreamCreateWithFlags(&p->s_gemm, cudaStreamNonBlocking));
  NF_CUDA(cudaStreamCreateWithFlags(&p->s_attn, cudaStreamNonBlocking));
  p->ev.resize(4 + 2 * NF_MAX_NANO);  // start, done, QKV and attention per nano-batch, joins
  for (auto& e : p->ev) NF_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  const int BMr = 128;
  if (!nf::make_tmap_bf16(&p->tm_n1, p->n1, T, H, BMr) ||
      !nf::make_tmap_bf16(&p->tm_o, p->o, T, QD, BMr) ||
      !nf::make_tmap_bf16(&p->tm_n2, p->n2, T, H, BMr) ||
      !nf::make_tmap_bf16(&p->tm_a, p->a, T, F, BMr))
    return fail(NF_ERR_CUDA, "tensor map creation failed (driver entry point missing?)");
  {
    const void* xb[4] = {p->n1, p->o, p->n2, p->a};
    const uint64_t xc[4] = {H, QD, H, F};
    for (int i = 0; i < 4; ++i)
      if (!nf::make_tmap_bf16(&p->tm_x64[i], xb[i], T, xc[i], 64) ||
          !nf::make_tmap_bf16(&p->tm_x128[i], xb[i], T, xc[i], 128))
        return fail(NF_ERR_CUDA, "tensor map creation failed");
  }
  return NF_OK;
}

nf_status build_plan(const nf_model_shape* shape, const nf_batch_desc* batch,
                     const nf_plan_opts* opts, nf_plan* out) {
  if (!out) return fail(NF_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  NF_TRY(check_shape(shape));
  if (!batch) return fail(NF_ERR_INVALID_ARG, "batch is NULL");
  if (batch->n_decode < 0 || batch->n_prefill < 0 || batch->n_decode + batch->n_prefill < 1)
    return fail(NF_ERR_INVALID_ARG, "batch needs at least one sequence");
  if (batch->n_prefill > 0 && !batch->prefill_q_lens)
    return fail(NF_ERR_INVALID_ARG, "prefill_q_lens is NULL");
  if (batch->max_pages_per_seq < 1 || batch->num_pages < 1)
    return fail(NF_ERR_INVALID_ARG, "max_pages_per_seq and num_pages must be >= 1");
  const int num_sms = device_sms();
  if (num_sms <= 0) return fail(NF_ERR_CUDA, "no CUDA device");

  nf_plan p = new nf_plan_s();
  p->shape = *shape;
  p->n_decode = batch->n_decode;
  p->n_prefill = batch->n_prefill;
  p->max_pages = batch->max_pages_per_seq;
  p->num_pages = batch->num_pages;
  p->n_seq = batch->n_decode + batch->n_prefill;
  p->num_sms = num_sms;
  p->tok_begin.push_back(0);
  for (int i = 0; i < p->n_seq; ++i) {
    int q = 1;
    if (i >= batch->n_decode) {
      q = batch->prefill_q_lens[i - batch->n_decode];
      if (q < 1) {
        delete p;
        return fail(NF_ERR_INVALID_ARG, "prefill_q_lens[%d] must be >= 1", i - batch->n_decode);
      }
      p->prefill_q.push_back(q);
    }
    p->q_lens.push_back(q);
    p->tok_begin.push_back(p->tok_begin.back() + q);
  }
  p->T = p->tok_begin.back();
  if (shape->n_experts > 0 && (int64_t)p->T * shape->top_k > 16384) {
    delete p;
    return fail(NF_ERR_UNSUPPORTED, "a MoE step routes at most 16384 (token, expert) pairs");
  }
  if (batch->seq_lens_hint) p->seq_hint.assign(batch->seq_lens_hint, batch->seq_lens_hint + p->n_seq);

  if (opts) {
    p->opts = *opts;
  } else {
    double pred = 0;
    nf_status s = nf_plan_search(shape, batch, nullptr, num_sms, &p->opts, &pred);
    if (s != NF_OK) {
      delete p;
      return s;
    }
  }
  if (p->opts.kv_chunk == 0) p->opts.kv_chunk = 1024;
  if (p->opts.timeout_ns == 0) p->opts.timeout_ns = kDefaultTimeoutNs;
  if (p->opts.attn_warps == 0) p->opts.attn_warps = 8;
  if (p->opts.gemm_stages == 0) p->opts.gemm_stages = 4;
  nf_status s = check_opts(&p->opts, p->T, num_sms);
  if (s != NF_OK) {
    delete p;
    return s;
  }
  {
    const nf_model_shape& sh = p->shape;
    const bool mma_ok = nf::attention_mma_supported(sh.n_q_heads, sh.n_kv_heads, sh.head_dim,
                                                    sh.page_size, p->num_pages);
    if (!mma_ok) {
      delete p;
      return fail(NF_ERR_UNSUPPORTED, "attention: unsupported shape or pool size (page 16, "
                  "head_dim 64 or 128, n_q / n_kv in 1, 2, 4, 8)");
    }
    p->attn_mma = true;
    if (p->opts.attn_impl == NF_ATTN_AUTO) p->opts.attn_impl = NF_ATTN_MMA;  // nf_plan_info reports it
  }
  s = alloc_plan(p);
  if (s != NF_OK) {
    std::string keep = g_err;
    free_plan(p);
    g_err = keep;
    return s;
  }
  *out = p;
  return NF_OK;
}

nf_status refresh_weight_maps(nf_plan p, const nf_layer_weights* w) {
  const bool moe = p->shape.n_experts > 0;
  const void* key[4] = {w->w_qkv, w->w_o, moe ? w->w_experts_gate_up : w->w_gate_up,
                        moe ? w->w_experts_down : w->w_down};
  if (std::memcmp(key, p->wkey, sizeof(key)) == 0) return NF_OK;
  for (const auto& c : p->wcache) {
    if (std::memcmp(key, c.key, sizeof(key)) == 0) {
      p->tm_wqkv = c.qkv;
      p->tm_wo = c.o;
      p->tm_wg = c.g;
      p->tm_wu = c.u;
      p->tm_wd = c.d;
      p->tm_wo224 = c.o224;
      p->tm_wd224 = c.d224;
      p->tm_wqkv_h = c.qkv_h;
      p->tm_wo128 = c.o128;
      p->tm_wd128 = c.d128;
      std::memcpy(p->wkey, key, sizeof(key));
      return NF_OK;
    }
  }
  const nf_model_shape& s = p->shape;
  const uint64_t H = s.hidden, F = s.ffn, QD = (uint64_t)s.n_q_heads * s.head_dim;
  const uint64_t NQKV = (uint64_t)(s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim;
  if (!nf::make_tmap_bf16(&p->tm_wqkv, w->w_qkv, NQKV, H, 256) ||
      !nf::make_tmap_bf16(&p->tm_wo, w->w_o, H, QD, 256) ||
      !nf::make_tmap_bf16(&p->tm_wo224, w->w_o, H, QD, 224) ||
      !nf::make_tmap_bf16(&p->tm_wqkv_h, w->w_qkv, NQKV, H, s.head_dim / 2) ||
      !nf::make_tmap_bf16(&p->tm_wo128, w->w_o, H, QD, 128))
    return fail(NF_ERR_INVALID_ARG, "weight tensor maps: pointers must be 16-byte aligned");
  if (moe) {  // one map over every expert's rows: [E * 2F, H] and [E * H, F]
    const uint64_t E = p->shape.n_experts;
    if (!nf::make_tmap_bf16(&p->tm_wg, w->w_experts_gate_up, E * 2 * F, H, 128) ||
        !nf::make_tmap_bf16(&p->tm_wd, w->w_experts_down, E * H, F, 256))
      return fail(NF_ERR_INVALID_ARG, "expert tensor maps: pointers must be 16-byte aligned");
    p->tm_wu = p->tm_wg;
  } else {
    const char* up = static_cast<const char*>(w->w_gate_up) + F * H * 2;
    if (!nf::make_tmap_bf16(&p->tm_wg, w->w_gate_up, F, H, 128) ||
        !nf::make_tmap_bf16(&p->tm_wu, up, F, H, 128) ||
        !nf::make_tmap_bf16(&p->tm_wd, w->w_down, H, F, 256) ||
        !nf::make_tmap_bf16(&p->tm_wd224, w->w_down, H, F, 224) ||
        !nf::make_tmap_bf16(&p->tm_wd128, w->w_down, H, F, 128))
      return fail(NF_ERR_INVALID_ARG, "weight tensor maps: pointers must be 16-byte aligned");
  }
  std::memcpy(p->wkey, key, sizeof(key));
  if (p->wcache.size() < 1024) {
    nf_plan_s::WeightMaps c;
    std::memcpy(c.key, key, sizeof(key));
    c.qkv = p->tm_wqkv;
    c.o = p->tm_wo;
    c.g = p->tm_wg;
    c.u = p->tm_wu;
    c.d = p->tm_wd;
    c.o224 = p->tm_wo224;
    c.d224 = p->tm_wd224;
    c.qkv_h = p->tm_wqkv_h;
    c.o128 = p->tm_wo128;
    c.d128 = p->tm_wd128;
    p->wcache.push_back(c);
  }
  return NF_OK;
}

GemmArgs base_args(nf_plan p) {
  GemmArgs g{};
  g.stages = p->opts.gemm_stages;
  g.splits = 1;
  g.part = p->gemm_part;
  g.tile_cnt = p->gemm_cnt;
  g.status = p->status;
  g.timeout_ns = (unsigned long long)p->opts.timeout_ns;
  g.n_q = p->shape.n_q_heads;
  g.n_kv = p->shape.n_kv_heads;
  g.head_dim = p->shape.head_dim;
  g.page_size = p->shape.page_size;
  g.log2_theta = std::log2(p->shape.rope_theta);
  g.rope_cs = p->rope_cs;
  g.rope_positions = p->max_pages * p->shape.page_size;
  return g;
}

// Token-row GEMMs of the sequential executor start as programmatic dependents
// of the kernel ahead of them on the stream (the one that writes their A) and
// request their first weights before they wait for it.  The two-stream
// executor puts event waits between its GEMMs, so it launches them plainly.
int weights_first(nf_plan p) { return p->opts.executor == NF_EXEC_SEQUENTIAL ? 1 : 0; }

int cap_grid(int tiles, int cap) { return tiles < cap ? tiles : cap; }

// Output columns per tile for a residual GEMM of m_tiles row tiles and N
// columns on `grid` CTAs: 224 when that turns a partial last wave into fewer
// tile-widths of work (256 tiles on 152 SMs take 2 rounds of 256 columns; 304
// tiles of 224 columns take 2 rounds of 224), else 256.
int pick_bn(int m_tiles, int N, int grid) {
  auto work = [&](int bn) {
    const int tiles = m_tiles * ((N + bn - 1) / bn);
    return (double)((tiles + grid - 1) / grid) * bn;
  };
  if (m_tiles * ((N + 255) / 256) * 2 <= grid) return 256;  // few tiles: split-K territory
  return work(224) < work(256) ? 224 : 256;
}

// Weight-row GEMM (gemm_wrows.cu) for nano-operations of few tokens: the
// token tile, the cluster size (K splits) and the cluster count.  Measured on
// GB300: with most SMs streaming, one CTA pulls weights at about 40 GB/s (its
// share of the device's read bandwidth; alone it reaches ~110 GB/s), the
// device as a whole up to 6.4 TB/s, and each tile ends in an exchange round of
// a few microseconds.  The time of a choice is the larger of
// the per-CTA stream and the weight stream at min(HBM, CTAs x per-CTA rate),
// plus one exchange per wave of tiles.  A cluster of several CTAs waits for its
// slowest member at every tile, which measured far slower than the model when
// clusters walk several tiles, so K is split only when every tile has its own
// cluster.  Two-operand tiles (QKV, SwiGLU) with 128 tokens measured slower
// than the token-row tiles (gate/up 72 vs 64 us): they take at most 64 tokens.
constexpr int kWrMaxTokens = 128;       // larger nano-operations take token-row tiles
constexpr int kWrMaxTokensDual = 64;
constexpr double kWrSmRate = 40e9;      // weight bytes/s one CTA streams
constexpr double kWrHbm = 6.4e12;       // weight bytes/s of the device
constexpr double kWrExchange1 = 2.0e-6; // seconds of a tile's epilogue, cluster of one
constexpr double kWrExchange = 4.0e-6;  // the same with an exchange between CTAs

struct WrChoice {
  int tok = 0, splits = 0, clusters = 0;  // splits = 0: not available
};

WrChoice wr_choose(int epi, int n_tok, int w_tiles, int K, int cap, int force_splits = 0) {
  WrChoice best;
  if (n_tok < 1 || n_tok > 256 || w_tiles < 1 || cap < 1) return best;
  const int tok = n_tok <= 64 ? 64 : 128;
  const int tiles = w_tiles * ((n_tok + tok - 1) / tok);
  const int nk = (K + 63) / 64;
  const double kb_bytes = (epi == nf::EPI_SWIGLU || epi == nf::EPI_QKV ? 2.0 : 1.0) * 128 * 64 * 2;
  const double w_total = (double)w_tiles * nk * kb_bytes;  // a second token tile hits L2
  double best_t = 1e30;
  for (int sp = 1; sp <= 8 && sp <= nk; ++sp) {
    if (force_splits > 0 && sp != force_splits) continue;
    const int fit = nf::gemm_wrows_max_clusters(epi, tok, sp);
    const int cl = std::min(tiles, std::min(fit, cap / sp));
    if (cl < 1) continue;
    const int waves = (tiles + cl - 1) / cl;
    if (sp > 1 && waves > 1 && force_splits == 0) continue;
    const double per_cta = (double)waves * ((nk + sp - 1) / sp) * kb_bytes;
    const double rate = std::min(kWrHbm, (double)cl * sp * kWrSmRate);
    const double t = std::max(per_cta / kWrSmRate, w_total / rate) +
                     waves * (sp > 1 ? kWrExchange : kWrExchange1);
    if (t < best_t * 0.99) {  // ties go to the smaller cluster
      best_t = t;
      best.tok = tok;
      best.splits = sp;
      best.clusters = cl;
    }
  }
  return best;
}

enum { XM_N1 = 0, XM_O = 1, XM_N2 = 2, XM_A = 3 };
const CUtensorMap& xmap(nf_plan p, int which, int tok) {
  return tok == 64 ? p->tm_x64[which] : p->tm_x128[which];
}

// The plan lets small nano-operations take the weight-row GEMM (gemm_split_k 0).
bool use_wrows(nf_plan p, int n_tok, bool dual = false) {
  return p->opts.gemm_split_k == 0 && n_tok >= 1 &&
         n_tok <= (dual ? kWrMaxTokensDual : kWrMaxTokens);
}

// The QKV weight-row tile pairs the two halves of 256 / head_dim heads.
bool qkv_wrows_ok(const nf_model_shape& s) {
  const int d = s.head_dim;
  return d >= 16 && d <= 256 && 256 % d == 0 && (d / 2) % 8 == 0;
}


cudaEvent_t pooled_event(nf_plan p) {
  cudaEvent_t e = nullptr;
  if (!p->ev_pool.empty()) {
    e = p->ev_pool.back();
    p->ev_pool.pop_back();
  } else if (cudaEventCreate(&e) != cudaSuccess) {
    return nullptr;
  }
  return e;
}

// Begin/end markers around one nano-operation (no-ops unless tracing).
struct TraceScope {
  nf_plan p;
  cudaStream_t st;
  int op, nano;
  cudaEvent_t b = nullptr;
  TraceScope(nf_plan p_, cudaStream_t st_, int op_, int nano_) : p(p_), st(st_), op(op_), nano(nano_) {
    if (p->trace_left > 0 && p->trace_s0 && ((p->trace_ops >> op) & 1u)) {
      b = pooled_event(p);
      if (b) cudaEventRecord(b, st);
    }
  }
  ~TraceScope() {
    if (!b) return;
    cudaEvent_t e = pooled_event(p);
    if (!e) return;
    cudaEventRecord(e, st);
    p->trace.push_back({op, nano, p->trace_step, b, e, p->trace_s0});
  }
};

// after_qkv: the step's RMSNorm-1 kernels write the token map, and this
// launch (the work list only) follows the first QKV GEMM as its programmatic
// dependent, on the SMs the GEMM's last wave leaves free.
nf_status run_meta(nf_plan p, const int32_t* bt, const int32_t* sl, cudaStream_t st,
                   bool after_qkv = false) {
  TraceScope ts_(p, st, NF_OP_META, 0);
  nf::MetaArgs m{};
  m.seq_lens = sl;
  m.block_table = bt;
  m.q_lens = p->d_q_lens;
  m.tok_begin = p->d_tok_begin;
  m.seg_bounds = p->d_seg_bounds;
  m.n_seq = p->n_seq;
  m.n_tok = p->T;
  m.n_seg = p->opts.n_attn;
  m.max_pages = p->max_pages;
  m.num_pages = p->num_pages;
  m.page_size = p->shape.page_size;
  m.kv_chunk = p->opts.kv_chunk;
  m.n_kv = p->shape.n_kv_heads;
  m.max_chunks = p->max_chunks;
  m.item_capacity = p->item_capacity;
  m.tok_seq = p->tok_seq;
  m.tok_pos = p->tok_pos;
  m.tok_slot = p->tok_slot;
  m.tok_nchunks = p->tok_nchunks;
  m.items = p->items;
  m.seg_items = p->seg_items;
  m.fetch = p->fetch;
  m.row_done = p->row_done;
  m.counter_sets = p->counter_sets;
  m.fetch_stride = NF_MAX_NANO;
  m.status = p->status;
  m.validate = p->opts.validate;
  m.map_done = after_qkv ? 1 : 0;
  NF_CUDA(nf::launch_meta(m, st));
  return NF_OK;
}

// The token map that RMSNorm-1 writes for its rows (see run_meta).
nf::TokMap token_map_args(nf_plan p, const int32_t* bt, const int32_t* sl) {
  nf::TokMap m{};
  m.seq_lens = sl;
  m.q_lens = p->d_q_lens;
  m.tok_begin = p->d_tok_begin;
  m.block_table = bt;
  m.n_seq = p->n_seq;
  m.n_decode = p->n_decode;
  m.max_pages = p->max_pages;
  m.num_pages = p->num_pages;
  m.page_size = p->shape.page_size;
  m.kv_chunk = p->opts.kv_chunk;
  m.max_chunks = p->max_chunks;
  m.validate = p->opts.validate;
  m.tok_seq = p->tok_seq;
  m.tok_pos = p->tok_pos;
  m.tok_slot = p->tok_slot;
  m.tok_nchunks = p->tok_nchunks;
  m.status = p->status;
  return m;
}

// Whether this step's trace records operation `op` (its events would sit
// between the kernels).
bool op_traced(nf_plan p, int op) {
  return p->trace_left > 0 && p->trace_s0 && ((p->trace_ops >> op) & 1u);
}

// How a QKV nano-operation takes part in the step metadata.  AHEAD (two
// streams): the one-CTA metadata kernel runs between RMSNorm-1 and the GEMM,
// whose operand loads and products proceed beside it while its epilogue (RoPE
// positions, cache slots) waits for the token map.  MAP_LIST / MAP (one
// stream): RMSNorm-1 writes the token map of its rows, the GEMM follows it as
// a programmatic dependent, and after the first one the work-list kernel runs
// on the SMs the GEMM's last wave leaves free.
struct MetaIn {
  const int32_t* bt;
  const int32_t* sl;
  enum Mode {
    AHEAD,      // the metadata kernel between RMSNorm-1 and the GEMM
    MAP_LIST,   // RMSNorm-1 maps the nano-batch's tokens; the work list of
                // the step follows the GEMM as its programmatic dependent
    MAP         // RMSNorm-1 maps the nano-batch's tokens
  } mode;
};

// The metadata goes inside the first QKV unless the trace records either
// operation (each keeps its own interval then).
bool fold_meta(nf_plan p) { return !op_traced(p, NF_OP_META) && !op_traced(p, NF_OP_QKV); }

// early: the kernel ahead on `st` is this nano-batch's QKV GEMM and the work
// list and token map are older; the decode kernel (when no prefill tiles go
// first) then starts as the GEMM's programmatic dependent and requests the K/V
// pages that the GEMM does not write before it waits for it.
nf_status run_attention(nf_plan p, int seg, const void* q, const void* kp, const void* vp,
                        const int32_t* bt, void* o, int grid, cudaStream_t st,
                        bool early = false) {
  TraceScope ts_(p, st, NF_OP_ATTN, seg);
  nf::AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_pool = static_cast<const __nv_bfloat16*>(kp);
  a.v_pool = static_cast<const __nv_bfloat16*>(vp);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.block_table = bt;
  a.tok_seq = p->tok_seq;
  a.tok_pos = p->tok_pos;
  a.tok_nchunks = p->tok_nchunks;
  a.items = p->items;
  a.seg_items = p->seg_items;
  a.fetch = p->fetch + (size_t)p->cur_set * NF_MAX_NANO;
  a.row_done = p->row_done + (size_t)p->cur_set * p->T * p->shape.n_kv_heads;
  a.partials = p->partials;
  a.seg = seg;
  a.n_q = p->shape.n_q_heads;
  a.n_kv = p->shape.n_kv_heads;
  a.head_dim = p->shape.head_dim;
  a.page_size = p->shape.page_size;
  a.max_pages = p->max_pages;
  a.num_pages = p->num_pages;
  a.kv_chunk = p->opts.kv_chunk;
  a.max_chunks = p->max_chunks;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->shape.head_dim));
  a.warps = p->opts.attn_warps;
  a.prefill_elsewhere = p->attn_mma && p->n_prefill > 0;
  a.n_decode_seqs = p->n_decode;
  a.status = p->status;
  a.timeout_ns = (unsigned long long)p->opts.timeout_ns;
  if (p->attn_mma) {
    const nf_plan_s::PoolMaps* pm = nullptr;
    for (const auto& c : p->pcache)
      if (c.k == kp && c.v == vp) pm = &c;
    if (!pm) {
      nf_plan_s::PoolMaps c{};
      c.k = kp;
      c.v = vp;
      const nf_model_shape& sh = p->shape;
      if (!nf::make_pool_tmap_groups(&c.tk, kp, p->num_pages, sh.n_kv_heads, sh.page_size,
                                     sh.head_dim) ||
          !nf::make_pool_tmap_groups(&c.tv, vp, p->num_pages, sh.n_kv_heads, sh.page_size,
                                     sh.head_dim) ||
          !nf::make_pool_tmap_pages(&c.dk, kp, p->num_pages, sh.n_kv_heads, sh.page_size,
                                    sh.head_dim) ||
          !nf::make_pool_tmap_pages(&c.dv, vp, p->num_pages, sh.n_kv_heads, sh.page_size,
                                    sh.head_dim))
        return fail(NF_ERR_INVALID_ARG, "KV pool tensor maps: pools must be 16-byte aligned");
      if (p->pcache.size() >= 4096) p->pcache.clear();
      p->pcache.push_back(c);
      pm = &p->pcache.back();
    }
    // the prefill tiles first; the decode kernel then starts, as their
    // programmatic dependent, on the SMs they leave free
    const int n_pf = a.prefill_elsewhere ? p->pf_seg[seg + 1] - p->pf_seg[seg] : 0;
    if (n_pf > 0)
      NF_CUDA(nf::launch_attention_prefill(a, pm->tk, pm->tv, p->pf_tiles + p->pf_seg[seg], n_pf, st));
    a.early = early && n_pf == 0 ? 1 : 0;
    NF_CUDA(nf::launch_attention_mma(a, pm->dk, pm->dv, grid, n_pf > 0 || a.early, st));
  }
  return NF_OK;
}

// On an early return from a two-stream schedule, orders the caller's stream
// after whatever the side streams already hold, so that no later work on it
// overtakes them (the normal end joins through the GEMM stream, which has
// waited for the last attention).
struct SideStreamJoin {
  nf_plan p;
  cudaStream_t st;
  bool done = false;
  ~SideStreamJoin() {
    if (done) return;
    cudaEvent_t eg = p->ev[2 + 2 * NF_MAX_NANO], ea = p->ev[3 + 2 * NF_MAX_NANO];
    if (cudaEventRecord(eg, p->s_gemm) == cudaSuccess) cudaStreamWaitEvent(st, eg, 0);
    if (cudaEventRecord(ea, p->s_attn) == cudaSuccess) cudaStreamWaitEvent(st, ea, 0);
  }
};

// One nano-operation of the layer; which = 0 QKV, 1 O, 2 RMSNorm-2 + gate/up + down.
// token_rows (optional, out): whether the GEMM ran the token-row kernel.
nf_status run_qkv(nf_plan p, const nf_layer_weights* w, const void* x, void* kp, void* vp, int r0,
                  int r1, int grid, cudaStream_t st, int nano = 0, const MetaIn* meta = nullptr,
                  bool* token_rows = nullptr) {
  if (token_rows) *token_rows = false;
  TraceScope ts_(p, st, NF_OP_QKV, nano);
  const nf_model_shape& s = p->shape;
  const bool map_in_norm = meta && meta->mode != MetaIn::AHEAD;
  const bool meta_ahead = meta && meta->mode == MetaIn::AHEAD;
  const nf::TokMap tm = map_in_norm ? token_map_args(p, meta->bt, meta->sl) : nf::TokMap{};
  NF_CUDA(nf::launch_rmsnorm(static_cast<const __nv_bfloat16*>(x),
                             static_cast<const __nv_bfloat16*>(w->norm1), p->n1, r0, r1, s.hidden,
                             s.rms_eps, st, map_in_norm ? &tm : nullptr));
  // Metadata between the norm and the GEMM: the weight-row kernel waits for it
  // in all its warps (after its weight prefetch), the token-row kernel only in
  // its epilogue.
  if (meta_ahead) NF_TRY(run_meta(p, meta->bt, meta->sl, st));
  // The step's work list right after the GEMM, on the SMs its last wave
  // leaves free; the attention that follows waits for both.
  struct ListAfter {
    nf_plan p;
    const MetaIn* m;
    cudaStream_t st;
    nf_status go() const {
      return m && m->mode == MetaIn::MAP_LIST ? run_meta(p, m->bt, m->sl, st, true) : NF_OK;
    }
  } const list_after{p, meta, st};
  GemmArgs g = base_args(p);
  g.wait_prior = meta_ahead ? 1 : 0;
  g.weights_first = meta_ahead ? 0 : weights_first(p);
  g.m_begin = r0;
  g.m_end = r1;
  g.N = (s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim;
  g.K = s.hidden;
  g.m_tiles = (r1 - r0 + 127) / 128;
  g.n_tiles = (g.N + 255) / 256;
  g.tok_pos = p->tok_pos;
  g.tok_slot = p->tok_slot;
  g.q_out = p->q;
  g.k_pool = static_cast<__nv_bfloat16*>(kp);
  g.v_pool = static_cast<__nv_bfloat16*>(vp);
  if (use_wrows(p, r1 - r0, true) && qkv_wrows_ok(s)) {
    const int hp = 256 / s.head_dim;
    const int w_tiles = (s.n_q_heads + 2 * s.n_kv_heads + hp - 1) / hp;
    const WrChoice c = wr_choose(nf::EPI_QKV, r1 - r0, w_tiles, g.K, grid);
    if (c.splits) {
      g.n_tiles = w_tiles;
      g.m_tiles = (r1 - r0 + c.tok - 1) / c.tok;
      g.splits = c.splits;
      NF_CUDA(nf::launch_gemm_wrows(nf::EPI_QKV, c.tok, p->tm_wqkv_h, p->tm_wqkv_h,
                                    xmap(p, XM_N1, c.tok), g, c.clusters, true, st));
      return list_after.go();
    }
  }
  g.splits = p->opts.gemm_split_k == 1 ? 1 : choose_splits(g.m_tiles * g.n_tiles, g.K, grid);
  NF_CUDA(nf::launch_gemm(nf::EPI_QKV, p->tm_n1, p->tm_wqkv, p->tm_wqkv, g,
                          cap_grid(g.m_tiles * g.n_tiles * g.splits, grid), st));
  if (token_rows) *token_rows = true;
  return list_after.go();
}

nf_status run_oproj(nf_plan p, const void* x, int r0, int r1, int grid, cudaStream_t st,
                    int nano = 0) {
  TraceScope ts_(p, st, NF_OP_OPROJ, nano);
  const nf_model_shape& s = p->shape;
  GemmArgs g = base_args(p);
  g.m_begin = r0;
  g.m_end = r1;
  g.N = s.hidden;
  g.K = s.n_q_heads * s.head_dim;
  g.m_tiles = (r1 - r0 + 127) / 128;
  g.n_tiles = (g.N + 255) / 256;
  g.C = p->h;
  g.ldc = s.hidden;
  g.R = static_cast<const __nv_bfloat16*>(x);
  g.ldr = s.hidden;
  if (use_wrows(p, r1 - r0)) {
    const int w_tiles = (g.N + 127) / 128;
    const WrChoice c = wr_choose(nf::EPI_RESID, r1 - r0, w_tiles, g.K, grid);
    if (c.splits) {
      g.n_tiles = w_tiles;
      g.m_tiles = (r1 - r0 + c.tok - 1) / c.tok;
      g.splits = c.splits;
      NF_CUDA(nf::launch_gemm_wrows(nf::EPI_RESID, c.tok, p->tm_wo128, p->tm_wo128,
                                    xmap(p, XM_O, c.tok), g, c.clusters, true, st));
      return NF_OK;
    }
  }
  g.bn = pick_bn(g.m_tiles, g.N, grid);
  g.n_tiles = (g.N + g.bn - 1) / g.bn;
  g.splits = p->opts.gemm_split_k == 1 ? 1 : choose_splits(g.m_tiles * g.n_tiles, g.K, grid);
  g.weights_first = weights_first(p);
  const CUtensorMap& wo = g.bn == 224 ? p->tm_wo224 : p->tm_wo;
  NF_CUDA(nf::launch_gemm(nf::EPI_RESID, p->tm_o, wo, wo, g,
                          cap_grid(g.m_tiles * g.n_tiles * g.splits, grid), st));
  return NF_OK;
}

// Mixture-of-experts FFN of the tokens [r0, r1): route, gather n2 into the
// expert-grouped order, grouped gate/up GEMM with SwiGLU, grouped down GEMM to
// fp32 rows, and the weighted combine with the residual.
nf_status run_moe_ffn(nf_plan p, const nf_layer_weights* w, void* y, int r0, int r1, int grid,
                      cudaStream_t st) {
  const nf_model_shape& s = p->shape;
  const int n = r1 - r0, k = s.top_k, E = s.n_experts;
  NF_CUDA(nf::launch_moe_route(static_cast<const float*>(w->router_logits), r0, n, E, k,
                               p->moe_off, p->moe_perm, p->moe_pair_row, p->moe_pair_w, st));
  NF_CUDA(nf::launch_gather_rows(p->n2, p->moe_perm, p->moe_a, n * k, s.hidden, p->T, p->status,
                                 st));
  GemmArgs g = base_args(p);
  g.N = s.ffn;
  g.K = s.hidden;
  g.n_tiles = (g.N + 127) / 128;
  g.C = p->moe_act;
  g.ldc = s.ffn;
  g.group_off = p->moe_off;
  g.n_groups = E;
  g.b_group_rows = 2 * s.ffn;
  g.b2_row_off = s.ffn;
  g.splits = 1;
  NF_CUDA(nf::launch_gemm(nf::EPI_SWIGLU, p->tm_moe_a, p->tm_wg, p->tm_wg, g, grid, st));
  GemmArgs d = base_args(p);
  d.N = s.hidden;
  d.K = s.ffn;
  d.n_tiles = (d.N + 255) / 256;
  d.Cf = p->moe_out;
  d.ldc = s.hidden;
  d.group_off = p->moe_off;
  d.n_groups = E;
  d.b_group_rows = s.hidden;
  d.splits = 1;
  NF_CUDA(nf::launch_gemm(nf::EPI_STORE_F32, p->tm_moe_act, p->tm_wd, p->tm_wd, d, grid, st));
  NF_CUDA(nf::launch_moe_combine(p->h, p->moe_out, p->moe_pair_row, p->moe_pair_w,
                                 static_cast<__nv_bfloat16*>(y), r0, n, k, s.hidden, st));
  return NF_OK;
}

nf_status run_ffn(nf_plan p, const nf_layer_weights* w, void* y, int r0, int r1, int grid,
                  cudaStream_t st, int nano = 0) {
  TraceScope ts_(p, st, NF_OP_FFN, nano);
  const nf_model_shape& s = p->shape;
  NF_CUDA(nf::launch_rmsnorm(p->h, static_cast<const __nv_bfloat16*>(w->norm2), p->n2, r0, r1,
                             s.hidden, s.rms_eps, st));
  if (s.n_experts > 0) return run_moe_ffn(p, w, y, r0, r1, grid, st);
  GemmArgs g = base_args(p);
  g.m_begin = r0;
  g.m_end = r1;
  g.N = s.ffn;
  g.K = s.hidden;
  g.m_tiles = (r1 - r0 + 127) / 128;
  g.n_tiles = (g.N + 127) / 128;
  g.C = p->a;
  g.ldc = s.ffn;
  const bool wr = use_wrows(p, r1 - r0);
  WrChoice c;
  if (use_wrows(p, r1 - r0, true)) c = wr_choose(nf::EPI_SWIGLU, r1 - r0, (g.N + 127) / 128, g.K, grid);
  if (c.splits) {
    g.n_tiles = (g.N + 127) / 128;
    g.m_tiles = (r1 - r0 + c.tok - 1) / c.tok;
    g.splits = c.splits;
    g.b2_row_off = 0;  // tm_wu starts at the up rows
    NF_CUDA(nf::launch_gemm_wrows(nf::EPI_SWIGLU, c.tok, p->tm_wg, p->tm_wu,
                                  xmap(p, XM_N2, c.tok), g, c.clusters, true, st));
  } else {
    g.splits = p->opts.gemm_split_k == 1 ? 1 : choose_splits(g.m_tiles * g.n_tiles, g.K, grid);
    g.weights_first = weights_first(p);
    NF_CUDA(nf::launch_gemm(nf::EPI_SWIGLU, p->tm_n2, p->tm_wg, p->tm_wu, g,
                            cap_grid(g.m_tiles * g.n_tiles * g.splits, grid), st));
  }
  GemmArgs d = base_args(p);
  d.m_begin = r0;
  d.m_end = r1;
  d.N = s.hidden;
  d.K = s.ffn;
  d.m_tiles = (r1 - r0 + 127) / 128;
  d.n_tiles = (d.N + 255) / 256;
  d.C = static_cast<__nv_bfloat16*>(y);
  d.ldc = s.hidden;
  d.R = p->h;
  d.ldr = s.hidden;
  if (wr) {
    const int w_tiles = (d.N + 127) / 128;
    const WrChoice cd = wr_choose(nf::EPI_RESID, r1 - r0, w_tiles, d.K, grid);
    if (cd.splits) {
      d.n_tiles = w_tiles;
      d.m_tiles = (r1 - r0 + cd.tok - 1) / cd.tok;
      d.splits = cd.splits;
      NF_CUDA(nf::launch_gemm_wrows(nf::EPI_RESID, cd.tok, p->tm_wd128, p->tm_wd128,
                                    xmap(p, XM_A, cd.tok), d, cd.clusters, true, st));
      return NF_OK;
    }
  }
  d.bn = pick_bn(d.m_tiles, d.N, grid);
  d.n_tiles = (d.N + d.bn - 1) / d.bn;
  d.splits = p->opts.gemm_split_k == 1 ? 1 : choose_splits(d.m_tiles * d.n_tiles, d.K, grid);
  d.weights_first = weights_first(p);
  const CUtensorMap& wd = d.bn == 224 ? p->tm_wd224 : p->tm_wd;
  NF_CUDA(nf::launch_gemm(nf::EPI_RESID, p->tm_a, wd, wd, d,
                          cap_grid(d.m_tiles * d.n_tiles * d.splits, grid), st));
  return NF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

nf_status check_step_args(nf_plan p, const nf_layer_weights* w, const void* x, void* kp, void* vp,
                          const int32_t* bt, const int32_t* sl, void* y) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (!w || !w->norm1 || !w->norm2 || !w->w_qkv || !w->w_o)
    return fail(NF_ERR_INVALID_ARG, "a weight pointer is NULL");
  if (p->shape.n_experts > 0) {
    if (!w->w_experts_gate_up || !w->w_experts_down || !w->router_logits)
      return fail(NF_ERR_INVALID_ARG, "a MoE layer needs expert weights and router logits");
    if (!aligned16(w->w_experts_gate_up) || !aligned16(w->w_experts_down))
      return fail(NF_ERR_INVALID_ARG, "expert weights must be 16-byte aligned");
  } else if (!w->w_gate_up || !w->w_down) {
    return fail(NF_ERR_INVALID_ARG, "a weight pointer is NULL");
  }
  if (!x || !y || !kp || !vp || !bt || !sl) return fail(NF_ERR_INVALID_ARG, "a pointer is NULL");
  if (x == y) return fail(NF_ERR_INVALID_ARG, "x and y must not alias");
  const bool moe = p->shape.n_experts > 0;
  const void* ptrs[] = {x, y, kp, vp, w->norm1, w->norm2, w->w_qkv, w->w_o,
                        moe ? w->w_experts_gate_up : w->w_gate_up,
                        moe ? w->w_experts_down : w->w_down};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(NF_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  return NF_OK;
}

// One layer.  with_meta: run the metadata kernel first (a stack runs it once
// per step and then gives each layer its own counter set, p->cur_set).
nf_status layer_step(nf_plan p, const nf_layer_weights* w, const void* x, void* kp, void* vp,
                     const int32_t* bt, const int32_t* sl, void* y, cudaStream_t st,
                     bool with_meta = true) {
  NF_TRY(refresh_weight_maps(p, w));
  if (p->trace_left > 0) {
    p->trace_s0 = pooled_event(p);
    if (p->trace_s0) cudaEventRecord(p->trace_s0, st);
  }
  struct StepEnd {
    nf_plan p;
    ~StepEnd() {
      if (p->trace_left > 0 && p->trace_s0) {
        --p->trace_left;
        ++p->trace_step;
      }
      p->trace_s0 = nullptr;
    }
  } step_end_{p};
  const nf_plan_opts& o = p->opts;
  const int all = p->num_sms;
  const bool fold = with_meta && fold_meta(p);
  if (o.executor == NF_EXEC_SEQUENTIAL) {
    // One stream: RMSNorm-1 of each nano-batch maps its tokens, and the work
    // list is built beside the first QKV GEMM.
    if (with_meta && !fold) NF_TRY(run_meta(p, bt, sl, st));
    const MetaIn first{bt, sl, MetaIn::MAP_LIST}, rest{bt, sl, MetaIn::MAP};
    for (int i = 0; i < o.n_attn; ++i) {
      const int r0 = o.attn_bounds[i], r1 = o.attn_bounds[i + 1];
      bool token_rows = false;
      NF_TRY(run_qkv(p, w, x, kp, vp, r0, r1, all, st, i,
                     !fold ? nullptr : i == 0 ? &first : &rest, &token_rows));
      // The attention starts early behind a token-row QKV GEMM (not right
      // after the work-list kernel).  Behind the weight-row kernel it measured
      // slower (the 64-row decode stack 4.87 -> 5.31 ms; the cause is not
      // known), so there it waits for the GEMM as before.
      NF_TRY(run_attention(p, i, p->q, kp, vp, bt, p->o, all, st,
                           token_rows && !(fold && i == 0)));
      NF_TRY(run_oproj(p, x, r0, r1, all, st, i));
    }
    for (int j = 0; j < o.n_ffn; ++j)
      NF_TRY(run_ffn(p, w, y, o.ffn_bounds[j], o.ffn_bounds[j + 1], all, st, j));
    return NF_OK;
  }
  // Two streams: GEMM-class nano-operations on s_gemm, attention on s_attn,
  // ordered by events on the token-range dependencies.
  const int n = o.n_attn;
  const int attn_grid = (n == 1) ? all : (o.attn_sms > 0 ? o.attn_sms : (all * 5) / 8);
  const int gemm_overlap = o.gemm_sms > 0 ? o.gemm_sms : (all - attn_grid > 0 ? all - attn_grid : all);
  cudaEvent_t ev_start = p->ev[0], ev_done = p->ev[1];
  cudaEvent_t* ev_q = &p->ev[2];
  cudaEvent_t* ev_a = &p->ev[2 + NF_MAX_NANO];
  NF_CUDA(cudaEventRecord(ev_start, st));
  NF_CUDA(cudaStreamWaitEvent(p->s_gemm, ev_start, 0));
  NF_CUDA(cudaStreamWaitEvent(p->s_attn, ev_start, 0));
  SideStreamJoin join_{p, st};
  if (with_meta && !fold) NF_TRY(run_meta(p, bt, sl, p->s_gemm));
  const MetaIn mi{bt, sl, MetaIn::AHEAD};
  for (int i = 0; i < n; ++i) {
    NF_TRY(run_qkv(p, w, x, kp, vp, o.attn_bounds[i], o.attn_bounds[i + 1],
                   i == 0 ? all : gemm_overlap, p->s_gemm, i, i == 0 && fold ? &mi : nullptr));
    NF_CUDA(cudaEventRecord(ev_q[i], p->s_gemm));
  }
  for (int i = 0; i < n; ++i) {
    NF_CUDA(cudaStreamWaitEvent(p->s_attn, ev_q[i], 0));
    NF_TRY(run_attention(p, i, p->q, kp, vp, bt, p->o, attn_grid, p->s_attn));
    NF_CUDA(cudaEventRecord(ev_a[i], p->s_attn));
  }
  int next_ffn = 0;
  for (int i = 0; i < n; ++i) {
    NF_CUDA(cudaStreamWaitEvent(p->s_gemm, ev_a[i], 0));
    const int grid = (i == n - 1) ? all : gemm_overlap;
    NF_TRY(run_oproj(p, x, o.attn_bounds[i], o.attn_bounds[i + 1], grid, p->s_gemm, i));
    while (next_ffn < o.n_ffn && o.ffn_bounds[next_ffn + 1] <= o.attn_bounds[i + 1]) {
      NF_TRY(run_ffn(p, w, y, o.ffn_bounds[next_ffn], o.ffn_bounds[next_ffn + 1], grid,
                     p->s_gemm, next_ffn));
      ++next_ffn;
    }
  }
  NF_CUDA(cudaEventRecord(ev_done, p->s_gemm));
  NF_CUDA(cudaStreamWaitEvent(st, ev_done, 0));
  join_.done = true;
  return NF_OK;
}

}  // namespace

nf_status nf::attention_on(nf_plan p, const void* q, const void* kp, const void* vp,
                           const int32_t* bt, const int32_t* sl, void* o, int grid,
                           cudaStream_t st) {
  NF_TRY(run_meta(p, bt, sl, st));
  for (int i = 0; i < p->opts.n_attn; ++i) NF_TRY(run_attention(p, i, q, kp, vp, bt, o, grid, st));
  return NF_OK;
}

nf_status nf::set_last_error(nf_status code, const char* msg) {
  g_err = msg ? msg : "";
  return code;
}

// ============================================================== C ABI
extern "C" {

const char* nf_last_error(void) { return g_err.c_str(); }

int32_t nf_device_sm_count(void) { return device_sms(); }

nf_status nf_plan_create(const nf_model_shape* shape, const nf_batch_desc* batch,
                         const nf_plan_opts* opts, nf_plan* out) {
  g_err.clear();
  return build_plan(shape, batch, opts, out);
}

nf_status nf_plan_info(nf_plan plan, nf_plan_opts* out, int32_t* n_tokens) {
  if (!plan) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (out) *out = plan->opts;
  if (n_tokens) *n_tokens = plan->T;
  return NF_OK;
}

void nf_plan_destroy(nf_plan plan) { free_plan(plan); }

nf_status nf_plan_save(nf_plan p, const char* path) {
  if (!p || !path) return fail(NF_ERR_INVALID_ARG, "plan or path is NULL");
  FILE* f = std::fopen(path, "w");
  if (!f) return fail(NF_ERR_INVALID_ARG, "cannot open %s", path);
  const nf_model_shape& s = p->shape;
  std::fprintf(f, "nanoflow-plan 2\n");
  std::fprintf(f, "shape %d %d %d %d %d %d %.9g %.9g\n", s.hidden, s.n_q_heads, s.n_kv_heads,
               s.head_dim, s.ffn, s.page_size, s.rms_eps, s.rope_theta);
  std::fprintf(f, "batch %d %d %d %d\n", p->n_decode, p->n_prefill, p->max_pages, p->num_pages);
  std::fprintf(f, "prefill");
  for (int q : p->prefill_q) std::fprintf(f, " %d", q);
  std::fprintf(f, "\n");
  const nf_plan_opts& o = p->opts;
  std::fprintf(f, "attn %d", o.n_attn);
  for (int i = 0; i <= o.n_attn; ++i) std::fprintf(f, " %d", o.attn_bounds[i]);
  std::fprintf(f, "\nffn %d", o.n_ffn);
  for (int i = 0; i <= o.n_ffn; ++i) std::fprintf(f, " %d", o.ffn_bounds[i]);
  std::fprintf(f, "\nexec %d %d %d %d %d %lld %d %d %d %d\n", o.executor, o.attn_sms,
               o.gemm_sms, o.kv_chunk, o.validate, (long long)o.timeout_ns, o.attn_warps,
               o.gemm_stages, o.gemm_split_k, o.attn_impl);
  std::fclose(f);
  return NF_OK;
}

nf_status nf_plan_load(const char* path, nf_plan* out) {
  if (!path || !out) return fail(NF_ERR_INVALID_ARG, "path or out is NULL");
  FILE* f = std::fopen(path, "r");
  if (!f) return fail(NF_ERR_INVALID_ARG, "cannot open %s", path);
  nf_model_shape s{};
  nf_plan_opts o{};
  int nd = 0, np = 0, mp = 0, npg = 0, ver = 0;
  long long tmo = 0;
  std::vector<int> pq;
  bool ok = std::fscanf(f, " nanoflow-plan %d", &ver) == 1 && ver == 2;
  ok = ok && std::fscanf(f, " shape %d %d %d %d %d %d %f %f", &s.hidden, &s.n_q_heads,
                         &s.n_kv_heads, &s.head_dim, &s.ffn, &s.page_size, &s.rms_eps,
                         &s.rope_theta) == 8;
  ok = ok && std::fscanf(f, " batch %d %d %d %d", &nd, &np, &mp, &npg) == 4;
  ok = ok && std::fscanf(f, " prefill") == 0;
  for (int i = 0; ok && i < np; ++i) {
    int q = 0;
    ok = std::fscanf(f, " %d", &q) == 1;
    pq.push_back(q);
  }
  ok = ok && std::fscanf(f, " attn %d", &o.n_attn) == 1 && o.n_attn >= 1 && o.n_attn <= NF_MAX_NANO;
  for (int i = 0; ok && i <= o.n_attn; ++i) ok = std::fscanf(f, " %d", &o.attn_bounds[i]) == 1;
  ok = ok && std::fscanf(f, " ffn %d", &o.n_ffn) == 1 && o.n_ffn >= 1 && o.n_ffn <= NF_MAX_NANO;
  for (int i = 0; ok && i <= o.n_ffn; ++i) ok = std::fscanf(f, " %d", &o.ffn_bounds[i]) == 1;
  ok = ok && std::fscanf(f, " exec %d %d %d %d %d %lld %d %d %d %d", &o.executor, &o.attn_sms,
                         &o.gemm_sms, &o.kv_chunk, &o.validate, &tmo, &o.attn_warps,
                         &o.gemm_stages, &o.gemm_split_k, &o.attn_impl) == 10;
  std::fclose(f);
  if (!ok) return fail(NF_ERR_INVALID_ARG, "%s is not a plan file", path);
  o.timeout_ns = tmo;
  nf_batch_desc b{};
  b.n_decode = nd;
  b.n_prefill = np;
  b.prefill_q_lens = pq.data();
  b.max_pages_per_seq = mp;
  b.num_pages = npg;
  return nf_plan_create(&s, &b, &o, out);
}

nf_status nf_layer_step(nf_plan plan, const nf_layer_weights* w, const void* x, void* k_pool,
                        void* v_pool, const int32_t* block_table, const int32_t* seq_lens, void* y,
                        void* stream) {
  NF_TRY(check_step_args(plan, w, x, k_pool, v_pool, block_table, seq_lens, y));
  return layer_step(plan, w, x, k_pool, v_pool, block_table, seq_lens, y,
                    static_cast<cudaStream_t>(stream));
}

namespace {
// Activation buffers and one split-KV counter set per layer for a run of
// n_layers layers (allocates, and synchronizes the device, only when it grows).
nf_status ensure_layers(nf_plan p, int n_layers) {
  const size_t xb = (size_t)p->T_cap * p->shape.hidden * 2;
  if (!p->xa) {
    NF_TRY(dalloc(&p->xa, xb));
    NF_TRY(dalloc(&p->xb, xb));
  }
  if (p->counter_sets < n_layers) {
    NF_CUDA(cudaDeviceSynchronize());
    cudaFree(p->fetch);
    cudaFree(p->row_done);
    p->fetch = nullptr;
    p->row_done = nullptr;
    NF_TRY(dalloc(&p->fetch, (size_t)NF_MAX_NANO * n_layers * 4));
    NF_TRY(dalloc(&p->row_done, (size_t)p->T_cap * p->shape.n_kv_heads * n_layers * 4));
    p->counter_sets = n_layers;
  }
  return NF_OK;
}

// Whether run_layers pipelines nano-batches across layers: the two-stream
// executor with at least two attention nano-batches.
bool cross_layer(nf_plan p, int n_layers) {
  const nf_plan_opts& o = p->opts;
  return o.executor == NF_EXEC_STREAMS && o.n_attn >= 2 && n_layers >= 2;
}

// The two-stream executor over several layers with no join between layers
// (the pages' cross-layer window, "Auto-Search Stage I": the pipeline search
// spans neighbouring layers): attention nano-batch i of layer l + 1 starts
// its QKV projection on the GEMM stream as soon as the FFN nano-batches of
// layer l that cover its rows are done, so its attention runs beside the
// GEMMs of the other nano-batches of layer l instead of waiting for the whole
// layer.  Order on the streams (FFN nano-batch j runs after the O projection
// that completes its rows, as in one layer):
//   GEMM:      QKV(0, 0..n-1) | O(l, i), FFN(l, j) ..., QKV(l+1, k) ... for l, then i
//   attention: A(0, 0..n-1)   | A(l+1, k) after QKV(l+1, k)
// Every buffer the plan shares between layers (n1, q, o, h, n2, a, the split-K
// and split-KV workspaces) is either written and read on one stream in that
// order, or touched on both streams only in rows of different nano-batches;
// the K/V that the attention of nano-batch i reads were appended by the QKV
// projections of nano-batches <= i of its layer, which precede it on the GEMM
// stream.
nf_status run_layers_pipelined(nf_plan p, const nf_layer_weights* layers, int n_layers,
                               const std::vector<const void*>& act, void* const* k_pools,
                               void* const* v_pools, const int32_t* bt, const int32_t* sl,
                               cudaStream_t st) {
  const nf_plan_opts& o = p->opts;
  const int n = o.n_attn, all = p->num_sms;
  const int attn_grid = o.attn_sms > 0 ? o.attn_sms : (all * 5) / 8;
  const int gsm = o.gemm_sms > 0 ? o.gemm_sms : (all - attn_grid > 0 ? all - attn_grid : all);
  struct Reset {
    nf_plan p;
    ~Reset() { p->cur_set = 0; }
  } reset_{p};
  // a traced window is one traced step: every layer's nano-operations, timed
  // from the step's start on the caller's stream
  if (p->trace_left > 0) {
    p->trace_s0 = pooled_event(p);
    if (p->trace_s0) cudaEventRecord(p->trace_s0, st);
  }
  struct StepEnd {
    nf_plan p;
    ~StepEnd() {
      if (p->trace_left > 0 && p->trace_s0) {
        --p->trace_left;
        ++p->trace_step;
      }
      p->trace_s0 = nullptr;
    }
  } step_end_{p};
  cudaEvent_t ev_start = p->ev[0], ev_done = p->ev[1];
  cudaEvent_t* ev_q = &p->ev[2];
  cudaEvent_t* ev_a = &p->ev[2 + NF_MAX_NANO];
  NF_CUDA(cudaEventRecord(ev_start, st));
  NF_CUDA(cudaStreamWaitEvent(p->s_gemm, ev_start, 0));
  NF_CUDA(cudaStreamWaitEvent(p->s_attn, ev_start, 0));
  SideStreamJoin join_{p, st};
  // the GEMM stream's order (schedule.h, also what the plan search simulates);
  // it opens with the QKV of layer 0's first nano-batch, which takes the metadata
  const std::vector<nf::WindowOp> sched = nf::window_schedule(o, n_layers);
  const bool fold = fold_meta(p) && !sched.empty() && sched[0].kind == nf::WOP_QKV &&
                    sched[0].layer == 0 && sched[0].nano == 0;
  const MetaIn mi{bt, sl, MetaIn::AHEAD};
  if (!fold) NF_TRY(run_meta(p, bt, sl, p->s_gemm));
  // QKV of nano-batch i of layer l on the GEMM stream, its attention on the other
  auto front = [&](int l, int i, int grid) -> nf_status {
    const nf_layer_weights* w = &layers[l];
    NF_TRY(refresh_weight_maps(p, w));
    NF_TRY(run_qkv(p, w, act[l], k_pools[l], v_pools[l], o.attn_bounds[i], o.attn_bounds[i + 1],
                   grid, p->s_gemm, i, fold && l == 0 && i == 0 ? &mi : nullptr));
    NF_CUDA(cudaEventRecord(ev_q[i], p->s_gemm));
    NF_CUDA(cudaStreamWaitEvent(p->s_attn, ev_q[i], 0));
    p->cur_set = l;
    NF_TRY(run_attention(p, i, p->q, k_pools[l], v_pools[l], bt, p->o, attn_grid, p->s_attn));
    NF_CUDA(cudaEventRecord(ev_a[i], p->s_attn));
    return NF_OK;
  };
  for (const nf::WindowOp& op : sched) {
    const int grid = op.full ? all : gsm;
    const int l = op.layer, i = op.nano;
    if (op.kind == nf::WOP_QKV) {
      NF_TRY(front(l, i, grid));
    } else if (op.kind == nf::WOP_O) {
      NF_CUDA(cudaStreamWaitEvent(p->s_gemm, ev_a[i], 0));  // attention i of layer l
      NF_TRY(refresh_weight_maps(p, &layers[l]));
      NF_TRY(run_oproj(p, act[l], o.attn_bounds[i], o.attn_bounds[i + 1], grid, p->s_gemm, i));
    } else {
      NF_TRY(refresh_weight_maps(p, &layers[l]));
      NF_TRY(run_ffn(p, &layers[l], const_cast<void*>(act[l + 1]), o.ffn_bounds[i],
                     o.ffn_bounds[i + 1], grid, p->s_gemm, i));
    }
  }
  NF_CUDA(cudaEventRecord(ev_done, p->s_gemm));
  NF_CUDA(cudaStreamWaitEvent(st, ev_done, 0));
  join_.done = true;
  return NF_OK;
}

// Metadata once (with layer 0), then layer l reads `in` (x for l = 0) and
// writes `out` (y for the last layer), ping-ponging between the plan's
// activation buffers.
nf_status run_layers(nf_plan p, const nf_layer_weights* layers, int n_layers, const void* x,
                     void* const* k_pools, void* const* v_pools, const int32_t* bt,
                     const int32_t* sl, void* y, cudaStream_t st) {
  if (cross_layer(p, n_layers)) {
    std::vector<const void*> act(n_layers + 1);
    act[0] = x;
    for (int l = 0; l < n_layers; ++l)
      act[l + 1] = l == n_layers - 1 ? y : (act[l] == p->xa ? (const void*)p->xb : (const void*)p->xa);
    return run_layers_pipelined(p, layers, n_layers, act, k_pools, v_pools, bt, sl, st);
  }
  const void* cur = x;
  for (int l = 0; l < n_layers; ++l) {
    // intermediate outputs alternate between xa and xb; the caller makes sure
    // that y is not the last layer's input
    void* nxt = l == n_layers - 1 ? y : (cur == p->xa ? (void*)p->xb : (void*)p->xa);
    p->cur_set = l;
    // the metadata runs once, inside layer 0 (it clears every layer's counters)
    const nf_status r = layer_step(p, &layers[l], cur, k_pools[l], v_pools[l], bt, sl, nxt, st,
                                   /*with_meta=*/l == 0);
    p->cur_set = 0;
    if (r != NF_OK) return r;
    cur = nxt;
  }
  return NF_OK;
}
}  // namespace

nf_status nf_layers_step(nf_plan p, const nf_layer_weights* layers, int32_t n_layers,
                         const void* x, void* const* k_pools, void* const* v_pools,
                         const int32_t* bt, const int32_t* sl, void* y, void* stream) {
  if (!p || !layers || !x || !k_pools || !v_pools || !bt || !sl || !y)
    return fail(NF_ERR_INVALID_ARG, "NULL argument");
  if (n_layers < 1) return fail(NF_ERR_INVALID_ARG, "n_layers must be positive");
  if (x == y) return fail(NF_ERR_INVALID_ARG, "x and y must be different buffers");
  NF_TRY(ensure_layers(p, n_layers));
  for (int l = 0; l < n_layers; ++l)
    NF_TRY(check_step_args(p, &layers[l], x, k_pools[l], v_pools[l], bt, sl, y));
  return run_layers(p, layers, n_layers, x, k_pools, v_pools, bt, sl, y,
                    static_cast<cudaStream_t>(stream));
}

namespace {
// The stack step; select: logits only for the n_rows rows listed in `rows`
// (device indices), gathered after the last layer, in that order.
nf_status stack_step(nf_plan p, const nf_stack_weights* sw, const int32_t* tokens,
                     void* const* k_pools, void* const* v_pools, const int32_t* bt,
                     const int32_t* sl, bool select, const int32_t* rows, int n_rows,
                     void* logits, void* stream) {
  if (!p || !sw || !tokens || !k_pools || !v_pools || !bt || !sl || !logits)
    return fail(NF_ERR_INVALID_ARG, "NULL argument");
  if (sw->n_layers < 1 || !sw->layers || !sw->embed || !sw->norm_f || !sw->lm_head)
    return fail(NF_ERR_INVALID_ARG, "stack weights incomplete");
  if (sw->vocab < 8 || sw->vocab % 8)
    return fail(NF_ERR_INVALID_ARG, "vocab must be a positive multiple of 8 (got %d)", sw->vocab);
  if (!aligned16(sw->embed) || !aligned16(sw->norm_f) || !aligned16(sw->lm_head) ||
      !aligned16(logits))
    return fail(NF_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  NF_TRY(ensure_layers(p, sw->n_layers));
  if (p->lm_key != sw->lm_head || p->lm_vocab != sw->vocab) {
    if (!nf::make_tmap_bf16(&p->tm_lm, sw->lm_head, sw->vocab, p->shape.hidden, 256) ||
        !nf::make_tmap_bf16(&p->tm_lm128, sw->lm_head, sw->vocab, p->shape.hidden, 128))
      return fail(NF_ERR_INVALID_ARG, "LM head tensor map failed");
    p->lm_key = sw->lm_head;
    p->lm_vocab = sw->vocab;
  }
  for (int l = 0; l < sw->n_layers; ++l) {
    NF_TRY(check_step_args(p, &sw->layers[l], p->xa, k_pools[l], v_pools[l], bt, sl, p->xb));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const nf_model_shape& s = p->shape;
  // embedding into xa, then the layers (metadata once for all of them); layer
  // l >= 1 reads xb when l is odd, so the last one writes the other buffer
  NF_CUDA(nf::launch_embed(tokens, static_cast<const __nv_bfloat16*>(sw->embed), p->xa, p->T,
                           s.hidden, sw->vocab, p->status, st));
  __nv_bfloat16* last = sw->n_layers % 2 ? p->xb : p->xa;
  NF_TRY(run_layers(p, sw->layers, sw->n_layers, p->xa, k_pools, v_pools, bt, sl, last, st));
  const __nv_bfloat16* cur = last;
  // final RMSNorm and the LM head: logits = RMSNorm(x) lm_head^T, for every
  // row, or for the selected rows gathered first (into n1, normalised into n2)
  const int M = select ? n_rows : p->T;
  if (M == 0) return NF_OK;
  const int xm = select ? XM_N2 : XM_N1;
  if (select) {
    NF_CUDA(nf::launch_gather_rows(cur, rows, p->n1, n_rows, s.hidden, p->T, p->status, st));
    NF_CUDA(nf::launch_rmsnorm(p->n1, static_cast<const __nv_bfloat16*>(sw->norm_f), p->n2, 0,
                               n_rows, s.hidden, s.rms_eps, st));
  } else {
    NF_CUDA(nf::launch_rmsnorm(cur, static_cast<const __nv_bfloat16*>(sw->norm_f), p->n1, 0, p->T,
                               s.hidden, s.rms_eps, st));
  }
  GemmArgs g = base_args(p);
  g.stages = 4;
  g.m_begin = 0;
  g.m_end = M;
  g.N = sw->vocab;
  g.K = s.hidden;
  g.m_tiles = (M + 127) / 128;
  g.n_tiles = (sw->vocab + 255) / 256;
  g.C = static_cast<__nv_bfloat16*>(logits);
  g.ldc = sw->vocab;
  if (use_wrows(p, M)) {
    const int w_tiles = (sw->vocab + 127) / 128;
    const WrChoice c = wr_choose(nf::EPI_STORE, M, w_tiles, g.K, p->num_sms);
    if (c.splits) {
      g.n_tiles = w_tiles;
      g.m_tiles = (M + c.tok - 1) / c.tok;
      g.splits = c.splits;
      NF_CUDA(nf::launch_gemm_wrows(nf::EPI_STORE, c.tok, p->tm_lm128, p->tm_lm128,
                                    xmap(p, xm, c.tok), g, c.clusters, true, st));
      return NF_OK;
    }
  }
  g.splits = p->opts.gemm_split_k == 1 ? 1 : choose_splits(g.m_tiles * g.n_tiles, g.K, p->num_sms);
  NF_CUDA(nf::launch_gemm(nf::EPI_STORE, select ? p->tm_n2 : p->tm_n1, p->tm_lm, p->tm_lm, g,
                          cap_grid(g.m_tiles * g.n_tiles * g.splits, p->num_sms), st));
  return NF_OK;
}
}  // namespace

nf_status nf_stack_step(nf_plan p, const nf_stack_weights* sw, const int32_t* tokens,
                        void* const* k_pools, void* const* v_pools, const int32_t* bt,
                        const int32_t* sl, void* logits, void* stream) {
  return stack_step(p, sw, tokens, k_pools, v_pools, bt, sl, false, nullptr, 0, logits, stream);
}

nf_status nf_stack_step_rows(nf_plan p, const nf_stack_weights* sw, const int32_t* tokens,
                             void* const* k_pools, void* const* v_pools, const int32_t* bt,
                             const int32_t* sl, const int32_t* rows, int32_t n_rows, void* logits,
                             void* stream) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (n_rows < 0 || n_rows > p->T || (n_rows > 0 && !rows))
    return fail(NF_ERR_INVALID_ARG, "n_rows must be in [0, %d] with a row list", p->T);
  return stack_step(p, sw, tokens, k_pools, v_pools, bt, sl, true, rows, n_rows, logits, stream);
}

namespace {
bool host_pinned(const void* ptr) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// The copies in, the step and the copy out, on stream st.  (Storing y straight
// into a pinned y_host from the last GEMM's epilogue was measured: the stores
// crossing to the host stall the epilogue, 1.10 -> 0.99 M tokens/s end to end.)
nf_status host_step_body(nf_plan p, const nf_layer_weights* w, const void* x_host, void* k_pool,
                         void* v_pool, const int32_t* bt_host, const int32_t* sl_host,
                         void* y_host, cudaStream_t st) {
  const size_t xb = (size_t)p->T * p->shape.hidden * 2;
  const size_t btb = (size_t)p->n_seq * p->max_pages * 4, slb = (size_t)p->n_seq * 4;
  NF_CUDA(cudaMemcpyAsync(p->x_stage, x_host, xb, cudaMemcpyHostToDevice, st));
  NF_CUDA(cudaMemcpyAsync(p->bt_stage, bt_host, btb, cudaMemcpyHostToDevice, st));
  NF_CUDA(cudaMemcpyAsync(p->sl_stage, sl_host, slb, cudaMemcpyHostToDevice, st));
  NF_TRY(layer_step(p, w, p->x_stage, k_pool, v_pool, p->bt_stage, p->sl_stage, p->y_stage, st));
  NF_CUDA(cudaMemcpyAsync(y_host, p->y_stage, xb, cudaMemcpyDeviceToHost, st));
  return NF_OK;
}
}  // namespace

nf_status nf_layer_step_host(nf_plan p, const nf_layer_weights* w, const void* x_host,
                             void* k_pool, void* v_pool, const int32_t* bt_host,
                             const int32_t* sl_host, void* y_host, void* stream) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (!w || !x_host || !y_host || !bt_host || !sl_host)
    return fail(NF_ERR_INVALID_ARG, "a host pointer is NULL");
  if (!p->x_stage) {  // sized for the plan's capacity
    NF_TRY(dalloc(&p->x_stage, (size_t)p->T_cap * p->shape.hidden * 2));
    NF_TRY(dalloc(&p->y_stage, (size_t)p->T_cap * p->shape.hidden * 2));
    NF_TRY(dalloc(&p->bt_stage, (size_t)p->seq_cap * p->max_pages * 4));
    NF_TRY(dalloc(&p->sl_stage, (size_t)p->seq_cap * 4));
  }
  NF_TRY(check_step_args(p, w, p->x_stage, k_pool, v_pool, p->bt_stage, p->sl_stage, p->y_stage));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  NF_CUDA(cudaStreamIsCapturing(st, &cap));
  // Replay a captured graph when the host buffers are pinned (the copies are then
  // asynchronous graph nodes), the caller is not capturing and no trace is taken.
  const bool graph_ok = cap == cudaStreamCaptureStatusNone && p->trace_left == 0 &&
                        host_pinned(x_host) && host_pinned(y_host) && host_pinned(bt_host) &&
                        host_pinned(sl_host);
  if (!graph_ok) {
    NF_TRY(host_step_body(p, w, x_host, k_pool, v_pool, bt_host, sl_host, y_host, st));
    NF_CUDA(cudaStreamSynchronize(st));
    return NF_OK;
  }
  const void* key[16] = {w->norm1, w->w_qkv, w->w_o, w->norm2, w->w_gate_up, w->w_down,
                         w->w_experts_gate_up, w->w_experts_down, w->router_logits, x_host,
                         k_pool, v_pool, bt_host, sl_host, y_host, nullptr};
  nf_plan_s::HostGraph* hg = nullptr;
  for (auto& h : p->hgraphs)
    if (h.version == p->batch_version && std::memcmp(h.key, key, sizeof(key)) == 0) hg = &h;
  if (!p->s_host) {
    NF_CUDA(cudaStreamCreateWithFlags(&p->s_host, cudaStreamNonBlocking));
    NF_CUDA(cudaEventCreateWithFlags(&p->ev_host, cudaEventDisableTiming));
  }
  // ordered after the caller's earlier work on `stream`
  NF_CUDA(cudaEventRecord(p->ev_host, st));
  NF_CUDA(cudaStreamWaitEvent(p->s_host, p->ev_host, 0));
  if (!hg || !hg->exec) {
    if (!hg) {  // first sight: run directly (lazy set-up happens outside any capture)
      if (p->hgraphs.size() >= 8) {
        if (p->hgraphs.front().exec) cudaGraphExecDestroy(p->hgraphs.front().exec);
        p->hgraphs.erase(p->hgraphs.begin());
      }
      nf_plan_s::HostGraph h{};
      std::memcpy(h.key, key, sizeof(key));
      h.version = p->batch_version;
      h.exec = nullptr;
      p->hgraphs.push_back(h);
      NF_TRY(host_step_body(p, w, x_host, k_pool, v_pool, bt_host, sl_host, y_host, p->s_host));
      NF_CUDA(cudaStreamSynchronize(p->s_host));
      return NF_OK;
    }
    NF_CUDA(cudaStreamSynchronize(p->s_host));
    cudaGraph_t g = nullptr;
    NF_CUDA(cudaStreamBeginCapture(p->s_host, cudaStreamCaptureModeThreadLocal));
    const nf_status s = host_step_body(p, w, x_host, k_pool, v_pool, bt_host, sl_host, y_host,
                                       p->s_host);
    const cudaError_t e = cudaStreamEndCapture(p->s_host, &g);
    if (s != NF_OK) {
      if (g) cudaGraphDestroy(g);
      return s;
    }
    if (e != cudaSuccess) return fail(NF_ERR_CUDA, "capture of the host step: %s", cudaGetErrorString(e));
    const cudaError_t ie = cudaGraphInstantiate(&hg->exec, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) {
      hg->exec = nullptr;
      return fail(NF_ERR_CUDA, "instantiation of the host step: %s", cudaGetErrorString(ie));
    }
  }
  NF_CUDA(cudaGraphLaunch(hg->exec, p->s_host));
  NF_CUDA(cudaStreamSynchronize(p->s_host));
  return NF_OK;
}

nf_status nf_layer_step_host_async(nf_plan p, const nf_layer_weights* w, const void* x_host,
                                   void* k_pool, void* v_pool, const int32_t* bt_host,
                                   const int32_t* sl_host, void* y_host, void* stream) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (!w || !x_host || !y_host || !bt_host || !sl_host)
    return fail(NF_ERR_INVALID_ARG, "a host pointer is NULL");
  auto& q = p->pipe;
  if (!q.s_in) {
    for (int i = 0; i < 2; ++i) {
      NF_TRY(dalloc(&q.x[i], (size_t)p->T_cap * p->shape.hidden * 2));
      NF_TRY(dalloc(&q.y[i], (size_t)p->T_cap * p->shape.hidden * 2));
      NF_TRY(dalloc(&q.bt[i], (size_t)p->seq_cap * p->max_pages * 4));
      NF_TRY(dalloc(&q.sl[i], (size_t)p->seq_cap * 4));
      NF_CUDA(cudaEventCreateWithFlags(&q.in_done[i], cudaEventDisableTiming));
      NF_CUDA(cudaEventCreateWithFlags(&q.step_done[i], cudaEventDisableTiming));
      NF_CUDA(cudaEventCreateWithFlags(&q.out_done[i], cudaEventDisableTiming));
    }
    NF_CUDA(cudaStreamCreateWithFlags(&q.s_in, cudaStreamNonBlocking));
    NF_CUDA(cudaStreamCreateWithFlags(&q.s_out, cudaStreamNonBlocking));
  }
  const int s = q.next;
  NF_TRY(check_step_args(p, w, q.x[s], k_pool, v_pool, q.bt[s], q.sl[s], q.y[s]));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)p->T * p->shape.hidden * 2;
  const size_t btb = (size_t)p->n_seq * p->max_pages * 4, slb = (size_t)p->n_seq * 4;
  // inputs into slot s once the step two calls back (the slot's last reader) is done
  NF_CUDA(cudaStreamWaitEvent(q.s_in, q.step_done[s], 0));
  NF_CUDA(cudaMemcpyAsync(q.x[s], x_host, xb, cudaMemcpyHostToDevice, q.s_in));
  NF_CUDA(cudaMemcpyAsync(q.bt[s], bt_host, btb, cudaMemcpyHostToDevice, q.s_in));
  NF_CUDA(cudaMemcpyAsync(q.sl[s], sl_host, slb, cudaMemcpyHostToDevice, q.s_in));
  NF_CUDA(cudaEventRecord(q.in_done[s], q.s_in));
  // the step, once its inputs landed and the slot's previous y was copied out
  NF_CUDA(cudaStreamWaitEvent(st, q.in_done[s], 0));
  NF_CUDA(cudaStreamWaitEvent(st, q.out_done[s], 0));
  NF_TRY(layer_step(p, w, q.x[s], k_pool, v_pool, q.bt[s], q.sl[s], q.y[s], st));
  NF_CUDA(cudaEventRecord(q.step_done[s], st));
  // y out
  NF_CUDA(cudaStreamWaitEvent(q.s_out, q.step_done[s], 0));
  NF_CUDA(cudaMemcpyAsync(y_host, q.y[s], xb, cudaMemcpyDeviceToHost, q.s_out));
  NF_CUDA(cudaEventRecord(q.out_done[s], q.s_out));
  q.next = s ^ 1;
  return NF_OK;
}

nf_status nf_plan_host_wait(nf_plan p) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (p->pipe.s_out) NF_CUDA(cudaStreamSynchronize(p->pipe.s_out));
  return NF_OK;
}

nf_status nf_plan_set_batch(nf_plan p, const nf_batch_desc* b, const nf_plan_opts* opts,
                            void* stream) {
  if (!p || !b) return fail(NF_ERR_INVALID_ARG, "plan or batch is NULL");
  const int n_seq = b->n_decode + b->n_prefill;
  if (b->n_decode < 0 || b->n_prefill < 0 || n_seq < 1 || n_seq > p->seq_cap)
    return fail(NF_ERR_INVALID_ARG, "the batch must hold 1 ... %d sequences (got %d)", p->seq_cap,
                n_seq);
  if (b->n_prefill > 0 && !b->prefill_q_lens) return fail(NF_ERR_INVALID_ARG, "prefill_q_lens is NULL");
  if (b->max_pages_per_seq != p->max_pages || b->num_pages != p->num_pages)
    return fail(NF_ERR_INVALID_ARG, "max_pages_per_seq and num_pages must stay as created");
  std::vector<int> q_lens, tok_begin{0}, prefill_q;
  for (int i = 0; i < n_seq; ++i) {
    const int q = i < b->n_decode ? 1 : b->prefill_q_lens[i - b->n_decode];
    if (q < 1) return fail(NF_ERR_INVALID_ARG, "prefill_q_lens[%d] must be >= 1", i - b->n_decode);
    if (i >= b->n_decode) prefill_q.push_back(q);
    q_lens.push_back(q);
    tok_begin.push_back(tok_begin.back() + q);
  }
  const int T = tok_begin.back();
  if (T > p->T_cap)
    return fail(NF_ERR_INVALID_ARG, "the batch holds %d tokens, the plan at most %d", T, p->T_cap);
  nf_plan_opts o = p->opts;
  if (opts) {
    o = *opts;
    if (o.kv_chunk == 0) o.kv_chunk = p->opts.kv_chunk;
    if (o.timeout_ns == 0) o.timeout_ns = p->opts.timeout_ns;
    if (o.attn_warps == 0) o.attn_warps = p->opts.attn_warps;
    if (o.gemm_stages == 0) o.gemm_stages = p->opts.gemm_stages;
    if (o.attn_impl == NF_ATTN_AUTO) o.attn_impl = p->opts.attn_impl;
    if (o.kv_chunk != p->opts.kv_chunk || o.attn_impl != p->opts.attn_impl ||
        o.attn_warps != p->opts.attn_warps)
      return fail(NF_ERR_INVALID_ARG,
                  "kv_chunk, attn_impl and attn_warps must stay as the plan was created");
  } else if (T != p->T) {  // the old split does not fit: one nano-batch
    o.n_attn = o.n_ffn = 1;
    o.attn_bounds[0] = o.ffn_bounds[0] = 0;
    o.attn_bounds[1] = o.ffn_bounds[1] = T;
    o.executor = NF_EXEC_SEQUENTIAL;
  }
  NF_TRY(check_opts(&o, T, p->num_sms));
  if (!p->set_stage)
    NF_CUDA(cudaHostAlloc(&p->set_stage, 2 * (2 * (size_t)p->seq_cap + 2 + NF_MAX_NANO + 1) * 4,
                          cudaHostAllocDefault));
  // Two halves, used alternately: a copy enqueued by the previous call may still
  // be pending when this one writes.  The host may run further ahead than one
  // call (steps are asynchronous), so before a half is written again the copies
  // that read it last must have run: wait for the event recorded after them.
  const int half = p->set_flip;
  if (p->set_ev_live[half]) NF_CUDA(cudaEventSynchronize(p->set_ev[half]));
  p->set_ev_live[half] = false;
  if (!p->set_ev[half]) NF_CUDA(cudaEventCreateWithFlags(&p->set_ev[half], cudaEventDisableTiming));
  int* h = p->set_stage + half * (2 * p->seq_cap + 2 + NF_MAX_NANO + 1);
  p->set_flip ^= 1;
  std::copy(q_lens.begin(), q_lens.end(), h);
  std::copy(tok_begin.begin(), tok_begin.end(), h + p->seq_cap);
  std::copy(o.attn_bounds, o.attn_bounds + o.n_attn + 1, h + 2 * p->seq_cap + 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  NF_CUDA(cudaMemcpyAsync(p->d_q_lens, h, n_seq * 4, cudaMemcpyHostToDevice, st));
  NF_CUDA(cudaMemcpyAsync(p->d_tok_begin, h + p->seq_cap, (n_seq + 1) * 4, cudaMemcpyHostToDevice,
                          st));
  NF_CUDA(cudaMemcpyAsync(p->d_seg_bounds, h + 2 * p->seq_cap + 1, (o.n_attn + 1) * 4,
                          cudaMemcpyHostToDevice, st));
  {
    std::vector<int4> tiles;
    int seg[NF_MAX_NANO + 1];
    build_prefill_tiles(p, b->n_decode, n_seq, tok_begin, o, tiles, seg);
    if (!p->pf_stage)
      NF_CUDA(cudaHostAlloc(&p->pf_stage, 2 * (size_t)p->T_cap * sizeof(int4), cudaHostAllocDefault));
    int4* hp = p->pf_stage + (size_t)half * p->T_cap;  // guarded by the same event
    std::copy(tiles.begin(), tiles.end(), hp);
    if (!tiles.empty())
      NF_CUDA(cudaMemcpyAsync(p->pf_tiles, hp, tiles.size() * sizeof(int4), cudaMemcpyHostToDevice,
                              st));
    std::copy(seg, seg + o.n_attn + 1, p->pf_seg);
  }
  NF_CUDA(cudaEventRecord(p->set_ev[half], st));
  p->set_ev_live[half] = true;
  p->n_decode = b->n_decode;
  p->n_prefill = b->n_prefill;
  p->n_seq = n_seq;
  p->T = T;
  p->q_lens = q_lens;
  p->tok_begin = tok_begin;
  p->prefill_q = prefill_q;
  p->seq_hint.clear();
  if (b->seq_lens_hint) p->seq_hint.assign(b->seq_lens_hint, b->seq_lens_hint + n_seq);
  p->opts = o;
  ++p->batch_version;  // captured host-buffer steps hold the old structure
  return NF_OK;
}

nf_status nf_plan_poll(nf_plan p, int wait) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (wait) NF_CUDA(cudaDeviceSynchronize());
  NF_CUDA(cudaGetLastError());
  uint32_t st = 0;
  NF_CUDA(cudaMemcpy(&st, p->status, 4, cudaMemcpyDeviceToHost));
  if (st) NF_CUDA(cudaMemset(p->status, 0, 4));
  if (st & nf::ST_TIMEOUT) return fail(NF_ERR_TIMEOUT, "a device wait timed out (status 0x%x)", st);
  if (st) return fail(NF_ERR_DEVICE, "device-side check failed (status 0x%x: %s%s%s)", st,
                      (st & nf::ST_BAD_PAGE) ? "page id out of range " : "",
                      (st & nf::ST_BAD_LEN) ? "bad sequence length " : "",
                      (st & nf::ST_OVERFLOW) ? "work list overflow" : "");
  return NF_OK;
}

nf_status nf_plan_selftest_wait(nf_plan p, int64_t timeout_ns, int32_t arrive, void* waited_ns,
                                void* stream) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  if (timeout_ns < 1 || timeout_ns > 10000000000LL)
    return fail(NF_ERR_INVALID_ARG, "timeout_ns must lie in [1, 1e10]");
  NF_CUDA(nf::launch_selftest_wait(p->status, static_cast<unsigned long long>(timeout_ns),
                                   arrive ? 1 : 0, static_cast<unsigned long long*>(waited_ns),
                                   static_cast<cudaStream_t>(stream)));
  return NF_OK;
}

nf_status nf_step_metadata(nf_plan p, const int32_t* bt, const int32_t* sl, void* stream) {
  if (!p || !bt || !sl) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  return run_meta(p, bt, sl, static_cast<cudaStream_t>(stream));
}

nf_status nf_attention(nf_plan p, const void* q, const void* kp, const void* vp,
                       const int32_t* bt, const int32_t* sl, void* o, void* stream) {
  if (!p || !q || !kp || !vp || !bt || !sl || !o) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(q) || !aligned16(kp) || !aligned16(vp) || !aligned16(o))
    return fail(NF_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  NF_TRY(run_meta(p, bt, sl, st));
  for (int i = 0; i < p->opts.n_attn; ++i)
    NF_TRY(run_attention(p, i, q, kp, vp, bt, o, p->num_sms, st));
  return NF_OK;
}

nf_status nf_rmsnorm(const void* x, const void* g, void* out, int32_t rows, int32_t hidden,
                     float eps, void* stream) {
  if (!x || !g || !out) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  if (rows < 0 || hidden <= 0 || hidden % 8)
    return fail(NF_ERR_INVALID_ARG, "hidden must be a positive multiple of 8");
  if (!aligned16(x) || !aligned16(g) || !aligned16(out))
    return fail(NF_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  NF_CUDA(nf::launch_rmsnorm(static_cast<const __nv_bfloat16*>(x),
                             static_cast<const __nv_bfloat16*>(g),
                             static_cast<__nv_bfloat16*>(out), 0, rows, hidden, eps,
                             static_cast<cudaStream_t>(stream)));
  return NF_OK;
}

nf_status nf_gemm(const void* A, const void* B, void* C, const void* R, int32_t M, int32_t N,
                  int32_t K, int32_t epilogue, int32_t max_sms, void* stream) {
  if (!A || !B || !C) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  if (M < 1 || N < 8 || K < 8 || N % 8 || K % 8)
    return fail(NF_ERR_INVALID_ARG, "need M >= 1 and N, K positive multiples of 8");
  if (epilogue < NF_EPI_STORE || epilogue > NF_EPI_SWIGLU)
    return fail(NF_ERR_INVALID_ARG, "unknown epilogue %d", epilogue);
  if (epilogue == NF_EPI_RESID && !R) return fail(NF_ERR_INVALID_ARG, "residual R is NULL");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (R && !aligned16(R)))
    return fail(NF_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int sms = device_sms();
  if (sms <= 0) return fail(NF_ERR_CUDA, "no CUDA device");
  CUtensorMap ta, tb, tb2;
  bool ok = nf::make_tmap_bf16(&ta, A, M, K, 128);
  if (epilogue == NF_EPI_SWIGLU) {
    ok = ok && nf::make_tmap_bf16(&tb, B, N, K, 128) &&
         nf::make_tmap_bf16(&tb2, static_cast<const char*>(B) + (size_t)N * K * 2, N, K, 128);
  } else {
    ok = ok && nf::make_tmap_bf16(&tb, B, N, K, 256);
    tb2 = tb;
  }
  if (!ok) return fail(NF_ERR_CUDA, "tensor map creation failed");
  GemmArgs g{};
  g.m_begin = 0;
  g.m_end = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + 127) / 128;
  g.n_tiles = (N + nf::gemm_block_n(epilogue) - 1) / nf::gemm_block_n(epilogue);
  g.C = static_cast<__nv_bfloat16*>(C);
  g.ldc = N;
  g.R = static_cast<const __nv_bfloat16*>(R);
  g.ldr = N;
  g.status = global_status();
  g.timeout_ns = kDefaultTimeoutNs;
  g.stages = 4;
  const int cap = (max_sms > 0 && max_sms < sms) ? max_sms : sms;
  g.splits = 1;
  const int splits = choose_splits(g.m_tiles * g.n_tiles, K, cap);
  if (splits > 1) {
    GlobalSplitWs* ws = global_split_ws();
    if (ws->part) {
      g.splits = splits;
      g.part = ws->part;
      g.tile_cnt = ws->cnt;
    }
  }
  NF_CUDA(nf::launch_gemm(epilogue, ta, tb, tb2, g,
                          cap_grid(g.m_tiles * g.n_tiles * g.splits, cap),
                          static_cast<cudaStream_t>(stream)));
  return NF_OK;
}

nf_status nf_gemm_wrows(const void* A, const void* B, void* C, const void* R, int32_t M,
                        int32_t N, int32_t K, int32_t epilogue, int32_t splits, int32_t max_sms,
                        void* stream) {
  if (!A || !B || !C) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  if (M < 1 || M > 256 || N < 8 || K < 8 || N % 8 || K % 8)
    return fail(NF_ERR_INVALID_ARG, "need 1 <= M <= 256 and N, K positive multiples of 8");
  if (epilogue < NF_EPI_STORE || epilogue > NF_EPI_SWIGLU)
    return fail(NF_ERR_INVALID_ARG, "unknown epilogue %d", epilogue);
  if (epilogue == NF_EPI_RESID && !R) return fail(NF_ERR_INVALID_ARG, "residual R is NULL");
  if (splits < 0 || splits > 8 || splits > (K + 63) / 64)
    return fail(NF_ERR_INVALID_ARG, "splits must be 0 or 1 .. min(8, ceil(K / 64))");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (R && !aligned16(R)))
    return fail(NF_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int sms = device_sms();
  if (sms <= 0) return fail(NF_ERR_CUDA, "no CUDA device");
  const int cap = (max_sms > 0 && max_sms < sms) ? max_sms : sms;
  const int w_tiles = (N + 127) / 128;
  const WrChoice c = wr_choose(epilogue, M, w_tiles, K, cap, splits);
  if (!c.splits) return fail(NF_ERR_UNSUPPORTED, "no cluster of %d CTAs fits in %d SMs", splits, cap);
  CUtensorMap tw, tw2, tx;
  bool ok = nf::make_tmap_bf16(&tx, A, M, K, c.tok) && nf::make_tmap_bf16(&tw, B, N, K, 128);
  if (epilogue == NF_EPI_SWIGLU)
    ok = ok && nf::make_tmap_bf16(&tw2, static_cast<const char*>(B) + (size_t)N * K * 2, N, K, 128);
  else
    tw2 = tw;
  if (!ok) return fail(NF_ERR_CUDA, "tensor map creation failed");
  GemmArgs g{};
  g.m_begin = 0;
  g.m_end = M;
  g.N = N;
  g.K = K;
  g.n_tiles = w_tiles;
  g.m_tiles = (M + c.tok - 1) / c.tok;
  g.splits = c.splits;
  g.C = static_cast<__nv_bfloat16*>(C);
  g.ldc = N;
  g.R = static_cast<const __nv_bfloat16*>(R);
  g.ldr = N;
  g.status = global_status();
  g.timeout_ns = kDefaultTimeoutNs;
  NF_CUDA(nf::launch_gemm_wrows(epilogue, c.tok, tw, tw2, tx, g, c.clusters, false,
                                static_cast<cudaStream_t>(stream)));
  return NF_OK;
}

nf_status nf_plan_trace_ops(nf_plan p, uint32_t op_mask) {
  if (!p) return fail(NF_ERR_INVALID_ARG, "plan is NULL");
  p->trace_ops = op_mask;
  return NF_OK;
}

nf_status nf_plan_trace_enable(nf_plan p, int32_t max_steps) {
  if (!p || max_steps < 0) return fail(NF_ERR_INVALID_ARG, "bad argument");
  NF_CUDA(cudaDeviceSynchronize());
  std::vector<cudaEvent_t> s0s;
  for (auto& r : p->trace) {
    p->ev_pool.push_back(r.b);
    p->ev_pool.push_back(r.e);
    if (std::find(s0s.begin(), s0s.end(), r.s0) == s0s.end()) s0s.push_back(r.s0);
  }
  for (cudaEvent_t e : s0s) p->ev_pool.push_back(e);
  p->trace.clear();
  p->trace_left = max_steps;
  p->trace_step = 0;
  return NF_OK;
}

nf_status nf_plan_trace_read(nf_plan p, nf_trace_entry* out, int32_t cap, int32_t* n_out) {
  if (!p || !n_out || (cap > 0 && !out)) return fail(NF_ERR_INVALID_ARG, "bad argument");
  NF_CUDA(cudaDeviceSynchronize());
  int n = 0;
  for (auto& r : p->trace) {
    if (n < cap) {
      float st = 0.f, ms = 0.f;
      NF_CUDA(cudaEventElapsedTime(&st, r.s0, r.b));
      NF_CUDA(cudaEventElapsedTime(&ms, r.b, r.e));
      out[n] = {r.op, r.nano, r.step, st, ms};
    }
    ++n;
  }
  *n_out = n;
  return NF_OK;
}

nf_status nf_plan_buffer_size(nf_plan p, int32_t which, size_t* bytes) {
  if (!p || !bytes) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  *bytes = buf_bytes(p, which);
  if (*bytes == 0) return fail(NF_ERR_INVALID_ARG, "unknown buffer %d", which);
  return NF_OK;
}

nf_status nf_plan_copy_buffer(nf_plan p, int32_t which, void* dst, size_t bytes) {
  if (!p || !dst) return fail(NF_ERR_INVALID_ARG, "NULL argument");
  const size_t have = buf_bytes(p, which);
  if (have == 0) return fail(NF_ERR_INVALID_ARG, "unknown buffer %d", which);
  if (bytes > have) return fail(NF_ERR_INVALID_ARG, "asked %zu bytes, buffer has %zu", bytes, have);
  NF_CUDA(cudaDeviceSynchronize());
  NF_CUDA(cudaMemcpy(dst, buf_ptr(p, which), bytes, cudaMemcpyDefault));
  return NF_OK;
}

}  // extern "C"
