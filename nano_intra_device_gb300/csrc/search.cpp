// Plan search: nano-batch count, token boundaries and SM shares that minimise
// the predicted step time of the two-stream pipeline.
//
// The pages' auto-search ("NanoFlow: Towards Optimal LLM Serving Throughput",
// "Auto-Search Stage I" and "Auto-Search Stage II") solves two MILPs: first the
// nano-batch structure (count, sizes in multiples of 128 summing to B_dense,
// order) with interference-free kernel times, then the resource share of each
// nano-operation from a measured R -> P table.  On one GPU with two resource
// classes (tensor-core GEMMs, HBM-bound attention) and a fixed operation order
// the space is small: n <= 4 nano-batches on a 128-token grid, an SM split on a
// 1/16 grid (1/64 for several layers).  This file enumerates it and scores each
// candidate with a list-scheduling simulation of the two streams, which is
// exact under the same time model the MILP would use, and needs no solver.
// For a step of several layers the simulation follows the cross-layer window
// of the executor (no join between layers; the pages search a window of
// neighbouring layers).
//
// Time model (per nano-operation, on S SMs):
//   GEMM M x N x K: waves = ceil(tiles / S) with 128 x 256 tiles, each tile
//     2*128*256*K / (per-SM tensor rate); plus a launch cost; beside attention
//     a GEMM keeps 1 - c u^2 of its rate, u the share of HBM bandwidth the
//     attention draws;
//   attention: decode K/V bytes / min(HBM bandwidth, S * per-SM attention
//     bandwidth), plus prefill rows' FLOPs at the tiled prefill kernel's per-SM
//     rate (a prefill row is charged a tile's share of its K/V bytes);
//     an SM share is an SM count because every kernel runs one CTA per SM;
//   a fixed cost per cross-stream dependency.
// The rates come from a profile written by nf_profile, else from built-in
// GB300 values: in-step measurements for the one-layer simulation, effective
// values fitted to measured window plans for the multi-layer one.  An
// overlapped plan must be predicted >= 2 % faster than the sequential one.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/nanoflow.h"
#include "schedule.h"

namespace {

// Defaults are GB300 measurements of this library's kernels (nf_profile on the
// 8B-shaped layer); a profile file overrides them.
struct Rates {
  double gemm_flops_per_sm = 11.45e12; // tensor rate of a GEMM, per SM (all 152 SMs busy)
  double qkv_row_sm_s = 3.5e-6;        // SM-seconds per token row of the QKV epilogue
                                       // (RoPE and the K/V append into the pools)
  double stream_sync_s = 25e-6;        // cost of one cross-stream dependency (event wait,
                                       // launch, pipeline fill of the waiting kernel)
  double hbm_bps = 6.75e12;            // attention bandwidth with every SM
  double attn_bps_per_sm = 78e9;       // attention bytes/s one SM sustains (tensor-core
                                       // kernel, 8 warps, measured on 57 SMs in the step)
  double gemm_launch_s = 4e-6;
  double attn_launch_s = 4e-6;
  // tiled prefill attention (tensor cores, K/V from L2): FLOPs/s one SM
  // sustains (a 2048-token chunk at the 8B shape: 34.4 GFLOP in 131.6 us on 152 SMs)
  double attn_prefill_flops_per_sm = 1.72e12;
  // Interference: attention keeps 0.85 of its alone bandwidth beside GEMMs on
  // other SMs.  A GEMM beside attention keeps 1 - c u^2 of its per-SM rate, u the
  // share of HBM bandwidth the attention draws: measured 0.6 ... 0.8 (0.65 taken)
  // at the 8B-shaped step with 76 attention SMs (u ~ 0.75), and at least 0.87
  // implied by the 70B-shaped step with 46 (u ~ 0.45); c = 0.62 fits both.  A
  // profile may fix the factor instead (overlap_gemm_factor).
  double overlap_bw_factor = 0.85;     // attention speed kept beside a GEMM on other SMs
  double gemm_interference = 0.62;     // c
  double overlap_gemm_factor = 0;      // > 0: GEMM speed kept beside attention, fixed
};

bool json_has(const std::string& s, const char* key) {
  return s.find(std::string("\"") + key + "\"") != std::string::npos;
}

double json_number(const std::string& s, const char* key, double dflt) {
  const std::string k = std::string("\"") + key + "\"";
  size_t p = s.find(k);
  if (p == std::string::npos) return dflt;
  p = s.find(':', p);
  if (p == std::string::npos) return dflt;
  return std::strtod(s.c_str() + p + 1, nullptr);
}

bool load_rates(const char* path, Rates* r) {
  if (!path) return true;
  FILE* f = std::fopen(path, "r");
  if (!f) return false;
  std::string s;
  char buf[4096];
  size_t n;
  while ((n = std::fread(buf, 1, sizeof(buf), f)) > 0) s.append(buf, n);
  std::fclose(f);
  r->gemm_flops_per_sm = json_number(s, "gemm_flops_per_sm", r->gemm_flops_per_sm);
  r->hbm_bps = json_number(s, "hbm_bps", r->hbm_bps);
  r->attn_bps_per_sm = json_number(s, "attn_bps_per_sm", r->attn_bps_per_sm);
  r->gemm_launch_s = json_number(s, "gemm_launch_s", r->gemm_launch_s);
  r->attn_launch_s = json_number(s, "attn_launch_s", r->attn_launch_s);
  r->overlap_bw_factor = json_number(s, "overlap_bw_factor", r->overlap_bw_factor);
  // a fitted interference coefficient takes precedence over a fixed factor
  if (json_has(s, "gemm_interference"))
    r->gemm_interference = json_number(s, "gemm_interference", r->gemm_interference);
  else
    r->overlap_gemm_factor = json_number(s, "overlap_gemm_factor", r->overlap_gemm_factor);
  r->qkv_row_sm_s = json_number(s, "qkv_row_sm_s", r->qkv_row_sm_s);
  r->attn_prefill_flops_per_sm =
      json_number(s, "attn_prefill_flops_per_sm", r->attn_prefill_flops_per_sm);
  r->stream_sync_s = json_number(s, "stream_sync_s", r->stream_sync_s);
  return true;
}

struct Model {
  nf_model_shape s;
  Rates r;
  int sms;
  // per token row: the K/V bytes its attention reads from HBM (a decode row
  // its whole visible K/V; a prefill row a share of it, since the tiled kernel
  // reads each page once for a tile of rows) and its prefill attention FLOPs
  std::vector<double> row_kv_bytes;
  std::vector<double> row_pf_flops;
  std::vector<double> prefix, prefix_flops;  // prefix sums of both
  std::vector<double> row_ctx;                // visible positions of each row
  std::vector<double> prefix_cost;            // prefix sums of the rows' attention seconds

  double gemm_time(int rows, int N, int K, int S, int bn) const {
    if (rows <= 0) return 0;
    const double tiles = std::ceil(rows / 128.0) * std::ceil(N / double(bn));
    const double waves = std::ceil(tiles / S);
    const double per_tile = 2.0 * 128 * bn * K / r.gemm_flops_per_sm;
    return waves * per_tile + r.gemm_launch_s;
  }
  // QKV + O for rows, or RMSNorm-2 + gate/up + down for rows
  double qkv_time(int rows, int S) const {
    return gemm_time(rows, (s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim, s.hidden, S, 256) +
           rows * r.qkv_row_sm_s / S;
  }
  double o_time(int rows, int S) const {
    return gemm_time(rows, s.hidden, s.n_q_heads * s.head_dim, S, 256);
  }
  double ffn_time(int rows, int S) const {
    if (s.n_experts > 0) rows *= s.top_k;  // every token runs top_k experts
    return gemm_time(rows, s.ffn, s.hidden, S, 128) + gemm_time(rows, s.hidden, s.ffn, S, 256);
  }
  // 1 / the share of its speed a GEMM keeps beside attention on attn_sms SMs
  double gemm_slow(int attn_sms) const {
    double f = r.overlap_gemm_factor;
    if (f <= 0) {
      const double u = std::min(r.hbm_bps, attn_sms * r.attn_bps_per_sm) * r.overlap_bw_factor / r.hbm_bps;
      f = 1.0 - r.gemm_interference * u * u;
    }
    return 1.0 / std::max(0.2, f);
  }
  double attn_time(int r0, int r1, int S, bool overlapped) const {
    const double bytes = prefix[r1] - prefix[r0];
    const double pf = (prefix_flops[r1] - prefix_flops[r0]) / (S * r.attn_prefill_flops_per_sm);
    double bw = std::min(r.hbm_bps, S * r.attn_bps_per_sm);
    if (overlapped) bw *= r.overlap_bw_factor;
    return bytes / bw + pf + r.attn_launch_s;
  }
};

// Simulate the two-stream pipeline of api.cu's stream executor.
double simulate(const Model& m, const nf_plan_opts& o) {
  const int all = m.sms;
  const int n = o.n_attn;
  if (o.executor == NF_EXEC_SEQUENTIAL) {
    double t = 0;
    for (int i = 0; i < n; ++i) {
      const int r0 = o.attn_bounds[i], r1 = o.attn_bounds[i + 1];
      t += m.qkv_time(r1 - r0, all) + m.attn_time(r0, r1, all, false) + m.o_time(r1 - r0, all);
    }
    for (int j = 0; j < o.n_ffn; ++j) t += m.ffn_time(o.ffn_bounds[j + 1] - o.ffn_bounds[j], all);
    return t;
  }
  const int attn_sms = n == 1 ? all : o.attn_sms;
  const int gsm = o.gemm_sms > 0 ? o.gemm_sms : std::max(1, all - attn_sms);
  double tg = 0, ta = 0;
  std::vector<double> q_done(n), a_done(n);
  const double slow = m.gemm_slow(attn_sms);
  for (int i = 0; i < n; ++i) {
    tg += m.qkv_time(o.attn_bounds[i + 1] - o.attn_bounds[i], i == 0 ? all : gsm) * (i == 0 ? 1.0 : slow);
    q_done[i] = tg;
  }
  const double sync = m.r.stream_sync_s;
  for (int i = 0; i < n; ++i) {
    ta = std::max(ta, q_done[i] + sync);  // attention i waits for QKV i on the other stream
    ta += m.attn_time(o.attn_bounds[i], o.attn_bounds[i + 1], attn_sms, n > 1);
    a_done[i] = ta;
  }
  int next_ffn = 0;
  for (int i = 0; i < n; ++i) {
    tg = std::max(tg, a_done[i] + sync);  // O projection i waits for attention i
    const int S = (i == n - 1) ? all : gsm;
    const double f = (i == n - 1) ? 1.0 : slow;
    tg += m.o_time(o.attn_bounds[i + 1] - o.attn_bounds[i], S) * f;
    while (next_ffn < o.n_ffn && o.ffn_bounds[next_ffn + 1] <= o.attn_bounds[i + 1]) {
      tg += m.ffn_time(o.ffn_bounds[next_ffn + 1] - o.ffn_bounds[next_ffn], S) * f;
      ++next_ffn;
    }
  }
  return tg;
}

// The cross-layer window over L layers (api.cu's run_layers_pipelined): the
// same operations in the same stream order, no join between layers; returns
// the time of all L layers.  Nothing overlaps the first QKV projection of the
// first layer and what follows the last attention of the last layer.
double simulate_window(const Model& m, const nf_plan_opts& o, int L) {
  const int all = m.sms, n = o.n_attn;
  const int attn_sms = o.attn_sms;
  const int gsm = o.gemm_sms > 0 ? o.gemm_sms : std::max(1, all - attn_sms);
  const double slow = m.gemm_slow(attn_sms), sync = m.r.stream_sync_s;
  double tg = 0, ta = 0;
  std::vector<double> a_done(n);
  for (const nf::WindowOp& op : nf::window_schedule(o, L)) {
    const int S = op.full ? all : gsm;
    const double f = op.full ? 1.0 : slow;
    const int i = op.nano;
    if (op.kind == nf::WOP_QKV) {  // QKV on the GEMM stream, then its attention
      tg += m.qkv_time(o.attn_bounds[i + 1] - o.attn_bounds[i], S) * f;
      ta = std::max(ta, tg + sync);
      ta += m.attn_time(o.attn_bounds[i], o.attn_bounds[i + 1], attn_sms, true);
      a_done[i] = ta;
    } else if (op.kind == nf::WOP_O) {
      tg = std::max(tg, a_done[i] + sync);  // O projection i waits for attention i
      tg += m.o_time(o.attn_bounds[i + 1] - o.attn_bounds[i], S) * f;
    } else {
      tg += m.ffn_time(o.ffn_bounds[i + 1] - o.ffn_bounds[i], S) * f;
    }
  }
  return tg;
}

// The time model of a batch: per-row attention bytes and prefill FLOPs, and
// the rates (a profile's, else the built-in ones).
nf_status build_model(const nf_model_shape* shape, const nf_batch_desc* batch,
                      const char* profile_json, int32_t num_sms, bool window, Model* m) {
  m->s = *shape;
  m->sms = num_sms;
  if (window && !profile_json) {
    // The cross-layer window's simulation, calibrated on measured window plans
    // (GB300; the 8B-shaped mixed batch through 16 layers, the 70B-shaped step,
    // an 8B decode stack, a serving-like mix and MoE layers): these effective
    // rates give the measured choice between overlap and the sequential plan
    // in each.  The single-layer simulation keeps the in-step measurements
    // above, which give its measured choices (the two simulations simplify
    // different schedules, and their parameters absorb that).
    m->r.attn_bps_per_sm = 95e9;
    m->r.qkv_row_sm_s = 7e-6;
  }
  if (!load_rates(profile_json, &m->r)) return NF_ERR_INVALID_ARG;
  const int n_seq = batch->n_decode + batch->n_prefill;
  const double kv_tok = 2.0 * shape->n_kv_heads * shape->head_dim * 2;
  // rows of a prefill tile (128 query vectors: 128 / GQA group rows)
  const double tile_rows = 128.0 / std::max(1, shape->n_q_heads / std::max(1, shape->n_kv_heads));
  const int default_ctx = batch->max_pages_per_seq * shape->page_size / 2;
  for (int s = 0; s < n_seq; ++s) {
    const int q = s < batch->n_decode ? 1 : batch->prefill_q_lens[s - batch->n_decode];
    if (q < 1) return NF_ERR_INVALID_ARG;
    const int L = batch->seq_lens_hint ? batch->seq_lens_hint[s]
                                       : (s < batch->n_decode ? default_ctx : q);
    const bool pre = s >= batch->n_decode;
    for (int i = 0; i < q; ++i) {
      const double vis = double(L - q + i + 1);
      m->row_kv_bytes.push_back(vis * kv_tok / (pre ? tile_rows : 1.0));
      m->row_pf_flops.push_back(pre ? 4.0 * shape->n_q_heads * shape->head_dim * vis : 0.0);
      m->row_ctx.push_back(vis);
    }
  }
  const int T = int(m->row_kv_bytes.size());
  if (T < 1) return NF_ERR_INVALID_ARG;
  m->prefix.assign(T + 1, 0.0);
  m->prefix_flops.assign(T + 1, 0.0);
  for (int t = 0; t < T; ++t) {
    m->prefix[t + 1] = m->prefix[t] + m->row_kv_bytes[t];
    m->prefix_flops[t + 1] = m->prefix_flops[t] + m->row_pf_flops[t];
  }

  // attention cost per row in seconds on the whole GPU: what nano-batch
  // boundaries balance
  m->prefix_cost.assign(T + 1, 0.0);
  for (int t = 0; t < T; ++t)
    m->prefix_cost[t + 1] = m->prefix_cost[t] + m->row_kv_bytes[t] / m->r.hbm_bps +
                            m->row_pf_flops[t] / (num_sms * m->r.attn_prefill_flops_per_sm);
  return NF_OK;
}

#define NF_MODEL_TRY(x)              \
  do {                               \
    const nf_status st_ = (x);       \
    if (st_ != NF_OK) return st_;    \
  } while (0)

// Boundaries that split the attention cost of the batch evenly, on a grid.
void balanced_bounds(const Model& m, int T, int n, int grid, int32_t* b) {
  b[0] = 0;
  b[n] = T;
  const double total = m.prefix_cost[T];
  for (int i = 1; i < n; ++i) {
    const double target = total * i / n;
    int t = int(std::lower_bound(m.prefix_cost.begin(), m.prefix_cost.end(), target) -
                m.prefix_cost.begin());
    t = std::max(1, std::min(T - 1, (t + grid / 2) / grid * grid));
    b[i] = std::max(t, b[i - 1] + 1);
  }
  for (int i = n - 1; i >= 1; --i) b[i] = std::min(b[i], b[i + 1] - 1);
}

nf_status search(const nf_model_shape* shape, const nf_batch_desc* batch, const char* profile_json,
                 int32_t num_sms, int32_t n_layers, nf_plan_opts* out, double* predicted_us) {
  if (!shape || !batch || !out || num_sms <= 0 || n_layers < 1) return NF_ERR_INVALID_ARG;
  Model m;
  NF_MODEL_TRY(build_model(shape, batch, profile_json, num_sms, n_layers > 1, &m));
  const int T = int(m.row_ctx.size());
  const int n_seq = batch->n_decode + batch->n_prefill;

  // Split-KV piece length: the longest that still gives the resident
  // attention warps about one and a half pieces each (load balance), so that a
  // small decode batch is not left to a few long pieces while most warps idle;
  // shorter pieces than that cost more in merges than they gain (measured on
  // 32-layer stacks at 64 and 256 decode requests).
  int kv_chunk = 128;
  {
    const double warps = 8.0 * num_sms;
    for (int cand : {1024, 512, 256, 128}) {
      double pieces = 0;
      int t = 0;
      for (int s = 0; s < n_seq; ++s) {
        const int q = s < batch->n_decode ? 1 : batch->prefill_q_lens[s - batch->n_decode];
        for (int i = 0; i < q; ++i, ++t) {
          const double ctx = m.row_ctx[t];
          pieces += std::ceil(ctx / cand);
        }
      }
      if (pieces * shape->n_kv_heads >= 1.5 * warps) {
        kv_chunk = cand;
        break;
      }
    }
  }
  nf_plan_opts best{};
  std::memset(&best, 0, sizeof(best));
  best.n_attn = 1;
  best.attn_bounds[1] = T;
  best.n_ffn = 1;
  best.ffn_bounds[1] = T;
  best.executor = NF_EXEC_SEQUENTIAL;
  best.kv_chunk = kv_chunk;
  best.attn_warps = 8;
  best.gemm_stages = 4;
  best.timeout_ns = 2000000000LL;
  double best_t = simulate(m, best) * n_layers;
  // An overlapped plan replaces the sequential one only when the model
  // predicts it at least 2 % faster: the model's error on measured plans is a
  // few per cent, the size of the gains it ranks.
  const double overlap_cap = 0.98 * best_t;

  const int grid = T >= 1024 ? 128 : 1;  // nano-batches are multiples of 128 tokens
  if (n_layers > 1) {
    // the cross-layer window: equal splits of both groups, or the pages' 70B
    // structure of 4 attention and 2 FFN nano-batches; attention shares on a
    // 1/64 grid (the step time moves steeply with it)
    for (int n = 2; n <= 4; ++n) {
      if (T / grid < n) break;
      nf_plan_opts o = best;
      o.executor = NF_EXEC_STREAMS;
      o.n_attn = n;
      balanced_bounds(m, T, n, grid, o.attn_bounds);
      for (int nf_ : {n, 2}) {
        if (nf_ == 2 && n != 4) continue;
        o.n_ffn = nf_;
        if (nf_ == n) {
          for (int i = 0; i <= n; ++i) o.ffn_bounds[i] = o.attn_bounds[i];
        } else {
          o.ffn_bounds[0] = 0;
          o.ffn_bounds[1] = o.attn_bounds[n / 2];
          o.ffn_bounds[2] = T;
        }
        for (int k = 8; k <= 40; ++k) {
          o.attn_sms = std::max(1, num_sms * k / 64);
          o.gemm_sms = 0;
          const double t = simulate_window(m, o, n_layers);
          if (t < best_t && t < overlap_cap) {
            best_t = t;
            best = o;
          }
        }
      }
    }
    *out = best;
    if (predicted_us) *predicted_us = best_t * 1e6;
    return NF_OK;
  }
  for (int n = 2; n <= 4; ++n) {
    if (T / grid < n) break;
    nf_plan_opts o = best;
    o.executor = NF_EXEC_STREAMS;
    o.n_attn = n;
    balanced_bounds(m, T, n, grid, o.attn_bounds);
    for (int nf_ = 1; nf_ <= 2; ++nf_) {
      o.n_ffn = nf_;
      if (nf_ == 1) {
        o.ffn_bounds[0] = 0;
        o.ffn_bounds[1] = T;
      } else {
        o.ffn_bounds[0] = 0;
        o.ffn_bounds[1] = o.attn_bounds[n / 2];
        o.ffn_bounds[2] = T;
      }
      for (int k = 2; k <= 15; ++k) {
        o.attn_sms = std::max(1, num_sms * k / 16);
        o.gemm_sms = 0;
        const double t = simulate(m, o);
        if (t < best_t && t < overlap_cap) {
          best_t = t;
          best = o;
        }
      }
    }
  }
  *out = best;
  if (predicted_us) *predicted_us = best_t * 1e6;
  return NF_OK;
}

// Predicted time of a given plan over n_layers layers, as the search scores it.
nf_status predict(const nf_model_shape* shape, const nf_batch_desc* batch, const char* profile_json,
                  int32_t num_sms, int32_t n_layers, const nf_plan_opts* o, double* us) {
  if (!shape || !batch || !o || !us || num_sms <= 0 || n_layers < 1) return NF_ERR_INVALID_ARG;
  const bool window = o->executor == NF_EXEC_STREAMS && o->n_attn >= 2 && n_layers >= 2;
  Model m;
  NF_MODEL_TRY(build_model(shape, batch, profile_json, num_sms, n_layers > 1, &m));
  const int T = int(m.row_ctx.size());
  for (int g = 0; g < 2; ++g) {  // bounds must describe this batch
    const int n = g ? o->n_ffn : o->n_attn;
    const int32_t* b = g ? o->ffn_bounds : o->attn_bounds;
    if (n < 1 || n > NF_MAX_NANO || b[0] != 0 || b[n] != T) return NF_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
      if (b[i + 1] <= b[i]) return NF_ERR_INVALID_ARG;
  }
  if (o->executor == NF_EXEC_STREAMS && (o->attn_sms < 0 || o->attn_sms > num_sms))
    return NF_ERR_INVALID_ARG;
  const double t = window ? simulate_window(m, *o, n_layers) : simulate(m, *o) * n_layers;
  *us = t * 1e6;
  return NF_OK;
}

}  // namespace

extern "C" nf_status nf_plan_predict(const nf_model_shape* shape, const nf_batch_desc* batch,
                                     const char* profile_json, int32_t num_sms, int32_t n_layers,
                                     const nf_plan_opts* plan, double* predicted_us) {
  return predict(shape, batch, profile_json, num_sms, n_layers, plan, predicted_us);
}

extern "C" nf_status nf_plan_search(const nf_model_shape* shape, const nf_batch_desc* batch,
                                    const char* profile_json, int32_t num_sms, nf_plan_opts* out,
                                    double* predicted_us) {
  return search(shape, batch, profile_json, num_sms, 1, out, predicted_us);
}

extern "C" nf_status nf_plan_search_layers(const nf_model_shape* shape, const nf_batch_desc* batch,
                                           const char* profile_json, int32_t num_sms,
                                           int32_t n_layers, nf_plan_opts* out,
                                           double* predicted_us) {
  return search(shape, batch, profile_json, num_sms, n_layers, out, predicted_us);
}

extern "C" nf_status nf_window_schedule(const nf_plan_opts* o, int32_t n_layers, int32_t* out,
                                        int32_t cap, int32_t* n_ops) {
  if (!o || !n_ops || n_layers < 1 || cap < 0 || (cap > 0 && !out)) return NF_ERR_INVALID_ARG;
  for (int g = 0; g < 2; ++g) {
    const int n = g ? o->n_ffn : o->n_attn;
    const int32_t* b = g ? o->ffn_bounds : o->attn_bounds;
    if (n < 1 || n > NF_MAX_NANO || b[0] != 0) return NF_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
      if (b[i + 1] <= b[i]) return NF_ERR_INVALID_ARG;
  }
  if (o->attn_bounds[o->n_attn] != o->ffn_bounds[o->n_ffn]) return NF_ERR_INVALID_ARG;
  const std::vector<nf::WindowOp> ops = nf::window_schedule(*o, n_layers);
  *n_ops = static_cast<int32_t>(ops.size());
  for (int k = 0; k < static_cast<int>(ops.size()) && k < cap; ++k) {
    out[4 * k] = ops[k].kind;
    out[4 * k + 1] = ops[k].layer;
    out[4 * k + 2] = ops[k].nano;
    out[4 * k + 3] = ops[k].full;
  }
  return NF_OK;
}
