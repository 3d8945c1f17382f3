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

#include <mutex>

#include "../../include/nanoflow.h"
#include "internal.h"
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
  // The R -> P table measured inside traced steps of the executor's own
  // schedule (nf_profile_step): for plans of rp_n[i] attention nano-batches
  // with attention on rp_sms[i] SMs overlapping GEMMs on the rest, the
  // attention's bytes/s per SM and the share of the model's GEMM rate the
  // GEMMs kept.  When present it replaces the parametric interference terms
  // above: the rows of the nearest profiled nano-batch count, interpolated
  // linearly in the SM count and clamped at the ends (rows sorted by n, then S).
  std::vector<double> rp_n, rp_sms, rp_attn_bps_per_sm, rp_gemm_factor;
  // the profiled plans' measured step times (all profiled layers), for the
  // batch structure and layer count they were measured on
  int prof_tokens = -1, prof_decode = -1, prof_layers = -1;
  std::vector<double> run_n, run_sms, run_ms;
  // a measured table is not extrapolated: the search stays inside its SM range
  bool in_table(int S) const {
    if (rp_sms.empty()) return true;
    const auto mm = std::minmax_element(rp_sms.begin(), rp_sms.end());
    return S >= *mm.first && S <= *mm.second;
  }
  double interp(const std::vector<double>& y, int n, double S) const {
    if (rp_sms.empty()) return 0;
    double nn = rp_n[0];
    for (double v : rp_n)
      if (std::fabs(v - n) < std::fabs(nn - n)) nn = v;
    size_t a = 0;
    while (rp_n[a] != nn) ++a;
    size_t b = a;
    while (b + 1 < rp_n.size() && rp_n[b + 1] == nn) ++b;
    if (S <= rp_sms[a]) return y[a];
    for (size_t i = a + 1; i <= b; ++i)
      if (S <= rp_sms[i]) {
        const double w = (S - rp_sms[i - 1]) / (rp_sms[i] - rp_sms[i - 1]);
        return y[i - 1] + w * (y[i] - y[i - 1]);
      }
    return y[b];
  }
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

// A JSON array of numbers under `key` ("key": [a, b, ...]); empty if absent.
std::vector<double> json_array(const std::string& s, const char* key) {
  std::vector<double> v;
  const std::string k = std::string("\"") + key + "\"";
  size_t p = s.find(k);
  if (p == std::string::npos) return v;
  p = s.find('[', p);
  const size_t e = s.find(']', p);
  if (p == std::string::npos || e == std::string::npos) return v;
  const char* c = s.c_str() + p + 1;
  const char* end = s.c_str() + e;
  while (c < end) {
    char* nx = nullptr;
    const double x = std::strtod(c, &nx);
    if (nx == c) {
      ++c;
      continue;
    }
    v.push_back(x);
    c = nx;
  }
  return v;
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
  r->rp_sms = json_array(s, "rp_sms");
  r->rp_n = json_array(s, "rp_n");
  if (r->rp_n.empty()) r->rp_n.assign(r->rp_sms.size(), 2.0);  // a table of one plan kind
  r->rp_attn_bps_per_sm = json_array(s, "rp_attn_bps_per_sm");
  r->rp_gemm_factor = json_array(s, "rp_gemm_factor");
  r->prof_tokens = int(json_number(s, "batch_tokens", -1));
  r->prof_decode = int(json_number(s, "batch_decode", -1));
  r->prof_layers = int(json_number(s, "n_layers", -1));
  r->run_n = json_array(s, "run_n");
  r->run_sms = json_array(s, "run_sms");
  r->run_ms = json_array(s, "run_ms");
  if (r->run_sms.size() != r->run_n.size() || r->run_ms.size() != r->run_n.size()) {
    r->run_n.clear();
    r->run_sms.clear();
    r->run_ms.clear();
  }
  if (r->rp_attn_bps_per_sm.size() != r->rp_sms.size() ||
      r->rp_gemm_factor.size() != r->rp_sms.size() || r->rp_n.size() != r->rp_sms.size()) {
    r->rp_n.clear();
    r->rp_sms.clear();
    r->rp_attn_bps_per_sm.clear();
    r->rp_gemm_factor.clear();
  }
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
  double gemm_slow(int attn_sms, int n_attn) const {
    if (!r.rp_sms.empty()) return 1.0 / std::max(0.2, r.interp(r.rp_gemm_factor, n_attn, attn_sms));
    double f = r.overlap_gemm_factor;
    if (f <= 0) {
      const double u = std::min(r.hbm_bps, attn_sms * r.attn_bps_per_sm) * r.overlap_bw_factor / r.hbm_bps;
      f = 1.0 - r.gemm_interference * u * u;
    }
    return 1.0 / std::max(0.2, f);
  }
  double attn_time(int r0, int r1, int S, bool overlapped, int n_attn = 2) const {
    const double bytes = prefix[r1] - prefix[r0];
    const double pf = (prefix_flops[r1] - prefix_flops[r0]) / (S * r.attn_prefill_flops_per_sm);
    double bw = std::min(r.hbm_bps, S * r.attn_bps_per_sm);
    if (overlapped && !r.rp_sms.empty())
      bw = std::min(r.hbm_bps, S * r.interp(r.rp_attn_bps_per_sm, n_attn, S));
    else if (overlapped)
      bw *= r.overlap_bw_factor;
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
  const double slow = m.gemm_slow(attn_sms, n);
  for (int i = 0; i < n; ++i) {
    tg += m.qkv_time(o.attn_bounds[i + 1] - o.attn_bounds[i], i == 0 ? all : gsm) * (i == 0 ? 1.0 : slow);
    q_done[i] = tg;
  }
  const double sync = m.r.stream_sync_s;
  for (int i = 0; i < n; ++i) {
    ta = std::max(ta, q_done[i] + sync);  // attention i waits for QKV i on the other stream
    ta += m.attn_time(o.attn_bounds[i], o.attn_bounds[i + 1], attn_sms, n > 1, n);
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
  const double slow = m.gemm_slow(attn_sms, n), sync = m.r.stream_sync_s;
  double tg = 0, ta = 0;
  std::vector<double> a_done(n);
  for (const nf::WindowOp& op : nf::window_schedule(o, L)) {
    const int S = op.full ? all : gsm;
    const double f = op.full ? 1.0 : slow;
    const int i = op.nano;
    if (op.kind == nf::WOP_QKV) {  // QKV on the GEMM stream, then its attention
      tg += m.qkv_time(o.attn_bounds[i + 1] - o.attn_bounds[i], S) * f;
      ta = std::max(ta, tg + sync);
      ta += m.attn_time(o.attn_bounds[i], o.attn_bounds[i + 1], attn_sms, true, n);
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
  // rows of a prefill tile (128 query vectors: 128 / GQA group rows), which
  // read each page once
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

  return NF_OK;
}

// Profiles registered for shapes (nf_profile_use, nf_profile_step): a NULL
// profile argument means the registered one, "" the built-in rates.
std::mutex g_prof_mu;
std::vector<std::pair<nf_model_shape, std::string>> g_profiles;

bool same_shape(const nf_model_shape& a, const nf_model_shape& b) {
  return a.hidden == b.hidden && a.n_q_heads == b.n_q_heads && a.n_kv_heads == b.n_kv_heads &&
         a.head_dim == b.head_dim && a.ffn == b.ffn && a.n_experts == b.n_experts &&
         a.top_k == b.top_k && a.page_size == b.page_size;
}

std::string profile_of(const nf_model_shape* shape, const char* profile_json) {
  if (profile_json) return profile_json;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const auto& e : g_profiles)
    if (same_shape(e.first, *shape)) return e.second;
  return std::string();
}
const char* path_or_null(const std::string& p) { return p.empty() ? nullptr : p.c_str(); }

#define NF_MODEL_TRY(x)              \
  do {                               \
    const nf_status st_ = (x);       \
    if (st_ != NF_OK) return st_;    \
  } while (0)

// The attention nano-batch bounds of the candidates: equal token shares on
// the grid.  (Splitting the attention's cost evenly instead measured slower
// in the cross-layer window, whose GEMMs split by tokens: the 8B step's batch
// through 16 layers 25.15 against 24.73 ms, the 70B-shaped step 69.2 against
// 68.1 ms.)
void nano_bounds(int T, int n, int grid, int32_t* b) {
  b[0] = 0;
  for (int i = 1; i < n; ++i) {
    const int t = (T * i / n + grid / 2) / grid * grid;
    b[i] = std::max(std::min(t, T - (n - i)), b[i - 1] + 1);
  }
  b[n] = T;
}

nf_status search(const nf_model_shape* shape, const nf_batch_desc* batch, const char* profile_json,
                 int32_t num_sms, int32_t n_layers, nf_plan_opts* out, double* predicted_us) {
  if (!shape || !batch || !out || num_sms <= 0 || n_layers < 1) return NF_ERR_INVALID_ARG;
  Model m;
  const std::string prof = profile_of(shape, profile_json);
  NF_MODEL_TRY(build_model(shape, batch, path_or_null(prof), num_sms, n_layers > 1, &m));
  const int T = int(m.row_ctx.size());
  const int n_seq = batch->n_decode + batch->n_prefill;

  // Split-KV piece length: the longest that still gives the resident
  // attention warps about one and a half pieces each, so that a small decode
  // batch is not left to a few long pieces while most warps idle; but not
  // below 512 positions while those still give the warps about one piece each
  // (4 for 5 warps): shorter pieces cost more in piece setup and merges than
  // they gain.  Measured on the 32-layer stacks at 64, 128, 256 and 1024
  // decode requests: 512, 512, 1024 and 1024 positions, each the fastest of
  // 256 ... 1024.
  int kv_chunk = 128;
  {
    const double warps = 8.0 * num_sms;
    auto pieces_of = [&](int cand) {
      double pieces = 0;
      int t = 0;
      for (int s = 0; s < n_seq; ++s) {
        const int q = s < batch->n_decode ? 1 : batch->prefill_q_lens[s - batch->n_decode];
        for (int i = 0; i < q; ++i, ++t) pieces += std::ceil(m.row_ctx[t] / cand);
      }
      return pieces * shape->n_kv_heads;
    };
    for (int cand : {1024, 512, 256, 128}) {
      if (pieces_of(cand) >= 1.5 * warps) {
        kv_chunk = cand;
        break;
      }
    }
    if (kv_chunk < 512 && pieces_of(512) >= 0.8 * warps) kv_chunk = 512;
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

  // The profile measured plans on this very batch structure and layer count:
  // pick the fastest of them by its measured (untraced) step time; an
  // overlapped plan must measure at least 1 % faster than the sequential one
  // (run-to-run noise).
  if (!m.r.run_n.empty() && m.r.prof_tokens == T && m.r.prof_decode == batch->n_decode &&
      m.r.prof_layers == std::min(n_layers, 32)) {
    double seq_ms = -1, best_ms = -1;
    int bn = 1, bs = 0;
    for (size_t i = 0; i < m.r.run_n.size(); ++i)
      if (m.r.run_n[i] <= 1 && m.r.run_ms[i] > 0) seq_ms = m.r.run_ms[i];
    for (size_t i = 0; i < m.r.run_n.size(); ++i) {
      const double t = m.r.run_ms[i];
      if (t <= 0) continue;
      const bool seq = m.r.run_n[i] <= 1;
      if (!seq && seq_ms > 0 && t > 0.99 * seq_ms) continue;
      if (best_ms < 0 || t < best_ms) {
        best_ms = t;
        bn = seq ? 1 : int(m.r.run_n[i]);
        bs = seq ? 0 : int(m.r.run_sms[i]);
      }
    }
    if (best_ms > 0) {
      if (bn > 1) {
        best.executor = NF_EXEC_STREAMS;
        best.n_attn = best.n_ffn = bn;
        nano_bounds(T, bn, T >= 1024 ? 128 : 1, best.attn_bounds);
        for (int i = 0; i <= bn; ++i) best.ffn_bounds[i] = best.attn_bounds[i];
        best.attn_sms = bs;
      }
      *out = best;
      if (predicted_us)
        *predicted_us = best_ms * 1e3 * n_layers / std::max(1, m.r.prof_layers);
      return NF_OK;
    }
  }
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
      nano_bounds(T, n, grid, o.attn_bounds);
      const int ffn_counts[2] = {n, n == 4 ? 2 : 0};
      for (int nf_ : ffn_counts) {
        if (nf_ == 0) continue;
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
          if (!m.r.in_table(o.attn_sms)) continue;
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
    nano_bounds(T, n, grid, o.attn_bounds);
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
        if (!m.r.in_table(o.attn_sms)) continue;
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
  const std::string prof = profile_of(shape, profile_json);
  NF_MODEL_TRY(build_model(shape, batch, path_or_null(prof), num_sms, n_layers > 1, &m));
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

namespace nf {

std::string registered_profile(const nf_model_shape* shape) { return profile_of(shape, nullptr); }

nf_status search_bounds(const nf_model_shape* shape, const nf_batch_desc* batch, int32_t num_sms,
                        int n, int32_t* b) {
  if (!shape || !batch || !b || num_sms <= 0 || n < 1 || n > NF_MAX_NANO) return NF_ERR_INVALID_ARG;
  Model m;
  NF_MODEL_TRY(build_model(shape, batch, nullptr, num_sms, false, &m));
  const int T = int(m.row_ctx.size());
  if (T < n) return NF_ERR_INVALID_ARG;
  nano_bounds(T, n, T >= 1024 && T / 128 >= n ? 128 : 1, b);
  return NF_OK;
}

namespace {

// [start, end) of an operation of a traced step, relative to the step start
struct Iv {
  double a, b;
};
double overlap(const Iv& x, const std::vector<Iv>& ys) {
  double o = 0;
  for (const Iv& y : ys) o += std::max(0.0, std::min(x.b, y.b) - std::max(x.a, y.a));
  return o;
}

// Model time of one traced GEMM-stream operation on S SMs (seconds).
double model_gemm_op(const Model& m, const nf_plan_opts& o, const nf_trace_entry& e, int S) {
  if (e.op == NF_OP_FFN) {
    if (e.nano < 0 || e.nano >= o.n_ffn) return 0;
    return m.ffn_time(o.ffn_bounds[e.nano + 1] - o.ffn_bounds[e.nano], S);
  }
  if (e.nano < 0 || e.nano >= o.n_attn) return 0;
  const int rows = o.attn_bounds[e.nano + 1] - o.attn_bounds[e.nano];
  return e.op == NF_OP_QKV ? m.qkv_time(rows, S) : e.op == NF_OP_OPROJ ? m.o_time(rows, S) : 0;
}

}  // namespace

std::string fit_step_profile(const nf_model_shape* shape, const nf_batch_desc* batch, int num_sms,
                             int n_layers, const std::vector<TracedRun>& runs) {
  if (!shape || !batch || runs.empty() || runs[0].opts.executor != NF_EXEC_SEQUENTIAL ||
      n_layers < 1 || num_sms < 2)
    return std::string();
  Model m;
  if (build_model(shape, batch, nullptr, num_sms, false, &m) != NF_OK) return std::string();
  Rates& r = m.r;
  // 1) interference-free rates from the sequential plan: one scale for the
  //    GEMM tensor rate (all four GEMM kinds), the attention's bandwidth
  const TracedRun& seq = runs[0];
  double g_meas = 0, g_model = 0, a_meas = 0;
  for (const nf_trace_entry& e : seq.ops) {
    if (e.op == NF_OP_ATTN) a_meas += e.ms * 1e-3;
    else if (e.op != NF_OP_META) {
      g_meas += e.ms * 1e-3;
      g_model += model_gemm_op(m, seq.opts, e, num_sms);
    }
  }
  const double steps = std::max(1, seq.steps);
  g_meas /= steps;
  a_meas /= steps;
  g_model /= steps;
  if (g_meas <= 0 || a_meas <= 0) return std::string();
  r.gemm_flops_per_sm *= g_model / g_meas;
  const double T = double(m.row_ctx.size());
  const double bytes_all = m.prefix.back() * n_layers;
  const double pf_all = m.prefix_flops.back() / (num_sms * r.attn_prefill_flops_per_sm) * n_layers;
  r.hbm_bps = bytes_all / std::max(1e-9, a_meas - pf_all - n_layers * r.attn_launch_s);
  (void)T;

  // 2) the R -> P table from the two-stream runs: attention bytes/s per SM and
  //    the share of the model's GEMM rate kept, over the operations that ran
  //    beside the other stream's
  struct Acc {
    double bytes = 0, attn_s = 0, gemm_model = 0, gemm_meas = 0;
  };
  std::vector<std::pair<std::pair<int, int>, Acc>> by_sms;  // (n_attn, S) -> sums
  for (size_t k = 1; k < runs.size(); ++k) {
    const TracedRun& run = runs[k];
    const nf_plan_opts& o = run.opts;
    if (o.executor != NF_EXEC_STREAMS || o.attn_sms < 1 || o.attn_sms >= num_sms) continue;
    const int S = o.attn_sms, gsm = o.gemm_sms > 0 ? o.gemm_sms : num_sms - S;
    std::vector<Iv> attn_iv, gemm_iv;
    for (const nf_trace_entry& e : run.ops) {
      const Iv iv{double(e.start_ms) + 1e6 * e.step, double(e.start_ms) + 1e6 * e.step + e.ms};
      if (e.op == NF_OP_ATTN) attn_iv.push_back(iv);
      else if (e.op != NF_OP_META) gemm_iv.push_back(iv);
    }
    Acc acc;
    for (const nf_trace_entry& e : run.ops) {
      const Iv iv{double(e.start_ms) + 1e6 * e.step, double(e.start_ms) + 1e6 * e.step + e.ms};
      if (e.op == NF_OP_ATTN) {
        if (e.nano < 0 || e.nano >= o.n_attn || overlap(iv, gemm_iv) < 0.5 * e.ms) continue;
        const int r0 = o.attn_bounds[e.nano], r1 = o.attn_bounds[e.nano + 1];
        const double pf = (m.prefix_flops[r1] - m.prefix_flops[r0]) / (S * r.attn_prefill_flops_per_sm);
        acc.bytes += m.prefix[r1] - m.prefix[r0];
        acc.attn_s += std::max(1e-9, e.ms * 1e-3 - pf - r.attn_launch_s);
      } else if (e.op != NF_OP_META) {
        if (overlap(iv, attn_iv) < 0.5 * e.ms) continue;  // ran alone, on every SM
        acc.gemm_model += model_gemm_op(m, o, e, gsm);
        acc.gemm_meas += e.ms * 1e-3;
      }
    }
    if (acc.attn_s <= 0 || acc.gemm_meas <= 0) continue;
    bool found = false;
    const std::pair<int, int> key{o.n_attn, S};
    for (auto& b : by_sms)
      if (b.first == key) {
        b.second.bytes += acc.bytes;
        b.second.attn_s += acc.attn_s;
        b.second.gemm_model += acc.gemm_model;
        b.second.gemm_meas += acc.gemm_meas;
        found = true;
      }
    if (!found) by_sms.push_back({key, acc});
  }
  std::sort(by_sms.begin(), by_sms.end(),
            [](const std::pair<std::pair<int, int>, Acc>& x,
               const std::pair<std::pair<int, int>, Acc>& y) { return x.first < y.first; });
  for (const auto& b : by_sms) {
    r.rp_n.push_back(b.first.first);
    r.rp_sms.push_back(b.first.second);
    r.rp_attn_bps_per_sm.push_back(b.second.bytes / b.second.attn_s / b.first.second);
    r.rp_gemm_factor.push_back(std::min(1.5, b.second.gemm_model / b.second.gemm_meas));
  }

  // 3) two scalars that the per-operation rates cannot give: the cost of a
  //    cross-stream dependency (0 ... 100 us), and one factor on the GEMM rates
  //    kept (0.85 ... 1.3: traced operations carry events between kernels,
  //    which the untraced step times do not), chosen together so that the
  //    simulated two-stream step times come closest to the measured ones
  auto sim = [&](const nf_plan_opts& o) {
    const bool window = o.executor == NF_EXEC_STREAMS && o.n_attn >= 2 && n_layers >= 2;
    return window ? simulate_window(m, o, n_layers) : simulate(m, o) * n_layers;
  };
  if (!r.rp_sms.empty()) {
    const std::vector<double> base = r.rp_gemm_factor;
    double best_sync = r.stream_sync_s, best_gamma = 1.0, best_err = -1;
    for (int gi = 85; gi <= 130; ++gi) {
      for (size_t i = 0; i < base.size(); ++i) r.rp_gemm_factor[i] = base[i] * gi * 0.01;
      for (int us = 0; us <= 100; us += 2) {
        r.stream_sync_s = us * 1e-6;
        double err = 0;
        for (size_t k = 1; k < runs.size(); ++k) {
          const double d = sim(runs[k].opts) * 1e3 / runs[k].step_ms - 1.0;
          err += d * d;
        }
        if (best_err < 0 || err < best_err) {
          best_err = err;
          best_sync = r.stream_sync_s;
          best_gamma = gi * 0.01;
        }
      }
    }
    r.stream_sync_s = best_sync;
    for (size_t i = 0; i < base.size(); ++i) r.rp_gemm_factor[i] = base[i] * best_gamma;
  }

  // JSON, with each run's measured and predicted step time
  std::string js = "{\n";
  char buf[512];
  auto num = [&](const char* k, double v) {
    std::snprintf(buf, sizeof(buf), "  \"%s\": %.9g,\n", k, v);
    js += buf;
  };
  auto arr = [&](const char* k, const std::vector<double>& v) {
    js += std::string("  \"") + k + "\": [";
    for (size_t i = 0; i < v.size(); ++i) {
      std::snprintf(buf, sizeof(buf), "%s%.9g", i ? ", " : "", v[i]);
      js += buf;
    }
    js += "],\n";
  };
  std::snprintf(buf, sizeof(buf),
                "  \"shape\": [%d, %d, %d, %d, %d, %d, %d, %d],\n  \"n_layers\": %d,\n  \"sms\": %d,\n",
                shape->hidden, shape->n_q_heads, shape->n_kv_heads, shape->head_dim, shape->ffn,
                shape->n_experts, shape->top_k, shape->page_size, n_layers, num_sms);
  js += buf;
  num("gemm_flops_per_sm", r.gemm_flops_per_sm);
  num("hbm_bps", r.hbm_bps);
  num("attn_bps_per_sm", r.attn_bps_per_sm);
  num("qkv_row_sm_s", r.qkv_row_sm_s);
  num("attn_prefill_flops_per_sm", r.attn_prefill_flops_per_sm);
  num("gemm_launch_s", r.gemm_launch_s);
  num("attn_launch_s", r.attn_launch_s);
  num("stream_sync_s", r.stream_sync_s);
  arr("rp_n", r.rp_n);
  arr("rp_sms", r.rp_sms);
  arr("rp_attn_bps_per_sm", r.rp_attn_bps_per_sm);
  arr("rp_gemm_factor", r.rp_gemm_factor);
  {
    std::vector<double> rn, rs, rm;
    for (const TracedRun& run : runs) {
      rn.push_back(run.opts.executor == NF_EXEC_STREAMS ? run.opts.n_attn : 1);
      rs.push_back(run.opts.executor == NF_EXEC_STREAMS ? run.opts.attn_sms : 0);
      rm.push_back(run.step_ms);
    }
    std::snprintf(buf, sizeof(buf), "  \"batch_tokens\": %d,\n  \"batch_decode\": %d,\n",
                  int(m.row_ctx.size()), batch->n_decode);
    js += buf;
    arr("run_n", rn);
    arr("run_sms", rs);
    arr("run_ms", rm);
  }
  js += "  \"runs\": [";
  for (size_t k = 0; k < runs.size(); ++k) {
    const nf_plan_opts& o = runs[k].opts;
    std::snprintf(buf, sizeof(buf),
                  "%s\n    {\"n_attn\": %d, \"n_ffn\": %d, \"attn_sms\": %d, \"measured_ms\": %.5g, "
                  "\"predicted_ms\": %.5g}",
                  k ? "," : "", o.n_attn, o.n_ffn, o.executor == NF_EXEC_STREAMS ? o.attn_sms : 0,
                  runs[k].step_ms, sim(o) * 1e3);
    js += buf;
  }
  js += "\n  ]\n}\n";
  return js;
}

}  // namespace nf

extern "C" nf_status nf_profile_use(const nf_model_shape* shape, const char* json_path) {
  if (!shape) return NF_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (size_t i = 0; i < g_profiles.size(); ++i)
    if (same_shape(g_profiles[i].first, *shape)) {
      if (json_path) g_profiles[i].second = json_path;
      else g_profiles.erase(g_profiles.begin() + static_cast<long>(i));
      return NF_OK;
    }
  if (json_path) g_profiles.push_back({*shape, std::string(json_path)});
  return NF_OK;
}

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
