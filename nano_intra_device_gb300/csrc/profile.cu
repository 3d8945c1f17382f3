// Offline profiler of the layer's nano-operations ("NanoFlow: Towards Optimal
// LLM Serving Throughput", "Kernel Profiling and Interference Modeling").
//
// What it measures on the current device, with synthetic data of the given
// layer shape:
//  * interference-free time of each GEMM of the layer (QKV, O, gate/up with
//    SwiGLU, down) at token counts that are multiples of 128 (the pages'
//    profiling grid), on the whole GPU;
//  * the per-SM tensor rate of a GEMM confined to S SMs;
//  * the bandwidth of paged decode attention confined to S SMs, alone;
//  * the same attention while a GEMM runs on the remaining SMs, and that
//    GEMM's slowdown: the measured counterpart of the pages' R -> P table,
//    with the resource share R expressed as an SM count.
// The JSON it writes is what nf_plan_search reads.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <string>
#include <vector>

#include "../../include/nanoflow.h"
#include "common.cuh"
#include "internal.h"

namespace {

__global__ void fill_bf16(__nv_bfloat16* p, size_t n, uint32_t seed, float scale) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B1u ^ seed;
    h ^= h >> 15;
    h *= 0x85EBCA77u;
    h ^= h >> 13;
    h *= 0xC2B2AE3Du;
    h ^= h >> 16;
    const float u = (h >> 8) * (1.0f / 16777216.0f) * 2.0f - 1.0f;
    p[i] = __float2bfloat16(u * scale);
  }
}

struct Bufs {
  std::vector<void*> all;
  ~Bufs() {
    for (void* p : all) cudaFree(p);
  }
  template <typename T>
  T* get(size_t bytes) {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return nullptr;
    all.push_back(p);
    return static_cast<T*>(p);
  }
};

template <typename F>
double time_ms(F&& fn, cudaStream_t st, int reps) {
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  fn();
  fn();
  std::vector<float> t;
  for (int r = 0; r < reps; ++r) {
    cudaEventRecord(a, st);
    fn();
    cudaEventRecord(b, st);
    cudaEventSynchronize(b);
    float ms = 0;
    cudaEventElapsedTime(&ms, a, b);
    t.push_back(ms);
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  std::sort(t.begin(), t.end());
  return t[t.size() / 2];
}

}  // namespace

extern "C" nf_status nf_profile(const nf_model_shape* shape, int32_t max_tokens, int32_t mean_ctx,
                                const char* out_json) {
  if (!shape || !out_json || max_tokens < 128 || mean_ctx < 1) return NF_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return NF_ERR_CUDA;
  const nf_model_shape& s = *shape;
  const int T = max_tokens / 128 * 128;
  const int H = s.hidden, F = s.ffn, QD = s.n_q_heads * s.head_dim;
  const int NQKV = (s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim;
  const int P = s.page_size;
  const int npp = (mean_ctx + P - 1) / P;
  const size_t num_pages = (size_t)T * npp;
  const size_t page_elems = (size_t)s.n_kv_heads * P * s.head_dim;
  const int KMAX = std::max(H, std::max(F, QD));
  const int NMAX = std::max(std::max(NQKV, H), F);

  Bufs B;
  auto* A = B.get<__nv_bfloat16>((size_t)T * KMAX * 2);
  auto* W = B.get<__nv_bfloat16>((size_t)2 * NMAX * KMAX * 2);
  auto* C = B.get<__nv_bfloat16>((size_t)T * NMAX * 2);
  auto* R = B.get<__nv_bfloat16>((size_t)T * NMAX * 2);
  auto* kp = B.get<__nv_bfloat16>(num_pages * page_elems * 2);
  auto* vp = B.get<__nv_bfloat16>(num_pages * page_elems * 2);
  auto* q = B.get<__nv_bfloat16>((size_t)T * QD * 2);
  auto* o = B.get<__nv_bfloat16>((size_t)T * QD * 2);
  auto* bt = B.get<int32_t>((size_t)T * npp * 4);
  auto* sl = B.get<int32_t>((size_t)T * 4);
  if (!A || !W || !C || !R || !kp || !vp || !q || !o || !bt || !sl) return NF_ERR_OOM;
  fill_bf16<<<1024, 256>>>(A, (size_t)T * KMAX, 1, 1.0f);
  fill_bf16<<<1024, 256>>>(W, (size_t)2 * NMAX * KMAX, 2, 0.03f);
  fill_bf16<<<1024, 256>>>(R, (size_t)T * NMAX, 3, 1.0f);
  fill_bf16<<<4096, 256>>>(kp, num_pages * page_elems, 4, 1.0f);
  fill_bf16<<<4096, 256>>>(vp, num_pages * page_elems, 5, 1.0f);
  fill_bf16<<<1024, 256>>>(q, (size_t)T * QD, 6, 1.0f);
  {
    std::vector<int32_t> hbt((size_t)T * npp), hsl(T, mean_ctx);
    // an affine permutation of the page ids (multiplier coprime with the count)
    size_t mul = 2654435761ull % num_pages;
    auto gcd = [](size_t a, size_t b) { while (b) { size_t t = a % b; a = b; b = t; } return a; };
    while (mul < 2 || gcd(mul, num_pages) != 1) mul = (mul + 1) % num_pages;
    for (size_t i = 0; i < hbt.size(); ++i) hbt[i] = (int32_t)((i * mul + 7) % num_pages);
    cudaMemcpy(bt, hbt.data(), hbt.size() * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(sl, hsl.data(), hsl.size() * 4, cudaMemcpyHostToDevice);
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return NF_ERR_CUDA;

  nf_batch_desc bd{};
  bd.n_decode = T;
  bd.max_pages_per_seq = npp;
  bd.num_pages = (int32_t)std::min<size_t>(num_pages, 0x7fffffff);
  nf_plan_opts po{};
  po.n_attn = 1;
  po.attn_bounds[1] = T;
  po.n_ffn = 1;
  po.ffn_bounds[1] = T;
  po.kv_chunk = 512;
  po.timeout_ns = 2000000000LL;
  nf_plan plan = nullptr;
  nf_status st = nf_plan_create(shape, &bd, &po, &plan);
  if (st != NF_OK) return st;

  cudaStream_t sa, sg;
  cudaStreamCreateWithFlags(&sa, cudaStreamNonBlocking);
  cudaStreamCreateWithFlags(&sg, cudaStreamNonBlocking);
  std::string js = "{\n";
  char buf[512];
  auto add = [&](const char* k, double v) {
    std::snprintf(buf, sizeof(buf), "  \"%s\": %.9g,\n", k, v);
    js += buf;
  };

  // 1) interference-free GEMM times per token count
  struct Op {
    const char* name;
    int N, K, epi;
  } ops[] = {{"qkv", NQKV, H, NF_EPI_STORE},
             {"oproj", H, QD, NF_EPI_RESID},
             {"gate_up", F, H, NF_EPI_SWIGLU},
             {"down", H, F, NF_EPI_RESID}};
  js += "  \"gemm_ms\": {\n";
  for (int oi = 0; oi < 4; ++oi) {
    const Op& op = ops[oi];
    js += std::string("    \"") + op.name + "\": [";
    bool first = true;
    for (int m = 128; m <= T; m += 128) {
      const double ms = time_ms([&] { nf_gemm(A, W, C, R, m, op.N, op.K, op.epi, 0, sa); }, sa, 5);
      std::snprintf(buf, sizeof(buf), "%s[%d, %.6g]", first ? "" : ", ", m, ms);
      js += buf;
      first = false;
    }
    js += oi == 3 ? "]\n" : "],\n";
  }
  js += "  },\n";

  // 2) per-SM tensor rate of the gate/up GEMM on S SMs
  double rate_sum = 0;
  int rate_n = 0;
  js += "  \"gemm_rate_by_sms\": [";
  for (int k = 1; k <= 4; ++k) {
    const int S = sms * k / 4;
    const double ms = time_ms([&] { nf_gemm(A, W, C, nullptr, T, F, H, NF_EPI_SWIGLU, S, sa); }, sa, 5);
    const double fl = 2.0 * T * (2.0 * F) * H;
    const double per_sm = fl / (ms * 1e-3) / S;
    rate_sum += per_sm;
    ++rate_n;
    std::snprintf(buf, sizeof(buf), "%s[%d, %.6g]", k == 1 ? "" : ", ", S, per_sm);
    js += buf;
  }
  js += "],\n";
  add("gemm_flops_per_sm", rate_sum / rate_n);

  // 3) attention alone on S SMs
  const double kv_bytes = (double)T * mean_ctx * 2.0 * s.n_kv_heads * s.head_dim * 2.0;
  std::vector<std::pair<int, double>> abw;
  js += "  \"attn_gbs_by_sms\": [";
  for (int S = 16; S <= sms; S += 16) {
    const double ms = time_ms([&] { nf::attention_on(plan, q, kp, vp, bt, sl, o, S, sa); }, sa, 5);
    abw.push_back({S, kv_bytes / (ms * 1e-3)});
    std::snprintf(buf, sizeof(buf), "%s[%d, %.6g]", S == 16 ? "" : ", ", S, kv_bytes / (ms * 1e-3) / 1e9);
    js += buf;
  }
  {
    const double ms = time_ms([&] { nf::attention_on(plan, q, kp, vp, bt, sl, o, sms, sa); }, sa, 5);
    abw.push_back({sms, kv_bytes / (ms * 1e-3)});
    std::snprintf(buf, sizeof(buf), ", [%d, %.6g]", sms, kv_bytes / (ms * 1e-3) / 1e9);
    js += buf;
  }
  js += "],\n";
  double hbm = 0;
  for (auto& e : abw) hbm = std::max(hbm, e.second);
  add("hbm_bps", hbm);
  add("attn_bps_per_sm", abw.front().second / abw.front().first);

  // 4) attention beside a GEMM on the other SMs (the measured R -> P table),
  //    and the GEMM's slowdown as a function of the share u of HBM bandwidth
  //    the attention draws: 1 - p_gemm = c u^2, c fitted by least squares
  js += "  \"overlap\": [";
  double fac_sum = 0, gfac_sum = 0, fit_num = 0, fit_den = 0;
  int fac_n = 0;
  for (int k = 2; k <= 6; ++k) {
    const int Sa = sms * k / 8, Sg = sms - Sa;
    const double alone_a = time_ms([&] { nf::attention_on(plan, q, kp, vp, bt, sl, o, Sa, sa); }, sa, 3);
    const double alone_g = time_ms([&] { nf_gemm(A, W, C, nullptr, T, F, H, NF_EPI_SWIGLU, Sg, sg); }, sg, 3);
    // keep the GEMM stream busy for the whole attention launch
    const int reps = std::max(2, (int)std::ceil(alone_a / alone_g) + 2);
    cudaEvent_t a0, a1, g0, g1;
    cudaEventCreate(&a0);
    cudaEventCreate(&a1);
    cudaEventCreate(&g0);
    cudaEventCreate(&g1);
    cudaEventRecord(g0, sg);
    for (int r = 0; r < reps; ++r) nf_gemm(A, W, C, nullptr, T, F, H, NF_EPI_SWIGLU, Sg, sg);
    cudaEventRecord(g1, sg);
    cudaEventRecord(a0, sa);
    nf::attention_on(plan, q, kp, vp, bt, sl, o, Sa, sa);
    cudaEventRecord(a1, sa);
    cudaDeviceSynchronize();
    float ta = 0, tg = 0;
    cudaEventElapsedTime(&ta, a0, a1);
    cudaEventElapsedTime(&tg, g0, g1);
    cudaEventDestroy(a0);
    cudaEventDestroy(a1);
    cudaEventDestroy(g0);
    cudaEventDestroy(g1);
    const double p_attn = alone_a / ta;
    const double p_gemm = alone_g * reps / tg;
    const double u = std::min(1.0, kv_bytes / (ta * 1e-3) / hbm);
    fac_sum += p_attn;
    gfac_sum += p_gemm;
    fit_num += (1.0 - p_gemm) * u * u;
    fit_den += u * u * u * u;
    ++fac_n;
    std::snprintf(buf, sizeof(buf),
                  "%s{\"attn_sms\": %d, \"gemm_sms\": %d, \"attn_alone_ms\": %.5g, "
                  "\"attn_overlap_ms\": %.5g, \"p_attn\": %.4g, \"p_gemm\": %.4g, \"u\": %.4g}",
                  k == 2 ? "" : ", ", Sa, Sg, alone_a, (double)ta, p_attn, p_gemm, u);
    js += buf;
  }
  js += "],\n";
  add("overlap_bw_factor", fac_sum / fac_n);
  add("overlap_gemm_factor", gfac_sum / fac_n);
  add("gemm_interference", fit_den > 0 ? std::max(0.0, fit_num / fit_den) : 0.62);
  // launch cost: a one-tile GEMM
  add("gemm_launch_s", time_ms([&] { nf_gemm(A, W, C, nullptr, 128, 256, 64, 0, 0, sa); }, sa, 9) * 1e-3);
  add("attn_launch_s", 4e-6);
  std::snprintf(buf, sizeof(buf), "  \"sms\": %d,\n  \"max_tokens\": %d,\n  \"mean_ctx\": %d\n}\n",
                sms, T, mean_ctx);
  js += buf;

  cudaStreamDestroy(sa);
  cudaStreamDestroy(sg);
  nf_plan_destroy(plan);
  if (cudaDeviceSynchronize() != cudaSuccess) return NF_ERR_CUDA;
  FILE* f = std::fopen(out_json, "w");
  if (!f) return NF_ERR_INVALID_ARG;
  std::fputs(js.c_str(), f);
  std::fclose(f);
  return NF_OK;
}
