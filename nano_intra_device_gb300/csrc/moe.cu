// Mixture-of-experts FFN plumbing around the grouped tensor-core GEMM: gate
// routing, the expert-grouped row order, the row gather and the weighted
// combine ("NanoFlow: Towards Optimal LLM Serving Throughput", MoE models: gate
// routing, then a grouped GEMM in which different experts compute on different
// tokens).
//
// Routing reading (the pages name only "gate routing"): each token takes the
// top_k experts by router logit, ties going to the lower expert index, weighted
// by a softmax over the selected logits.  The grouped order is expert by expert
// and, within an expert, by increasing token: a stable counting sort, so the
// integer outputs are bit-exact and independent of thread timing.
#include "common.cuh"
#include "kernels.h"

namespace nf {

constexpr int ROUTE_THREADS = 1024;
constexpr int ROUTE_MAX_K = 2;

// Exclusive prefix sum over the block of one int per thread; returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) warp_sums[lane] = wi - w;  // exclusive prefix of each warp
    if (lane == nw - 1) *total = wi;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();  // warp_sums is reused by the next scan
  return r;
}

__global__ void __launch_bounds__(ROUTE_THREADS) moe_route_kernel(
    const float* __restrict__ logits, int r0, int n, int E, int k, int* group_off,
    int* perm_tok, int* pair_row, float* pair_w) {
  __shared__ int warp_sums[32];
  __shared__ int total;
  const int pairs = n * k;
  // pass 1: each token's experts (best first) into pair_row as scratch
  for (int i = threadIdx.x; i < n; i += ROUTE_THREADS) {
    const float* r = logits + static_cast<size_t>(r0 + i) * E;
    int e0 = 0;
    float l0 = r[0];
    for (int e = 1; e < E; ++e)
      if (r[e] > l0) {  // strict: an equal logit keeps the lower index
        l0 = r[e];
        e0 = e;
      }
    if (k == 1) {
      pair_row[i] = e0;
      pair_w[i] = 1.0f;
    } else {
      int e1 = -1;
      float l1 = 0.f;
      for (int e = 0; e < E; ++e)
        if (e != e0 && (e1 < 0 || r[e] > l1)) {
          l1 = r[e];
          e1 = e;
        }
      // softmax over (l0, l1) with l0 >= l1: w0 = 1 / (1 + 2^((l1 - l0) log2 e))
      const float w0 = 1.0f / (1.0f + exp2f((l1 - l0) * 1.4426950408889634f));
      pair_row[2 * i] = e0;
      pair_row[2 * i + 1] = e1;
      pair_w[2 * i] = w0;
      pair_w[2 * i + 1] = 1.0f - w0;
    }
  }
  __syncthreads();
  // pass 2: stable grouping.  Thread j owns the contiguous pairs
  // [j * per, (j + 1) * per); for each expert a block scan of the owners'
  // counts gives every pair its row.
  const int per = (pairs + ROUTE_THREADS - 1) / ROUTE_THREADS;
  const int p0 = min(pairs, threadIdx.x * per), p1 = min(pairs, p0 + per);
  int exp_of[16];  // per <= 16 (pairs <= 16384): the experts of the owned pairs
#pragma unroll
  for (int q = 0; q < 16; ++q) exp_of[q] = (p0 + q < p1) ? pair_row[p0 + q] : -1;
  __syncthreads();  // every read of pair_row happens before it is overwritten below
  int base = 0;
  for (int e = 0; e < E; ++e) {
    int c = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) c += exp_of[q] == e;
    const int pre = block_exclusive_scan(c, warp_sums, &total);
    if (threadIdx.x == 0) group_off[e] = base;
    int at = base + pre;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (exp_of[q] == e) {
        const int p = p0 + q;
        perm_tok[at] = r0 + p / k;
        pair_row[p] = at;
        ++at;
      }
    base += total;
    __syncthreads();  // `total` is rewritten by the next scan
  }
  if (threadIdx.x == 0) group_off[E] = base;
}

cudaError_t launch_moe_route(const float* logits, int r0, int n, int n_experts, int top_k,
                             int* group_off, int* perm_tok, int* pair_row, float* pair_w,
                             cudaStream_t stream) {
  if (n < 0 || n_experts < 1 || n_experts > GEMM_MAX_GROUPS || top_k < 1 ||
      top_k > ROUTE_MAX_K || top_k > n_experts || n * top_k > 16 * ROUTE_THREADS)
    return cudaErrorInvalidValue;
  moe_route_kernel<<<1, ROUTE_THREADS, 0, stream>>>(logits, r0, n, n_experts, top_k, group_off,
                                                    perm_tok, pair_row, pair_w);
  return cudaGetLastError();
}

__global__ void gather_rows_kernel(const uint4* __restrict__ src, const int* __restrict__ perm_tok,
                                   uint4* __restrict__ dst, int rows, int vec_per_row, int src_rows,
                                   uint32_t* status) {
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int from = perm_tok[row];
    uint4* d = dst + static_cast<size_t>(row) * vec_per_row;
    if (from < 0 || from >= src_rows) {  // never read outside src: a zero row, flagged
      if (threadIdx.x == 0) raise_status(status, ST_BAD_LEN);
      for (int i = threadIdx.x; i < vec_per_row; i += blockDim.x) d[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* s = src + static_cast<size_t>(from) * vec_per_row;
    for (int i = threadIdx.x; i < vec_per_row; i += blockDim.x) d[i] = s[i];
  }
}

cudaError_t launch_gather_rows(const __nv_bfloat16* src, const int* perm_tok, __nv_bfloat16* dst,
                               int rows, int cols, int src_rows, uint32_t* status,
                               cudaStream_t stream) {
  if (cols % 8 || rows < 0) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  const int grid = rows < 2048 ? rows : 2048;
  gather_rows_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(src), perm_tok,
                                               reinterpret_cast<uint4*>(dst), rows, cols / 8,
                                               src_rows, status);
  return cudaGetLastError();
}

__global__ void moe_combine_kernel(const __nv_bfloat16* __restrict__ h,
                                   const float* __restrict__ part,
                                   const int* __restrict__ pair_row,
                                   const float* __restrict__ pair_w, __nv_bfloat16* __restrict__ y,
                                   int r0, int n, int k, int hidden) {
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const size_t t = static_cast<size_t>(r0 + i);
    for (int c = threadIdx.x * 4; c < hidden; c += blockDim.x * 4) {
      const uint2 hv = *reinterpret_cast<const uint2*>(h + t * hidden + c);
      float acc[4] = {bf16lo(hv.x), bf16hi(hv.x), bf16lo(hv.y), bf16hi(hv.y)};
      for (int j = 0; j < k; ++j) {
        const float w = pair_w[i * k + j];
        const float4 pv =
            *reinterpret_cast<const float4*>(part + static_cast<size_t>(pair_row[i * k + j]) * hidden + c);
        acc[0] += w * pv.x;
        acc[1] += w * pv.y;
        acc[2] += w * pv.z;
        acc[3] += w * pv.w;
      }
      uint2 o;
      o.x = pack_bf16(acc[0], acc[1]);
      o.y = pack_bf16(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(y + t * hidden + c) = o;
    }
  }
}

cudaError_t launch_moe_combine(const __nv_bfloat16* h, const float* part, const int* pair_row,
                               const float* pair_w, __nv_bfloat16* y, int r0, int n, int top_k,
                               int hidden, cudaStream_t stream) {
  if (hidden % 4 || n < 0) return cudaErrorInvalidValue;
  if (n == 0) return cudaSuccess;
  const int grid = n < 4096 ? n : 4096;
  moe_combine_kernel<<<grid, 256, 0, stream>>>(h, part, pair_row, pair_w, y, r0, n, top_k, hidden);
  return cudaGetLastError();
}

}  // namespace nf
