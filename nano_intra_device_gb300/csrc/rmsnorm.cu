// RMSNorm rows of a [rows, hidden] bf16 matrix: out = x * g / sqrt(mean(x^2) + eps).
// Pre-norm of the decoder layer ("CSE 451 Lecture 25", slide 25, decoder-only
// transformer layer).  HBM-bound: one CTA per row, 16-byte loads, fp32 sums.
#include "common.cuh"
#include "kernels.h"
#include "tokmap.cuh"

namespace nf {

constexpr int RMS_THREADS = 128;

__global__ void __launch_bounds__(RMS_THREADS)
    rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ g,
                   __nv_bfloat16* __restrict__ out, int row_begin, int hidden, float eps,
                   const TokMap map, int with_map) {
  pdl_trigger();
  const int row = row_begin + blockIdx.x;
  if (with_map && threadIdx.x == RMS_THREADS - 32) {
    // RMSNorm-1: row `row` is token `row` of the step.  The first n_decode
    // sequences own one token each, so a decode row is its own sequence;
    // otherwise search the token starts.
    const int t = row;
    int s = -1;
    if (t < map.n_decode && t < map.n_seq && map.tok_begin[t] == t && map.tok_begin[t + 1] == t + 1)
      s = t;
    if (s < 0) s = tok_seq_search(map.tok_begin, 0, map.n_seq, t);
    const TokEntry e = token_entry(map, s, map.tok_begin[s], t, true);
    map.tok_seq[t] = s;
    map.tok_pos[t] = e.pos;
    map.tok_slot[t] = e.slot;
    map.tok_nchunks[t] = e.nch;
  }
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * hidden);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4* orow = reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * hidden);
  const int nvec = hidden / 8;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nvec; i += RMS_THREADS) {
    uint4 u = xr[i];
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16lo(w[j]), b = bf16hi(w[j]);
      ss += a * a + b * b;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  __shared__ float red[RMS_THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < RMS_THREADS / 32; ++i) tot += red[i];
  const float r = rsqrtf(tot / hidden + eps);
  for (int i = threadIdx.x; i < nvec; i += RMS_THREADS) {
    uint4 u = xr[i], gv = gr[i];
    uint32_t w[4] = {u.x, u.y, u.z, u.w}, gg[4] = {gv.x, gv.y, gv.z, gv.w}, o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16(bf16lo(w[j]) * r * bf16lo(gg[j]), bf16hi(w[j]) * r * bf16hi(gg[j]));
    orow[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* out,
                           int row_begin, int row_end, int hidden, float eps, cudaStream_t stream,
                           const TokMap* map) {
  if (row_end <= row_begin) return cudaSuccess;
  const TokMap m = map ? *map : TokMap{};
  rmsnorm_kernel<<<row_end - row_begin, RMS_THREADS, 0, stream>>>(x, g, out, row_begin, hidden,
                                                                   eps, m, map ? 1 : 0);
  return cudaGetLastError();
}

// Embedding lookup, one CTA per token: the row is copied with 16-byte accesses.
__global__ void __launch_bounds__(RMS_THREADS)
    embed_kernel(const int* __restrict__ tokens, const __nv_bfloat16* __restrict__ embed,
                 __nv_bfloat16* __restrict__ x, int hidden, int vocab, uint32_t* status) {
  const int t = blockIdx.x;
  const int id = tokens[t];
  uint4* dst = reinterpret_cast<uint4*>(x + static_cast<size_t>(t) * hidden);
  const int nvec = hidden / 8;
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) raise_status(status, ST_BAD_LEN);
    for (int i = threadIdx.x; i < nvec; i += RMS_THREADS) dst[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(embed + static_cast<size_t>(id) * hidden);
  for (int i = threadIdx.x; i < nvec; i += RMS_THREADS) dst[i] = src[i];
}

cudaError_t launch_embed(const int* tokens, const __nv_bfloat16* embed, __nv_bfloat16* x, int n_tok,
                         int hidden, int vocab, uint32_t* status, cudaStream_t stream) {
  if (n_tok <= 0) return cudaSuccess;
  embed_kernel<<<n_tok, RMS_THREADS, 0, stream>>>(tokens, embed, x, hidden, vocab, status);
  return cudaGetLastError();
}

}  // namespace nf
