// Split-KV merge shared by the attention kernels.
//
// A row whose history is cut into several pieces gets one partial record per
// (piece, KV head): the unnormalised output acc[GRP][d], then the reference
// maxima m[GRP] (base-2 logits) and the denominators l[GRP] = sum 2^(s - m).
// The warp that finishes a row's last piece combines the records by
// log-sum-exp: M = max_c m_c, w_c = 2^(m_c - M), o = sum_c w_c acc_c /
// sum_c w_c l_c.  This is exact: a softmax over the union of the pieces equals
// the rescaled combination of the pieces' own exponentials and sums.  The
// records are read in piece order, so the result does not depend on which warp
// finished last.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace nf {

// Lane (ts = lane / 8, dg = lane % 8) handles the heads h with h % 4 == ts and
// the dims ch * 64 + dg * 8 .. + 7 of each.
template <int GRP, int NCH>
__device__ __forceinline__ void merge_row_partials(const AttnArgs& a, int t, int g, int nch,
                                                   int lane) {
  constexpr int D = NCH * 64;
  constexpr int REC = partial_rec_floats(GRP, D);
  const int ts = lane >> 3, dg = lane & 7;
  const size_t row_rec = static_cast<size_t>(t) * a.max_chunks;
  const int n_kv = a.n_kv;
#pragma unroll
  for (int h = 0; h < GRP; ++h) {
    if ((h & 3) != ts) continue;
    float M = -INFINITY;
    for (int cc = 0; cc < nch; ++cc) {
      const float* r = a.partials + ((row_rec + cc) * n_kv + g) * REC;
      M = fmaxf(M, __ldcg(r + GRP * D + h));
    }
    float L = 0.f, O[NCH * 8];
#pragma unroll
    for (int e = 0; e < NCH * 8; ++e) O[e] = 0.f;
    for (int cc = 0; cc < nch; ++cc) {
      const float* r = a.partials + ((row_rec + cc) * n_kv + g) * REC;
      const float w = exp2f(__ldcg(r + GRP * D + h) - M);
      L += w * __ldcg(r + GRP * D + GRP + h);
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const float4* src = reinterpret_cast<const float4*>(r + h * D + ch * 64 + dg * 8);
        const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
        O[ch * 8 + 0] += w * x0.x; O[ch * 8 + 1] += w * x0.y;
        O[ch * 8 + 2] += w * x0.z; O[ch * 8 + 3] += w * x0.w;
        O[ch * 8 + 4] += w * x1.x; O[ch * 8 + 5] += w * x1.y;
        O[ch * 8 + 6] += w * x1.z; O[ch * 8 + 7] += w * x1.w;
      }
    }
    const float inv = 1.f / L;
    __nv_bfloat16* orow = a.o + (static_cast<size_t>(t) * a.n_q + g * GRP + h) * D;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      uint4 u;
      u.x = pack_bf16(O[ch * 8 + 0] * inv, O[ch * 8 + 1] * inv);
      u.y = pack_bf16(O[ch * 8 + 2] * inv, O[ch * 8 + 3] * inv);
      u.z = pack_bf16(O[ch * 8 + 4] * inv, O[ch * 8 + 5] * inv);
      u.w = pack_bf16(O[ch * 8 + 6] * inv, O[ch * 8 + 7] * inv);
      *reinterpret_cast<uint4*>(orow + ch * 64 + dg * 8) = u;
    }
  }
}

// Publish-and-count step after a piece wrote its record: returns true (to every
// lane) in the warp that completed the row's last piece.
__device__ __forceinline__ bool finish_piece(const AttnArgs& a, int t, int g, int nch, int lane) {
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&a.row_done[t * a.n_kv + g], 1) == nch - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

}  // namespace nf
