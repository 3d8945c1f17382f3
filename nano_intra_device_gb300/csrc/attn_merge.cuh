// Split-KV merge shared by the attention kernels.
//
// A row whose history is cut into several pieces gets one partial record per
// (piece, KV head): the unnormalised output acc[GRP][d], then the reference
// maxima m[GRP] (base-2 logits) and the denominators l[GRP] = sum 2^(s - m).
// The warp that finishes a row's last piece combines the records by
// log-sum-exp: M = max_c m_c, w_c = 2^(m_c - M), o = sum_c w_c acc_c /
// sum_c w_c l_c.  This is exact: a softmax over the union of the pieces equals
// the rescaled combination of the pieces' own exponentials and sums.  The
// combination order is fixed (records in piece order, lanes in a fixed
// shuffle tree), so the result does not depend on which warp finished last.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace nf {

// Lane (ts = lane / 8, dg = lane % 8) handles the heads h with h % 4 == ts and
// the dims ch * 64 + dg * 8 .. + 7 of each.  Latency, not bandwidth, bounds a
// merge (a long row has dozens of records and one warp merges them), so the
// loads are batched: the maxima and denominators with the lanes over the
// records (one round trip per 32 records), then the accumulators MB records
// at a time.  Sums stay in record order.
// MB: records per batch of accumulator loads (MB x heads per lane x NCH x 2
// float4 registers): 4 where the kernel has registers to spare, else 2.
template <int GRP, int NCH, int MB = 2>
__device__ __forceinline__ void merge_row_partials(const AttnArgs& a, int t, int g, int nch,
                                                   int lane) {
  constexpr int D = NCH * 64;
  constexpr int REC = partial_rec_floats(GRP, D);
  constexpr int HPL = (GRP + 3) / 4;                // heads per lane
  const int ts = lane >> 3, dg = lane & 7;
  const size_t cstride = static_cast<size_t>(a.n_kv) * REC;  // from one record of the row to the next
  const float* rec0 = a.partials + (static_cast<size_t>(t) * a.max_chunks * a.n_kv + g) * REC;
  // 1) per head: M = max_c m_c and L = sum_c 2^(m_c - M) l_c, lanes over records c,
  //    each lane folding its records (in order) into (M, L), then a fixed
  //    shuffle tree combining the lanes
  float Mh[GRP], Lh[GRP];
#pragma unroll
  for (int h = 0; h < GRP; ++h) {
    float M = -INFINITY, L = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const float* r = rec0 + c * cstride;
      const float m = __ldcg(r + GRP * D + h), l = __ldcg(r + GRP * D + GRP + h);
      const float nM = fmaxf(M, m);
      L = L * exp2f(M - nM) + l * exp2f(m - nM);
      M = nM;
    }
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o_);
      const float L2 = __shfl_xor_sync(0xffffffffu, L, o_);
      const float nM = fmaxf(M, M2);
      // a lane without records holds (-inf, 0): its term is 0
      L = (M == -INFINITY ? 0.f : L * exp2f(M - nM)) + (M2 == -INFINITY ? 0.f : L2 * exp2f(M2 - nM));
      M = nM;
    }
    Mh[h] = M;
    Lh[h] = L;
  }
  // 2) o = sum_c w_c acc_c / L with w_c = 2^(m_c - M): lane j of a group of 32
  //    records holds their weights; accumulators in record order
  float O[HPL][NCH * 8];
#pragma unroll
  for (int k = 0; k < HPL; ++k)
#pragma unroll
    for (int e = 0; e < NCH * 8; ++e) O[k][e] = 0.f;
  for (int c32 = 0; c32 < nch; c32 += 32) {
    float wl[GRP];  // weights of record c32 + lane, per head
    {
      const int c = c32 + lane;
      const float* r = rec0 + (c < nch ? c : 0) * cstride;
#pragma unroll
      for (int h = 0; h < GRP; ++h)
        wl[h] = c < nch ? exp2f(__ldcg(r + GRP * D + h) - Mh[h]) : 0.f;
    }
    const int cn = min(32, nch - c32);
    for (int j0 = 0; j0 < cn; j0 += MB) {
      float4 x[MB][HPL][2 * NCH];
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        const float* r = rec0 + (c32 + min(j0 + j, cn - 1)) * cstride;
#pragma unroll
        for (int k = 0; k < HPL; ++k) {
          const int h = ts + 4 * k;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            const float4* src =
                reinterpret_cast<const float4*>(r + (h < GRP ? h : 0) * D + ch * 64 + dg * 8);
            x[j][k][2 * ch] = __ldcg(src);
            x[j][k][2 * ch + 1] = __ldcg(src + 1);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        float w[HPL];
#pragma unroll
        for (int k = 0; k < HPL; ++k) w[k] = 0.f;
#pragma unroll
        for (int h = 0; h < GRP; ++h) {  // every lane shuffles every head; keeps its own
          const float wh = __shfl_sync(0xffffffffu, wl[h], (j0 + j) & 31);
          if ((h & 3) == ts) w[h >> 2] = wh;
        }
        if (j0 + j < cn) {
#pragma unroll
          for (int k = 0; k < HPL; ++k)
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              const float4 u = x[j][k][2 * ch], v = x[j][k][2 * ch + 1];
              float* o = O[k] + ch * 8;
              o[0] += w[k] * u.x; o[1] += w[k] * u.y; o[2] += w[k] * u.z; o[3] += w[k] * u.w;
              o[4] += w[k] * v.x; o[5] += w[k] * v.y; o[6] += w[k] * v.z; o[7] += w[k] * v.w;
            }
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < HPL; ++k) {
    const int h = ts + 4 * k;
    if (h >= GRP) continue;
    float Lsel = 1.f;  // Lh[h] with h lane-dependent: selected, not indexed (no local array)
#pragma unroll
    for (int hh = 0; hh < GRP; ++hh)
      if (hh == h) Lsel = Lh[hh];
    const float inv = 1.f / Lsel;
    __nv_bfloat16* orow = a.o + (static_cast<size_t>(t) * a.n_q + g * GRP + h) * D;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      const float* o = O[k] + ch * 8;
      uint4 u;
      u.x = pack_bf16(o[0] * inv, o[1] * inv);
      u.y = pack_bf16(o[2] * inv, o[3] * inv);
      u.z = pack_bf16(o[4] * inv, o[5] * inv);
      u.w = pack_bf16(o[6] * inv, o[7] * inv);
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
