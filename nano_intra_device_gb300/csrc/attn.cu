// Paged GQA attention over the KV cache, split-KV, one warp per work piece.
//
// Decode attention is the step's memory-bound operation: each request streams
// its own K/V history, which no other token shares ("NanoFlow: Towards Optimal
// LLM Serving Throughput", "The Intra-Device Parallelism Mechanism"; "LLM
// Inference Performance", "PagedAttention: virtual memory for the KV cache").
// Every token of the batch (decode or prefill) is a query row: row t of
// sequence s at position p attends to positions 0..p of s, read through the
// block table.
//
// Work: a piece = (row, chunk of kv_chunk positions, KV head).  The kernel is
// persistent; each warp fetches pieces from a per-nano-batch counter, so a
// grid of S CTAs (one per SM) is the SM share of the nano-operation.
// Per piece the warp:
//   * stages each (page, KV head) block of K and of V (P x d bf16, contiguous)
//     into shared memory with 1-D bulk copies (TMA engine), STAGES pages in
//     flight per warp, completion on an mbarrier;
//   * lane (ts = lane/8, dg = lane%8) owns tokens ts, ts+4, ts+8, ts+12 of a
//     page and the 8*NCH dims {ch*64 + dg*8 ...}: 16-byte, conflict-free loads;
//     all GRP query heads of the KV group share every K/V read;
//   * scores are reduced over dg with three xor-shuffles, then an online
//     softmax (running max and sum, base 2) per page;
//   * a piece that is a row's only chunk writes o directly; otherwise it
//     writes (acc, m, l) and the warp that finishes the row's last piece merges
//     them by log-sum-exp.
#include "attn_merge.cuh"
#include "common.cuh"
#include "kernels.h"

namespace nf {

constexpr int ATT_P = 16;              // page size the kernel is built for
constexpr int ATT_MIN_SMEM = 120 * 1024;  // > half an SM: one CTA per SM
constexpr int ATT_MAX_PIECE_PAGES = 2048 / ATT_P;  // longest split-KV piece, in pages

int attn_partial_floats(int n_q, int n_kv, int head_dim) {
  return partial_rec_floats(n_q / n_kv, head_dim);
}

// Dynamic shared memory of an attention CTA: per warp its ring, barriers and
// page-id list.  `share` configurations leave room for one GEMM CTA (two ring
// stages) on the same SM; the 4-warp one is padded past half an SM so that two
// attention CTAs never pair up on one SM instead.
static int attn_smem_bytes_cfg(int head_dim, int page_size, int warps, int stages, bool share) {
  const int blk = page_size * head_dim * 2;
  const int need = warps * (stages * 2 * blk + stages * 8 + ATT_MAX_PIECE_PAGES * 4) + 128;
  if (!share) return need < ATT_MIN_SMEM ? ATT_MIN_SMEM : need;
  const int half_sm = 117 * 1024;
  return (warps == 4 && need < half_sm) ? half_sm : need;
}

// 8*NCH bf16 of one row -> NCH*4 fp32 pairs (dims ch*64 + dg*8 + 0..7).
template <int NCH>
__device__ __forceinline__ void load_row_pairs(const uint8_t* base, int dg,
                                               float2 (&out)[NCH * 4]) {
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const uint4 u = *reinterpret_cast<const uint4*>(base + (ch * 64 + dg * 8) * 2);
    out[ch * 4 + 0] = make_float2(bf16lo(u.x), bf16hi(u.x));
    out[ch * 4 + 1] = make_float2(bf16lo(u.y), bf16hi(u.y));
    out[ch * 4 + 2] = make_float2(bf16lo(u.z), bf16hi(u.z));
    out[ch * 4 + 3] = make_float2(bf16lo(u.w), bf16hi(u.w));
  }
}

template <int GRP, int NCH, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32, 1) attn_kernel(const AttnArgs a) {
  constexpr int D = NCH * 64;
  constexpr int P = ATT_P;
  constexpr int BLK = P * D * 2;  // bytes of one (page, KV head) block
  constexpr int E2 = NCH * 4;     // dim pairs per lane
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ts = lane >> 3, dg = lane & 7;
  uint8_t* ring = smem + warp * (STAGES * 2 * BLK);
  uint64_t* bar =
      reinterpret_cast<uint64_t*>(smem + WARPS * STAGES * 2 * BLK) + warp * STAGES;
  int* wpages = reinterpret_cast<int*>(smem + WARPS * STAGES * 2 * BLK + WARPS * STAGES * 8) +
                warp * ATT_MAX_PIECE_PAGES;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int seg = a.seg;
  const int begin = a.seg_items[seg];
  const int total = (a.seg_items[seg + 1] - begin) * a.n_kv;
  const int n_kv = a.n_kv, n_q = a.n_q, C = a.kv_chunk;
  const size_t page_stride = static_cast<size_t>(n_kv) * P * D;  // elements per page
  const uint64_t policy = l2_policy_evict_first();
  uint32_t gk = 0;  // pages this warp has consumed (ring position)
  bool failed = false;

  // the next piece is claimed one piece ahead, so the atomic's latency hides
  // behind the current piece
  int next_idx = 0;
  if (lane == 0) next_idx = atomicAdd(&a.fetch[seg], 1);
  for (;;) {
    const int idx = __shfl_sync(0xffffffffu, next_idx, 0);
    if (idx >= total) break;
    if (lane == 0) next_idx = atomicAdd(&a.fetch[seg], 1);
    const int pair = begin + idx / n_kv, g = idx % n_kv;
    const int t = a.items[2 * pair], c = a.items[2 * pair + 1];
    const int s = a.tok_seq[t];
    const int ctx = a.tok_pos[t] + 1;
    const int b0 = c * C;
    const int n = min(C, ctx - b0);
    const int npg = (n + P - 1) / P;
    // the piece's page ids, checked once and kept in shared memory for issue()
    {
      const int* bt = a.block_table + static_cast<size_t>(s) * a.max_pages + b0 / P;
      for (int i = lane; i < npg; i += 32) {
        int page = bt[i];
        if (page < 0 || page >= a.num_pages) {  // never read outside the pool
          raise_status(a.status, ST_BAD_PAGE);
          page = 0;
        }
        wpages[i] = page;
      }
      __syncwarp();
    }

    auto issue = [&](int k) {
      const uint32_t st = (gk + k) % STAGES;
      const size_t off =
          static_cast<size_t>(wpages[k]) * page_stride + static_cast<size_t>(g) * P * D;
      uint8_t* kb = ring + st * 2 * BLK;
      mbar_arrive_expect_tx(&bar[st], 2 * BLK);
      bulk_g2s_evict_first(kb, a.k_pool + off, BLK, &bar[st], policy);
      bulk_g2s_evict_first(kb + BLK, a.v_pool + off, BLK, &bar[st], policy);
    };
    int issued = 0;  // pages of this piece whose copies were started (lane 0)
    if (lane == 0) {
      const int pre = npg < STAGES ? npg : STAGES;
      for (int k = 0; k < pre; ++k) issue(k);
      issued = pre;
    }

    // q of the GRP heads of this KV group, scaled to base-2 logits
    float2 qv[GRP][E2];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(
          a.q + (static_cast<size_t>(t) * n_q + g * GRP + h) * D);
      load_row_pairs<NCH>(qrow, dg, qv[h]);
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
      for (int e = 0; e < E2; ++e) qv[h][e] = __fmul2_rn(qv[h][e], sc2);
    }
    // Softmax state.  m_ref[h] is a warp-uniform reference maximum of head h
    // (base-2 logits); probabilities are exp2(s - m_ref) and the reference is
    // only raised when a score exceeds it by more than kLazy, so p <= 2^kLazy.
    // Each lane's value slots always hold the same heads (see below), so the
    // lane keeps its share of the denominators per slot (lslot).
    constexpr int V = 4 * GRP;                 // (token slot, head) values per lane
    constexpr bool kTransposed = V >= 8;       // scores reduced by transposition
    constexpr int R = kTransposed ? V / 8 : V; // totals a lane holds after the reduction
    constexpr float kLazy = 8.0f;
    float m_ref[GRP], lslot[R], msel[R];
    int hsel[R];                               // head of each slot
    float2 acc[GRP][E2];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      m_ref[h] = -INFINITY;
#pragma unroll
      for (int e = 0; e < E2; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int idx = kTransposed ? dg * R + r : r;
      hsel[r] = idx % GRP;
      lslot[r] = 0.f;
      msel[r] = -INFINITY;
    }

    // partial q.k of one page over this lane's dims: v[jj * GRP + h], token ts + 4 jj
    auto partial_qk = [&](const uint8_t* kb, float (&v)[V]) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        float2 kv[E2];
        load_row_pairs<NCH>(kb + (ts + 4 * jj) * D * 2, dg, kv);
#pragma unroll
        for (int h = 0; h < GRP; ++h) {
          float2 d0 = __fmul2_rn(qv[h][0], kv[0]);
          float2 d1 = __fmul2_rn(qv[h][1], kv[1]);
#pragma unroll
          for (int e = 2; e < E2; e += 2) {
            d0 = __ffma2_rn(qv[h][e], kv[e], d0);
            d1 = __ffma2_rn(qv[h][e + 1], kv[e + 1], d1);
          }
          v[jj * GRP + h] = (d0.x + d0.y) + (d1.x + d1.y);
        }
      }
    };
    auto page_ready = [&](int k) {
      return __all_sync(0xffffffffu, mbar_wait(&bar[(gk + k) % STAGES], ((gk + k) / STAGES) & 1,
                                               a.timeout_ns));
    };
    // on a failed wait: every copy this warp started must land before the CTA exits
    auto drain_from = [&](int k) {
      if (lane == 0)
        for (int kk = k; kk < issued; ++kk)
          mbar_wait(&bar[(gk + kk) % STAGES], ((gk + kk) / STAGES) & 1, a.timeout_ns);
    };

    // Software pipeline: the partial q.k of page k+1 is computed before the
    // softmax and PV of page k, so the two dependency chains overlap.
    float vq[V];
    if (page_ready(0)) {
      partial_qk(ring + (gk % STAGES) * 2 * BLK, vq);
    } else {
      drain_from(0);
      failed = true;
    }
    for (int k = 0; k < npg && !failed; ++k) {
      float v[V];
#pragma unroll
      for (int i = 0; i < V; ++i) v[i] = vq[i];
      if (k + 1 < npg) {
        if (!page_ready(k + 1)) {
          drain_from(k + 1);
          failed = true;
          break;
        }
        partial_qk(ring + ((gk + k + 1) % STAGES) * 2 * BLK, vq);
      }
      const uint8_t* vb = ring + ((gk + k) % STAGES) * 2 * BLK + BLK;
      // Sum over the 8 dim-group lanes.  Transposed form: at each level a
      // lane keeps half of its values and adds the partner's matching half, so
      // after three levels lane dg holds the totals of values dg*R .. dg*R+R-1.
      if constexpr (kTransposed) {
#pragma unroll
        for (int lvl = 0; lvl < 3; ++lvl) {
          const int mask = 4 >> lvl;
          const int half = V >> (lvl + 1);
          const bool upper = (lane & mask) != 0;
#pragma unroll
          for (int i = 0; i < half; ++i) {
            const float keep = upper ? v[i + half] : v[i];
            const float send = upper ? v[i] : v[i + half];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) {
          v[i] += __shfl_xor_sync(0xffffffffu, v[i], 1);
          v[i] += __shfl_xor_sync(0xffffffffu, v[i], 2);
          v[i] += __shfl_xor_sync(0xffffffffu, v[i], 4);
        }
      }
      bool valid[R];
      bool raise = false;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int idx = kTransposed ? dg * R + r : r;
        valid[r] = k * P + ts + 4 * (idx / GRP) < n;
        raise |= valid[r] && v[r] > msel[r] + kLazy;
      }
      if (__any_sync(0xffffffffu, raise)) {  // rare: move the reference maxima up
#pragma unroll
        for (int h = 0; h < GRP; ++h) {
          float x = -INFINITY;
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (valid[r] && hsel[r] == h) x = fmaxf(x, v[r]);
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
          const float mn = fmaxf(m_ref[h], x);
          if (mn > m_ref[h]) {  // warp-uniform
            const float corr = exp2f(m_ref[h] - mn);
            const float2 c2 = make_float2(corr, corr);
#pragma unroll
            for (int e = 0; e < E2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], c2);
#pragma unroll
            for (int r = 0; r < R; ++r)
              if (hsel[r] == h) lslot[r] *= corr;
            m_ref[h] = mn;
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float mm = m_ref[0];
#pragma unroll
          for (int h = 1; h < GRP; ++h) mm = hsel[r] == h ? m_ref[h] : mm;
          msel[r] = mm;
        }
      }
      float pr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        pr[r] = valid[r] ? exp2f(v[r] - msel[r]) : 0.f;
        lslot[r] += pr[r];
      }
      // probabilities of this lane's tokens for every head
      float pg[V];
      if constexpr (kTransposed) {
#pragma unroll
        for (int i = 0; i < V; ++i)
          pg[i] = __shfl_sync(0xffffffffu, pr[i % R], (lane & 24) | (i / R));
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) pg[i] = pr[i];
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (k * P + ts + 4 * jj < n) {  // positions past the piece may hold anything (even NaN)
          float2 vv[E2];
          load_row_pairs<NCH>(vb + (ts + 4 * jj) * D * 2, dg, vv);
#pragma unroll
          for (int h = 0; h < GRP; ++h) {
            const float2 p2 = make_float2(pg[jj * GRP + h], pg[jj * GRP + h]);
#pragma unroll
            for (int e = 0; e < E2; ++e) acc[h][e] = __ffma2_rn(p2, vv[e], acc[h][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && k + STAGES < npg) {
        fence_proxy_async_smem();
        issue(k + STAGES);
        ++issued;
      }
    }
    if (failed) break;
    gk += npg;

    // denominators: gather each head's slots from every lane that holds them
    float l[GRP], m[GRP];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      float x = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) x += hsel[r] == h ? lslot[r] : 0.f;
      if constexpr (kTransposed) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      } else {
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
      }
      l[h] = x;
      m[h] = m_ref[h];
    }
    // merge the four token slots of the accumulators
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
#pragma unroll
      for (int e = 0; e < E2; ++e) {
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, 8);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, 8);
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, 16);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, 16);
      }
    }
    const int nch = a.tok_nchunks[t];
    if (nch == 1) {
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        if ((h & 3) != ts) continue;
        const float inv = 1.f / l[h];
        __nv_bfloat16* orow = a.o + (static_cast<size_t>(t) * n_q + g * GRP + h) * D;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          uint4 u;
          const float2* v = &acc[h][ch * 4];
          u.x = pack_bf16(v[0].x * inv, v[0].y * inv);
          u.y = pack_bf16(v[1].x * inv, v[1].y * inv);
          u.z = pack_bf16(v[2].x * inv, v[2].y * inv);
          u.w = pack_bf16(v[3].x * inv, v[3].y * inv);
          *reinterpret_cast<uint4*>(orow + ch * 64 + dg * 8) = u;
        }
      }
      continue;
    }
    // several pieces: publish this one, the last finisher merges
    constexpr int REC = partial_rec_floats(GRP, D);
    static_assert(REC % 4 == 0, "partial records must stay 16-byte aligned");
    const size_t row_rec = static_cast<size_t>(t) * a.max_chunks;
    float* rec = a.partials + ((row_rec + c) * n_kv + g) * REC;
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      if ((h & 3) != ts) continue;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        float4* dst = reinterpret_cast<float4*>(rec + h * D + ch * 64 + dg * 8);
        const float2* v = &acc[h][ch * 4];
        dst[0] = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
        dst[1] = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        rec[GRP * D + h] = m[h];
        rec[GRP * D + GRP + h] = l[h];
      }
    }
    if (finish_piece(a, t, g, nch, lane)) merge_row_partials<GRP, NCH>(a, t, g, nch, lane);
  }

  if (failed) raise_status(a.status, ST_TIMEOUT);
}

template <int GRP, int NCH, int WARPS, int STAGES>
static cudaError_t launch_t(const AttnArgs& a, int grid, cudaStream_t stream) {
  const int smem = attn_smem_bytes_cfg(NCH * 64, ATT_P, WARPS, STAGES, WARPS < 8);
  const cudaError_t e =
      set_smem_limit(reinterpret_cast<const void*>(attn_kernel<GRP, NCH, WARPS, STAGES>), smem);
  if (e != cudaSuccess) return e;
  attn_kernel<GRP, NCH, WARPS, STAGES><<<grid, WARPS * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int GRP, int NCH>
static cudaError_t launch_cfg(const AttnArgs& a, int grid, cudaStream_t stream) {
  switch (a.warps) {
    case 4: return launch_t<GRP, NCH, 4, 3>(a, grid, stream);
    case 5: return launch_t<GRP, NCH, 5, 2>(a, grid, stream);
    case 12:
    case 16:  // warp pairs split the head dims (head_dim 128 only)
      if (NCH == 2) return launch_attention_pair(a, grid, stream);
      return launch_t<GRP, NCH, 8, 3>(a, grid, stream);
    default: return launch_t<GRP, NCH, 8, 3>(a, grid, stream);
  }
}

cudaError_t launch_attention(const AttnArgs& a, int grid, cudaStream_t stream) {
  if (a.page_size != ATT_P || grid <= 0) return cudaErrorInvalidValue;
  const int grp = a.n_q / a.n_kv;
  const int nch = a.head_dim / 64;
#define NF_ATT_CASE(G, N) \
  if (grp == G && nch == N) return launch_cfg<G, N>(a, grid, stream);
  NF_ATT_CASE(1, 1) NF_ATT_CASE(2, 1) NF_ATT_CASE(4, 1) NF_ATT_CASE(8, 1)
  NF_ATT_CASE(1, 2) NF_ATT_CASE(2, 2) NF_ATT_CASE(4, 2) NF_ATT_CASE(8, 2)
#undef NF_ATT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace nf
