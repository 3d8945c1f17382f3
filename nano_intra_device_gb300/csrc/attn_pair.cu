// Paged GQA attention, head_dim 128, one warp PAIR per work piece.
//
// Same computation and work list as attn.cu (paged decode/causal attention
// over the KV cache, split-KV pieces merged by log-sum-exp; "NanoFlow: Towards
// Optimal LLM Serving Throughput", "The Intra-Device Parallelism Mechanism";
// "LLM Inference Performance", "PagedAttention").  The difference is how a
// piece is spread over threads: two warps share one shared-memory ring of
// (page, KV head) blocks and each owns half of the 128 head dims, so a lane
// keeps 8 dims of q and of the accumulators per query head instead of 16.  The
// halved register footprint fits 12-16 warps per SM, which is what hides the
// latency of the per-page dependency chain (q.k -> reduction -> softmax ->
// p.v).  The two halves of each score are added through shared memory once
// per page.  Every wait, including the pair's synchronisation, is an mbarrier
// wait with a time limit: no named barrier, so a timed-out warp cannot leave
// its partner blocked.
#include "common.cuh"
#include "kernels.h"

namespace nf {

namespace {

constexpr int PD = 128;                  // head_dim this kernel is built for
constexpr int PP = 16;                   // page size
constexpr int PBLK = PP * PD * 2;        // bytes of one (page, KV head) block
constexpr int PMAX_PAGES = 2048 / PP;    // longest split-KV piece, in pages

template <int STAGES, int R>
struct PairSmem {
  uint64_t full[STAGES];                 // TMA completion, one arrival (expect_tx)
  uint64_t empty[STAGES];                // both warps done with the stage (2 arrivals)
  uint64_t sync;                         // pair rendezvous (2 arrivals)
  int next_idx;                          // next piece, published by the leader
  int last;                              // merge decision of the piece
  float xbuf[2][2][32][R];               // [slot][half][lane][value] partial scores
  int pages[PMAX_PAGES];
};

// 8 bf16 (16 bytes) at dims dbase + dg*8 .. of one row -> 4 fp32 pairs.
__device__ __forceinline__ void load8(const uint8_t* row, int dbase, int dg, float2 (&o)[4]) {
  const uint4 u = *reinterpret_cast<const uint4*>(row + (dbase + dg * 8) * 2);
  o[0] = make_float2(bf16lo(u.x), bf16hi(u.x));
  o[1] = make_float2(bf16lo(u.y), bf16hi(u.y));
  o[2] = make_float2(bf16lo(u.z), bf16hi(u.z));
  o[3] = make_float2(bf16lo(u.w), bf16hi(u.w));
}

}  // namespace

template <int GRP, int PAIRS, int STAGES>
__global__ void __launch_bounds__(PAIRS * 64, 1) attn_pair_kernel(const AttnArgs a) {
  constexpr int E2 = 4;                      // dim pairs per lane
  constexpr int V = 4 * GRP;                 // (token slot, head) values per lane
  constexpr bool kTransposed = V >= 8;
  constexpr int R = kTransposed ? V / 8 : V; // totals a lane holds after the reduction
  constexpr float kLazy = 8.0f;
  using Smem = PairSmem<STAGES, R>;
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp >> 1, half = warp & 1;
  const int ts = lane >> 3, dg = lane & 7;
  const int dbase = half * 64;
  const bool leader = half == 0 && lane == 0;
  uint8_t* ring = smem + pair * (STAGES * 2 * PBLK);
  Smem* sm = reinterpret_cast<Smem*>(smem + PAIRS * STAGES * 2 * PBLK) + pair;
  if (leader) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], 2);
    }
    mbar_init(&sm->sync, 2);
    fence_mbar_init();
  }
  __syncthreads();

  const int seg = a.seg;
  const int begin = a.seg_items[seg];
  const int total = (a.seg_items[seg + 1] - begin) * a.n_kv;
  const int n_kv = a.n_kv, n_q = a.n_q, C = a.kv_chunk;
  const size_t page_stride = static_cast<size_t>(n_kv) * PP * PD;
  const uint64_t policy = l2_policy_evict_first();
  const uint64_t tmo = a.timeout_ns;
  uint32_t gk = 0;      // pages this pair has consumed (ring position)
  uint32_t nsync = 0;   // pair rendezvous so far (phase of sm->sync)
  uint32_t nempty = 0;  // refills the leader has issued after the first fill of each stage
  bool failed = false;

  // Rendezvous of the two warps (bounded).  Orders shared-memory writes made
  // before it by either warp before reads after it.
  auto pair_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->sync);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm->sync, nsync & 1, tmo));
    ++nsync;
    return ok;
  };

  if (leader) sm->next_idx = atomicAdd(&a.fetch[seg], 1);
  if (!pair_sync()) failed = true;

  while (!failed) {
    const int idx = sm->next_idx;
    if (idx >= total) break;
    // everyone has read next_idx (and finished the previous piece's stages)
    if (!pair_sync()) {
      failed = true;
      break;
    }
    if (leader) sm->next_idx = atomicAdd(&a.fetch[seg], 1);
    const int pr_ = begin + idx / n_kv, g = idx % n_kv;
    const int t = a.items[2 * pr_], c = a.items[2 * pr_ + 1];
    const int s = a.tok_seq[t];
    const int ctx = a.tok_pos[t] + 1;
    const int b0 = c * C;
    const int n = min(C, ctx - b0);
    const int npg = (n + PP - 1) / PP;
    {
      const int* bt = a.block_table + static_cast<size_t>(s) * a.max_pages + b0 / PP;
      for (int i = half * 32 + lane; i < npg; i += 64) {
        int page = bt[i];
        if (page < 0 || page >= a.num_pages) {  // never read outside the pool
          raise_status(a.status, ST_BAD_PAGE);
          page = 0;
        }
        sm->pages[i] = page;
      }
    }
    if (!pair_sync()) {
      failed = true;
      break;
    }
    auto issue = [&](int k) {
      const uint32_t st = (gk + k) % STAGES;
      const size_t off =
          static_cast<size_t>(sm->pages[k]) * page_stride + static_cast<size_t>(g) * PP * PD;
      uint8_t* kb = ring + st * 2 * PBLK;
      mbar_arrive_expect_tx(&sm->full[st], 2 * PBLK);
      bulk_g2s_evict_first(kb, a.k_pool + off, PBLK, &sm->full[st], policy);
      bulk_g2s_evict_first(kb + PBLK, a.v_pool + off, PBLK, &sm->full[st], policy);
    };
    int issued = 0;
    if (leader) {
      const int pre = npg < STAGES ? npg : STAGES;
      for (int k = 0; k < pre; ++k) issue(k);
      issued = pre;
    }

    float2 qv[GRP][E2];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(
          a.q + (static_cast<size_t>(t) * n_q + g * GRP + h) * PD);
      load8(qrow, dbase, dg, qv[h]);
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
      for (int e = 0; e < E2; ++e) qv[h][e] = __fmul2_rn(qv[h][e], sc2);
    }
    float m_ref[GRP], lslot[R], msel[R];
    int hsel[R];
    float2 acc[GRP][E2];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      m_ref[h] = -INFINITY;
#pragma unroll
      for (int e = 0; e < E2; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int idx2 = kTransposed ? dg * R + r : r;
      hsel[r] = idx2 % GRP;
      lslot[r] = 0.f;
      msel[r] = -INFINITY;
    }

    auto partial_qk = [&](const uint8_t* kb, float (&v)[V]) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        float2 kv[E2];
        load8(kb + (ts + 4 * jj) * PD * 2, dbase, dg, kv);
#pragma unroll
        for (int h = 0; h < GRP; ++h) {
          float2 d0 = __fmul2_rn(qv[h][0], kv[0]);
          float2 d1 = __fmul2_rn(qv[h][1], kv[1]);
          d0 = __ffma2_rn(qv[h][2], kv[2], d0);
          d1 = __ffma2_rn(qv[h][3], kv[3], d1);
          v[jj * GRP + h] = (d0.x + d0.y) + (d1.x + d1.y);
        }
      }
    };
    auto page_ready = [&](int k) {
      return __all_sync(0xffffffffu,
                        mbar_wait(&sm->full[(gk + k) % STAGES], ((gk + k) / STAGES) & 1, tmo));
    };
    // both warps are done with page k's stage: release it, and let the leader
    // refill it with page k + STAGES once its partner has released it too
    auto release = [&](int k) -> bool {
      __syncwarp();
      const uint32_t st = (gk + k) % STAGES;
      if (lane == 0) mbar_arrive(&sm->empty[st]);
      if (k + STAGES < npg) {
        bool ok = true;
        if (leader) {
          ok = mbar_wait(&sm->empty[st], ((gk + k) / STAGES) & 1, tmo);
          if (ok) {
            fence_proxy_async_smem();
            issue(k + STAGES);
            ++issued;
          }
        }
        return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
      return true;
    };
    auto drain_from = [&](int k) {
      if (leader)
        for (int kk = k; kk < issued; ++kk)
          mbar_wait(&sm->full[(gk + kk) % STAGES], ((gk + kk) / STAGES) & 1, tmo);
    };

    float vq[V];
    if (page_ready(0)) {
      partial_qk(ring + (gk % STAGES) * 2 * PBLK, vq);
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
        partial_qk(ring + ((gk + k + 1) % STAGES) * 2 * PBLK, vq);
      }
      const uint8_t* vb = ring + ((gk + k) % STAGES) * 2 * PBLK + PBLK;
      // reduce over this warp's 8 dim groups (transposed), then add the other half
      if constexpr (kTransposed) {
#pragma unroll
        for (int lvl = 0; lvl < 3; ++lvl) {
          const int mask = 4 >> lvl;
          const int hv = V >> (lvl + 1);
          const bool upper = (lane & mask) != 0;
#pragma unroll
          for (int i = 0; i < hv; ++i) {
            const float keep = upper ? v[i + hv] : v[i];
            const float send = upper ? v[i] : v[i + hv];
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
      const int slot = nsync & 1;
#pragma unroll
      for (int r = 0; r < R; ++r) sm->xbuf[slot][half][lane][r] = v[r];
      if (!pair_sync()) {
        drain_from(k + 1);
        failed = true;
        break;
      }
#pragma unroll
      for (int r = 0; r < R; ++r) v[r] += sm->xbuf[slot][half ^ 1][lane][r];

      bool valid[R];
      bool raise = false;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int idx2 = kTransposed ? dg * R + r : r;
        valid[r] = k * PP + ts + 4 * (idx2 / GRP) < n;
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
          if (mn > m_ref[h]) {
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
        if (k * PP + ts + 4 * jj < n) {  // positions past the piece may hold anything
          float2 vv[E2];
          load8(vb + (ts + 4 * jj) * PD * 2, dbase, dg, vv);
#pragma unroll
          for (int h = 0; h < GRP; ++h) {
            const float2 p2 = make_float2(pg[jj * GRP + h], pg[jj * GRP + h]);
#pragma unroll
            for (int e = 0; e < E2; ++e) acc[h][e] = __ffma2_rn(p2, vv[e], acc[h][e]);
          }
        }
      }
      if (!release(k)) {
        drain_from(k + 1);
        failed = true;
        break;
      }
    }
    if (failed) break;
    gk += npg;

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
#pragma unroll
    for (int h = 0; h < GRP; ++h)
#pragma unroll
      for (int e = 0; e < E2; ++e) {
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, 8);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, 8);
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, 16);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, 16);
      }
    const int nch = a.tok_nchunks[t];
    if (nch == 1) {
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        if ((h & 3) != ts) continue;
        const float inv = 1.f / l[h];
        __nv_bfloat16* orow = a.o + (static_cast<size_t>(t) * n_q + g * GRP + h) * PD;
        uint4 u;
        u.x = pack_bf16(acc[h][0].x * inv, acc[h][0].y * inv);
        u.y = pack_bf16(acc[h][1].x * inv, acc[h][1].y * inv);
        u.z = pack_bf16(acc[h][2].x * inv, acc[h][2].y * inv);
        u.w = pack_bf16(acc[h][3].x * inv, acc[h][3].y * inv);
        *reinterpret_cast<uint4*>(orow + dbase + dg * 8) = u;
      }
      continue;
    }
    // several pieces: publish this one (each warp its dims, the leader warp m
    // and l), and the pair that finishes a row's last piece merges
    constexpr int REC = partial_rec_floats(GRP, PD);
    const size_t row_rec = static_cast<size_t>(t) * a.max_chunks;
    float* rec = a.partials + ((row_rec + c) * n_kv + g) * REC;
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      if ((h & 3) != ts) continue;
      float4* dst = reinterpret_cast<float4*>(rec + h * PD + dbase + dg * 8);
      dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
      dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
    }
    if (leader) {
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        rec[GRP * PD + h] = m[h];
        rec[GRP * PD + GRP + h] = l[h];
      }
    }
    __threadfence();
    if (!pair_sync()) {
      failed = true;
      break;
    }
    if (leader) sm->last = atomicAdd(&a.row_done[t * n_kv + g], 1) == nch - 1;
    if (!pair_sync()) {
      failed = true;
      break;
    }
    if (!sm->last) continue;
    __threadfence();
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      if ((h & 3) != ts) continue;
      float M = -INFINITY;
      for (int cc = 0; cc < nch; ++cc) {
        const float* r = a.partials + ((row_rec + cc) * n_kv + g) * REC;
        M = fmaxf(M, __ldcg(r + GRP * PD + h));
      }
      float L = 0.f, O[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) O[e] = 0.f;
      for (int cc = 0; cc < nch; ++cc) {
        const float* r = a.partials + ((row_rec + cc) * n_kv + g) * REC;
        const float w = exp2f(__ldcg(r + GRP * PD + h) - M);
        L += w * __ldcg(r + GRP * PD + GRP + h);
        const float4* src = reinterpret_cast<const float4*>(r + h * PD + dbase + dg * 8);
        const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
        O[0] += w * x0.x; O[1] += w * x0.y; O[2] += w * x0.z; O[3] += w * x0.w;
        O[4] += w * x1.x; O[5] += w * x1.y; O[6] += w * x1.z; O[7] += w * x1.w;
      }
      const float inv = 1.f / L;
      __nv_bfloat16* orow = a.o + (static_cast<size_t>(t) * n_q + g * GRP + h) * PD;
      uint4 u;
      u.x = pack_bf16(O[0] * inv, O[1] * inv);
      u.y = pack_bf16(O[2] * inv, O[3] * inv);
      u.z = pack_bf16(O[4] * inv, O[5] * inv);
      u.w = pack_bf16(O[6] * inv, O[7] * inv);
      *reinterpret_cast<uint4*>(orow + dbase + dg * 8) = u;
    }
  }
  if (failed) raise_status(a.status, ST_TIMEOUT);
  (void)nempty;
}

template <int GRP, int PAIRS, int STAGES>
static cudaError_t launch_pair_t(const AttnArgs& a, int grid, cudaStream_t stream) {
  constexpr int V = 4 * GRP;
  constexpr int R = V >= 8 ? V / 8 : V;
  const int smem = PAIRS * (STAGES * 2 * PBLK) + PAIRS * static_cast<int>(sizeof(PairSmem<STAGES, R>)) + 128;
  const cudaError_t attr =
      set_smem_limit(reinterpret_cast<const void*>(attn_pair_kernel<GRP, PAIRS, STAGES>), smem);
  if (attr != cudaSuccess) return attr;
  attn_pair_kernel<GRP, PAIRS, STAGES><<<grid, PAIRS * 64, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attention_pair(const AttnArgs& a, int grid, cudaStream_t stream) {
  if (a.head_dim != PD || a.page_size != PP || grid <= 0) return cudaErrorInvalidValue;
  const int grp = a.n_q / a.n_kv;
  const bool sixteen = a.warps == 16;
#define NF_PAIR_CASE(G)                                                              \
  if (grp == G)                                                                      \
    return sixteen ? launch_pair_t<G, 8, 3>(a, grid, stream)                         \
                   : launch_pair_t<G, 6, 4>(a, grid, stream);
  NF_PAIR_CASE(1) NF_PAIR_CASE(2) NF_PAIR_CASE(4) NF_PAIR_CASE(8)
#undef NF_PAIR_CASE
  return cudaErrorInvalidValue;
}

}  // namespace nf
