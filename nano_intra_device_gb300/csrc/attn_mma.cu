// Paged GQA attention with the dot products on the tensor cores.
//
// Each token row attends to positions 0..pos of its sequence through the block
// table.  The work list cuts every row into split-KV pieces (row, chunk of
// kv_chunk positions); one warp takes one piece for one KV head, fetched from a
// per-nano-batch counter by a persistent grid, and pieces of a row that was cut
// are merged by log-sum-exp (attn_merge.cuh).  Decode attention moves far more
// bytes than it computes on ("NanoFlow: Towards Optimal LLM Serving
// Throughput", "The Intra-Device Parallelism Mechanism": the memory-bound
// operation); with the dot products on the tensor cores one page costs about 60
// warp instructions, so that part of the SMs can keep HBM busy while the rest
// run the GEMMs of another nano-batch.
//
// Per page (16 positions) and KV head, with the GQA group of GRP query heads
// padded to the 8 columns of an m16n8k16 tile:
//   * S^T[16 pos x 8 heads] = K_page[16 x d] . Q^T[d x 8]   (d/16 MMAs);
//   * online softmax down each column (base 2, lazily rescaled);
//   * P^T goes from accumulator to operand layout with movmatrix.trans;
//   * O^T[d x 8] += V_page^T[d x 16] . P^T[16 x 8]         (d/16 MMAs).
// K and V pages arrive by 2-D TMA copies over the pool viewed as
// [num_pages * n_kv * 16, d] with 128-byte swizzle, so that the ldmatrix loads
// of 8 positions at the same dims hit 8 different bank groups.  Positions past
// the end of a piece read row 0 of its page instead (P is 0 there), so a stale
// or poisoned slot never reaches the accumulators.  P enters the PV product
// as two bf16 operands, hi = bf16(p) and lo = bf16(p - hi), in two MMAs on the
// same V fragment: p keeps 16 significant bits instead of 8 (one bf16 P alone
// perturbs each weight by up to 2^-9, which shows in o at the 1e-3 level and
// then moves bf16 roundings of every tensor downstream), and the denominators
// sum the fp32 values.
#include "attn_merge.cuh"
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace nf {

int attn_partial_floats(int n_q, int n_kv, int head_dim) {
  return partial_rec_floats(n_q / n_kv, head_dim);
}

constexpr int AMMA_MAX_PIECE_PAGES = 2048 / AMMA_P;  // longest piece: 4 page ids per lane
constexpr int AMMA_MIN_SMEM = 120 * 1024;            // > half an SM: one CTA per SM

// The 4-warp configuration shares its SM with one GEMM CTA of 2 ring stages
// (98 KB, <= 248 registers a thread): it takes 117 KB (more than half an SM, so
// two attention CTAs never pair up) and at most 128 registers a thread.  The
// others fill an SM alone.
constexpr int AMMA_SHARE_WARPS = 4;
constexpr int AMMA_SHARE_SMEM = 117 * 1024;

static int amma_smem_bytes(int head_dim, int warps, int stages) {
  const int slot = 2 * AMMA_P * head_dim * 2;  // K and V of one (page, KV head)
  const int need = 1024 + warps * stages * (slot + 8);
  const int floor = warps == AMMA_SHARE_WARPS ? AMMA_SHARE_SMEM : AMMA_MIN_SMEM;
  return need < floor ? floor : need;
}

template <int GRP, int NCH, int WARPS, int STAGES, int PPI>
__global__ void __launch_bounds__(WARPS * 32, WARPS == AMMA_SHARE_WARPS ? 4 : 1)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnArgs a) {
  constexpr int D = NCH * 64;
  constexpr int P = AMMA_P;
  constexpr int BOX = P * 128;      // one 64-column box of a page: 2 KB
  constexpr int BLK = NCH * BOX;    // K (or V) of one (page, KV head)
  constexpr int SLOT = 2 * BLK;
  constexpr int KS = D / 16;        // k-steps of S, m-tiles of O
  static_assert(GRP >= 1 && GRP <= 8, "the GQA group must fit the 8 columns of a tile");
  static_assert(STAGES >= 2 * PPI, "S of the next group is formed while this one is in use");
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzled boxes: 1 KB aligned
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lr = lane >> 2, lc = lane & 3;  // fragment row / column pair of this lane
  uint8_t* ring = smem + warp * (STAGES * SLOT);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + WARPS * STAGES * SLOT) + warp * STAGES;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncwarp();

  const int seg = a.seg;
  const int begin = a.seg_items[seg];
  const int total = (a.seg_items[seg + 1] - begin) * a.n_kv;
  const int n_kv = a.n_kv, n_q = a.n_q, C = a.kv_chunk;
  const uint64_t policy = l2_policy_evict_first();
  uint32_t gk = 0;  // pages this warp has consumed (ring position)
  bool failed = false;
  const int h0 = 2 * lc, h1 = 2 * lc + 1;  // the two heads of this lane's accumulator columns
  constexpr float kLazy = 8.0f;

  const float scale = a.scale_log2;
  const uint32_t ring_u32 = smem_u32(ring);
  // ldmatrix row addresses (lane 8 j + r supplies row r of matrix j), fixed per
  // lane: S^T takes matrix j = (positions 8 (j & 1) .., dims 16 kk + 8 (j >> 1) ..),
  // O^T takes matrix j = (positions 8 (j >> 1) .., dims 16 mi + 8 (j & 1) ..), transposed.
  const int mj = lane >> 3, mr = lane & 7;
  const int k_row = mr + 8 * (mj & 1), k_ci = mj >> 1;
  const int v_row = mr + 8 * (mj >> 1), v_ci = mj & 1;
  uint32_t koff[KS], voff[KS];
#pragma unroll
  for (int i = 0; i < KS; ++i) {
    koff[i] = page_chunk_off(k_row, 2 * i + k_ci);
    voff[i] = BLK + page_chunk_off(v_row, 2 * i + v_ci);
  }

  bool waited = !a.early;  // warp-uniform: this warp has waited for the QKV GEMM
  int next_idx = 0;
  if (lane == 0) next_idx = atomicAdd(&a.fetch[seg], 1);
  for (;;) {
    const int idx = __shfl_sync(0xffffffffu, next_idx, 0);
    if (idx >= total) break;
    if (lane == 0) next_idx = atomicAdd(&a.fetch[seg], 1);
    const int pair = begin + idx / n_kv, g = idx % n_kv;
    const int t = a.items[2 * pair], c = a.items[2 * pair + 1];
    const int s = a.tok_seq[t];
    if (a.prefill_elsewhere && s >= a.n_decode_seqs) continue;  // the prefill kernel's row
    const int ctx = a.tok_pos[t] + 1;
    const int b0 = c * C;
    const int n = min(C, ctx - b0);
    const int npg = (n + P - 1) / P;
    int pid[4];  // page ids of the piece: page lane + 32 i in pid[i]
    {
      const int* bt = a.block_table + static_cast<size_t>(s) * a.max_pages + b0 / P;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = lane + 32 * i;
        int page = 0;
        if (j < npg) {
          page = bt[j];
          if (page < 0 || page >= a.num_pages) {  // never read outside the pool
            raise_status(a.status, ST_BAD_PAGE);
            page = 0;
          }
        }
        pid[i] = page;
      }
    }
    // id of page k of the piece (k warp-uniform; every lane must call)
    auto page_id = [&](int k) {
      const int v = k < 32 ? pid[0] : k < 64 ? pid[1] : k < 96 ? pid[2] : pid[3];
      return __shfl_sync(0xffffffffu, v, k & 31);
    };
    auto issue_into = [&](uint32_t st, int page) {
      uint8_t* sl = ring + st * SLOT;
      const int y = (page * n_kv + g) * P;  // first pool row of the (page, KV head)
      mbar_arrive_expect_tx(&bar[st], SLOT);
      if (NCH == 2) {  // one box per (page, KV head): both 64-column halves
        tma_load_3d_hint(sl, &tmK, &bar[st], 0, y, 0, policy);
        tma_load_3d_hint(sl + BLK, &tmV, &bar[st], 0, y, 0, policy);
      } else {
        tma_load_2d_hint(sl, &tmK, &bar[st], 0, y, policy);
        tma_load_2d_hint(sl + BLK, &tmV, &bar[st], 0, y, policy);
      }
    };
    int issued = 0;
    {
      const int pre = npg < STAGES ? npg : STAGES;
      int first[STAGES];
#pragma unroll
      for (int k = 0; k < STAGES; ++k) first[k] = page_id(k < pre ? k : 0);
      // Before the wait for the QKV GEMM only pages that it does not write: a
      // decode row appends position ctx - 1; other rows are left whole.
      int ahead = pre;
      if (!waited) {
        const int fresh = s < a.n_decode_seqs ? ctx - 1 : 0;
        const int clean = fresh > b0 ? (fresh - b0) / P : 0;
        ahead = clean < pre ? clean : pre;
      }
      if (lane == 0) {
        fence_proxy_async_smem();  // the previous piece's reads of these slots come first
#pragma unroll
        for (int k = 0; k < STAGES; ++k)
          if (k < ahead) issue_into((gk + k) % STAGES, first[k]);
      }
      if (!waited) {
        pdl_wait();  // q and this step's K/V are written
        waited = true;
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < STAGES; ++k)
            if (k >= ahead && k < pre) issue_into((gk + k) % STAGES, first[k]);
        }
      }
      issued = pre;
    }

    // Q^T as the B operand of S^T = K Q^T: column n = head lr of the group
    // (zero past GRP), rows = dims 16 kk + 2 lc (+1) and + 8.
    uint32_t qb[KS][2];
    {
      const bool hv = lr < GRP;
      const __nv_bfloat16* qrow = a.q + (static_cast<size_t>(t) * n_q + g * GRP + (hv ? lr : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint32_t x0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * lc);
        const uint32_t x1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * lc);
        qb[kk][0] = hv ? x0 : 0u;
        qb[kk][1] = hv ? x1 : 0u;
      }
    }
    float o[KS][4];
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // reference maxima of heads h0, h1 (base 2)
    float l0 = 0.f, l1 = 0.f;              // this lane's share of their denominators

    auto qk = [&](uint32_t slot, float (&sacc)[4]) {
      float s2[4] = {0.f, 0.f, 0.f, 0.f};  // odd k-steps: two independent MMA chains
      sacc[0] = sacc[1] = sacc[2] = sacc[3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t af[4];
        ldsm_x4(slot + koff[kk], af);
        if (kk & 1)
          mma_16816(s2, af, qb[kk][0], qb[kk][1]);
        else
          mma_16816(sacc, af, qb[kk][0], qb[kk][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i] += s2[i];
    };
    auto slot_ready = [&](uint32_t st, uint32_t ph) {
      return __all_sync(0xffffffffu, mbar_wait(&bar[st], ph, a.timeout_ns));
    };
    auto drain_from = [&](int k) {
      if (lane == 0)
        for (int kk = k; kk < issued; ++kk)
          mbar_wait(&bar[(gk + kk) % STAGES], ((gk + kk) / STAGES) & 1, a.timeout_ns);
    };

    // Software pipeline over groups of PPI pages: S of the next group is formed
    // before the softmax and PV of the current one.  (rs, rph): ring slot and
    // barrier phase of the group's first page; page i of a group sits i slots on.
    auto slot_at = [&](uint32_t base, uint32_t ph, int i, uint32_t& st, uint32_t& p) {
      st = base + i;
      p = ph;
      if (st >= STAGES) {
        st -= STAGES;
        p ^= 1;
      }
    };
    uint32_t rs = gk % STAGES, rph = (gk / STAGES) & 1;
    float sn[PPI][4];
#pragma unroll
    for (int i = 0; i < PPI; ++i) {
      if (i < npg && !failed) {
        uint32_t st, ph;
        slot_at(rs, rph, i, st, ph);
        if (slot_ready(st, ph)) {
          qk(ring_u32 + st * SLOT, sn[i]);
        } else {
          drain_from(i);
          failed = true;
        }
      }
    }
    for (int k = 0; k < npg && !failed; k += PPI) {
      uint32_t ns, nph;  // first slot of the next group
      slot_at(rs, rph, PPI, ns, nph);
      float sc[PPI][4];
#pragma unroll
      for (int i = 0; i < PPI; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) sc[i][r] = sn[i][r];  // raw q.k: (pos lr, h0), (lr, h1), (lr+8, h0), (lr+8, h1)
#pragma unroll
      for (int i = 0; i < PPI; ++i) {
        if (k + PPI + i < npg && !failed) {
          uint32_t st, ph;
          slot_at(ns, nph, i, st, ph);
          if (slot_ready(st, ph)) {
            qk(ring_u32 + st * SLOT, sn[i]);
          } else {
            drain_from(k + PPI + i);
            failed = true;
          }
        }
      }
      if (failed) break;
      // positions past the piece (the last page's tail, or a missing last page
      // of the group) may hold anything, even NaN: they become -inf
      const bool tail = (k + PPI) * P > n;  // warp-uniform
      if (tail) {
#pragma unroll
        for (int i = 0; i < PPI; ++i) {
          const int kb = (k + i) * P;
          const bool v0 = kb + lr < n, v1 = kb + lr + 8 < n;
          sc[i][0] = v0 ? sc[i][0] : -INFINITY;
          sc[i][1] = v0 ? sc[i][1] : -INFINITY;
          sc[i][2] = v1 ? sc[i][2] : -INFINITY;
          sc[i][3] = v1 ? sc[i][3] : -INFINITY;
        }
      }
      // Lazy softmax: p = 2^(s * scale - m) with m only raised when some score
      // passes it by more than kLazy, so p <= 2^kLazy; no lane then needs the
      // column maximum, which costs shuffles.
      float x0 = fmaxf(sc[0][0], sc[0][2]), x1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
      for (int i = 1; i < PPI; ++i) {
        x0 = fmaxf(x0, fmaxf(sc[i][0], sc[i][2]));
        x1 = fmaxf(x1, fmaxf(sc[i][1], sc[i][3]));
      }
      x0 *= scale;
      x1 *= scale;
      if (__any_sync(0xffffffffu, x0 > m0 + kLazy || x1 > m1 + kLazy)) {
        float y0 = x0, y1 = x1;
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {  // over the 8 position rows of the tile
          y0 = fmaxf(y0, __shfl_xor_sync(0xffffffffu, y0, o_));
          y1 = fmaxf(y1, __shfl_xor_sync(0xffffffffu, y1, o_));
        }
        const float n0 = fmaxf(m0, y0), n1 = fmaxf(m1, y1);
        const float c0 = ex2_approx(m0 - n0), c1 = ex2_approx(m1 - n1);  // 0 on the first page
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
          o[mi][0] *= c0;
          o[mi][1] *= c1;
          o[mi][2] *= c0;
          o[mi][3] *= c1;
        }
        l0 *= c0;
        l1 *= c1;
        m0 = n0;
        m1 = n1;
      }
#pragma unroll
      for (int i = 0; i < PPI; ++i) {
        if (k + i >= npg) break;  // warp-uniform
        const float e0 = ex2_approx(fmaf(sc[i][0], scale, -m0));
        const float e1 = ex2_approx(fmaf(sc[i][1], scale, -m1));
        const float e2 = ex2_approx(fmaf(sc[i][2], scale, -m0));
        const float e3 = ex2_approx(fmaf(sc[i][3], scale, -m1));
        const uint32_t p01 = pack_bf16(e0, e1), p23 = pack_bf16(e2, e3);
        const uint32_t r01 = pack_bf16(e0 - bf16lo(p01), e1 - bf16hi(p01));
        const uint32_t r23 = pack_bf16(e2 - bf16lo(p23), e3 - bf16hi(p23));
        l0 += e0 + e2;
        l1 += e1 + e3;
        // P^T operands (hi and lo): (positions 2 lc (+1), head lr) and positions + 8
        const uint32_t pb0 = movmatrix_trans(p01);
        const uint32_t pb1 = movmatrix_trans(p23);
        const uint32_t rb0 = movmatrix_trans(r01);
        const uint32_t rb1 = movmatrix_trans(r23);
        uint32_t st, ph;
        slot_at(rs, rph, i, st, ph);
        const uint32_t slot = ring_u32 + st * SLOT;
        const int kb = (k + i) * P;
        if (kb + P <= n) {
#pragma unroll
          for (int mi = 0; mi < KS; ++mi) {
            uint32_t vf[4];
            ldsm_x4_trans(slot + voff[mi], vf);
            mma_16816(o[mi], vf, rb0, rb1);
            mma_16816(o[mi], vf, pb0, pb1);
          }
        } else {  // rows past the piece read row 0 instead (weighted 0)
          const bool past = kb + v_row >= n;
#pragma unroll
          for (int mi = 0; mi < KS; ++mi) {
            uint32_t vf[4];
            ldsm_x4_trans(slot + (past ? BLK + page_chunk_off(0, 2 * mi + v_ci) : voff[mi]), vf);
            mma_16816(o[mi], vf, rb0, rb1);
            mma_16816(o[mi], vf, pb0, pb1);
          }
        }
      }
      // refill the group's slots with the pages STAGES further on
      int pg[PPI];
#pragma unroll
      for (int i = 0; i < PPI; ++i) pg[i] = k + i + STAGES < npg ? page_id(k + i + STAGES) : -1;
      __syncwarp();
      if (lane == 0 && pg[0] >= 0) fence_proxy_async_smem();
#pragma unroll
      for (int i = 0; i < PPI; ++i) {
        if (pg[i] >= 0) {
          if (lane == 0) {
            uint32_t st, ph;
            slot_at(rs, rph, i, st, ph);
            issue_into(st, pg[i]);
          }
          ++issued;
        }
      }
      rs = ns;
      rph = nph;
    }
    if (failed) break;
    gk += npg;

#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
    }
    // o[mi]: (dim 16 mi + lr, h0), (.., h1), (dim 16 mi + lr + 8, h0), (.., h1)
    const int nch = a.tok_nchunks[t];
    const bool w0 = h0 < GRP, w1 = h1 < GRP;
    if (nch == 1) {
      const float i0 = 1.f / l0, i1 = 1.f / l1;
      __nv_bfloat16* o0 = a.o + (static_cast<size_t>(t) * n_q + g * GRP + h0) * D;
      __nv_bfloat16* o1 = o0 + D;
#pragma unroll
      for (int mi = 0; mi < KS; ++mi) {
        const int d0 = 16 * mi + lr;
        if (w0) {
          o0[d0] = __float2bfloat16_rn(o[mi][0] * i0);
          o0[d0 + 8] = __float2bfloat16_rn(o[mi][2] * i0);
        }
        if (w1) {
          o1[d0] = __float2bfloat16_rn(o[mi][1] * i1);
          o1[d0 + 8] = __float2bfloat16_rn(o[mi][3] * i1);
        }
      }
      continue;
    }
    constexpr int REC = partial_rec_floats(GRP, D);
    static_assert(REC % 4 == 0, "partial records must stay 16-byte aligned");
    const size_t row_rec = static_cast<size_t>(t) * a.max_chunks;
    float* rec = a.partials + ((row_rec + c) * n_kv + g) * REC;
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      const int d0 = 16 * mi + lr;
      if (w0) {
        rec[h0 * D + d0] = o[mi][0];
        rec[h0 * D + d0 + 8] = o[mi][2];
      }
      if (w1) {
        rec[h1 * D + d0] = o[mi][1];
        rec[h1 * D + d0 + 8] = o[mi][3];
      }
    }
    if (lr == 0) {
      if (w0) {
        rec[GRP * D + h0] = m0;
        rec[GRP * D + GRP + h0] = l0;
      }
      if (w1) {
        rec[GRP * D + h1] = m1;
        rec[GRP * D + GRP + h1] = l1;
      }
    }
    if (finish_piece(a, t, g, nch, lane))
      merge_row_partials<GRP, NCH, (WARPS <= 8 && GRP <= 4) ? 4 : 2>(a, t, g, nch, lane);
  }

  if (failed) raise_status(a.status, ST_TIMEOUT);
  // Launched as a programmatic dependent of the prefill kernel of the same
  // nano-batch (which writes other rows of o), this grid completes only after
  // that one, so whatever follows sees both.
  pdl_wait();
}

template <int GRP, int NCH, int WARPS, int STAGES, int PPI>
static cudaError_t launch_mma_t(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                int grid, bool programmatic, cudaStream_t stream) {
  const int smem = amma_smem_bytes(NCH * 64, WARPS, STAGES);
  const cudaError_t e = set_smem_limit(
      reinterpret_cast<const void*>(attn_mma_kernel<GRP, NCH, WARPS, STAGES, PPI>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(WARPS * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_mma_kernel<GRP, NCH, WARPS, STAGES, PPI>, tk, tv, a);
}

bool attention_mma_supported(int n_q, int n_kv, int head_dim, int page_size, int num_pages) {
  if (n_kv <= 0 || n_q % n_kv) return false;
  const int grp = n_q / n_kv;
  if (page_size != AMMA_P || (head_dim != 64 && head_dim != 128)) return false;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return false;
  // TMA row coordinates are 32-bit
  return static_cast<int64_t>(num_pages) * n_kv * page_size < (int64_t(1) << 31);
}

bool make_pool_tmap(CUtensorMap* map, const void* pool, int num_pages, int n_kv, int page_size,
                    int head_dim) {
  return make_tmap_bf16(map, pool, static_cast<uint64_t>(num_pages) * n_kv * page_size,
                        static_cast<uint64_t>(head_dim), static_cast<uint32_t>(page_size));
}

bool make_pool_tmap_pages(CUtensorMap* map, const void* pool, int num_pages, int n_kv,
                          int page_size, int head_dim) {
  if (head_dim != 128)
    return make_pool_tmap(map, pool, num_pages, n_kv, page_size, head_dim);
  return make_tmap_bf16_rows128(map, pool, static_cast<uint64_t>(num_pages) * n_kv * page_size,
                                static_cast<uint32_t>(page_size));
}

bool make_pool_tmap_groups(CUtensorMap* map, const void* pool, int num_pages, int n_kv,
                           int page_size, int head_dim) {
  if (head_dim != 128)
    return make_pool_tmap(map, pool, num_pages, n_kv, page_size, head_dim);
  return make_tmap_bf16_groups128(map, pool, static_cast<uint64_t>(num_pages) * n_kv * page_size);
}

cudaError_t launch_attention_mma(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                 int grid, bool programmatic, cudaStream_t stream) {
  if (grid <= 0 || !attention_mma_supported(a.n_q, a.n_kv, a.head_dim, a.page_size, a.num_pages))
    return cudaErrorInvalidValue;
  const int grp = a.n_q / a.n_kv, nch = a.head_dim / 64;
  // warps per CTA -> ring stages per warp (as deep as 227 KB of shared memory
  // allows) and pages per iteration (two pages per iteration measured slower
  // than one on every configuration, so all use one)
#define NF_AMMA_CFG(G, N)                                                  \
  switch (a.warps) {                                                       \
    case 4: return launch_mma_t<G, N, 4, 3, 1>(a, tk, tv, grid, programmatic, stream);   \
    case 5: return launch_mma_t<G, N, 5, 5, 1>(a, tk, tv, grid, programmatic, stream);   \
    case 6: return launch_mma_t<G, N, 6, 4, 1>(a, tk, tv, grid, programmatic, stream);   \
    case 7: return launch_mma_t<G, N, 7, 4, 1>(a, tk, tv, grid, programmatic, stream);   \
    case 8: return launch_mma_t<G, N, 8, 3, 1>(a, tk, tv, grid, programmatic, stream);   \
    case 10: return launch_mma_t<G, N, 10, 2, 1>(a, tk, tv, grid, programmatic, stream); \
    case 12: return launch_mma_t<G, N, 12, 2, 1>(a, tk, tv, grid, programmatic, stream); \
    case 14: return launch_mma_t<G, N, 14, 2, 1>(a, tk, tv, grid, programmatic, stream); \
    default: return cudaErrorInvalidValue;                                 \
  }
#define NF_AMMA_CASE(G, N) \
  if (grp == G && nch == N) { NF_AMMA_CFG(G, N) }
  NF_AMMA_CASE(1, 1) NF_AMMA_CASE(2, 1) NF_AMMA_CASE(4, 1) NF_AMMA_CASE(8, 1)
  NF_AMMA_CASE(1, 2) NF_AMMA_CASE(2, 2) NF_AMMA_CASE(4, 2) NF_AMMA_CASE(8, 2)
#undef NF_AMMA_CASE
#undef NF_AMMA_CFG
  return cudaErrorInvalidValue;
}

}  // namespace nf
