// Paged GQA decode attention, warp-specialised: one producer warp streams the
// K/V pages of every consumer warp, the consumer warps compute.
//
// Same operation, work list, split-KV records and per-page arithmetic as the
// tensor-core kernel in attn_mma.cu (S^T = K Q^T and O^T += V^T P^T with
// mma.sync m16n8k16, base-2 online softmax, P as bf16 hi + lo operands), so the
// two give the same bits.  What differs is who moves the bytes.  Decode
// attention is the memory-bound operation of the layer ("NanoFlow: Towards
// Optimal LLM Serving Throughput", "The Intra-Device Parallelism Mechanism");
// to run beside the GEMMs of another nano-batch it must draw HBM bandwidth from
// a fraction of the SMs, so what counts is bytes per second per SM.  In
// attn_mma.cu each warp issues its own copies between its pages, so its ring
// waits on the warp.  Here:
//   * consumer warp c owns a ring of SPC page slots; lane c of the producer
//     warp (warp WS_NC) keeps it full with TMA copies of the pages of c's
//     pieces, and can ask L2 to fetch pages ahead of the ring;
//   * the producer never waits on global memory: consumer c takes its pieces
//     (row, chunk, KV head) from the nano-batch's counter itself and publishes
//     each one, with its page ids, in one of two descriptor slots in shared
//     memory.  It fetches piece i + 1 while it computes piece i, one dependent
//     load per page (counter, work item, row data, page ids), so the loads'
//     latency hides behind its pages; only a piece shorter than the stages
//     finishes the fetch at its end;
//   * a consumer waits on its slot's full barrier, computes the page, and
//     arrives on the slot's empty barrier as soon as the V fragments are in
//     registers.
// Every wait is bounded; on expiry the kernel sets ST_TIMEOUT, the producer
// waits (bounded) for the copies it issued, and the CTA exits.
#include "attn_merge.cuh"
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace nf {

namespace {

// consumer warps: with the producer 12 warps, three on each SM sub-partition,
// which leaves 168 registers a thread
constexpr int WS_NC = 11;
constexpr int WS_MAX_PIECE_PAGES = 2048 / AMMA_P;

template <int NCH>
struct WsCfg {
  static constexpr int D = NCH * 64;
  static constexpr int BOX = AMMA_P * 128;       // one 64-column box of a page: 2 KB
  static constexpr int BLK = NCH * BOX;          // K (or V) of one (page, KV head)
  static constexpr int SLOT = 2 * BLK;
  static constexpr int SPC = NCH == 2 ? 2 : 4;   // slots per consumer
  static constexpr int NSLOT = WS_NC * SPC;
  // per consumer two piece descriptors: (t, chunk, KV head | stop, positions)
  // and the piece's page ids
  static constexpr int DESC_INTS = 4 + WS_MAX_PIECE_PAGES;
  static constexpr int OFF_DESC = NSLOT * SLOT;  // slots 1 KB aligned (128-byte swizzle)
  static constexpr int OFF_BAR = OFF_DESC + WS_NC * 2 * DESC_INTS * 4;
  // full and empty per slot, then one "published" barrier per descriptor
  static constexpr int OFF_FLAG = OFF_BAR + (2 * NSLOT + 2 * WS_NC) * 8;
  static constexpr int SMEM = 1024 + OFF_FLAG + 16;
};

constexpr int DESC_STOP = 1 << 30;  // in the KV-head word: no more pieces

}  // namespace

template <int GRP, int NCH>
__global__ void __launch_bounds__((WS_NC + 1) * 32, 1)
    attn_ws_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const AttnArgs a) {
  using Cfg = WsCfg<NCH>;
  constexpr int D = Cfg::D, P = AMMA_P, BOX = Cfg::BOX, BLK = Cfg::BLK, SLOT = Cfg::SLOT;
  constexpr int SPC = Cfg::SPC, KS = D / 16, DI = Cfg::DESC_INTS;
  static_assert(GRP >= 1 && GRP <= 8, "the GQA group must fit the 8 columns of a tile");
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  int* desc = reinterpret_cast<int*>(smem + Cfg::OFF_DESC);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* empty = full + Cfg::NSLOT;
  uint64_t* pub = empty + Cfg::NSLOT;  // [consumer][descriptor]
  volatile int* failed = reinterpret_cast<volatile int*>(smem + Cfg::OFF_FLAG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::NSLOT; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2 * WS_NC; ++s) mbar_init(&pub[s], 1);
    *failed = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int seg = a.seg;
  const int n_kv = a.n_kv;
  const uint64_t tmo = a.timeout_ns;

  if (warp == WS_NC) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    const uint64_t policy = l2_policy_evict_first();
    const bool feeder = lane < WS_NC;
    const int pfd = a.l2_prefetch;
    const size_t blk_elems = static_cast<size_t>(P) * D;  // one (page, KV head) block of a pool
    // this lane's consumer: the descriptor being issued and the ring position
    int g = 0, npg = 0, k = 0;
    const int* pid = nullptr;
    bool have = false, done = !feeder;
    uint32_t pieces = 0;  // descriptors taken
    uint32_t issued = 0;  // pages issued into the ring
    uint64_t last_progress = globaltimer_ns();
    bool timed_out = false;
    auto prefetch_page = [&](int j) {
      const size_t off = (static_cast<size_t>(pid[j]) * n_kv + g) * blk_elems;
      bulk_prefetch_l2(a.k_pool + off, BLK);
      bulk_prefetch_l2(a.v_pool + off, BLK);
    };
    for (;;) {
      bool progressed = false;
      if (!done && !have) {  // the consumer's next piece, once published
        const int q = static_cast<int>(pieces & 1);
        if (mbar_try_wait(&pub[lane * 2 + q], (pieces >> 1) & 1)) {
          const int* d = desc + (lane * 2 + q) * DI;
          ++pieces;
          progressed = true;
          if (d[2] & DESC_STOP) {
            done = true;
          } else {
            g = d[2];
            npg = (d[3] + P - 1) / P;
            pid = d + 4;
            k = 0;
            have = true;
            for (int j = SPC; j < npg && j < SPC + pfd; ++j) prefetch_page(j);
          }
        }
      }
      if (have) {  // one page into the consumer's next slot
        const int sl = lane * SPC + static_cast<int>(issued % SPC);
        if (issued < SPC || mbar_try_wait(&empty[sl], ((issued / SPC) - 1) & 1)) {
          uint8_t* dst = smem + static_cast<size_t>(sl) * SLOT;
          const int y = (pid[k] * n_kv + g) * P;
          if (issued >= SPC) fence_proxy_async_smem();  // the consumer's reads of the slot first
          mbar_arrive_expect_tx(&full[sl], SLOT);
#pragma unroll
          for (int b = 0; b < NCH; ++b)
            tma_load_2d_hint(dst + b * BOX, &tmK, &full[sl], b * 64, y, policy);
#pragma unroll
          for (int b = 0; b < NCH; ++b)
            tma_load_2d_hint(dst + BLK + b * BOX, &tmV, &full[sl], b * 64, y, policy);
          if (pfd > 0 && k + SPC + pfd < npg) prefetch_page(k + SPC + pfd);
          if (++k == npg) have = false;
          ++issued;
          progressed = true;
        }
      }
      const uint64_t now = globaltimer_ns();
      if (__any_sync(0xffffffffu, progressed)) last_progress = now;
      if (__all_sync(0xffffffffu, done)) break;
      const bool other = __any_sync(0xffffffffu, *failed != 0);
      if (other || __any_sync(0xffffffffu, now - last_progress > tmo)) {
        timed_out = !other;
        break;
      }
    }
    if (timed_out) {
      *failed = 1;
      if (lane == 0) raise_status(a.status, ST_TIMEOUT);
    }
    // no copy may land after the CTA exits: wait (bounded) for the last slots
    // this lane filled
    if (feeder) {
      const uint32_t from = issued > SPC ? issued - SPC : 0;
      for (uint32_t i = from; i < issued; ++i)
        mbar_wait(&full[lane * SPC + static_cast<int>(i % SPC)], (i / SPC) & 1, tmo);
    }
    pdl_wait();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int lr = lane >> 2, lc = lane & 3;  // fragment row / column pair of this lane
  const int mj = lane >> 3, mr = lane & 7;
  const int k_row = mr + 8 * (mj & 1), k_ci = mj >> 1;
  const int v_row = mr + 8 * (mj >> 1), v_ci = mj & 1;
  const int h0 = 2 * lc, h1 = 2 * lc + 1;  // the two heads of this lane's accumulator columns
  const bool w0 = h0 < GRP, w1 = h1 < GRP;
  constexpr float kLazy = 8.0f;
  const float scale = a.scale_log2;
  const uint32_t slots_u32 = smem_u32(smem);
  const int begin = a.seg_items[seg];
  const int total = (a.seg_items[seg + 1] - begin) * n_kv;
  const int C = a.kv_chunk;

  // The next piece, fetched in stages (one per computed page): 0 take an index
  // from the counter; 1 read the work item; 2 read the row's sequence,
  // position and piece count; 3 read the page ids and the row's q; 4 publish
  // it.  5: published (or no piece left: nx_stop).
  int st = 0, nx_idx = 0, nx_t = 0, nx_ch = 0, nx_g = 0, nx_s = 0, nx_pos = 0, nx_nch = 0;
  int nx_n = 0;
  bool nx_stop = false;
  int nx_pid[WS_MAX_PIECE_PAGES / 32];
  uint32_t nx_q[KS][2];
  uint32_t published = 0;
  auto stage = [&]() {  // warp-uniform
    switch (st) {
      case 0:
        if (lane == 0) nx_idx = atomicAdd(&a.fetch[seg], 1);
        st = 1;
        break;
      case 1: {
        nx_idx = __shfl_sync(0xffffffffu, nx_idx, 0);
        if (nx_idx >= total) {
          nx_stop = true;
          st = 4;
          break;
        }
        const int pair = begin + nx_idx / n_kv;
        nx_g = nx_idx % n_kv;
        nx_t = a.items[2 * pair];
        nx_ch = a.items[2 * pair + 1];
        st = 2;
        break;
      }
      case 2:
        nx_s = a.tok_seq[nx_t];
        nx_pos = a.tok_pos[nx_t];
        nx_nch = a.tok_nchunks[nx_t];
        st = 3;
        break;
      case 3: {
        if (a.prefill_elsewhere && nx_s >= a.n_decode_seqs) {  // the prefill kernel's row
          st = 0;
          break;
        }
        const int b0 = nx_ch * C;
        nx_n = min(C, nx_pos + 1 - b0);
        const int npg = (nx_n + P - 1) / P;
        const int* bt = a.block_table + static_cast<size_t>(nx_s) * a.max_pages + b0 / P;
#pragma unroll
        for (int r = 0; r < WS_MAX_PIECE_PAGES / 32; ++r) {
          const int j = lane + 32 * r;
          nx_pid[r] = j < npg ? bt[j] : 0;
        }
        // Q^T as the B operand of S^T = K Q^T: column n = head lr of the group
        // (zero past GRP), rows = dims 16 kk + 2 lc (+1) and + 8
        const bool hv = lr < GRP;
        const __nv_bfloat16* qrow =
            a.q + (static_cast<size_t>(nx_t) * a.n_q + nx_g * GRP + (hv ? lr : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint32_t x0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * lc);
          const uint32_t x1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * lc);
          nx_q[kk][0] = hv ? x0 : 0u;
          nx_q[kk][1] = hv ? x1 : 0u;
        }
        st = 4;
        break;
      }
      case 4: {
        int* d = desc + (warp * 2 + static_cast<int>(published & 1)) * DI;
        if (nx_stop) {
          if (lane == 0) d[2] = DESC_STOP;
        } else {
          const int npg = (nx_n + P - 1) / P;
#pragma unroll
          for (int r = 0; r < WS_MAX_PIECE_PAGES / 32; ++r) {
            const int j = lane + 32 * r;
            if (j < npg) {
              int page = nx_pid[r];
              if (page < 0 || page >= a.num_pages) {  // never read outside the pool
                raise_status(a.status, ST_BAD_PAGE);
                page = 0;
              }
              d[4 + j] = page;
            }
          }
          if (lane == 0) {
            d[0] = nx_t;
            d[1] = nx_ch;
            d[2] = nx_g;
            d[3] = nx_n;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pub[warp * 2 + static_cast<int>(published & 1)]);
        ++published;
        st = 5;
        break;
      }
      default:
        break;
    }
  };

  // the first piece at once, then each next one in stages
  while (st < 5) stage();
  uint32_t qb[KS][2];
  float o[KS][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  uint32_t r = 0;  // pages taken from the ring
  while (!nx_stop && !__any_sync(0xffffffffu, *failed != 0)) {
    // the published piece becomes the current one; the fetch of the next starts
    const int t = nx_t, ch = nx_ch, g = nx_g, n = nx_n, nch = nx_nch;
    const int npg = (n + P - 1) / P;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qb[kk][0] = nx_q[kk][0];
      qb[kk][1] = nx_q[kk][1];
    }
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
    st = 0;
    bool ok = true;
    for (int k = 0; k < npg; ++k, ++r) {
      const int sl = warp * SPC + static_cast<int>(r % SPC);
      if (!__all_sync(0xffffffffu, mbar_wait(&full[sl], (r / SPC) & 1, tmo, failed))) {
        ok = false;
        break;
      }
      const uint32_t slot = slots_u32 + static_cast<uint32_t>(sl) * SLOT;
      // S^T[16 pos x 8 heads] = K Q^T, two independent MMA chains
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t af[4];
        ldsm_x4(slot + page_chunk_off(k_row, 2 * kk + k_ci), af);
        if (kk & 1)
          mma_16816(s2, af, qb[kk][0], qb[kk][1]);
        else
          mma_16816(sc, af, qb[kk][0], qb[kk][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[i] += s2[i];
      // positions past the piece may hold anything, even NaN: they become -inf
      const int kb = k * P;
      const bool tail = kb + P > n;  // warp-uniform
      if (tail) {
        const bool v0 = kb + lr < n, v1 = kb + lr + 8 < n;
        sc[0] = v0 ? sc[0] : -INFINITY;
        sc[1] = v0 ? sc[1] : -INFINITY;
        sc[2] = v1 ? sc[2] : -INFINITY;
        sc[3] = v1 ? sc[3] : -INFINITY;
      }
      // lazy softmax: the reference maximum rises only when a score passes it by kLazy
      const float x0 = fmaxf(sc[0], sc[2]) * scale, x1 = fmaxf(sc[1], sc[3]) * scale;
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
      const float e0 = ex2_approx(fmaf(sc[0], scale, -m0));
      const float e1 = ex2_approx(fmaf(sc[1], scale, -m1));
      const float e2 = ex2_approx(fmaf(sc[2], scale, -m0));
      const float e3 = ex2_approx(fmaf(sc[3], scale, -m1));
      const uint32_t p01 = pack_bf16(e0, e1), p23 = pack_bf16(e2, e3);
      const uint32_t r01 = pack_bf16(e0 - bf16lo(p01), e1 - bf16hi(p01));
      const uint32_t r23 = pack_bf16(e2 - bf16lo(p23), e3 - bf16hi(p23));
      l0 += e0 + e2;
      l1 += e1 + e3;
      const uint32_t pb0 = movmatrix_trans(p01), pb1 = movmatrix_trans(p23);
      const uint32_t rb0 = movmatrix_trans(r01), rb1 = movmatrix_trans(r23);
      // O^T[d x 8] += V^T P^T; V rows past the piece read row 0 instead (weighted 0)
      const bool past = tail && kb + v_row >= n;
      uint32_t vf[KS][4];
#pragma unroll
      for (int mi = 0; mi < KS; ++mi)
        ldsm_x4_trans(slot + BLK + page_chunk_off(past ? 0 : v_row, 2 * mi + v_ci), vf[mi]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sl]);  // the slot's data is in registers
#pragma unroll
      for (int mi = 0; mi < KS; ++mi) {
        mma_16816(o[mi], vf[mi], rb0, rb1);
        mma_16816(o[mi], vf[mi], pb0, pb1);
      }
      stage();  // one step of the next piece's fetch
    }
    if (!ok) {
      if (!*failed) {
        *failed = 1;
        if (lane == 0) raise_status(a.status, ST_TIMEOUT);
      }
      break;
    }
    while (st < 5) stage();  // a short piece: finish the next one's fetch now

    // the piece is done: write o (a row in one piece) or its partial record
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
    }
    if (nch == 1) {
      const float i0 = 1.f / l0, i1 = 1.f / l1;
      __nv_bfloat16* o0 = a.o + (static_cast<size_t>(t) * a.n_q + g * GRP + h0) * D;
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
    float* rec = a.partials + ((static_cast<size_t>(t) * a.max_chunks + ch) * n_kv + g) * REC;
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
    if (finish_piece(a, t, g, nch, lane)) merge_row_partials<GRP, NCH, 2>(a, t, g, nch, lane);
  }
  // Launched as a programmatic dependent of the prefill kernel of the same
  // nano-batch (which writes other rows of o), this grid completes only after
  // that one, so whatever follows sees both.
  pdl_wait();
}

template <int GRP, int NCH>
static cudaError_t launch_ws_t(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                               int grid, bool programmatic, cudaStream_t stream) {
  const int smem = WsCfg<NCH>::SMEM;
  const cudaError_t e =
      set_smem_limit(reinterpret_cast<const void*>(attn_ws_kernel<GRP, NCH>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3((WS_NC + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_ws_kernel<GRP, NCH>, tk, tv, a);
}

cudaError_t launch_attention_ws(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                int grid, bool programmatic, cudaStream_t stream) {
  if (grid <= 0 || !attention_mma_supported(a.n_q, a.n_kv, a.head_dim, a.page_size, a.num_pages) ||
      a.kv_chunk > WS_MAX_PIECE_PAGES * AMMA_P)
    return cudaErrorInvalidValue;
  const int grp = a.n_q / a.n_kv;
  const int nch = a.head_dim / 64;
#define NF_WS_CASE(G, N) \
  if (grp == G && nch == N) return launch_ws_t<G, N>(a, tk, tv, grid, programmatic, stream);
  NF_WS_CASE(1, 1) NF_WS_CASE(2, 1) NF_WS_CASE(4, 1) NF_WS_CASE(8, 1)
  NF_WS_CASE(1, 2) NF_WS_CASE(2, 2) NF_WS_CASE(4, 2) NF_WS_CASE(8, 2)
#undef NF_WS_CASE
  return cudaErrorInvalidValue;
}

}  // namespace nf
