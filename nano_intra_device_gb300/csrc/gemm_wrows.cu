// Tensor-core GEMM for nano-operations of few tokens (decode-sized batches):
// the weight rows are the 128-row MMA operand and the tokens its N side.
//
// The KQV, O and Up/Gate/Down projections ("NanoFlow: Towards Optimal LLM
// Serving Throughput", "The Intra-Device Parallelism Mechanism") stream their
// weights once when a nano-operation holds at most 128 tokens, so they are
// bound by HBM, and the 128 x 256 token-row tiles of gemm_tc.cu then compute
// half-empty tiles on a few dozen SMs.  Here:
//  * a tile is 128 output features x TOK tokens (TOK = 64 or 128), so every
//    accumulator lane is a real output feature;
//  * the K range of a tile is split over the CTAs of a thread-block cluster
//    (up to 8), so that a hundred or more SMs stream disjoint slices of the
//    weights.  The partial tiles are summed through distributed shared memory:
//    each CTA copies its accumulator to its own shared memory, then each rank
//    adds the copies of all ranks, in rank order, for a disjoint share of the
//    tile's tokens and runs the epilogue on it.  No global partials, no serial
//    reduction tail, and the sum does not depend on timing;
//  * SwiGLU loads the gate and the up rows of the same 128 features as two A
//    operands into two accumulators, and QKV the first and the second half of
//    each head's dimensions, so that every pair the epilogue combines (gate
//    with up, RoPE's dimensions i and i + d/2) is in one thread;
//  * when every CTA has at most one tile (the usual case: clusters are sized
//    so), the exchange copy reuses the ring, which is idle by then, and the
//    ring gets the room: more weight bytes in flight per SM;
//  * launched as a programmatic dependent, a CTA fills its ring with weights
//    (which no kernel writes) before it waits for the kernel ahead of it, so
//    the weight stream starts while that kernel finishes;
//  * every wait is bounded.  The CTAs of a cluster walk the same tiles and
//    exchange rounds, also after an error (with zeros in place of the
//    accumulator), and meet at a cluster barrier before they exit, so no CTA
//    leaves while a peer may still address its shared memory.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace nf {
namespace {

constexpr int WR_BM = 128;             // weight rows (output features) per tile
constexpr int WR_BK = 64;              // K per ring stage: one 128-byte swizzled row
constexpr int WR_XC = 64;              // tokens per exchange round
constexpr int WR_THREADS = 192;
constexpr int WR_MAX_STAGES = 12;
constexpr int WR_MAX_CLUSTER = 8;      // portable cluster size
constexpr int WR_SMEM_LIMIT = 232448;  // opt-in shared memory of a CTA
constexpr int WR_TAIL = 512;

// ONE: every CTA has at most one tile, and the exchange copy (XBUF) reuses
// the ring; otherwise it has room of its own.
template <int EPI, int TOK, bool ONE>
struct WrCfg {
  static constexpr int NA = (EPI == EPI_SWIGLU || EPI == EPI_QKV) ? 2 : 1;  // A operands
  static constexpr int W_BYTES = WR_BM * WR_BK * 2;
  static constexpr int X_BYTES = TOK * WR_BK * 2;
  static constexpr int STAGE = NA * W_BYTES + X_BYTES;
  static constexpr int XBUF = NA * WR_XC * WR_BM * 4;  // fp32 copy of one round
  static constexpr int FIT = (WR_SMEM_LIMIT - 1024 - WR_TAIL - (ONE ? 0 : XBUF)) / STAGE;
  static constexpr int STAGES = FIT < WR_MAX_STAGES ? FIT : WR_MAX_STAGES;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM =
      1024 + (ONE ? (RING > XBUF ? RING : XBUF) : RING + XBUF) + WR_TAIL;
  static constexpr int ACC = NA * TOK;  // TMEM columns of one accumulator set
  static constexpr int TMEM = 2 * ACC;  // double buffered
  static_assert(STAGES >= 2 && SMEM <= WR_SMEM_LIMIT, "ring");
  static_assert(TMEM == 128 || TMEM == 256 || TMEM == 512, "TMEM allocation");
  static_assert(TOK % WR_XC == 0 && TOK <= 256, "token tile");
};

struct WrTail {
  uint64_t full[WR_MAX_STAGES];
  uint64_t empty[WR_MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t epi_sync;  // rendezvous of the four epilogue warps
  uint64_t xready;    // every rank has written its copy of the round
  uint64_t xdone;     // every rank has read this CTA's copy of the round
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(WrTail) <= WR_TAIL, "barrier block exceeds its reservation");

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  return make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}

template <int EPI, int TOK, bool ONE>
__global__ void __launch_bounds__(WR_THREADS, 1)
    gemm_wrows_kernel(const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmW2,
                      const __grid_constant__ CUtensorMap tmX, const GemmArgs args) {
  using Cfg = WrCfg<EPI, TOK, ONE>;
  pdl_trigger();
  constexpr int NA = Cfg::NA, STAGES = Cfg::STAGES;
  constexpr uint32_t IDESC = idesc_bf16_f32(WR_BM, TOK);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float* xbuf = reinterpret_cast<float*>(ONE ? smem : smem + Cfg::RING);
  WrTail* tail = reinterpret_cast<WrTail*>(smem + Cfg::SMEM - 1024 - WR_TAIL);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = args.splits;  // CTAs of a cluster = K splits of a tile
  const int rank = static_cast<int>(cluster_rank());
  const int first = static_cast<int>(cluster_id_x());
  const int stride = static_cast<int>(cluster_count_x());
  const int n_tiles = args.n_tiles * args.m_tiles;  // weight tiles x token tiles
  const int nk = (args.K + WR_BK - 1) / WR_BK;
  const int kb0 = rank * nk / S, kb1 = (rank + 1) * nk / S;
  // A tile walks its K range from an offset that spreads the tiles evenly over
  // it, so that the CTAs, which start together, do not all read the same
  // 128-byte column of the weight rows (rows 2K bytes apart) at once; the sum
  // order is a function of the tile alone.
  const int klen = kb1 - kb0;
  auto kb_at = [&](int wt, int i) {
    const int rot = static_cast<int>((static_cast<long long>(wt) * klen) / args.n_tiles) % klen;
    const int j = i + rot;
    return kb0 + (j >= klen ? j - klen : j);
  };
  const uint64_t tmo = args.timeout_ns;
  // QKV: a tile holds 256 / d heads; its first A operand is dimensions
  // [0, d/2) of each, its second [d/2, d)
  const int d = args.head_dim, half = d / 2;
  const int hp = EPI == EPI_QKV ? 2 * WR_BM / d : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tail->tfull[a], 1);
      mbar_init(&tail->tempty[a], 128);
    }
    mbar_init(&tail->drain, 1);
    mbar_init(&tail->epi_sync, 4);
    mbar_init(&tail->xready, S);
    mbar_init(&tail->xdone, S);
    tail->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmW);
    if (EPI == EPI_SWIGLU) prefetch_tensormap(&tmW2);
    prefetch_tensormap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, Cfg::TMEM);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // every peer's barriers exist before anyone arrives on them
  const uint32_t tmem_base = tail->tmem_base;
  volatile int* abort_flag = &tail->abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      // the weight rows of k block kb of weight tile wt into ring stage sa
      auto load_w = [&](uint8_t* sa, uint64_t* bar, int kb, int wt) {
        const int kx = kb * WR_BK;
        mbar_arrive_expect_tx(bar, Cfg::STAGE);
        if (EPI == EPI_QKV) {
          for (int i = 0; i < hp; ++i) {
            const int row = (wt * hp + i) * d;
            tma_load_2d(sa + i * half * 128, &tmW, bar, kx, row);
            tma_load_2d(sa + Cfg::W_BYTES + i * half * 128, &tmW, bar, kx, row + half);
          }
        } else if (EPI == EPI_SWIGLU) {
          tma_load_2d(sa, &tmW, bar, kx, wt * WR_BM);
          tma_load_2d(sa + Cfg::W_BYTES, &tmW2, bar, kx, args.b2_row_off + wt * WR_BM);
        } else {
          tma_load_2d(sa, &tmW, bar, kx, wt * WR_BM);
        }
      };
      // the first ring of weights does not depend on the kernel ahead
      const int pre = first < n_tiles ? min(STAGES, klen) : 0;
      for (int i = 0; i < pre; ++i)
        load_w(smem + i * Cfg::STAGE, &tail->full[i], kb_at(first / args.m_tiles, i),
               first / args.m_tiles);
      pdl_wait();
      uint32_t st = 0, ph = 0;
      uint32_t issued_mask = 0, last_ph[WR_MAX_STAGES] = {};
      bool ok = true;
      for (int tile = first; tile < n_tiles && ok; tile += stride) {
        const int wt = tile / args.m_tiles, tt = tile % args.m_tiles;
        const int x_row = args.m_begin + tt * TOK;
        for (int i = 0; i < klen; ++i) {
          const int kb = kb_at(wt, i);
          if (!mbar_wait(&tail->empty[st], ph ^ 1, tmo, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + st * Cfg::STAGE;
          uint64_t* bar = &tail->full[st];
          if (tile != first || i >= pre) load_w(sa, bar, kb, wt);
          tma_load_2d(sa + NA * Cfg::W_BYTES, &tmX, bar, kb * WR_BK, x_row);
          issued_mask |= 1u << st;
          last_ph[st] = ph;
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        raise_status(args.status, ST_TIMEOUT);
        *abort_flag = 1;
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) mbar_wait(&tail->full[s], last_ph[s], tmo);
      }
    }
    if (lane != 0) pdl_wait();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    pdl_wait();
    if (lane == 0) {
      uint32_t st = 0, ph = 0, acc = 0, aph = 0;
      bool ok = true, any = false;
      for (int tile = first; tile < n_tiles && ok; tile += stride) {
        if (!mbar_wait(&tail->tempty[acc], aph ^ 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * Cfg::ACC;
        for (int i = 0; i < klen; ++i) {
          if (!mbar_wait(&tail->full[st], ph, tmo, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + st * Cfg::STAGE);
          const uint64_t a0 = desc_sw128_kmajor(sa);
          const uint64_t a1 = desc_sw128_kmajor(sa + Cfg::W_BYTES);
          const uint64_t xd = desc_sw128_kmajor(sa + NA * Cfg::W_BYTES);
#pragma unroll
          for (int k = 0; k < WR_BK / 16; ++k) {
            const uint32_t accum = (i != 0) || (k != 0);
            tc_mma_bf16(d_tmem, a0 + 2 * k, xd + 2 * k, IDESC, accum);
            if (NA == 2) tc_mma_bf16(d_tmem + TOK, a1 + 2 * k, xd + 2 * k, IDESC, accum);
          }
          any = true;
          tc_commit(&tail->empty[st]);
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tail->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1;
        }
      }
      if (!ok) {
        raise_status(args.status, ST_TIMEOUT);
        *abort_flag = 1;
        if (any) {
          tc_commit(&tail->drain);
          mbar_wait(&tail->drain, 0, tmo);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    pdl_wait();
    const int et = threadIdx.x - 64;  // 0 .. 127
    const int quarter = warp & 3;     // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t xready_addr = smem_u32(&tail->xready), xdone_addr = smem_u32(&tail->xdone);
    uint32_t acc = 0, aph = 0, esync = 0, xr = 0;
    bool ok = true;  // false after a failed wait; the exchange rounds still run
    auto fail = [&]() {
      if (ok) {
        raise_status(args.status, ST_TIMEOUT);
        *abort_flag = 1;
        ok = false;
      }
    };
    auto epi_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->epi_sync);
      const bool got =
          __all_sync(0xffffffffu, mbar_wait(&tail->epi_sync, esync & 1, tmo, abort_flag));
      ++esync;
      if (!got) fail();
    };
    // elected thread: one arrival on the barrier at `addr` of every rank
    auto arrive_all = [&](uint32_t addr) {
      if (warp == 2 && lane == 0) {
        fence_acq_rel_cluster();
        for (int j = 0; j < S; ++j) mbar_arrive_remote(cluster_map(addr, j));
      }
    };
    // The epilogue of one batch of this rank's share of a round: quads (4
    // consecutive features of one token) eb, eb + 128, ..., eb + 128 (QB - 1)
    // of the share's nq quads, token c0 + e / 32 of the round and features
    // (e % 32) * 4 of the tile.  Global operands are fetched for the whole
    // batch first and the partial tiles of RG ranks next, all loaded before
    // any is added (a peer's shared memory is a round trip away, about a
    // microsecond under load), so their latencies overlap instead of adding up
    // rank by rank; this CTA's own copy is read from its shared memory.
    constexpr int QB = 4, RG = EPI == EPI_QKV ? 3 : 4;
    // QKV: the positions, cache slots and RoPE (cos, sin) of a batch's quads,
    // which do not depend on the products (a tile's first batch is fetched
    // before its products are ready)
    struct QkvIn {
      int pos[QB], slot[QB];
      float4 cs0[QB], cs1[QB];
    };
    auto qkv_fetch = [&](int wt, int tr0, int c0, int eb, int nq, QkvIn& q) {
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const int e = eb + 128 * i;
        q.pos[i] = 0;
        q.slot[i] = -1;
        q.cs0[i] = q.cs1[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < nq) {
          const int t = tr0 + c0 + e / 32;
          q.pos[i] = __ldg(args.tok_pos + t);
          q.slot[i] = __ldg(args.tok_slot + t);
        }
      }
#pragma unroll
      for (int i = 0; i < QB; ++i) {  // RoPE (cos, sin) from the table
        const int e = eb + 128 * i;
        const int q4 = (e % 32) * 4, jh = q4 % half;
        if (e < nq && wt * hp + q4 / half < args.n_q + args.n_kv && q.pos[i] < args.rope_positions) {
          const float4* cs =
              reinterpret_cast<const float4*>(args.rope_cs + static_cast<size_t>(q.pos[i]) * half + jh);
          q.cs0[i] = __ldg(cs);
          q.cs1[i] = __ldg(cs + 1);
        }
      }
    };
    auto reduce_batch = [&](int wt, int tr0, int c0, int eb, int nq, const QkvIn* pre) {
      uint2 rr[QB];
      QkvIn qi;
      if (EPI == EPI_QKV) {
        if (pre) qi = *pre;
        else qkv_fetch(wt, tr0, c0, eb, nq, qi);
      }
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const int e = eb + 128 * i;
        rr[i] = make_uint2(0u, 0u);
        if (e < nq) {
          const int t = tr0 + c0 + e / 32, q4 = (e % 32) * 4;
          if (EPI == EPI_RESID && wt * WR_BM + q4 < args.N)
            rr[i] = __ldg(reinterpret_cast<const uint2*>(args.R + static_cast<size_t>(t) * args.ldr +
                                                         wt * WR_BM + q4));
        }
      }
      float4 s0[QB], s1[QB];
#pragma unroll
      for (int i = 0; i < QB; ++i) s0[i] = s1[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j0 = 0; j0 < WR_MAX_CLUSTER; j0 += RG) {
        if (j0 < S) {
          float4 p0[RG][QB], p1[RG][QB];
#pragma unroll
          for (int jj = 0; jj < RG; ++jj) {
            const int j = j0 + jj, jv = j < S ? j : rank;  // jv: an address that exists
            const float* src = jv == rank
                                   ? xbuf
                                   : static_cast<const float*>(__cluster_map_shared_rank(xbuf, jv));
#pragma unroll
            for (int i = 0; i < QB; ++i) {
              const int e = eb + 128 * i;
              const int idx = (c0 + e / 32) * WR_BM + (e % 32) * 4;
              const bool on = j < S && e < nq;
              p0[jj][i] = on ? *reinterpret_cast<const float4*>(src + idx) : z4;
              if (NA == 2)
                p1[jj][i] = on ? *reinterpret_cast<const float4*>(src + WR_XC * WR_BM + idx) : z4;
            }
          }
          // rank order: the sum does not depend on timing
#pragma unroll
          for (int jj = 0; jj < RG; ++jj) {
            if (j0 + jj < S) {
#pragma unroll
              for (int i = 0; i < QB; ++i) {
                s0[i].x += p0[jj][i].x; s0[i].y += p0[jj][i].y;
                s0[i].z += p0[jj][i].z; s0[i].w += p0[jj][i].w;
                if (NA == 2) {
                  s1[i].x += p1[jj][i].x; s1[i].y += p1[jj][i].y;
                  s1[i].z += p1[jj][i].z; s1[i].w += p1[jj][i].w;
                }
              }
            }
          }
        }
      }
      if (EPI == EPI_QKV) {
        const int nqh = args.n_q, nkv = args.n_kv;
#pragma unroll
        for (int i = 0; i < QB; ++i) {
          const int e = eb + 128 * i;
          if (e >= nq) continue;
          const int t = tr0 + c0 + e / 32, q4 = (e % 32) * 4;
          const int head = wt * hp + q4 / half, j = q4 % half;
          if (head >= nqh + 2 * nkv) continue;
          __nv_bfloat16* dst;
          if (head < nqh) {
            dst = args.q_out + static_cast<size_t>(t) * nqh * d + static_cast<size_t>(head) * d + j;
          } else {
            if (qi.slot[i] < 0) continue;
            const bool is_k = head < nqh + nkv;
            const int gh = is_k ? head - nqh : head - nqh - nkv;
            const int P = args.page_size;
            __nv_bfloat16* pool = is_k ? args.k_pool : args.v_pool;
            dst = pool + static_cast<size_t>(qi.slot[i] / P) * nkv * P * d +
                  static_cast<size_t>(gh) * P * d + static_cast<size_t>(qi.slot[i] % P) * d + j;
          }
          float lo[4] = {s0[i].x, s0[i].y, s0[i].z, s0[i].w};
          float hi[4] = {s1[i].x, s1[i].y, s1[i].z, s1[i].w};
          if (head < nqh + nkv) {  // RoPE on q and k: rotate (i, i + d/2) by pos theta^(-2i/d)
            float c[4], sn[4];
            if (qi.pos[i] < args.rope_positions) {
              c[0] = qi.cs0[i].x; sn[0] = qi.cs0[i].y; c[1] = qi.cs0[i].z; sn[1] = qi.cs0[i].w;
              c[2] = qi.cs1[i].x; sn[2] = qi.cs1[i].y; c[3] = qi.cs1[i].z; sn[3] = qi.cs1[i].w;
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float inv_freq = exp2f(-(2.0f * (j + k) / d) * args.log2_theta);
                sincosf(static_cast<float>(qi.pos[i]) * inv_freq, &sn[k], &c[k]);
              }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a = lo[k], b = hi[k];
              lo[k] = a * c[k] - b * sn[k];
              hi[k] = b * c[k] + a * sn[k];
            }
          }
          *reinterpret_cast<uint2*>(dst) = pack4_bf16(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint2*>(dst + half) = pack4_bf16(hi[0], hi[1], hi[2], hi[3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < QB; ++i) {
          const int e = eb + 128 * i;
          if (e >= nq) continue;
          const int t = tr0 + c0 + e / 32, f = wt * WR_BM + (e % 32) * 4;
          if (f >= args.N) continue;  // N is a multiple of 4
          float o[4] = {s0[i].x, s0[i].y, s0[i].z, s0[i].w};
          if (EPI == EPI_SWIGLU) {
            const float u[4] = {s1[i].x, s1[i].y, s1[i].z, s1[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = __fdividef(o[k], 1.0f + __expf(-o[k])) * u[k];
          } else if (EPI == EPI_RESID) {
            o[0] += bf16lo(rr[i].x);
            o[1] += bf16hi(rr[i].x);
            o[2] += bf16lo(rr[i].y);
            o[3] += bf16hi(rr[i].y);
          }
          *reinterpret_cast<uint2*>(args.C + static_cast<size_t>(t) * args.ldc + f) =
              pack4_bf16(o[0], o[1], o[2], o[3]);
        }
      }
    };

    for (int tile = first; tile < n_tiles; tile += stride) {
      const int wt = tile / args.m_tiles, tt = tile % args.m_tiles;
      const int t0 = args.m_begin + tt * TOK;
      const int nv = min(TOK, args.m_end - t0);  // tokens of this tile
      QkvIn qpre;  // QKV: the inputs of this thread's first batch of round 0
      if (EPI == EPI_QKV) {
        const int ntok = min(WR_XC, nv);
        const int c0 = rank * ntok / S, c1 = (rank + 1) * ntok / S;
        qkv_fetch(wt, t0, c0, et, (c1 - c0) * 32, qpre);
      }
      // warp-uniform: tcgen05.ld below is .sync.aligned
      const bool have =
          ok && __all_sync(0xffffffffu, mbar_wait(&tail->tfull[acc], aph, tmo, abort_flag));
      if (!have) fail();
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * Cfg::ACC;
      if (EPI != EPI_QKV && S == 1) {
        // The whole K range is in this accumulator: each thread finishes its
        // feature (accumulator row) for the tile's tokens straight from tensor
        // memory, 32 tokens a load, without the exchange copy.  A warp's stores
        // of one token cover 32 consecutive features (64 bytes).
        const int f = wt * WR_BM + row;
#pragma unroll 1
        for (int c = 0; c * 32 < nv; ++c) {
          uint32_t v0[32], v1[32];
          if (have) {
            tc_ld_32x32b_x32(tb + c * 32, v0);
            if (NA == 2) tc_ld_32x32b_x32(tb + TOK + c * 32, v1);
            tc_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v0[i] = v1[i] = 0u;
          }
          const int nt = min(32, nv - c * 32);
          if (f < args.N) {
            const size_t r0 = static_cast<size_t>(t0 + c * 32);
            float rv[32];
            if (EPI == EPI_RESID) {  // all residual loads in flight before the stores
#pragma unroll
              for (int i = 0; i < 32; ++i)
                rv[i] = i < nt ? __bfloat162float(__ldg(args.R + (r0 + i) * args.ldr + f)) : 0.f;
            }
            __nv_bfloat16* dst = args.C + r0 * args.ldc + f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i < nt) {
                float o = __uint_as_float(v0[i]);
                if (EPI == EPI_SWIGLU) o = __fdividef(o, 1.0f + __expf(-o)) * __uint_as_float(v1[i]);
                if (EPI == EPI_RESID) o += rv[i];
                dst[static_cast<size_t>(i) * args.ldc] = __float2bfloat16_rn(o);
              }
            }
          }
        }
        tc_fence_before();  // the accumulator is free for the tile after next
        mbar_arrive(&tail->tempty[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1;
        }
        continue;
      }
      const int rounds = (nv + WR_XC - 1) / WR_XC;
      for (int g = 0; g < rounds; ++g) {
        // every rank must have read this CTA's previous copy before it is overwritten
        if (xr > 0 &&
            !__all_sync(0xffffffffu, mbar_wait_cluster(&tail->xdone, (xr - 1) & 1, tmo, abort_flag)))
          fail();
        // accumulator columns [g XC, g XC + XC) of each A operand -> xbuf[a][token][row]
        // (both 32-column loads of an operand in flight before the wait)
        static_assert(WR_XC == 64, "two 32-column loads a round");
#pragma unroll 1
        for (int a = 0; a < NA; ++a) {
          uint32_t v0[32], v1[32];
          if (have) {
            tc_ld_32x32b_x32(tb + a * TOK + g * WR_XC, v0);
            tc_ld_32x32b_x32(tb + a * TOK + g * WR_XC + 32, v1);
            tc_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v0[i] = v1[i] = 0u;
          }
          float* dst = xbuf + a * WR_XC * WR_BM + row;
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[i * WR_BM] = __uint_as_float(v0[i]);
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[(32 + i) * WR_BM] = __uint_as_float(v1[i]);
        }
        if (g == rounds - 1) {  // the accumulator is free for the tile after next
          tc_fence_before();
          mbar_arrive(&tail->tempty[acc]);
        }
        epi_sync();
        arrive_all(xready_addr);
        const bool ready =
            __all_sync(0xffffffffu, mbar_wait_cluster(&tail->xready, xr & 1, tmo, abort_flag));
        if (!ready) fail();
        if (ready) {
          // this rank's share of the round: tokens [c0, c1), 32 quads each
          const int ntok = min(WR_XC, nv - g * WR_XC);
          const int c0 = rank * ntok / S, c1 = (rank + 1) * ntok / S;
          const int nq = (c1 - c0) * 32;
          for (int eb = et; eb < nq; eb += 128 * QB)
            reduce_batch(wt, t0 + g * WR_XC, c0, eb, nq,
                         EPI == EPI_QKV && g == 0 && eb == et ? &qpre : nullptr);
        }
        // the last round of the last tile needs no release: the cluster barrier
        // before exit keeps every copy alive until all ranks have read it
        if (tile + stride < n_tiles || g + 1 < rounds) {
          epi_sync();
          arrive_all(xdone_addr);
          ++xr;
        }
      }
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM);
  }
  cluster_sync_all();  // no CTA leaves while a peer may still address it
}

template <int EPI, int TOK, bool ONE>
cudaError_t wr_prepare() {
  return set_smem_limit(reinterpret_cast<const void*>(gemm_wrows_kernel<EPI, TOK, ONE>),
                        WrCfg<EPI, TOK, ONE>::SMEM);
}

template <int EPI, int TOK, bool ONE>
void wr_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* at, int clusters, int S,
               cudaStream_t stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(static_cast<unsigned>(clusters * S), 1, 1);
  cfg->blockDim = dim3(WR_THREADS, 1, 1);
  cfg->dynamicSmemBytes = WrCfg<EPI, TOK, ONE>::SMEM;
  cfg->stream = stream;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(S);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg->attrs = at;
  cfg->numAttrs = 1;
}

template <int EPI, int TOK, bool ONE>
cudaError_t wr_launch(const CUtensorMap& tmW, const CUtensorMap& tmW2, const CUtensorMap& tmX,
                      const GemmArgs& args, int clusters, bool programmatic,
                      cudaStream_t stream) {
  cudaError_t e = wr_prepare<EPI, TOK, ONE>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute at[2];
  wr_config<EPI, TOK, ONE>(&cfg, at, clusters, args.splits, stream);
  if (programmatic) {
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, gemm_wrows_kernel<EPI, TOK, ONE>, tmW, tmW2, tmX, args);
}

// Both variants take one SM per CTA, so one query serves them.
template <int EPI, int TOK>
int wr_max_clusters(int S) {
  static std::atomic<int> cache[WR_MAX_CLUSTER + 1];  // 0: not asked yet
  if (cache[S].load(std::memory_order_relaxed) == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute at[1];
    wr_config<EPI, TOK, false>(&cfg, at, 1, S, nullptr);
    if (wr_prepare<EPI, TOK, false>() != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, gemm_wrows_kernel<EPI, TOK, false>, &cfg) !=
            cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[S].store(n > 0 ? n : -1, std::memory_order_relaxed);
  }
  const int c = cache[S].load(std::memory_order_relaxed);
  return c > 0 ? c : 0;
}

template <int EPI, int TOK>
cudaError_t wr_launch_any(const CUtensorMap& tmW, const CUtensorMap& tmW2, const CUtensorMap& tmX,
                          const GemmArgs& args, int clusters, bool programmatic,
                          cudaStream_t stream) {
  if (clusters >= args.n_tiles * args.m_tiles)  // at most one tile per CTA
    return wr_launch<EPI, TOK, true>(tmW, tmW2, tmX, args, clusters, programmatic, stream);
  return wr_launch<EPI, TOK, false>(tmW, tmW2, tmX, args, clusters, programmatic, stream);
}

}  // namespace

int gemm_wrows_max_clusters(int epi, int tok, int cluster) {
  if (cluster < 1 || cluster > WR_MAX_CLUSTER) return 0;
  const bool t64 = tok == 64;
  if (!t64 && tok != 128) return 0;
  switch (epi) {
    case EPI_STORE: return t64 ? wr_max_clusters<EPI_STORE, 64>(cluster)
                               : wr_max_clusters<EPI_STORE, 128>(cluster);
    case EPI_RESID: return t64 ? wr_max_clusters<EPI_RESID, 64>(cluster)
                               : wr_max_clusters<EPI_RESID, 128>(cluster);
    case EPI_SWIGLU: return t64 ? wr_max_clusters<EPI_SWIGLU, 64>(cluster)
                                : wr_max_clusters<EPI_SWIGLU, 128>(cluster);
    case EPI_QKV: return t64 ? wr_max_clusters<EPI_QKV, 64>(cluster)
                             : wr_max_clusters<EPI_QKV, 128>(cluster);
    default: return 0;
  }
}

cudaError_t launch_gemm_wrows(int epi, int tok, const CUtensorMap& tmW, const CUtensorMap& tmW2,
                              const CUtensorMap& tmX, const GemmArgs& args, int clusters,
                              bool programmatic, cudaStream_t stream) {
  if (clusters <= 0) return cudaSuccess;
  if (args.splits < 1 || args.splits > WR_MAX_CLUSTER || args.m_tiles < 1 || args.n_tiles < 1 ||
      args.N % 4 || (args.K + WR_BK - 1) / WR_BK < args.splits)
    return cudaErrorInvalidValue;
  if (epi == EPI_QKV && (args.head_dim < 16 || (2 * WR_BM) % args.head_dim ||
                         (args.head_dim / 2) % 8 || args.head_dim > 2 * WR_BM))
    return cudaErrorInvalidValue;
  const bool t64 = tok == 64;
  if (!t64 && tok != 128) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_STORE:
      return t64 ? wr_launch_any<EPI_STORE, 64>(tmW, tmW2, tmX, args, clusters, programmatic, stream)
                 : wr_launch_any<EPI_STORE, 128>(tmW, tmW2, tmX, args, clusters, programmatic, stream);
    case EPI_RESID:
      return t64 ? wr_launch_any<EPI_RESID, 64>(tmW, tmW2, tmX, args, clusters, programmatic, stream)
                 : wr_launch_any<EPI_RESID, 128>(tmW, tmW2, tmX, args, clusters, programmatic, stream);
    case EPI_SWIGLU:
      return t64 ? wr_launch_any<EPI_SWIGLU, 64>(tmW, tmW2, tmX, args, clusters, programmatic, stream)
                 : wr_launch_any<EPI_SWIGLU, 128>(tmW, tmW2, tmX, args, clusters, programmatic,
                                                  stream);
    case EPI_QKV:
      return t64 ? wr_launch_any<EPI_QKV, 64>(tmW, tmW2, tmX, args, clusters, programmatic, stream)
                 : wr_launch_any<EPI_QKV, 128>(tmW, tmW2, tmX, args, clusters, programmatic, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nf
