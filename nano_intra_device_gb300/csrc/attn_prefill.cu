// Causal attention of the rows of prefill chunks on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// A prefill chunk's rows attend to their sequence's earlier positions and to
// the chunk up to themselves ("NanoFlow: Towards Optimal LLM Serving
// Throughput", "The Intra-Device Parallelism Mechanism": prefill attention, the
// compute-bound kind; "CSE 451 Lecture 25", causal self-attention).  A CTA
// takes a tile of consecutive rows of one chunk and one KV head and reads each
// page of the sequence once for the whole tile:
//  * the tile is 128 query vectors: 128 / GRP rows x the GQA group's GRP query
//    heads (vector v is row v / GRP of the tile, query head v % GRP of the
//    group), one per tensor-memory lane;
//  * two producer warps stream key blocks of 128 positions (8 pages) of K and
//    of V of the KV head by TMA (one box per page: at d = 128 a 4-D box that
//    lands as [8-position group][64-column half][8 positions], 1024-byte atoms
//    of the 128-byte swizzle), into a three-stage K ring and a two-stage V ring; warp 1 issues the MMAs from one thread; eight softmax warps own
//    half a vector (lane) each: 64 positions of every block and d / 2 columns
//    of O; they write Q into shared memory, run the online softmax and the
//    epilogue;
//  * per block j: S_j = Q K_j^T (M 128, N 128, K d) into one of two S
//    accumulators in tensor memory; the softmax threads read their row of S
//    (both halves, for the row maximum), mask keys past the row's position,
//    and write their half of P_j = 2^(S scale - m) as bf16 into shared memory
//    (the denominators sum the fp32 values); then O += P_j V_j (M 128, N d,
//    K 128) with V read MN-major straight from the TMA boxes.  The reference
//    maximum m of a row is raised only when a score passes it by more than
//    2^8, and then the row of O in tensor memory is rescaled before the next
//    PV product;
//  * S_{j+1} runs on the tensor cores while the softmax of block j runs;
//  * every wait is bounded; on expiry the kernel flags ST_TIMEOUT, every role
//    leaves its loop, the MMA thread drains the products it issued and the
//    producers the copies they issued before tensor memory is freed.
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace nf {
namespace {

constexpr int TP_SM_WARPS = 8;      // softmax warps: two per tensor-memory lane quarter
constexpr int TP_V_WARP = 2 + TP_SM_WARPS;           // the V producer
constexpr int TP_THREADS = (3 + TP_SM_WARPS) * 32;  // + warp 0 K producer, warp 1 MMA
constexpr int TP_SM_THREADS = TP_SM_WARPS * 32;
constexpr int TP_M = 128;           // query vectors of a tile (tensor-memory lanes)
constexpr int TP_N = 128;           // positions of a key block
constexpr int TP_H = TP_N / 2;      // positions of a block one softmax thread owns
constexpr int TP_PAGES = TP_N / AMMA_P;
constexpr int TP_REGION = 128 * 128;  // 128 rows x 128 bytes: 64 bf16 columns of 128 rows
constexpr float TP_SLACK = 8.f;     // a row's reference maximum may trail its scores by 2^8
constexpr uint32_t TP_TMEM_COLS = 512;
constexpr int TP_KST = 3;           // K ring stages (the MMAs wait on K first)
constexpr int TP_VST = 2;           // V ring stages

struct TpBars {
  uint64_t q_full;                  // TP_SM_THREADS arrivals: Q written
  uint64_t k_full[TP_KST], k_empty[TP_KST];  // K ring
  uint64_t v_full[TP_VST], v_empty[TP_VST];  // V ring
  uint64_t s_full[2], s_free[2];    // S accumulators (s_free: TP_SM_THREADS arrivals)
  uint64_t p_full;                  // TP_SM_THREADS arrivals: P written (and O rescaled)
  uint64_t p_free;                  // a PV product finished (P and O free)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  uint64_t pair[4];                 // 64 arrivals: the two warps of a lane quarter
  float xch[2][TP_M];               // the two halves of a row exchange their sums
};

template <int NCH>
struct TpLayout {
  static constexpr int D = NCH * 64;
  static constexpr int Q_BYTES = NCH * TP_REGION;   // [d/64][128 vectors][128 B]
  // per stage: 16 groups of 8 positions, each [d/64][8 positions][128 B]
  static constexpr int KV_BYTES = NCH * TP_REGION;
  static constexpr int KV_GROUP = NCH * 1024;      // bytes between 8-position groups
  static constexpr int P_BYTES = 2 * TP_REGION;     // [keys/64][128 vectors][128 B]
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;
  static constexpr int V_OFF = K_OFF + TP_KST * KV_BYTES;
  static constexpr int P_OFF = V_OFF + TP_VST * KV_BYTES;
  static constexpr int BAR_OFF = P_OFF + P_BYTES;
  static constexpr int SMEM = 1024 + BAR_OFF + static_cast<int>(sizeof(TpBars));
};

// Byte offset of 16-byte chunk c (elements 8c .. 8c + 7 of a 64-column
// region) of row r, in the 128-byte swizzle the TMA boxes and the MMA
// descriptors use (regions are 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

template <int GRP, int NCH>
__global__ void __launch_bounds__(TP_THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnArgs a,
                        const int4* __restrict__ tiles) {
  using Lay = TpLayout<NCH>;
  constexpr int D = Lay::D;
  static_assert(TP_M % GRP == 0, "a tile holds whole rows of the GQA group");
  constexpr uint32_t IDESC_S = idesc_bf16_f32(TP_M, TP_N);
  constexpr uint32_t IDESC_PV = idesc_bf16_f32_bmn(TP_M, D);
  pdl_trigger();  // the decode kernel of the same nano-batch may start on the free SMs
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  TpBars* bars = reinterpret_cast<TpBars*>(smem + Lay::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kv = a.n_kv;
  const int g = blockIdx.x % n_kv;
  // tiles of a chunk are listed by increasing position, so a later tile reads
  // more blocks: the grid takes them from the end, longest first
  const int4 tl = tiles[gridDim.x / n_kv - 1 - blockIdx.x / n_kv];
  const int t0 = tl.x, t1 = tl.y, sq = tl.z;  // rows [t0, t1) of sequence sq
  const int last_pos = a.tok_pos[t1 - 1];
  const int npages = last_pos / AMMA_P + 1;
  const int nb = (last_pos + TP_N) / TP_N;    // key blocks
  const uint64_t tmo = a.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, TP_SM_THREADS);
    for (int i = 0; i < TP_KST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < TP_VST; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], TP_SM_THREADS);
    }
    mbar_init(&bars->p_full, TP_SM_THREADS);
    mbar_init(&bars->p_free, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bars->pair[i], 64);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, TP_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;  // columns [0, 256): S x 2; [256, 256 + d): O
  volatile int* abort_flag = &bars->abort;
  auto give_up = [&]() {
    raise_status(a.status, ST_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 || warp == TP_V_WARP) {
    // --------------------------------------------- producers: K (warp 0), V
    // Each ring has its own warp, so a K block is fetched as soon as its stage
    // is free, whatever the V ring waits for.
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
    uint8_t* ring = smem + (is_k ? Lay::K_OFF : Lay::V_OFF);
    const int nst = is_k ? TP_KST : TP_VST;
    const int* bt = a.block_table + static_cast<size_t>(sq) * a.max_pages;
    int out[TP_KST];  // block whose copy a stage awaits
#pragma unroll
    for (int i = 0; i < TP_KST; ++i) out[i] = -1;
    for (int j = 0; j < nb; ++j) {
      // pages 8 j .. 8 j + 7; past the sequence's last page, its last page again
      // (those positions are masked, and their V rows zeroed before use)
      int page = 0;
      if (lane < TP_PAGES) {
        const int pi = min(j * TP_PAGES + lane, npages - 1);
        page = bt[pi];
        if (page < 0 || page >= a.num_pages) {  // never read outside the pool
          raise_status(a.status, ST_BAD_PAGE);
          page = 0;
        }
      }
      int rows[TP_PAGES];
#pragma unroll
      for (int p = 0; p < TP_PAGES; ++p)
        rows[p] = (__shfl_sync(0xffffffffu, page, p) * n_kv + g) * AMMA_P;
      const int s = j % nst;
      int good = 1;
      if (lane == 0) {
        good = mbar_wait(&empty[s], ((j / nst) & 1) ^ 1, tmo, abort_flag);
        if (good) {
          uint8_t* dst = ring + s * Lay::KV_BYTES;
          mbar_arrive_expect_tx(&full[s], Lay::KV_BYTES);
          // one box per (page, KV head): [group][half][8 positions][64 columns]
#pragma unroll
          for (int p = 0; p < TP_PAGES; ++p) {
            if (NCH == 2)
              tma_load_4d(dst + p * 2 * Lay::KV_GROUP, map, &full[s], 0, 0, 0, rows[p] / 8);
            else
              tma_load_2d(dst + p * 2 * Lay::KV_GROUP, map, &full[s], 0, rows[p]);
          }
          out[s] = j;
        }
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        if (lane == 0 && !*abort_flag) give_up();
        break;
      }
    }
    if (lane == 0) {
      // the copies still in flight land before the CTA may exit
      for (int s = 0; s < nst; ++s)
        if (out[s] >= 0) mbar_wait(&full[s], (out[s] / nst) & 1, tmo);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(&bars->q_full, 0, tmo, abort_flag);
      bool any = false;
      const uint32_t q_addr = sbase + Lay::Q_OFF;
      const uint32_t o_tmem = tmem + 256;
      const uint32_t p_addr = sbase + Lay::P_OFF;
      auto pv = [&](int i) -> bool {
        const int s = i % TP_VST;
        if (!mbar_wait(&bars->v_full[s], (i / TP_VST) & 1, tmo, abort_flag)) return false;
        if (!mbar_wait(&bars->p_full, i & 1, tmo, abort_flag)) return false;
        tc_fence_after();
        const uint32_t v_addr = sbase + Lay::V_OFF + s * Lay::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < TP_N / 16; ++kk) {
          // A = P: K-major, keys 16 kk .. in region kk / 4; B = V: MN-major,
          // positions 16 kk .. = two 8-position groups; the 64-column halves of a
          // group 1024 bytes apart
          const uint64_t bdesc =
              desc_sw128_mnmajor(v_addr + kk * 2 * Lay::KV_GROUP, 1024, Lay::KV_GROUP);
          const uint64_t adesc = desc_sw128_kmajor(p_addr + (kk >> 2) * TP_REGION) + 2 * (kk & 3);
          tc_mma_bf16(o_tmem, adesc, bdesc, IDESC_PV, (i > 0) || (kk > 0));
        }
        any = true;
        tc_commit(&bars->p_free);
        tc_commit(&bars->v_empty[s]);
        return true;
      };
      for (int j = 0; j < nb && ok; ++j) {
        const int s = j & 1, ks = j % TP_KST;
        ok = mbar_wait(&bars->k_full[ks], (j / TP_KST) & 1, tmo, abort_flag) &&
             mbar_wait(&bars->s_free[s], ((j >> 1) & 1) ^ 1, tmo, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t k_addr = sbase + Lay::K_OFF + ks * Lay::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t adesc = desc_sw128_kmajor(q_addr + (kk >> 2) * TP_REGION) + 2 * (kk & 3);
          const uint64_t bdesc =
              desc_sw128_kmajor_sbo(k_addr + (kk >> 2) * 1024, Lay::KV_GROUP) + 2 * (kk & 3);
          tc_mma_bf16(tmem + s * TP_N, adesc, bdesc, IDESC_S, kk > 0);
        }
        any = true;
        tc_commit(&bars->s_full[s]);
        tc_commit(&bars->k_empty[ks]);
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok) ok = pv(nb - 1);
      if (!ok) {
        if (!*abort_flag) give_up();
        if (any) {  // the products already issued finish before tensor memory goes away
          tc_commit(&bars->drain);
          mbar_wait(&bars->drain, 0, tmo);
        }
      }
    }
  } else {
    // ------------------------------------------- softmax and epilogue
    const int quarter = warp & 3;           // tensor-memory lanes this warp may access
    const int half = (warp - 2) >> 2;       // which 64 keys of a block (and d/2 of O) it owns
    const int r = quarter * 32 + lane;      // the vector (lane) this thread owns
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int row = t0 + r / GRP;
    const bool live = row < t1;
    const int qt = live ? row : t1 - 1;
    const int qh = g * GRP + r % GRP;
    const int qpos = a.tok_pos[qt];
    // Q into shared memory, K-major in the 128-byte swizzle (each half of the
    // row writes half of its chunks)
    {
      const uint4* q4 = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(qt) * a.n_q + qh) * D);
#pragma unroll
      for (int c = half * (D / 16); c < (half + 1) * (D / 16); ++c)
        st_shared_v4(sbase + Lay::Q_OFF + (c >> 3) * TP_REGION + sw128(r, c & 7), q4[c]);
      fence_proxy_async_smem();
      mbar_arrive(&bars->q_full);
    }
    const float scale = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // PV product n (of block n) finished: completion n of p_free.  Every wait
    // of a thread targets the completion after the one it waited for last, or
    // the same, so the parity is never two phases stale.
    auto pv_done = [&](int n) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(&bars->p_free, n & 1, tmo, abort_flag));
    };
    for (int j = 0; j < nb; ++j) {
      const int s = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[s], (j >> 1) & 1, tmo, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this half's 64 scores, and the other half's for the row maximum
      float x[TP_H];
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
      {
        uint32_t u[TP_H], w[TP_H];
#pragma unroll
        for (int c = 0; c < TP_H / 32; ++c) {
          tc_ld_32x32b_x32(tmem + lane_off + s * TP_N + half * TP_H + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
          tc_ld_32x32b_x32(tmem + lane_off + s * TP_N + (half ^ 1) * TP_H + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&w[c * 32]));
        }
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_free[s]);
        // maxima of the raw scores in 8 independent chains; positions past the
        // row's own are masked (only in the blocks that reach past it)
        if (j * TP_N + TP_N - 1 <= qpos) {
#pragma unroll
          for (int i = 0; i < TP_H; ++i) {
            x[i] = __uint_as_float(u[i]);
            mx8[i & 7] = fmax3(mx8[i & 7], x[i], __uint_as_float(w[i]));
          }
        } else {
          const int kb_own = j * TP_N + half * TP_H, kb_oth = j * TP_N + (half ^ 1) * TP_H;
#pragma unroll
          for (int i = 0; i < TP_H; ++i) {
            x[i] = kb_own + i <= qpos ? __uint_as_float(u[i]) : -INFINITY;
            const float y = kb_oth + i <= qpos ? __uint_as_float(w[i]) : -INFINITY;
            mx8[i & 7] = fmax3(mx8[i & 7], x[i], y);
          }
        }
      }
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7])) * scale;
      float corr = 1.f;
      if (m_ref == -INFINITY) {
        m_ref = mx;  // block 0: position 0 is visible to every row
      } else if (mx > m_ref + TP_SLACK) {
        corr = ex2_approx(m_ref - mx);
        m_ref = mx;
        l *= corr;
      }
      // p = 2^(s scale - m): the affine step two lanes at a time, the sums in 4
      // independent pairs of chains
      {
        const float2 sc2 = make_float2(scale, scale), nm2 = make_float2(-m_ref, -m_ref);
        float2 ls4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ls4[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < TP_H / 2; ++i) {
          const float2 t = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), sc2, nm2);
          x[2 * i] = ex2_approx(t.x);
          x[2 * i + 1] = ex2_approx(t.y);
          ls4[i & 3] = __fadd2_rn(ls4[i & 3], make_float2(x[2 * i], x[2 * i + 1]));
        }
        const float2 a2 = __fadd2_rn(__fadd2_rn(ls4[0], ls4[1]), __fadd2_rn(ls4[2], ls4[3]));
        l += a2.x + a2.y;
      }
      // a raised maximum rescales this half of the row of O, once the PV
      // product of the previous block is done with it
      if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
        if (!pv_done(j - 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t u[32];
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t ta = tmem + lane_off + 256 + half * (D / 2) + c * 32;
          tc_ld_32x32b_x32(ta, u);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * corr);
          tc_st_32x32b_x32(ta, u);
        }
        tc_wait_st();
      }
      // P (free once the previous PV product is done), K-major in the 128-byte
      // swizzle: this half's 64 keys fill one region
      if (j >= 1 && !pv_done(j - 1)) {
        ok = false;
        break;
      }
      const uint32_t p_reg = sbase + Lay::P_OFF + half * TP_REGION;
#pragma unroll
      for (int c = 0; c < TP_H / 8; ++c) {
        uint4 w;
        w.x = pack_bf16(x[8 * c + 0], x[8 * c + 1]);
        w.y = pack_bf16(x[8 * c + 2], x[8 * c + 3]);
        w.z = pack_bf16(x[8 * c + 4], x[8 * c + 5]);
        w.w = pack_bf16(x[8 * c + 6], x[8 * c + 7]);
        st_shared_v4(p_reg + sw128(r, c), w);
      }
      if (j == nb - 1 && j * TP_N + TP_N - 1 > last_pos) {
        // V rows past the tile's last position may lie past the sequence and
        // hold anything (even NaN): P is 0 there, and 0 x NaN must not reach O
        const int vs = j % TP_VST;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars->v_full[vs], (j / TP_VST) & 1, tmo, abort_flag))) {
          ok = false;
          break;
        }
        if (half < NCH && j * TP_N + r > last_pos) {
          const uint32_t vrow = sbase + Lay::V_OFF + vs * Lay::KV_BYTES + (r >> 3) * Lay::KV_GROUP +
                                half * 1024 + (r & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_v4(vrow + c * 16, make_uint4(0, 0, 0, 0));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    if (ok && !pv_done(nb - 1)) ok = false;
    if (!ok) {
      if (!*abort_flag) give_up();
    } else {
      tc_fence_after();
      // the row's denominator: the two halves' sums, met at a bounded barrier
      bars->xch[half][r] = l;
      mbar_arrive(&bars->pair[quarter]);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->pair[quarter], 0, tmo, abort_flag))) ok = false;
    }
    if (!ok) {
      if (!*abort_flag) give_up();
    } else {
      const float inv = 1.f / (bars->xch[0][r] + bars->xch[1][r]);
      uint4* dst = reinterpret_cast<uint4*>(a.o + (static_cast<size_t>(qt) * a.n_q + qh) * D +
                                            half * (D / 2));
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t u[32];
        tc_ld_32x32b_x32(tmem + lane_off + 256 + half * (D / 2) + c * 32, u);
        tc_wait_ld();
        if (live) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(u[8 * i + 0]) * inv, __uint_as_float(u[8 * i + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(u[8 * i + 2]) * inv, __uint_as_float(u[8 * i + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(u[8 * i + 4]) * inv, __uint_as_float(u[8 * i + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(u[8 * i + 6]) * inv, __uint_as_float(u[8 * i + 7]) * inv);
            dst[c * 4 + i] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TP_TMEM_COLS);
  }
}

template <int GRP, int NCH>
cudaError_t launch_pf_t(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        const int4* tiles, int n_tiles, cudaStream_t stream) {
  const int smem = TpLayout<NCH>::SMEM;
  const void* fn = reinterpret_cast<const void*>(attn_prefill_kernel<GRP, NCH>);
  const cudaError_t attr = set_smem_limit(fn, smem);
  if (attr != cudaSuccess) return attr;
  attn_prefill_kernel<GRP, NCH><<<n_tiles * a.n_kv, TP_THREADS, smem, stream>>>(tk, tv, a, tiles);
  return cudaGetLastError();
}

}  // namespace

int prefill_tile_rows(int n_q, int n_kv) { return TP_M / (n_q / n_kv); }

cudaError_t launch_attention_prefill(const AttnArgs& a, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const int4* tiles, int n_tiles,
                                     cudaStream_t stream) {
  if (n_tiles <= 0) return cudaSuccess;
  if (!attention_mma_supported(a.n_q, a.n_kv, a.head_dim, a.page_size, a.num_pages))
    return cudaErrorInvalidValue;
  const int grp = a.n_q / a.n_kv, nch = a.head_dim / 64;
#define NF_PF_CASE(G, N) \
  if (grp == G && nch == N) return launch_pf_t<G, N>(a, tk, tv, tiles, n_tiles, stream);
  NF_PF_CASE(1, 1) NF_PF_CASE(2, 1) NF_PF_CASE(4, 1) NF_PF_CASE(8, 1)
  NF_PF_CASE(1, 2) NF_PF_CASE(2, 2) NF_PF_CASE(4, 2) NF_PF_CASE(8, 2)
#undef NF_PF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace nf
