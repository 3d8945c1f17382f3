// Causal attention of the rows of prefill chunks, flash style on the tensor
// cores.
//
// A prefill chunk's rows attend to their sequence's earlier positions and to
// the chunk up to themselves ("NanoFlow: Towards Optimal LLM Serving
// Throughput", "The Intra-Device Parallelism Mechanism": prefill attention, the
// compute-bound kind; "CSE 451 Lecture 25", causal self-attention).  Through
// the decode kernel every row would read its sequence's K/V once; here a CTA
// takes a tile of consecutive rows of one chunk and one KV head and reads each
// page once for the whole tile:
//  * the tile is QP = 128 / GRP rows x the GQA group's GRP query heads = 128
//    query vectors, 16 per compute warp (8 warps): vector v is row v / GRP of
//    the tile, query head v % GRP of the group;
//  * a producer warp streams pages 0 .. (position of the tile's last row) / 16
//    of the sequence (K and V of the KV head) by 2-D TMA into a ring that the
//    compute warps share; a page is released when all 8 have used it;
//  * per page and warp: S[16 x 16] = Q K^T (Q the A operand, from registers;
//    K by ldmatrix), the causal mask by position, an online softmax per row in
//    base 2, P moved to the A-operand layout straight from the accumulators,
//    and O[16 x d] += P V (V by ldmatrix.trans).  P enters PV as two bf16
//    operands (hi = bf16(p), lo = bf16(p - hi)) and the denominators sum the
//    fp32 values, as in the decode kernel;
//  * every wait is bounded; on expiry the kernel flags ST_TIMEOUT and the
//    producer waits (bounded) for the copies it issued before the CTA exits.
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace nf {
namespace {

constexpr int PF_WARPS = 8;                  // compute warps
constexpr int PF_THREADS = (PF_WARPS + 1) * 32;
constexpr int PF_STAGES = 8;                 // pages in the ring
constexpr int PF_VECS = 16 * PF_WARPS;       // query vectors of a tile

int pf_smem_bytes(int head_dim) {
  const int slot = 2 * AMMA_P * head_dim * 2;
  return 1024 + PF_STAGES * slot + 2 * PF_STAGES * 8;
}

template <int GRP, int NCH>
__global__ void __launch_bounds__(PF_THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnArgs a,
                        const int4* __restrict__ tiles) {
  constexpr int D = NCH * 64;
  constexpr int KS = D / 16;           // k-steps of S, pairs of n8 tiles of O
  static_assert(PF_VECS % GRP == 0, "a tile holds whole rows of the GQA group");
  pdl_trigger();  // the decode kernel of the same nano-batch may start on the free SMs
  constexpr int BOX = AMMA_P * 128;    // one 64-column box of a page: 2 KB
  constexpr int BLK = NCH * BOX;       // K (or V) of one (page, KV head)
  constexpr int SLOT = 2 * BLK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PF_STAGES * SLOT);
  uint64_t* empty = full + PF_STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kv = a.n_kv;
  const int g = blockIdx.x % n_kv;
  // tiles of a chunk are listed by increasing position, so a later tile reads
  // more pages: the grid takes them from the end, longest first
  const int4 tl = tiles[gridDim.x / n_kv - 1 - blockIdx.x / n_kv];
  const int t0 = tl.x, t1 = tl.y, sq = tl.z;  // rows [t0, t1) of sequence sq
  const int last_pos = a.tok_pos[t1 - 1];
  const int npages = last_pos / AMMA_P + 1;
  const uint64_t tmo = a.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < PF_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], PF_WARPS);
    }
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();

  if (warp == PF_WARPS) {
    // ---------------------------------------------------------- producer
    const int* bt = a.block_table + static_cast<size_t>(sq) * a.max_pages;
    bool ok = true;
    int issued = 0;
    for (int k0 = 0; k0 < npages && ok; k0 += 32) {
      int page = 0;  // page id of page k0 + lane
      if (k0 + lane < npages) {
        page = bt[k0 + lane];
        if (page < 0 || page >= a.num_pages) {  // never read outside the pool
          raise_status(a.status, ST_BAD_PAGE);
          page = 0;
        }
      }
      const int cnt = min(32, npages - k0);
      for (int j = 0; j < cnt; ++j) {
        const int pg = __shfl_sync(0xffffffffu, page, j);
        const int k = k0 + j;
        const int st = k % PF_STAGES;
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(&empty[st], ((k / PF_STAGES) & 1) ^ 1, tmo);
          if (good) {
            fence_proxy_async_smem();  // the compute warps' reads of the slot come first
            uint8_t* sl = smem + st * SLOT;
            const int y = (pg * n_kv + g) * AMMA_P;  // first pool row of the (page, KV head)
            mbar_arrive_expect_tx(&full[st], SLOT);
#pragma unroll
            for (int b = 0; b < NCH; ++b) tma_load_2d(sl + b * BOX, &tmK, &full[st], b * 64, y);
#pragma unroll
            for (int b = 0; b < NCH; ++b)
              tma_load_2d(sl + BLK + b * BOX, &tmV, &full[st], b * 64, y);
          }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        ++issued;
      }
    }
    if (lane == 0) {
      if (!ok) raise_status(a.status, ST_TIMEOUT);
      // the copies still in flight land before the CTA may exit
      for (int k = issued - PF_STAGES > 0 ? issued - PF_STAGES : 0; k < issued; ++k)
        mbar_wait(&full[k % PF_STAGES], (k / PF_STAGES) & 1, tmo);
    }
    return;
  }

  // -------------------------------------------------------------- compute
  const int lr = lane >> 2, lc = lane & 3;  // fragment row / column pair of this lane
  // this lane's two rows of the warp's m16 tile: query vectors v, v + 8
  const int n_q = a.n_q;
  int qt[2], qh[2], qpos[2];
  bool live[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int v = warp * 16 + lr + 8 * r;
    const int row = t0 + v / GRP;
    live[r] = row < t1;
    qt[r] = live[r] ? row : t1 - 1;
    qh[r] = g * GRP + v % GRP;
    qpos[r] = a.tok_pos[qt[r]];
  }
  // Q as the A operand: k-step kk holds dims 16 kk + 2 lc (+1) and + 8
  uint32_t qa[KS][4];
  {
    const __nv_bfloat16* q0 = a.q + (static_cast<size_t>(qt[0]) * n_q + qh[0]) * D;
    const __nv_bfloat16* q1 = a.q + (static_cast<size_t>(qt[1]) * n_q + qh[1]) * D;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qa[kk][0] = *reinterpret_cast<const uint32_t*>(q0 + 16 * kk + 2 * lc);
      qa[kk][1] = *reinterpret_cast<const uint32_t*>(q1 + 16 * kk + 2 * lc);
      qa[kk][2] = *reinterpret_cast<const uint32_t*>(q0 + 16 * kk + 8 + 2 * lc);
      qa[kk][3] = *reinterpret_cast<const uint32_t*>(q1 + 16 * kk + 8 + 2 * lc);
    }
  }
  // ldmatrix row addresses, fixed per lane (lane 8 j + r supplies row r of matrix j):
  // K (for S = Q K^T): matrix j = positions 8 (j >> 1) .., dims 16 kk + 8 (j & 1) ..
  // V (for O += P V, transposed): matrix j = positions 8 (j & 1) .., dims 16 nn + 8 (j >> 1) ..
  const int mj = lane >> 3, mr = lane & 7;
  // On the last page, positions past the tile's last row may lie past the
  // sequence's end and hold anything (even NaN): P is 0 there, and their V rows
  // read position 0 of the page instead, so 0 x NaN never reaches O.
  const int vpos = mr + 8 * (mj & 1);
  const bool v_past = (npages - 1) * AMMA_P + vpos > last_pos;
  uint32_t koff[KS], voff[KS];
#pragma unroll
  for (int i = 0; i < KS; ++i) {
    koff[i] = page_chunk_off(mr + 8 * (mj >> 1), 2 * i + (mj & 1));
    voff[i] = BLK + page_chunk_off(vpos, 2 * i + (mj >> 1));
  }
  const float scale = a.scale_log2;
  float o[2 * KS][4];  // n8 tile j of O: (row lr, dims 8 j + 2 lc, +1), (row lr + 8, ..)
#pragma unroll
  for (int j = 0; j < 2 * KS; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const uint32_t ring_u32 = smem_u32(smem);
  bool failed = false;
  for (int k = 0; k < npages; ++k) {
    const int st = k % PF_STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (k / PF_STAGES) & 1, tmo))) {
      failed = true;
      break;
    }
    const uint32_t slot = ring_u32 + st * SLOT;
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t kb[4];
      ldsm_x4(slot + koff[kk], kb);
      mma_16816(sc[0], qa[kk], kb[0], kb[1]);
      mma_16816(sc[1], qa[kk], kb[2], kb[3]);
    }
    // scores in base 2, keys past the row's position masked
    float x[2][4];
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        const int kp = k * AMMA_P + 8 * j + 2 * lc + (e & 1);
        x[j][e] = kp <= qpos[r] ? sc[j][e] * scale : -INFINITY;
        mx[r] = fmaxf(mx[r], x[j][e]);
      }
    float c[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float nm = fmaxf(m[r], mx[r]);  // finite from the first page on (key 0 is visible)
      c[r] = ex2_approx(m[r] - nm);
      m[r] = nm;
      l[r] *= c[r];
    }
#pragma unroll
    for (int j = 0; j < 2 * KS; ++j) {
      o[j][0] *= c[0];
      o[j][1] *= c[0];
      o[j][2] *= c[1];
      o[j][3] *= c[1];
    }
    // P as the A operand of a k16 step: (row lr, keys 2 lc ..), (lr + 8, ..), then
    // keys + 8; as two bf16 operands, hi = bf16(p) and lo = bf16(p - hi), so that
    // each weight keeps 16 significant bits; the denominators sum the fp32 values
    uint32_t pa[4], pr[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float e0 = ex2_approx(x[j][0] - m[0]), e1 = ex2_approx(x[j][1] - m[0]);
      const float e2 = ex2_approx(x[j][2] - m[1]), e3 = ex2_approx(x[j][3] - m[1]);
      const uint32_t p0 = pack_bf16(e0, e1), p1 = pack_bf16(e2, e3);
      l[0] += e0 + e1;
      l[1] += e2 + e3;
      pa[2 * j] = p0;
      pa[2 * j + 1] = p1;
      pr[2 * j] = pack_bf16(e0 - bf16lo(p0), e1 - bf16hi(p0));
      pr[2 * j + 1] = pack_bf16(e2 - bf16lo(p1), e3 - bf16hi(p1));
    }
    const bool redirect = v_past && k == npages - 1;
#pragma unroll
    for (int nn = 0; nn < KS; ++nn) {
      uint32_t vb[4];
      ldsm_x4_trans(slot + (redirect ? BLK + page_chunk_off(0, 2 * nn + (mj >> 1)) : voff[nn]), vb);
      mma_16816(o[2 * nn], pr, vb[0], vb[1]);
      mma_16816(o[2 * nn + 1], pr, vb[2], vb[3]);
      mma_16816(o[2 * nn], pa, vb[0], vb[1]);
      mma_16816(o[2 * nn + 1], pa, vb[2], vb[3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (failed) {
    raise_status(a.status, ST_TIMEOUT);
    return;
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  const float inv0 = 1.f / l[0], inv1 = 1.f / l[1];
  __nv_bfloat16* o0 = a.o + (static_cast<size_t>(qt[0]) * n_q + qh[0]) * D;
  __nv_bfloat16* o1 = a.o + (static_cast<size_t>(qt[1]) * n_q + qh[1]) * D;
#pragma unroll
  for (int j = 0; j < 2 * KS; ++j) {
    const int d0 = 8 * j + 2 * lc;
    if (live[0]) *reinterpret_cast<uint32_t*>(o0 + d0) = pack_bf16(o[j][0] * inv0, o[j][1] * inv0);
    if (live[1]) *reinterpret_cast<uint32_t*>(o1 + d0) = pack_bf16(o[j][2] * inv1, o[j][3] * inv1);
  }
}

template <int GRP, int NCH>
cudaError_t launch_pf_t(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        const int4* tiles, int n_tiles, cudaStream_t stream) {
  const int smem = pf_smem_bytes(NCH * 64);
  const cudaError_t attr =
      set_smem_limit(reinterpret_cast<const void*>(attn_prefill_kernel<GRP, NCH>), smem);
  if (attr != cudaSuccess) return attr;
  attn_prefill_kernel<GRP, NCH><<<n_tiles * a.n_kv, PF_THREADS, smem, stream>>>(tk, tv, a, tiles);
  return cudaGetLastError();
}

}  // namespace

int prefill_tile_rows(int n_q, int n_kv) { return PF_VECS / (n_q / n_kv); }

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
