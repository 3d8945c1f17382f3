// Tensor-core GEMM for sm_103a: C = A * B^T, bf16 in, fp32 accumulate in TMEM.
//
// The projections and the FFN of the decoder layer are the step's dense
// contractions ("NanoFlow: Towards Optimal LLM Serving Throughput", "The
// Intra-Device Parallelism Mechanism": KQV, O, Up/Gate/Down are the
// compute-bound operations).  Design:
//  * persistent CTAs, one per SM (the shared-memory ring fills the SM), so a
//    grid of S CTAs occupies exactly S SMs: the SM share of a nano-operation;
//  * warp 0: one thread issues TMA tile loads (128-byte swizzle) into a
//    4-stage ring; warp 1: one thread issues tcgen05.mma (M=128, N=256, K=16)
//    into a double-buffered TMEM accumulator; warps 2-5: epilogue, tcgen05.ld
//    of the accumulator rows, fused RoPE + KV append, residual or SwiGLU;
//  * every wait is bounded; on expiry the kernel flags the status word, drains
//    what it has in flight (bounded) and frees TMEM before returning.
#include "common.cuh"
#include "kernels.h"

namespace nf {

constexpr int BM = 128, BK = 64;
constexpr int BN_DEFAULT = 256;     // output columns of a tile (224 for the O / down
                                    // projections when it turns a partial last wave into
                                    // whole ones)
constexpr int MAX_STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int TMEM_COLS = 512;      // two accumulators of up to 256 columns
constexpr int GEMM_THREADS = 192;
// Dynamic shared memory of a CTA with `stages` ring stages of `bn`-column B
// tiles: the ring, slack to align it to 1024 bytes, and the barrier block.  4
// stages fill an SM (one CTA per SM, exclusive); 3 or 2 leave room for an
// attention CTA beside it.
constexpr int gemm_smem_bytes(int stages, int bn) {
  return stages * (A_BYTES + bn * BK * 2) + 1024 + 640;
}

struct GemmSmemTail {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t epi_sync;   // rendezvous of the 4 epilogue warps (split-K)
  uint32_t tmem_base;
  int abort;
  int last;            // this CTA finishes the tile's last split (split-K)
  int gpre[GEMM_MAX_GROUPS + 1];  // grouped GEMM: first tile of each group
};
static_assert(sizeof(GemmSmemTail) <= 640, "barrier block exceeds its reservation");

// One output tile: A rows [m0, m0 + BM) (rows >= m_lim are not stored), B rows
// from brow + tn * (columns per tile), split sp of the K range.
struct GemmTile {
  int t, sp, m0, m_lim, tn, brow;
};

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float* v) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16(v[8 * i + 6], v[8 * i + 7]);
    d4[i] = u;
  }
}

// Store 32 consecutive columns starting at column n of row `row`, keeping
// only columns < ncols (ncols is a multiple of 8).
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16* row, int n, int ncols,
                                                const float* v) {
  if (n + 32 <= ncols) {
    store32_bf16(row + n, v);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(row + n);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (n + 8 * i + 8 <= ncols) {
        uint4 u;
        u.x = pack_bf16(v[8 * i + 0], v[8 * i + 1]);
        u.y = pack_bf16(v[8 * i + 2], v[8 * i + 3]);
        u.z = pack_bf16(v[8 * i + 4], v[8 * i + 5]);
        u.w = pack_bf16(v[8 * i + 6], v[8 * i + 7]);
        d4[i] = u;
      }
    }
  }
}

__device__ __forceinline__ void tmem_load32(uint32_t taddr, float* v) {
  uint32_t r[32];
  tc_ld_32x32b_x32(taddr, r);
  tc_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int EPI, int STAGES, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  static_assert(BN % 32 == 0 && BN <= 256, "tile width");
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  GemmSmemTail* tail = reinterpret_cast<GemmSmemTail*>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work units: (output tile, K split).  The splits of one tile are adjacent
  // unit numbers, so they run on different CTAs at the same time.
  const int splits = args.splits > 1 && args.n_groups == 0 ? args.splits : 1;
  const int nk = (args.K + BK - 1) / BK;
  const uint64_t tmo = args.timeout_ns;

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
    tail->abort = 0;
    if (args.n_groups > 0) {  // tiles per group from the device-side row offsets
      int acc = 0;
      for (int e = 0; e < args.n_groups; ++e) {
        tail->gpre[e] = acc;
        const int rows = args.group_off[e + 1] - args.group_off[e];
        acc += rows > 0 ? ((rows + BM - 1) / BM) * args.n_tiles : 0;
      }
      tail->gpre[args.n_groups] = acc;
    }
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (EPI == EPI_SWIGLU) prefetch_tensormap(&tmB2);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  volatile int* abort_flag = &tail->abort;
  const int total_tiles =
      args.n_groups > 0 ? tail->gpre[args.n_groups] : args.m_tiles * args.n_tiles * splits;
  auto decode = [&](int u) {
    GemmTile x;
    if (args.n_groups > 0) {
      int e = 0;
      while (e + 1 < args.n_groups && tail->gpre[e + 1] <= u) ++e;
      const int local = u - tail->gpre[e];
      const int g0 = args.group_off[e], g1 = args.group_off[e + 1];
      const int mt = (g1 - g0 + BM - 1) / BM;
      x.t = u;
      x.sp = 0;
      x.m0 = g0 + (local % mt) * BM;
      x.m_lim = g1;
      x.tn = local / mt;
      x.brow = e * args.b_group_rows;
    } else {
      x.t = u / splits;
      x.sp = u % splits;
      x.m0 = args.m_begin + (x.t % args.m_tiles) * BM;
      x.m_lim = args.m_end;
      x.tn = x.t / args.m_tiles;
      x.brow = 0;
    }
    return x;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t st = 0, ph = 0;
      uint32_t issued_mask = 0, last_ph[MAX_STAGES] = {0, 0, 0, 0};
      bool ok = true;
      // the B part of a stage: k block kb of output-column tile tn
      auto load_b = [&](uint8_t* sb, uint64_t* bar, int kb, int tn, int brow) {
        if (EPI == EPI_SWIGLU) {
          tma_load_2d(sb, &tmB, bar, kb * BK, brow + tn * (BN / 2));
          tma_load_2d(sb + B_BYTES / 2, &tmB2, bar, kb * BK, brow + args.b2_row_off + tn * (BN / 2));
        } else {
          tma_load_2d(sb, &tmB, bar, kb * BK, brow + tn * BN);
        }
      };
      // Programmatic dependent: the weights of the first tile's first stages
      // (no kernel writes them) are requested before the wait for the kernel
      // that writes A; each such stage's barrier expects its A bytes too.
      int pre = 0;
      if (args.weights_first) {
        if (static_cast<int>(blockIdx.x) < total_tiles) {
          const GemmTile x = decode(blockIdx.x);
          const int kb0 = x.sp * nk / splits, kb1 = (x.sp + 1) * nk / splits;
          pre = kb1 - kb0 < STAGES ? kb1 - kb0 : STAGES;
          for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(&tail->full[i], STAGE_BYTES);
            load_b(smem + i * STAGE_BYTES + A_BYTES, &tail->full[i], kb0 + i, x.tn, x.brow);
          }
        }
        pdl_wait();
      }
      for (int u = blockIdx.x; u < total_tiles && ok; u += gridDim.x) {
        const GemmTile x = decode(u);
        const int sp = x.sp, tn = x.tn, m0 = x.m0;
        const int kb0 = sp * nk / splits, kb1 = (sp + 1) * nk / splits;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&tail->empty[st], ph ^ 1, tmo, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + st * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          // the first tile's first `pre` stages (st = kb - kb0, phase 0) hold
          // their weights already
          const bool have_b = u == static_cast<int>(blockIdx.x) && kb - kb0 < pre;
          if (!have_b) mbar_arrive_expect_tx(&tail->full[st], STAGE_BYTES);
          tma_load_2d(sa, &tmA, &tail->full[st], kb * BK, m0);
          if (!have_b) load_b(sb, &tail->full[st], kb, tn, x.brow);
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
        // drain: every stage we filled must have landed before smem is released
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) mbar_wait(&tail->full[s], last_ph[s], tmo);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t st = 0, ph = 0, acc = 0, aph = 0;
      bool ok = true, any = false;
      for (int u = blockIdx.x; u < total_tiles && ok; u += gridDim.x) {
        const int sp = decode(u).sp;
        const int kb0 = sp * nk / splits, kb1 = (sp + 1) * nk / splits;
        if (!mbar_wait(&tail->tempty[acc], aph ^ 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&tail->full[st], ph, tmo, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + st * STAGE_BYTES);
          const uint64_t adesc = desc_sw128_kmajor(sa);
          const uint64_t bdesc = desc_sw128_kmajor(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // advance 16 bf16 = 32 bytes along K inside the swizzled row
            tc_mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb != kb0) || (k != 0));
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
        if (any) {  // wait for the MMAs already issued before TMEM goes away
          tc_commit(&tail->drain);
          mbar_wait(&tail->drain, 0, tmo);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // Every CTA's epilogue waits here, so the grid ends after the kernel it
    // depends on even where a CTA has no tile.
    if (args.wait_prior || args.weights_first) pdl_wait();
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row_in_tile = quarter * 32 + lane;
    uint32_t acc = 0, aph = 0, esync = 0;
    // rendezvous of the four epilogue warps (bounded)
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->epi_sync);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tail->epi_sync, esync & 1, tmo, abort_flag));
      ++esync;
      return ok;
    };
    for (int u = blockIdx.x; u < total_tiles; u += gridDim.x) {
      const GemmTile x = decode(u);
      const int t = x.t, sp = x.sp;
      // Residual epilogue: the residual's 32 columns of a chunk, loaded one
      // chunk ahead; the first chunk's before the wait for the accumulator, so
      // that its latency hides under the tile's MMAs.
      uint4 r_next[4];
      auto load_r = [&](int c) {
        const int m_ = x.m0 + (warp & 3) * 32 + lane;
        const int n_ = x.tn * BN + c * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          r_next[i] = make_uint4(0u, 0u, 0u, 0u);
          if (m_ < x.m_lim && n_ + 8 * i + 8 <= args.N)
            r_next[i] = __ldg(reinterpret_cast<const uint4*>(args.R + static_cast<size_t>(m_) * args.ldr +
                                                            n_ + 8 * i));
        }
      };
      if (EPI == EPI_RESID) load_r(0);
      // the wait result must be warp-uniform: tcgen05.ld below is .sync.aligned
      const bool got = __all_sync(0xffffffffu, mbar_wait(&tail->tfull[acc], aph, tmo, abort_flag));
      if (!got) {
        raise_status(args.status, ST_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int tn = x.tn;
      const int m = x.m0 + row_in_tile;
      const bool row_ok = m < x.m_lim;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      float v[32];
      // Split-K: publish this split's fp32 tile, and let the CTA that finishes
      // the tile's last split add the others and run the epilogue.
      bool reduce = false;
      float* part_tile = nullptr;
      if (splits > 1) {
        // Partial layout per split: float4 (chunk c of 32 columns, quad i, row),
        // rows fastest, so a warp's 32 rows write 512 contiguous bytes.
        part_tile = args.part + static_cast<size_t>(t) * splits * BM * BN;
        float4* mine = reinterpret_cast<float4*>(part_tile + static_cast<size_t>(sp) * BM * BN) +
                       row_in_tile;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          tmem_load32(tbase + c * 32, v);
          if (row_ok) {  // rows past the range are never read back
#pragma unroll
            for (int i = 0; i < 8; ++i)
              mine[(c * 8 + i) * BM] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
        __threadfence();
        bool ok = epi_sync();
        if (ok && warp == 2 && lane == 0)
          tail->last = atomicAdd(&args.tile_cnt[t], 1) == splits - 1;
        ok = ok && epi_sync();
        if (!ok) {
          raise_status(args.status, ST_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        if (!tail->last) {  // another split finishes this tile
          tc_fence_before();
          mbar_arrive(&tail->tempty[acc]);
          if (++acc == 2) {
            acc = 0;
            aph ^= 1;
          }
          continue;
        }
        __threadfence();
        reduce = true;
        if (warp == 2 && lane == 0) args.tile_cnt[t] = 0;  // ready for the next GEMM
      }
      // 32 accumulator columns starting at column col.  Split-K: the sum of the
      // splits' partials, always in split order, so the result does not depend
      // on which CTA arrived last.
      auto fetch32 = [&](int col, float* out) {
        tmem_load32(tbase + col, out);  // keeps every lane in the .sync.aligned load
        if (reduce && row_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) out[i] = 0.f;
          const float4* src = reinterpret_cast<const float4*>(part_tile) + (col / 32) * 8 * BM +
                              row_in_tile;
          constexpr int kSplit4 = BM * BN / 4;  // float4 per split
          // two splits' loads in flight at a time; the sum stays in split order
          for (int o = 0; o < splits; o += 2) {
            const bool two = o + 1 < splits;
            float4 x[8], y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __ldcg(src + static_cast<size_t>(o) * kSplit4 + i * BM);
            if (two) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                y[i] = __ldcg(src + static_cast<size_t>(o + 1) * kSplit4 + i * BM);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              out[4 * i] += x[i].x;
              out[4 * i + 1] += x[i].y;
              out[4 * i + 2] += x[i].z;
              out[4 * i + 3] += x[i].w;
            }
            if (two) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                out[4 * i] += y[i].x;
                out[4 * i + 1] += y[i].y;
                out[4 * i + 2] += y[i].z;
                out[4 * i + 3] += y[i].w;
              }
            }
          }
        }
      };

      if (EPI == EPI_STORE || EPI == EPI_RESID) {
        __nv_bfloat16* crow = args.C + static_cast<size_t>(m) * args.ldc;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint4 r_cur[4];
          if (EPI == EPI_RESID) {
#pragma unroll
            for (int i = 0; i < 4; ++i) r_cur[i] = r_next[i];
            if (c + 1 < BN / 32) load_r(c + 1);
          }
          fetch32(c * 32, v);
          const int n = tn * BN + c * 32;
          if (row_ok && n < args.N) {
            if (EPI == EPI_RESID) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (n + 8 * i + 8 <= args.N) {
                  const uint4 u = r_cur[i];
                  v[8 * i + 0] += bf16lo(u.x); v[8 * i + 1] += bf16hi(u.x);
                  v[8 * i + 2] += bf16lo(u.y); v[8 * i + 3] += bf16hi(u.y);
                  v[8 * i + 4] += bf16lo(u.z); v[8 * i + 5] += bf16hi(u.z);
                  v[8 * i + 6] += bf16lo(u.w); v[8 * i + 7] += bf16hi(u.w);
                }
              }
            }
            store_row_chunk(crow, n, args.N, v);
          }
        }
      } else if (EPI == EPI_STORE_F32) {
        float* crow = args.Cf + static_cast<size_t>(m) * args.ldc;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          fetch32(c * 32, v);
          const int n = tn * BN + c * 32;
          if (row_ok && n < args.N) {
            float4* d4 = reinterpret_cast<float4*>(crow + n);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (n + 4 * i + 4 <= args.N)
                d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      } else if (EPI == EPI_SWIGLU) {
        __nv_bfloat16* crow = args.C + static_cast<size_t>(m) * args.ldc;
        float u[32];
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          fetch32(c * 32, v);            // gate columns
          fetch32(BN / 2 + c * 32, u);   // matching up columns
          const int n = tn * (BN / 2) + c * 32;
          if (row_ok && n < args.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = v[i] / (1.0f + __expf(-v[i])) * u[i];
            store_row_chunk(crow, n, args.N, v);
          }
        }
      } else {  // EPI_QKV
        const int d = args.head_dim;
        const int nq = args.n_q, nkv = args.n_kv;
        const int pos = row_ok ? args.tok_pos[m] : 0;
        const int slot = row_ok ? args.tok_slot[m] : -1;
        const int P = args.page_size;
        const size_t page_stride = static_cast<size_t>(nkv) * P * d;
#pragma unroll 1
        for (int hh = 0; hh < BN / d; ++hh) {
          const int col0 = tn * BN + hh * d;
          const int head = col0 / d;
          const bool is_q = head < nq;
          const bool is_k = !is_q && head < nq + nkv;
          const bool in_range = col0 < args.N;
          __nv_bfloat16* dst = nullptr;
          if (row_ok && in_range) {
            if (is_q) {
              dst = args.q_out + static_cast<size_t>(m) * nq * d + static_cast<size_t>(head) * d;
            } else if (slot >= 0) {
              const int g = is_k ? head - nq : head - nq - nkv;
              __nv_bfloat16* pool = is_k ? args.k_pool : args.v_pool;
              dst = pool + static_cast<size_t>(slot / P) * page_stride +
                    static_cast<size_t>(g) * P * d + static_cast<size_t>(slot % P) * d;
            }
          }
          const int hb = hh * d;  // first accumulator column of this head
          if (is_q || is_k) {
            float w[32];
#pragma unroll 1
            for (int j0 = 0; j0 < d / 2; j0 += 32) {
              fetch32(hb + j0, v);
              fetch32(hb + d / 2 + j0, w);
              if (dst != nullptr) {
                if (pos < args.rope_positions) {  // table of (cos, sin), 16-byte loads
                  const float4* cs = reinterpret_cast<const float4*>(
                      args.rope_cs + static_cast<size_t>(pos) * (d / 2) + j0);
#pragma unroll
                  for (int i2 = 0; i2 < 16; ++i2) {
                    const float4 t = __ldg(cs + i2);
                    const float a0 = v[2 * i2], b0 = w[2 * i2];
                    const float a1 = v[2 * i2 + 1], b1 = w[2 * i2 + 1];
                    v[2 * i2] = a0 * t.x - b0 * t.y;
                    w[2 * i2] = b0 * t.x + a0 * t.y;
                    v[2 * i2 + 1] = a1 * t.z - b1 * t.w;
                    w[2 * i2 + 1] = b1 * t.z + a1 * t.w;
                  }
                } else {
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    // angle = pos * theta^(-2 i / d)
                    const float inv_freq = exp2f(-(2.0f * (j0 + i) / d) * args.log2_theta);
                    float s, c;
                    sincosf(static_cast<float>(pos) * inv_freq, &s, &c);
                    const float a = v[i], b = w[i];
                    v[i] = a * c - b * s;
                    w[i] = b * c + a * s;
                  }
                }
                store32_bf16(dst + j0, v);
                store32_bf16(dst + d / 2 + j0, w);
              }
            }
          } else {
#pragma unroll 1
            for (int j0 = 0; j0 < d; j0 += 32) {
              fetch32(hb + j0, v);
              if (dst != nullptr) store32_bf16(dst + j0, v);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tail->tempty[acc]);
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
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

int gemm_block_n(int epi) { return epi == EPI_SWIGLU ? BN_DEFAULT / 2 : BN_DEFAULT; }

int gemm_tiles(int epi, int m_rows, int N) {
  const int bn = gemm_block_n(epi);
  return ((m_rows + BM - 1) / BM) * ((N + bn - 1) / bn);
}

template <int EPI, int STAGES, int BN>
static cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap& tmB2, const GemmArgs& args, int grid,
                              cudaStream_t stream) {
  constexpr int smem = gemm_smem_bytes(STAGES, BN);
  const cudaError_t attr =
      set_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<EPI, STAGES, BN>), smem);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = args.wait_prior || args.weights_first ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI, STAGES, BN>, tmA, tmB, tmB2, args);
}

template <int EPI, int BN>
static cudaError_t launch_stages(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const CUtensorMap& tmB2, const GemmArgs& args, int grid,
                                 cudaStream_t stream) {
  switch (args.stages) {
    case 2: return launch_one<EPI, 2, BN>(tmA, tmB, tmB2, args, grid, stream);
    case 3: return launch_one<EPI, 3, BN>(tmA, tmB, tmB2, args, grid, stream);
    default: return launch_one<EPI, 4, BN>(tmA, tmB, tmB2, args, grid, stream);
  }
}

cudaError_t launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const CUtensorMap& tmB2, const GemmArgs& args, int grid,
                        cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  // the grouped GEMM reads the group offsets before any wait: never a
  // programmatic dependent
  if (args.n_groups < 0 || args.n_groups > GEMM_MAX_GROUPS ||
      (args.n_groups > 0 && (!args.group_off || args.splits > 1 || args.wait_prior ||
                             args.weights_first)))
    return cudaErrorInvalidValue;
  const int bn = args.bn ? args.bn : BN_DEFAULT;
  if (bn == 224) {  // residual epilogue only (the O and down projections)
    if (epi != EPI_RESID) return cudaErrorInvalidValue;
    return launch_stages<EPI_RESID, 224>(tmA, tmB, tmB2, args, grid, stream);
  }
  if (bn != BN_DEFAULT) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_STORE: return launch_stages<EPI_STORE, 256>(tmA, tmB, tmB2, args, grid, stream);
    case EPI_RESID: return launch_stages<EPI_RESID, 256>(tmA, tmB, tmB2, args, grid, stream);
    case EPI_SWIGLU: return launch_stages<EPI_SWIGLU, 256>(tmA, tmB, tmB2, args, grid, stream);
    case EPI_QKV: return launch_stages<EPI_QKV, 256>(tmA, tmB, tmB2, args, grid, stream);
    case EPI_STORE_F32: return launch_stages<EPI_STORE_F32, 256>(tmA, tmB, tmB2, args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  // looked up once; the initialisation of a function-local static is
  // thread-safe, so no caller sees it half done
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16 || rows == 0 || cols == 0)
    return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_groups128(CUtensorMap* map, const void* base, uint64_t rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || rows == 0 || rows % 16) return false;
  // dims (column within a half, row within an 8-row group, half, group): a box
  // of two groups lands as [group][half][8 rows][64 columns], each 8 x 64 block
  // a 1024-byte atom of the 128-byte swizzle
  cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  cuuint64_t strides[3] = {256, 128, 2048};
  cuuint32_t box[4] = {64, 8, 2, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_rows128(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || rows == 0) return false;
  // dims (column within a half, row, half): a box of box_rows rows lands as
  // [half][row][64 columns], each half in the 128-byte swizzle of a 64-column box
  cuuint64_t dims[3] = {64, rows, 2};
  cuuint64_t strides[2] = {256, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace nf
