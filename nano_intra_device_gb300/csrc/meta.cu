// Step metadata: per token its sequence, position and cache slot; per
// attention nano-batch the split-KV work list.
//
// * position: sequence s owns q_lens[s] consecutive tokens of the step, at
//   positions seq_lens[s] - q_lens[s] ... seq_lens[s] - 1;
// * slot = block_table[s][pos / P] * P + pos % P ("Inside nano-vLLM", 4.2 Paged
//   KV: the block table and the slot mapping of new KV writes);
// * work list: token t sees pos+1 positions, cut into pieces of kv_chunk
//   positions; a piece is the unit one warp of the attention kernel handles
//   (for one KV head).  Pieces are grouped by attention nano-batch (the token
//   range of each nano-operation, "NanoFlow: Towards Optimal LLM Serving
//   Throughput", "Auto-Search Stage I", constraints on dependencies) and,
//   inside a nano-batch, ordered longest first so the last pieces any warp
//   picks up are the short ones.
// One CTA does it all: a few thousand tokens, microseconds.
#include "common.cuh"
#include "kernels.h"

namespace nf {

constexpr int META_THREADS = 1024;
constexpr int META_MAX_SEG = 8;
constexpr int META_MAX_BUCKETS = 128;

__device__ __forceinline__ int upper_index(const int* bounds, int n, int t) {
  // largest i in [0, n) with bounds[i] <= t
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bounds[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int META_SMEM_SEQ = 8192;  // sequences whose token starts fit in shared memory

__global__ void __launch_bounds__(META_THREADS) meta_kernel(const MetaArgs a) {
  // The first QKV GEMM of the step may start now on the other SMs: only its
  // epilogue reads the token map, after waiting for this grid.
  pdl_trigger();
  __shared__ int hist[META_MAX_SEG * META_MAX_BUCKETS];
  __shared__ int cursor[META_MAX_SEG * META_MAX_BUCKETS];
  __shared__ int sbegin[META_SMEM_SEQ + 1];
  __shared__ int sseg[META_MAX_SEG + 1];
  const int P = a.page_size, C = a.kv_chunk;
  const int nb = C / P;  // buckets: pieces of 1..nb pages
  for (int i = threadIdx.x; i < META_MAX_SEG * META_MAX_BUCKETS; i += META_THREADS) hist[i] = 0;
  // the token starts of the sequences and the nano-batch bounds are searched
  // once per token: keep them in shared memory when they fit
  const bool in_smem = a.n_seq <= META_SMEM_SEQ;
  if (in_smem)
    for (int i = threadIdx.x; i <= a.n_seq; i += META_THREADS) sbegin[i] = a.tok_begin[i];
  for (int i = threadIdx.x; i <= a.n_seg; i += META_THREADS) sseg[i] = a.seg_bounds[i];
  __syncthreads();
  const int* tb = in_smem ? sbegin : a.tok_begin;

  // pass 1: token map, slots, piece histogram
  for (int t = threadIdx.x; t < a.n_tok; t += META_THREADS) {
    const int s = upper_index(tb, a.n_seq, t);
    const int L = a.seq_lens[s], q = a.q_lens[s];
    int pos = L - q + (t - tb[s]);
    bool ok = true;
    if (q < 1 || L < q || pos >= a.max_pages * P) {
      raise_status(a.status, ST_BAD_LEN);
      ok = false;
      pos = 0;
    }
    int slot = -1;
    if (ok) {
      const int page = a.block_table[static_cast<size_t>(s) * a.max_pages + pos / P];
      if (page >= 0 && page < a.num_pages) {
        slot = page * P + pos % P;
      } else {
        raise_status(a.status, ST_BAD_PAGE);
      }
      if (a.validate) {  // every page the token's attention will read
        for (int j = 0; j <= pos / P; ++j) {
          const int pg = a.block_table[static_cast<size_t>(s) * a.max_pages + j];
          if (pg < 0 || pg >= a.num_pages) {
            raise_status(a.status, ST_BAD_PAGE);
            break;
          }
        }
      }
    }
    const int ctx = ok ? pos + 1 : 0;
    int nch = (ctx + C - 1) / C;
    if (nch > a.max_chunks) {
      raise_status(a.status, ST_OVERFLOW);
      nch = a.max_chunks;
    }
    a.tok_seq[t] = s;
    a.tok_pos[t] = pos;
    a.tok_slot[t] = slot;
    a.tok_nchunks[t] = nch;
    const int seg = upper_index(sseg, a.n_seg, t);
    for (int c = 0; c < nch; ++c) {
      const int len = min(C, ctx - c * C);
      const int npg = (len + P - 1) / P;
      atomicAdd(&hist[seg * META_MAX_BUCKETS + (nb - npg)], 1);
    }
  }
  __syncthreads();

  // exclusive scan over (segment, bucket) in order
  if (threadIdx.x == 0) {
    int run = 0;
    for (int sg = 0; sg < a.n_seg; ++sg) {
      a.seg_items[sg] = min(run, a.item_capacity);
      for (int b = 0; b < nb; ++b) {
        cursor[sg * META_MAX_BUCKETS + b] = run;
        run += hist[sg * META_MAX_BUCKETS + b];
      }
    }
    if (run > a.item_capacity) raise_status(a.status, ST_OVERFLOW);
    a.seg_items[a.n_seg] = min(run, a.item_capacity);
  }
  __syncthreads();

  // pass 2: scatter pieces
  for (int t = threadIdx.x; t < a.n_tok; t += META_THREADS) {
    const int ctx = a.tok_pos[t] + 1;
    const int nch = a.tok_nchunks[t];
    const int seg = upper_index(sseg, a.n_seg, t);
    for (int c = 0; c < nch; ++c) {
      const int len = min(C, ctx - c * C);
      const int npg = (len + P - 1) / P;
      const int at = atomicAdd(&cursor[seg * META_MAX_BUCKETS + (nb - npg)], 1);
      if (at < a.item_capacity) {
        a.items[2 * at] = t;
        a.items[2 * at + 1] = c;
      }
    }
  }
  const int sets = a.counter_sets > 0 ? a.counter_sets : 1;
  for (int i = threadIdx.x; i < a.fetch_stride * sets; i += META_THREADS) a.fetch[i] = 0;
  const int4 z = make_int4(0, 0, 0, 0);
  const int n_done = a.n_tok * a.n_kv * sets;  // multiple of 4: row_done is 16-byte aligned
  for (int i = threadIdx.x; i < n_done / 4; i += META_THREADS) reinterpret_cast<int4*>(a.row_done)[i] = z;
  for (int i = (n_done / 4) * 4 + threadIdx.x; i < n_done; i += META_THREADS) a.row_done[i] = 0;
}

cudaError_t launch_meta(const MetaArgs& a, cudaStream_t stream) {
  if (a.n_seg > META_MAX_SEG || a.kv_chunk / a.page_size > META_MAX_BUCKETS)
    return cudaErrorInvalidValue;
  meta_kernel<<<1, META_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace nf
