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
// One CTA does it all: a few thousand tokens, microseconds.  In the
// sequential executor the token map comes from RMSNorm-1 (rmsnorm.cu) and this
// kernel, which then only builds the work list, runs beside the first QKV GEMM.
#include "common.cuh"
#include "kernels.h"
#include "tokmap.cuh"

namespace nf {

constexpr int META_THREADS = 1024;
constexpr int META_MAX_SEG = 8;
constexpr int META_MAX_BUCKETS = 128;

constexpr int META_SMEM_SEQ = 8192;  // sequences whose token starts fit in shared memory

__global__ void __launch_bounds__(META_THREADS) meta_kernel(const MetaArgs a) {
  // A programmatic dependent (the first QKV GEMM of a two-stream step, which
  // reads the token map only in its epilogue, after waiting for this grid) may
  // start now on the other SMs.
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
  TokMap tm{};
  tm.seq_lens = a.seq_lens;
  tm.q_lens = a.q_lens;
  tm.block_table = a.block_table;
  tm.max_pages = a.max_pages;
  tm.num_pages = a.num_pages;
  tm.page_size = P;
  tm.kv_chunk = C;
  tm.max_chunks = a.max_chunks;
  tm.validate = a.validate;
  tm.status = a.status;
  for (int t = threadIdx.x; t < a.n_tok; t += META_THREADS) {
    const int s = tok_seq_search(tb, 0, a.n_seq, t);
    const TokEntry e = token_entry(tm, s, tb[s], t, !a.map_done);
    if (!a.map_done) {
      a.tok_seq[t] = s;
      a.tok_pos[t] = e.pos;
      a.tok_slot[t] = e.slot;
      a.tok_nchunks[t] = e.nch;
    }
    const int ctx = e.nch > 0 ? e.pos + 1 : 0;
    const int seg = tok_seq_search(sseg, 0, a.n_seg, t);
    for (int c = 0; c < e.nch; ++c) {
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

  // pass 2: scatter pieces (the token map is this kernel's own output, or
  // derived again where the RMSNorm kernels write it)
  for (int t = threadIdx.x; t < a.n_tok; t += META_THREADS) {
    int ctx, nch;
    if (a.map_done) {
      const int s = tok_seq_search(tb, 0, a.n_seq, t);
      const TokEntry e = token_entry(tm, s, tb[s], t, false);
      nch = e.nch;
      ctx = nch > 0 ? e.pos + 1 : 0;
    } else {
      ctx = a.tok_pos[t] + 1;
      nch = a.tok_nchunks[t];
    }
    const int seg = tok_seq_search(sseg, 0, a.n_seg, t);
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
  // Launched as a programmatic dependent of the first QKV GEMM: end only after
  // it, so that whatever follows on the stream sees both.
  pdl_wait();
}

cudaError_t launch_meta(const MetaArgs& a, cudaStream_t stream) {
  if (a.n_seg > META_MAX_SEG || a.kv_chunk / a.page_size > META_MAX_BUCKETS)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(META_THREADS, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = a.map_done ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, meta_kernel, a);
}

}  // namespace nf
