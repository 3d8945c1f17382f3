// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nf {

// ------------------------------------------------------------------ GEMM
enum GemmEpi : int { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_QKV = 3, EPI_STORE_F32 = 4 };
constexpr int GEMM_MAX_GROUPS = 64;

struct GemmArgs {
  int m_begin, m_end;   // output rows [m_begin, m_end)
  int N;                // output columns (F for SwiGLU)
  int K;
  int m_tiles, n_tiles; // tiles over the row range / the output columns
  __nv_bfloat16* C;     // STORE/RESID/SWIGLU output, row stride ldc
  int ldc;
  const __nv_bfloat16* R;  // RESID residual, row stride ldr
  int ldr;
  // QKV epilogue: RoPE on q and k, q to q_out, k and v appended to the pools
  const int* tok_pos;
  const int* tok_slot;
  __nv_bfloat16* q_out;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  int n_q, n_kv, head_dim, page_size;
  float log2_theta;
  // RoPE table: (cos, sin) of pos * theta^(-2i/d) at [pos][i], i < d/2, for
  // positions below rope_positions (computed in double precision on the host);
  // positions past it fall back to sincosf
  const float2* rope_cs;
  int rope_positions;
  int stages;           // ring stages: 4 (fills an SM), 3 or 2 (room for attention)
  int bn;               // output columns per tile: 0 or 256; 224 (residual epilogue only)
  // split-K (for few output tiles): each tile's K range is cut into `splits`
  // pieces on different CTAs; fp32 partials in `part` [tiles][splits][128][BN],
  // per-tile arrival counters `tile_cnt` (zero between launches)
  int splits;
  float* part;
  int* tile_cnt;
  // grouped GEMM (mixture of experts): with n_groups > 0, row group e of A is
  // [group_off[e], group_off[e+1]) (device array: the sizes are known only on
  // the GPU) and multiplies the B rows from e * b_group_rows; tiles are
  // enumerated on the device.  For SwiGLU the up rows of a group start
  // b2_row_off rows after its gate rows (tmB2 may then be tmB).  No split-K.
  const int* group_off;
  int n_groups;
  int b_group_rows;
  int b2_row_off;
  float* Cf;            // EPI_STORE_F32 output, row stride ldc
  // 1: launched as a programmatic dependent of the step-metadata kernel, whose
  // outputs (token positions and cache slots) only the epilogue reads; A was
  // complete before that kernel started.  The TMA and MMA warps start at once,
  // the epilogue warps wait for the metadata before their first tile.
  int wait_prior;
  // 1: launched as a programmatic dependent of the kernel that writes A (not
  // B): the producer issues the B (weight) loads of its first ring stages
  // before it waits for that kernel; A, the residual and every output come
  // after the wait.  Not with the grouped GEMM.
  int weights_first;
  uint32_t* status;
  unsigned long long timeout_ns;
};

// Build a 2-D bf16 tensor map over a row-major [rows, cols] matrix with a
// box of box_rows x 64 columns and 128-byte swizzle.  Returns false on error.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);

// C = A * B^T (+ epilogue).  tmA over A [*, K], tmB over B; for SwiGLU tmB is
// the gate rows and tmB2 the up rows.  grid = persistent CTA count.
cudaError_t launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const CUtensorMap& tmB2, const GemmArgs& args, int grid,
                        cudaStream_t stream);
int gemm_block_n(int epi);
int gemm_tiles(int epi, int m_rows, int N);

// Weight-row GEMM for few tokens (gemm_wrows.cu): tiles of 128 output
// features x tok tokens (tok = 64 or 128), the tokens [m_begin, m_end).
// tmW: weight rows, 128-row boxes (QKV: head_dim / 2-row boxes; SwiGLU: the
// gate rows, tmW2 the up rows from b2_row_off); tmX: the tokens' activations,
// tok-row boxes.  n_tiles = weight tiles (ceil(N / 128); QKV: ceil(heads /
// (256 / head_dim))), m_tiles = token tiles, splits = CTAs per cluster (1..8,
// at most the K blocks of 64), which split K and sum through distributed
// shared memory.  grid = clusters x splits CTAs.  EPI_STORE, EPI_RESID,
// EPI_SWIGLU, EPI_QKV; N a multiple of 4.  programmatic: launch as a
// programmatic dependent of the kernel ahead in the stream, which must be one
// of this library's kernels launched after every write to the weights (the
// first ring of weights is read before that kernel has finished).
cudaError_t launch_gemm_wrows(int epi, int tok, const CUtensorMap& tmW, const CUtensorMap& tmW2,
                              const CUtensorMap& tmX, const GemmArgs& args, int clusters,
                              bool programmatic, cudaStream_t stream);
// Clusters of `cluster` CTAs of that kernel that fit on the device at once
// (0 when the query fails).  Cached per process.
int gemm_wrows_max_clusters(int epi, int tok, int cluster);

// ------------------------------------------------------ mixture of experts
// Top-k routing of the tokens [r0, r0 + n) from router logits [*, E] fp32
// (ties to the lower expert index, weights = softmax over the selected logits)
// and their grouping by expert: rows of the grouped order are pairs (token,
// choice), expert by expert, tokens increasing within an expert.  Writes
// group_off [E + 1], perm_tok [n * k] (token of each grouped row), pair_row
// [n * k] (grouped row of pair t * k + j) and pair_w [n * k].  One CTA.
cudaError_t launch_moe_route(const float* logits, int r0, int n, int n_experts, int top_k,
                             int* group_off, int* perm_tok, int* pair_row, float* pair_w,
                             cudaStream_t stream);
// dst[row] = src[perm_tok[row]] for row < rows (bf16 rows of `cols`, cols % 8 == 0);
// an index outside [0, src_rows) gives a zero row and flags ST_BAD_LEN.
cudaError_t launch_gather_rows(const __nv_bfloat16* src, const int* perm_tok, __nv_bfloat16* dst,
                               int rows, int cols, int src_rows, uint32_t* status,
                               cudaStream_t stream);
// y[t] = h[t] + sum_j pair_w[i k + j] * part[pair_row[i k + j]] for t = r0 + i, i < n
// (fp32 sum in choice order, one bf16 rounding).
cudaError_t launch_moe_combine(const __nv_bfloat16* h, const float* part, const int* pair_row,
                               const float* pair_w, __nv_bfloat16* y, int r0, int n, int top_k,
                               int hidden, cudaStream_t stream);

// ----------------------------------------------------------- token map
// Inputs and outputs of the per-token map (tokmap.cuh): sequence, position,
// cache slot and split-KV piece count of each token of the step.
struct TokMap {
  const int* seq_lens;      // device [n_seq]
  const int* q_lens;        // device [n_seq]
  const int* tok_begin;     // device [n_seq + 1]
  const int* block_table;   // device [n_seq, max_pages]
  int n_seq, n_decode;      // sequences; the first n_decode own one token each
  int max_pages, num_pages, page_size, kv_chunk, max_chunks, validate;
  int* tok_seq;             // out [n_tok]
  int* tok_pos;             // out [n_tok]
  int* tok_slot;            // out [n_tok]
  int* tok_nchunks;         // out [n_tok]
  uint32_t* status;
};

// --------------------------------------------------------------- RMSNorm
// map != nullptr: the CTA of row t also writes the token map of token t
// (RMSNorm-1 of a step, whose rows are the step's tokens).
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* out,
                           int row_begin, int row_end, int hidden, float eps, cudaStream_t stream,
                           const TokMap* map = nullptr);

// Embedding lookup: x[t] = embed[tokens[t]] (rows of H bf16); an id outside
// [0, vocab) flags ST_BAD_LEN and writes a zero row.
cudaError_t launch_embed(const int* tokens, const __nv_bfloat16* embed, __nv_bfloat16* x, int n_tok,
                         int hidden, int vocab, uint32_t* status, cudaStream_t stream);

// ---------------------------------------------------------- step metadata
struct MetaArgs {
  const int* seq_lens;      // device [n_seq]
  const int* block_table;   // device [n_seq, max_pages]
  const int* q_lens;        // device [n_seq]
  const int* tok_begin;     // device [n_seq + 1]
  const int* seg_bounds;    // device [n_seg + 1], attention nano-batch token bounds
  int n_seq, n_tok, n_seg, max_pages, num_pages, page_size, kv_chunk, n_kv;
  int max_chunks;           // per-row chunk capacity = ceil(max_pages*page/kv_chunk)
  int item_capacity;        // pairs the item buffer holds
  int* tok_seq;             // out [n_tok]
  int* tok_pos;             // out [n_tok]
  int* tok_slot;            // out [n_tok]
  int* tok_nchunks;         // out [n_tok]
  int* items;               // out [2 * item_capacity] (row, chunk)
  int* seg_items;           // out [n_seg + 1] segment starts in items
  int* fetch;               // out [counter_sets * n_seg] dynamic fetch counters, zeroed
  int* row_done;            // out [counter_sets * n_tok * n_kv] split-combine counters, zeroed
  int counter_sets;         // one set per layer that attends with this metadata
  int fetch_stride;         // fetch counters per set
  uint32_t* status;
  int validate;
  // 1: the step's RMSNorm-1 kernels write the token map; this kernel derives
  // positions for the work list itself, writes no token map, and is launched
  // as a programmatic dependent of the first QKV GEMM (which reads nothing it
  // writes): it waits for that GEMM only before it ends
  int map_done;
};
cudaError_t launch_meta(const MetaArgs& a, cudaStream_t stream);

// -------------------------------------------------------------- attention
struct AttnArgs {
  const __nv_bfloat16* q;    // [T, n_q, d]
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  __nv_bfloat16* o;          // [T, n_q, d]
  const int* block_table;
  const int* tok_seq;
  const int* tok_pos;
  const int* tok_nchunks;
  const int* items;          // (row, chunk) pairs
  const int* seg_items;      // segment starts
  int* fetch;                // per-segment fetch counter
  int* row_done;             // [T, n_kv]
  float* partials;           // [T, max_chunks, n_kv, rec]
  int seg;                   // which attention nano-batch
  int n_q, n_kv, head_dim, page_size, max_pages, num_pages, kv_chunk, max_chunks;
  float scale_log2;          // log2(e) / sqrt(d)
  int warps;                 // warps per CTA: 8 (3 pages in flight each); 4 leaves room for a
                             // 2-stage GEMM CTA on the same SM
  // tensor-core decode kernel: with prefill_elsewhere set, rows of sequences
  // n_decode_seqs and up (the prefill chunks) are left to the prefill kernel
  int prefill_elsewhere;
  int n_decode_seqs;
  // tensor-core decode kernel, 1: launched as a programmatic dependent of the
  // QKV GEMM that writes q and this step's K/V, with the work list and token
  // map from earlier kernels.  A warp's first piece requests its pages that lie
  // wholly before the first position the step writes, then waits for the GEMM.
  int early;
  uint32_t* status;
  unsigned long long timeout_ns;
};
int attn_partial_floats(int n_q, int n_kv, int head_dim);  // floats per (row, chunk, kv head)
// Floats of one split-KV partial record: acc [GRP][d], then m [GRP] and
// l [GRP], padded so every record starts on a 16-byte boundary (the record is
// written and read with 16-byte vector accesses).
__host__ __device__ constexpr int partial_rec_floats(int grp, int head_dim) {
  return grp * head_dim + ((2 * grp + 3) / 4) * 4;
}
// Tensor-core variant (mma.sync m16n8k16, bf16 operands, fp32 accumulators) of
// the same operation with the same records; K and V pages arrive by TMA
// copies through maps over the pools viewed as [num_pages * n_kv * 16, d]
// (make_pool_tmap_pages).  Supported: page 16, d 64 or 128, GQA group 1, 2, 4 or 8.
bool attention_mma_supported(int n_q, int n_kv, int head_dim, int page_size, int num_pages);
bool make_pool_tmap(CUtensorMap* map, const void* pool, int num_pages, int n_kv, int page_size,
                    int head_dim);
// The decode kernel's map over a pool: for d = 128 one 3-D box fetches a whole
// (page, KV head) block of K or V (both 64-column halves, the same shared
// layout as two 2-D boxes); for d = 64 the 2-D map above.
bool make_pool_tmap_pages(CUtensorMap* map, const void* pool, int num_pages, int n_kv,
                          int page_size, int head_dim);
// The prefill kernel's map over a pool: for d = 128 one 4-D box fetches a
// (page, KV head) block of K or V as [8-row group][64-column half][8 rows]
// (1024-byte atoms of the 128-byte swizzle, groups 2048 bytes apart); for
// d = 64 the 2-D map above.
bool make_pool_tmap_groups(CUtensorMap* map, const void* pool, int num_pages, int n_kv,
                           int page_size, int head_dim);
// A 4-D map over rows of 128 bf16 (rows a multiple of 16): box = 16 rows as
// [8-row group][64-column half][8 rows][64 columns].
bool make_tmap_bf16_groups128(CUtensorMap* map, const void* base, uint64_t rows);
// A 3-D map over rows of 128 bf16: box = box_rows rows, landing as two
// 128-byte-swizzled 64-column halves one after the other.
bool make_tmap_bf16_rows128(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);
// programmatic: launch as a programmatic dependent of the kernel ahead (the
// prefill kernel of the same nano-batch); the grid waits for it before it ends.
cudaError_t launch_attention_mma(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                 int grid, bool programmatic, cudaStream_t stream);
// Causal attention of prefill-chunk rows (attn_prefill.cu), flash style on the
// tensor cores: tiles[i] = (first row, end row, sequence, 0), rows of one
// prefill sequence, at most prefill_tile_rows(n_q, n_kv) of them; one CTA per
// (tile, KV head) writes o for the tile's rows.  Same shapes as
// attention_mma_supported; K/V through the same pool maps.
int prefill_tile_rows(int n_q, int n_kv);
cudaError_t launch_attention_prefill(const AttnArgs& a, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const int4* tiles, int n_tiles,
                                     cudaStream_t stream);

// Failure-detection self-test (selftest.cu): one warp waits, with the bounded
// wait of every kernel here, on a barrier nothing arrives at (arrive = 0) or
// that it arrived at itself (1); an expired wait sets ST_TIMEOUT in *status.
// waited_ns (device, optional) receives the time waited.
cudaError_t launch_selftest_wait(uint32_t* status, unsigned long long timeout_ns, int arrive,
                                 unsigned long long* waited_ns, cudaStream_t stream);

}  // namespace nf
