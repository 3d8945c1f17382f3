/*
 * nanoflow.h — C ABI of the GB300 (sm_103a) nano-batched decoder-layer step.
 *
 * One call, nf_layer_step, runs one pre-norm decoder layer over a mixed batch
 * of decode requests and prefill chunks whose K/V live in a paged cache:
 *
 *   n1 = RMSNorm(x; g1)                 [T, H]
 *   q|k|v = n1 W_qkv^T, RoPE on q and k, k and v appended to the paged cache
 *   o = GQA softmax attention of each token over positions 0..pos of its
 *       sequence (decode: the whole history; prefill: causal)
 *   h = x + o W_o^T
 *   y = h + (silu(n2 W_g^T) * (n2 W_u^T)) W_d^T,  n2 = RMSNorm(h; g2)
 *
 * The batch is cut into nano-batches of tokens so that the tensor-core GEMMs of
 * one nano-batch run on the GPU while the HBM-bound decode attention of another
 * runs beside them ("NanoFlow: Towards Optimal LLM Serving Throughput",
 * "The Intra-Device Parallelism Mechanism").  A plan fixes the split, the order
 * and the SM share of each nano-operation ("Auto-Search Stage I" and
 * "Auto-Search Stage II" of the same page); the result never depends on it.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device pointers on the current device;
 *    "host" pointers are ordinary host memory.  The caller owns all buffers it
 *    passes; the library never frees or reallocates them.
 *  - Tensors are dense, row-major, bf16 (stored as 16-bit words) unless stated.
 *  - Calls that take a `stream` (a cudaStream_t, NULL = legacy default stream)
 *    only enqueue work and return; results are ready when the stream completes.
 *  - Argument errors are detected on the host before anything is launched and
 *    return NF_ERR_INVALID_ARG with a message in nf_last_error().  Device-side
 *    problems (a page id outside the pool, a bounded wait that gave up) set a
 *    status word in the plan; nf_plan_poll reports it.  Nothing traps.
 *  - No entry point throws across the ABI.  Functions are thread-safe except
 *    that one plan must not be used by two threads at once.
 */
#ifndef NANOFLOW_H
#define NANOFLOW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NF_MAX_NANO 8

typedef enum {
  NF_OK = 0,
  NF_ERR_INVALID_ARG = 1, /* a size, pointer or layout the library does not accept */
  NF_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement */
  NF_ERR_OOM = 3,         /* device or host allocation failed */
  NF_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  NF_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (from nf_plan_poll) */
  NF_ERR_DEVICE = 6,      /* device-side check failed, e.g. page id out of range */
  NF_ERR_INTERNAL = 7
} nf_status;

typedef enum {
  NF_EXEC_SEQUENTIAL = 0, /* every nano-operation in order on the caller's stream */
  NF_EXEC_STREAMS = 1     /* GEMMs and attention on two streams ordered by events,
                             each kernel capped to its SM share */
} nf_executor;

typedef enum {
  NF_ATTN_AUTO = 0, /* NF_ATTN_MMA */
  NF_ATTN_MMA = 2   /* dot products on the tensor cores (mma.sync, bf16 x bf16 -> fp32), each
                       warp streaming its own pages; values 1 (a CUDA-core kernel) and 3 (a
                       warp-specialised variant), both removed, are refused */
} nf_attn_impl;

/* Shape of one Llama-style decoder layer.  head_dim in {64, 128};
 * n_q_heads a multiple of n_kv_heads with n_q/n_kv in {1, 2, 4, 8};
 * hidden and ffn multiples of 16; page_size = 16.
 * n_experts = 0: dense SwiGLU FFN.  n_experts in [1, 64]: a mixture of that
 * many SwiGLU experts of width ffn, each token routed to top_k (1 or 2) of them
 * ("NanoFlow: Towards Optimal LLM Serving Throughput", MoE models: gate
 * routing and a grouped GEMM in which experts compute on different tokens). */
typedef struct {
  int32_t hidden;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t ffn;
  int32_t page_size;
  float rms_eps;
  float rope_theta;
  int32_t n_experts;
  int32_t top_k;
} nf_model_shape;

/* Structure of the mixed batch a plan serves ("NanoFlow: Towards Optimal LLM
 * Serving Throughput", "The NanoFlow Runtime System", batch formation: decode
 * requests first, prefill chunks fill the rest of a constant dense batch).
 * Tokens [0, n_decode) are decode requests, one token each (sequence i = token
 * i); then n_prefill chunks, chunk j holding prefill_q_lens[j] consecutive
 * tokens of sequence n_decode + j.  T = n_decode + sum(prefill_q_lens). */
typedef struct {
  int32_t n_decode;
  int32_t n_prefill;
  const int32_t* prefill_q_lens; /* host [n_prefill]; copied by nf_plan_create */
  const int32_t* seq_lens_hint;  /* host [n_decode + n_prefill] or NULL: typical KV
                                    lengths, used only by the plan search */
  int32_t max_pages_per_seq;     /* row stride of the block table */
  int32_t num_pages;             /* pages in each of the K and V pools */
} nf_batch_desc;

/* A plan: the nano-batch split and the resources of each nano-operation
 * (the output of the pages' two-stage auto-search).  Passed to nf_plan_create
 * to force a plan, or read back with nf_plan_info.
 * attn_bounds: token boundaries of the attention group (QKV projection,
 *   attention, O projection): nano-batch i is [attn_bounds[i], attn_bounds[i+1]),
 *   attn_bounds[0] = 0, attn_bounds[n_attn] = T, strictly increasing.
 * ffn_bounds: the same for the FFN group (RMSNorm-2, gate/up, down). */
typedef struct {
  int32_t n_attn;
  int32_t attn_bounds[NF_MAX_NANO + 1];
  int32_t n_ffn;
  int32_t ffn_bounds[NF_MAX_NANO + 1];
  int32_t executor;   /* nf_executor */
  int32_t attn_sms;   /* SMs for attention while it overlaps GEMMs (0 = automatic) */
  int32_t gemm_sms;   /* SMs for a GEMM while it overlaps attention (0 = the rest) */
  int32_t kv_chunk;   /* split-KV piece in tokens, multiple of page_size, <= 2048 (0 = 1024) */
  int32_t attn_warps; /* warps per attention CTA (0 = 8): 4 shares each SM with one GEMM
                         CTA of gemm_stages = 2 (3-page rings, 117 KB, <= 128 registers a
                         thread); 5 ... 8, 10, 12 or 14 fill an SM, ring stages per warp as
                         deep as shared memory allows (5: 5, 6: 4, 7: 4, 8: 3, more warps:
                         2 pages) */
  int32_t gemm_stages; /* shared-memory ring stages of the GEMM kernel: 4 fills an SM;
                          2 lets an attention CTA of 4 warps run on the same SM (0 = 4) */
  int32_t gemm_split_k; /* 0: a GEMM of at most 128 tokens runs the weight-row kernel (128
                           output features x 64 or 128 tokens a tile, K split over the CTAs
                           of a cluster, partial tiles summed in distributed shared memory);
                           a larger one splits K across CTAs when it has fewer output tiles
                           than half its SMs.  1: token-row tiles, never split.  2: token-row
                           tiles, split as in 0 (no weight-row kernel) */
  int32_t attn_impl;  /* nf_attn_impl; nf_plan_info reports the kernel chosen */
  int32_t validate;   /* 1 = check page ids and lengths on the device */
  int64_t timeout_ns; /* limit of every device-side wait (0 = 2e9) */
} nf_plan_opts;

typedef struct nf_plan_s* nf_plan;

/* Layer weights, all device, bf16.
 * norm1, norm2: [H].  w_qkv: [(n_q + 2 n_kv) * head_dim, H], rows are the q
 * heads, then the k heads, then the v heads.  w_o: [H, n_q * head_dim].
 * w_gate_up: [2 F, H], gate rows then up rows.  w_down: [H, F]. */
typedef struct {
  const void* norm1;
  const void* w_qkv;
  const void* w_o;
  const void* norm2;
  const void* w_gate_up;   /* dense FFN (n_experts = 0); NULL for a MoE layer */
  const void* w_down;      /* dense FFN; NULL for a MoE layer */
  /* Mixture of experts (n_experts > 0), device:
   * w_experts_gate_up [E, 2F, H] bf16 (per expert its gate rows, then its up rows),
   * w_experts_down [E, H, F] bf16, router_logits [T, E] fp32: this step's router
   * logits, one row per token.  Routing: the top_k logits of a token, ties to
   * the lower expert index, weighted by a softmax over the selected logits. */
  const void* w_experts_gate_up;
  const void* w_experts_down;
  const void* router_logits;
} nf_layer_weights;

/* Create a plan for one model shape and batch structure
 * ("Auto-Search Stage I" / "Stage II": split, order, resource share).
 * opts NULL: search the split and the SM shares with the library's cost
 * model (uses seq_lens_hint when given).  opts non-NULL: use it as given
 * (validated).  Allocates the plan's device workspace on the current device.
 * Errors: NF_ERR_INVALID_ARG (shape/batch/opts), NF_ERR_OOM, NF_ERR_CUDA. */
nf_status nf_plan_create(const nf_model_shape* shape, const nf_batch_desc* batch,
                         const nf_plan_opts* opts, nf_plan* out);

/* Give the plan the structure of the next step's batch (the runtime's batch
 * formation changes it every iteration): at most the sequences and tokens the
 * plan was created for, the same max_pages_per_seq and num_pages.  opts: a
 * new split and SM shares for it (kv_chunk, attn_impl and attn_warps must stay
 * as created; 0 fields take the plan's values), or NULL to keep the current
 * split, or to fall back to one sequential nano-batch when the token count
 * changed.  The device copies are enqueued on `stream` (pinned staging, no
 * allocation after the first call); steps enqueued after it on that stream see
 * the new batch.  A plan serves one stream at a time. */
nf_status nf_plan_set_batch(nf_plan plan, const nf_batch_desc* batch, const nf_plan_opts* opts,
                            void* stream);

/* The plan's split and resources, and the batch's token count. */
nf_status nf_plan_info(nf_plan plan, nf_plan_opts* out, int32_t* n_tokens);

/* Write / read a plan (shape, batch structure and opts) as a text file. */
nf_status nf_plan_save(nf_plan plan, const char* path);
nf_status nf_plan_load(const char* path, nf_plan* out);

/* Free a plan and its device workspace.  The caller must make sure no step
 * that uses the plan is still running.  NULL is ignored. */
void nf_plan_destroy(nf_plan plan);

/* One decoder-layer step (see the top of this file).
 * x, y: device [T, H]; x != y (no aliasing).
 * k_pool, v_pool: device [num_pages, n_kv, page_size, head_dim]; the step
 *   writes this step's k (after RoPE) and v at slot(seq, pos) =
 *   block_table[seq][pos / page_size] * page_size + pos % page_size, and reads
 *   positions 0..pos of each token's sequence.
 * block_table: device int32 [n_seq, max_pages_per_seq]; must cover every
 *   position < seq_lens[s].
 * seq_lens: device int32 [n_seq], KV length of each sequence AFTER this step:
 *   decode token i sits at position seq_lens[i] - 1; prefill chunk j continues
 *   its prompt at position seq_lens[s] - prefill_q_lens[j].
 * A slot this step writes must not be read by another sequence of the step
 *   (a page that two sequences share may hold only positions before both
 *   sequences' new tokens).
 * Returns after enqueueing on `stream`.  The step's first kernel waits for all
 * work enqueued on `stream` before it and work enqueued after it waits for the
 * step's last kernel; inside the step, kernels may start as programmatic
 * dependents of the one ahead and wait for it before they read its output. */
nf_status nf_layer_step(nf_plan plan, const nf_layer_weights* w, const void* x, void* k_pool,
                        void* v_pool, const int32_t* block_table, const int32_t* seq_lens, void* y,
                        void* stream);

/* A stack of decoder layers over one mixed step ("NanoFlow: Towards Optimal
 * LLM Serving Throughput", "Example Pipelines for Different Model Scales": the
 * per-layer pipeline repeated over the model): x = embed[tokens], then every
 * layer l with its own weights and K/V pools (the block table and lengths are
 * shared), then logits = RMSNorm(x; norm_f) lm_head^T.
 * embed, lm_head: device [vocab, H] bf16, vocab a multiple of 8; norm_f: [H].
 * layers: HOST array [n_layers] of device weight sets.
 * tokens: device int32 [T] token ids (an id outside [0, vocab) gives a zero
 *   row and sets the device status NF_ERR_DEVICE).
 * k_pools, v_pools: HOST arrays [n_layers] of device pools, laid out as for
 *   nf_layer_step.  logits: device [T, vocab] bf16.
 * The first call for a given n_layers may allocate (activation buffers and
 * one split-KV counter set per layer) and synchronizes the device once;
 * later calls only enqueue work and can be captured in a CUDA graph. */
typedef struct {
  const void* embed;
  const void* norm_f;
  const void* lm_head;
  int32_t vocab;
  int32_t n_layers;
  const nf_layer_weights* layers;
} nf_stack_weights;
nf_status nf_stack_step(nf_plan plan, const nf_stack_weights* w, const int32_t* tokens,
                        void* const* k_pools, void* const* v_pools, const int32_t* block_table,
                        const int32_t* seq_lens, void* logits, void* stream);

/* The same step with logits only for the rows that need them (a serving loop
 * samples one token per emitting row): rows [n_rows] are device int32 token
 * indices in [0, T) (an index outside makes nf_plan_poll report NF_ERR_DEVICE and
 * gives a zero row), logits [n_rows, vocab] row i for token rows[i].  The last
 * hidden states of those rows are gathered before the final RMSNorm, so the
 * LM head multiplies n_rows rows instead of T.  0 <= n_rows <= T. */
nf_status nf_stack_step_rows(nf_plan plan, const nf_stack_weights* w, const int32_t* tokens,
                             void* const* k_pools, void* const* v_pools,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const int32_t* rows, int32_t n_rows, void* logits, void* stream);

/* n_layers decoder layers over one mixed step, hidden states in and out
 * ("NanoFlow: Towards Optimal LLM Serving Throughput", "Example Pipelines for
 * Different Model Scales": the per-layer pipeline repeated over the layers a
 * GPU holds): layer l reads the previous layer's output (x for l = 0) and
 * appends this step's K/V into its own pools; the last layer writes y.
 * layers, k_pools, v_pools: HOST arrays [n_layers] (device weights and pools
 * as for nf_layer_step).  x, y: device [T, H] bf16, distinct; x is not
 * modified.  The step metadata is computed once for all layers.  Allocation
 * and capture behave as for nf_stack_step.  With the two-stream executor and
 * the same n >= 2 nano-batches in both groups (the same holds for
 * nf_stack_step), the layers are not joined: nano-batch i of layer l + 1
 * starts right after the FFN of nano-batch i of layer l (the pages'
 * cross-layer window); results do not depend on it. */
nf_status nf_layers_step(nf_plan plan, const nf_layer_weights* layers, int32_t n_layers,
                         const void* x, void* const* k_pools, void* const* v_pools,
                         const int32_t* block_table, const int32_t* seq_lens, void* y,
                         void* stream);

/* The same step with the per-step inputs and the output in HOST memory:
 * x_host [T, H] bf16, block_table_host and seq_lens_host as above, y_host
 * [T, H].  Copies them through plan-owned device staging buffers on `stream`
 * and synchronizes the stream before returning (y_host is then valid).
 * Pinned host memory gives full copy bandwidth; pageable memory works.  With
 * pinned buffers (and no capture or trace in progress) the second call with the
 * same pointers captures the copies and the step into a CUDA graph, and later
 * calls replay it on a plan-owned stream ordered after `stream`: one launch per
 * step instead of one per copy and kernel.  nf_plan_set_batch invalidates the
 * captured graphs.  The host buffers' contents are read at each call. */
nf_status nf_layer_step_host(nf_plan plan, const nf_layer_weights* w, const void* x_host,
                             void* k_pool, void* v_pool, const int32_t* block_table_host,
                             const int32_t* seq_lens_host, void* y_host, void* stream);

/* The same step, pipelined: enqueues the copies of the inputs on a plan-owned
 * copy stream into one of two staging slots, the step on `stream`, and the copy
 * of y back to y_host on a second plan-owned copy stream, and returns without
 * waiting.  Consecutive calls overlap one step's copies with the neighbouring
 * steps' compute (events keep a slot from being refilled before the step that
 * read it has finished, and from being rewritten before its y was copied out).
 * Host buffers should be pinned; x_host, block_table_host and seq_lens_host
 * must stay unchanged, and y_host unread, until nf_plan_host_wait returns.
 * Steps run in call order on `stream` (the KV pools carry from one to the next). */
nf_status nf_layer_step_host_async(nf_plan plan, const nf_layer_weights* w, const void* x_host,
                                   void* k_pool, void* v_pool, const int32_t* block_table_host,
                                   const int32_t* seq_lens_host, void* y_host, void* stream);

/* Wait until every step enqueued by nf_layer_step_host_async has copied its y
 * out to the host. */
nf_status nf_plan_host_wait(nf_plan plan);

/* Report device-side errors of earlier steps.  wait != 0 synchronizes the
 * device first.  Returns NF_OK, NF_ERR_TIMEOUT or NF_ERR_DEVICE (and clears
 * the status word), or NF_ERR_CUDA for an asynchronous CUDA error. */
nf_status nf_plan_poll(nf_plan plan, int wait);

/* Failure-detection self-test: enqueues one warp that waits, through the
 * bounded wait that every kernel of this library uses, on a shared-memory
 * barrier that nothing arrives at (arrive = 0), or, as the control, one that
 * it has arrived at itself (arrive = 1), for at most timeout_ns.  An expired
 * wait sets the plan's status word as a kernel's would, so nf_plan_poll then
 * returns NF_ERR_TIMEOUT; nothing else is affected and the plan stays usable.
 * waited_ns: NULL or a device uint64 that receives the nanoseconds waited.
 * NF_ERR_INVALID_ARG for a NULL plan or timeout_ns outside [1, 1e10]. */
nf_status nf_plan_selftest_wait(nf_plan plan, int64_t timeout_ns, int32_t arrive, void* waited_ns,
                                void* stream);

/* Text of the last error on the calling thread ("" if none). */
const char* nf_last_error(void);

/* Number of SMs the plan's device has (the unit of SM shares). */
int32_t nf_device_sm_count(void);

/* ---------------------------------------------------------------------------
 * Single steps of the path, for tests and for the profiler.  Each runs exactly
 * the kernel nf_layer_step runs for that step.
 */

/* Step metadata (integer, bit-exact): per token its sequence, position and
 * cache slot, and the split-KV attention work list of each attention
 * nano-batch.  ("NanoFlow: Towards Optimal LLM Serving Throughput",
 * "Auto-Search Stage I", constraints on dependencies: a nano-operation's token
 * range; "Inside nano-vLLM", 4.2 Paged KV: slot mapping.)  Reads block_table and
 * seq_lens (device, as in nf_layer_step); results stay in the plan, read them
 * with nf_plan_copy_buffer. */
nf_status nf_step_metadata(nf_plan plan, const int32_t* block_table, const int32_t* seq_lens,
                           void* stream);

/* Paged GQA attention of every token of the batch, from q already computed:
 * q: device [T, n_q, head_dim] (RoPE applied); o: device [T, n_q, head_dim].
 * The cache must already hold this step's K/V.  Runs nf_step_metadata first.
 * ("NanoFlow: Towards Optimal LLM Serving Throughput", "The Intra-Device
 * Parallelism Mechanism": decode attention is the memory-bound operation;
 * "LLM Inference Performance", "PagedAttention".) */
nf_status nf_attention(nf_plan plan, const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* block_table, const int32_t* seq_lens, void* o, void* stream);

/* Size of the fixed device working memory of nf_attention_noalloc, and the
 * largest number of prefill chunks one call takes. */
#define NF_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
#define NF_NOALLOC_MAX_PREFILL 64

/* nf_attention for callers that cannot allocate device memory.  No counterpart
 * on the pages: it exists for callers of this library that must not call
 * cudaMalloc, e.g. a host runtime that owns all device memory through its own
 * pool and gives an operator only its input and output pointers, or a hot
 * loop that cannot take the device synchronisation an allocation may cause.
 * It needs no plan.  Inputs and outputs are those of nf_attention (shape and
 * batch structure as for nf_plan_create, with at most NF_NOALLOC_MAX_PREFILL
 * prefill chunks; q, o device [T, n_q, head_dim]; pools, block table and
 * seq_lens device, the cache already holding this step's K/V).  The batch
 * structure travels by value in a kernel's arguments: no host table is copied.
 *
 * Working memory: one static device array of NF_NOALLOC_SCRATCH_BYTES, present
 * on every GPU that loads the library until the process exits.  With
 * grp = n_q / n_kv, n_seq = n_decode + n_prefill and
 * C = ceil(max_pages_per_seq * 16 / 2048) split-KV pieces per row, a call
 * needs 256 bytes (the status word) plus these regions, each rounded up to a
 * multiple of 256 bytes:
 *   4 n_seq, 4 (n_seq + 1), 8, four of 4 T, 8 T C, 8, 4, 4 T n_kv, and
 *   4 T C n_kv (grp head_dim + 4 ceil(2 grp / 4))   (the split-KV partials).
 * E.g. 1024 tokens of the Llama-3-8B shape with contexts up to 2048 fit.  A
 * batch that needs more returns NF_ERR_INVALID_ARG with the required size in
 * nf_last_error().
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call uses the same array and overwrites what the previous call left;
 * the counters that must start at zero are cleared by each call.  Calls whose
 * work overlaps on the GPU (two streams, or two threads) race on the array and
 * give wrong results: serialise them.
 *
 * Errors found on the device (a page id outside the pool, an inconsistent
 * length, a bounded wait that gave up) never fault: reads stay inside the pool
 * and the kernels set bits in a status word kept in the array.  The bits stay
 * set across calls until nf_attention_noalloc_poll reports and clears them.
 * This call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine. */
nf_status nf_attention_noalloc(const nf_model_shape* shape, const nf_batch_desc* batch,
                               const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_table, const int32_t* seq_lens, void* o,
                               void* stream);

/* Waits for `stream`, then reads and clears the status word that
 * nf_attention_noalloc calls on the current device have set since the last
 * poll: NF_OK if none, NF_ERR_TIMEOUT if a wait gave up, else NF_ERR_DEVICE
 * (the reason in nf_last_error()).  Allocates nothing. */
nf_status nf_attention_noalloc_poll(void* stream);

/* RMSNorm of rows [0, rows): out = x * g / sqrt(mean(x^2) + eps), fp32
 * arithmetic, bf16 out.  x, out: device [rows, hidden]; g: device [hidden]. */
nf_status nf_rmsnorm(const void* x, const void* g, void* out, int32_t rows, int32_t hidden,
                     float eps, void* stream);

/* Tensor-core GEMM, C = A * B^T with fp32 accumulation.
 * A: device [M, K], B: device [N, K], both bf16 row-major, K a multiple of 8,
 * 16-byte aligned rows.  epilogue:
 *   NF_EPI_STORE   C[M, N] = acc
 *   NF_EPI_RESID   C[M, N] = R[M, N] + acc          (R device [M, N])
 *   NF_EPI_SWIGLU  B holds 2F rows (gate rows then up rows), N = F:
 *                  C[M, F] = silu(A Bg^T) * (A Bu^T)
 * max_sms caps the persistent grid (0 = all SMs).  A GEMM with fewer 128 x 256
 * output tiles than half the SMs splits K across CTAs (split-K, fp32 partials
 * summed before the epilogue, the same result up to fp32 rounding order); its
 * partials use one workspace shared by every nf_gemm call (allocated on first
 * use), so such calls must not run concurrently on different streams. */
typedef enum { NF_EPI_STORE = 0, NF_EPI_RESID = 1, NF_EPI_SWIGLU = 2 } nf_epilogue;
nf_status nf_gemm(const void* A, const void* B, void* C, const void* R, int32_t M, int32_t N,
                  int32_t K, int32_t epilogue, int32_t max_sms, void* stream);

/* The same product through the weight-row kernel that layer steps use for
 * nano-operations of at most 128 tokens ("NanoFlow: Towards Optimal LLM
 * Serving Throughput", "The Intra-Device Parallelism Mechanism": the dense
 * projections): a tile is 128 rows of B (output columns) x 64 or 128 rows of
 * A, and K is split over the `splits` CTAs of a thread-block cluster whose
 * fp32 partial tiles are summed, in rank order, through distributed shared
 * memory.  Arguments as nf_gemm, with 1 <= M <= 256, N a multiple of 8;
 * splits 0 = chosen from the shape, else 1 .. 8 and at most ceil(K / 64).
 * No workspace: calls may run concurrently. */
nf_status nf_gemm_wrows(const void* A, const void* B, void* C, const void* R, int32_t M,
                        int32_t N, int32_t K, int32_t epilogue, int32_t splits, int32_t max_sms,
                        void* stream);

/* Copy one of the plan's device buffers (written by the last step or
 * metadata call on the plan's device) to dst (host or device), synchronously.
 * bytes must not exceed the buffer size (nf_plan_buffer_size). */
typedef enum {
  NF_BUF_TOK_SEQ = 0,   /* int32 [T] */
  NF_BUF_TOK_POS = 1,   /* int32 [T] */
  NF_BUF_TOK_SLOT = 2,  /* int32 [T], -1 where the page id was invalid */
  NF_BUF_ITEMS = 3,     /* int32 [2 * capacity]: (row, chunk) pairs of the work
                           list, nano-batch segments back to back */
  NF_BUF_ITEM_SEG = 4,  /* int32 [n_attn + 1]: start of each segment in ITEMS;
                           the last entry is the total */
  NF_BUF_N1 = 5,        /* bf16 [T, H] */
  NF_BUF_Q = 6,         /* bf16 [T, n_q * head_dim] */
  NF_BUF_O = 7,         /* bf16 [T, n_q * head_dim] */
  NF_BUF_H = 8,         /* bf16 [T, H] */
  NF_BUF_N2 = 9,        /* bf16 [T, H] */
  NF_BUF_A = 10,        /* bf16 [T, F] */
  /* mixture of experts, for the last FFN nano-batch of the last step (rows
   * of the grouped order are counted from that nano-batch's first token): */
  NF_BUF_MOE_OFF = 11,      /* int32 [E + 1]: first grouped row of each expert */
  NF_BUF_MOE_PERM = 12,     /* int32 [T * top_k]: token of each grouped row */
  NF_BUF_MOE_PAIR_ROW = 13, /* int32 [T * top_k]: grouped row of pair (token, choice) */
  NF_BUF_MOE_PAIR_W = 14    /* fp32 [T * top_k]: routing weight of pair (token, choice) */
} nf_buffer;
nf_status nf_plan_buffer_size(nf_plan plan, int32_t which, size_t* bytes);
nf_status nf_plan_copy_buffer(nf_plan plan, int32_t which, void* dst, size_t bytes);

/* Tracing: CUDA-event timestamps of every nano-operation of a step, taken on
 * the stream each one is launched on (the pages' per-microsecond utilisation
 * timelines, "NanoFlow: Towards Optimal LLM Serving Throughput", evaluation of
 * resource usage).  nf_plan_trace_enable(plan, max_steps) starts recording the
 * next max_steps steps (0 stops and drops the record).  nf_plan_trace_read
 * synchronizes the plan's streams and returns one entry per nano-operation
 * per recorded step: op (NF_OP_*), nano-batch index, step index, start time
 * relative to that step's start and duration, both in milliseconds. */
typedef enum { NF_OP_META = 0, NF_OP_QKV = 1, NF_OP_ATTN = 2, NF_OP_OPROJ = 3, NF_OP_FFN = 4 } nf_op;
typedef struct {
  int32_t op;
  int32_t nano;
  int32_t step;
  float start_ms;
  float ms;
} nf_trace_entry;
nf_status nf_plan_trace_enable(nf_plan plan, int32_t max_steps);
/* Which operations the trace records: bit NF_OP_x of op_mask (default: all).
 * Each recorded operation adds a CUDA event before and after it on its
 * stream, and an event between two kernels keeps the second from starting as
 * a programmatic dependent of the first; recording only what is measured
 * (e.g. 1 << NF_OP_ATTN) leaves the rest of the step as it runs untraced. */
nf_status nf_plan_trace_ops(nf_plan plan, uint32_t op_mask);
nf_status nf_plan_trace_read(nf_plan plan, nf_trace_entry* out, int32_t cap, int32_t* n_out);

/* ---------------------------------------------------------------------------
 * Profiler and plan search ("NanoFlow: Towards Optimal LLM Serving
 * Throughput", "Kernel Profiling and Interference Modeling", "Auto-Search
 * Stage I/II").
 */

/* Measure, on the current device, the interference-free time of each
 * operation of the layer at token counts that are multiples of 128 (up to
 * max_tokens) and SM counts, and the time of attention when it shares the GPU
 * with a GEMM at several SM splits; write them to out_json.  Allocates and
 * frees its own buffers; takes seconds to minutes. */
nf_status nf_profile(const nf_model_shape* shape, int32_t max_tokens, int32_t mean_ctx,
                     const char* out_json);

/* Measure the R -> P table inside the step itself ("Kernel Profiling and
 * Interference Modeling": the performance P a kernel keeps for a resource
 * share R): run this batch structure (seq_lens_hint required, synthetic
 * weights and K/V) through min(n_layers, 32) layers under the sequential plan
 * and under two-stream plans of 2, 3 and 4 nano-batches with attention on
 * 3/16 ... 10/16 of the SMs (the cross-layer window when n_layers > 1), tracing
 * every nano-operation; fit the search's rates to what ran (the GEMM tensor
 * rate and attention bandwidth alone; per nano-batch count and attention SM
 * count the attention's bytes/s per SM and the share of its rate a GEMM kept
 * while the two overlapped; the cost of a cross-stream dependency and one
 * factor on the GEMM shares, from the untraced step times; the sequential plan
 * and the three fastest overlapped plans are timed again, interleaved over
 * three rounds, and keep the median); write them with each plan's measured
 * and predicted step time to out_json, and register the file for this shape
 * (nf_profile_use), so that plan creation without options and the searches
 * below use it.  Allocates its own buffers (weights of one layer, one K/V pool
 * of batch->num_pages pages); takes seconds. */
nf_status nf_profile_step(const nf_model_shape* shape, const nf_batch_desc* batch,
                          int32_t n_layers, const char* out_json);

/* Register a profile (JSON written by nf_profile_step or nf_profile) for this
 * shape in this process; json_path NULL forgets it.  The path is read when a
 * search runs. */
nf_status nf_profile_use(const nf_model_shape* shape, const char* json_path);

/* Plan search on the host only (no device work): given a profile table
 * (a JSON path; NULL for the profile registered for the shape, else the
 * built-in rates; "" for the built-in rates), pick the split and SM shares that
 * minimise the predicted step time.  Fills `out` and the predicted time in
 * microseconds.  nf_plan_create with opts NULL runs it with NULL. */
nf_status nf_plan_search(const nf_model_shape* shape, const nf_batch_desc* batch,
                         const char* profile_json, int32_t num_sms, nf_plan_opts* out,
                         double* predicted_us);

/* The same for a step of n_layers layers run by nf_layers_step or
 * nf_stack_step, whose two-stream plans pipeline nano-batches across layers
 * (the pages search a window of neighbouring layers): candidates are the
 * sequential plan and cross-layer plans of 2-4 attention nano-batches (equal
 * FFN splits, or 2 FFN nano-batches under 4) with the attention share on a
 * 1/64 grid, each scored by simulating the two streams over all the layers.
 * The predicted time is that of all n_layers layers.  n_layers = 1 is
 * nf_plan_search; NF_ERR_INVALID_ARG for n_layers < 1. */
nf_status nf_plan_search_layers(const nf_model_shape* shape, const nf_batch_desc* batch,
                                const char* profile_json, int32_t num_sms, int32_t n_layers,
                                nf_plan_opts* out, double* predicted_us);

/* The time the search's model predicts for a given plan over n_layers layers
 * (the cross-layer window for a two-stream plan of >= 2 attention nano-batches
 * when n_layers > 1), in microseconds: for comparing the model with measured
 * plans.  NF_ERR_INVALID_ARG when the plan's bounds do not describe the batch. */
nf_status nf_plan_predict(const nf_model_shape* shape, const nf_batch_desc* batch,
                          const char* profile_json, int32_t num_sms, int32_t n_layers,
                          const nf_plan_opts* plan, double* predicted_us);

/* The order in which the two-stream executor issues the nano-operations of
 * n_layers layers under the cross-layer window (host only; the executor and
 * the search's simulation both follow it).  Operations in the order of the
 * GEMM stream, 4 int32 each in out[]: kind (0 QKV projection, followed on the
 * attention stream by that nano-batch's attention; 1 O projection, which waits
 * for it; 2 FFN nano-batch), layer, nano-batch index, and 1 where the
 * operation overlaps nothing and gets every SM.  Writes at most cap
 * operations and the total count to *n_ops.  NF_ERR_INVALID_ARG when the
 * plan's bounds are not increasing from 0 to one common end. */
nf_status nf_window_schedule(const nf_plan_opts* plan, int32_t n_layers, int32_t* out, int32_t cap,
                             int32_t* n_ops);

/* ---------------------------------------------------------------------------
 * Runtime around the step ("NanoFlow: Towards Optimal LLM Serving Throughput",
 * "The NanoFlow Runtime System"): requests in, greedy tokens out.
 *
 * Batch formation keeps a constant token budget b_dense per iteration: every
 * decoding request gets one token first, then prompts are cut into chunks,
 * first come first served, that fill the rest.  nf_runtime_step forms the next
 * iteration and enqueues it (token composition from each request's previous
 * output kept on the device, the stack step, argmax sampling, an asynchronous
 * copy of the sampled tokens) without waiting for the GPU; the tokens of an
 * iteration are taken in when the iteration two later is formed, so a request
 * that produced eos_token runs one more (wasted) iteration, as in the pages.
 * KV pages of every layer share one page allocator of num_pages pages; a
 * finished request returns its pages and its token slot.  The plan follows
 * each batch (nf_plan_set_batch); the plan search runs again when the decode
 * share of the batch moved by more than replan_threshold since the last search
 * or the token count changed (the pages' pipeline is static; this re-plans it
 * online). */
typedef struct nf_runtime_s* nf_runtime;
typedef struct {
  int32_t b_dense;            /* tokens per iteration */
  int32_t max_requests;       /* requests admitted at once (device token slots) */
  int32_t max_pages_per_seq;  /* block-table width: longest prompt + output */
  int32_t num_pages;          /* pages in each layer's K and V pools */
  int32_t vocab;              /* the LM head's rows, a multiple of 8 */
  int32_t eos_token;          /* -1: requests end after max_new_tokens only */
  float replan_threshold;     /* < 0: never re-plan (one sequential nano-batch) */
  int32_t host_only;          /* 1: no device resources; batches are formed with
                                 nf_runtime_form and results given with
                                 nf_runtime_apply (the scheduler alone) */
} nf_runtime_opts;

/* One iteration's batch as formed (arrays owned by the runtime, valid until the
 * same iteration slot is formed again, two iterations later).  Rows: decode
 * sequences first (one row each), then the prompt chunks. */
typedef struct {
  int32_t iteration;
  int32_t n_tokens;
  int32_t n_decode;               /* decode sequences (= decode rows) */
  int32_t n_prefill;              /* prompt chunks */
  const int32_t* row_request;     /* [n_tokens] request id */
  const int32_t* row_pos;         /* [n_tokens] position in the request's sequence */
  const int32_t* row_token;       /* [n_tokens] prompt token, or -1: the request's last output */
  const int32_t* row_emit;        /* [n_tokens] 1 where the row's output is the request's next token */
  const int32_t* seq_lens;        /* [n_decode + n_prefill] KV length after the step */
  const int32_t* block_table;     /* [n_decode + n_prefill][max_pages_per_seq], -1 past the end */
  const int32_t* prefill_q_lens;  /* [n_prefill] */
  int32_t replanned;              /* the plan search ran for this batch */
  int32_t free_pages;             /* pages left after forming it */
} nf_runtime_batch;

nf_status nf_runtime_create(const nf_model_shape* shape, const nf_runtime_opts* opts,
                            nf_runtime* out);
/* Waits for the iterations in flight, then frees everything. */
void nf_runtime_destroy(nf_runtime rt);
/* A request: prompt tokens (host, copied), at most max_new_tokens outputs. */
nf_status nf_runtime_submit(nf_runtime rt, const int32_t* prompt, int32_t prompt_len,
                            int32_t max_new_tokens, int32_t* id);
/* Form and enqueue the next iteration on `stream` (see above).  A batch of 0
 * tokens means nothing could run (all requests finished). */
nf_status nf_runtime_step(nf_runtime rt, const nf_stack_weights* w, void* const* k_pools,
                          void* const* v_pools, void* stream, nf_runtime_batch* out);
/* Wait for the iterations in flight and take in their tokens. */
nf_status nf_runtime_sync(nf_runtime rt);
/* A request's outputs so far (tokens: host, up to cap). */
nf_status nf_runtime_result(nf_runtime rt, int32_t id, int32_t* finished, int32_t* n_tokens,
                            int32_t* tokens, int32_t cap);
nf_status nf_runtime_counts(nf_runtime rt, int32_t* waiting, int32_t* active, int32_t* free_pages);
/* The logits of the last iteration that nf_runtime_step launched, for its
 * emitting rows in row order: dst [n_rows, vocab] bf16, host or device (e.g. to
 * check a model against a reference, or to sample differently).  Waits for that
 * iteration's stream; the buffer is overwritten by the next step.  With dst
 * NULL only n_rows is set.  cap_rows: rows dst holds. */
nf_status nf_runtime_logits(nf_runtime rt, void* dst, int32_t cap_rows, int32_t* n_rows);
/* Host-only runtimes: form the next batch / give the sampled tokens of an
 * iteration ([n_tokens], read where row_emit is 1).  At most two iterations
 * may await results. */
nf_status nf_runtime_form(nf_runtime rt, nf_runtime_batch* out);
nf_status nf_runtime_apply(nf_runtime rt, int32_t iteration, const int32_t* sampled);

#ifdef __cplusplus
}
#endif
#endif /* NANOFLOW_H */
