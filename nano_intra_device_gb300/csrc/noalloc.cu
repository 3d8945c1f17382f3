// Paged attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a host runtime that
// owns every byte of device memory through its own pool and hands a custom
// operator nothing but input and output pointers, or a latency-critical loop
// that cannot afford the implicit device synchronisation an allocation may
// cause.  nf_attention needs a plan, and a plan allocates its workspace.  This
// file gives those callers the same attention through nf_attention_noalloc,
// whose working memory (token map, work list, counters, split-KV partials) is
// one file-scope device array of fixed size, set aside when the library's
// device code is loaded and held by every GPU that loads it until the process
// exits.  A small kernel writes the batch structure (passed by value) into
// that array; then the metadata kernel and the tensor-core attention kernel of
// nf_attention run on it.  Device-side checks (page ids, lengths, bounded
// waits) OR their bits into a status word at the start of the array, which
// stays set until nf_attention_noalloc_poll reads and clears it.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <vector>

#include "../../include/nanoflow.h"
#include "common.cuh"
#include "internal.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = NF_NOALLOC_SCRATCH_BYTES;
constexpr int kChunk = 2048;  // split-KV piece of this entry point (fewest partial records)
constexpr int kMaxDevices = 64;
constexpr int kMaxPrefill = NF_NOALLOC_MAX_PREFILL;
constexpr size_t kStatusOff = 0;    // the status word: first 256 bytes, never moved
constexpr size_t kCarveBegin = 256; // per-call regions start here

// The working memory.  Host code never dereferences this name: on the host it
// is only a stand-in for the symbol, whose device address comes from
// cudaGetSymbolAddress below.  Zero when the module loads, so the status word
// starts clear.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
nf_status scratch_address(void** out, const char* who) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    char msg[128];
    std::snprintf(msg, sizeof(msg), "%s: no usable current device", who);
    return nf::set_last_error(NF_ERR_CUDA, msg);
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      std::snprintf(msg, sizeof(msg), "%s: cudaGetSymbolAddress failed: %s", who,
                    cudaGetErrorString(e));
      return nf::set_last_error(NF_ERR_CUDA, msg);
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return NF_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The batch structure, passed by value: decode sequences own one token each,
// prefill chunk j owns tokens n_decode + pf_begin[j] ... n_decode + pf_begin[j+1] - 1.
struct FillArgs {
  int n_decode, n_seq, T;
  int pf_begin[kMaxPrefill + 1];
};

// Writes the metadata kernel's inputs (q_lens, token starts, the one segment's
// bounds) into the working memory, so no host table is copied.
__global__ void noalloc_fill_kernel(const FillArgs f, int* q_lens, int* tok_begin, int* seg_bounds) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= f.n_seq; i += gridDim.x * blockDim.x) {
    const int j = i - f.n_decode;
    tok_begin[i] = j <= 0 ? i : f.n_decode + f.pf_begin[j];
    if (i < f.n_seq) q_lens[i] = j < 0 ? 1 : f.pf_begin[j + 1] - f.pf_begin[j];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    seg_bounds[0] = 0;
    seg_bounds[1] = f.T;
  }
}

}  // namespace

extern "C" nf_status nf_attention_noalloc(const nf_model_shape* shape, const nf_batch_desc* batch,
                                          const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* block_table, const int32_t* seq_lens,
                                          void* o, void* stream) {
  if (!shape || !batch || !q || !k_pool || !v_pool || !block_table || !seq_lens || !o)
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: NULL argument");
  const nf_model_shape& s = *shape;
  if ((s.head_dim != 64 && s.head_dim != 128) || s.n_kv_heads <= 0 || s.n_q_heads <= 0 ||
      s.n_q_heads % s.n_kv_heads || s.page_size != 16)
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: unsupported shape");
  const int grp = s.n_q_heads / s.n_kv_heads;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 8)
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: n_q/n_kv must be 1, 2, 4 or 8");
  if (!nf::attention_mma_supported(s.n_q_heads, s.n_kv_heads, s.head_dim, s.page_size,
                                   batch->num_pages > 0 ? batch->num_pages : 1))
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: the pool is too large");
  if (batch->n_decode < 0 || batch->n_prefill < 0 || batch->n_decode + batch->n_prefill < 1 ||
      (batch->n_prefill > 0 && !batch->prefill_q_lens) || batch->max_pages_per_seq < 1 ||
      batch->num_pages < 1)
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: invalid batch");
  if (batch->n_prefill > kMaxPrefill) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "nf_attention_noalloc: at most %d prefill chunks (got %d)",
                  kMaxPrefill, batch->n_prefill);
    return nf::set_last_error(NF_ERR_INVALID_ARG, msg);
  }
  for (const void* p : {q, k_pool, v_pool, (const void*)o})
    if (reinterpret_cast<uintptr_t>(p) & 15)
      return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: tensors must be 16-byte aligned");

  // the batch structure, by value
  FillArgs f{};
  f.n_decode = batch->n_decode;
  f.n_seq = batch->n_decode + batch->n_prefill;
  long long T_ll = batch->n_decode;
  for (int j = 0; j < batch->n_prefill; ++j) {
    const int ql = batch->prefill_q_lens[j];
    if (ql < 1)
      return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: prefill_q_lens must be >= 1");
    f.pf_begin[j] = static_cast<int>(T_ll - batch->n_decode);
    T_ll += ql;
    if (T_ll > (1 << 24))
      return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: too many tokens");
  }
  f.pf_begin[batch->n_prefill] = static_cast<int>(T_ll - batch->n_decode);
  const int n_seq = f.n_seq;
  const int T = f.T = static_cast<int>(T_ll);
  const int max_chunks = (batch->max_pages_per_seq * s.page_size + kChunk - 1) / kChunk;

  // carve the fixed array (after the status word)
  const size_t rec = nf::attn_partial_floats(s.n_q_heads, s.n_kv_heads, s.head_dim);
  size_t off = kCarveBegin;
  auto take = [&](size_t bytes) { const size_t at = off; off = align256(off + bytes); return at; };
  const size_t o_qlens = take((size_t)n_seq * 4), o_begin = take((size_t)(n_seq + 1) * 4);
  const size_t o_segb = take(8), o_seq = take((size_t)T * 4), o_pos = take((size_t)T * 4);
  const size_t o_slot = take((size_t)T * 4), o_nch = take((size_t)T * 4);
  const size_t o_items = take((size_t)T * max_chunks * 8), o_segi = take(8), o_fetch = take(4);
  const size_t o_done = take((size_t)T * s.n_kv_heads * 4);
  const size_t o_part = take((size_t)T * max_chunks * s.n_kv_heads * rec * 4);
  if (off > kScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "nf_attention_noalloc: this batch needs %zu bytes of working memory, more than "
                  "the fixed %zu; use nf_attention with a plan",
                  off, kScratchBytes);
    return nf::set_last_error(NF_ERR_INVALID_ARG, msg);
  }
  void* base_v = nullptr;
  nf_status st = scratch_address(&base_v, "nf_attention_noalloc");
  if (st != NF_OK) return st;
  unsigned char* base = static_cast<unsigned char*>(base_v);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: cannot read the SM count");

  nf::MetaArgs m{};
  m.q_lens = reinterpret_cast<const int*>(base + o_qlens);
  m.tok_begin = reinterpret_cast<const int*>(base + o_begin);
  m.seg_bounds = reinterpret_cast<const int*>(base + o_segb);
  {
    const int grid = std::min(64, (n_seq + 1 + 255) / 256);
    noalloc_fill_kernel<<<grid, 256, 0, cs>>>(f, const_cast<int*>(m.q_lens),
                                              const_cast<int*>(m.tok_begin),
                                              const_cast<int*>(m.seg_bounds));
    if (cudaGetLastError() != cudaSuccess)
      return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: launch failed");
  }
  m.seq_lens = seq_lens;
  m.block_table = block_table;
  m.n_seq = n_seq;
  m.n_tok = T;
  m.n_seg = 1;
  m.max_pages = batch->max_pages_per_seq;
  m.num_pages = batch->num_pages;
  m.page_size = s.page_size;
  m.kv_chunk = kChunk;
  m.n_kv = s.n_kv_heads;
  m.max_chunks = max_chunks;
  m.item_capacity = T * max_chunks;
  m.tok_seq = reinterpret_cast<int*>(base + o_seq);
  m.tok_pos = reinterpret_cast<int*>(base + o_pos);
  m.tok_slot = reinterpret_cast<int*>(base + o_slot);
  m.tok_nchunks = reinterpret_cast<int*>(base + o_nch);
  m.items = reinterpret_cast<int*>(base + o_items);
  m.seg_items = reinterpret_cast<int*>(base + o_segi);
  m.fetch = reinterpret_cast<int*>(base + o_fetch);     // zeroed by the metadata kernel
  m.row_done = reinterpret_cast<int*>(base + o_done);   // zeroed by the metadata kernel
  m.counter_sets = 1;
  m.fetch_stride = 1;
  m.status = reinterpret_cast<uint32_t*>(base + kStatusOff);  // sticky until polled
  m.validate = 1;  // every page id a token reads is checked against num_pages
  if (nf::launch_meta(m, cs) != cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: metadata launch failed");

  nf::AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
  a.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.block_table = block_table;
  a.tok_seq = m.tok_seq;
  a.tok_pos = m.tok_pos;
  a.tok_nchunks = m.tok_nchunks;
  a.items = m.items;
  a.seg_items = m.seg_items;
  a.fetch = m.fetch;
  a.row_done = m.row_done;
  a.partials = reinterpret_cast<float*>(base + o_part);
  a.seg = 0;
  a.n_q = s.n_q_heads;
  a.n_kv = s.n_kv_heads;
  a.head_dim = s.head_dim;
  a.page_size = s.page_size;
  a.max_pages = batch->max_pages_per_seq;
  a.num_pages = batch->num_pages;
  a.kv_chunk = kChunk;
  a.max_chunks = max_chunks;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.head_dim));
  a.warps = 8;
  a.prefill_elsewhere = 0;  // prefill rows too go through the decode kernel, row by row
  a.n_decode_seqs = batch->n_decode;
  a.status = m.status;
  a.timeout_ns = 2000000000ull;
  // tensor maps over the pools: host-side descriptors, passed by value
  CUtensorMap tk, tv;
  if (!nf::make_pool_tmap_pages(&tk, k_pool, batch->num_pages, s.n_kv_heads, s.page_size,
                                s.head_dim) ||
      !nf::make_pool_tmap_pages(&tv, v_pool, batch->num_pages, s.n_kv_heads, s.page_size,
                                s.head_dim))
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: KV pool tensor maps failed");
  if (nf::launch_attention_mma(a, tk, tv, sms, false, cs) != cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: attention launch failed");
  return NF_OK;
}

extern "C" nf_status nf_attention_noalloc_poll(void* stream) {
  void* base = nullptr;
  nf_status st = scratch_address(&base, "nf_attention_noalloc_poll");
  if (st != NF_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc_poll: the stream reported an error");
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, static_cast<unsigned char*>(base) + kStatusOff, 4, cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc_poll: cannot read the status word");
  if (!bits) return NF_OK;
  if (cudaMemset(static_cast<unsigned char*>(base) + kStatusOff, 0, 4) != cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc_poll: cannot clear the status word");
  char msg[200];
  std::snprintf(msg, sizeof(msg), "nf_attention_noalloc: device-side check failed (status 0x%x:%s%s%s%s)",
                bits, (bits & nf::ST_TIMEOUT) ? " a wait timed out" : "",
                (bits & nf::ST_BAD_PAGE) ? " page id out of range" : "",
                (bits & nf::ST_BAD_LEN) ? " bad sequence length" : "",
                (bits & nf::ST_OVERFLOW) ? " work list overflow" : "");
  return nf::set_last_error((bits & nf::ST_TIMEOUT) ? NF_ERR_TIMEOUT : NF_ERR_DEVICE, msg);
}
