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
// exits.  It runs the same metadata and attention kernels as nf_attention.
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

// The working memory.  Host code never dereferences this name: on the host it
// is only a stand-in for the symbol, whose device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
nf_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: no usable current device");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      std::snprintf(msg, sizeof(msg), "nf_attention_noalloc: cudaGetSymbolAddress failed: %s",
                    cudaGetErrorString(e));
      return nf::set_last_error(NF_ERR_CUDA, msg);
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return NF_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

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
  if (batch->n_decode < 0 || batch->n_prefill < 0 || batch->n_decode + batch->n_prefill < 1 ||
      (batch->n_prefill > 0 && !batch->prefill_q_lens) || batch->max_pages_per_seq < 1 ||
      batch->num_pages < 1)
    return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: invalid batch");
  for (const void* p : {q, k_pool, v_pool, (const void*)o})
    if (reinterpret_cast<uintptr_t>(p) & 15)
      return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: tensors must be 16-byte aligned");

  // host-side token map inputs
  const int n_seq = batch->n_decode + batch->n_prefill;
  std::vector<int32_t> q_lens(n_seq), tok_begin(n_seq + 1, 0);
  for (int i = 0; i < n_seq; ++i) {
    q_lens[i] = i < batch->n_decode ? 1 : batch->prefill_q_lens[i - batch->n_decode];
    if (q_lens[i] < 1) return nf::set_last_error(NF_ERR_INVALID_ARG, "nf_attention_noalloc: prefill_q_lens must be >= 1");
    tok_begin[i + 1] = tok_begin[i] + q_lens[i];
  }
  const int T = tok_begin[n_seq];
  const int32_t seg_bounds[2] = {0, T};
  const int max_chunks = (batch->max_pages_per_seq * s.page_size + kChunk - 1) / kChunk;

  // carve the fixed array
  const size_t rec = nf::attn_partial_floats(s.n_q_heads, s.n_kv_heads, s.head_dim);
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t at = off; off = align256(off + bytes); return at; };
  const size_t o_qlens = take((size_t)n_seq * 4), o_begin = take((size_t)(n_seq + 1) * 4);
  const size_t o_segb = take(8), o_seq = take((size_t)T * 4), o_pos = take((size_t)T * 4);
  const size_t o_slot = take((size_t)T * 4), o_nch = take((size_t)T * 4);
  const size_t o_items = take((size_t)T * max_chunks * 8), o_segi = take(8), o_fetch = take(4);
  const size_t o_done = take((size_t)T * s.n_kv_heads * 4), o_status = take(4);
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
  nf_status st = scratch_address(&base_v);
  if (st != NF_OK) return st;
  unsigned char* base = static_cast<unsigned char*>(base_v);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: cannot read the SM count");

  // Inputs of the metadata kernel.  The host vectors may go away on return: a
  // copy from pageable memory is staged before cudaMemcpyAsync returns.
  if (cudaMemcpyAsync(base + o_qlens, q_lens.data(), (size_t)n_seq * 4, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
      cudaMemcpyAsync(base + o_begin, tok_begin.data(), (size_t)(n_seq + 1) * 4, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
      cudaMemcpyAsync(base + o_segb, seg_bounds, 8, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
      cudaMemsetAsync(base + o_status, 0, 4, cs) != cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: copy into the working memory failed");

  nf::MetaArgs m{};
  m.seq_lens = seq_lens;
  m.block_table = block_table;
  m.q_lens = reinterpret_cast<const int*>(base + o_qlens);
  m.tok_begin = reinterpret_cast<const int*>(base + o_begin);
  m.seg_bounds = reinterpret_cast<const int*>(base + o_segb);
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
  m.status = reinterpret_cast<uint32_t*>(base + o_status);
  m.validate = 0;
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
  a.status = m.status;
  a.timeout_ns = 2000000000ull;
  if (nf::launch_attention(a, sms, cs) != cudaSuccess)
    return nf::set_last_error(NF_ERR_CUDA, "nf_attention_noalloc: attention launch failed");
  return NF_OK;
}
