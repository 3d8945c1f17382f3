// Where one token of a step sits: its sequence, position, cache slot and
// split-KV piece count.  Used by the step-metadata kernel and by RMSNorm-1,
// which maps the tokens of its rows while it normalises them.
//
// Sequence s owns q_lens[s] consecutive tokens of the step, at positions
// seq_lens[s] - q_lens[s] ... seq_lens[s] - 1; the token's new K/V goes to
// slot block_table[s][pos / P] * P + pos % P ("Inside nano-vLLM", 4.2 Paged
// KV: the block table and the slot mapping of new KV writes).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace nf {

// largest i in [lo, hi) with tb[i] <= t (tb ascending, tb[lo] <= t)
__device__ __forceinline__ int tok_seq_search(const int* tb, int lo, int hi, int t) {
  hi -= 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct TokEntry {
  int pos, slot, nch;
};

// Token t of sequence s (tb_s = the sequence's first token).  full: also the
// cache slot and, with m.validate, every page the token's attention reads;
// otherwise slot is -1 and no page is read.  Inconsistent lengths give
// position 0 and no context; a bad page id gives slot -1; both set status bits.
__device__ __forceinline__ TokEntry token_entry(const TokMap& m, int s, int tb_s, int t,
                                                bool full) {
  const int P = m.page_size, C = m.kv_chunk;
  const int L = m.seq_lens[s], q = m.q_lens[s];
  TokEntry e;
  e.pos = L - q + (t - tb_s);
  e.slot = -1;
  bool ok = true;
  if (q < 1 || L < q || e.pos >= m.max_pages * P) {
    raise_status(m.status, ST_BAD_LEN);
    ok = false;
    e.pos = 0;
  }
  if (ok && full) {
    const int* row = m.block_table + static_cast<size_t>(s) * m.max_pages;
    const int page = row[e.pos / P];
    if (page >= 0 && page < m.num_pages) {
      e.slot = page * P + e.pos % P;
    } else {
      raise_status(m.status, ST_BAD_PAGE);
    }
    if (m.validate) {  // every page the token's attention will read
      for (int j = 0; j <= e.pos / P; ++j) {
        const int pg = row[j];
        if (pg < 0 || pg >= m.num_pages) {
          raise_status(m.status, ST_BAD_PAGE);
          break;
        }
      }
    }
  }
  const int ctx = ok ? e.pos + 1 : 0;
  e.nch = (ctx + C - 1) / C;
  if (e.nch > m.max_chunks) {
    raise_status(m.status, ST_OVERFLOW);
    e.nch = m.max_chunks;
  }
  return e;
}

}  // namespace nf
