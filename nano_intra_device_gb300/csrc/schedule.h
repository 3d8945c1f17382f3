// The order of nano-operations of the cross-layer window, shared by the
// executor (api.cu, run_layers_pipelined) and the plan search's simulation
// (search.cpp, simulate_window), so that the search scores the schedule that
// runs.  Host code only.
//
// The GEMM stream runs the listed operations in order; a QKV entry is
// followed on the attention stream by the attention of the same nano-batch
// (waiting for that QKV), and an O entry waits for that attention.  Order:
//   QKV(0, 0 .. n-1); then for each layer l and attention nano-batch i:
//   O(l, i), the FFN nano-batches of layer l whose rows that O completes,
//   and after each FFN the QKV of layer l + 1's nano-batches whose rows are
//   now complete.
// full = 1 marks the operations that nothing overlaps (the first QKV and what
// follows the last attention), which get every SM.
#pragma once
#include <vector>

#include "../../include/nanoflow.h"

namespace nf {

enum WindowOpKind : int { WOP_QKV = 0, WOP_O = 1, WOP_FFN = 2 };

struct WindowOp {
  int kind, layer, nano, full;
};

inline std::vector<WindowOp> window_schedule(const nf_plan_opts& o, int n_layers) {
  std::vector<WindowOp> ops;
  const int n = o.n_attn;
  for (int i = 0; i < n; ++i) ops.push_back({WOP_QKV, 0, i, i == 0 ? 1 : 0});
  for (int l = 0; l < n_layers; ++l) {
    int next_ffn = 0, next_front = 0;
    for (int i = 0; i < n; ++i) {
      const int full = (l == n_layers - 1 && i == n - 1) ? 1 : 0;
      ops.push_back({WOP_O, l, i, full});
      while (next_ffn < o.n_ffn && o.ffn_bounds[next_ffn + 1] <= o.attn_bounds[i + 1]) {
        ops.push_back({WOP_FFN, l, next_ffn, full});
        ++next_ffn;
        while (l + 1 < n_layers && next_front < n &&
               o.attn_bounds[next_front + 1] <= o.ffn_bounds[next_ffn]) {
          ops.push_back({WOP_QKV, l + 1, next_front, 0});
          ++next_front;
        }
      }
    }
  }
  return ops;
}

}  // namespace nf
