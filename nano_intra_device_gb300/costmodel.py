"""Cost model of the layer step: algorithmic FLOPs and bytes, roofline time.

The pages' cost model ("NanoFlow: Towards Optimal LLM Serving Throughput",
"The Cost Model and the Compute-Bound Classification") bounds an iteration by
its compute time 2 * B_dense * P_model / Compute and its memory time; Eq. 4
(TR = T_mem / T_compute) says which bound binds, and Eq. 5 gives the optimal
throughput Compute / (2 * P_model).  This module states the same quantities
for ONE decoder-layer step over a concrete mixed batch, counting what the step
must move at least once:

* FLOPs: 2 * T * P_layer for the projections and FFN (for a mixture of
  experts, top_k experts per token), plus the attention products (2 FLOPs per
  multiply-add, QK^T and PV, per query head and visible position);
* bytes: bf16 weights once (every expert of a mixture: a step of thousands of
  tokens hits them all), the KV each sequence reads (its whole visible
  history, including this step's tokens), the K/V appended, x in and y out.

Nano-batch weight re-reads are not counted: they are the cost of the method,
not algorithmic work.  The KV-size formula is the one of "LLM Inference
Performance", KV cache sizing: 2 * n_layers * n_kv_heads * head_dim * bytes.
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """K and V bytes one token occupies across all layers."""
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes


def optimal_throughput(compute_flops: float, params: float) -> float:
    """Eq. 5: tokens/s when compute is fully busy = Compute / (2 * P_model)."""
    return compute_flops / (2.0 * params)


def compute_time(b_dense: float, params: float, compute_flops: float) -> float:
    """T_compute ~= 2 * B_dense * P_model / Compute."""
    return 2.0 * b_dense * params / compute_flops


def memory_time(mem_bytes: float, mem_bw: float) -> float:
    """T_mem = MemSize / MemBW."""
    return mem_bytes / mem_bw


def transfer_ratio(mem_bytes: float, mem_bw: float, b_dense: float, params: float,
                   compute_flops: float) -> float:
    """Eq. 4: TR = T_mem / T_compute (> 1 memory-bound, < 1 compute-bound)."""
    return memory_time(mem_bytes, mem_bw) / compute_time(b_dense, params, compute_flops)


def effective_intensity(batch: float, params: float, kv_bytes_per_seq: float) -> float:
    """FLOP per byte of a decode step that streams weights once and every
    sequence's KV: B * 2P / (2P + B * kv_bytes) ("LLM Inference Performance",
    batching moves decode up the roofline)."""
    return batch * 2.0 * params / (2.0 * params + batch * kv_bytes_per_seq)


def layer_params(shape) -> int:
    """Weights of one layer's projections and FFN (norm gains excluded); a
    mixture-of-experts layer counts every expert."""
    H, d, F = shape.hidden, shape.head_dim, shape.ffn
    experts = max(1, getattr(shape, "n_experts", 0))
    return H * (shape.n_q + 2 * shape.n_kv) * d + shape.n_q * d * H + experts * 3 * H * F


def active_params(shape) -> int:
    """Weights one token multiplies: the projections and, for a mixture of
    experts, top_k experts' FFNs."""
    H, d, F = shape.hidden, shape.head_dim, shape.ffn
    k = getattr(shape, "top_k", 1) if getattr(shape, "n_experts", 0) else 1
    return H * (shape.n_q + 2 * shape.n_kv) * d + shape.n_q * d * H + k * 3 * H * F


def step_work(shape, seq_lens, q_lens, elem_bytes: int = 2) -> dict:
    """Algorithmic FLOPs and bytes of one layer step over the batch."""
    seq_lens = np.asarray(seq_lens, np.int64)
    q_lens = np.asarray(q_lens, np.int64)
    T = int(q_lens.sum())
    d, nq, nkv, H = shape.head_dim, shape.n_q, shape.n_kv, shape.hidden
    P = layer_params(shape)
    # visible positions summed over the step's tokens: a token at position p sees p+1
    vis = 0
    for L, q in zip(seq_lens.tolist(), q_lens.tolist()):
        first = L - q + 1
        vis += (first + L) * q // 2 if q > 0 else 0
    gemm_flops = 2 * T * active_params(shape)
    attn_flops = 4 * nq * d * vis
    kv_tok = 2 * nkv * d * elem_bytes
    bytes_w = P * elem_bytes
    bytes_kv_read = int(seq_lens.sum()) * kv_tok
    bytes_kv_write = T * kv_tok
    bytes_act = 2 * T * H * elem_bytes
    return {
        "tokens": T,
        "gemm_flops": gemm_flops,
        "attn_flops": attn_flops,
        "flops": gemm_flops + attn_flops,
        "weight_bytes": bytes_w,
        "kv_read_bytes": bytes_kv_read,
        "kv_write_bytes": bytes_kv_write,
        "act_bytes": bytes_act,
        "bytes": bytes_w + bytes_kv_read + bytes_kv_write + bytes_act,
    }


def roofline_time(work: dict, peak_flops: float, peak_bw: float) -> dict:
    """t_roof = max(FLOPs / peak_flops, bytes / peak_bw) and which binds."""
    t_f = work["flops"] / peak_flops
    t_b = work["bytes"] / peak_bw
    return {"t_flop": t_f, "t_byte": t_b, "t_roof": max(t_f, t_b),
            "bound": "tensor" if t_f >= t_b else "hbm"}


def decode_attention_bytes(shape, seq_lens, q_lens, elem_bytes: int = 2) -> int:
    """Bytes the decode-attention kernel must move: every decode row's KV
    history once (K and V, all KV heads), its q in and o out."""
    seq_lens = np.asarray(seq_lens, np.int64)
    q_lens = np.asarray(q_lens, np.int64)
    dec = q_lens == 1
    kv_tok = 2 * shape.n_kv * shape.head_dim * elem_bytes
    n = int(dec.sum())
    return int(seq_lens[dec].sum()) * kv_tok + 2 * n * shape.n_q * shape.head_dim * elem_bytes


def stack_work(shape, seq_lens, q_lens, n_layers: int, vocab: int, elem_bytes: int = 2) -> dict:
    """Algorithmic work of a stack step: n_layers layer steps (each reads its own
    K/V and weights once), the embedding rows gathered, the final norm and the
    LM head (its weights read once, 2*T*H*vocab FLOPs)."""
    lw = step_work(shape, seq_lens, q_lens, elem_bytes)
    T = lw["tokens"]
    H = shape.hidden
    head_flops = 2 * T * H * vocab
    head_bytes = vocab * H * elem_bytes + T * vocab * elem_bytes
    flops = n_layers * lw["flops"] + head_flops
    # per layer: weights + K/V once; activations stay on chip or in L2 between kernels
    per_layer_bytes = lw["weight_bytes"] + lw["kv_read_bytes"] + lw["kv_write_bytes"]
    byts = n_layers * per_layer_bytes + head_bytes + T * H * elem_bytes
    return {"tokens": T, "flops": flops, "bytes": byts, "layer": lw}
