"""Seeded synthetic inputs for the mixed prefill+decode decoder-layer step.

This module draws numbers and lays them out; it holds none of the layer's
arithmetic.  It produces model shapes, weights, activations, per-sequence KV
lengths, block tables and KV-pool contents.  The CUDA path's tests and bench
and the CPU oracle's tests both consume what it returns, so the two sides
always see the same bytes.

Layout conventions fixed here (they are the library's input formats):

* Tokens of a step are ordered decode requests first (one token each), then the
  prefill chunks, each chunk contiguous.  This follows the NanoFlow runtime's
  batch formation ("NanoFlow: Towards Optimal LLM Serving Throughput",
  "The NanoFlow Runtime System", batch formation: decode requests are placed
  first and prefill chunks fill the remaining dense-batch capacity).
* ``seq_lens[s]`` is sequence s's KV length *after* this step's tokens are
  appended; its ``q_lens[s]`` newest positions are produced by this step.
* KV pools are ``[num_pages, n_kv, page_size, head_dim]`` bf16, one pool for K
  and one for V; ``block_table[s, j]`` is the physical page holding logical
  positions ``[j*page_size, (j+1)*page_size)`` of sequence s ("LLM Inference
  Performance", "PagedAttention: virtual memory for the KV cache": fixed
  16-token blocks and a per-sequence block table).
* Pool positions that hold no cached token before the step (pages no sequence
  owns, the tail of each sequence's last page, and the positions this step
  will append) are filled with NaN, so that a read of a wrong position shows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16 = torch.bfloat16


@dataclass(frozen=True)
class Shape:
    """Shape of one Llama-style decoder layer."""

    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    page_size: int = 16
    n_experts: int = 0    # 0: dense SwiGLU FFN; else a mixture of that many SwiGLU experts
    top_k: int = 2        # experts per token when n_experts > 0

    @property
    def qkv_rows(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim


@dataclass
class Batch:
    """One mixed step: ``n_decode`` one-token requests, then prefill chunks."""

    n_decode: int
    prefill_q_lens: list
    seq_lens: np.ndarray          # int32 [n_seq], KV length after the step
    q_lens: np.ndarray            # int32 [n_seq], tokens this step per sequence
    block_table: np.ndarray       # int32 [n_seq, max_pages], -1 = unused entry
    num_pages: int
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_seq(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def n_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def tiny_shape() -> Shape:
    return Shape(hidden=256, n_q=4, n_kv=2, head_dim=64, ffn=688,
                 rms_eps=1e-5, rope_theta=1e4, page_size=16)


def llama8b_shape() -> Shape:
    return Shape(hidden=4096, n_q=32, n_kv=8, head_dim=128, ffn=14336,
                 rms_eps=1e-5, rope_theta=5e5, page_size=16)


def llama70b_shape() -> Shape:
    """LLaMA-2-70B-shaped layer: GQA group of 8, FFN 28672, RoPE theta 1e4."""
    return Shape(hidden=8192, n_q=64, n_kv=8, head_dim=128, ffn=28672,
                 rms_eps=1e-5, rope_theta=1e4, page_size=16)


def _assign_pages(seq_lens, page_size, seed_bt, slack, max_pages=None):
    need = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    total = int(sum(need))
    num_pages = total + int(math.ceil(slack * total))
    perm = np.random.default_rng(seed_bt).permutation(num_pages).astype(np.int32)
    width = max(need) if max_pages is None else max_pages
    width = max(width, 1)
    bt = np.full((len(seq_lens), width), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    return bt, num_pages


def make_batch(shape: Shape, decode_ctx, prefill_q_lens, prefill_prefix=None,
               seed_bt: int = 2, slack: float = 0.0, max_pages=None,
               name: str = "") -> Batch:
    """Build a batch from explicit per-request KV lengths.

    ``decode_ctx[i]`` is decode request i's KV length after the step (its new
    token sits at position ``decode_ctx[i] - 1``).  Prefill chunk j has
    ``prefill_q_lens[j]`` tokens after ``prefill_prefix[j]`` cached ones.
    """
    decode_ctx = [int(c) for c in decode_ctx]
    prefill_q_lens = [int(q) for q in prefill_q_lens]
    if prefill_prefix is None:
        prefill_prefix = [0] * len(prefill_q_lens)
    seq_lens = decode_ctx + [p + q for p, q in zip(prefill_prefix, prefill_q_lens)]
    q_lens = [1] * len(decode_ctx) + prefill_q_lens
    bt, num_pages = _assign_pages(seq_lens, shape.page_size, seed_bt, slack, max_pages)
    return Batch(n_decode=len(decode_ctx), prefill_q_lens=prefill_q_lens,
                 seq_lens=np.asarray(seq_lens, np.int32),
                 q_lens=np.asarray(q_lens, np.int32), block_table=bt,
                 num_pages=num_pages, name=name)


def lognormal_contexts(n: int, median: float, sigma: float, lo: int, hi: int,
                       seed: int = 1) -> np.ndarray:
    """Decode KV lengths: ``clip(round(exp(ln(median) + sigma*z)), lo, hi)``."""
    z = np.random.default_rng(seed).standard_normal(n)
    return np.clip(np.rint(np.exp(math.log(median) + sigma * z)), lo, hi).astype(np.int32)


def tiny_batch() -> Batch:
    """4 decode requests with KV lengths {17,33,48,64} plus one 32-token chunk."""
    return make_batch(tiny_shape(), [17, 33, 48, 64], [32], [0], seed_bt=2,
                      slack=0.0, name="tiny")


def llama8b_batch(n_decode: int = 1792, prefill: int = 256) -> Batch:
    """1792 decode requests (lognormal median 600, sigma 1, clip [1, 8192]) and
    one 256-token prefill chunk starting a prompt; 16-token pages, 1% slack."""
    ctx = lognormal_contexts(n_decode, 600.0, 1.0, 1, 8192, seed=1)
    return make_batch(llama8b_shape(), ctx, [prefill] if prefill else [], None,
                      seed_bt=2, slack=0.01, max_pages=8192 // 16, name="llama8b")


def llama70b_batch(n_decode: int = 3584, prefill: int = 512) -> Batch:
    """3584 decode requests (lognormal median 1000, sigma 1, clip [1, 4096]) and
    one 512-token prefill chunk starting a prompt; 16-token pages, 1% slack."""
    ctx = lognormal_contexts(n_decode, 1000.0, 1.0, 1, 4096, seed=1)
    return make_batch(llama70b_shape(), ctx, [prefill] if prefill else [], None,
                      seed_bt=2, slack=0.01, max_pages=4096 // 16, name="llama70b")


def mixtral_shape() -> Shape:
    """Mixtral-8x7B-shaped layer: Llama-3-8B-like attention, 8 SwiGLU experts of
    FFN 14336, top-2 routing, RoPE theta 1e6."""
    return Shape(hidden=4096, n_q=32, n_kv=8, head_dim=128, ffn=14336,
                 rms_eps=1e-5, rope_theta=1e6, page_size=16, n_experts=8, top_k=2)


def tiny_moe_shape() -> Shape:
    """The small config's attention with 4 SwiGLU experts of FFN 688, top-2."""
    return Shape(hidden=256, n_q=4, n_kv=2, head_dim=64, ffn=688, rms_eps=1e-5,
                 rope_theta=1e4, page_size=16, n_experts=4, top_k=2)


def moe_batch(n_decode: int = 1920, prefill: int = 128) -> Batch:
    """1920 decode requests (lognormal median 600, sigma 1, clip [1, 8192]) and
    one 128-token prefill chunk; 16-token pages, 1% slack."""
    ctx = lognormal_contexts(n_decode, 600.0, 1.0, 1, 8192, seed=1)
    return make_batch(mixtral_shape(), ctx, [prefill] if prefill else [], None,
                      seed_bt=2, slack=0.01, max_pages=8192 // 16, name="mixtral")


def make_router_logits(n_tokens: int, n_experts: int, seed: int = 4) -> torch.Tensor:
    """Router logits N(0, 1) per token and expert, float32 (CPU)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(n_tokens, n_experts, generator=g, dtype=torch.float32)


# --------------------------------------------------------------------------
# weights and activations

def make_weights(shape: Shape, seed: int = 0, gain_std: float = 0.0,
                 std: float = 0.02) -> dict:
    """Random bf16 layer weights (CPU tensors).

    Projection and FFN matrices are N(0, std); RMSNorm gains are 1, or
    ``1 + gain_std * N(0,1)`` when ``gain_std > 0`` (used by parity tests so
    that a gain applied to the wrong element cannot hide).

    Layouts: ``w_qkv [(n_q + 2 n_kv) d, H]`` (rows: q heads, k heads, v heads),
    ``w_o [H, n_q d]``, ``w_gate_up [2F, H]`` (gate rows then up rows),
    ``w_down [H, F]``, gains ``[H]``.
    """
    g = torch.Generator().manual_seed(seed)
    H, F = shape.hidden, shape.ffn
    qd = shape.n_q * shape.head_dim

    def rn(*sz):
        return (torch.randn(*sz, generator=g) * std).to(BF16)

    w = {
        "w_qkv": rn(shape.qkv_rows, H),
        "w_o": rn(H, qd),
        "w_gate_up": rn(2 * F, H),
        "w_down": rn(H, F),
    }
    if gain_std > 0:
        g2 = torch.Generator().manual_seed(seed + 1000)
        w["norm1"] = (1.0 + gain_std * torch.randn(H, generator=g2)).to(BF16)
        w["norm2"] = (1.0 + gain_std * torch.randn(H, generator=g2)).to(BF16)
    else:
        w["norm1"] = torch.ones(H, dtype=BF16)
        w["norm2"] = torch.ones(H, dtype=BF16)
    return w


def make_moe_weights(shape: Shape, seed: int = 0, gain_std: float = 0.0,
                     std: float = 0.02) -> dict:
    """Attention weights as make_weights, and the experts in place of the dense
    FFN: w_experts_gate_up [E, 2F, H] (gate rows, then up rows, per expert) and
    w_experts_down [E, H, F], N(0, std), bf16 (CPU)."""
    w = make_weights(Shape(shape.hidden, shape.n_q, shape.n_kv, shape.head_dim, 16,
                           shape.rms_eps, shape.rope_theta, shape.page_size),
                     seed=seed, gain_std=gain_std, std=std)
    del w["w_gate_up"], w["w_down"]
    g = torch.Generator().manual_seed(seed + 2000)
    E, H, F = shape.n_experts, shape.hidden, shape.ffn
    w["w_experts_gate_up"] = (torch.randn(E, 2 * F, H, generator=g) * std).to(BF16)
    w["w_experts_down"] = (torch.randn(E, H, F, generator=g) * std).to(BF16)
    return w


def make_x(shape: Shape, n_tokens: int, seed: int = 0) -> torch.Tensor:
    """Layer input activations ``[T, H]`` bf16, N(0,1)."""
    g = torch.Generator().manual_seed(seed + 7)
    return torch.randn(n_tokens, shape.hidden, generator=g).to(BF16)


# --------------------------------------------------------------------------
# KV pools

def page_fill_counts(shape: Shape, batch: Batch, appended: bool = False) -> np.ndarray:
    """Per physical page, how many leading positions hold a cached token
    before the step (after it, with appended=True); 0 for pages no sequence
    owns."""
    P = shape.page_size
    cnt = np.zeros(batch.num_pages, np.int32)
    for s in range(batch.n_seq):
        cached = int(batch.seq_lens[s]) - (0 if appended else int(batch.q_lens[s]))
        n_pages = (int(batch.seq_lens[s]) + P - 1) // P
        for j in range(n_pages):
            cnt[batch.block_table[s, j]] = min(P, max(0, cached - j * P))
    return cnt


def make_pools(shape: Shape, batch: Batch, device="cpu", seed: int = 3, appended: bool = False):
    """K and V pools ``[num_pages, n_kv, page_size, head_dim]`` bf16.

    Cached positions are N(0,1); every other position is NaN.  With
    appended=True the positions of this step's tokens count as cached too (a
    cache as it stands after the step's append).  On a CUDA
    device the values come from torch's CUDA generator (seeded), so that a
    multi-GB pool is drawn in place.
    """
    dev = torch.device(device)
    sz = (batch.num_pages, shape.n_kv, shape.page_size, shape.head_dim)
    g = torch.Generator(device=dev).manual_seed(seed)
    k = torch.randn(sz, generator=g, device=dev, dtype=BF16)
    v = torch.randn(sz, generator=g, device=dev, dtype=BF16)
    cnt = torch.from_numpy(page_fill_counts(shape, batch, appended)).to(dev)
    empty = torch.arange(shape.page_size, device=dev)[None, :] >= cnt[:, None]
    empty = empty[:, None, :, None]
    k.masked_fill_(empty, float("nan"))
    v.masked_fill_(empty, float("nan"))
    return k, v
