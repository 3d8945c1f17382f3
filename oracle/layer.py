"""CPU oracle for one pre-norm decoder-layer step over a mixed, paged batch.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The library never
does, and it shares no code with the CUDA path.

What it computes is the plain definition of the layer.  The method this
repository accelerates (nano-batching with overlapped execution) reaches exactly
that result, because nano-batches share no data dependencies ("NanoFlow:
Towards Optimal LLM Serving Throughput", "The Intra-Device Parallelism
Mechanism").  So the oracle never splits the batch: it walks tokens in order.

Arithmetic: float64 throughout.  bf16 inputs are converted exactly.  By
default nothing is rounded back to bf16 (not even the K/V it appends).  With
``store="bf16"`` the tensors that a layer keeps in memory between its
operations — n1, q and the appended k, v (after RoPE), the attention output o,
h, n2, the SwiGLU product a, and a layer's output when another layer or the
final norm reads it — are rounded to the nearest bf16 value (ties to even)
where they are produced; every arithmetic step between them stays float64, and
the returned outputs (y, logits) are not rounded.  The pages fix no precision;
this mode is the plain reading of "a layer whose stored tensors are bf16",
used to separate the error that storage in bf16 causes from the rest.

Readings taken where the pages leave a step open (each is listed with its
reason in the design notes):

* layer structure: Llama pre-norm, no biases — x -> RMSNorm -> QKV -> RoPE ->
  paged GQA attention -> O-proj + residual -> RMSNorm -> SwiGLU FFN + residual.
  The pages give only the operation list (KQV, attention, O, Up/Gate/Down;
  "NanoFlow: Towards Optimal LLM Serving Throughput", "The Intra-Device
  Parallelism Mechanism"; "CSE 451 Lecture 25", slide 81 names RoPE).
* RoPE: rotate-half pairing (i, i + d/2), angle pos * theta^(-2i/d).
* ``seq_lens`` is the KV length after this step's tokens are appended.
* GQA: query head h reads KV head h // (n_q / n_kv) (contiguous groups).
* softmax scale 1/sqrt(d); masked positions are excluded, not -inf-added.
* mixture-of-experts FFN (the Mixtral-shaped config): router logits are an
  input of the step; each token takes its top-k experts (ties to the lower
  index) weighted by a softmax over the selected logits, and the FFN output is
  the weighted sum of those experts' SwiGLU FFNs.  The pages name only "gate
  routing" and grouped GEMMs over experts.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force and printed values); none is unpinned.
"""
from __future__ import annotations

import numpy as np
import torch


# --------------------------------------------------------------------------
# conversions

def f64(t) -> np.ndarray:
    """Exact conversion of a bf16/fp32 tensor or array to float64."""
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


class _LazyExperts:
    """Per-expert float64 view of a stacked [E, rows, cols] bf16 tensor,
    converted one expert at a time on first use (the Mixtral-shaped experts
    hold 1.4 G parameters; a sampled-row check touches a few of them)."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = f64(self.t[e])
        return self.cache[e]


def weights_f64(w: dict) -> dict:
    """Convert a weight dict (bf16 tensors) to float64 arrays once (expert
    stacks lazily, expert by expert)."""
    return {k: (_LazyExperts(v) if k.startswith("w_experts") else f64(v)) for k, v in w.items()}


def bf16(v) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even,
    returned as float64.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and float32's
    exponent range.  With v = m * 2^e, 0.5 <= |m| < 1, the representable
    neighbours are the multiples of 2^(e-8); numpy's round() breaks ties to the
    even multiple.  Normal range only (|v| >= 2^-126; values here are far
    from it), zeros keep their sign.
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)


def _storage(store):
    if store is None:
        return lambda v: v
    if store == "bf16":
        return bf16
    raise ValueError(f"store must be None or 'bf16', not {store!r}")


# --------------------------------------------------------------------------
# elementary steps

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of each row: x * g / sqrt(mean(x^2) + eps).

    Pre-norm placement as in a Llama decoder layer ("CSE 451 Lecture 25",
    slide 25, decoder-only transformer layer diagram).
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * g / np.sqrt(ms + eps)


def rope(u: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half form.

    u: [N, heads, d]; pos: [N].  For i < d/2 the pair (u_i, u_{i+d/2}) is
    rotated by the angle pos * theta^(-2i/d).  ("CSE 451 Lecture 25",
    slide 81 lists RoPE among the layer's operations; the pairing convention
    is this library's reading.)
    """
    d = u.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = pos.astype(np.float64)[:, None] * inv_freq[None, :]          # [N, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = u[..., :half], u[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def attention_one(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_q: int, n_kv: int) -> np.ndarray:
    """Softmax attention of one token's query heads over its KV positions.

    q: [n_q, d]; K, V: [L, n_kv, d] (every position the token may see).
    Query head h uses KV head h // (n_q / n_kv): grouped-query attention, where
    several query heads share one K/V head ("LLM Inference Performance", KV
    cache sizing; "NanoFlow: Towards Optimal LLM Serving Throughput",
    "Factor 1").  Returns o: [n_q, d].
    """
    d = q.shape[-1]
    grp = n_q // n_kv
    o = np.empty_like(q)
    for h in range(n_q):
        g = h // grp
        s = K[:, g, :] @ q[h] / np.sqrt(d)
        p = np.exp(s - s.max())
        o[h] = (p @ V[:, g, :]) / p.sum()
    return o


# --------------------------------------------------------------------------
# step metadata (integer)

def token_map(q_lens: np.ndarray, seq_lens: np.ndarray):
    """Sequence id and position of each token of the step.

    Sequence s owns q_lens[s] consecutive tokens, at positions
    seq_lens[s] - q_lens[s] ... seq_lens[s] - 1 (a decode request has one token
    at seq_lens[s] - 1; a prefill chunk continues its prompt after the cached
    prefix).  Returns (seq [T], pos [T]) as int64.
    """
    seq, pos = [], []
    for s, (q, L) in enumerate(zip(q_lens.tolist(), seq_lens.tolist())):
        for i in range(q):
            seq.append(s)
            pos.append(L - q + i)
    return np.asarray(seq, np.int64), np.asarray(pos, np.int64)


def slot_of(seq: np.ndarray, pos: np.ndarray, block_table: np.ndarray, page: int) -> np.ndarray:
    """Physical pool slot of (sequence, position): block_table[s][pos // P] * P
    + pos % P.  The block table maps logical blocks to physical blocks
    ("LLM Inference Performance", "PagedAttention: virtual memory for the KV
    cache"; "Inside nano-vLLM", 4.2 Paged KV, slot mapping of new KV writes).
    """
    return block_table[seq, pos // page].astype(np.int64) * page + pos % page


def split_kv_items(ctx_len: np.ndarray, chunk: int, row_begin: int = 0, row_end: int | None = None):
    """Work items of split-KV attention for rows [row_begin, row_end).

    Row t sees ctx_len[t] positions; they are cut into pieces of ``chunk``
    positions, the last one ragged.  Returns a sorted list of
    (row, first_position, n_positions).  The set is unique; the order in which
    a kernel visits the items is not part of the result.
    """
    if row_end is None:
        row_end = len(ctx_len)
    out = []
    for t in range(row_begin, row_end):
        L = int(ctx_len[t])
        for b in range(0, L, chunk):
            out.append((t, b, min(chunk, L - b)))
    return sorted(out)


# --------------------------------------------------------------------------
# the layer step

def route(logits, top_k: int):
    """Top-k gate routing of a mixture-of-experts FFN ("NanoFlow: Towards
    Optimal LLM Serving Throughput", MoE models: gate routing, then experts
    computing on different tokens).  Reading taken: per token the top_k
    experts by router logit, ties going to the lower expert index, weighted by
    a softmax over the selected logits.  logits [T, E]; returns (experts
    [T, top_k] int64, weights [T, top_k] float64), best first."""
    r = np.asarray(logits, np.float64)
    T, E = r.shape
    experts = np.zeros((T, top_k), np.int64)
    weights = np.zeros((T, top_k))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-r[t, e], e))
        sel = order[:top_k]
        z = np.exp(r[t, sel] - r[t, sel].max())
        experts[t] = sel
        weights[t] = z / z.sum()
    return experts, weights


def expert_groups(experts, n_experts: int):
    """The grouped order of the (token, choice) pairs that the expert GEMMs
    consume: expert by expert, and within an expert by increasing token.
    Returns (pairs [T*k, 2] of (token, choice), offsets [n_experts + 1])."""
    experts = np.asarray(experts)
    pairs, offsets = [], [0]
    for e in range(n_experts):
        for t in range(experts.shape[0]):
            for j in range(experts.shape[1]):
                if experts[t, j] == e:
                    pairs.append((t, j))
        offsets.append(len(pairs))
    return np.asarray(pairs, np.int64).reshape(-1, 2), np.asarray(offsets, np.int64)


def moe_ffn(n2, w64: dict, logits, top_k: int, F: int, store=None):
    """sum over the token's selected experts e of weight_e * FFN_e(n2), with
    FFN_e(z) = (silu(z W_g,e^T) * (z W_u,e^T)) W_d,e^T; w64["w_experts_gate_up"][e]
    holds the gate rows then the up rows of expert e, w64["w_experts_down"][e]
    its down matrix.  n2 [R, H], logits [R, E] for the same rows.  With
    store="bf16" each expert's SwiGLU product is rounded to bf16."""
    rnd = _storage(store)
    experts, weights = route(logits, top_k)
    out = np.zeros_like(n2)
    for i in range(n2.shape[0]):
        for j in range(top_k):
            e = int(experts[i, j])
            gu = w64["w_experts_gate_up"][e]
            a = rnd(silu(n2[i] @ gu[:F].T) * (n2[i] @ gu[F:].T))
            out[i] += weights[i, j] * (a @ w64["w_experts_down"][e].T)
    return out


def _needed_rows(seq, rows):
    """rows plus every earlier token of the same sequence in this step: a
    prefill row attends to the K/V this step appends for earlier rows of its
    chunk (the dependency rule of the pages: a nano-operation depends on
    another when their parent operations depend and their token ranges
    intersect)."""
    need = set(int(r) for r in rows)
    for r in list(need):
        s = seq[r]
        t = r - 1
        while t >= 0 and seq[t] == s:
            need.add(t)
            t -= 1
    return np.asarray(sorted(need), np.int64)


def layer_step(shape, w64: dict, x, k_pool, v_pool, block_table, seq_lens, q_lens,
               rows=None, keep=False, router_logits=None, store=None) -> dict:
    """One decoder-layer step over a mixed prefill+decode batch.

    shape: a Shape (hidden, n_q, n_kv, head_dim, ffn, rms_eps, rope_theta,
    page_size).  w64: float64 weights (see ``weights_f64``).  x: [T, H] layer
    input.  k_pool, v_pool: [num_pages, n_kv, P, d] caches holding the
    positions cached before the step (bf16 tensors; only the pages a computed
    row reads are converted).  block_table [n_seq, max_pages], seq_lens and
    q_lens [n_seq] as in the workload module.

    rows: the token rows whose outputs are wanted (default: all).  Returns a
    dict with ``rows``, ``y`` [len(rows), H], the appended ``k_new`` / ``v_new``
    [len(rows), n_kv, d] and their ``slots``, plus the integer ``seq``/``pos``
    maps.  With keep=True the intermediates n1, q, o, h, n2, a are returned
    for the same rows.

    Steps, in the order of a pre-norm layer:
      n1 = RMSNorm(x; g1); [q|k|v] = n1 W_qkv^T; q, k <- RoPE(pos);
      K/V of the step appended at slot(seq, pos);
      o = GQA softmax attention over positions 0..pos of the token's sequence;
      h = x + o W_o^T; n2 = RMSNorm(h; g2); a = silu(n2 W_g^T) * (n2 W_u^T);
      y = h + a W_d^T.
    A mixture-of-experts layer (shape.n_experts > 0, weights w_experts_gate_up
    and w_experts_down) replaces the last two lines by y = h + moe_ffn(n2)
    with router_logits [T, n_experts] given for the step.

    store: None (float64 throughout) or "bf16" (n1, q, k, v, o, h, n2 and a
    rounded to bf16 where they are produced; y is returned unrounded).
    """
    rnd = _storage(store)
    H, nq, nkv, d, F = shape.hidden, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn
    P = shape.page_size
    q_lens = np.asarray(q_lens, np.int64)
    seq_lens = np.asarray(seq_lens, np.int64)
    block_table = np.asarray(block_table)
    seq, pos = token_map(q_lens, seq_lens)
    T = len(seq)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    need = _needed_rows(seq, rows)

    # projections for every needed row
    xn = f64(x[torch.as_tensor(need)]) if isinstance(x, torch.Tensor) else f64(x)[need]
    n1 = rnd(rmsnorm(xn, w64["norm1"], shape.rms_eps))
    qkv = n1 @ w64["w_qkv"].T
    q = qkv[:, : nq * d].reshape(-1, nq, d)
    k = qkv[:, nq * d: (nq + nkv) * d].reshape(-1, nkv, d)
    v = rnd(qkv[:, (nq + nkv) * d:].reshape(-1, nkv, d))
    q = rnd(rope(q, pos[need], shape.rope_theta))
    k = rnd(rope(k, pos[need], shape.rope_theta))
    new_k = {int(t): k[i] for i, t in enumerate(need)}
    new_v = {int(t): v[i] for i, t in enumerate(need)}
    qrow = {int(t): q[i] for i, t in enumerate(need)}
    xrow = {int(t): xn[i] for i, t in enumerate(need)}
    n1row = {int(t): n1[i] for i, t in enumerate(need)}

    # first token index of each sequence (tokens of one sequence are contiguous)
    first_tok = {}
    for t in range(T):
        first_tok.setdefault(int(seq[t]), t)

    o = np.empty((len(rows), nq, d))
    for i, t in enumerate(rows.tolist()):
        s, p = int(seq[t]), int(pos[t])
        cached = int(seq_lens[s] - q_lens[s])      # positions already in the pool
        L = p + 1                                    # causal: positions 0..p
        K = np.empty((L, nkv, d))
        V = np.empty((L, nkv, d))
        n_old = min(cached, L)
        if n_old > 0:
            j = np.arange(n_old)
            pages = torch.as_tensor(block_table[s, j // P].astype(np.int64))
            offs = torch.as_tensor(j % P)
            K[:n_old] = f64(k_pool[pages, :, offs, :])
            V[:n_old] = f64(v_pool[pages, :, offs, :])
        for pp in range(n_old, L):                   # positions appended this step
            tt = first_tok[s] + (pp - cached)
            K[pp] = new_k[tt]
            V[pp] = new_v[tt]
        o[i] = attention_one(qrow[t], K, V, nq, nkv)
    o = rnd(o)

    xr = np.stack([xrow[t] for t in rows.tolist()])
    h = rnd(xr + o.reshape(len(rows), nq * d) @ w64["w_o"].T)
    n2 = rnd(rmsnorm(h, w64["norm2"], shape.rms_eps))
    if getattr(shape, "n_experts", 0):
        lg = np.asarray(router_logits, np.float64)[rows]
        a = None
        y = h + moe_ffn(n2, w64, lg, shape.top_k, F, store=store)
    else:
        gate = n2 @ w64["w_gate_up"][:F].T
        up = n2 @ w64["w_gate_up"][F:].T
        a = rnd(silu(gate) * up)
        y = h + a @ w64["w_down"].T

    out = {
        "rows": rows,
        "y": y,
        "k_new": np.stack([new_k[t] for t in rows.tolist()]),
        "v_new": np.stack([new_v[t] for t in rows.tolist()]),
        "slots": slot_of(seq[rows], pos[rows], block_table, P),
        "seq": seq,
        "pos": pos,
    }
    if keep:
        out.update(n1=np.stack([n1row[t] for t in rows.tolist()]),
                   q=np.stack([qrow[t] for t in rows.tolist()]),
                   o=o, h=h, n2=n2, a=a)
    return out


# --------------------------------------------------------------------------
# a stack of layers with embedding and LM head

def layers_step(shape, layers64: list, x, pools: list, block_table, seq_lens, q_lens,
                rows=None, store=None) -> dict:
    """Several decoder layers over one mixed step: layer l takes the previous
    layer's output (x for the first) and reads its own K/V pools; the block
    table and lengths are shared ("NanoFlow: Towards Optimal LLM Serving
    Throughput", "Example Pipelines for Different Model Scales": the per-layer
    step repeated over the layers).

    layers64: float64 weight dicts; pools: (k_pool, v_pool) per layer; x: [T, H].
    rows: the tokens whose output is wanted; every layer computes the rows
    those need (their earlier prefill rows).  Returns {"rows", "y" [len(rows),
    H], "x_all" [T, H] (rows outside the needed set are left as given),
    "appended": per layer (slots, k_new, v_new) of the computed rows}.
    store: as in layer_step; with "bf16" every layer's output but the last is
    rounded to bf16 before the next layer reads it.
    """
    rnd = _storage(store)
    q_lens = np.asarray(q_lens, np.int64)
    seq_lens = np.asarray(seq_lens, np.int64)
    seq, _ = token_map(q_lens, seq_lens)
    T = len(seq)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    need = _needed_rows(seq, rows)
    x = np.array(f64(x), copy=True)
    n_layers = len(layers64)
    appended = []
    for li, (w64, (kp, vp)) in enumerate(zip(layers64, pools)):
        out = layer_step(shape, w64, x, kp, vp, block_table, seq_lens, q_lens, rows=need,
                         store=store)
        appended.append((out["slots"], out["k_new"], out["v_new"]))
        x = x.copy()
        x[need] = out["y"] if li == n_layers - 1 else rnd(out["y"])
    return {"rows": rows, "y": x[rows], "x_all": x, "appended": appended}


def stack_step(shape, embed, norm_f, lm_head, layers64: list, tokens, pools: list, block_table,
               seq_lens, q_lens, rows=None, store=None) -> dict:
    """A decoder stack over one mixed step: x = embed[tokens]; each layer's step
    (its own K/V pools, the shared block table and lengths); logits =
    RMSNorm(x; norm_f) lm_head^T.

    layers64: float64 weight dicts, one per layer (see weights_f64); pools:
    (k_pool, v_pool) per layer.  rows: the tokens whose logits are wanted;
    every layer computes the rows those need (their earlier prefill rows).
    Returns {"rows", "logits" [len(rows), vocab], "x_final", "appended" (as in
    layers_step)}.
    store: as in layers_step; with "bf16" the last layer's output and the
    final norm's output are rounded too (the logits are not).
    """
    rnd = _storage(store)
    q_lens = np.asarray(q_lens, np.int64)
    seq_lens = np.asarray(seq_lens, np.int64)
    seq, _ = token_map(q_lens, seq_lens)
    T = len(seq)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    need = _needed_rows(seq, rows)
    E = f64(embed)
    x = np.zeros((T, shape.hidden))
    x[need] = E[np.asarray(tokens)[need]]
    out = layers_step(shape, layers64, x, pools, block_table, seq_lens, q_lens, rows=rows,
                      store=store)
    xf = rnd(rmsnorm(rnd(out["y"]), f64(norm_f), shape.rms_eps))
    return {"rows": rows, "logits": xf @ f64(lm_head).T, "x_final": out["y"],
            "appended": out["appended"]}
