"""Serving a real (random-weight) model through the runtime, replayed through
the oracle: the model, and the oracle's side of the replay.

The model is a small stack with non-zero projections and norm gains other
than 1, whose LM head is a scaled copy of the embedding shifted by one row plus
noise, so the greedy token has a clear margin while the logits still depend on
every layer's attention (over K/V appended in earlier iterations) and FFN.
The replay runs each batch the runtime formed through the oracle's stack step,
with the oracle's own K/V pools updated from the K/V it appends."""
import numpy as np
import torch

from nano_intra_device_gb300 import workload as wl
from oracle import layer as orc


def serving_model(shape, n_layers, vocab, seed=0, proj_scale=3.0, head_scale=0.1,
                  head_noise=0.05):
    """(embed, norm_f, lm_head, layers) as bf16 CPU tensors.  With the small
    shape and these scales the top logit leads the second by about 7 or more
    (logits RMS ~2.5), while dropping the K/V of earlier iterations moves
    logits by 1.5 to 4: tokens are robust to rounding and logits are not
    blind to attention."""
    g = torch.Generator().manual_seed(seed)
    H = shape.hidden
    embed = torch.randn(vocab, H, generator=g)
    lm_head = head_scale * torch.roll(embed, shifts=1, dims=0) + head_noise * torch.randn(vocab, H, generator=g)
    norm_f = 1 + 0.1 * torch.randn(H, generator=g)
    layers = []
    for i in range(n_layers):
        w = wl.make_weights(shape, seed=seed + 10 + i, gain_std=0.1)
        layers.append({k: ((v.float() * proj_scale).to(torch.bfloat16) if k.startswith("w_") else v)
                       for k, v in w.items()})
    bf = torch.bfloat16
    return embed.to(bf), norm_f.to(bf), lm_head.to(bf), layers


class OracleServer:
    """The oracle's side of a serving replay: one float64 K and V pool per
    layer (zeros at the start, like the runtime's), the batches the runtime
    formed, and the tokens its decode rows consumed."""

    def __init__(self, shape, model, num_pages, max_pages, store=None):
        self.shape, self.store, self.max_pages = shape, store, max_pages
        embed, norm_f, lm_head, layers = model
        self.embed, self.norm_f, self.lm_head = embed, norm_f, lm_head
        self.layers64 = [orc.weights_f64(w) for w in layers]
        sz = (num_pages, shape.n_kv, shape.page_size, shape.head_dim)
        self.pools = [(torch.zeros(sz, dtype=torch.float64), torch.zeros(sz, dtype=torch.float64))
                      for _ in layers]

    def step(self, b, tokens):
        """Run batch view b (as nf_runtime_step / nf_runtime_form describe it)
        on the given row tokens; append its K/V; return the emitting rows'
        logits [n_emit, vocab] float64."""
        n_seq = b["n_decode"] + b["n_prefill"]
        bt = np.asarray(b["block_table"], np.int64).reshape(n_seq, self.max_pages)
        sl = np.asarray(b["seq_lens"], np.int64)
        ql = np.asarray([1] * b["n_decode"] + list(b["prefill_q_lens"]), np.int64)
        out = orc.stack_step(self.shape, self.embed, self.norm_f, self.lm_head, self.layers64,
                             np.asarray(tokens, np.int64), self.pools, bt, sl, ql,
                             store=self.store)
        P = self.shape.page_size
        for (slots, k, v), (kp, vp) in zip(out["appended"], self.pools):
            pg = torch.as_tensor(slots // P)
            off = torch.as_tensor(slots % P)
            kp[pg, :, off, :] = torch.from_numpy(np.ascontiguousarray(k))
            vp[pg, :, off, :] = torch.from_numpy(np.ascontiguousarray(v))
        emit = np.asarray(b["row_emit"], bool)
        return out["logits"][emit]


def row_tokens(b, prompts, generated):
    """Each row's input token: its prompt token, or for a decode row at
    position p the request's output number p - len(prompt)."""
    toks = []
    for rid, pos, tok in zip(b["row_request"], b["row_pos"], b["row_token"]):
        toks.append(tok if tok >= 0 else generated[rid][pos - len(prompts[rid])])
    return toks


def greedy(logits):
    """Index of the largest value per row, the lowest on ties."""
    return np.argmax(np.asarray(logits), axis=1)
