"""A stack of layers (embedding, layers with their own KV pools, final norm,
LM head) through nf_stack_step against the oracle, and the same step replayed
from a CUDA graph."""
import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
from oracle import layer as orc
from tests.helpers import compare, f64, parity


def both(fn, *args, **kw):
    """An oracle function's result under exact and bf16-storage arithmetic."""
    return fn(*args, store=None, **kw), fn(*args, store="bf16", **kw)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _stack(shape, batch, n_layers, vocab, seed=0, gain_std=0.1):
    g = torch.Generator().manual_seed(seed + 100)
    embed = torch.randn(vocab, shape.hidden, generator=g).to(torch.bfloat16)
    lm_head = (torch.randn(vocab, shape.hidden, generator=g) * 0.02).to(torch.bfloat16)
    norm_f = (1 + 0.1 * torch.randn(shape.hidden, generator=g)).to(torch.bfloat16)
    tokens = torch.randint(0, vocab, (batch.n_tokens,), generator=g).to(torch.int32)
    layers = [wl.make_weights(shape, seed=seed + 10 + i, gain_std=gain_std) for i in range(n_layers)]
    pools = [wl.make_pools(shape, batch, DEV, seed=seed + 50 + i) for i in range(n_layers)]
    return embed, norm_f, lm_head, tokens, layers, pools


def _run(shape, batch, opts, embed, norm_f, lm_head, tokens, layers, pools):
    plan = _lib.Plan(shape, batch, opts)
    dl = [{k: v.to(DEV) for k, v in w.items()} for w in layers]
    dp = [(k.clone(), v.clone()) for k, v in pools]
    args = _lib.StackArgs(embed.to(DEV), norm_f.to(DEV), lm_head.to(DEV), dl, dp)
    logits = torch.empty(batch.n_tokens, embed.shape[0], dtype=torch.bfloat16, device=DEV)
    bt = torch.from_numpy(batch.block_table).to(DEV)
    sl = torch.from_numpy(batch.seq_lens).to(DEV)
    tok = tokens.to(DEV)
    _lib.stack_step(plan, args, tok, bt, sl, logits)
    plan.poll()
    return plan, args, logits, (tok, bt, sl), dp


@pytest.mark.parametrize("executor,bounds", [(_lib.NF_EXEC_SEQUENTIAL, None),
                                             (_lib.NF_EXEC_STREAMS, [0, 20, 36]),
                                             (_lib.NF_EXEC_STREAMS, [0, 6, 21, 36])])
def test_tiny_stack_matches_oracle(executor, bounds):
    """Two-stream plans with the same nano-batches in both groups run the
    cross-layer window (no join between layers); the tiny batch's prefill
    sequences cross the nano-batch bounds."""
    shape, batch = wl.tiny_shape(), wl.tiny_batch()
    embed, norm_f, lm_head, tokens, layers, pools = _stack(shape, batch, 3, 96)
    ex, em = both(orc.stack_step, shape, embed, norm_f, lm_head,
                  [orc.weights_f64(w) for w in layers], tokens.numpy(), pools, batch.block_table,
                  batch.seq_lens, batch.q_lens)
    T = batch.n_tokens
    opts = _lib.make_opts(T, bounds, executor=executor, attn_sms=24, kv_chunk=32)
    plan, args, logits, _, dp = _run(shape, batch, opts, embed, norm_f, lm_head, tokens, layers, pools)
    plan.close()
    parity(f64(logits), ex["logits"], em["logits"], "3-layer tiny stack logits")
    # each layer appended this step's K/V into its own pool
    seq, pos = orc.token_map(batch.q_lens, batch.seq_lens)
    slots = orc.slot_of(seq, pos, batch.block_table, shape.page_size)
    P = shape.page_size
    for (k, v) in dp:
        sl_ = torch.as_tensor(slots, device=DEV)
        assert torch.isfinite(k[sl_ // P, :, sl_ % P, :]).all()
        assert torch.isfinite(v[sl_ // P, :, sl_ % P, :]).all()


def test_stack_logits_for_selected_rows_only():
    """nf_stack_step_rows: logits of listed rows (any order) equal those rows of
    the full step within the GEMM's rounding; no rows is valid; a row index
    outside the batch is reported by poll, never read."""
    shape, batch = wl.tiny_shape(), wl.tiny_batch()
    embed, norm_f, lm_head, tokens, layers, pools = _stack(shape, batch, 2, 96)
    T = batch.n_tokens
    opts = _lib.make_opts(T, None, kv_chunk=32)
    plan, args, full, (tok, bt, sl), _ = _run(shape, batch, opts, embed, norm_f, lm_head, tokens,
                                              layers, pools)
    for sel in ([35, 0, 3, 17, 4], list(range(T)), [2]):
        rows = torch.tensor(sel, dtype=torch.int32, device=DEV)
        part = torch.empty(len(sel), embed.shape[0], dtype=torch.bfloat16, device=DEV)
        # the pools carry this step's K/V already: re-running the step rewrites the same slots
        _lib.stack_step_rows(plan, args, tok, bt, sl, rows, part)
        plan.poll()
        compare(f64(part), f64(full)[sel], f"rows {sel[:5]}")
    empty = torch.empty(0, dtype=torch.int32, device=DEV)
    _lib.stack_step_rows(plan, args, tok, bt, sl, empty, torch.empty(1, 96, dtype=torch.bfloat16,
                                                                      device=DEV))
    plan.poll()
    bad = torch.tensor([1, T + 5], dtype=torch.int32, device=DEV)
    out = torch.empty(2, 96, dtype=torch.bfloat16, device=DEV)
    _lib.stack_step_rows(plan, args, tok, bt, sl, bad, out)
    with pytest.raises(_lib.NanoflowError):
        plan.poll()
    assert bool((out[1] == 0).all())
    plan.close()


@pytest.mark.parametrize("bounds,attn_sms", [(None, 0), ([0, 112, 128], 76)])
def test_llama8b_shaped_two_layer_stack_sampled_rows(bounds, attn_sms):
    """Sequential, and the cross-layer window with the nano-batch bound inside
    the 32-token prefill chunk (its second part attends to K/V the first part's
    QKV projection appended)."""
    shape = wl.llama8b_shape()
    ctx = wl.lognormal_contexts(96, 600.0, 1.0, 1, 4096, seed=1)
    batch = wl.make_batch(shape, ctx, [32], None, seed_bt=2, max_pages=4096 // 16)
    embed, norm_f, lm_head, tokens, layers, pools = _stack(shape, batch, 2, 32000, gain_std=0.0)
    rows = [0, 5, int(np.argmax(ctx)), 95, 96, 127]
    ref, em = both(orc.stack_step, shape, embed, norm_f, lm_head,
                   [orc.weights_f64(w) for w in layers], tokens.numpy(), pools, batch.block_table,
                   batch.seq_lens, batch.q_lens, rows=rows)
    ex = _lib.NF_EXEC_SEQUENTIAL if bounds is None else _lib.NF_EXEC_STREAMS
    opts = _lib.make_opts(batch.n_tokens, bounds, executor=ex, attn_sms=attn_sms)
    plan, args, logits, _, _ = _run(shape, batch, opts, embed, norm_f, lm_head, tokens, layers, pools)
    plan.close()
    parity(f64(logits)[rows], ref["logits"], em["logits"], "8B-shaped 2-layer stack logits")


@pytest.mark.parametrize("bounds", [None, [0, 32, 64]])
def test_stack_cuda_graph_replay_equals_eager(bounds):
    """A captured stack step replays bit for bit, also with the cross-layer
    window (two streams forked from and joined to the capturing stream)."""
    shape = wl.llama8b_shape()
    ctx = wl.lognormal_contexts(64, 600.0, 1.0, 1, 2048, seed=3)
    batch = wl.make_batch(shape, ctx, [], None, seed_bt=4, max_pages=2048 // 16)
    embed, norm_f, lm_head, tokens, layers, pools = _stack(shape, batch, 4, 8192, gain_std=0.0)
    ex = _lib.NF_EXEC_SEQUENTIAL if bounds is None else _lib.NF_EXEC_STREAMS
    opts = _lib.make_opts(batch.n_tokens, bounds, executor=ex, attn_sms=64)
    plan, args, logits, (tok, bt, sl), dp = _run(shape, batch, opts, embed, norm_f, lm_head, tokens,
                                                 layers, pools)
    eager = logits.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                      # warm path before capture
        _lib.stack_step(plan, args, tok, bt, sl, logits, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _lib.stack_step(plan, args, tok, bt, sl, logits)
    logits.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    plan.poll()
    assert torch.equal(logits, eager)
    plan.close()


# ------------------------------------------------------------ layers only

def _run_layers(shape, batch, opts, layers, pools, x):
    plan = _lib.Plan(shape, batch, opts)
    dl = [{k: v.to(DEV) for k, v in w.items()} for w in layers]
    dp = [(k.clone(), v.clone()) for k, v in pools]
    args = _lib.LayersArgs(dl, dp)
    y = torch.empty(batch.n_tokens, shape.hidden, dtype=torch.bfloat16, device=DEV)
    bt = torch.from_numpy(batch.block_table).to(DEV)
    sl = torch.from_numpy(batch.seq_lens).to(DEV)
    xd = x.to(DEV)
    _lib.layers_step(plan, args, xd, bt, sl, y)
    plan.poll()
    assert torch.equal(xd.cpu(), x)   # the input is not modified
    return plan, y


@pytest.mark.parametrize("n_layers", [1, 2, 3])
@pytest.mark.parametrize("executor,bounds", [(_lib.NF_EXEC_SEQUENTIAL, None),
                                             (_lib.NF_EXEC_STREAMS, [0, 20, 36]),
                                             (_lib.NF_EXEC_STREAMS, [0, 5, 19, 30, 36])])
def test_tiny_layers_step_matches_oracle(n_layers, executor, bounds):
    shape, batch = wl.tiny_shape(), wl.tiny_batch()
    layers = [wl.make_weights(shape, seed=70 + i, gain_std=0.1) for i in range(n_layers)]
    pools = [wl.make_pools(shape, batch, DEV, seed=80 + i) for i in range(n_layers)]
    x = wl.make_x(shape, batch.n_tokens, seed=9)
    ex, em = both(orc.layers_step, shape, [orc.weights_f64(w) for w in layers], x, pools,
                  batch.block_table, batch.seq_lens, batch.q_lens)
    opts = _lib.make_opts(batch.n_tokens, bounds, executor=executor, attn_sms=24, kv_chunk=32)
    plan, y = _run_layers(shape, batch, opts, layers, pools, x)
    plan.close()
    parity(f64(y), ex["y"], em["y"], f"{n_layers} tiny layers")


@pytest.mark.parametrize("ab,fb", [([0, 5, 19, 30, 36], [0, 19, 36]),   # 4-way attention, 2-way FFN
                                   ([0, 20, 36], [0, 10, 36]),          # FFN bound inside a nano-batch
                                   ([0, 12, 24, 36], [0, 36])])
def test_tiny_cross_layer_window_with_other_ffn_splits(ab, fb):
    """The cross-layer window when the FFN group is split differently from
    the attention group: a next-layer nano-batch starts once the FFN
    nano-batches covering its rows are done."""
    shape, batch = wl.tiny_shape(), wl.tiny_batch()
    layers = [wl.make_weights(shape, seed=90 + i, gain_std=0.1) for i in range(3)]
    pools = [wl.make_pools(shape, batch, DEV, seed=95 + i) for i in range(3)]
    x = wl.make_x(shape, batch.n_tokens, seed=11)
    ex, em = both(orc.layers_step, shape, [orc.weights_f64(w) for w in layers], x, pools,
                  batch.block_table, batch.seq_lens, batch.q_lens)
    opts = _lib.make_opts(batch.n_tokens, ab, fb, executor=_lib.NF_EXEC_STREAMS, attn_sms=24,
                          kv_chunk=32)
    plan, y = _run_layers(shape, batch, opts, layers, pools, x)
    plan.close()
    parity(f64(y), ex["y"], em["y"], f"3 tiny layers, attention {ab}, FFN {fb}")


@pytest.mark.parametrize("bounds", [None, [0, 128, 256]])
def test_llama8b_shaped_decode_layers_on_one_stream(bounds):
    """A decode-only batch past the weight-row kernel's token range (256 rows,
    so every QKV projection runs the token-row kernel) through two layers on
    one stream.  After the first layer's first attention (and for the second
    nano-batch of each layer) the decode attention starts as the programmatic
    dependent of its QKV GEMM and requests, before it waits for the GEMM, the
    pages that lie wholly before its row's new position.  Split-KV pieces of
    256 positions put piece starts inside long rows; the sampled rows include
    contexts that end on a page boundary, one past it, the shortest and the
    longest, against both oracles."""
    shape = wl.llama8b_shape()
    ctx = wl.lognormal_contexts(256, 600.0, 1.0, 1, 4096, seed=21)
    ctx[7], ctx[130] = 48, 49            # the new position ends / starts a page
    ctx[200] = 1
    batch = wl.make_batch(shape, ctx, [], None, seed_bt=22, max_pages=4096 // 16)
    T = batch.n_tokens
    layers = [wl.make_weights(shape, seed=40 + i, gain_std=0.1) for i in range(2)]
    pools = [wl.make_pools(shape, batch, DEV, seed=45 + i) for i in range(2)]
    x = wl.make_x(shape, T, seed=23)
    rows = sorted({0, 7, 127, 128, 130, 200, 255, int(np.argmax(ctx)), int(np.argmin(ctx))})
    ex, em = both(orc.layers_step, shape, [orc.weights_f64(w) for w in layers], x, pools,
                  batch.block_table, batch.seq_lens, batch.q_lens, rows=rows)
    opts = _lib.make_opts(T, bounds, executor=_lib.NF_EXEC_SEQUENTIAL, kv_chunk=256)
    plan, y = _run_layers(shape, batch, opts, layers, pools, x)
    plan.close()
    parity(f64(y)[rows], ex["y"], em["y"], f"8B-shaped decode layers on one stream, bounds {bounds}")


def test_llama70b_shaped_layer_sampled_rows():
    """One LLaMA-2-70B-shaped layer (hidden 8192, 64 query heads over 8 KV heads,
    FFN 28672) on a mixed batch, sampled rows against both oracles at the
    stated bounds (the bf16-storage oracle) and the stated relative L2 (the
    exact one)."""
    shape = wl.llama70b_shape()
    ctx = wl.lognormal_contexts(64, 1000.0, 1.0, 1, 4096, seed=4)
    batch = wl.make_batch(shape, ctx, [48], None, seed_bt=5, max_pages=4096 // 16)
    w = wl.make_weights(shape, seed=1, gain_std=0.1)
    pools = [wl.make_pools(shape, batch, DEV, seed=6)]
    x = wl.make_x(shape, batch.n_tokens, seed=7)
    rows = [0, int(np.argmax(ctx)), int(np.argmin(ctx)), 63, 64, 90, batch.n_tokens - 1]
    ex, em = both(orc.layers_step, shape, [orc.weights_f64(w)], x, pools, batch.block_table,
                  batch.seq_lens, batch.q_lens, rows=rows)
    plan, y = _run_layers(shape, batch, _lib.make_opts(batch.n_tokens), [w], pools, x)
    info, _ = plan.info()
    assert info.attn_impl == _lib.NF_ATTN_MMA     # GQA group 8 fills the tensor-core tile
    plan.close()
    parity(f64(y)[rows], ex["y"], em["y"], "70B-shaped layer y")


@pytest.mark.parametrize("n_attn,attn_sms", [(2, 46), (3, 45)])
def test_llama70b_shaped_layers_overlapped_window(n_attn, attn_sms):
    """Two LLaMA-2-70B-shaped layers through the cross-layer window, the plan
    kind that wins at this shape: 2 or 3 attention nano-batches on about 45 of
    the SMs (two streams, no join between the layers), FFN in 2 nano-batches.
    A mixed batch of 240 decode rows (lognormal KV lengths, median 1000) and a
    48-token prefill chunk; the nano-batch bounds cut the decode rows and the
    chunk.  Sampled rows include the longest context and the chunk's last
    row, against both oracles."""
    shape = wl.llama70b_shape()
    ctx = wl.lognormal_contexts(240, 1000.0, 1.0, 1, 4096, seed=14)
    batch = wl.make_batch(shape, ctx, [48], None, seed_bt=15, max_pages=4096 // 16)
    T = batch.n_tokens
    layers = [wl.make_weights(shape, seed=20 + i, gain_std=0.1) for i in range(2)]
    pools = [wl.make_pools(shape, batch, DEV, seed=30 + i) for i in range(2)]
    x = wl.make_x(shape, T, seed=17)
    ab = [0] + [int(round(T * i / n_attn)) for i in range(1, n_attn)] + [T]
    if n_attn == 3:
        ab[-2] = 260                                      # a bound inside the prefill chunk
    fb = [0, T // 2, T]
    rows = sorted({0, int(np.argmax(ctx)), int(np.argmin(ctx)), 120, 239, 240, 259, 260, T - 1})
    ex, em = both(orc.layers_step, shape, [orc.weights_f64(w) for w in layers], x, pools,
                  batch.block_table, batch.seq_lens, batch.q_lens, rows=rows)
    opts = _lib.make_opts(T, ab, fb, executor=_lib.NF_EXEC_STREAMS, attn_sms=attn_sms)
    plan, y = _run_layers(shape, batch, opts, layers, pools, x)
    info, _ = plan.info()
    assert info.n_attn == n_attn and info.executor == _lib.NF_EXEC_STREAMS
    plan.close()
    parity(f64(y)[rows], ex["y"], em["y"], f"70B-shaped 2 layers, window n={n_attn}")
