"""nf_attention_noalloc: the attention entry point for callers that cannot
allocate device memory (a runtime that owns all device memory and passes an
operator only its inputs and outputs, or a hot loop that cannot take an
allocation's device synchronisation).  Its working memory is a fixed array
inside the library.

Checked here: on two calls in a row (the second reuses the array the first one
left behind) its output matches the float64 oracle row by row at the
attention tolerance and the plan-based nf_attention on the same inputs; a
batch whose working memory would not fit is refused on the host; a page id
outside the pool is reported by nf_attention_noalloc_poll (once: the poll
clears it) without any read outside the pool.  This file is collected last so
that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
from oracle import layer as orc
from tests.helpers import compare, f64

pytestmark = pytest.mark.gpu


def _case(shape, batch, seed):
    T = batch.n_tokens
    kp, vp = wl.make_pools(shape, batch, "cuda", seed=seed, appended=True)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(T, shape.n_q, shape.head_dim, generator=g).to(torch.bfloat16).cuda()
    bt = torch.from_numpy(batch.block_table).cuda()
    sl = torch.from_numpy(batch.seq_lens).cuda()
    return q, kp, vp, bt, sl


def _oracle_rows(shape, batch, q, kp, vp, rows):
    """Softmax attention of each listed row over its cached positions 0..pos."""
    seq, pos = orc.token_map(batch.q_lens, batch.seq_lens)
    P = shape.page_size
    out = []
    for t in rows:
        s, L = int(seq[t]), int(pos[t]) + 1
        j = np.arange(L)
        pages = torch.as_tensor(batch.block_table[s, j // P].astype(np.int64), device=kp.device)
        offs = torch.as_tensor(j % P, device=kp.device)
        out.append(orc.attention_one(f64(q[t]), f64(kp[pages, :, offs, :]), f64(vp[pages, :, offs, :]),
                                     shape.n_q, shape.n_kv))
    return np.stack(out)


@pytest.mark.parametrize("which", ["small", "llama8b-shaped"])
def test_noalloc_attention_matches_the_oracle_twice(which):
    if which == "small":
        shape = wl.tiny_shape()
        batch = wl.make_batch(shape, [17, 33, 48, 64, 1, 2047], [32], [5], seed_bt=3)
        rows = list(range(batch.n_tokens))
    else:
        shape = wl.llama8b_shape()
        ctx = wl.lognormal_contexts(300, 600.0, 1.0, 1, 4096, seed=1)
        batch = wl.make_batch(shape, ctx, [64], [100], seed_bt=2, max_pages=4096 // 16)
        rows = sorted({0, 1, int(np.argmax(ctx)), int(np.argmin(ctx)), 150, 299, 300, 331, 363})
    q, kp, vp, bt, sl = _case(shape, batch, seed=7)
    T = batch.n_tokens
    ref = _oracle_rows(shape, batch, q, kp, vp, rows)
    plan_o = torch.empty_like(q)
    plan = _lib.Plan(shape, batch, _lib.make_opts(T, kv_chunk=2048))
    _lib.attention(plan, q, kp, vp, bt, sl, plan_o)
    plan.poll()
    plan.close()
    _lib.attention_noalloc_poll()            # start from a clear status word
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        _lib.attention_noalloc(shape, batch, q, kp, vp, bt, sl, o)
        _lib.attention_noalloc_poll()          # waits for the stream; raises on a device error
        got = f64(o)
        compare(got[rows], ref, f"no-alloc attention vs oracle, call {call + 1}")
        compare(got, f64(plan_o), f"no-alloc attention vs nf_attention, call {call + 1}")


def test_noalloc_attention_refuses_a_batch_that_does_not_fit():
    shape = wl.llama8b_shape()
    batch = wl.make_batch(shape, [8192] * 2048, [], seed_bt=2, max_pages=8192 // 16)
    q = torch.empty(batch.n_tokens, shape.n_q, shape.head_dim, dtype=torch.bfloat16, device="cuda")
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.NanoflowError) as e:
        _lib.attention_noalloc(shape, batch, q, dummy, dummy, bt, bt, q)
    assert e.value.code == _lib.NF_ERR_INVALID_ARG
    assert "working memory" in str(e.value)


def test_noalloc_attention_reports_a_bad_page_id_once():
    """A block-table entry past the pool: the call still returns, reads stay
    inside the pool, the next poll reports NF_ERR_DEVICE and clears the word,
    and a following call on valid inputs is clean again."""
    shape = wl.tiny_shape()
    batch = wl.tiny_batch()
    q, kp, vp, bt, sl = _case(shape, batch, seed=9)
    o = torch.empty_like(q)
    _lib.attention_noalloc_poll()
    bad = bt.clone()
    bad[1, 1] = batch.num_pages + 7
    _lib.attention_noalloc(shape, batch, q, kp, vp, bad, sl, o)
    with pytest.raises(_lib.NanoflowError) as e:
        _lib.attention_noalloc_poll()
    assert e.value.code == _lib.NF_ERR_DEVICE and "page id" in str(e.value)
    _lib.attention_noalloc_poll()            # reported once
    _lib.attention_noalloc(shape, batch, q, kp, vp, bt, sl, o)
    _lib.attention_noalloc_poll()
    rows = list(range(batch.n_tokens))
    compare(f64(o), _oracle_rows(shape, batch, q, kp, vp, rows), "no-alloc attention after a bad call")
