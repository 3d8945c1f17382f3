"""nf_attention_noalloc: the attention entry point for callers that cannot
allocate device memory (a runtime that owns all device memory and passes an
operator only its inputs and outputs, or a hot loop that cannot take an
allocation's device synchronisation).  Its working memory is a fixed array
inside the library.

It must give what nf_attention (plan-based) gives on the same inputs, on two
calls in a row (the second call reuses the array the first one left behind),
and refuse a batch whose working memory would not fit.  This file is collected
last so that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
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


@pytest.mark.parametrize("which", ["small", "llama8b-shaped"])
def test_noalloc_attention_matches_plan_attention_twice(which):
    if which == "small":
        shape = wl.tiny_shape()
        batch = wl.make_batch(shape, [17, 33, 48, 64, 1, 2047], [32], [5], seed_bt=3)
    else:
        shape = wl.llama8b_shape()
        ctx = wl.lognormal_contexts(300, 600.0, 1.0, 1, 4096, seed=1)
        batch = wl.make_batch(shape, ctx, [64], [100], seed_bt=2, max_pages=4096 // 16)
    q, kp, vp, bt, sl = _case(shape, batch, seed=7)
    T = batch.n_tokens
    ref = torch.empty_like(q)
    plan = _lib.Plan(shape, batch, _lib.make_opts(T, kv_chunk=2048))
    _lib.attention(plan, q, kp, vp, bt, sl, ref)
    plan.poll()
    plan.close()
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        _lib.attention_noalloc(shape, batch, q, kp, vp, bt, sl, o)
        torch.cuda.synchronize()
        compare(f64(o), f64(ref), f"no-alloc attention, call {call + 1}")


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
