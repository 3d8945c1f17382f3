"""Mixture-of-experts layer step (Mixtral-shaped and small): routing and expert
grouping bit-exact against the oracle, the layer output within the stated
tolerance, every executor and FFN split."""
import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
from oracle import layer as orc
from tests.helpers import f64, parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(shape, batch, seed=0, logits=None):
    w = wl.make_moe_weights(shape, seed=seed, gain_std=0.1)
    if logits is None:
        logits = wl.make_router_logits(batch.n_tokens, shape.n_experts, seed=seed + 4)
    w["router_logits"] = logits
    kp, vp = wl.make_pools(shape, batch, DEV, seed=seed + 3)
    x = wl.make_x(shape, batch.n_tokens, seed=seed + 5)
    return w, kp, vp, x


def _oracles(shape, w, x, kp, vp, batch, logits, rows=None):
    """(exact, bf16-storage) oracle results of the MoE layer."""
    w64 = orc.weights_f64(w)
    return tuple(orc.layer_step(shape, w64, x, kp, vp, batch.block_table, batch.seq_lens,
                                batch.q_lens, rows=rows, router_logits=logits, store=st)
                 for st in (None, "bf16"))


def _run(shape, batch, opts, w, kp, vp, x):
    plan = _lib.Plan(shape, batch, opts)
    wd = {k: v.to(DEV) for k, v in w.items()}
    k2, v2 = kp.clone(), vp.clone()
    y = torch.empty(batch.n_tokens, shape.hidden, dtype=torch.bfloat16, device=DEV)
    _lib.layer_step(plan, wd, x.to(DEV), k2, v2, torch.from_numpy(batch.block_table).to(DEV),
                    torch.from_numpy(batch.seq_lens).to(DEV), y)
    plan.poll()
    return plan, y


def _routing(plan, shape, n):
    k = shape.top_k
    off = plan.buffer(_lib.NF_BUF_MOE_OFF, torch.int32, (shape.n_experts + 1,)).numpy()
    perm = plan.buffer(_lib.NF_BUF_MOE_PERM, torch.int32, (plan_T(plan) * k,)).numpy()[: n * k]
    prow = plan.buffer(_lib.NF_BUF_MOE_PAIR_ROW, torch.int32, (plan_T(plan) * k,)).numpy()[: n * k]
    pw = plan.buffer(_lib.NF_BUF_MOE_PAIR_W, torch.float32, (plan_T(plan) * k,)).numpy()[: n * k]
    return off, perm, prow, pw


def plan_T(plan):
    return plan.info()[1]


@pytest.mark.parametrize("shape_fn,batch_fn", [(wl.tiny_moe_shape, wl.tiny_batch),
                                               (wl.mixtral_shape, lambda: wl.moe_batch(200, 56))])
def test_moe_routing_and_grouping_bit_exact(shape_fn, batch_fn):
    shape, batch = shape_fn(), batch_fn()
    T = batch.n_tokens
    w, kp, vp, x = _case(shape, batch, seed=1)
    plan, _ = _run(shape, batch, _lib.make_opts(T), w, kp, vp, x)
    off, perm, prow, pw = _routing(plan, shape, T)
    plan.close()
    experts, weights = orc.route(w["router_logits"].numpy(), shape.top_k)
    pairs, ref_off = orc.expert_groups(experts, shape.n_experts)
    assert np.array_equal(off, ref_off)
    assert np.array_equal(perm, pairs[:, 0])
    ref_prow = np.empty(T * shape.top_k, np.int64)
    ref_prow[pairs[:, 0] * shape.top_k + pairs[:, 1]] = np.arange(len(pairs))
    assert np.array_equal(prow, ref_prow)
    np.testing.assert_allclose(pw, weights.reshape(-1), rtol=2e-6, atol=1e-7)


def test_moe_routing_ties_and_idle_experts():
    """Equal logits go to the lower expert; experts nobody picks get empty
    groups (the grouped GEMM must skip them)."""
    shape, batch = wl.tiny_moe_shape(), wl.tiny_batch()
    T = batch.n_tokens
    logits = torch.zeros(T, shape.n_experts)
    logits[: T // 2, 3] = 1.0          # first half: expert 3, then the tie 0
    w, kp, vp, x = _case(shape, batch, seed=2, logits=logits)
    ex, em = _oracles(shape, w, x, kp, vp, batch, logits.numpy())
    plan, y = _run(shape, batch, _lib.make_opts(T), w, kp, vp, x)
    off, _, _, _ = _routing(plan, shape, T)
    plan.close()
    assert list(np.diff(off)) == [T, T - T // 2, 0, T // 2]   # expert 2 idle
    parity(f64(y), ex["y"], em["y"], "MoE y (ties)")


@pytest.mark.parametrize("executor,ab,fb", [
    (_lib.NF_EXEC_SEQUENTIAL, [0, 36], [0, 36]),
    (_lib.NF_EXEC_SEQUENTIAL, [0, 20, 36], [0, 11, 36]),
    (_lib.NF_EXEC_STREAMS, [0, 18, 36], [0, 18, 36]),
    (_lib.NF_EXEC_STREAMS, [0, 9, 20, 36], [0, 30, 36])])
def test_tiny_moe_layer_matches_oracle(executor, ab, fb):
    shape, batch = wl.tiny_moe_shape(), wl.tiny_batch()
    w, kp, vp, x = _case(shape, batch, seed=3)
    ex, em = _oracles(shape, w, x, kp, vp, batch, w["router_logits"].numpy())
    opts = _lib.make_opts(batch.n_tokens, ab, fb, executor=executor, attn_sms=24, kv_chunk=32)
    plan, y = _run(shape, batch, opts, w, kp, vp, x)
    plan.close()
    parity(f64(y), ex["y"], em["y"], "tiny MoE y")


def test_mixtral_shaped_layer_sampled_rows():
    shape = wl.mixtral_shape()
    batch = wl.moe_batch(240, 48)
    T = batch.n_tokens
    w, kp, vp, x = _case(shape, batch, seed=4)
    ctx = batch.seq_lens[: batch.n_decode]
    rows = [0, int(np.argmax(ctx)), int(np.argmin(ctx)), 239, 240, 260, T - 1]
    ex, em = _oracles(shape, w, x, kp, vp, batch, w["router_logits"].numpy(), rows=rows)
    for ab in ([0, T], [0, 128, T]):
        opts = _lib.make_opts(T, ab, ab, executor=_lib.NF_EXEC_STREAMS if len(ab) > 2 else 0,
                              attn_sms=76)
        plan, y = _run(shape, batch, opts, w, kp, vp, x)
        plan.close()
        parity(f64(y)[rows], ex["y"], em["y"], f"Mixtral-shaped y, bounds {ab}")
