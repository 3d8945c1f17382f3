"""The cost model against numbers the pages print (tests/golden/page_values.json)."""
import json
import os

import numpy as np
import pytest

from nano_intra_device_gb300 import costmodel as cm
from nano_intra_device_gb300 import workload as wl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))


@pytest.mark.parametrize("e", GOLD["kv_bytes_per_token"], ids=lambda e: str(e["value"]))
def test_kv_bytes_per_token(e):
    assert cm.kv_bytes_per_token(e["n_layers"], e["n_kv_heads"], e["head_dim"], e["dtype_bytes"]) == e["value"]


def test_kv_bytes_per_sequence():
    a, b = GOLD["kv_bytes_sequence"]
    v = cm.kv_bytes_per_token(a["n_layers"], a["n_kv_heads"], a["head_dim"], a["dtype_bytes"]) * a["tokens"]
    assert abs(v / 1e9 - a["value_gb"]) <= a["rel_tol"] * a["value_gb"]
    v = cm.kv_bytes_per_token(b["n_layers"], b["n_kv_heads"], b["head_dim"], b["dtype_bytes"]) * b["tokens"]
    assert v == b["value_mib"] * 2**20


def test_optimal_throughput_eq5():
    e = GOLD["optimal_throughput"]
    assert cm.optimal_throughput(e["compute_flops"], e["params"]) == pytest.approx(e["value"], rel=1e-12)


def test_ridge_and_batch1_decode():
    r = GOLD["ridge"]
    assert abs(r["peak_flops"] / r["hbm_bw"] - r["value"]) <= r["abs_tol"]
    e = GOLD["batch1_decode"]
    t = cm.memory_time(e["weight_bytes"], e["hbm_bw"])
    assert t * 1e3 == pytest.approx(e["value_ms"], rel=e["rel_tol"])
    assert 1 / t == pytest.approx(e["tokens_per_s"], rel=e["rel_tol"])


@pytest.mark.parametrize("e", GOLD["effective_intensity"], ids=lambda e: str(e["live_tokens"]))
def test_effective_intensity(e):
    v = cm.effective_intensity(e["batch"], e["params"], e["live_tokens"] * e["kv_bytes_per_token"])
    assert abs(v - e["value"]) <= e["abs_tol"]


def test_transfer_ratio_is_ratio_of_times():
    tr = cm.transfer_ratio(80e9, 2e12, 2048, 70e9, 300e12)
    assert tr == pytest.approx((80e9 / 2e12) / (2 * 2048 * 70e9 / 300e12))


def test_layer_params_llama8b():
    # 32 layers of these weights plus embeddings ~ 8B parameters
    p = cm.layer_params(wl.llama8b_shape())
    assert p == 4096 * 6144 + 4096 * 4096 + 3 * 4096 * 14336
    assert 6.9e9 < 32 * p < 7.0e9


def test_step_work_counts_every_visible_position():
    shape = wl.tiny_shape()
    b = wl.tiny_batch()
    w = cm.step_work(shape, b.seq_lens, b.q_lens)
    vis = 17 + 33 + 48 + 64 + sum(range(1, 33))
    assert w["attn_flops"] == 4 * shape.n_q * shape.head_dim * vis
    assert w["gemm_flops"] == 2 * 36 * cm.layer_params(shape)
    kv_tok = 2 * shape.n_kv * shape.head_dim * 2
    assert w["kv_read_bytes"] == int(b.seq_lens.sum()) * kv_tok
    assert w["kv_write_bytes"] == 36 * kv_tok


def test_nanobatch_examples_from_pages_are_multiples_of_128():
    e = GOLD["pipeline_70b_split"]
    assert sum(e["sizes"]) == e["b_dense"] and all(s % 128 == 0 for s in e["sizes"])
    s = GOLD["nanobatch_example"]["split"]
    assert s[-1] == GOLD["nanobatch_example"]["b_dense"]


def test_moe_work_counts_top_k_experts_for_flops_and_all_for_bytes():
    """Mixtral-shaped layer, 2048 tokens: FLOPs use the projections plus two
    experts per token, the weight bytes all eight experts (closed forms)."""
    shape = wl.mixtral_shape()
    H, F = shape.hidden, shape.ffn
    attn = H * (32 + 16) * 128 + 32 * 128 * H
    seq = np.array([1] * 10)
    q = np.ones(10, np.int64)
    w = cm.step_work(shape, seq, q)
    assert w["gemm_flops"] == 2 * 10 * (attn + 2 * 3 * H * F)
    assert w["weight_bytes"] == 2 * (attn + 8 * 3 * H * F)
    assert abs(w["weight_bytes"] / 1e9 - 2.90) < 0.01
