"""The C ABI library loads without a GPU, exports every declared function, and
its host-only plan search returns valid plans."""
import ctypes
import os

import pytest

from nano_intra_device_gb300 import _lib, workload as wl


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        from nano_intra_device_gb300 import build
        build.build()
    return _lib.lib()


def test_header_declares_the_boundary():
    names = _lib.header_functions()
    for must in ("nf_plan_create", "nf_layer_step", "nf_plan_poll", "nf_profile",
                 "nf_plan_search", "nf_attention", "nf_gemm", "nf_step_metadata"):
        assert must in names


def test_library_exports_every_declared_function(L):
    missing = [n for n in _lib.header_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert set(_lib._SIGS) >= set(_lib.header_functions())


def _check_plan(o, T, grid):
    b = list(o.attn_bounds[: o.n_attn + 1])
    assert b[0] == 0 and b[-1] == T and all(x < y for x, y in zip(b, b[1:]))
    assert all(x % grid == 0 for x in b[1:-1])
    f = list(o.ffn_bounds[: o.n_ffn + 1])
    assert f[0] == 0 and f[-1] == T and all(x < y for x, y in zip(f, f[1:]))
    assert 1 <= o.n_attn <= 4


def test_plan_search_llama8b_follows_the_rates(L, tmp_path):
    shape, batch = wl.llama8b_shape(), wl.llama8b_batch()
    # with the measured GB300 rates attention needs most of the SMs to reach HBM
    # speed, so splitting the GPU cannot win: the search keeps one nano-batch
    o, t = _lib.plan_search(shape, batch, None, 152)
    _check_plan(o, batch.n_tokens, 128)
    assert o.n_attn == 1 and o.executor == _lib.NF_EXEC_SEQUENTIAL
    assert 1000.0 < t < 3000.0
    # if one SM streamed attention 1.7x faster and neighbours did not slow each
    # other down, overlap with an SM split would pay
    prof = tmp_path / "fast_attention.json"
    prof.write_text('{"attn_bps_per_sm": 132e9, "hbm_bps": 6.75e12, "gemm_flops_per_sm": 11.45e12, '
                    '"overlap_bw_factor": 0.95, "overlap_gemm_factor": 0.95}')
    o2, t2 = _lib.plan_search(shape, batch, str(prof), 152)
    _check_plan(o2, batch.n_tokens, 128)
    assert o2.n_attn >= 2 and o2.executor == _lib.NF_EXEC_STREAMS
    assert 0 < o2.attn_sms < 152 and t2 < t


def test_plan_search_tiny_is_valid(L):
    shape, batch = wl.tiny_shape(), wl.tiny_batch()
    o, t = _lib.plan_search(shape, batch, None, 152)
    _check_plan(o, batch.n_tokens, 1)
    assert t > 0


def test_invalid_shape_is_rejected_on_host(L):
    shape = wl.Shape(hidden=100, n_q=4, n_kv=2, head_dim=64, ffn=688)
    batch = wl.tiny_batch()
    with pytest.raises(_lib.NanoflowError) as e:
        _lib.Plan(shape, batch, _lib.make_opts(batch.n_tokens))
    assert e.value.code in (_lib.NF_ERR_INVALID_ARG, _lib.NF_ERR_CUDA)


def _bounds(T, k):
    g = 128 if T >= 128 * k else 1
    return [0] + [int(round(T * i / k / g)) * g for i in range(1, k)] + [T]


def test_layer_search_follows_the_measured_regimes(L):
    """The layer-aware search scores the cross-layer window: it keeps the
    sequential plan where attention is bound by HBM or the prefill attention by
    the tensor cores (the 8B-shaped decode stack and a serving-like mix, both
    measured slower when overlapped) and splits the GPU for the GEMM-dominated
    70B-shaped step (measured faster overlapped)."""
    s8, s70 = wl.llama8b_shape(), wl.llama70b_shape()
    dec = wl.make_batch(s8, wl.lognormal_contexts(1024, 600.0, 1.0, 1, 8192, seed=1), [], None,
                        seed_bt=2, max_pages=8192 // 16)
    mix = wl.make_batch(s8, wl.lognormal_contexts(512, 600.0, 1.0, 1, 4096, seed=1),
                        [512, 512, 512], [0, 1024, 2048], seed_bt=2, max_pages=4096 // 16)
    for b in (dec, mix):
        o, t = _lib.plan_search(s8, b, None, 152, n_layers=32)
        _check_plan(o, b.n_tokens, 128)
        assert o.executor == _lib.NF_EXEC_SEQUENTIAL and o.n_attn == 1
    b70 = wl.llama70b_batch()
    o, t = _lib.plan_search(s70, b70, None, 152, n_layers=10)
    _check_plan(o, b70.n_tokens, 128)
    assert o.executor == _lib.NF_EXEC_STREAMS and o.n_attn >= 2
    assert 0.2 * 152 <= o.attn_sms <= 0.45 * 152
    seq = _lib.plan_predict(s70, b70, _lib.make_opts(b70.n_tokens), None, 152, 10)
    assert t < 0.98 * seq          # an overlapped plan must be predicted >= 2 % faster
    # the prediction entry scores a plan exactly as the search did
    assert _lib.plan_predict(s70, b70, o, None, 152, 10) == pytest.approx(t, rel=1e-12)
    o1, t1 = _lib.plan_search(s8, wl.llama8b_batch(), None, 152)
    assert _lib.plan_predict(s8, wl.llama8b_batch(), o1, None, 152, 1) == pytest.approx(t1, rel=1e-12)


def test_plan_predict_model_properties(L):
    """Properties of the time model: sequential layers add up (multi-layer
    predictions share one calibration, the window's); a longer window costs
    more; a prefill chunk costs more after a longer cached prefix; bounds that
    do not describe the batch are rejected."""
    s70, b70 = wl.llama70b_shape(), wl.llama70b_batch()
    T = b70.n_tokens
    seq = _lib.make_opts(T)
    two = _lib.plan_predict(s70, b70, seq, None, 152, 2)
    assert _lib.plan_predict(s70, b70, seq, None, 152, 10) == pytest.approx(5 * two, rel=1e-12)
    o = _lib.make_opts(T, _bounds(T, 2), _bounds(T, 2), executor=_lib.NF_EXEC_STREAMS, attn_sms=46)
    w2 = _lib.plan_predict(s70, b70, o, None, 152, 2)
    w4 = _lib.plan_predict(s70, b70, o, None, 152, 4)
    assert w2 < w4 < 2 * w2
    s8 = wl.llama8b_shape()
    short = wl.make_batch(s8, [100] * 64, [512], [0], seed_bt=2, max_pages=256)
    long_ = wl.make_batch(s8, [100] * 64, [512], [3000], seed_bt=2, max_pages=256)
    ts = _lib.plan_predict(s8, short, _lib.make_opts(short.n_tokens), None, 152, 1)
    tl = _lib.plan_predict(s8, long_, _lib.make_opts(long_.n_tokens), None, 152, 1)
    assert tl > ts
    with pytest.raises(_lib.NanoflowError):
        _lib.plan_predict(s70, b70, _lib.make_opts(T - 1), None, 152, 1)
    with pytest.raises(_lib.NanoflowError):
        _lib.plan_search(s70, b70, None, 152, n_layers=0)


def test_empty_batch_is_rejected_on_host(L):
    shape, batch = wl.tiny_shape(), wl.make_batch(wl.tiny_shape(), [], [], None, max_pages=4)
    with pytest.raises(_lib.NanoflowError) as e:
        _lib.Plan(shape, batch, _lib.make_opts(1))
    assert e.value.code == _lib.NF_ERR_INVALID_ARG
