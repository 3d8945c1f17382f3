"""The C ABI library loads without a GPU, exports every declared function, and
its host-only plan search returns valid plans."""
import ctypes
import os

import numpy as np
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


def _overlaps(a0, a1, b0, b1):
    return a0 < b1 and b0 < a1


@pytest.mark.parametrize("ab,fb", [([0, 1024, 2048], [0, 1024, 2048]),
                                   ([0, 512, 1024, 1536, 2048], [0, 1024, 2048]),
                                   ([0, 20, 36], [0, 10, 36]),
                                   ([0, 12, 24, 36], [0, 36]),
                                   ([0, 5, 19, 30, 36], [0, 19, 36])])
@pytest.mark.parametrize("layers", [1, 2, 3, 5])
def test_window_schedule_respects_every_dependency(L, ab, fb, layers):
    """The cross-layer window's issue order (the one list the executor runs and
    the search simulates), checked against dependencies derived here from the
    nano-batch bounds: every operation once; O(l, i) after QKV(l, i); FFN(l, j)
    after every O(l, i) sharing rows with it; QKV(l+1, k) after every FFN(l, j)
    sharing rows with it (its input) and after O(l, k) (its q and o rows are
    free again); QKV projections of a layer in row order (a prefill chunk across
    a bound reads the K/V its earlier rows appended); FFN(l+1, j), which
    overwrites layer l's input rows, after their last reader; and every SM only
    for the first QKV and what follows the last attention."""
    T = ab[-1]
    opts = _lib.make_opts(T, ab, fb, executor=_lib.NF_EXEC_STREAMS, attn_sms=64)
    ops = _lib.window_schedule(opts, layers)
    pos = {}
    for k, (kind, l, i, full) in enumerate(ops):
        assert (kind, l, i) not in pos
        pos[(kind, l, i)] = k
    na, nf = len(ab) - 1, len(fb) - 1
    assert len(ops) == layers * (2 * na + nf)
    for l in range(layers):
        for i in range(na):
            assert pos[("o", l, i)] > pos[("qkv", l, i)]
            if i:
                assert pos[("qkv", l, i)] > pos[("qkv", l, i - 1)]
        for j in range(nf):
            for i in range(na):
                if _overlaps(fb[j], fb[j + 1], ab[i], ab[i + 1]):
                    assert pos[("ffn", l, j)] > pos[("o", l, i)]
            if l + 1 < layers:
                for i in range(na):          # layer l's readers of its input rows
                    if _overlaps(fb[j], fb[j + 1], ab[i], ab[i + 1]):
                        assert pos[("ffn", l + 1, j)] > pos[("o", l, i)]
                        assert pos[("ffn", l + 1, j)] > pos[("qkv", l, i)]
        if l + 1 < layers:
            for k in range(na):
                assert pos[("qkv", l + 1, k)] > pos[("o", l, k)]
                for j in range(nf):
                    if _overlaps(fb[j], fb[j + 1], ab[k], ab[k + 1]):
                        assert pos[("qkv", l + 1, k)] > pos[("ffn", l, j)]
    last_o = pos[("o", layers - 1, na - 1)]
    for k, (kind, l, i, full) in enumerate(ops):
        assert full == (1 if (k == 0 or k >= last_o) else 0), (k, kind, l, i)


def test_window_schedule_rejects_bad_bounds(L):
    o = _lib.make_opts(36, [0, 20, 36], [0, 10, 30])
    with pytest.raises(_lib.NanoflowError):
        _lib.window_schedule(o, 2)


def test_search_returns_valid_plans_on_random_batches(L):
    """Random shapes, decode/prefill mixes and layer counts: every plan the
    search returns is valid for its batch (bounds increasing from 0 to T on the
    128-token grid at T >= 1024, counts within NF_MAX_NANO, an SM share below
    the SM count), and nf_plan_predict reproduces the score it was chosen by."""
    rng = np.random.default_rng(7)
    shapes = [wl.tiny_shape(), wl.llama8b_shape(), wl.llama70b_shape()]
    for trial in range(40):
        shape = shapes[trial % 3]
        n_dec = int(rng.integers(0, 1500))
        pq = [int(q) for q in rng.integers(1, 700, int(rng.integers(0 if n_dec else 1, 4)))]
        pp = [int(p) for p in rng.integers(0, 2000, len(pq))]
        ctx = wl.lognormal_contexts(max(n_dec, 1), 600.0, 1.0, 1, 4096, seed=trial)[:n_dec]
        b = wl.make_batch(shape, list(ctx), pq, pp, seed_bt=trial, max_pages=256)
        layers = int(rng.choice([1, 4, 16]))
        sms = int(rng.choice([76, 132, 152]))
        o, t = _lib.plan_search(shape, b, None, sms, n_layers=layers)
        T = b.n_tokens
        _check_plan(o, T, 128 if T >= 1024 else 1)
        assert 0 <= o.attn_sms < sms and t > 0
        assert _lib.plan_predict(shape, b, o, None, sms, layers) == pytest.approx(t, rel=1e-9)


def _profile(tmp_path, name, rp_sms, attn_bps, gemm_factor, sync=25e-6):
    import json
    p = tmp_path / name
    p.write_text(json.dumps({"gemm_flops_per_sm": 11.45e12, "hbm_bps": 6.75e12,
                             "attn_bps_per_sm": 78e9, "stream_sync_s": sync,
                             "rp_sms": rp_sms, "rp_attn_bps_per_sm": attn_bps,
                             "rp_gemm_factor": gemm_factor}))
    return str(p)


def test_search_reads_a_measured_rp_table(L, tmp_path):
    """A profile's R -> P table (attention bytes/s per SM and the GEMM rate kept,
    by attention SM count) drives the overlapped predictions: with no
    interference and fast attention per SM the 70B-shaped window plan is
    predicted faster than with strong interference, the sequential plan does
    not depend on the table, and between two table points the prediction lies
    between those of the points' values."""
    s70 = wl.llama70b_shape()
    b70 = wl.llama70b_batch()
    T = b70.n_tokens
    good = _profile(tmp_path, "good.json", [40, 80], [150e9, 150e9], [1.0, 1.0])
    bad = _profile(tmp_path, "bad.json", [40, 80], [60e9, 60e9], [0.5, 0.5])
    win = _lib.make_opts(T, [0, T // 2, T], [0, T // 2, T], executor=_lib.NF_EXEC_STREAMS,
                         attn_sms=57)
    seq = _lib.make_opts(T)
    assert _lib.plan_predict(s70, b70, win, good, 152, 10) < _lib.plan_predict(s70, b70, win, bad, 152, 10)
    assert _lib.plan_predict(s70, b70, seq, good, 152, 10) == pytest.approx(
        _lib.plan_predict(s70, b70, seq, bad, 152, 10), rel=1e-12)
    mixed = _profile(tmp_path, "mixed.json", [40, 80], [60e9, 150e9], [0.5, 1.0])
    at40 = _lib.make_opts(T, [0, T // 2, T], [0, T // 2, T], executor=_lib.NF_EXEC_STREAMS, attn_sms=40)
    at60 = _lib.make_opts(T, [0, T // 2, T], [0, T // 2, T], executor=_lib.NF_EXEC_STREAMS, attn_sms=60)
    t_bad = _lib.plan_predict(s70, b70, at60, bad, 152, 10)
    t_good = _lib.plan_predict(s70, b70, at60, good, 152, 10)
    t_mid = _lib.plan_predict(s70, b70, at60, mixed, 152, 10)
    assert t_good < t_mid < t_bad
    # clamped below the table's first point: the first point's values
    assert _lib.plan_predict(s70, b70, at40, mixed, 152, 10) == pytest.approx(
        _lib.plan_predict(s70, b70, at40, bad, 152, 10), rel=1e-12)


def test_registered_profile_is_the_default(L, tmp_path):
    """nf_profile_use registers a profile for a shape: a NULL profile then
    means that file, "" the built-in rates; other shapes are unaffected;
    forgetting it restores the built-in rates."""
    s70 = wl.llama70b_shape()
    b70 = wl.llama70b_batch()
    T = b70.n_tokens
    bad = _profile(tmp_path, "bad.json", [40, 80], [60e9, 60e9], [0.5, 0.5])
    win = _lib.make_opts(T, [0, T // 2, T], [0, T // 2, T], executor=_lib.NF_EXEC_STREAMS,
                         attn_sms=57)
    builtin = _lib.plan_predict(s70, b70, win, "", 152, 10)
    assert _lib.plan_predict(s70, b70, win, None, 152, 10) == pytest.approx(builtin, rel=1e-12)
    _lib.profile_use(s70, bad)
    try:
        assert _lib.plan_predict(s70, b70, win, None, 152, 10) == pytest.approx(
            _lib.plan_predict(s70, b70, win, bad, 152, 10), rel=1e-12)
        assert _lib.plan_predict(s70, b70, win, "", 152, 10) == pytest.approx(builtin, rel=1e-12)
        o_reg, _ = _lib.plan_search(s70, b70, None, 152, n_layers=10)
        o_bad, _ = _lib.plan_search(s70, b70, bad, 152, n_layers=10)
        assert _lib.opts_dict(o_reg) == _lib.opts_dict(o_bad)
        s8, b8 = wl.llama8b_shape(), wl.llama8b_batch()
        assert _lib.plan_search(s8, b8, None, 152)[1] == pytest.approx(
            _lib.plan_search(s8, b8, "", 152)[1], rel=1e-12)
    finally:
        _lib.profile_use(s70, None)
    assert _lib.plan_predict(s70, b70, win, None, 152, 10) == pytest.approx(builtin, rel=1e-12)


def test_search_picks_the_fastest_profiled_plan_of_the_same_batch(L, tmp_path):
    """A profile measured on this very batch structure and layer count: the
    search returns its fastest measured plan (an overlapped one only when it
    measured at least 1 % faster than the sequential one), with the profile's
    bounds rule; for another batch it falls back to the model."""
    import json
    s8, b8 = wl.llama8b_shape(), wl.llama8b_batch()
    T = b8.n_tokens
    prof = {"gemm_flops_per_sm": 11.45e12, "hbm_bps": 6.75e12, "attn_bps_per_sm": 78e9,
            "rp_n": [2, 2], "rp_sms": [47, 95], "rp_attn_bps_per_sm": [78e9, 60e9],
            "rp_gemm_factor": [0.8, 0.7], "batch_tokens": T, "batch_decode": b8.n_decode,
            "n_layers": 16, "run_n": [1, 2, 2, 3], "run_sms": [0, 57, 66, 66],
            "run_ms": [26.3, 25.4, 24.9, 25.0]}
    p = tmp_path / "p.json"
    p.write_text(json.dumps(prof))
    o, t = _lib.plan_search(s8, b8, str(p), 152, n_layers=16)
    assert o.executor == _lib.NF_EXEC_STREAMS and o.n_attn == 2 and o.attn_sms == 66
    assert t == pytest.approx(24.9e3, rel=1e-9)
    # the bounds are those the model path generates for 2 nano-batches (the
    # profile measured the search's own plans): a table that makes 2 nano-batches
    # the only good choice there gives the same bounds
    b = list(o.attn_bounds[:3])
    assert b[0] == 0 and b[2] == T and b[1] % 128 == 0 and 0 < b[1] < T
    assert list(o.ffn_bounds[:3]) == b
    model = dict(prof, batch_tokens=-1, stream_sync_s=0.0, rp_n=[2, 2, 3, 3, 4, 4],
                 rp_sms=[47, 95] * 3, rp_attn_bps_per_sm=[200e9] * 6,
                 rp_gemm_factor=[1.0, 1.0, 0.2, 0.2, 0.2, 0.2])
    pm = tmp_path / "m.json"
    pm.write_text(json.dumps(model))
    om, _ = _lib.plan_search(s8, b8, str(pm), 152, n_layers=16)
    assert om.n_attn == 2 and list(om.attn_bounds[:3]) == b
    prof["run_ms"] = [26.3, 26.2, 26.1, 26.2]          # less than 1 % better: sequential
    p.write_text(json.dumps(prof))
    o, t = _lib.plan_search(s8, b8, str(p), 152, n_layers=16)
    assert o.executor == _lib.NF_EXEC_SEQUENTIAL and o.n_attn == 1 and t == pytest.approx(26.3e3)
    o8, _ = _lib.plan_search(s8, b8, str(p), 152, n_layers=8)  # another layer count: the model
    assert _lib.plan_predict(s8, b8, o8, str(p), 152, 8) > 0
