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
