"""The whole layer step on the GPU through nf_layer_step against the oracle:
every two-way split of the small batch, both executors, the 8B-shaped batch at
1-4 nano-batches on sampled rows, and the host-buffer entry point."""
import itertools
import os
import tempfile

import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
from oracle import layer as orc
from tests.helpers import compare, f64, parity, record, rounding_floor, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Case:
    def __init__(self, shape, batch, gain_std=0.1, seed=0):
        self.shape, self.batch = shape, batch
        self.w = wl.make_weights(shape, seed=seed, gain_std=gain_std)
        self.x = wl.make_x(shape, batch.n_tokens, seed=seed)
        self.kp, self.vp = wl.make_pools(shape, batch, DEV, seed=seed + 3)
        self.wd = to_dev(self.w)
        self.xd = self.x.to(DEV)
        self.bt = torch.from_numpy(batch.block_table).to(DEV)
        self.sl = torch.from_numpy(batch.seq_lens).to(DEV)

    def oracle(self, rows=None, keep=False):
        """(exact, bf16-storage) oracle results for the given rows."""
        w64 = orc.weights_f64(self.w)
        return tuple(orc.layer_step(self.shape, w64, self.x, self.kp, self.vp,
                                    self.batch.block_table, self.batch.seq_lens,
                                    self.batch.q_lens, rows=rows, keep=keep, store=st)
                     for st in (None, "bf16"))

    def run(self, opts):
        kp, vp = self.kp.clone(), self.vp.clone()
        y = torch.empty_like(self.xd)
        plan = _lib.Plan(self.shape, self.batch, opts)
        _lib.layer_step(plan, self.wd, self.xd, kp, vp, self.bt, self.sl, y)
        plan.poll()
        return plan, y, kp, vp


def _check_layer(case, refs, y, kp, vp, rows):
    """y, y - x and the appended K, V of the given rows against both oracles."""
    ex, em = refs
    P = case.shape.page_size
    yg = f64(y)[rows]
    xr = f64(case.x)[rows]
    parity(yg, ex["y"], em["y"], "y")
    # y - x isolates the attention and FFN terms: its relative L2 (the element
    # errors are y's, checked above).  The GPU's y is bf16, so an exact y - x
    # scores rounding_floor on it already; the bound adds that floor to the
    # stated relative L2 (exact: recorded).
    floor = rounding_floor(em["y"], xr)
    compare(yg - xr, em["y"] - xr, "y - x", rel_l2=1e-2 + floor, max_abs=None,
            oracle="bf16-storage")
    record("y - x", (yg - xr) - (ex["y"] - xr), ex["y"] - xr, "exact")
    sl = torch.as_tensor(ex["slots"], device=DEV)
    kg = f64(kp[sl // P, :, sl % P, :])
    vg = f64(vp[sl // P, :, sl % P, :])
    parity(kg, ex["k_new"], em["k_new"], "appended k")
    parity(vg, ex["v_new"], em["v_new"], "appended v")


@pytest.fixture(scope="module")
def tiny():
    c = Case(wl.tiny_shape(), wl.tiny_batch())
    return c, c.oracle(keep=True)


@pytest.mark.parametrize("executor", [_lib.NF_EXEC_SEQUENTIAL, _lib.NF_EXEC_STREAMS])
def test_tiny_every_two_way_split(tiny, executor):
    case, ref = tiny
    T = case.batch.n_tokens
    rows = np.arange(T)
    first = None
    for cut in range(1, T):
        opts = _lib.make_opts(T, [0, cut, T], [0, cut, T], executor=executor, attn_sms=20,
                              kv_chunk=32)
        plan, y, kp, vp = case.run(opts)
        plan.close()
        _check_layer(case, ref, y, kp, vp, rows)
        if first is None:
            first = y.clone()
        else:  # the split never changes the bits
            assert torch.equal(y, first), f"split {cut} changed the result"


def test_tiny_intermediates_and_untouched_pool(tiny):
    case, ref = tiny
    T = case.batch.n_tokens
    s = case.shape
    plan, y, kp, vp = case.run(_lib.make_opts(T, [0, 18, T], kv_chunk=32))
    ex, em = ref
    for buf, key, shp in ((_lib.NF_BUF_N1, "n1", (T, s.hidden)),
                          (_lib.NF_BUF_Q, "q", (T, s.n_q, s.head_dim)),
                          (_lib.NF_BUF_O, "o", (T, s.n_q, s.head_dim)),
                          (_lib.NF_BUF_H, "h", (T, s.hidden)),
                          (_lib.NF_BUF_N2, "n2", (T, s.hidden)),
                          (_lib.NF_BUF_A, "a", (T, s.ffn))):
        parity(f64(plan.buffer(buf, torch.bfloat16, shp)), ex[key], em[key], key)
    plan.close()
    # nothing but this step's slots changed in the pools (NaN poison included)
    P = s.page_size
    mask = torch.ones(case.kp.shape[0] * P, dtype=torch.bool)
    mask[torch.as_tensor(ex["slots"])] = False
    def flat(t):
        return t.permute(0, 2, 1, 3).reshape(-1, s.n_kv * s.head_dim).cpu()[mask]
    assert torch.equal(flat(kp).isnan(), flat(case.kp).isnan())
    assert torch.equal(torch.nan_to_num(flat(kp)), torch.nan_to_num(flat(case.kp)))
    assert torch.equal(torch.nan_to_num(flat(vp)), torch.nan_to_num(flat(case.vp)))


@pytest.mark.parametrize("ab,fb", [([0, 5, 19, 36], [0, 19, 36]), ([0, 1, 2, 3, 36], [0, 36]),
                                   ([0, 4, 36], [0, 2, 4, 30, 36])])
def test_tiny_multiway_splits_both_executors(tiny, ab, fb):
    case, ref = tiny
    T = case.batch.n_tokens
    for ex in (_lib.NF_EXEC_SEQUENTIAL, _lib.NF_EXEC_STREAMS):
        plan, y, kp, vp = case.run(_lib.make_opts(T, ab, fb, executor=ex, attn_sms=16, kv_chunk=16))
        plan.close()
        _check_layer(case, ref, y, kp, vp, np.arange(T))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_tiny_gemm_kinds_match_the_oracle(tiny, mode):
    """gemm_split_k 0: the weight-row kernel (every nano-operation here has at
    most 128 tokens); 1: token-row tiles; 2: token-row tiles split over K."""
    case, ref = tiny
    T = case.batch.n_tokens
    for ab, ex in (([0, T], _lib.NF_EXEC_SEQUENTIAL), ([0, 18, T], _lib.NF_EXEC_STREAMS)):
        plan, y, kp, vp = case.run(_lib.make_opts(T, ab, ab, executor=ex, attn_sms=20,
                                                  kv_chunk=32, gemm_split_k=mode))
        plan.close()
        _check_layer(case, ref, y, kp, vp, np.arange(T))


def test_tiny_host_entry_point_matches_device(tiny):
    case, ref = tiny
    T = case.batch.n_tokens
    opts = _lib.make_opts(T, [0, 18, T], executor=_lib.NF_EXEC_STREAMS, attn_sms=30)
    plan, y, _, _ = case.run(opts)
    kp, vp = case.kp.clone(), case.vp.clone()
    yh = torch.empty(T, case.shape.hidden, dtype=torch.bfloat16).pin_memory()
    _lib.layer_step_host(plan, case.wd, case.x.pin_memory(), kp, vp,
                         torch.from_numpy(case.batch.block_table), torch.from_numpy(case.batch.seq_lens), yh)
    plan.close()
    assert torch.equal(yh, y.cpu())


@pytest.mark.parametrize("executor", [_lib.NF_EXEC_SEQUENTIAL, _lib.NF_EXEC_STREAMS])
def test_host_entry_point_graph_replay_reads_fresh_inputs(tiny, executor):
    """Pinned host buffers: the first call runs directly, the second captures a
    graph and later calls replay it.  Every call must read the host buffers
    anew (a different x each time) and match the device entry point bit for bit;
    after nf_plan_set_batch (another nano-batch split) the old graph is not
    reused."""
    case, _ = tiny
    T, H = case.batch.n_tokens, case.shape.hidden
    bt, sl = torch.from_numpy(case.batch.block_table), torch.from_numpy(case.batch.seq_lens)
    xh = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    yh = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    bth, slh = bt.pin_memory(), sl.pin_memory()
    plan = _lib.Plan(case.shape, case.batch,
                     _lib.make_opts(T, [0, 18, T], executor=executor, attn_sms=30))
    kp, vp = case.kp.clone(), case.vp.clone()   # the same pools every call: one graph
    for i, bounds in enumerate([None] * 4 + [[0, 7, T]] * 2):
        if bounds is not None and i == 4:
            plan.set_batch(case.batch, _lib.make_opts(T, bounds, executor=executor, attn_sms=30))
        x = wl.make_x(case.shape, T, seed=100 + i)
        xh.copy_(x)
        _lib.layer_step_host(plan, case.wd, xh, kp, vp, bth, slh, yh)
        kd, vd = case.kp.clone(), case.vp.clone()
        yd = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        _lib.layer_step(plan, case.wd, x.to(DEV), kd, vd, bt.to(DEV), sl.to(DEV), yd)
        torch.cuda.synchronize()
        assert torch.equal(yh, yd.cpu()), f"call {i}"
    plan.poll()
    plan.close()


@pytest.mark.parametrize("executor", [_lib.NF_EXEC_SEQUENTIAL, _lib.NF_EXEC_STREAMS])
def test_host_entry_point_pipelined_steps(tiny, executor):
    """nf_layer_step_host_async: five steps enqueued back to back (different x,
    separate y buffers; the staging slots alternate), then one wait; each y
    matches the device entry point bit for bit."""
    case, _ = tiny
    T, H = case.batch.n_tokens, case.shape.hidden
    bt, sl = torch.from_numpy(case.batch.block_table), torch.from_numpy(case.batch.seq_lens)
    bth, slh = bt.pin_memory(), sl.pin_memory()
    plan = _lib.Plan(case.shape, case.batch,
                     _lib.make_opts(T, [0, 18, T], executor=executor, attn_sms=30))
    kp, vp = case.kp.clone(), case.vp.clone()
    xs = [wl.make_x(case.shape, T, seed=200 + i).pin_memory() for i in range(5)]
    ys = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(5)]
    for xh, yh in zip(xs, ys):
        _lib.layer_step_host_async(plan, case.wd, xh, kp, vp, bth, slh, yh)
    _lib.host_wait(plan)
    for i, (xh, yh) in enumerate(zip(xs, ys)):
        kd, vd = case.kp.clone(), case.vp.clone()
        yd = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        _lib.layer_step(plan, case.wd, xh.to(DEV), kd, vd, bt.to(DEV), sl.to(DEV), yd)
        torch.cuda.synchronize()
        assert torch.equal(yh, yd.cpu()), f"step {i}"
    plan.poll()
    plan.close()


def test_plan_save_load_and_search(tiny, tmp_path):
    case, ref = tiny
    T = case.batch.n_tokens
    plan = _lib.Plan(case.shape, case.batch, None)          # library search
    o, n = plan.info()
    assert n == T and o.attn_bounds[0] == 0 and o.attn_bounds[o.n_attn] == T
    path = str(tmp_path / "plan.txt")
    _lib.check(_lib.lib().nf_plan_save(plan.h, path.encode()))
    h = _lib.ctypes.c_void_p()
    _lib.check(_lib.lib().nf_plan_load(path.encode(), _lib.ctypes.byref(h)))
    p2 = _lib.Plan.from_handle(h)
    o2, n2 = p2.info()
    assert n2 == T and list(o2.attn_bounds) == list(o.attn_bounds) and o2.attn_sms == o.attn_sms
    kp, vp = case.kp.clone(), case.vp.clone()
    y = torch.empty_like(case.xd)
    _lib.layer_step(p2, case.wd, case.xd, kp, vp, case.bt, case.sl, y)
    p2.poll()
    _check_layer(case, ref, y, kp, vp, np.arange(T))
    plan.close()
    p2.close()


def test_prefill_with_prefix_and_several_chunks():
    shape = wl.tiny_shape()
    b = wl.make_batch(shape, [1, 2, 100, 31], [7, 20, 1], [0, 45, 16], seed_bt=11)
    case = Case(shape, b, gain_std=0.2, seed=4)
    ref = case.oracle()
    T = b.n_tokens
    for ab in ([0, T], [0, 3, 9, 20, T]):
        plan, y, kp, vp = case.run(_lib.make_opts(T, ab, executor=_lib.NF_EXEC_STREAMS,
                                                  attn_sms=12, kv_chunk=48))
        plan.close()
        _check_layer(case, ref, y, kp, vp, np.arange(T))


# ------------------------------------------------------------ 8B-shaped
@pytest.fixture(scope="module")
def big():
    shape, b = wl.llama8b_shape(), wl.llama8b_batch()
    case = Case(shape, b, gain_std=0.0, seed=0)
    T = b.n_tokens
    rng = np.random.default_rng(1)
    ctx = b.seq_lens[: b.n_decode]
    rows = sorted(set([0, 1023, 1024, b.n_decode - 1, int(np.argmax(ctx)), int(np.argmin(ctx))] +
                      rng.choice(b.n_decode, 24, replace=False).tolist() +
                      [b.n_decode, T - 1] + (b.n_decode + rng.choice(256, 6, replace=False)).tolist()))
    return case, rows, case.oracle(rows=rows)


@pytest.mark.parametrize("n,warps,stages", [(1, 8, 4), (2, 8, 4), (3, 14, 4), (4, 12, 4),
                                            (2, 4, 2), (1, 10, 4)])
def test_llama8b_sampled_rows_by_nano_batch_count(big, n, warps, stages):
    case, rows, ref = big
    T = case.batch.n_tokens
    ab = [0] + [int(round(T * i / n / 128)) * 128 for i in range(1, n)] + [T]
    ex = _lib.NF_EXEC_SEQUENTIAL if n == 1 else _lib.NF_EXEC_STREAMS
    plan, y, kp, vp = case.run(_lib.make_opts(T, ab, ab, executor=ex, attn_sms=96,
                                              attn_warps=warps, gemm_stages=stages))
    plan.close()
    _check_layer(case, ref, y, kp, vp, np.asarray(rows))
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("n_tok,nano", [(64, 1), (100, 1), (128, 2), (17, 1), (256, 1)])
def test_llama8b_small_decode_batches(n_tok, nano):
    """Decode-sized batches of the 8B shape: every GEMM on the weight-row kernel
    (token tiles of 64 and 128; head_dim 128 pairs two heads per QKV tile)."""
    shape = wl.llama8b_shape()
    ctx = wl.lognormal_contexts(n_tok, 600.0, 1.0, 1, 8192, seed=n_tok)
    b = wl.make_batch(shape, ctx, [], None, seed_bt=3, slack=0.01, max_pages=8192 // 16)
    case = Case(shape, b, gain_std=0.0, seed=1)
    ref = case.oracle()
    ab = [0, n_tok] if nano == 1 else [0, n_tok // 2, n_tok]
    ex = _lib.NF_EXEC_SEQUENTIAL if nano == 1 else _lib.NF_EXEC_STREAMS
    plan, y, kp, vp = case.run(_lib.make_opts(n_tok, ab, ab, executor=ex, attn_sms=64))
    plan.close()
    _check_layer(case, ref, y, kp, vp, np.arange(n_tok))


def test_expired_device_wait_is_reported_and_the_plan_stays_usable(tiny):
    """Failure detection without a fault: a bounded wait on a barrier that
    nothing arrives at gives up after its limit, nf_plan_poll reports
    NF_ERR_TIMEOUT once (and clears it), and the same plan then runs a layer
    step that matches the oracle; the control (a barrier already arrived at)
    reports nothing."""
    case, ref = tiny
    T = case.batch.n_tokens
    plan = _lib.Plan(case.shape, case.batch, _lib.make_opts(T))
    waited = torch.zeros(1, dtype=torch.int64, device=DEV)
    plan.selftest_wait(1_000_000, arrive=False, waited_ns=waited)      # 1 ms limit
    with pytest.raises(_lib.NanoflowError) as err:
        plan.poll()
    assert err.value.code == _lib.NF_ERR_TIMEOUT
    assert 1_000_000 <= int(waited.item()) < 1_000_000_000
    plan.poll()                                    # reported once: the status was cleared
    plan.selftest_wait(2_000_000_000, arrive=True, waited_ns=waited)
    plan.poll()
    assert int(waited.item()) < 1_000_000
    kp, vp = case.kp.clone(), case.vp.clone()
    y = torch.empty_like(case.xd)
    _lib.layer_step(plan, case.wd, case.xd, kp, vp, case.bt, case.sl, y)
    plan.poll()
    parity(f64(y), ref[0]["y"], ref[1]["y"], "y after an expired wait")
    with pytest.raises(_lib.NanoflowError):
        plan.selftest_wait(0, arrive=True)
    plan.close()


def test_profile_writes_rates_that_the_search_reads(tmp_path):
    """nf_profile on a small shape: every rate the search reads is present and
    physically sane (bandwidths below the measured copy peak's order, shares in
    (0, 1]), and the search accepts the file."""
    import ctypes
    import json
    shape = wl.tiny_shape()
    path = tmp_path / "rates.json"
    s = _lib.make_shape(shape)
    _lib.check(_lib.lib().nf_profile(ctypes.byref(s), 256, 64, str(path).encode()))
    d = json.loads(path.read_text())
    for k in ("gemm_flops_per_sm", "hbm_bps", "attn_bps_per_sm", "overlap_bw_factor",
              "overlap_gemm_factor", "gemm_interference", "gemm_launch_s"):
        assert k in d and d[k] >= 0, k
    assert 0 < d["hbm_bps"] < 2e13 and 0 < d["attn_bps_per_sm"] < 1e12
    assert 0 < d["overlap_bw_factor"] <= 1.5 and 0 < d["overlap_gemm_factor"] <= 1.5
    assert len(d["overlap"]) == 5 and all(0 <= e["u"] <= 1 for e in d["overlap"])
    o, t = _lib.plan_search(shape, wl.tiny_batch(), str(path), _lib.device_sm_count())
    assert o.n_attn >= 1 and t > 0


@pytest.mark.parametrize("decode_ctx,pq,pp,max_pages", [
    ([1], [], [], 4),                       # one token that attends only to itself
    ([], [1], [0], 4),                      # a one-token prompt
    ([64, 16, 17, 33], [], [], 4),          # a row that fills its block table; page edges
    ([64], [3], [61], 4),                   # a chunk that ends on the last slot of the table
])
def test_degenerate_batches_match_the_oracle(decode_ctx, pq, pp, max_pages):
    """Edge cases of the step: a single token, a one-token prompt, rows whose
    KV length fills every page of their block table or sits on a page edge,
    and a prefill chunk whose last token takes the table's last slot."""
    shape = wl.tiny_shape()
    batch = wl.make_batch(shape, decode_ctx, pq, pp, seed_bt=9, max_pages=max_pages)
    case = Case(shape, batch, seed=4)
    ref = case.oracle()
    T = batch.n_tokens
    execs = [(_lib.NF_EXEC_SEQUENTIAL, None)]
    if T >= 2:
        execs.append((_lib.NF_EXEC_STREAMS, [0, T // 2, T]))
    for ex, bounds in execs:
        plan, y, _, _ = case.run(_lib.make_opts(T, bounds, executor=ex, attn_sms=24, kv_chunk=32))
        plan.close()
        parity(f64(y), ref[0]["y"], ref[1]["y"], f"degenerate batch {decode_ctx} {pq}/{pp}, executor {ex}")


def test_trace_records_only_the_selected_operations(tiny):
    """nf_plan_trace_ops: with only attention selected, the trace holds one
    entry per attention nano-batch per step and nothing else; with all
    selected, every operation of the step."""
    case, _ = tiny
    T = case.batch.n_tokens
    plan = _lib.Plan(case.shape, case.batch, _lib.make_opts(T, [0, 18, T]))
    kp, vp = case.kp.clone(), case.vp.clone()
    y = torch.empty_like(case.xd)
    for ops, want in ((["attn"], {"attn"}), (None, {"meta", "qkv", "attn", "oproj", "ffn"})):
        plan.trace_ops(ops)
        plan.trace_enable(2)
        for _ in range(2):
            _lib.layer_step(plan, case.wd, case.xd, kp, vp, case.bt, case.sl, y)
        plan.poll()
        tr = plan.trace_read()
        plan.trace_enable(0)
        assert {e["op"] for e in tr} == want
        assert sum(e["op"] == "attn" for e in tr) == 2 * 2          # 2 nano-batches x 2 steps
        assert all(e["ms"] >= 0 for e in tr)
    plan.close()


def test_step_profile_measures_the_rp_table_and_drives_plan_creation(tmp_path):
    """nf_profile_step on the small batch through 2 layers: the JSON holds the
    R -> P table (attention bytes/s per SM and GEMM rate kept, per nano-batch
    count and SM count, all positive), every profiled plan with its measured
    step time; it is registered, so plan creation without options returns the
    fastest profiled plan, and forgetting it restores the built-in model."""
    import json
    shape, batch = wl.tiny_shape(), wl.tiny_batch()
    path = str(tmp_path / "step.json")
    _lib.profile_step(shape, batch, 2, path)
    try:
        d = json.load(open(path))
        n = len(d["rp_sms"])
        assert n > 0 and len(d["rp_n"]) == n and len(d["rp_gemm_factor"]) == n
        assert all(v > 0 for v in d["rp_attn_bps_per_sm"]) and all(v > 0 for v in d["rp_gemm_factor"])
        assert d["n_layers"] == 2 and d["batch_tokens"] == batch.n_tokens
        assert len(d["run_ms"]) == 1 + 3 * 8 and all(t > 0 for t in d["run_ms"])
        o, t = _lib.plan_search(shape, batch, None, _lib.device_sm_count(), n_layers=2)
        i = min(range(len(d["run_ms"])), key=lambda k: d["run_ms"][k])
        if d["run_n"][i] > 1 and d["run_ms"][i] <= 0.99 * d["run_ms"][0]:
            assert o.n_attn == d["run_n"][i] and o.attn_sms == d["run_sms"][i]
        assert t == pytest.approx(min(d["run_ms"][k] for k in range(len(d["run_ms"]))
                                      if k == 0 or d["run_ms"][k] <= 0.99 * d["run_ms"][0]) * 1e3)
    finally:
        _lib.profile_use(shape, None)
