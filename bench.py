#!/usr/bin/env python
"""Benchmark of the nano-batched decoder-layer step on one GB300 (or N replicas).

Workload: one Llama-3-8B-shaped decoder layer (hidden 4096, 32 q / 8 KV heads,
head_dim 128, FFN 14336, bf16) over a mixed step of T = 2048 tokens: 1792
decode requests with lognormal KV lengths (median 600, sigma 1, clipped to
[1, 8192]) plus one 256-token prefill chunk, KV in 16-token pages under a
random block table.  Synthetic, seeded inputs; random N(0, 0.02) weights.

Metric: tokens/s of the layer step (T / step time, summed over replicas) and
the fraction of the layer roofline, max(FLOPs / bf16 peak, bytes / HBM peak)
divided by the step time.

The JSON line also carries: e2e (the same step through the pipelined
host-buffer entry point: every step copies its inputs in from pinned host
memory and its output back, overlapped with the neighbouring steps' compute), the roofline of the dominant kernel (paged decode
attention, HBM-bound) measured inside the timed steps, clocks sampled during
the timed region, the CPU oracle timed on a bounded sample (cpu_baseline),
and the sequential / nanobatch-only / overlapped comparison, with the same
batch also run through 8 layers, sequential against the two-stream plan that
pipelines nano-batches across layers (ablation_tokens_per_s.cross_layer).

`--impl reference` times the CPU oracle itself on the same workload (bounded
sample per step) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nano_intra_device_gb300 import costmodel as cm  # noqa: E402
from nano_intra_device_gb300 import replicas  # noqa: E402
from nano_intra_device_gb300 import workload as wl  # noqa: E402

METRIC = "tokens/s per GB300 for mixed prefill+decode layer step; % of layer roofline"
WORKLOAD = ("llama3-8b-shaped decoder layer, mixed step of 2048 tokens: 1792 decode "
            "(lognormal KV median 600, sigma 1, clip [1,8192]) + one 256-token prefill chunk, "
            "16-token pages, random block table")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nanoflow", choices=["nanoflow", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--plan", default="auto", help="auto | search | n=<k>,sms=<s>")
    ap.add_argument("--workload", default="layer",
                    choices=["layer", "stack", "70b", "layers8b", "moe", "serve"],
                    help="layer: the single 8B-shaped layer step (default); stack: the 32-layer "
                         "8B-shaped stack with embedding and LM head, decode batches; 70b: ten "
                         "70B-shaped layers over a 4096-token mixed step; layers8b: the layer "
                         "step's 8B-shaped mixed batch through 16 layers; moe: one Mixtral-shaped "
                         "layer (8 experts, top-2) over a 2048-token mixed step; serve: the "
                         "runtime serving synthetic requests on the 32-layer 8B-shaped stack")
    ap.add_argument("--batch", type=int, default=256, help="decode requests of the stack workload")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi samples (every 200 ms) during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = tempfile.mktemp(suffix=".csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        want = vis.split(",")[0] if vis and vis.split(",")[0].isdigit() else None
        if want is not None and any(r[0] == want for r in rows):
            rows = [r for r in rows if r[0] == want]
        elif rows:
            rows = [r for r in rows if r[0] == rows[0][0]]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- workload
class Workload:
    def __init__(self, dev):
        self.shape = wl.llama8b_shape()
        self.batch = wl.llama8b_batch()
        self.T = self.batch.n_tokens
        self.w_cpu = wl.make_weights(self.shape, seed=0)
        self.x_cpu = wl.make_x(self.shape, self.T, seed=0)
        self.dev = dev
        self.w = {k: v.to(dev) for k, v in self.w_cpu.items()}
        self.x = self.x_cpu.to(dev)
        self.kp, self.vp = wl.make_pools(self.shape, self.batch, dev, seed=3)
        self.bt = torch.from_numpy(self.batch.block_table).to(dev)
        self.sl = torch.from_numpy(self.batch.seq_lens).to(dev)
        self.y = torch.empty_like(self.x)
        self.work = cm.step_work(self.shape, self.batch.seq_lens, self.batch.q_lens)
        self.attn_bytes = self._attn_bytes()

    def _attn_bytes(self):
        """Bytes attention must move per step: every token's visible K/V once
        (decode history; prefill rows share their chunk's K/V), q in, o out."""
        s, b = self.shape, self.batch
        kv_tok = 2 * s.n_kv * s.head_dim * 2
        qo = 2 * self.T * s.n_q * s.head_dim * 2
        return int(b.seq_lens.sum()) * kv_tok + qo


def cross_layer_ablation(wk: Workload, stream, L: int = 8, attn_frac: float = 0.45):
    """The step's batch through L layers (the step's weights in every layer,
    each layer its own KV pools), sequential against the two-stream plan with
    2 nano-batches, which pipelines them across layers: per-layer milliseconds
    and tokens/s of each."""
    from nano_intra_device_gb300 import _lib
    T = wk.T
    sms = _lib.device_sm_count()
    pools = [wl.make_pools(wk.shape, wk.batch, wk.dev, seed=200 + l) for l in range(L)]
    la = _lib.LayersArgs([wk.w] * L, pools)
    y = torch.empty_like(wk.x)
    half = int(round(T / 2 / 128)) * 128
    a_sms = int(round(sms * attn_frac))
    out = {"layers": L, "overlap_plan": f"n=2,attn_sms={a_sms}"}
    for name, o in (("sequential", _lib.make_opts(T)),
                    ("overlap", _lib.make_opts(T, [0, half, T], [0, half, T],
                                               executor=_lib.NF_EXEC_STREAMS, attn_sms=a_sms))):
        plan = _lib.Plan(wk.shape, wk.batch, o)
        ms = time_steps(lambda: _lib.layers_step(plan, la, wk.x, wk.bt, wk.sl, y), 5, 3, 1, stream)
        plan.poll()
        plan.close()
        out[f"{name}_ms_per_layer"] = ms / L
        out[f"{name}_tokens_per_s"] = T / (ms / L * 1e-3)
    del pools, la
    torch.cuda.empty_cache()
    return out


def oracle_sample(wk: Workload, n_decode: int, n_prefill: int, seed: int = 0):
    """A bounded piece of the workload the CPU oracle can run: n_decode random
    decode requests plus the first n_prefill rows of the prefill chunk, with
    only their pages copied to host memory."""
    b, s = wk.batch, wk.shape
    rng = np.random.default_rng(seed)
    dec = sorted(rng.choice(b.n_decode, n_decode, replace=False).tolist())
    seqs = dec + ([b.n_decode] if n_prefill > 0 else [])
    P = s.page_size
    pages, bt_rows = [], []
    for sq in seqs:
        n = (int(b.seq_lens[sq]) + P - 1) // P
        ids = b.block_table[sq, :n]
        bt_rows.append(list(range(len(pages), len(pages) + n)))
        pages.extend(ids.tolist())
    width = max(len(r) for r in bt_rows)
    bt = np.full((len(seqs), width), -1, np.int32)
    for i, r in enumerate(bt_rows):
        bt[i, :len(r)] = r
    idx = torch.as_tensor(pages, device=wk.kp.device)
    kp = wk.kp[idx].cpu()
    vp = wk.vp[idx].cpu()
    sl = b.seq_lens[seqs].astype(np.int32)
    ql = b.q_lens[seqs].astype(np.int32)
    tok = dec + (list(range(b.n_decode, b.n_decode + int(b.q_lens[b.n_decode]))) if n_prefill else [])
    x = wk.x_cpu[torch.as_tensor(tok)]
    rows = list(range(len(dec))) + list(range(len(dec), len(dec) + n_prefill))
    return dict(shape=s, w=wk.w_cpu, x=x, kp=kp, vp=vp, bt=bt, sl=sl, ql=ql, rows=rows,
                desc=f"{n_decode} random decode rows + first {n_prefill} prefill rows of the "
                     f"8B-shaped step, one oracle call (float64 weights converted per call)")


def time_oracle(sample):
    from oracle import layer as orc   # CPU baseline leg only
    t0 = time.perf_counter()
    orc.layer_step(sample["shape"], orc.weights_f64(sample["w"]), sample["x"], sample["kp"],
                   sample["vp"], sample["bt"], sample["sl"], sample["ql"], rows=sample["rows"])
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ---------------------------------------------------------------- replicas
def dist_setup(n):
    """One process per GPU, each an independent replica (no data-path collective)."""
    return replicas.setup()


def barrier(world):
    replicas.barrier(world)


def max_over_ranks(v, world):
    return replicas.max_over_ranks(v, world)


# --------------------------------------------------------------- reference
def run_reference(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wk = Workload(dev)
    sample = oracle_sample(wk, 24, 8, seed=1)
    n_tok = len(sample["rows"])
    for _ in range(args.warmup):
        time_oracle(sample)
    ts = [time_oracle(sample) for _ in range(args.steps)]
    t = sum(ts) / len(ts)
    v = n_tok / t
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step_sample": n_tok},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample["desc"]},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- main
def step_profile(shape, batch, n_layers):
    """nf_profile_step on this batch structure (the R -> P table measured in
    traced steps; registered for the shape, so plan creation without options
    and the searches use it): its wall time, and each profiled plan's measured
    against predicted step time."""
    import tempfile
    from nano_intra_device_gb300 import _lib
    path = os.path.join(tempfile.mkdtemp(prefix="nf_profile_"), "step_profile.json")
    t0 = time.perf_counter()
    _lib.profile_step(shape, batch, n_layers, path)
    d = json.load(open(path))
    runs = d.get("runs", [])
    err = [abs(r["predicted_ms"] / r["measured_ms"] - 1) for r in runs if r["measured_ms"] > 0]
    return {"seconds": round(time.perf_counter() - t0, 2), "layers_profiled": d.get("n_layers"),
            "rp_sms": d.get("rp_sms"), "rp_attn_gbs_per_sm": [round(x / 1e9, 1) for x in d.get("rp_attn_bps_per_sm", [])],
            "rp_gemm_factor": [round(x, 3) for x in d.get("rp_gemm_factor", [])],
            "stream_sync_us": round(d.get("stream_sync_s", 0) * 1e6, 1),
            "model_error_mean": round(sum(err) / max(1, len(err)), 4),
            "model_error_max": round(max(err, default=0), 4),
            "runs": [[r["n_attn"], r["attn_sms"], round(r["measured_ms"], 3), round(r["predicted_ms"], 3)]
                     for r in runs]}


def time_steps(fn, steps, warmup, world, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / steps


def run_stack(args):
    """32-layer 8B-shaped stack, decode-only batch, eager and CUDA-graph replay."""
    from nano_intra_device_gb300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shape = wl.llama8b_shape()
    L, vocab, B = 32, 128256, args.batch
    ctx = wl.lognormal_contexts(B, 600.0, 1.0, 1, 8192, seed=1)
    batch = wl.make_batch(shape, ctx, [], None, seed_bt=2, slack=0.01, max_pages=8192 // 16)
    g = torch.Generator(device=dev).manual_seed(0)

    def rn(*sz, std=0.02):
        return (torch.randn(*sz, generator=g, device=dev) * std).to(torch.bfloat16)
    H, F = shape.hidden, shape.ffn
    layers = [{"w_qkv": rn(shape.qkv_rows, H), "w_o": rn(H, shape.n_q * shape.head_dim),
               "w_gate_up": rn(2 * F, H), "w_down": rn(H, F),
               "norm1": torch.ones(H, dtype=torch.bfloat16, device=dev),
               "norm2": torch.ones(H, dtype=torch.bfloat16, device=dev)} for _ in range(L)]
    embed, lm_head = rn(vocab, H, std=1.0), rn(vocab, H)
    norm_f = torch.ones(H, dtype=torch.bfloat16, device=dev)
    pools = [wl.make_pools(shape, batch, dev, seed=100 + l) for l in range(L)]
    tokens = torch.randint(0, vocab, (B,), generator=g, device=dev, dtype=torch.int32)
    bt = torch.from_numpy(batch.block_table).to(dev)
    sl = torch.from_numpy(batch.seq_lens).to(dev)
    logits = torch.empty(B, vocab, dtype=torch.bfloat16, device=dev)
    opts = None  # the library's search
    if args.plan.startswith("n="):
        # a forced two-stream plan: with the same nano-batches in both groups the
        # stack runs the cross-layer window
        kv = dict(p.split("=") for p in args.plan.split(","))
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        n, a_sms = int(kv["n"]), int(kv.get("sms", sms * 5 // 8))
        T = batch.n_tokens
        g = 128 if T >= 128 * n else 1
        ab = [0] + [max(1, int(round(T * i / n / g))) * g for i in range(1, n)] + [T]
        opts = _lib.make_opts(T, ab, ab, executor=_lib.NF_EXEC_STREAMS, attn_sms=a_sms)
    plan = _lib.Plan(shape, batch, opts)
    sa = _lib.StackArgs(embed, norm_f, lm_head, layers, pools)
    stream = torch.cuda.current_stream()
    step = lambda: _lib.stack_step(plan, sa, tokens, bt, sl, logits)  # noqa: E731
    eager_ms = time_steps(step, args.steps, args.warmup, 1, stream)
    graph = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    s2.wait_stream(stream)
    with torch.cuda.stream(s2):
        step()
    stream.wait_stream(s2)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step()
    graph_ms = time_steps(graph.replay, args.steps, args.warmup, 1, stream)
    plan.poll()
    pk = peaks()
    work = cm.stack_work(shape, batch.seq_lens, batch.q_lens, L, vocab)
    rf = cm.roofline_time(work, pk["bf16_tflops_sustained"] * 1e12, pk["hbm_gbs"] * 1e9)
    ms = min(eager_ms, graph_ms)
    line = {"metric": "end-to-end layer-stack tokens/s (decode step, 32 layers + LM head)",
            "value": B / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "eager_ms": eager_ms, "graph_ms": graph_ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"llama3-8b-shaped 32-layer stack, vocab {vocab}, {B} decode "
                                   "requests (lognormal KV median 600, sigma 1, clip [1,8192])",
                       "kv_read_gb_per_step": L * work["layer"]["kv_read_bytes"] / 1e9,
                       "plan": _lib.opts_dict(plan.info()[0])},
            "stack_roofline": {"frac": rf["t_roof"] / (ms * 1e-3), "t_roof_ms": rf["t_roof"] * 1e3,
                               "bound": rf["bound"], "flops": work["flops"], "bytes": work["bytes"]}}
    print(json.dumps(line), flush=True)
    plan.close()


def run_layers_workload(args, shape, batch, L, metric, workload, fracs_by_n):
    """L layers of `shape`, each with its own weights and KV pools, over one
    mixed step through nf_layers_step.  Plans: the layer-aware search's pick,
    sequential, and two-stream candidates (n attention nano-batches, n_ffn FFN
    ones, attention on a fraction of the SMs), each timed; the fastest is
    reported, with every candidate's time and the search model's prediction."""
    from nano_intra_device_gb300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T, H, F = batch.n_tokens, shape.hidden, shape.ffn
    # the step profile first: it allocates (and frees) its own weights and pool
    prof = step_profile(shape, batch, L)
    g = torch.Generator(device=dev).manual_seed(0)

    def rn(*sz, std=0.02):
        return (torch.randn(*sz, generator=g, device=dev) * std).to(torch.bfloat16)
    layers = [{"w_qkv": rn(shape.qkv_rows, H), "w_o": rn(H, shape.n_q * shape.head_dim),
               "w_gate_up": rn(2 * F, H), "w_down": rn(H, F),
               "norm1": torch.ones(H, dtype=torch.bfloat16, device=dev),
               "norm2": torch.ones(H, dtype=torch.bfloat16, device=dev)} for _ in range(L)]
    pools = [wl.make_pools(shape, batch, dev, seed=100 + l) for l in range(L)]
    x = (torch.randn(T, H, generator=g, device=dev)).to(torch.bfloat16)
    y = torch.empty_like(x)
    bt = torch.from_numpy(batch.block_table).to(dev)
    sl = torch.from_numpy(batch.seq_lens).to(dev)
    la = _lib.LayersArgs(layers, pools)
    stream = torch.cuda.current_stream()
    sms = _lib.device_sm_count()
    # the two-stream candidates run the cross-layer window (no join between
    # layers); "search" is the layer-aware search's pick (it scores the window
    # over all the layers), and each candidate's model prediction is reported
    # beside its measured time
    searched, _ = _lib.plan_search(shape, batch, None, sms, n_layers=L)   # the profile's rates
    builtin, _ = _lib.plan_search(shape, batch, "", sms, n_layers=L)      # the built-in rates
    cands = [("search", searched), ("search_builtin", builtin), ("sequential", _lib.make_opts(T))]

    def bounds(n):
        return [0] + [int(round(T * i / n / 128)) * 128 for i in range(1, n)] + [T]
    for (n, nf), fracs in fracs_by_n.items():
        for f in fracs:
            a_sms = int(round(sms * f))
            name = f"n={n},attn_sms={a_sms}" + (f",n_ffn={nf}" if nf != n else "")
            cands.append((name, _lib.make_opts(T, bounds(n), bounds(nf),
                                               executor=_lib.NF_EXEC_STREAMS, attn_sms=a_sms)))
    tried, model = {}, {}
    for name, o in cands:
        plan = _lib.Plan(shape, batch, o)
        tried[name] = (time_steps(lambda: _lib.layers_step(plan, la, x, bt, sl, y), 3, 1, 1, stream),
                       _lib.opts_dict(plan.info()[0]))
        model[name] = round(_lib.plan_predict(shape, batch, plan.info()[0], None, sms, L) / 1e3, 3)
        plan.poll()
        plan.close()
    best = min(tried, key=lambda k: tried[k][0])
    plan = _lib.Plan(shape, batch, dict(cands)[best])
    clocks = Clocks()
    for _ in range(args.warmup):
        _lib.layers_step(plan, la, x, bt, sl, y)
    torch.cuda.synchronize()
    clocks.start()
    ms = time_steps(lambda: _lib.layers_step(plan, la, x, bt, sl, y), args.steps, 0, 1, stream)
    clk = clocks.stop()
    plan.poll()
    pk = peaks()
    lw = cm.step_work(shape, batch.seq_lens, batch.q_lens)
    rf = cm.roofline_time({"flops": L * lw["flops"], "bytes": L * lw["bytes"]},
                          pk["bf16_tflops_sustained"] * 1e12, pk["hbm_gbs"] * 1e9)
    line = {"metric": metric,
            "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_layer": ms / L,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "clocks": clk,
            "config": {"workload": workload, "layers": L,
                       "kv_read_gb_per_step": L * lw["kv_read_bytes"] / 1e9,
                       "plan": dict(tried[best][1], chosen=best)},
            f"roofline_{L}_layers": {"frac": rf["t_roof"] / (ms * 1e-3), "t_roof_ms": rf["t_roof"] * 1e3,
                                     "t_flop_ms": rf["t_flop"] * 1e3, "t_byte_ms": rf["t_byte"] * 1e3,
                                     "bound": rf["bound"]},
            "candidates_ms": {k: round(v[0], 3) for k, v in tried.items()},
            "candidates_model_ms": model,
            "search": {"pick": tried["search"][1], "pick_over_best": round(tried["search"][0] / tried[best][0], 4),
                       "builtin_pick_over_best": round(tried["search_builtin"][0] / tried[best][0], 4),
                       "step_profile": prof}}
    print(json.dumps(line), flush=True)
    plan.close()


def run_70b(args):
    """Ten LLaMA-2-70B-shaped layers over one 4096-token mixed step (3584 decode
    requests, lognormal KV median 1000 clipped to [1, 4096], plus a 512-token
    prefill chunk).  Measured on GB300 the optimum is 2 nano-batches with 29-31 %
    of the SMs on attention, and the step time moves steeply with that share;
    the pages' 70B structure (4 attention nano-batches, 2 FFN ones) is among the
    candidates."""
    run_layers_workload(
        args, wl.llama70b_shape(), wl.llama70b_batch(), 10,
        "tokens/s per GB300 for a 10-layer 70B-shaped mixed step; % of its roofline",
        "llama2-70b-shaped, 10 layers, 4096-token step: 3584 decode (lognormal KV median 1000, "
        "sigma 1, clip [1,4096]) + one 512-token prefill chunk, 16-token pages",
        {(2, 2): (0.27, 0.28, 0.29, 0.30, 0.31, 0.32), (3, 3): (0.26, 0.27), (4, 2): (0.26, 0.29)})


def run_layers8b(args):
    """The 8B-shaped mixed batch of the layer step (1792 decode requests +
    one 256-token prefill chunk) through 16 layers, each with its own weights
    and KV pools: the layer step as a model runs it, where the two-stream
    executor can pipeline nano-batches across layers.  Measured on GB300 the
    optimum is 2 nano-batches with ~42 % of the SMs on attention."""
    run_layers_workload(
        args, wl.llama8b_shape(), wl.llama8b_batch(), 16,
        "tokens/s per GB300 for the 8B-shaped mixed batch through 16 layers; % of its roofline",
        "llama3-8b-shaped, 16 layers, 2048-token step: 1792 decode (lognormal KV) + one "
        "256-token prefill chunk, 16-token pages",
        {(2, 2): (0.37, 0.39, 0.42, 0.45, 0.47, 0.50), (3, 3): (0.42, 0.46)})


def run_moe(args):
    """One Mixtral-shaped layer (8 SwiGLU experts of FFN 14336, top-2 routing
    from N(0, 1) router logits) over a 2048-token mixed step: 1920 decode
    requests (lognormal KV median 600, sigma 1, clip [1, 8192]) plus a 128-token
    prefill chunk.  Plans: search, sequential and SM-split overlap candidates,
    each timed; the fastest is reported."""
    from nano_intra_device_gb300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shape, batch = wl.mixtral_shape(), wl.moe_batch()
    T, H, F, E = batch.n_tokens, shape.hidden, shape.ffn, shape.n_experts
    g = torch.Generator(device=dev).manual_seed(0)

    def rn(*sz, std=0.02):
        return (torch.randn(*sz, generator=g, device=dev) * std).to(torch.bfloat16)
    w = {"w_qkv": rn(shape.qkv_rows, H), "w_o": rn(H, shape.n_q * shape.head_dim),
         "norm1": torch.ones(H, dtype=torch.bfloat16, device=dev),
         "norm2": torch.ones(H, dtype=torch.bfloat16, device=dev),
         "w_experts_gate_up": torch.cat([rn(1, 2 * F, H) for _ in range(E)]),
         "w_experts_down": torch.cat([rn(1, H, F) for _ in range(E)]),
         "router_logits": torch.randn(T, E, generator=g, device=dev)}
    kp, vp = wl.make_pools(shape, batch, dev, seed=3)
    x = torch.randn(T, H, generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty_like(x)
    bt = torch.from_numpy(batch.block_table).to(dev)
    sl = torch.from_numpy(batch.seq_lens).to(dev)
    stream = torch.cuda.current_stream()
    sms = _lib.device_sm_count()
    prof = step_profile(shape, batch, 1)
    cands = [("search", None), ("search_builtin", _lib.plan_search(shape, batch, "", sms)[0]),
             ("sequential", _lib.make_opts(T))]
    for n in (2, 3):
        ab = [0] + [int(round(T * i / n / 128)) * 128 for i in range(1, n)] + [T]
        for a_sms in (sms * 6 // 16, sms * 8 // 16, sms * 10 // 16):
            cands.append((f"n={n},attn_sms={a_sms}",
                          _lib.make_opts(T, ab, ab, executor=_lib.NF_EXEC_STREAMS, attn_sms=a_sms)))
    tried, plans = {}, {}
    for name, o in cands:
        plan = _lib.Plan(shape, batch, o)
        tried[name] = time_steps(lambda: _lib.layer_step(plan, w, x, kp, vp, bt, sl, y), 5, 2, 1,
                                 stream)
        plan.poll()
        plans[name] = plan
    best = min(tried, key=tried.get)
    plan = plans.pop(best)
    for p in plans.values():
        p.close()
    clocks = Clocks()
    for _ in range(args.warmup):
        _lib.layer_step(plan, w, x, kp, vp, bt, sl, y)
    torch.cuda.synchronize()
    clocks.start()
    ms = time_steps(lambda: _lib.layer_step(plan, w, x, kp, vp, bt, sl, y), args.steps, 0, 1, stream)
    clk = clocks.stop()
    plan.poll()
    # the per-operation breakdown from three more steps, traced (events between
    # kernels would perturb the timed ones)
    plan.trace_enable(3)
    for _ in range(3):
        _lib.layer_step(plan, w, x, kp, vp, bt, sl, y)
    plan.poll()
    trace = plan.trace_read()
    plan.trace_enable(0)
    ops = {}
    for e in trace:
        ops.setdefault(f"{e['op']}{e['nano']}", []).append(e["ms"])
    pk = peaks()
    work = cm.step_work(shape, batch.seq_lens, batch.q_lens)
    rf = cm.roofline_time(work, pk["bf16_tflops_sustained"] * 1e12, pk["hbm_gbs"] * 1e9)
    line = {"metric": "tokens/s per GB300 for a Mixtral-shaped MoE layer step; % of layer roofline",
            "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "clocks": clk,
            "config": {"workload": "mixtral-8x7b-shaped layer (8 experts x FFN 14336, top-2 from "
                                   "N(0,1) router logits), 2048-token step: 1920 decode (lognormal "
                                   "KV median 600, sigma 1, clip [1,8192]) + one 128-token prefill "
                                   "chunk, 16-token pages",
                       "kv_read_gb_per_step": work["kv_read_bytes"] / 1e9,
                       "plan": dict(_lib.opts_dict(plan.info()[0]), chosen=best)},
            "layer_roofline": {"frac": rf["t_roof"] / (ms * 1e-3), "t_roof_ms": rf["t_roof"] * 1e3,
                               "t_flop_ms": rf["t_flop"] * 1e3, "t_byte_ms": rf["t_byte"] * 1e3,
                               "bound": rf["bound"], "flops": work["flops"], "bytes": work["bytes"]},
            "ops_ms": {k: round(float(np.mean(v)), 4) for k, v in ops.items()},
            "candidates_ms": {k: round(v, 3) for k, v in tried.items()},
            "search": {"pick_over_best": round(tried["search"] / tried[best], 4),
                       "builtin_pick_over_best": round(tried["search_builtin"] / tried[best], 4),
                       "step_profile": prof}}
    print(json.dumps(line), flush=True)
    plan.close()


def run_serve(args):
    """The runtime (batch formation, async scheduling, pages, re-planning) serving
    synthetic requests on the 32-layer 8B-shaped stack with a 128256-token
    vocabulary: prompts lognormal (median 512, sigma 1, clip [16, 4096]), outputs
    lognormal (median 200, sigma 0.7, clip [16, 1024]), enough requests queued
    that every iteration is full.  After warm-up iterations, args.steps
    iterations are timed (host and device, the runtime's own loop)."""
    from nano_intra_device_gb300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shape = wl.llama8b_shape()
    L, vocab, B = 32, 128256, 2048
    max_requests, max_pages, num_pages = 768, 320, 40000
    g = torch.Generator(device=dev).manual_seed(0)

    def rn(*sz, std=0.02):
        return (torch.randn(*sz, generator=g, device=dev) * std).to(torch.bfloat16)
    H, F = shape.hidden, shape.ffn
    layers = [{"w_qkv": rn(shape.qkv_rows, H), "w_o": rn(H, shape.n_q * shape.head_dim),
               "w_gate_up": rn(2 * F, H), "w_down": rn(H, F),
               "norm1": torch.ones(H, dtype=torch.bfloat16, device=dev),
               "norm2": torch.ones(H, dtype=torch.bfloat16, device=dev)} for _ in range(L)]
    embed, lm_head = rn(vocab, H, std=1.0), rn(vocab, H)
    norm_f = torch.ones(H, dtype=torch.bfloat16, device=dev)
    pools = [(torch.zeros(num_pages, shape.n_kv, 16, shape.head_dim, dtype=torch.bfloat16, device=dev),
              torch.zeros(num_pages, shape.n_kv, 16, shape.head_dim, dtype=torch.bfloat16, device=dev))
             for _ in range(L)]
    sa = _lib.StackArgs(embed, norm_f, lm_head, layers, pools)
    rt = _lib.Runtime(shape, B, max_requests, max_pages, num_pages, vocab, eos_token=-1,
                      replan_threshold=0.1)
    rng = np.random.default_rng(5)
    n_req = 3000
    plens = np.clip(np.round(np.exp(np.log(512) + rng.standard_normal(n_req))), 16, 4096).astype(int)
    olens = np.clip(np.round(np.exp(np.log(200) + 0.7 * rng.standard_normal(n_req))), 16, 1024).astype(int)
    for pl, ol in zip(plens, olens):
        rt.submit(rng.integers(0, vocab, int(pl)).tolist(), int(ol))
    stream = torch.cuda.current_stream()
    # warm-up long enough for the admitted requests to finish their prompts, so
    # that the timed iterations see the steady decode share
    warm = max(args.warmup, 400)
    for _ in range(warm):
        rt.step(sa, stream)
    torch.cuda.synchronize()
    clocks = Clocks()
    clocks.start()
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    tok = dec = replans = full = 0
    for _ in range(args.steps):
        b = rt.step(sa, stream)
        tok += b["n_tokens"]
        dec += b["n_decode"]
        replans += b["replanned"]
        full += b["n_tokens"] == B
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    rt.sync()
    dev_s = e0.elapsed_time(e1) * 1e-3
    waiting, active, free_pages = rt.counts()
    line = {"metric": "serving-loop tokens/s (runtime + 32-layer 8B-shaped stack, greedy decode)",
            "value": tok / wall, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": warm, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "clocks": clk,
            "config": {"workload": f"runtime, b_dense {B}, {L} layers, vocab {vocab}, {n_req} queued "
                                   "requests: prompts lognormal median 512 sigma 1 clip [16,4096], "
                                   "outputs lognormal median 200 sigma 0.7 clip [16,1024]",
                       "max_requests": max_requests, "num_pages": num_pages},
            "decode_tokens_per_s": dec / wall, "device_ms_per_step": dev_s / args.steps * 1e3,
            "full_iterations": full, "replans": replans,
            "state_after": {"waiting": waiting, "active": active, "free_pages": free_pages}}
    print(json.dumps(line), flush=True)
    rt.close()


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "stack":
        return run_stack(args)
    if args.workload == "70b":
        return run_70b(args)
    if args.workload == "layers8b":
        return run_layers8b(args)
    if args.workload == "moe":
        return run_moe(args)
    if args.workload == "serve":
        return run_serve(args)
    from nano_intra_device_gb300 import _lib

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _lib.lib()
    wk = Workload(dev)
    T = wk.T
    stream = torch.cuda.current_stream()
    pk = peaks()
    sms = _lib.device_sm_count()

    def make_plan(opts):
        return _lib.Plan(wk.shape, wk.batch, opts)

    def stepper(plan):
        return lambda: _lib.layer_step(plan, wk.w, wk.x, wk.kp, wk.vp, wk.bt, wk.sl, wk.y)

    # candidates: the library's search, then measured neighbours (real timing of
    # the best predicted plans, the last step of the plan search)
    prof = step_profile(wk.shape, wk.batch, 1) if args.plan == "auto" else None
    searched = make_plan(None)   # plan creation without options: the profile's rates
    so, _ = searched.info()
    cands = [("search", searched), ("sequential", make_plan(_lib.make_opts(T)))]
    if prof is not None:
        cands.append(("search_builtin", make_plan(_lib.plan_search(wk.shape, wk.batch, "", sms)[0])))
    if args.plan == "auto":
        for n in (2, 3, 4):
            ab = [0] + [int(round(T * i / n / 128)) * 128 for i in range(1, n)] + [T]
            for a_sms in (sms * 7 // 16, sms * 8 // 16, sms * 9 // 16, sms * 10 // 16):
                o = _lib.make_opts(T, ab, ab, executor=_lib.NF_EXEC_STREAMS, attn_sms=a_sms)
                cands.append((f"n={n},attn_sms={a_sms}", make_plan(o)))
    elif args.plan.startswith("n="):
        kv = dict(p.split("=") for p in args.plan.split(","))
        n, a_sms = int(kv["n"]), int(kv.get("sms", sms * 5 // 8))
        ab = [0] + [int(round(T * i / n / 128)) * 128 for i in range(1, n)] + [T]
        cands = [(args.plan, make_plan(_lib.make_opts(T, ab, ab, executor=_lib.NF_EXEC_STREAMS,
                                                      attn_sms=a_sms)))]
    tried = {}
    for name, p in cands:
        tried[name] = time_steps(stepper(p), 5, 2, 1, stream)
        p.poll()
    best_name = min(tried, key=tried.get)
    plan = dict(cands)[best_name]
    # the fastest overlapped candidate (two streams, n >= 2), for the ablation
    ovl = [nm for nm in tried if nm.startswith("n=")]
    ovl_name = min(ovl, key=tried.get) if ovl else None
    ovl_opts = dict(cands)[ovl_name].info()[0] if ovl_name else None
    for name, p in cands:
        if p is not plan:
            p.close()
    po, _ = plan.info()

    # timed region: events around the attention only (the dominant kernel's
    # duration for the roofline); an event between two kernels would keep the
    # second from starting as a programmatic dependent of the first
    clocks = Clocks()
    plan.trace_ops(["attn"])
    plan.trace_enable(args.steps)
    for _ in range(args.warmup):
        stepper(plan)()
    torch.cuda.synchronize()
    plan.trace_enable(args.steps)      # record exactly the timed steps
    clocks.start()
    ms = time_steps(stepper(plan), args.steps, 0, world, stream)
    clk = clocks.stop()
    plan.poll()
    trace = plan.trace_read()
    plan.trace_enable(0)
    # every operation of two more steps, for the timeline (outside the timed region)
    plan.trace_ops(None)
    plan.trace_enable(2)
    for _ in range(2):
        stepper(plan)()
    plan.poll()
    full_trace = plan.trace_read()
    plan.trace_enable(0)
    ms = max_over_ranks(ms, world)
    value = T * world / (ms * 1e-3)

    # roofline of the dominant kernel (attention) from the timed steps
    attn = [e["ms"] for e in trace if e["op"] == "attn"]
    n_attn = po.n_attn
    attn_bytes_per_launch = wk.attn_bytes / n_attn
    attn_ms = sum(attn) / max(1, len(attn))
    achieved = attn_bytes_per_launch / (attn_ms * 1e-3) / 1e9
    src_name = "attn_mma.cu"
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath)).get(src_name, {})
        src = open(os.path.join(ROOT, "nano_intra_device_gb300", "csrc", src_name), "rb").read()
        if tj.get("source_sha256") == hashlib.sha256(src).hexdigest():
            traffic = tj.get("bytes_per_launch", {}).get(str(n_attn))
    kname = "attn_mma_kernel (paged GQA attention, tensor cores)"
    roof = {"bound": "hbm", "kernel": kname,
            "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
            "peak_source": pk["source"] + " hbm_gbs (copy)",
            "algorithmic_bytes_per_launch": attn_bytes_per_launch, "launches_per_step": n_attn,
            "avg_launch_ms": attn_ms}

    # layer roofline
    rf = cm.roofline_time(wk.work, pk["bf16_tflops_sustained"] * 1e12, pk["hbm_gbs"] * 1e9)
    layer_frac = rf["t_roof"] / (ms * 1e-3)

    # timeline summary of the last fully traced step: overlap of attention with GEMMs
    last = max((e["step"] for e in full_trace), default=0)
    ev = [e for e in full_trace if e["step"] == last]
    a_iv = [(e["start_ms"], e["start_ms"] + e["ms"]) for e in ev if e["op"] == "attn"]
    g_iv = [(e["start_ms"], e["start_ms"] + e["ms"]) for e in ev if e["op"] in ("qkv", "oproj", "ffn")]
    overlap = sum(max(0.0, min(a1, g1) - max(a0, g0)) for a0, a1 in a_iv for g0, g1 in g_iv)
    timeline = [{k: (round(v, 4) if isinstance(v, float) else v) for k, v in e.items() if k != "step"}
                for e in sorted(ev, key=lambda e: e["start_ms"])]

    # e2e through the host-buffer entry point: every step copies its inputs in
    # from pinned host memory and its y out; nf_layer_step_host_async pipelines
    # them (a step's copies overlap the neighbouring steps' compute), and the
    # clock stops once the last y is on the host
    xh = wk.x_cpu.pin_memory()
    yhs = [torch.empty_like(xh).pin_memory() for _ in range(2)]
    bth = torch.from_numpy(wk.batch.block_table).pin_memory()
    slh = torch.from_numpy(wk.batch.seq_lens).pin_memory()
    for i in range(max(1, args.warmup)):
        _lib.layer_step_host_async(plan, wk.w, xh, wk.kp, wk.vp, bth, slh, yhs[i % 2])
    _lib.host_wait(plan)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _lib.layer_step_host_async(plan, wk.w, xh, wk.kp, wk.vp, bth, slh, yhs[i % 2])
    _lib.host_wait(plan)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world)
    h2d = xh.numel() * 2 + bth.numel() * 4 + slh.numel() * 4
    d2h = yhs[0].numel() * 2

    # ablation: sequential, nanobatch-only, overlapped (same kernels)
    # (the pages' Fig. 9 ablation: non-overlap, nanobatch-only, overlap): the
    # sequential plan; the best overlapped candidate's split run on one stream;
    # that candidate itself.  Each timed the same way, 10 steps after 3.
    ablation = None
    if not args.no_ablation:
        ablation = {}
        seq = make_plan(_lib.make_opts(T))
        ablation["sequential_n1"] = T / (time_steps(stepper(seq), 10, 3, world, stream) * 1e-3)
        seq.close()
        if ovl_opts is not None:
            ab = list(ovl_opts.attn_bounds[: ovl_opts.n_attn + 1])
            fb = list(ovl_opts.ffn_bounds[: ovl_opts.n_ffn + 1])
            nb = make_plan(_lib.make_opts(T, ab, fb, executor=_lib.NF_EXEC_SEQUENTIAL))
            ablation["nanobatch_only"] = T / (time_steps(stepper(nb), 10, 3, world, stream) * 1e-3)
            nb.close()
            ov = make_plan(_lib.make_opts(T, ab, fb, executor=_lib.NF_EXEC_STREAMS,
                                          attn_sms=ovl_opts.attn_sms))
            ablation["overlap"] = T / (time_steps(stepper(ov), 10, 3, world, stream) * 1e-3)
            ov.close()
            ablation["overlap_plan"] = ovl_name
            ablation["nanobatch_only_plan"] = f"{ovl_name.split(',')[0]}, one stream"
        if world == 1:
            # the same batch through several layers, where the overlap can run
            # across layer boundaries (the single step has a head and a tail
            # that nothing overlaps)
            ablation["cross_layer"] = cross_layer_ablation(wk, stream)

    # metadata; per attention nano-batch RMSNorm-1, QKV, decode attention, O, and
    # the prefill-chunk attention where the nano-batch holds prefill rows (the
    # tensor-core attention); per FFN nano-batch RMSNorm-2, gate/up, down
    bounds = list(po.attn_bounds[: po.n_attn + 1])
    n_dec = wk.batch.n_decode
    with_prefill = sum(1 for a, b in zip(bounds, bounds[1:]) if b > n_dec) \
        if po.attn_impl == _lib.NF_ATTN_MMA else 0
    launches_per_step = 1 + 4 * po.n_attn + with_prefill + 3 * po.n_ffn
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens": T, "decode": wk.batch.n_decode,
                       "prefill": wk.batch.prefill_q_lens,
                       "kv_read_gb_per_step": wk.work["kv_read_bytes"] / 1e9,
                       "l2": "inputs larger than L2 (KV read per step > 7 GB, weights 0.44 GB)",
                       "plan": dict(_lib.opts_dict(po), chosen=best_name),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "layer_roofline": {"frac": layer_frac, "t_roof_ms": rf["t_roof"] * 1e3,
                               "t_flop_ms": rf["t_flop"] * 1e3, "t_byte_ms": rf["t_byte"] * 1e3,
                               "bound": rf["bound"], "flops": wk.work["flops"],
                               "bytes": wk.work["bytes"],
                               "peaks": f"{pk['source']}: {pk['bf16_tflops_sustained']} TF/s bf16 sustained, {pk['hbm_gbs']} GB/s"},
            "clocks": clk,
            "e2e": {"value": T * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roof,
            "overlap": {"attn_gemm_concurrent_ms": overlap, "timeline_last_step": timeline},
            "ablation_tokens_per_s": ablation,
            "plan_candidates_ms": tried,
            "search": None if prof is None else {
                "pick": _lib.opts_dict(so), "pick_over_best": round(tried["search"] / tried[best_name], 4),
                "builtin_pick_over_best": round(tried["search_builtin"] / tried[best_name], 4),
                "step_profile": prof}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = oracle_sample(wk, 128, 16, seed=1)
        t = time_oracle(sample)
        line["cpu_baseline"] = {"value": len(sample["rows"]) / t, "unit": "tokens/s",
                                "cores": cpu_cores(), "kind": "oracle", "sample": sample["desc"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    replicas.teardown(world)


if __name__ == "__main__":
    main()
