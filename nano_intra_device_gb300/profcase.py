"""Small, self-contained runs of single kernels for Nsight Compute captures.

Each case builds seeded inputs of the 8B-shaped layer at a reduced size (so a
capture holds a few GB at most but still streams more than L2), runs a couple
of warm-up launches and then the launches to capture, and prints the mean
time of those launches (CUDA events on the launching stream; meaningless under
a profiler, which serialises and replays them).

    python -m nano_intra_device_gb300.profcase attn --decode 512
    python -m nano_intra_device_gb300.profcase gemm --m 1024 --n 6144 --k 4096
    python -m nano_intra_device_gb300.profcase wrows --m 64 --n 14336 --k 4096 --epi 2
    python -m nano_intra_device_gb300.profcase step --decode 1792 --prefill 256 --nano 2 --sms 96
    python -m nano_intra_device_gb300.profcase stepprofile --decode 1792 --prefill 256 --out p.json
"""
from __future__ import annotations

import argparse
import sys

import numpy as np
import torch

from . import _lib, workload as wl


def _timed(fn, warmup, launches):
    """Run fn warmup times, then `launches` times between two CUDA events;
    the mean milliseconds per launch."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(launches):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / max(1, launches)


def _batch(decode, prefill, prefix=0):
    shape = wl.llama8b_shape()
    ctx = wl.lognormal_contexts(decode, 600.0, 1.0, 1, 8192, seed=1)
    b = wl.make_batch(shape, ctx, [prefill] if prefill else [], [prefix] if prefill else None,
                      seed_bt=2, slack=0.01, max_pages=8192 // 16)
    return shape, b


def case_attn(a):
    shape, b = _batch(a.decode, a.prefill, a.prefix)
    T = b.n_tokens
    kp, vp = wl.make_pools(shape, b, "cuda", seed=3, appended=True)
    q = torch.randn(T, shape.n_q, shape.head_dim, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    plan = _lib.Plan(shape, b, _lib.make_opts(T, kv_chunk=a.chunk))
    bt = torch.from_numpy(b.block_table).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    ms = _timed(lambda: _lib.attention(plan, q, kp, vp, bt, sl, o), a.warmup, a.launches)
    plan.poll()
    kv = int(b.seq_lens.sum()) * 2 * shape.n_kv * shape.head_dim * 2
    print(f"attn case: {b.n_decode} decode + {a.prefill} prefill rows (prefix {a.prefix}), "
          f"KV read {kv / 1e9:.3f} GB/launch, {ms * 1e3:.1f} us per launch (metadata included)")


def case_gemm(a):
    A = torch.randn(a.m, a.k, device="cuda").to(torch.bfloat16)
    nb = 2 * a.n if a.epi == 2 else a.n
    B = (torch.randn(nb, a.k, device="cuda") * 0.02).to(torch.bfloat16)
    C = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
    R = torch.randn(a.m, a.n, device="cuda").to(torch.bfloat16) if a.epi == 1 else None
    ms = _timed(lambda: _lib.gemm(A, B, C, R=R, epilogue=a.epi, max_sms=a.sms), a.warmup, a.launches)
    fl = 2.0 * a.m * nb * a.k
    print(f"gemm case: {a.m}x{a.n}x{a.k} epilogue {a.epi}: {ms * 1e3:.1f} us, {fl / ms / 1e9:.0f} TFLOP/s")


def case_wrows(a):
    """The weight-row GEMM of decode-sized nano-operations (nf_gemm_wrows)."""
    A = torch.randn(a.m, a.k, device="cuda").to(torch.bfloat16)
    nb = 2 * a.n if a.epi == 2 else a.n
    B = (torch.randn(nb, a.k, device="cuda") * 0.02).to(torch.bfloat16)
    C = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
    R = torch.randn(a.m, a.n, device="cuda").to(torch.bfloat16) if a.epi == 1 else None
    ms = _timed(lambda: _lib.gemm_wrows(A, B, C, R=R, epilogue=a.epi, splits=a.splits, max_sms=a.sms),
                a.warmup, a.launches)
    wbytes = nb * a.k * 2
    print(f"wrows case: {a.m}x{a.n}x{a.k} epilogue {a.epi} splits {a.splits}: {ms * 1e3:.1f} us, "
          f"weights at {wbytes / ms / 1e9:.2f} TB/s")


def case_step(a):
    shape, b = _batch(a.decode, a.prefill)
    T = b.n_tokens
    w = {k: v.cuda() for k, v in wl.make_weights(shape, seed=0).items()}
    x = wl.make_x(shape, T, seed=0).cuda()
    kp, vp = wl.make_pools(shape, b, "cuda", seed=3)
    bt = torch.from_numpy(b.block_table).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    y = torch.empty_like(x)
    g = 128 if T >= 1024 else 1
    ab = [0] + [max(1, int(round(T * i / a.nano / g)) * g) for i in range(1, a.nano)] + [T]
    ex = _lib.NF_EXEC_STREAMS if a.nano > 1 else _lib.NF_EXEC_SEQUENTIAL
    plan = _lib.Plan(shape, b, _lib.make_opts(T, ab, ab, executor=ex, attn_sms=a.sms))
    ms = _timed(lambda: _lib.layer_step(plan, w, x, kp, vp, bt, sl, y), a.warmup, a.launches)
    plan.poll()
    print(f"step case: T={T}, plan {ab}, attn_sms {a.sms}: {ms:.3f} ms per step")


def case_stepprofile(a):
    """nf_profile_step on the 8B-shaped mixed batch (decode rows + one prefill
    chunk) over --layers layers; writes the profile JSON to --out."""
    shape, b = _batch(a.decode, a.prefill, a.prefix)
    _lib.profile_step(shape, b, a.layers, a.out)
    print(f"step profile: T={b.n_tokens}, {a.layers} layers -> {a.out}")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["attn", "gemm", "wrows", "step", "stepprofile"])
    ap.add_argument("--decode", type=int, default=512)
    ap.add_argument("--prefill", type=int, default=0)
    ap.add_argument("--prefix", type=int, default=0, help="cached positions before the prefill chunk")
    ap.add_argument("--chunk", type=int, default=512)
    ap.add_argument("--m", type=int, default=1024)
    ap.add_argument("--n", type=int, default=6144)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--epi", type=int, default=0)
    ap.add_argument("--sms", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--nano", type=int, default=2)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--launches", type=int, default=2)
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--out", default="step_profile.json")
    a = ap.parse_args(argv)
    {"attn": case_attn, "gemm": case_gemm, "wrows": case_wrows, "step": case_step,
     "stepprofile": case_stepprofile}[a.case](a)


if __name__ == "__main__":
    sys.exit(main())
