"""Small, self-contained runs of single kernels for Nsight Compute captures.

Each case builds seeded inputs of the 8B-shaped layer at a reduced size (so a
capture holds a few GB at most but still streams more than L2), runs a couple
of warm-up launches and then the launches to capture, and exits.

    python -m nano_intra_device_gb300.profcase attn --decode 512
    python -m nano_intra_device_gb300.profcase gemm --m 1024 --n 6144 --k 4096
    python -m nano_intra_device_gb300.profcase wrows --m 64 --n 14336 --k 4096 --epi 2
    python -m nano_intra_device_gb300.profcase step --decode 1792 --prefill 256 --nano 2 --sms 96
"""
from __future__ import annotations

import argparse
import sys

import numpy as np
import torch

from . import _lib, workload as wl


def _batch(decode, prefill):
    shape = wl.llama8b_shape()
    ctx = wl.lognormal_contexts(decode, 600.0, 1.0, 1, 8192, seed=1)
    b = wl.make_batch(shape, ctx, [prefill] if prefill else [], None, seed_bt=2, slack=0.01,
                      max_pages=8192 // 16)
    return shape, b


def case_attn(a):
    shape, b = _batch(a.decode, a.prefill)
    T = b.n_tokens
    kp, vp = wl.make_pools(shape, b, "cuda", seed=3, appended=True)
    q = torch.randn(T, shape.n_q, shape.head_dim, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    plan = _lib.Plan(shape, b, _lib.make_opts(T, kv_chunk=a.chunk))
    bt = torch.from_numpy(b.block_table).cuda()
    sl = torch.from_numpy(b.seq_lens).cuda()
    for _ in range(a.warmup + a.launches):
        _lib.attention(plan, q, kp, vp, bt, sl, o)
    plan.poll()
    kv = int(b.seq_lens.sum()) * 2 * shape.n_kv * shape.head_dim * 2
    print(f"attn case: {b.n_decode} decode + {a.prefill} prefill rows, KV read {kv / 1e9:.3f} GB/launch")


def case_gemm(a):
    A = torch.randn(a.m, a.k, device="cuda").to(torch.bfloat16)
    nb = 2 * a.n if a.epi == 2 else a.n
    B = (torch.randn(nb, a.k, device="cuda") * 0.02).to(torch.bfloat16)
    C = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
    R = torch.randn(a.m, a.n, device="cuda").to(torch.bfloat16) if a.epi == 1 else None
    for _ in range(a.warmup + a.launches):
        _lib.gemm(A, B, C, R=R, epilogue=a.epi, max_sms=a.sms)
    torch.cuda.synchronize()
    print(f"gemm case: {a.m}x{a.n}x{a.k} epilogue {a.epi}")


def case_wrows(a):
    """The weight-row GEMM of decode-sized nano-operations (nf_gemm_wrows)."""
    A = torch.randn(a.m, a.k, device="cuda").to(torch.bfloat16)
    nb = 2 * a.n if a.epi == 2 else a.n
    B = (torch.randn(nb, a.k, device="cuda") * 0.02).to(torch.bfloat16)
    C = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
    R = torch.randn(a.m, a.n, device="cuda").to(torch.bfloat16) if a.epi == 1 else None
    for _ in range(a.warmup + a.launches):
        _lib.gemm_wrows(A, B, C, R=R, epilogue=a.epi, splits=a.splits, max_sms=a.sms)
    torch.cuda.synchronize()
    print(f"wrows case: {a.m}x{a.n}x{a.k} epilogue {a.epi} splits {a.splits}")


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
    for _ in range(a.warmup + a.launches):
        _lib.layer_step(plan, w, x, kp, vp, bt, sl, y)
    plan.poll()
    print(f"step case: T={T}, plan {ab}, attn_sms {a.sms}")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["attn", "gemm", "wrows", "step"])
    ap.add_argument("--decode", type=int, default=512)
    ap.add_argument("--prefill", type=int, default=0)
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
    a = ap.parse_args(argv)
    {"attn": case_attn, "gemm": case_gemm, "wrows": case_wrows, "step": case_step}[a.case](a)


if __name__ == "__main__":
    sys.exit(main())
