"""Shared helpers for the GPU parity tests.

Bounds (the layer's stated tolerance for its bf16 outputs): relative L2
<= 1e-2, and element by element |gpu - ref| <= 3e-2 + half a bf16 step of ref.
The second term is the rounding of the stored output itself: the GPU's outputs
are bf16, so even the exact value, rounded, is off by up to half a step, which
is 2^(e-8) for |ref| in [2^e, 2^(e+1)) (between 2^-9 and 2^-8 of |ref|).

Two oracles serve the layer-level tests.  The exact one computes in float64
throughout.  The bf16-storage one (oracle ``store="bf16"``) is the same
definition with the tensors the layer keeps in memory between its operations
(n1, q, k, v, o, h, n2, a, and a layer's output read by the next) rounded to
bf16 where they are produced: the GPU keeps exactly these in bf16, because
they are bf16 tensor-core operands or live in bf16 buffers.  ``parity`` holds
the GPU to both stated bounds against the bf16-storage oracle and to the stated
relative L2 against the exact one, and records the max-abs against the exact
oracle, which is bounded by the stated bound plus the storage term
|bf16-storage - exact| that the oracle itself measures.

Every comparison is appended to RECORD (test, quantity, size, max-abs,
relative L2, RMS of the reference); the session writes it out as JSON when the
environment names a file in NF_PARITY_LOG.
"""
import os

import numpy as np
import torch

REL_L2 = 1e-2
MAX_ABS = 3e-2
RECORD = []


def half_step(ref):
    """Half the spacing of the bf16 grid at |ref| (0 at 0)."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def record(name, d, ref, oracle):
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    ma = float(np.abs(d).max()) if d.size else 0.0
    rl = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)) if d.size else 0.0
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RECORD.append(dict(test=test, name=name, oracle=oracle, n=int(d.size), max_abs=ma,
                       rel_l2=rl, rms_ref=rms))
    print(f"parity {name} [{oracle}]: n {d.size}, max-abs {ma:.4g}, rel-L2 {rl:.3g}, rms {rms:.3g}")
    return ma, rl


def compare(gpu, ref, name="", rel_l2=REL_L2, max_abs=MAX_ABS, oracle="oracle"):
    """Assert rel-L2 <= rel_l2 and |gpu - ref| <= max_abs + half_step(ref)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    d = gpu - ref
    ma, rl = record(name, d, ref, oracle)
    assert rl <= rel_l2, f"{name}: rel-L2 {rl:.3g} > {rel_l2}"
    bound = max_abs + half_step(ref)
    if d.size:
        worst = int(np.argmax(np.abs(d) - bound))
        assert np.all(np.abs(d) <= bound), (
            f"{name}: |err| {np.abs(d).flat[worst]:.3g} > bound {bound.flat[worst]:.3g} at ref "
            f"{ref.flat[worst]:.3g} (max-abs {ma:.3g})")
    return ma, rl


def parity(gpu, exact, emul, name):
    """The GPU's bf16 output against the bf16-storage oracle (both stated
    bounds) and against the exact oracle (stated relative L2; max-abs
    recorded, and checked against its derived bound)."""
    gpu = np.asarray(gpu, np.float64)
    exact = np.asarray(exact, np.float64)
    emul = np.asarray(emul, np.float64)
    compare(gpu, emul, name, oracle="bf16-storage")
    d = gpu - exact
    _, rl = record(name, d, exact, "exact")
    record(name + " (storage term)", emul - exact, exact, "bf16-storage vs exact")
    assert rl <= REL_L2, f"{name}: rel-L2 {rl:.3g} against the exact oracle > {REL_L2}"
    derived = MAX_ABS + half_step(emul) + np.abs(emul - exact)
    assert np.all(np.abs(d) <= derived), f"{name}: beyond the stated bound plus the storage term"


def rounding_floor(out, base):
    """Relative L2 that an exact result scores on out - base once out is
    rounded to bf16: the floor of a check on a small difference of a bf16
    output (e.g. y - x when the residual dominates y)."""
    from oracle.layer import bf16
    out = np.asarray(out, np.float64)
    base = np.asarray(base, np.float64)
    return float(np.linalg.norm(bf16(out) - out) / max(np.linalg.norm(out - base), 1e-30))


def to_dev(w, dev="cuda"):
    return {k: v.to(dev) for k, v in w.items()}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()
