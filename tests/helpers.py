"""Shared helpers for the GPU parity tests."""
import numpy as np
import torch

# Tolerances for bf16 outputs against the float64 oracle.  Relative L2 <= 1e-2
# as stated for the layer; max-abs <= 3e-2 in units of the reference's RMS
# (floored at 1): a bf16 value of magnitude >= 4 already carries a rounding
# step of 3e-2 or more, so an absolute bound cannot hold for outputs of RMS ~3.
REL_L2 = 1e-2
MAX_ABS = 3e-2


def compare(gpu, ref, name="", rel_l2=REL_L2, max_abs=MAX_ABS):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    d = gpu - ref
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    ma = float(np.abs(d).max()) if d.size else 0.0
    rl = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    assert rl <= rel_l2, f"{name}: rel-L2 {rl:.3g} > {rel_l2}"
    assert ma <= max_abs * max(1.0, rms), f"{name}: max-abs {ma:.3g} > {max_abs} x max(1, rms={rms:.3g})"
    return ma, rl


def to_dev(w, dev="cuda"):
    return {k: v.to(dev) for k, v in w.items()}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()
