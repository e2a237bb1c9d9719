"""Tolerances of the GPU-vs-oracle parity tests.

fp32 inputs: max|x - ref| / max|ref| <= 1e-4 per tensor (normwise max).
bf16 inputs: |x - ref| <= 2e-2 |ref| + 1e-2 elementwise.
Both apply to outputs and final states.
"""
import numpy as np
import torch

F32_REL = 1e-4
BF16_REL, BF16_ABS = 2e-2, 1e-2


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def assert_close(got, ref, dtype, what=""):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if dtype in ("f32", torch.float32):
        scale = max(np.abs(ref).max(), 1e-30)
        err = np.abs(got - ref).max() / scale
        assert err <= F32_REL, f"{what}: normwise max rel err {err:.3e} > {F32_REL}"
        return err
    excess = np.abs(got - ref) - (BF16_REL * np.abs(ref) + BF16_ABS)
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: |x-ref| exceeds 2e-2|ref|+1e-2 at {worst}: "
                               f"got {got[worst]:.6f} ref {ref[worst]:.6f}")
    return float(np.abs(got - ref).max())
