"""Tolerances of the GPU-vs-oracle parity tests.

fp32 inputs: max|x - ref| / max|ref| <= 1e-4 per tensor (normwise max).
bf16 inputs: |x - ref| <= 2e-2 |ref| + 1e-2 elementwise.
Both apply to outputs and final states.

The fp32 bound is read normwise: "max relative error 1e-4" taken over the
whole tensor, with the tensor's largest magnitude as the scale.  The stricter
elementwise reading (|x - ref| / |ref| per element) is also measured, without
asserting on it, over the elements with |ref| above F32_ELEM_FLOOR times the
tensor's largest magnitude (below that, relative error measures rounding of
near-cancelled sums rather than the kernel); the worst value seen in a test
run is printed in the session summary.
"""
import numpy as np
import torch

F32_REL = 1e-4
BF16_REL, BF16_ABS = 2e-2, 1e-2
F32_ELEM_FLOOR = 1e-3
F32_ELEMENTWISE = []     # (what, normwise error, worst elementwise relative error)


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
        big = np.abs(ref) > F32_ELEM_FLOOR * scale
        elem = float((np.abs(got - ref)[big] / np.abs(ref)[big]).max()) if big.any() else 0.0
        F32_ELEMENTWISE.append((what, float(err), elem))
        assert err <= F32_REL, f"{what}: normwise max rel err {err:.3e} > {F32_REL}"
        return err
    excess = np.abs(got - ref) - (BF16_REL * np.abs(ref) + BF16_ABS)
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: |x-ref| exceeds 2e-2|ref|+1e-2 at {worst}: "
                               f"got {got[worst]:.6f} ref {ref[worst]:.6f}")
    return float(np.abs(got - ref).max())


def assert_close_gated(got, o_ref, gate, dtype, what=""):
    """The output epilogue y = o / sqrt(mean(o^2) + eps) * w * sigmoid(z),
    checked against the oracle's o (o_ref, before the epilogue).

    fp32: the normwise 1e-4 bound on y itself.  bf16: the elementwise bound
    on o carried through the epilogue.  A change do in one element of o moves
    y by at most |do| rinv |w sigmoid(z)| plus the change of the row's rinv,
    which is at most the row's relative change of o; with the bf16 bound
    |do| <= 2e-2 |o| + 1e-2 that gives
        |y - y_ref| <= 2e-2 |y_ref| + 1e-2 rinv |w sigmoid(z)|     (each element)
                     + 2e-2 |y_ref|                                  (the row's rinv)
                     + 2^-8 |y_ref|                                  (bf16 rounding of y)
    with rinv = 1 / sqrt(mean(o_ref^2) + eps) of the row.
    """
    import oracle
    z, w, eps = gate
    o_ref = to64(o_ref)
    y_ref = oracle.output_gate(o_ref, z, w, eps)
    got = to64(got)
    assert got.shape == y_ref.shape, (what, got.shape, y_ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if dtype in ("f32", torch.float32):
        return assert_close(got, y_ref, dtype, what)
    zz, ww = to64(z), to64(w)
    rinv = 1.0 / np.sqrt(np.mean(o_ref * o_ref, axis=-1, keepdims=True) + float(eps))
    amp = rinv * np.abs(ww) / (1.0 + np.exp(-zz))
    bound = (2 * BF16_REL + 2.0 ** -8) * np.abs(y_ref) + BF16_ABS * amp
    excess = np.abs(got - y_ref) - bound
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: gated |y-ref| exceeds the propagated bf16 bound at "
                               f"{worst}: got {got[worst]:.6f} ref {y_ref[worst]:.6f} "
                               f"bound {bound[worst]:.6f}")
    return float(np.abs(got - y_ref).max())
