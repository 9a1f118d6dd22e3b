"""Helpers shared by the GPU parity tests (input marshalling and the error metrics)."""
import numpy as np
import torch

from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32

# Tolerances.  Forward: the evaluation targets for out and lse.  Gradients (no
# target is stated for them): the kernels round P and dS to bf16 before the
# products and the outputs to bf16 once; bf16 keeps 8 significant bits, so each
# rounding moves a value by at most 2^-8 of itself (about 2^-9 in rms), and a
# gradient element stays within a few 2^-8 of max(1, |ref|).
F32_MAX_ABS = 1e-5
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-2
GRAD_MAX_REL = 2e-2   # max |err| / max(1, |ref|)
GRAD_MEAN_ABS = 2e-3


def to_dev(x: np.ndarray, dtype: str, dev="cuda"):
    if x is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    if x.dtype == np.int32:
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x).astype(np.float64) if dtype == "bf16" else x.astype(np.float64)


def check_out(got, ref, dtype, what="out", scale=1.0):
    """Forward output check.  The absolute bounds are the evaluation targets for
    unit-scale inputs; for inputs scaled by `scale` > 1 (stress cases outside
    the evaluation distributions) the same bounds apply relative to
    max(1, |ref|) and the mean bound grows with the scale, because bf16
    rounding of P and of the output is relative to the magnitude."""
    err = np.abs(got - ref)
    if scale > 1.0 and dtype == "bf16":
        rel = (err / np.maximum(1.0, np.abs(ref))).max()
        assert rel <= BF16_MAX_ABS, f"{what}: max rel err {rel:.3e}"
        assert err.mean() <= BF16_MEAN_ABS * scale, f"{what}: mean abs err {err.mean():.3e}"
        return err.max(), err.mean()
    if dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    else:
        assert err.max() <= BF16_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
        assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    return err.max(), err.mean()


def check_lse(got, ref, dtype):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "lse: -inf pattern differs"
    err = np.abs(got[fin] - ref[fin]) if fin.any() else np.zeros(1)
    tol = F32_MAX_ABS if dtype == "f32" else LSE_MAX_ABS
    assert err.max() <= tol, f"lse: max abs err {err.max():.3e}"
    return err.max()


def check_grad(got, ref, what):
    err = np.abs(got - ref)
    rel = (err / np.maximum(1.0, np.abs(ref))).max()
    assert rel <= GRAD_MAX_REL, f"{what}: max rel err {rel:.3e}"
    assert err.mean() <= GRAD_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    return rel, err.mean()
