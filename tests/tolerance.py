"""Per-element acceptance bound for GPU results against the oracle.

|Y_gpu - Y_ref| <= 2e-3 * sum_k |A[m,k] w[n,k]| + 1e-5  (+ u_out * |Y_ref|)

The first two terms are the stated tolerance for fp32 and bf16 activations.
The last term is the representation error of the output dtype, which no
kernel can avoid: a bf16 output is the fp32 result rounded to nearest even,
whose relative error is at most u = 2^-8 (8-bit significand). It is 0 for
fp32 outputs. Without it a single-term dot product (K = 1) could not pass in
bf16 however exact the arithmetic.
"""
import numpy as np
import torch

REL = 2e-3
ABS = 1e-5
U_OUT = {torch.float32: 0.0, torch.bfloat16: 2.0 ** -8}


def bound(absdot: np.ndarray, ref: np.ndarray, out_dtype: torch.dtype) -> np.ndarray:
    return REL * absdot + ABS + U_OUT[out_dtype] * np.abs(ref)


def check(y_gpu: torch.Tensor, ref: np.ndarray, absdot: np.ndarray, what: str = ""):
    """Assert the bound element by element; return max(err / bound)."""
    y = y_gpu.detach().float().cpu().double().numpy()
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    b = bound(absdot, ref, y_gpu.dtype)
    ratio = err / b
    if ratio.size == 0:
        return 0.0
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert np.all(err <= b), (
        f"{what}: max err/bound = {ratio.max():.3g} at {worst}: gpu={y[worst]!r} "
        f"ref={ref[worst]!r} absdot={absdot[worst]!r}")
    return float(ratio.max())
