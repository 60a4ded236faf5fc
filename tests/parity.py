"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (the method's stated bars):
  FP32 forward         max |gpu - ref| <= 2e-4
  FP32 gradients       ||gpu - ref||_2 / ||ref||_2 <= 5e-3 (TF32 allowed in backward)
  BF16 outputs, grads  max |gpu - ref| / max(1, |ref|) <= 3e-2  and  rel-L2 <= 1e-2

The BF16 max-abs bar is applied elementwise relative to max(1, |ref|): outputs
have a standard deviation near 3 and reach ~16, where half a bf16 unit in the
last place is already 0.03-0.06, so an absolute 3e-2 cannot hold for any
correctly rounded bf16 result.  Below magnitude 1 the bar is absolute.

One further reading applies to the gradients that are sums of bf16-rounded
dK products: dW and dbias (every pixel of every image summed into one entry)
and dy (all 3*C*K*K taps of a pixel summed through the weight).  bf16 training
rounds each product dK = grad * x to bf16 before those sums (PyTorch's bf16
autograd semantics), and the error of a sum of N such terms grows like
sqrt(N) * 2^-9 * |term|, i.e. with the magnitude of the whole tensor (its RMS),
not with each entry.  At 256x256 the dW entries are ~256 and their rounding
error ~0.5; the dy entries have an RMS near 5 and a rounding error up to ~0.03.
Entries that happen to lie near zero can only be held to the tensor's scale:
for dy, dW and dbias the denominator is max(1, |ref|, rms(ref)).  Outputs, dx
and dtaps (no sum of rounded products) use max(1, |ref|).  rel-L2 is applied
as written everywhere.

Every comparison is recorded in MARGINS (what, measure, value, bar) so that the
test session can print the achieved errors next to their bars.
"""
import numpy as np
import torch

FP32_FWD_MAX_ABS = 2e-4
FP32_GRAD_REL_L2 = 5e-3
BF16_MAX_REL = 3e-2
BF16_REL_L2 = 1e-2

# gradients that are sums of bf16-rounded dK products (held to the tensor's scale in bf16)
DK_SUMS = ("dy", "dW", "dbias")

# (what, measure, value, bar, full_size) of every comparison made in this session
MARGINS = []
_full_size = [False]


class full_size_section:
    """Context manager: comparisons made inside it are flagged as full-size."""

    def __enter__(self):
        _full_size[0] = True
        return self

    def __exit__(self, *exc):
        _full_size[0] = False


def _record(what, measure, value, bar):
    MARGINS.append((what, measure, float(value), float(bar), _full_size[0]))


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
    """max |got - ref| / max(1, |ref|) (the bf16 max-abs reading)."""
    got, ref = to64(got), to64(ref)
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref)))) if got.size else 0.0


def max_rel_scale(got, ref) -> float:
    """max |got - ref| / max(1, |ref|, rms(ref)) (bf16 sums of rounded dK products only)."""
    got, ref = to64(got), to64(ref)
    if not got.size:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref) / np.maximum(max(1.0, rms), np.abs(ref))))


def _bf16(got, ref, what, dk_sum):
    if dk_sum:
        e1, m1 = max_rel_scale(got, ref), "max|d|/max(1,|ref|,rms)"
    else:
        e1, m1 = max_rel1(got, ref), "max|d|/max(1,|ref|)"
    e2 = rel_l2(got, ref)
    _record(what, m1, e1, BF16_MAX_REL)
    _record(what, "rel-L2", e2, BF16_REL_L2)
    assert e1 <= BF16_MAX_REL, f"{what}: bf16 {m1} {e1:.3e} > {BF16_MAX_REL}"
    assert e2 <= BF16_REL_L2, f"{what}: bf16 rel-L2 {e2:.3e} > {BF16_REL_L2}"


def assert_forward_close(got, ref, dtype: str, what: str = "out"):
    if dtype == "float32":
        e = max_abs(got, ref)
        _record(what, "max|d|", e, FP32_FWD_MAX_ABS)
        assert e <= FP32_FWD_MAX_ABS, f"{what}: fp32 max-abs {e:.3e} > {FP32_FWD_MAX_ABS}"
    else:
        _bf16(got, ref, what, dk_sum=False)


def assert_grad_close(got, ref, dtype: str, what: str):
    """`what` starts with the gradient's name; dy, dW and dbias are sums of rounded dK."""
    if dtype == "float32":
        e = rel_l2(got, ref)
        _record(what, "rel-L2", e, FP32_GRAD_REL_L2)
        assert e <= FP32_GRAD_REL_L2, f"{what}: fp32 rel-L2 {e:.3e} > {FP32_GRAD_REL_L2}"
    else:
        _bf16(got, ref, what, dk_sum=what.split()[0] in DK_SUMS)


# ------------------------------------------------- bf16 tap-rounding ties --
# In bf16 mode every generated tap is rounded to bf16 before the filter uses it
# (a quantisation decision).  The GPU decides it on the FP32 tensor-core sum
# W.y + bias, the oracle on the FP64 sum: where the exact tap lies within the
# FP32 accumulation error of a rounding midpoint, both roundings are correct
# results, and they differ by one bf16 spacing.  Elements above the bar are
# accepted only if the taps they use include such ties and the excess is at
# most what flipping those ties can change: sum over tied taps of
# |round(T + eps) - round(T - eps)| * |operand|, eps = 2^-16 * (sum_j |W y| + |b|)
# (well above the FP32 accumulation error of 65 terms, 65 * 2^-24 * sum |terms|).

TIE_EPS = 2.0 ** -16


def tap_tie_flip(oracle, y64, w64, b64, K, dil, b, o, h, w) -> float:
    """|round(T + eps) - round(T - eps)| for tap o at (b, h, w): 0 unless the tap is a tie."""
    T = oracle.tap(y64, w64, b64, K, dil, b, o, h, w, bf16=False)
    mag = float(np.abs(w64[o]) @ np.abs(y64[b, :, h, w])) + (abs(float(b64[o])) if b64 is not None else 0.0)
    eps = TIE_EPS * mag
    return abs(oracle.round_bf16(T + eps) - oracle.round_bf16(T - eps))


def forward_tie_allowance(oracle, h64, K, dil, flat_idx) -> np.ndarray:
    """Per output element (flat index into [B, 4C, H, W]): the most that flipping tied
    taps can change it, sum over its taps of flip(T) * |x at the tap's source|."""
    x64, y64, w64, b64 = h64["x"], h64["y"], h64["weight"], h64.get("bias")
    B, C, H, W = x64.shape
    r = K // 2
    out = np.zeros(len(flat_idx))
    for n, f in enumerate(flat_idx):
        b, ch, hh, ww = np.unravel_index(int(f), (B, 4 * C, H, W))
        if ch < C:
            continue
        di, c = ch // C - 1, ch % C
        d = dil[di]
        for k in range(K * K):
            ky, kx = divmod(k, K)
            hs, ws = hh + (ky - r) * d, ww + (kx - r) * d
            if 0 <= hs < H and 0 <= ws < W and x64[b, c, hs, ws] != 0.0:
                o = (di * C + c) * K * K + k
                out[n] += tap_tie_flip(oracle, y64, w64, b64, K, dil, b, o, hh, ww) * abs(x64[b, c, hs, ws])
    return out


def dx_tie_allowance(oracle, h64, K, dil, flat_idx) -> np.ndarray:
    """Per dx element (flat index into [B, C, H, W]): sum over the taps it gathers of
    flip(T at the source pixel) * |grad at the source pixel|."""
    g64, y64, w64, b64 = h64["grad_out"], h64["y"], h64["weight"], h64.get("bias")
    B, C, H, W = y64.shape
    r = K // 2
    out = np.zeros(len(flat_idx))
    for n, f in enumerate(flat_idx):
        b, c, hh, ww = np.unravel_index(int(f), (B, C, H, W))
        for di in range(3):
            d = dil[di]
            for k in range(K * K):
                ky, kx = divmod(k, K)
                hs, ws = hh - (ky - r) * d, ww - (kx - r) * d
                gv = g64[b, (1 + di) * C + c, hs, ws] if (0 <= hs < H and 0 <= ws < W) else 0.0
                if gv != 0.0:
                    o = (di * C + c) * K * K + k
                    out[n] += tap_tie_flip(oracle, y64, w64, b64, K, dil, b, o, hs, ws) * abs(gv)
    return out


def assert_bf16_close_with_ties(got, ref, what, allowance_fn, limit=20000):
    """The bf16 bar of assert_forward_close / assert_grad_close (max(1, |ref|) reading),
    where an element above it must be explained by tap-rounding ties: its excess
    may not exceed allowance_fn(flat indices) and that allowance must be nonzero."""
    got, ref = to64(got), to64(ref)
    err = np.abs(got - ref).reshape(-1)
    scale = np.maximum(1.0, np.abs(ref)).reshape(-1)
    over = np.nonzero(err > BF16_MAX_REL * scale)[0]
    e2 = rel_l2(got, ref)
    _record(what, "rel-L2", e2, BF16_REL_L2)
    assert e2 <= BF16_REL_L2, f"{what}: bf16 rel-L2 {e2:.3e} > {BF16_REL_L2}"
    inside = np.ones_like(err, dtype=bool)
    inside[over] = False
    e1 = float(np.max(err[inside] / scale[inside])) if inside.any() else 0.0
    _record(what, "max|d|/max(1,|ref|) untied", e1, BF16_MAX_REL)
    assert len(over) <= limit, f"{what}: {len(over)} elements above the bar"
    if len(over):
        allow = allowance_fn(over)
        excess = err[over] - BF16_MAX_REL * scale[over]
        bad = np.nonzero((allow <= 0.0) | (excess > allow))[0]
        assert len(bad) == 0, (f"{what}: {len(bad)} of {len(over)} elements above the bar are not explained by "
                               f"tap-rounding ties (first: flat index {over[bad[0]]}, error {err[over[bad[0]]]:.4e}, "
                               f"allowance {allow[bad[0]]:.4e})")
        worst = float(np.max(err[over] / (BF16_MAX_REL * scale[over] + allow)))
        _record(what, f"tied elements: {len(over)}; max|d|/(bar+flip)", worst * BF16_MAX_REL, BF16_MAX_REL)
