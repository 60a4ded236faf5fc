"""Pins of the CPU FP64 oracle to things other than itself (CPU only).

Each test ties the oracle to an independent fact about the method in the
"lartpang/DynamicConvolutionOperator" README:

* Unfold math reference ("问题与目标": out_d = taps x Unfold_d(x), taps from a
  1x1 generator) -- computed here with torch's own ``F.unfold`` / ``F.conv2d``;
* constant taps reduce to an ordinary dilated depthwise convolution
  (``F.conv2d(groups=C, dilation=d)``, a library routine);
* K = 1 reduces to per-pixel channel scaling (closed form);
* one-hot taps on position-coded x return the shifted image (offset sign,
  zero padding), bit-exact;
* FP64 central differences for every gradient (the map is linear in each of
  x, y, W, bias separately, so central differences are exact up to rounding);
* adjoint identities <g,out> = <dx,x> and <g,out_d> = <dW,W> + <dbias,bias>
  = <dy,y> + <dbias,bias>;
* the bf16 rounding against torch's float32 -> bfloat16 conversion;
* a hand-worked example (tests/golden/handworked_k3_3x3.json);
* the filter-only backward (taps given) against torch autograd through the
  Unfold reference, the adjoint identities <g,out> = <dx,x> = <dT,T> + <g_0,x>,
  and sum_{b,p} dT = the fused backward's dbias.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from dynamic_dilated_depthwise_gb300.inputs import Problem, make_inputs, make_integer_inputs

HERE = os.path.dirname(os.path.abspath(__file__))

SMALL = [
    Problem(1, 2, 5, 6, 3),
    Problem(2, 3, 7, 5, 3),
    Problem(1, 2, 6, 7, 5),
    Problem(2, 3, 4, 5, 1),
    Problem(1, 2, 9, 8, 3, dilations=(2, 2, 4)),
]


def _id(p):
    return f"{p.B}x{p.C}x{p.H}x{p.W}k{p.K}d{''.join(map(str, p.dilations))}"


def _np(t):
    return t.detach().to(torch.float64).numpy()


def unfold_reference(x, T, K, dils):
    """The pages' Unfold math reference, written with torch library primitives."""
    x = torch.as_tensor(x, dtype=torch.float64)
    T = torch.as_tensor(T, dtype=torch.float64)
    B, C, H, W = x.shape
    K2 = K * K
    outs = [x]
    for di, d in enumerate(dils):
        U = F.unfold(x, K, dilation=d, padding=d * (K // 2))          # [B, C*K2, H*W], order (c, ky, kx)
        Td = T[:, di * C * K2:(di + 1) * C * K2].reshape(B, C * K2, H * W)
        outs.append((U * Td).reshape(B, C, K2, H * W).sum(2).reshape(B, C, H, W))
    return torch.cat(outs, 1).numpy()


def generator_reference(y, Wg, bias):
    y = torch.as_tensor(y, dtype=torch.float64)
    Wg = torch.as_tensor(Wg, dtype=torch.float64)
    b = None if bias is None else torch.as_tensor(bias, dtype=torch.float64)
    return F.conv2d(y, Wg[:, :, None, None], b).numpy()


def _inputs(p, seed=7):
    t = make_inputs(p, seed, "float32", grad=True, taps=True)
    return {k: _np(v) for k, v in t.items()}


# ------------------------------------------------------------------ bf16 --

def test_round_bf16_matches_torch_conversion():
    g = torch.Generator().manual_seed(3)
    vals = torch.cat([
        torch.randn(4000, generator=g) * 10.0 ** torch.randint(-6, 6, (4000,), generator=g).float(),
        torch.tensor([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 1.0078125, -1.0078125, 3e38, -3.4e38,
                      1e-40, -3e-39, 9.2e-41, 2.0 ** -133, 3 * 2.0 ** -134, 65504.0, 1.5e-38]),
    ]).to(torch.float32)
    want = vals.to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals.to(torch.float64)])
    np.testing.assert_array_equal(got, want)


def test_round_bf16_ties_to_even():
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0                      # halfway: even is 1.0
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6      # halfway: even is 1+2^-6
    assert oracle.round_bf16(-(1.0 + 2.0 ** -8)) == -1.0


# --------------------------------------------------------------- forward --

@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_generator_matches_conv1x1(p):
    t = _inputs(p)
    T = oracle.generate_taps(t["y"], t["weight"], t["bias"], p.K, p.dilations)
    np.testing.assert_allclose(T, generator_reference(t["y"], t["weight"], t["bias"]), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_forward_matches_unfold_reference(p):
    t = _inputs(p)
    out = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations)
    T = generator_reference(t["y"], t["weight"], t["bias"])
    np.testing.assert_allclose(out, unfold_reference(t["x"], T, p.K, p.dilations), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_filter_matches_unfold_reference(p):
    t = _inputs(p)
    out = oracle.filter_pregenerated(t["x"], t["taps"], p.K, p.dilations)
    np.testing.assert_allclose(out, unfold_reference(t["x"], t["taps"], p.K, p.dilations), rtol=1e-12, atol=1e-12)


def test_forward_without_bias_matches_unfold_reference():
    p = Problem(1, 3, 6, 5, 3)
    t = _inputs(p)
    out = oracle.forward(t["x"], t["y"], t["weight"], None, p.K, p.dilations)
    T = generator_reference(t["y"], t["weight"], None)
    np.testing.assert_allclose(out, unfold_reference(t["x"], T, p.K, p.dilations), rtol=1e-12, atol=1e-12)


def test_forward_bf16_mode_rounds_taps_before_use():
    p = Problem(1, 3, 6, 7, 3)
    t = make_inputs(p, 11, "bfloat16", grad=False)
    t = {k: _np(v) for k, v in t.items()}
    out = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations, bf16=True)
    T = generator_reference(t["y"], t["weight"], t["bias"])
    # torch's conversion of the float32-rounded taps agrees with direct rounding almost everywhere
    Tq = torch.as_tensor(T).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    direct = np.vectorize(oracle.round_bf16)(T)
    assert np.mean(direct == Tq) > 0.99
    np.testing.assert_allclose(out, unfold_reference(t["x"], direct, p.K, p.dilations), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("K", [1, 3, 5])
@pytest.mark.parametrize("dils", [(1, 3, 5), (2, 2, 4)])
def test_constant_taps_are_dilated_depthwise_conv(K, dils):
    p = Problem(2, 3, 11, 9, K, dilations=dils)
    t = _inputs(p, seed=5)
    Wg = np.zeros_like(t["weight"])
    bias = t["bias"] * 10.0
    out = oracle.forward(t["x"], t["y"], Wg, bias, K, dils)
    x = torch.as_tensor(t["x"])
    C, K2 = p.C, K * K
    for di, d in enumerate(dils):
        ker = torch.as_tensor(bias[di * C * K2:(di + 1) * C * K2]).reshape(C, 1, K, K)
        want = F.conv2d(x, ker, padding=d * (K // 2), dilation=d, groups=C).numpy()
        np.testing.assert_allclose(out[:, (1 + di) * C:(2 + di) * C], want, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(out[:, :C], t["x"])


def test_k1_is_per_pixel_channel_scaling():
    p = Problem(2, 4, 5, 6, 1)
    t = _inputs(p)
    out = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], 1, p.dilations)
    T = generator_reference(t["y"], t["weight"], t["bias"])
    for di in range(3):
        np.testing.assert_allclose(out[:, (1 + di) * p.C:(2 + di) * p.C],
                                   T[:, di * p.C:(di + 1) * p.C] * t["x"], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("K,dils", [(3, (1, 3, 5)), (5, (1, 3, 5)), (3, (2, 2, 4))])
def test_one_hot_taps_shift_position_coded_x(K, dils):
    B, C, H, W = 1, 2, 9, 12
    x = np.zeros((B, C, H, W))
    for c in range(C):
        x[0, c] = (np.arange(H)[:, None] * W + np.arange(W)[None, :] + 1) * (c + 1)
    r = K // 2
    O = 3 * C * K * K
    for di, d in enumerate(dils):
        for ky in range(K):
            for kx in range(K):
                T = np.zeros((B, O, H, W))
                for c in range(C):
                    T[0, (di * C + c) * K * K + ky * K + kx] = 1.0
                out = oracle.filter_pregenerated(x, T, K, dils)
                sy, sx = (ky - r) * d, (kx - r) * d
                want = np.zeros((B, C, H, W))
                h0, h1 = max(0, -sy), min(H, H - sy)
                w0, w1 = max(0, -sx), min(W, W - sx)
                if h0 < h1 and w0 < w1:
                    want[:, :, h0:h1, w0:w1] = x[:, :, h0 + sy:h1 + sy, w0 + sx:w1 + sx]
                np.testing.assert_array_equal(out[:, (1 + di) * C:(2 + di) * C], want)
                for dj in range(3):
                    if dj != di:
                        assert not out[:, (1 + dj) * C:(2 + dj) * C].any()


def test_passthrough_channels_bitwise():
    p = Problem(2, 3, 7, 5, 3)
    t = _inputs(p)
    out = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations)
    np.testing.assert_array_equal(out[:, :p.C], t["x"])


def test_forward_points_match_full():
    p = Problem(2, 3, 7, 6, 5)
    t = _inputs(p)
    full = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations)
    idx = np.random.default_rng(0).integers(0, full.size, 300)
    np.testing.assert_array_equal(oracle.forward_points(t["x"], t["y"], t["weight"], t["bias"], p.K, idx,
                                                        p.dilations), full.reshape(-1)[idx])
    fullf = oracle.filter_pregenerated(t["x"], t["taps"], p.K, p.dilations)
    np.testing.assert_array_equal(oracle.filter_points(t["x"], t["taps"], p.K, idx, p.dilations),
                                  fullf.reshape(-1)[idx])


# -------------------------------------------------------------- backward --

def _loss(g, x, y, Wg, bias, K, dils):
    return float(np.sum(g * oracle.forward(x, y, Wg, bias, K, dils)))


@pytest.mark.parametrize("p", [Problem(1, 2, 5, 6, 3), Problem(2, 2, 6, 5, 3, dilations=(2, 2, 4)),
                               Problem(1, 2, 6, 7, 5), Problem(1, 3, 4, 4, 1)], ids=_id)
def test_gradients_match_central_differences(p):
    t = _inputs(p, seed=21)
    g, x, y, Wg, bias = t["grad_out"], t["x"], t["y"], t["weight"], t["bias"]
    dx, dy, dW, db = oracle.backward(g, x, y, Wg, bias, p.K, p.dilations)
    rng = np.random.default_rng(1)
    h = 1e-3
    for name, arr, grad in (("x", x, dx), ("y", y, dy), ("W", Wg, dW), ("bias", bias, db)):
        for flat in rng.integers(0, arr.size, 6):
            args = {"x": x, "y": y, "W": Wg, "bias": bias}
            plus = {k: v.copy() for k, v in args.items()}
            minus = {k: v.copy() for k, v in args.items()}
            plus[name].reshape(-1)[flat] += h
            minus[name].reshape(-1)[flat] -= h
            fd = (_loss(g, plus["x"], plus["y"], plus["W"], plus["bias"], p.K, p.dilations) -
                  _loss(g, minus["x"], minus["y"], minus["W"], minus["bias"], p.K, p.dilations)) / (2 * h)
            got = grad.reshape(-1)[flat]
            assert abs(fd - got) <= 1e-7 * max(1.0, abs(fd)), (name, flat, fd, got)


@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_adjoint_identities(p):
    t = _inputs(p, seed=33)
    g, x, y, Wg, bias = t["grad_out"], t["x"], t["y"], t["weight"], t["bias"]
    out = oracle.forward(x, y, Wg, bias, p.K, p.dilations)
    dx, dy, dW, db = oracle.backward(g, x, y, Wg, bias, p.K, p.dilations)
    C = p.C
    total = float(np.sum(g * out))
    filt = float(np.sum(g[:, C:] * out[:, C:]))
    scale = float(np.sum(np.abs(g * out))) + 1.0
    assert abs(total - float(np.sum(dx * x))) <= 1e-12 * scale
    assert abs(filt - (float(np.sum(dW * Wg)) + float(np.sum(db * bias)))) <= 1e-12 * scale
    assert abs(filt - (float(np.sum(dy * y)) + float(np.sum(db * bias)))) <= 1e-12 * scale


def test_backward_points_match_full():
    p = Problem(2, 3, 6, 7, 3)
    t = _inputs(p, seed=2)
    g, x, y, Wg, bias = t["grad_out"], t["x"], t["y"], t["weight"], t["bias"]
    full = dict(zip(("dx", "dy", "dW", "dbias"), oracle.backward(g, x, y, Wg, bias, p.K, p.dilations)))
    rng = np.random.default_rng(4)
    for name, arr in full.items():
        idx = rng.integers(0, arr.size, 50)
        np.testing.assert_array_equal(oracle.backward_points(g, x, y, Wg, bias, p.K, name, idx, p.dilations),
                                      arr.reshape(-1)[idx])


def test_bf16_mode_equals_fp64_mode_on_bf16_exact_taps():
    """With integer inputs every tap is exactly representable in bf16, so the
    rounding step is the identity and both modes coincide exactly."""
    p = Problem(2, 3, 6, 5, 3)
    t = {k: _np(v) for k, v in make_integer_inputs(p, 9).items()}
    a = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations, bf16=False)
    b = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations, bf16=True)
    np.testing.assert_array_equal(a, b)
    ga = oracle.backward(t["grad_out"], t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations, bf16=False)
    gb = oracle.backward(t["grad_out"], t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations, bf16=True)
    for u, v in zip(ga, gb):
        np.testing.assert_array_equal(u, v)


def test_bf16_backward_uses_rounded_taps_for_dx():
    """Straight-through rounding: dx pairs grad with the rounded taps that
    multiplied x; dy/dW/dbias do not involve the taps at all."""
    p = Problem(1, 2, 6, 5, 3)
    t = {k: _np(v) for k, v in make_inputs(p, 17, "bfloat16").items()}
    args = (t["grad_out"], t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations)
    dx32, dy32, dW32, db32 = oracle.backward(*args, bf16=False)
    dx16, dy16, dW16, db16 = oracle.backward(*args, bf16=True)
    np.testing.assert_array_equal(dy32, dy16)
    np.testing.assert_array_equal(dW32, dW16)
    np.testing.assert_array_equal(db32, db16)
    out16 = oracle.forward(t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations, bf16=True)
    assert abs(float(np.sum(t["grad_out"] * out16)) - float(np.sum(dx16 * t["x"]))) < 1e-10
    assert not np.array_equal(dx32, dx16)


# ---------------------------------------------------------------- golden --

def test_handworked_golden():
    gold = json.load(open(os.path.join(HERE, "golden", "handworked_k3_3x3.json")))
    s = gold["shape"]
    B, C, H, W, K = s["B"], s["C"], s["H"], s["W"], s["K"]
    dils = tuple(s["dilations"])
    x = np.array(gold["x"], dtype=np.float64).reshape(B, C, H, W)
    y = np.full((B, C, H, W), gold["y_constant"])
    Wg = np.zeros((3 * C * K * K, C))
    bias = np.array(gold["bias_per_dilation"] * 3, dtype=np.float64)
    out = oracle.forward(x, y, Wg, bias, K, dils)
    np.testing.assert_array_equal(out[0, 0], x[0, 0])
    np.testing.assert_array_equal(out[0, 1], np.array(gold["out_d1"], dtype=np.float64))
    np.testing.assert_array_equal(out[0, 2], np.array(gold["out_d3"], dtype=np.float64))
    np.testing.assert_array_equal(out[0, 3], np.array(gold["out_d5"], dtype=np.float64))
    g = np.zeros((B, 4 * C, H, W))
    oh = gold["grad_onehot"]
    g[0, oh["channel"], oh["h"], oh["w"]] = 1.0
    dx, dy, dW, db = oracle.backward(g, x, y, Wg, bias, K, dils)
    np.testing.assert_array_equal(dx[0, 0], np.array(gold["dx"], dtype=np.float64))
    want_db = np.array(gold["dbias_d1"] + gold["dbias_d3"] + gold["dbias_d5"], dtype=np.float64)
    np.testing.assert_array_equal(db, want_db)
    np.testing.assert_array_equal(dW[:, 0], want_db)
    assert not dy.any()


# ------------------------------------------------------- planted mistakes --

def test_pins_catch_planted_mistakes():
    """Plausible oracle mistakes must fail the pins: emulate each on the oracle's
    own inputs and check that the Unfold reference disagrees."""
    p = Problem(1, 2, 7, 6, 3)
    t = _inputs(p)
    ref = unfold_reference(t["x"], t["taps"], p.K, p.dilations)
    T = t["taps"]
    # convolution instead of correlation (flipped taps)
    Tflip = T.reshape(p.B, 3 * p.C, p.K, p.K, p.H, p.W)[:, :, ::-1, ::-1].reshape(T.shape)
    wrong = oracle.filter_pregenerated(t["x"], np.ascontiguousarray(Tflip), p.K, p.dilations)
    assert np.max(np.abs(wrong - ref)) > 1e-3
    # channel-major vs dilation-major tap order swapped
    Tswap = T.reshape(p.B, 3, p.C, p.K * p.K, p.H, p.W).transpose(0, 2, 1, 3, 4, 5).reshape(T.shape)
    wrong = oracle.filter_pregenerated(t["x"], np.ascontiguousarray(Tswap), p.K, p.dilations)
    assert np.max(np.abs(wrong - ref)) > 1e-3
    # dropped bias
    out_nb = oracle.forward(t["x"], t["y"], t["weight"], None, p.K, p.dilations)
    Tg = generator_reference(t["y"], t["weight"], t["bias"])
    assert np.max(np.abs(out_nb - unfold_reference(t["x"], Tg, p.K, p.dilations))) > 1e-3


# ------------------------------------------------- filter-only backward --
# README section "CUDA 动态过滤": with the taps given, the backward forms dX and
# dK (the taps' gradient) without a patch matrix.  Pinned to torch autograd
# through the Unfold reference, and to the adjoint identities of a bilinear map.

def _unfold_filter_autograd(x, T, g, K, dils):
    """(dx, dT) of L = <g, filter(x, T)> by torch autograd through F.unfold."""
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    Tt = torch.tensor(T, dtype=torch.float64, requires_grad=True)
    B, C, H, W = x.shape
    K2 = K * K
    outs = [xt]
    for di, d in enumerate(dils):
        U = F.unfold(xt, K, dilation=d, padding=d * (K // 2))
        Td = Tt[:, di * C * K2:(di + 1) * C * K2].reshape(B, C * K2, H * W)
        outs.append((U * Td).reshape(B, C, K2, H * W).sum(2).reshape(B, C, H, W))
    L = (torch.cat(outs, 1) * torch.as_tensor(g, dtype=torch.float64)).sum()
    L.backward()
    return _np(xt.grad), _np(Tt.grad)


@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_filter_backward_matches_unfold_autograd(p):
    t = _inputs(p)
    dx, dT = oracle.filter_backward(t["grad_out"], t["x"], t["taps"], p.K, p.dilations)
    rdx, rdT = _unfold_filter_autograd(t["x"], t["taps"], t["grad_out"], p.K, p.dilations)
    np.testing.assert_allclose(dx, rdx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dT, rdT, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_filter_backward_adjoint_identities(p):
    """The filter is linear in x and in T: <g,out> = <dx,x> = <dT,T> + <g_0,x>."""
    t = _inputs(p, seed=21)
    x, T, g = t["x"], t["taps"], t["grad_out"]
    L = float((g * oracle.filter_pregenerated(x, T, p.K, p.dilations)).sum())
    dx, dT = oracle.filter_backward(g, x, T, p.K, p.dilations)
    assert abs(float((dx * x).sum()) - L) <= 1e-12 * max(1.0, abs(L))
    assert abs(float((dT * T).sum() + (g[:, :p.C] * x).sum()) - L) <= 1e-12 * max(1.0, abs(L))


def test_filter_backward_dT_sums_to_fused_dbias():
    """dT is the fused path's dK: summed over batch and pixels it is dbias."""
    p = Problem(2, 3, 6, 5, 3)
    t = _inputs(p, seed=5)
    _, dT = oracle.filter_backward(t["grad_out"], t["x"], t["taps"], p.K, p.dilations)
    _, _, _, db = oracle.backward(t["grad_out"], t["x"], t["y"], t["weight"], t["bias"], p.K, p.dilations)
    np.testing.assert_allclose(dT.sum(axis=(0, 2, 3)), db, rtol=1e-12, atol=1e-12)


def test_filter_backward_pins_catch_planted_mistakes():
    """A gather at +offset (flipped taps) or a dropped identity term must fail the autograd pin."""
    p = Problem(1, 2, 7, 6, 3)
    t = _inputs(p)
    x, T, g = t["x"], t["taps"], t["grad_out"]
    rdx, _ = _unfold_filter_autograd(x, T, g, p.K, p.dilations)
    Tflip = np.ascontiguousarray(T.reshape(p.B, 3 * p.C, p.K, p.K, p.H, p.W)[:, :, ::-1, ::-1].reshape(T.shape))
    wrong, _ = oracle.filter_backward(g, x, Tflip, p.K, p.dilations)
    assert np.max(np.abs(wrong - rdx)) > 1e-3
    g_no_id = g.copy()
    g_no_id[:, :p.C] = 0.0
    wrong, _ = oracle.filter_backward(g_no_id, x, T, p.K, p.dilations)
    assert np.max(np.abs(wrong - rdx)) > 1e-3
