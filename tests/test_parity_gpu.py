"""GPU parity: the CUDA library (through its C ABI) against the CPU FP64 oracle.

Same seeded inputs on both sides (dynamic_dilated_depthwise_gb300.inputs).
Every problem, the five workloads at full size included, is compared element
by element over whole tensors.  Integer-valued inputs make every intermediate exact,
so addressing (tap order, offset signs, zero padding, tile tails) is checked
bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_dilated_depthwise_gb300 import binding, build
from dynamic_dilated_depthwise_gb300.inputs import (SEEDS, WORKLOADS, Problem, make_inputs,
                                                    make_integer_inputs)
from parity import (assert_bf16_close_with_ties, assert_forward_close, assert_grad_close, dx_tie_allowance,
                    forward_tie_allowance, full_size_section, to64)

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "bfloat16"]

SMALL = [
    Problem(2, 24, 15, 17, 3),               # the regression shape: non-pow2 C, odd borders
    Problem(1, 16, 9, 130, 3),               # rows wider than one 128-pixel tile, ragged
    Problem(2, 40, 37, 45, 3),               # several tiles and a ragged tail, C % 16 != 0
    Problem(1, 64, 32, 32, 3),               # C = 64 as in the main workloads
    Problem(1, 8, 12, 11, 5),                # K = 5
    Problem(2, 5, 6, 7, 1),                  # K = 1
    Problem(1, 6, 13, 9, 7),                 # K = 7
    Problem(1, 12, 20, 19, 3, (2, 2, 4)),    # other dilations
    Problem(1, 3, 1, 1, 3),                  # 1x1 image: every neighbour is padding
    Problem(3, 4, 2, 33, 3),                 # image thinner than the halo
]


# Shapes the tensor-core forward takes (bf16, K = 3, C % 8 == 0, C <= 64, W % 8 == 0):
# ragged row tiles, partial channel groups, several rows per tile, H below the tile height.
TC_SHAPES = [
    Problem(1, 16, 5, 136, 3),               # W = 136: one full and one 8-pixel tile per row
    Problem(2, 24, 10, 24, 3),               # C = 24: partial second channel group; 5 rows per tile
    Problem(1, 48, 12, 256, 3),              # two tiles per row, three channel groups
    Problem(1, 8, 3, 40, 3, (2, 2, 4)),      # C = 8, other dilations, image shorter than a tile
    Problem(2, 64, 7, 200, 3),               # second tile of each row holds 72 pixels
    Problem(1, 32, 1, 8, 3),                 # a single 8-pixel row
    Problem(3, 64, 40, 40, 3),               # several images, 3 rows per tile
]


def _id(p):
    return f"B{p.B}C{p.C}_{p.H}x{p.W}_K{p.K}_d{''.join(map(str, p.dilations))}"


@pytest.fixture(scope="session", autouse=True)
def library():
    build.build()
    binding.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()


def _dev(t):
    return {k: v.cuda() for k, v in t.items()}


def run_forward(d, p):
    return binding.forward(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations)


def run_backward(d, p, flags=0, workspace=None):
    return binding.backward(d["grad_out"], d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations, flags=flags,
                            workspace=workspace)


def min_workspace(d, p):
    """The smallest workspace the backward accepts (the dW/dbias partials alone),
    so dX stages its operands itself."""
    prob = binding.make_problem(p.B, p.C, p.H, p.W, p.K, p.dilations,
                                binding.DDPM_BFLOAT16 if d["x"].dtype == torch.bfloat16 else binding.DDPM_FLOAT32)
    n = binding.ddpm_backward_workspace_min(prob)
    assert n < binding.ddpm_backward_workspace_size(prob)
    return torch.empty(n, dtype=torch.uint8, device=d["x"].device)


# ------------------------------------------------------------ small, full --

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_forward_matches_oracle(p, dtype):
    h = make_inputs(p, 100, dtype)
    d = _dev(h)
    out = run_forward(d, p)
    torch.cuda.synchronize()
    ref = oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=dtype == "bfloat16")
    assert_forward_close(out, ref, dtype)
    assert torch.equal(out[:, :p.C].cpu(), h["x"]), "passthrough channels must be a bit-exact copy of x"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_filter_pregenerated_matches_oracle(p, dtype):
    h = make_inputs(p, 200, dtype, grad=False, taps=True)
    d = _dev(h)
    out = binding.filter_pregenerated(d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    ref = oracle.filter_pregenerated(h["x"], h["taps"], p.K, p.dilations)
    assert_forward_close(out, ref, dtype)
    assert torch.equal(out[:, :p.C].cpu(), h["x"])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_backward_matches_oracle(p, dtype):
    h = make_inputs(p, 300, dtype)
    d = _dev(h)
    dx, dy, dw, db = run_backward(d, p, flags=binding.DDPM_FLAG_TF32_BACKWARD)
    torch.cuda.synchronize()
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations,
                          bf16=dtype == "bfloat16")
    for name, got, want in zip(("dx", "dy", "dW", "dbias"), (dx, dy, dw, db), ref):
        assert_grad_close(got, want, dtype, name)


# Shapes whose rows are whole 16-byte vectors (W % 8 == 0): the filter takes its tiled
# shared-memory kernel.  Ragged 64-column and row tiles,
# halo radius 10 (K = 5), 15 (K = 7) and 16 (K = 3, the widest the x window takes), a
# 1-row image, other dilations, and W a multiple of the FP32 vector only.
FILTER_TILED = TC_SHAPES + [
    Problem(1, 8, 40, 72, 5),                # K = 5: halo radius 10
    Problem(1, 4, 19, 24, 7),                # K = 7: halo radius 15
    Problem(2, 6, 33, 64, 3, (2, 3, 4)),
    Problem(1, 4, 40, 64, 3, (4, 8, 16)),    # K = 3: halo radius 16
    Problem(2, 8, 10, 36, 3),                # W % 8 != 0: bf16 takes the per-element kernel
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", FILTER_TILED, ids=_id)
def test_filter_tiled_matches_oracle(p, dtype):
    h = make_inputs(p, 250, dtype, grad=False, taps=True)
    d = _dev(h)
    out = binding.filter_pregenerated(d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    ref = oracle.filter_pregenerated(h["x"], h["taps"], p.K, p.dilations)
    assert_forward_close(out, ref, dtype)
    assert torch.equal(out[:, :p.C].cpu(), h["x"])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", FILTER_TILED[:4], ids=_id)
def test_filter_tiled_integer_bit_exact(p, dtype):
    """Integer-valued x and taps: every product and sum is exact, so the tiled
    kernel's neighbour addressing must match the oracle bit for bit."""
    g = torch.Generator().manual_seed(11)
    x = torch.randint(-2, 3, (p.B, p.C, p.H, p.W), generator=g).to(torch.float32)
    taps = torch.randint(-2, 3, (p.B, p.O, p.H, p.W), generator=g).to(torch.float32)
    td = torch.bfloat16 if dtype == "bfloat16" else torch.float32
    out = binding.filter_pregenerated(x.to(td).cuda(), taps.to(td).cuda(), p.K, p.dilations)
    torch.cuda.synchronize()
    ref = oracle.filter_pregenerated(x.double().numpy(), taps.double().numpy(), p.K, p.dilations)
    np.testing.assert_array_equal(out.double().cpu().numpy(), ref)


# ------------------------------------------------- tensor-core forward path --

def _traced_kernels(fn):
    binding.ddpm_trace_read()
    binding.ddpm_trace_enable(True)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        binding.ddpm_trace_enable(False)
    return [name for name, _ in binding.ddpm_trace_read()]


@pytest.mark.parametrize("p", TC_SHAPES, ids=_id)
def test_tc_forward_matches_oracle_and_cuda_cores(p):
    h = make_inputs(p, 700, "bfloat16", grad=False)
    d = _dev(h)
    names = _traced_kernels(lambda: run_forward(d, p))
    assert names == ["forward_tc"], f"expected the tensor-core forward, got {names}"
    out = run_forward(d, p)
    simt = binding.forward(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations,
                           flags=binding.DDPM_FLAG_CUDA_CORES)
    torch.cuda.synchronize()
    ref = oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=True)
    assert_forward_close(out, ref, "bfloat16")
    assert_forward_close(simt, ref, "bfloat16")
    assert torch.equal(out[:, :p.C].cpu(), h["x"])


# K = 5 shapes the tensor-core forward takes (4-channel groups, halo radius up to 10)
TC_SHAPES_K5 = [
    Problem(1, 8, 12, 64, 5),                # one row of 64-column tiles, halo radius 10
    Problem(2, 16, 9, 136, 5),               # ragged row tile, odd row count
    Problem(1, 64, 20, 128, 5),              # C = 64 as in the K = 5 workload
    Problem(1, 24, 5, 24, 5, (1, 2, 3)),     # whole-row tiles, other dilations
    Problem(1, 8, 7, 40, 5, (2, 4, 5)),      # whole-row tiles of 3 rows, halo radius 10
]


@pytest.mark.parametrize("p", TC_SHAPES_K5, ids=_id)
def test_tc_forward_k5_matches_oracle_and_cuda_cores(p):
    test_tc_forward_matches_oracle_and_cuda_cores(p)


@pytest.mark.parametrize("p", TC_SHAPES[:5] + TC_SHAPES_K5[:3], ids=_id)
def test_tc_forward_integer_bit_exact(p):
    h = make_integer_inputs(p, 9, "bfloat16", grad=False)
    out = run_forward(_dev(h), p)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to64(out), oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K,
                                                            p.dilations, bf16=True))


def test_tc_forward_without_bias():
    p = Problem(1, 24, 6, 64, 3)
    h = make_inputs(p, 701, "bfloat16", grad=False)
    d = _dev(h)
    out = binding.forward(d["x"], d["y"], d["weight"], None, p.K, p.dilations)
    torch.cuda.synchronize()
    assert_forward_close(out, oracle.forward(h["x"], h["y"], h["weight"], None, p.K, p.dilations, bf16=True),
                         "bfloat16")


def test_tc_forward_repeated_calls_identical():
    p = Problem(1, 64, 64, 128, 3)
    d = _dev(make_inputs(p, 702, "bfloat16", grad=False))
    a = run_forward(d, p)
    b = run_forward(d, p)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert binding.ddpm_get_device_error() == 0


# ------------------------------------- FP32 forward on TF32 tensor cores (3xTF32) --

# Shapes the 3xTF32 forward takes (FP32, K = 3 with halo radius <= 8 or K = 5 with halo
# radius <= 12; C % 4 == 0, C <= 64, W % 4 == 0): ragged 64-column
# tiles, whole-row tiles (W < 64), several images, a single-row image, other dilations,
# C below one K block, and for K = 5 the radius-10 halo of dilation 5.
TF32X3_SHAPES = [
    Problem(1, 16, 5, 136, 3),               # two full tiles and an 8-pixel one per row
    Problem(2, 24, 10, 24, 3),               # whole-row tiles of 5 rows, C = 24
    Problem(1, 64, 12, 256, 3),              # C = 64, four tiles per row
    Problem(1, 8, 3, 40, 3, (2, 2, 4)),      # other dilations, image shorter than a tile
    Problem(2, 64, 7, 200, 3),               # last tile of each row 8 pixels wide
    Problem(1, 4, 1, 12, 3),                 # one row, C = 4
    Problem(3, 64, 40, 40, 3),               # several images
]
TF32X3_K5_SHAPES = [
    Problem(1, 64, 12, 256, 5),              # C = 64, four tiles per row, halo radius 10
    Problem(2, 16, 10, 24, 5),               # whole-row tiles of 5 rows
    Problem(1, 4, 7, 200, 5),                # C = 4 (two channel groups), 8-pixel last tile
    Problem(1, 8, 3, 40, 5, (1, 2, 2)),      # other dilations, image shorter than a tile
    Problem(3, 24, 33, 36, 5, (2, 4, 6)),    # radius 12, several images, ragged rows
]
TF32X3 = binding.DDPM_FLAG_TF32X3_FORWARD


@pytest.mark.parametrize("p", TF32X3_SHAPES + TF32X3_K5_SHAPES, ids=_id)
def test_tf32x3_forward_matches_oracle(p):
    h = make_inputs(p, 720, "float32", grad=False)
    d = _dev(h)
    run = lambda: binding.forward(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations, flags=TF32X3)
    names = _traced_kernels(run)
    assert names == ["forward_tf32"], f"expected the 3xTF32 forward, got {names}"
    out = run()
    torch.cuda.synchronize()
    ref = oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations)
    assert_forward_close(out, ref, "float32", "out (3xTF32)")
    assert torch.equal(out[:, :p.C].cpu(), h["x"])


@pytest.mark.parametrize("p", TF32X3_SHAPES[:5] + TF32X3_K5_SHAPES[:3], ids=_id)
def test_tf32x3_forward_integer_bit_exact(p):
    """Integer inputs: every operand is exact in TF32 (the lo parts are zero), so the
    split GEMM and the FP32 filter must match the oracle bit for bit."""
    h = make_integer_inputs(p, 21, "float32", grad=False)
    d = _dev(h)
    out = binding.forward(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations, flags=TF32X3)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to64(out), oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations))


def test_tf32x3_forward_without_bias_and_ineligible_shapes():
    p = Problem(1, 24, 6, 64, 3)
    h = make_inputs(p, 721, "float32", grad=False)
    d = _dev(h)
    out = binding.forward(d["x"], d["y"], d["weight"], None, p.K, p.dilations, flags=TF32X3)
    torch.cuda.synchronize()
    assert_forward_close(out, oracle.forward(h["x"], h["y"], h["weight"], None, p.K, p.dilations), "float32",
                         "out (3xTF32, no bias)")
    # a K = 5 halo radius above 12, C % 4 != 0 and W % 4 != 0 keep the IEEE kernel under
    # the flag
    for q in (Problem(1, 8, 12, 16, 5, (1, 3, 7)), Problem(1, 6, 6, 16, 5), Problem(1, 8, 9, 10, 3)):
        hq = _dev(make_inputs(q, 722, "float32", grad=False))
        names = _traced_kernels(lambda: binding.forward(hq["x"], hq["y"], hq["weight"], hq["bias"], q.K, q.dilations,
                                                        flags=TF32X3))
        assert names == ["forward_simt"], names


# ------------------------------------------------ tensor-core backward path --

# + H*W a multiple of 2048 with several images and fewer than eight channel chunks:
# the persistent TMA pack
# + enough 8x64 super tiles (>= half the SMs) that dY keeps four sub-tiles per CTA, with
# ragged rows and columns
TC_BWD_SHAPES = list(TC_SHAPES) + [Problem(2, 24, 32, 64, 3), Problem(4, 16, 70, 136, 3)]


@pytest.mark.parametrize("p", TC_BWD_SHAPES, ids=_id)
def test_tc_backward_matches_oracle_and_cuda_cores(p):
    h = make_inputs(p, 800, "bfloat16")
    d = _dev(h)
    names = _traced_kernels(lambda: run_backward(d, p))
    assert {"pack_chunks", "bwd_dx_tc_packed", "bwd_dy_tc", "bwd_dw_tc"} <= set(names), \
        f"expected the tensor-core backward, got {names}"
    ws = min_workspace(d, p)
    names_small = _traced_kernels(lambda: run_backward(d, p, workspace=ws))
    assert {"bwd_dx_tc", "bwd_dy_tc", "bwd_dw_tc"} <= set(names_small), names_small
    assert "bwd_dx_tc_packed" not in names_small
    got = run_backward(d, p)
    staged = run_backward(d, p, workspace=ws)
    simt = run_backward(d, p, flags=binding.DDPM_FLAG_CUDA_CORES)
    torch.cuda.synchronize()
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=True)
    for name, a, b, want in zip(("dx", "dy", "dW", "dbias"), got, simt, ref):
        assert_grad_close(a, want, "bfloat16", name)
        assert_grad_close(b, want, "bfloat16", name + " (cuda cores)")
    assert_grad_close(staged[0], ref[0], "bfloat16", "dx (operands staged in the kernel)")


@pytest.mark.parametrize("p", [Problem(1, 16, 8, 16, 3), Problem(1, 24, 4, 24, 3, (2, 2, 4)), Problem(2, 64, 4, 16, 3)],
                         ids=_id)
def test_tc_backward_integer_bit_exact(p):
    """Integer inputs with at most 256 pixels: every dW / dbias sum is exact in bf16."""
    h = make_integer_inputs(p, 11, "bfloat16")
    d = _dev(h)
    assert {"bwd_dx_tc_packed", "bwd_dw_tc"} <= set(_traced_kernels(lambda: run_backward(d, p)))
    dx, dy, dw, db = run_backward(d, p)
    dx_staged = run_backward(d, p, workspace=min_workspace(d, p))[0]
    torch.cuda.synchronize()
    rdx, rdy, rdw, rdb = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations,
                                         bf16=True)
    np.testing.assert_array_equal(to64(dx), rdx)
    np.testing.assert_array_equal(to64(dx_staged), rdx)
    np.testing.assert_array_equal(to64(dy), rdy)
    np.testing.assert_array_equal(to64(dw), rdw)
    np.testing.assert_array_equal(to64(db), rdb)


# K = 5: dW and dY on tensor cores (blocks of 5 channels x 25 taps, 96-column x
# windows, halo radius up to 10); dX on tensor cores with grad gathered from L2 when the
# workspace holds the channel-chunked copies, on CUDA cores with the minimum workspace.
TC_BWD_K5_SHAPES = [
    Problem(1, 64, 16, 64, 5),               # C = 64: 13 channel blocks per dilation, halo radius 10
    Problem(2, 24, 10, 72, 5),               # ragged 64-column tiles, several images, a partial block
    Problem(1, 8, 6, 128, 5, (1, 2, 3)),     # other dilations, one full and one partial block
    Problem(1, 16, 3, 16, 5, (2, 4, 5)),     # image smaller than the halo
    Problem(6, 8, 38, 136, 5),               # dY with four sub-tiles per CTA, ragged rows and columns
]


@pytest.mark.parametrize("p", TC_BWD_K5_SHAPES, ids=_id)
def test_tc_backward_k5_matches_oracle_and_cuda_cores(p):
    h = make_inputs(p, 810, "bfloat16")
    d = _dev(h)
    names = set(_traced_kernels(lambda: run_backward(d, p)))
    assert {"pack_chunks", "bwd_dx_gather", "bwd_dy_tc", "bwd_dw_tc"} <= names, names
    ws = min_workspace(d, p)
    names_small = set(_traced_kernels(lambda: run_backward(d, p, workspace=ws)))
    assert {"bwd_dx_simt", "bwd_dy_tc", "bwd_dw_tc"} <= names_small, names_small
    got = run_backward(d, p)
    small = run_backward(d, p, workspace=ws)
    simt = run_backward(d, p, flags=binding.DDPM_FLAG_CUDA_CORES)
    torch.cuda.synchronize()
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=True)
    for name, a, b, want in zip(("dx", "dy", "dW", "dbias"), got, simt, ref):
        assert_grad_close(a, want, "bfloat16", name + " (K = 5)")
        assert_grad_close(b, want, "bfloat16", name + " (K = 5, cuda cores)")
    assert_grad_close(small[0], ref[0], "bfloat16", "dx (K = 5, minimum workspace)")


@pytest.mark.parametrize("p", [Problem(1, 16, 8, 16, 5), Problem(2, 8, 4, 16, 5, (1, 2, 3))], ids=_id)
def test_tc_backward_k5_integer_bit_exact(p):
    """Integer inputs with at most 256 pixels: every dW / dbias sum is exact in bf16."""
    h = make_integer_inputs(p, 12, "bfloat16")
    d = _dev(h)
    assert {"bwd_dx_gather", "bwd_dy_tc", "bwd_dw_tc"} <= set(_traced_kernels(lambda: run_backward(d, p)))
    got = run_backward(d, p)
    torch.cuda.synchronize()
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=True)
    for a, want in zip(got, ref):
        np.testing.assert_array_equal(to64(a), want)


# ----------------------------------------- filter-only backward (taps given) --

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", SMALL, ids=_id)
def test_filter_backward_matches_oracle(p, dtype):
    h = make_inputs(p, 900, dtype, grad=True, taps=True)
    d = _dev(h)
    names = _traced_kernels(lambda: binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K,
                                                                         p.dilations))
    assert names == ["filter_bwd_dx", "filter_bwd_dtaps"], names
    dx, dT = binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K, p.dilations)
    dx_only, none = binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K, p.dilations,
                                                         with_dtaps=False)
    torch.cuda.synchronize()
    rdx, rdT = oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
    assert_grad_close(dx, rdx, dtype, "dx")
    assert_grad_close(dT, rdT, dtype, "dtaps")
    assert none is None and torch.equal(dx_only, dx)


# Shapes the tiled filter-backward kernels take (W a multiple of 8): every K, ragged
# tile rows, several tiles per row, several images, other dilations.
FILTER_TILED_BWD = [
    Problem(1, 3, 9, 24, 3), Problem(2, 2, 19, 16, 5), Problem(1, 2, 7, 40, 7), Problem(2, 3, 5, 8, 1),
    Problem(1, 2, 21, 136, 3, (2, 2, 4)), Problem(1, 2, 10, 72, 3, (1, 6, 2)), Problem(2, 2, 17, 64, 5, (3, 1, 2)),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", FILTER_TILED_BWD, ids=_id)
def test_filter_backward_tiled_matches_oracle(p, dtype):
    h = make_inputs(p, 905, dtype, grad=True, taps=True)
    d = _dev(h)
    dx, dT = binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    rdx, rdT = oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
    assert_grad_close(dx, rdx, dtype, "dx")
    assert_grad_close(dT, rdT, dtype, "dtaps")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", FILTER_TILED_BWD, ids=_id)
def test_filter_backward_tiled_integer_bit_exact(p, dtype):
    h = make_integer_inputs(p, 19, dtype, taps=True)
    d = _dev(h)
    dx, dT = binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    rdx, rdT = oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
    np.testing.assert_array_equal(to64(dx), rdx)
    np.testing.assert_array_equal(to64(dT), rdT)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", [Problem(2, 24, 15, 17, 3), Problem(1, 8, 12, 11, 5), Problem(1, 12, 20, 19, 3, (2, 2, 4)),
                               Problem(2, 5, 6, 7, 1), Problem(1, 6, 13, 9, 7)], ids=_id)
def test_filter_backward_integer_bit_exact(p, dtype):
    """Integer inputs: every product and sum is a small integer, exact in bf16 and fp32."""
    h = make_integer_inputs(p, 17, dtype, taps=True)
    d = _dev(h)
    dx, dT = binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    rdx, rdT = oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
    np.testing.assert_array_equal(to64(dx), rdx)
    np.testing.assert_array_equal(to64(dT), rdT)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("name", ["b1_c64_128x128_k3", "b1_c64_128x128_k5"])
def test_filter_backward_full_size(name, dtype):
    """The 128x128, C=64 filter workloads (K = 3 and 5), compared over whole tensors."""
    p = WORKLOADS[name]
    h = make_inputs(p, SEEDS[name], dtype, grad=True, taps=True)
    d = _dev(h)
    dx, dT = binding.filter_pregenerated_backward(d["grad_out"], d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    rdx, rdT = oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
    with full_size_section():
        assert_grad_close(dx, rdx, dtype, f"dx {name} {dtype} (filter)")
        assert_grad_close(dT, rdT, dtype, f"dtaps {name} {dtype} (filter)")
    assert binding.ddpm_get_device_error() == 0


# --------------------------------------------- FP32 backward, TF32 dW / dbias --

# Shapes the TF32 dW kernel takes (FP32, K = 3, C <= 64, W % 4 == 0, dilations <= 6; K = 5 below):
# ragged 64-pixel row tiles, partial blocks of 14 channels, other dilations, several images.
TF32_SHAPES = [
    Problem(1, 16, 9, 132, 3),               # three tiles per row, the last 4 pixels wide
    Problem(2, 24, 10, 24, 3),               # C = 24: a partial channel block; one short tile per row
    Problem(1, 64, 12, 64, 3),               # C = 64 as in the main workloads
    Problem(1, 12, 7, 40, 3, (2, 2, 4)),     # other dilations
    Problem(3, 8, 5, 68, 3, (1, 6, 2)),      # halo radius 6, several images
    Problem(2, 32, 9, 36, 3, (1, 6, 2)),     # TF32 dY: ragged 4 x 32 tiles, halo radius 6, two images
    Problem(1, 48, 6, 64, 3),                # TF32 dY with N = 48
    Problem(1, 10, 6, 36, 3),                # C % 4 != 0: dX and dY stay IEEE FP32
    Problem(2, 20, 19, 28, 3, (3, 1, 2)),    # TF32 dX: C % 8 == 4 (a zero chunk), ragged 16 x 8 tiles
]


def _tf32_dx_applies(p):
    return p.C % 4 == 0 and p.W % 4 == 0 and max(p.dilations) * (p.K // 2) <= 6


@pytest.mark.parametrize("p", TF32_SHAPES, ids=_id)
def test_tf32_backward_matches_oracle(p):
    h = make_inputs(p, 850, "float32")
    d = _dev(h)
    flags = binding.DDPM_FLAG_TF32_BACKWARD
    names = _traced_kernels(lambda: run_backward(d, p, flags=flags))
    assert "bwd_dw_tf32" in names and "bwd_dw_partial_simt" not in names, names
    tf32_dy = p.C % 16 == 0
    assert ("bwd_dy_tf32" in names) == tf32_dy and ("bwd_dy_simt" in names) != tf32_dy, names
    tf32_dx = _tf32_dx_applies(p)
    assert ("bwd_dx_tf32" in names) == tf32_dx and ("bwd_dx_simt" in names) != tf32_dx, names
    got = run_backward(d, p, flags=flags)
    ieee = run_backward(d, p)
    torch.cuda.synchronize()
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=False)
    for name, a, want in zip(("dx", "dy", "dW", "dbias"), got, ref):
        assert_grad_close(a, want, "float32", name)
        assert_grad_close(ieee[("dx", "dy", "dW", "dbias").index(name)], want, "float32", name + " (IEEE)")
    # where a TF32 kernel does not apply the flag leaves that gradient in IEEE FP32
    if not tf32_dx:
        assert torch.equal(got[0], ieee[0])
    if not tf32_dy:
        assert torch.equal(got[1], ieee[1])


def test_tf32_backward_workspace_fallbacks():
    """A workspace without room for the copy of y keeps dX on CUDA cores (dY still on
    TF32); the partials alone keep both there.  Each result still matches the oracle."""
    p = Problem(1, 32, 20, 40, 3)
    h = make_inputs(p, 851, "float32")
    d = _dev(h)
    flags = binding.DDPM_FLAG_TF32_BACKWARD
    prob = binding.make_problem(p.B, p.C, p.H, p.W, p.K, p.dilations, binding.DDPM_FLOAT32, flags)
    full = binding.ddpm_backward_workspace_size(prob)
    ymin = binding.ddpm_backward_workspace_min(prob)
    wt = 27 * p.C * p.C * 4
    dy_only = (ymin + 255) // 256 * 256 + wt
    assert full >= dy_only + 4 * p.B * p.C * p.H * p.W * 4
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=False)
    for nbytes, want in ((full, {"bwd_dx_tf32", "bwd_dy_tf32"}), (dy_only, {"bwd_dx_simt", "bwd_dy_tf32"}),
                         (ymin, {"bwd_dx_simt", "bwd_dy_simt"})):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        names = set(_traced_kernels(lambda: run_backward(d, p, flags=flags, workspace=ws)))
        assert want <= names, (nbytes, names)
        got = run_backward(d, p, flags=flags, workspace=ws)
        torch.cuda.synchronize()
        for name, a, r in zip(("dx", "dy", "dW", "dbias"), got, ref):
            assert_grad_close(a, r, "float32", f"{name} (workspace {nbytes})")


@pytest.mark.parametrize("p", TF32_SHAPES, ids=_id)
def test_tf32_backward_integer_bit_exact(p):
    """Integer inputs: every product and partial sum is exact in TF32 / FP32."""
    h = make_integer_inputs(p, 13, "float32")
    d = _dev(h)
    dx, dy, dw, db = run_backward(d, p, flags=binding.DDPM_FLAG_TF32_BACKWARD)
    torch.cuda.synchronize()
    rdx, rdy, rdw, rdb = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations,
                                         bf16=False)
    np.testing.assert_array_equal(to64(dw), rdw)
    np.testing.assert_array_equal(to64(db), rdb)
    np.testing.assert_array_equal(to64(dx), rdx)
    np.testing.assert_array_equal(to64(dy), rdy)


# K = 5: the TF32 dW kernel takes blocks of 5 channels (125 taps of the 128 MMA rows) and
# 96-column x windows (halo radius <= 10); dX and dY stay IEEE FP32 on CUDA cores.
TF32_DW_K5_SHAPES = [
    Problem(1, 10, 12, 72, 5),               # two channel blocks, a ragged 8-pixel tile
    Problem(2, 64, 9, 64, 5),                # C = 64: 13 blocks, the last holds 4 channels
    Problem(1, 12, 23, 36, 5, (1, 5, 3)),    # halo radius 10 (dilation 5), a short tile
    Problem(1, 7, 6, 132, 5, (2, 3, 4)),     # odd C, three tiles per row, radius 8
]


@pytest.mark.parametrize("p", TF32_DW_K5_SHAPES, ids=_id)
def test_tf32_backward_k5_matches_oracle(p):
    h = make_inputs(p, 852, "float32")
    d = _dev(h)
    flags = binding.DDPM_FLAG_TF32_BACKWARD
    names = _traced_kernels(lambda: run_backward(d, p, flags=flags))
    assert "bwd_dw_tf32" in names and "bwd_dw_partial_simt" not in names, names
    assert "bwd_dx_simt" in names and "bwd_dy_simt" in names, names
    got = run_backward(d, p, flags=flags)
    ieee = run_backward(d, p)
    torch.cuda.synchronize()
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=False)
    for name, a, want in zip(("dx", "dy", "dW", "dbias"), got, ref):
        assert_grad_close(a, want, "float32", name)
    assert torch.equal(got[0], ieee[0]) and torch.equal(got[1], ieee[1])


@pytest.mark.parametrize("p", TF32_DW_K5_SHAPES, ids=_id)
def test_tf32_backward_k5_integer_bit_exact(p):
    h = make_integer_inputs(p, 14, "float32")
    dx, dy, dw, db = run_backward(_dev(h), p, flags=binding.DDPM_FLAG_TF32_BACKWARD)
    torch.cuda.synchronize()
    rdx, rdy, rdw, rdb = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations,
                                         bf16=False)
    np.testing.assert_array_equal(to64(dw), rdw)
    np.testing.assert_array_equal(to64(db), rdb)
    np.testing.assert_array_equal(to64(dx), rdx)
    np.testing.assert_array_equal(to64(dy), rdy)


# ----------------------------------------------------- integer, bit-exact --

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", [Problem(2, 24, 15, 17, 3), Problem(1, 16, 9, 130, 3), Problem(1, 8, 12, 11, 5),
                               Problem(1, 12, 20, 19, 3, (2, 2, 4)), Problem(2, 5, 6, 7, 1),
                               Problem(1, 64, 16, 24, 3)], ids=_id)
def test_integer_inputs_bit_exact(p, dtype):
    h = make_integer_inputs(p, 7, dtype, taps=True)
    d = _dev(h)
    bf = dtype == "bfloat16"
    out = run_forward(d, p)
    filt = binding.filter_pregenerated(d["x"], d["taps"], p.K, p.dilations)
    dx, dy, dw, db = run_backward(d, p, flags=binding.DDPM_FLAG_TF32_BACKWARD)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to64(out), oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K,
                                                            p.dilations, bf16=bf))
    np.testing.assert_array_equal(to64(filt), oracle.filter_pregenerated(h["x"], h["taps"], p.K, p.dilations))
    rdx, rdy, rdw, rdb = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K,
                                         p.dilations, bf16=bf)
    np.testing.assert_array_equal(to64(dx), rdx)
    np.testing.assert_array_equal(to64(dy), rdy)
    if not bf or p.B * p.H * p.W <= 256:   # bf16 holds every integer sum only up to 256
        np.testing.assert_array_equal(to64(dw), rdw)
        np.testing.assert_array_equal(to64(db), rdb)


def test_integer_bf16_weight_grads_bit_exact_small_image():
    p = Problem(1, 24, 15, 17, 3)             # 255 pixels: every dW / dbias sum stays <= 255
    h = make_integer_inputs(p, 8, "bfloat16")
    dx, dy, dw, db = run_backward(_dev(h), p)
    torch.cuda.synchronize()
    _, _, rdw, rdb = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations,
                                     bf16=True)
    np.testing.assert_array_equal(to64(dw), rdw)
    np.testing.assert_array_equal(to64(db), rdb)


# ------------------------------------------------------------ edge cases --

@pytest.mark.parametrize("dtype", DTYPES)
def test_no_bias(dtype):
    p = Problem(2, 24, 15, 17, 3)
    h = make_inputs(p, 400, dtype)
    d = _dev(h)
    out = binding.forward(d["x"], d["y"], d["weight"], None, p.K, p.dilations)
    dx, dy, dw, db = binding.backward(d["grad_out"], d["x"], d["y"], d["weight"], None, p.K, p.dilations,
                                      with_dbias=False)
    torch.cuda.synchronize()
    bf = dtype == "bfloat16"
    assert db is None
    assert_forward_close(out, oracle.forward(h["x"], h["y"], h["weight"], None, p.K, p.dilations, bf16=bf), dtype)
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], None, p.K, p.dilations, bf16=bf)
    for name, got, want in zip(("dx", "dy", "dW"), (dx, dy, dw), ref[:3]):
        assert_grad_close(got, want, dtype, name)


@pytest.mark.parametrize("dtype", DTYPES)
def test_backward_deterministic(dtype):
    p = Problem(1, 64, 64, 64, 3)
    d = _dev(make_inputs(p, 500, dtype))
    a = run_backward(d, p)
    b = run_backward(d, p)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v), "backward must be bit-reproducible run to run"


def test_autograd_wrapper():
    p = Problem(1, 8, 10, 12, 3)
    h = make_inputs(p, 600, "float32")
    d = {k: v.cuda().requires_grad_(k in ("x", "y", "weight", "bias")) for k, v in h.items()}
    out = binding.DDPMCoreFunction.apply(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations)
    out.backward(d["grad_out"])
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations)
    for name, t, want in zip(("dx", "dy", "dW", "dbias"), ("x", "y", "weight", "bias"), ref):
        assert_grad_close(d[t].grad, want, "float32", name)


@pytest.mark.parametrize("dtype", DTYPES)
def test_filter_autograd_wrapper(dtype):
    p = Problem(1, 8, 10, 16, 3)
    h = make_inputs(p, 610, dtype, grad=True, taps=True)
    d = {k: v.cuda().requires_grad_(k in ("x", "taps")) for k, v in h.items()}
    out = binding.DDPMFilterFunction.apply(d["x"], d["taps"], p.K, p.dilations)
    out.backward(d["grad_out"])
    rdx, rdT = oracle.filter_backward(h["grad_out"], h["x"], h["taps"], p.K, p.dilations)
    assert_grad_close(d["x"].grad, rdx, dtype, "dx")
    assert_grad_close(d["taps"].grad, rdT, dtype, "dtaps")


def test_device_error_word_is_clear():
    p = Problem(1, 16, 8, 8, 3)
    run_forward(_dev(make_inputs(p, 1, "bfloat16", grad=False)), p)
    assert binding.ddpm_get_device_error() == 0


# ------------------------------------------------ full-size, whole tensors --
# Every workload at its full size, every element of every output compared with the
# oracle (the oracle takes ~1.5 s per 256x256 image on the host cores).

FULL_FORWARD = [("b1_c64_128x128_k3", "float32"), ("b1_c64_128x128_k3", "bfloat16"),
                ("b1_c64_128x128_k5", "float32"), ("b1_c64_128x128_k5", "bfloat16")]
FULL_TRAINING = [("b2_c24_15x17_k3", "float32"), ("b2_c24_15x17_k3", "bfloat16"),
                 ("b1_c64_256x256_k3", "bfloat16"), ("b1_c64_256x256_k3", "float32"),
                 ("b1_c64_128x128_k5", "bfloat16"), ("b1_c64_128x128_k5", "float32"),
                 ("b8_c64_256x256_k3", "bfloat16")]


def _f64_inputs(h):
    return {k: v.double().numpy() for k, v in h.items() if k != "taps"}


def _check_forward(out, h, p, dtype, what):
    """The fused forward over whole tensors; in bf16 an element above the bar must be
    explained by bf16 tap-rounding ties (see parity.assert_bf16_close_with_ties)."""
    bf = dtype == "bfloat16"
    ref = oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=bf)
    if not bf:
        assert_forward_close(out, ref, dtype, what)
        return
    h64 = _f64_inputs(h)
    assert_bf16_close_with_ties(out, ref, what, lambda idx: forward_tie_allowance(oracle, h64, p.K, p.dilations, idx))


@pytest.mark.parametrize("name,dtype", FULL_FORWARD, ids=lambda v: v)
def test_full_size_forward_and_filter(name, dtype):
    """Fused forward and filter-only (taps given) over whole output tensors."""
    p = WORKLOADS[name]
    h = make_inputs(p, SEEDS[name], dtype, grad=False, taps=True)
    d = _dev(h)
    out = run_forward(d, p)
    filt = binding.filter_pregenerated(d["x"], d["taps"], p.K, p.dilations)
    torch.cuda.synchronize()
    bf = dtype == "bfloat16"
    with full_size_section():
        _check_forward(out, h, p, dtype, f"{name} {dtype} out (fused)")
        assert_forward_close(filt, oracle.filter_pregenerated(h["x"], h["taps"], p.K, p.dilations), dtype,
                             f"{name} {dtype} out (filter)")
    assert torch.equal(out[:, :p.C].cpu(), h["x"])
    assert torch.equal(filt[:, :p.C].cpu(), h["x"])
    assert binding.ddpm_get_device_error() == 0


@pytest.mark.parametrize("name", ["b1_c64_128x128_k3", "b1_c64_256x256_k3", "b1_c64_128x128_k5"])
def test_full_size_tf32x3_forward(name):
    """The FP32 forward with the 3xTF32 generator GEMM, whole tensors, FP32 bar."""
    p = WORKLOADS[name]
    h = make_inputs(p, SEEDS[name], "float32", grad=False)
    d = _dev(h)
    out = binding.forward(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations, flags=TF32X3)
    torch.cuda.synchronize()
    with full_size_section():
        assert_forward_close(out, oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations),
                             "float32", f"{name} float32 out (3xTF32)")
    assert torch.equal(out[:, :p.C].cpu(), h["x"])
    assert binding.ddpm_get_device_error() == 0


@pytest.mark.parametrize("name,dtype", FULL_TRAINING, ids=lambda v: v)
def test_full_size_training(name, dtype):
    """Forward and backward (dx, dy, dW, dbias) over whole tensors, in the launch
    configuration the benchmark times (TF32 allowed in an FP32 backward)."""
    p = WORKLOADS[name]
    h = make_inputs(p, SEEDS[name], dtype)
    d = _dev(h)
    out = run_forward(d, p)
    grads = run_backward(d, p, flags=binding.DDPM_FLAG_TF32_BACKWARD)
    torch.cuda.synchronize()
    assert binding.ddpm_get_device_error() == 0
    bf = dtype == "bfloat16"
    with full_size_section():
        _check_forward(out, h, p, dtype, f"{name} {dtype} out")
        del out
        ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=bf)
        for gname, got, want in zip(("dx", "dy", "dW", "dbias"), grads, ref):
            if bf and gname == "dx":
                h64 = _f64_inputs(h)
                assert_bf16_close_with_ties(got, want, f"dx {name} {dtype}",
                                            lambda idx: dx_tie_allowance(oracle, h64, p.K, p.dilations, idx))
            else:
                assert_grad_close(got, want, dtype, f"{gname} {name} {dtype}")
