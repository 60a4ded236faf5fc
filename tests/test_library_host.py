"""Host-side tests of the C ABI (no GPU needed, no compute call made).

* The library builds for sm_103a and loads.
* It exports every function that include/ddpm.h declares.
* Invalid arguments are rejected on the host, before anything touches CUDA.
* The workspace size is the documented <= 16 FP32 partials of [O, C+1].
"""
import ctypes
import os
import re

import pytest
import torch

from dynamic_dilated_depthwise_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        names += re.findall(r"DDPM_API\s+[\w\s\*]+?\b(ddpm_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("ddpm_forward", "ddpm_filter_pregenerated", "ddpm_backward", "ddpm_backward_workspace_size"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    for name in binding.EXPORTED:
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    for code, name in binding.STATUS.items():
        assert binding.status_string(code).startswith(name)
    assert "unknown" in binding.status_string(99)
    assert binding.ddpm_version() >= 100


def _prob(**kw):
    base = dict(B=1, C=4, H=5, W=6, K=3, dilations=(1, 3, 5), dtype=binding.DDPM_FLOAT32, flags=0)
    base.update(kw)
    return binding.make_problem(**base)


BAD = [
    dict(B=0), dict(C=0), dict(H=0), dict(W=-1), dict(K=2), dict(K=0), dict(K=4),
    dict(dilations=(1, 0, 5)), dict(dilations=(-1, 3, 5)), dict(dtype=7), dict(flags=0x80),
]


@pytest.mark.parametrize("kw", BAD, ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_invalid_problems_rejected_on_host(lib, kw):
    p = _prob(**kw)
    n = ctypes.c_size_t(0)
    assert lib.ddpm_backward_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 1
    assert lib.ddpm_forward(ctypes.byref(p), 16, 16, 16, 16, 16, None) == 1
    assert lib.ddpm_filter_pregenerated(ctypes.byref(p), 16, 16, 16, None) == 1
    assert lib.ddpm_filter_pregenerated_backward(ctypes.byref(p), 16, 16, 16, 16, 16, None) == 1


def test_unsupported_sizes(lib):
    n = ctypes.c_size_t(0)
    for kw in (dict(K=9), dict(B=70000), dict(dilations=(1, 3, 1 << 22))):
        p = _prob(**kw)
        assert lib.ddpm_backward_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 2


def test_null_and_misaligned_pointers(lib):
    p = _prob()
    assert lib.ddpm_forward(ctypes.byref(p), None, 16, 16, 16, 16, None) == 1          # x NULL
    assert lib.ddpm_forward(ctypes.byref(p), 16, 16, 16, 16, None, None) == 1          # out NULL
    assert lib.ddpm_forward(ctypes.byref(p), 18, 16, 16, 16, 16, None) == 3            # fp32 x at 2 bytes
    pb = _prob(dtype=binding.DDPM_BFLOAT16)
    assert lib.ddpm_forward(ctypes.byref(pb), 16, 16, 16, 17, 16, None) == 3           # bias odd address
    assert lib.ddpm_filter_pregenerated(ctypes.byref(p), 16, None, 16, None) == 1
    assert lib.ddpm_forward(None, 16, 16, 16, 16, 16, None) == 1
    # filter backward: a NULL grad, x, taps or dx is rejected; dtaps may be NULL
    assert lib.ddpm_filter_pregenerated_backward(ctypes.byref(p), 16, 16, 16, None, 16, None) == 1
    assert lib.ddpm_filter_pregenerated_backward(ctypes.byref(p), None, 16, 16, 16, None, None) == 1
    assert lib.ddpm_filter_pregenerated_backward(ctypes.byref(p), 16, 16, 18, 16, 16, None) == 3   # taps at 2 bytes
    assert lib.ddpm_filter_pregenerated_backward(ctypes.byref(p), 16, 16, 16, 16, 22, None) == 3   # dtaps at 2 bytes
    # backward: NULL grad, misaligned workspace, too-small workspace
    assert lib.ddpm_backward(ctypes.byref(p), None, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.ddpm_backward(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, 16, 24, 1 << 30, None) == 3
    assert lib.ddpm_backward(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 8, None) == 4
    n = ctypes.c_size_t(0)
    assert lib.ddpm_backward_workspace_size(ctypes.byref(p), None) == 1
    assert lib.ddpm_backward_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0


@pytest.mark.parametrize("B,C,H,W,K", [(1, 64, 256, 256, 3), (8, 64, 256, 256, 3), (2, 24, 15, 17, 3),
                                       (1, 64, 128, 128, 5), (1, 1, 1, 1, 1)])
def test_workspace_is_at_most_16_partials(lib, B, C, H, W, K):
    p = _prob(B=B, C=C, H=H, W=W, K=K)
    n = binding.ddpm_backward_workspace_size(p)
    O = 3 * C * K * K
    assert 0 < n <= 16 * O * (C + 1) * 4
    assert n % (O * (C + 1) * 4) == 0
    if B * H * W >= 16 * 2048:
        assert n == 16 * O * (C + 1) * 4
    assert n < 64 << 20  # "a few MiB", independent of the image size


def _partials_bytes(B, C, H, W, K):
    S = min(16, max(1, -(-B * H * W // 2048)))
    return S * 3 * C * K * K * (C + 1) * 4


@pytest.mark.parametrize("B,C,H,W,K,dil,packed", [
    (1, 64, 256, 256, 3, (1, 3, 5), True),    # partials + channel-chunked copies of y and grad for dX
    (2, 24, 16, 32, 3, (1, 3, 5), True),
    (2, 24, 15, 17, 3, (1, 3, 5), False),     # W not a multiple of 8: no tensor-core backward
    (1, 64, 64, 64, 3, (2, 4, 6), False),     # halo radius 6 with wide windows: dX tiles do not fit
    (1, 64, 128, 128, 5, (1, 3, 5), True),    # K = 5: the same copies, for the dX that gathers grad from L2
    (1, 64, 128, 128, 5, (1, 3, 6), False),   # K = 5, halo radius 12: CUDA-core backward
])
def test_bf16_workspace_adds_packed_copies(lib, B, C, H, W, K, dil, packed):
    p = _prob(B=B, C=C, H=H, W=W, K=K, dilations=dil, dtype=binding.DDPM_BFLOAT16)
    n = binding.ddpm_backward_workspace_size(p)
    parts = _partials_bytes(B, C, H, W, K)
    if packed:
        assert n == ((parts + 255) // 256) * 256 + 4 * B * C * H * W * 2
    else:
        assert n == parts
    # the smallest workspace the backward accepts is the partials alone, in every dtype
    assert binding.ddpm_backward_workspace_min(p) == parts
    assert binding.ddpm_backward_workspace_min(p) <= 16 * 3 * C * K * K * (C + 1) * 4


def test_binding_rejects_host_and_mixed_tensors():
    """The binding checks its tensors before any library call: host tensors and mixed
    dtypes raise in Python and never reach the kernels (no GPU needed)."""
    x = torch.zeros(1, 2, 4, 8)
    taps = torch.zeros(1, 3 * 2 * 9, 4, 8)
    g = torch.zeros(1, 8, 4, 8)
    with pytest.raises(ValueError):
        binding.filter_pregenerated(x, taps, 3)
    with pytest.raises(ValueError):
        binding.filter_pregenerated_backward(g, x, taps, 3)
    w, b = torch.zeros(54, 2), torch.zeros(54)
    with pytest.raises(ValueError):
        binding.forward(x, x, w, b, 3)
    with pytest.raises(ValueError):
        binding.backward(g, x, x, w, b, 3)


def test_wait_probe_rejects_limits_out_of_range(lib):
    """The failure probe's limit is checked on the host: nothing is enqueued."""
    assert lib.ddpm_debug_wait_probe(0, None) == 1
    assert lib.ddpm_debug_wait_probe(1000001, None) == 1


@pytest.mark.parametrize("C,tf32_dy", [(64, True), (32, True), (16, True), (24, False), (8, False), (10, False)])
def test_fp32_tf32_workspace_adds_rearranged_weight(lib, C, tf32_dy):
    """FP32 problems with DDPM_FLAG_TF32_BACKWARD: where the TF32 dY kernel applies
    (C a multiple of 16), the workspace also holds the rearranged weight (27*C*C FP32);
    where the TF32 dX applies (C a multiple of 4), it then holds, 256-byte aligned,
    channel-chunked FP32 copies of y and of grad's three dilation blocks (4*B*C*H*W values)."""
    p = _prob(B=1, C=C, H=64, W=64, K=3, flags=binding.DDPM_FLAG_TF32_BACKWARD)
    n = binding.ddpm_backward_workspace_size(p)
    parts = _partials_bytes(1, C, 64, 64, 3)
    up = lambda v: (v + 255) // 256 * 256
    wt = 27 * C * C * 4 if tf32_dy else 0
    if C % 4 == 0:
        assert n == up(up(parts) + wt) + 4 * C * 64 * 64 * 4
    elif tf32_dy:
        assert n == up(parts) + wt
    else:
        assert n == parts
    assert binding.ddpm_backward_workspace_min(p) == parts
