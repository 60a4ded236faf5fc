"""ddpm_backward_noalloc against ddpm_backward, through the C ABI (GPU).

ddpm_backward_noalloc serves callers that cannot allocate device memory when
they run the backward (a plugin inside an application that owns all device
allocations, a loop that forbids allocation after start-up, a C caller with
no allocator for temporaries): it keeps the dW/dbias partial sums in a fixed
array inside the library instead of a caller-supplied workspace.

Its results must match the workspace entry point's within the parity
tolerances, on two calls in a row (the shared array keeps the previous call's
contents) and across two problem sizes.  This file is collected last so that
a run stopping at the first failure has already run every other test; it
builds and loads the library itself, so it also passes alone.
"""
import ctypes

import pytest
import torch

from dynamic_dilated_depthwise_gb300 import binding, build
from dynamic_dilated_depthwise_gb300.inputs import SEEDS, WORKLOADS, Problem, make_inputs
from parity import assert_grad_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    assert torch.cuda.is_available(), "needs a CUDA device"
    return binding.load()


# FP32 regression shape; a small BF16 image whose packed copies also fit in the array
# (dX takes the packed kernel); the 256x256 BF16 workload (dX stages its operands)
CASES = [(Problem(2, 24, 15, 17, 3), "float32", 41),
         (Problem(1, 64, 32, 32, 3), "bfloat16", 42),
         (WORKLOADS["b1_c64_256x256_k3"], "bfloat16", SEEDS["b1_c64_256x256_k3"])]


def test_noalloc_backward_matches_workspace_backward(lib):
    for p, dtype, seed in CASES:
        h = make_inputs(p, seed, dtype)
        d = {k: v.cuda() for k, v in h.items()}
        flags = binding.DDPM_FLAG_TF32_BACKWARD
        ref = binding.backward(d["grad_out"], d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations, flags=flags)
        prob = binding.make_problem(p.B, p.C, p.H, p.W, p.K, p.dilations,
                                    binding.DDPM_BFLOAT16 if dtype == "bfloat16" else binding.DDPM_FLOAT32, flags)
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):
            outs = [torch.full_like(r, float("nan")) for r in ref]
            status = lib.ddpm_backward_noalloc(ctypes.byref(prob), d["grad_out"].data_ptr(), d["x"].data_ptr(),
                                               d["y"].data_ptr(), d["weight"].data_ptr(), d["bias"].data_ptr(),
                                               outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                                               outs[3].data_ptr(), stream)
            assert status == 0, binding.status_string(status)
            torch.cuda.synchronize()
            for name, got, want in zip(("dx", "dy", "dW", "dbias"), outs, ref):
                assert torch.isfinite(got).all(), f"call {call}: {name} not fully written"
                assert_grad_close(got, want, dtype, f"{name} (call {call})")


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    p = WORKLOADS["b1_c64_128x128_k5"]          # partials need 16 x 4800 x 65 x 4 B = 20 MB > 8 MiB
    prob = binding.make_problem(p.B, p.C, p.H, p.W, p.K, p.dilations, binding.DDPM_BFLOAT16)
    assert binding.ddpm_backward_workspace_size(prob) > 8 << 20
    # real device buffers of the problem's shapes: were the size check ever to let the
    # problem through, the backward would run on valid memory and the status would say so
    h = make_inputs(p, 5, "bfloat16")
    d = {k: v.cuda() for k, v in h.items()}
    outs = [torch.empty_like(d["x"]), torch.empty_like(d["x"]), torch.empty_like(d["weight"]),
            torch.empty_like(d["bias"])]
    status = lib.ddpm_backward_noalloc(ctypes.byref(prob), d["grad_out"].data_ptr(), d["x"].data_ptr(),
                                       d["y"].data_ptr(), d["weight"].data_ptr(), d["bias"].data_ptr(),
                                       outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                                       outs[3].data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert status == 2  # DDPM_ERR_UNSUPPORTED, rejected on the host before any launch
