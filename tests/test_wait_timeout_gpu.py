"""The bounded-wait failure path on the GPU, without faulting it.

Every tensor-core kernel of the library waits on shared-memory barriers with
a time limit.  ddpm_debug_wait_probe runs a block with the kernels' warp roles
whose wait can never be satisfied, with a limit of a few milliseconds: the
wait must expire on its own, the host must then read DDPM_ERR_DEVICE_TIMEOUT
from ddpm_get_device_error (which clears it), and the same CUDA context must
keep working -- a forward and a backward right after it match the oracle.
No trap, no unbounded wait, no bad address is involved.
"""
import time

import pytest
import torch

import oracle
from dynamic_dilated_depthwise_gb300 import binding, build
from dynamic_dilated_depthwise_gb300.inputs import Problem, make_inputs
from parity import assert_forward_close, assert_grad_close

pytestmark = pytest.mark.gpu

DDPM_ERR_DEVICE_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    binding.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_bounded_wait_expires_and_the_context_stays_usable():
    p = Problem(1, 64, 16, 64, 3)                # takes the tensor-core forward and backward
    h = make_inputs(p, 77, "bfloat16")
    d = {k: v.cuda() for k, v in h.items()}
    torch.cuda.synchronize()
    assert binding.ddpm_get_device_error() == 0
    for limit_us in (2000, 5000):
        t0 = time.perf_counter()
        binding.ddpm_debug_wait_probe(limit_us)
        status = binding.ddpm_get_device_error()
        elapsed = time.perf_counter() - t0
        assert status == DDPM_ERR_DEVICE_TIMEOUT, binding.status_string(status)
        # the probe ended by its own short limit, far below the kernels' 2 s
        assert elapsed < 0.5, f"probe took {elapsed:.3f} s"
        assert binding.ddpm_get_device_error() == 0, "reading the error must clear it"
    out = binding.forward(d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations)
    grads = binding.backward(d["grad_out"], d["x"], d["y"], d["weight"], d["bias"], p.K, p.dilations)
    torch.cuda.synchronize()
    assert binding.ddpm_get_device_error() == 0
    assert_forward_close(out, oracle.forward(h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=True),
                         "bfloat16", "out after the probe")
    ref = oracle.backward(h["grad_out"], h["x"], h["y"], h["weight"], h["bias"], p.K, p.dilations, bf16=True)
    for name, got, want in zip(("dx", "dy", "dW", "dbias"), grads, ref):
        assert_grad_close(got, want, "bfloat16", f"{name} after the probe")
