"""ctypes binding of libddpm_gb300.so -- argument marshalling only.

The functions named ``ddpm_*`` mirror the C ABI in ``include/ddpm.h`` one to
one and take either torch tensors (their ``data_ptr()`` is passed) or raw
integer device pointers.  The helpers ``forward``, ``filter_pregenerated`` and
``backward`` allocate outputs with torch (device memory is PyTorch's job here)
and call the library on torch's current stream.  Every step of the method
runs in the library's CUDA kernels; there is no CPU fallback: if the library
is missing or no GPU is present, these calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libddpm_gb300.so")

DDPM_FLOAT32 = 0
DDPM_BFLOAT16 = 1
DDPM_FLAG_TF32_BACKWARD = 0x1
DDPM_FLAG_CUDA_CORES = 0x2
DDPM_FLAG_TF32X3_FORWARD = 0x4

STATUS = {
    0: "DDPM_OK", 1: "DDPM_ERR_INVALID_ARGUMENT", 2: "DDPM_ERR_UNSUPPORTED", 3: "DDPM_ERR_MISALIGNED",
    4: "DDPM_ERR_WORKSPACE_TOO_SMALL", 5: "DDPM_ERR_CUDA", 6: "DDPM_ERR_DEVICE_TIMEOUT",
}
EXPORTED = ("ddpm_forward", "ddpm_filter_pregenerated", "ddpm_backward_workspace_size", "ddpm_backward",
            "ddpm_get_device_error", "ddpm_status_string", "ddpm_version", "ddpm_trace_enable",
            "ddpm_trace_read", "ddpm_kernel_name", "ddpm_backward_noalloc", "ddpm_measure_ffma_tflops",
            "ddpm_filter_pregenerated_backward", "ddpm_debug_wait_probe",
            "ddpm_backward_workspace_min_size")


class ddpm_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("C", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("K", ctypes.c_int), ("dilations", ctypes.c_int * 3), ("dtype", ctypes.c_int),
                ("flags", ctypes.c_uint)]


class DDPMError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libddpm_gb300.so not built ({path}); run dynamic_dilated_depthwise_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(ddpm_problem)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        lib.ddpm_forward.argtypes = [P, vp, vp, vp, vp, vp, vp]
        lib.ddpm_filter_pregenerated.argtypes = [P, vp, vp, vp, vp]
        lib.ddpm_filter_pregenerated_backward.argtypes = [P, vp, vp, vp, vp, vp, vp]
        lib.ddpm_backward_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
        lib.ddpm_backward_workspace_min_size.argtypes = [P, ctypes.POINTER(sz)]
        lib.ddpm_backward_workspace_min_size.restype = ctypes.c_int
        lib.ddpm_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.ddpm_get_device_error.argtypes = [vp]
        lib.ddpm_backward_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.ddpm_backward_noalloc.restype = ctypes.c_int
        lib.ddpm_status_string.argtypes = [ctypes.c_int]
        lib.ddpm_status_string.restype = ctypes.c_char_p
        lib.ddpm_version.argtypes = []
        lib.ddpm_trace_enable.argtypes = [ctypes.c_int]
        lib.ddpm_trace_enable.restype = ctypes.c_int
        lib.ddpm_trace_read.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float), ctypes.c_int]
        lib.ddpm_trace_read.restype = ctypes.c_int
        lib.ddpm_measure_ffma_tflops.argtypes = [ctypes.POINTER(ctypes.c_double)]
        lib.ddpm_measure_ffma_tflops.restype = ctypes.c_int
        lib.ddpm_debug_wait_probe.argtypes = [ctypes.c_uint, vp]
        lib.ddpm_debug_wait_probe.restype = ctypes.c_int
        lib.ddpm_kernel_name.argtypes = [ctypes.c_int]
        lib.ddpm_kernel_name.restype = ctypes.c_char_p
        for f in ("ddpm_forward", "ddpm_filter_pregenerated", "ddpm_backward_workspace_size", "ddpm_backward",
                  "ddpm_get_device_error", "ddpm_version"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().ddpm_status_string(int(status)).decode()


def _p(t):
    """A device pointer from a tensor, an int or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise DDPMError(status, what)


def make_problem(B, C, H, W, K, dilations=(1, 3, 5), dtype=DDPM_FLOAT32, flags=0) -> ddpm_problem:
    p = ddpm_problem()
    p.B, p.C, p.H, p.W, p.K = int(B), int(C), int(H), int(W), int(K)
    for i in range(3):
        p.dilations[i] = int(dilations[i])
    p.dtype = int(dtype)
    p.flags = int(flags)
    return p


# ------------------------------------------------------------ C ABI mirror --

def ddpm_forward(problem, x, y, weight, bias, out, stream=None) -> None:
    _check(load().ddpm_forward(ctypes.byref(problem), _p(x), _p(y), _p(weight), _p(bias), _p(out),
                               _stream(stream)), "ddpm_forward")


def ddpm_filter_pregenerated(problem, x, taps, out, stream=None) -> None:
    _check(load().ddpm_filter_pregenerated(ctypes.byref(problem), _p(x), _p(taps), _p(out), _stream(stream)),
           "ddpm_filter_pregenerated")


def ddpm_filter_pregenerated_backward(problem, grad_out, x, taps, dx, dtaps, stream=None) -> None:
    _check(load().ddpm_filter_pregenerated_backward(ctypes.byref(problem), _p(grad_out), _p(x), _p(taps), _p(dx),
                                                    _p(dtaps), _stream(stream)),
           "ddpm_filter_pregenerated_backward")


def ddpm_backward_workspace_size(problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load().ddpm_backward_workspace_size(ctypes.byref(problem), ctypes.byref(n)),
           "ddpm_backward_workspace_size")
    return int(n.value)


def ddpm_backward_workspace_min(problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load().ddpm_backward_workspace_min_size(ctypes.byref(problem), ctypes.byref(n)),
           "ddpm_backward_workspace_min_size")
    return int(n.value)


def ddpm_backward(problem, grad_out, x, y, weight, bias, dx, dy, dweight, dbias, workspace, workspace_bytes,
                  stream=None) -> None:
    _check(load().ddpm_backward(ctypes.byref(problem), _p(grad_out), _p(x), _p(y), _p(weight), _p(bias), _p(dx),
                                _p(dy), _p(dweight), _p(dbias), _p(workspace), int(workspace_bytes),
                                _stream(stream)), "ddpm_backward")


def ddpm_backward_noalloc(problem, grad_out, x, y, weight, bias, dx, dy, dweight, dbias, stream=None) -> None:
    """ddpm_backward with the library's own fixed scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/ddpm.h)."""
    _check(load().ddpm_backward_noalloc(ctypes.byref(problem), _p(grad_out), _p(x), _p(y), _p(weight), _p(bias),
                                        _p(dx), _p(dy), _p(dweight), _p(dbias), _stream(stream)),
           "ddpm_backward_noalloc")


def ddpm_get_device_error(stream=None) -> int:
    return int(load().ddpm_get_device_error(_stream(stream)))


def ddpm_debug_wait_probe(limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait failure probe (a wait that expires after limit_us)."""
    _check(load().ddpm_debug_wait_probe(int(limit_us), _stream(stream)), "ddpm_debug_wait_probe")


def ddpm_version() -> int:
    return int(load().ddpm_version())


def ddpm_trace_enable(enable: bool) -> None:
    _check(load().ddpm_trace_enable(1 if enable else 0), "ddpm_trace_enable")


def ddpm_trace_read(max_records: int = 65536):
    """[(kernel name, milliseconds), ...] of the traced launches, in launch order."""
    ids = (ctypes.c_int * max_records)()
    ms = (ctypes.c_float * max_records)()
    n = load().ddpm_trace_read(ids, ms, max_records)
    if n < 0:
        raise DDPMError(5, "ddpm_trace_read")
    return [(ddpm_kernel_name(ids[i]), float(ms[i])) for i in range(n)]


def ddpm_measure_ffma_tflops() -> float:
    """Measured FP32 FMA throughput of the current device, TFLOP/s (synchronises)."""
    v = ctypes.c_double(0.0)
    _check(load().ddpm_measure_ffma_tflops(ctypes.byref(v)), "ddpm_measure_ffma_tflops")
    return float(v.value)


def ddpm_kernel_name(kernel_id: int) -> str:
    return load().ddpm_kernel_name(int(kernel_id)).decode()


# ------------------------------------------------------------- tensor helpers --

_DT = {torch.float32: DDPM_FLOAT32, torch.bfloat16: DDPM_BFLOAT16}


def _problem_of(x, K, dilations, flags=0):
    if x.dtype not in _DT:
        raise TypeError(f"unsupported dtype {x.dtype}; use float32 or bfloat16")
    B, C, H, W = x.shape
    return make_problem(B, C, H, W, K, dilations, _DT[x.dtype], flags)


def _same(x, *ts):
    """Every tensor a contiguous CUDA tensor on x's device with x's dtype (the library
    takes raw device pointers: a host tensor must never reach it)."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    for t in ts:
        if t is None:
            continue
        if t.dtype != x.dtype:
            raise TypeError("all tensors must share one dtype")
        if t.device != x.device or not t.is_contiguous():
            raise ValueError("tensors must be contiguous and on the same CUDA device")


def forward(x, y, weight, bias, K, dilations=(1, 3, 5), out=None, stream=None, flags=0):
    """[x, d1, d3, d5] = DDPM core forward; returns out [B, 4C, H, W]."""
    _same(x, y, weight, bias)
    B, C, H, W = x.shape
    if out is None:
        out = torch.empty((B, 4 * C, H, W), dtype=x.dtype, device=x.device)
    ddpm_forward(_problem_of(x, K, dilations, flags), x, y, weight, bias, out, stream)
    return out


def filter_pregenerated(x, taps, K, dilations=(1, 3, 5), out=None, stream=None):
    """The dynamic filter with given taps [B, 3*C*K*K, H, W]."""
    _same(x, taps)
    B, C, H, W = x.shape
    if out is None:
        out = torch.empty((B, 4 * C, H, W), dtype=x.dtype, device=x.device)
    ddpm_filter_pregenerated(_problem_of(x, K, dilations), x, taps, out, stream)
    return out


def filter_pregenerated_backward(grad_out, x, taps, K, dilations=(1, 3, 5), with_dtaps=True, stream=None):
    """Gradients (dx, dtaps) of <grad_out, filter_pregenerated(x, taps)>; dtaps is
    None when with_dtaps is False (dx alone)."""
    _same(x, grad_out, taps)
    dx = torch.empty_like(x)
    dtaps = torch.empty_like(taps) if with_dtaps else None
    ddpm_filter_pregenerated_backward(_problem_of(x, K, dilations), grad_out, x, taps, dx, dtaps, stream)
    return dx, dtaps


def backward_workspace_size(x, K, dilations=(1, 3, 5), flags=0) -> int:
    return ddpm_backward_workspace_size(_problem_of(x, K, dilations, flags))


def backward(grad_out, x, y, weight, bias, K, dilations=(1, 3, 5), workspace=None, flags=0, outs=None,
             stream=None, with_dbias=True):
    """Gradients (dx, dy, dweight, dbias) of <grad_out, forward(...)>."""
    _same(x, grad_out, y, weight, bias)
    prob = _problem_of(x, K, dilations, flags)
    nbytes = ddpm_backward_workspace_size(prob)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    if outs is None:
        dx = torch.empty_like(x)
        dy = torch.empty_like(y)
        dw = torch.empty_like(weight)
        db = torch.empty((weight.shape[0],), dtype=x.dtype, device=x.device) if with_dbias else None
    else:
        dx, dy, dw, db = outs
    ddpm_backward(prob, grad_out, x, y, weight, bias, dx, dy, dw, db, workspace, workspace.numel(), stream)
    return dx, dy, dw, db


class DDPMCoreFunction(torch.autograd.Function):
    """autograd wrapper: forward and backward both run in the CUDA library."""

    @staticmethod
    def forward(ctx, x, y, weight, bias, K, dilations):
        ctx.save_for_backward(x, y, weight, bias)
        ctx.K, ctx.dilations = K, tuple(dilations)
        return forward(x, y, weight, bias, K, dilations)

    @staticmethod
    def backward(ctx, grad_out):
        x, y, weight, bias = ctx.saved_tensors
        dx, dy, dw, db = backward(grad_out.contiguous(), x, y, weight, bias, ctx.K, ctx.dilations,
                                  with_dbias=bias is not None)
        return dx, dy, dw, db, None, None


class DDPMFilterFunction(torch.autograd.Function):
    """autograd wrapper of the filter with given taps: forward and backward (dx, dtaps)
    both run in the CUDA library; dtaps is computed only when taps needs a gradient."""

    @staticmethod
    def forward(ctx, x, taps, K, dilations):
        ctx.save_for_backward(x, taps)
        ctx.K, ctx.dilations = K, tuple(dilations)
        return filter_pregenerated(x, taps, K, dilations)

    @staticmethod
    def backward(ctx, grad_out):
        x, taps = ctx.saved_tensors
        dx, dtaps = filter_pregenerated_backward(grad_out.contiguous(), x, taps, ctx.K, ctx.dilations,
                                                 with_dtaps=ctx.needs_input_grad[1])
        return dx, dtaps, None, None
