"""libselscan: Mamba's selective scan on one NVIDIA B300 (sm_103a).

A thin binding over the C ABI declared in ``include/selscan.h``; it only
checks and marshals arguments. Every step of the scan runs in the library's
CUDA kernels; PyTorch provides device memory and streams. There is no CPU
path: if ``libselscan.so`` is missing the first call raises.

    y = selscan_fwd(x, delta, A, B, C, delta_softplus=True)
    y, hT = selscan_fwd(x, delta, A, B, C, h0=h0, return_final_state=True)
    y = selscan_step(state, x, delta, A, B, C)     # state updated in place
    y, hT = selective_scan(x, delta, A, B, C, True)  # differentiable (fp32)

Tensors may live on the current CUDA device (the call is asynchronous on the
current stream) or in host memory (preferably pinned): host inputs are copied
to the device, the kernels run, and the outputs are copied back before the
call returns.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["selscan_fwd", "selscan_bwd", "selective_scan", "selscan_fwd_noalloc", "selscan_step", "conv1d", "conv1d_step",
           "ssd_fwd", "fwd_plan", "last_error", "check_device_error",
           "release_workspace", "version", "library_path", "SelscanError", "host_empty",
           "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_NO_MEMORY", "ERR_TIMEOUT",
           "MAX_N", "FLAG_SOFTPLUS", "FLAG_ZOH"]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_NO_MEMORY, ERR_TIMEOUT = 0, 1, 2, 3, 4, 5
FLAG_SOFTPLUS, FLAG_ZOH = 1, 2
F32, BF16 = 0, 1
MAX_N = 64
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libselscan.so")
_lib = None


class SelscanError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libselscan error {code}: {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with `python -m selective_state_space_157_b300.build`"
                " (there is no fallback path)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I64, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.selscan_fwd.restype = INT
        L.selscan_fwd.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_step.restype = INT
        L.selscan_step.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, P]
        L.selscan_last_error.restype = ctypes.c_char_p
        L.selscan_last_error.argtypes = []
        L.selscan_check_device_error.restype = INT
        L.selscan_check_device_error.argtypes = [P]
        L.selscan_release_workspace.restype = None
        L.selscan_release_workspace.argtypes = []
        L.selscan_version.restype = ctypes.c_char_p
        L.selscan_version.argtypes = []
        L.selscan_fwd_noalloc.restype = INT
        L.selscan_fwd_noalloc.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_fwd_gated.restype = INT
        L.selscan_fwd_gated.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_step_gated.restype = INT
        L.selscan_step_gated.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I64, P]
        L.selscan_fwd_ex.restype = INT
        L.selscan_fwd_ex.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_step_ex.restype = INT
        L.selscan_step_ex.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I64, INT, P]
        L.selscan_conv1d.restype = INT
        L.selscan_conv1d.argtypes = [P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_conv1d_step.restype = INT
        L.selscan_conv1d_step.argtypes = [P, P, P, P, P, I64, I64, I64, INT, P]
        L.selscan_fwd_host.restype = INT
        L.selscan_fwd_host.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_fwd_host_ex.restype = INT
        L.selscan_fwd_host_ex.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, P, P, P]
        L.selscan_fwd_plan.restype = INT
        L.selscan_fwd_plan.argtypes = [I64, I64, I64, I64, INT, P, P, P, P]
        L.selscan_ssd_fwd.restype = INT
        L.selscan_ssd_fwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, INT, INT, P]
        L.selscan_test_fault_injection.restype = INT
        L.selscan_test_fault_injection.argtypes = [INT, INT]
        L.selscan_bwd.restype = INT
        L.selscan_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT, P]
        L.selscan_host_alloc.restype = P
        L.selscan_host_alloc.argtypes = [ctypes.c_size_t]
        L.selscan_host_free.restype = INT
        L.selscan_host_free.argtypes = [P]
        L.selscan_bwd_gated.restype = INT
        L.selscan_bwd_gated.argtypes = [P] * 18 + [I64, I64, I64, I64, INT, P]
        _lib = L
    return _lib


def last_error() -> str:
    return lib().selscan_last_error().decode()


def version() -> str:
    return lib().selscan_version().decode()


def fwd_plan(Bsz: int, L: int, D: int, N: int, bf16: bool = False) -> dict:
    """How selscan_fwd would split this problem on the current device:
    {"chunks", "chunk_len", "launches", "workspace_bytes"} (16-byte aligned tensors)."""
    k = ctypes.c_int(0)
    t = ctypes.c_int64(0)
    n = ctypes.c_int(0)
    w = ctypes.c_int64(0)
    _check(lib().selscan_fwd_plan(Bsz, L, D, N, BF16 if bf16 else F32, ctypes.byref(k),
                                  ctypes.byref(t), ctypes.byref(n), ctypes.byref(w)))
    return {"chunks": k.value, "chunk_len": t.value, "launches": n.value, "workspace_bytes": w.value}


def host_empty(shape, dtype=None):
    """An uninitialised host tensor in page-locked memory from
    ``selscan_host_alloc`` (see ``include/selscan.h``): the DMA engines read
    and write it at the link's full rate. The memory is given back with
    ``selscan_host_free`` when the tensor is no longer referenced."""
    import math
    import weakref
    import torch
    dtype = torch.float32 if dtype is None else dtype
    shape = tuple(int(v) for v in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    nbytes = max(1, math.prod(shape) * torch.empty((), dtype=dtype).element_size())
    ptr = lib().selscan_host_alloc(nbytes)
    if not ptr:
        raise SelscanError(ERR_NO_MEMORY, last_error())
    buf = (ctypes.c_uint8 * nbytes).from_address(ptr)
    weakref.finalize(buf, lib().selscan_host_free, ptr)
    n = math.prod(shape)
    return torch.frombuffer(buf, dtype=torch.uint8)[:n * torch.empty((), dtype=dtype).element_size()] \
        .view(dtype).view(shape)


def release_workspace() -> None:
    lib().selscan_release_workspace()


def _check(rc: int) -> None:
    if rc != OK:
        raise SelscanError(rc, last_error())


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def check_device_error(stream=None) -> None:
    """Wait for the stream and raise if work on it failed."""
    _check(lib().selscan_check_device_error(_stream_ptr(stream)))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"x, delta, B, C must be float32 or bfloat16, got {t.dtype}")


def _need(t, name, shape, dtype, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def selscan_fwd(x, delta, A, B, C, delta_softplus: bool = False, h0=None,
                return_final_state: bool = False, y=None, hT=None, stream=None,
                D_skip=None, z=None, zoh: bool = False, check: bool = False):
    """Forward selective scan (see ``include/selscan.h``).

    x, delta: (Bsz, L, D) float32 or bfloat16; A: (D, N) float32;
    B, C: (Bsz, L, N) same dtype as x; h0: (Bsz, D, N) float32 or None.
    Returns y (Bsz, L, D), or (y, hT) with hT (Bsz, D, N) float32 when
    ``return_final_state``. ``y`` / ``hT`` may be passed preallocated.
    ``D_skip`` (D,) float32 and ``z`` (like x) add the block's skip and gate
    (selscan_fwd_gated): y = (scan + D_skip * x) * silu(z). ``zoh`` selects
    the zero-order-hold discretisation (selscan_fwd_ex). Host (CPU) tensors
    take the host-buffer entry points (selscan_fwd_host, selscan_fwd_host_ex).
    ``check`` waits for the call and raises if a wait inside the
    kernel ran out (``check_device_error``): the outputs are invalid then.
    """
    import torch
    gated = D_skip is not None or z is not None
    if x.device.type == "cpu":
        return _fwd_host(x, delta, A, B, C, delta_softplus, h0, return_final_state, y, hT, D_skip, z, zoh)
    dev = x.device
    Bsz, L, D = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    code = _dtype_code(x)
    _need(delta, "delta", (Bsz, L, D), x.dtype, dev)
    _need(A, "A", (D, N), torch.float32, dev)
    _need(B, "B", (Bsz, L, N), x.dtype, dev)
    _need(C, "C", (Bsz, L, N), x.dtype, dev)
    _need(x, "x", (Bsz, L, D), x.dtype, dev)
    if h0 is not None:
        _need(h0, "h0", (Bsz, D, N), torch.float32, dev)
    if y is None:
        y = torch.empty((Bsz, L, D), dtype=x.dtype, device=dev)
    else:
        _need(y, "y", (Bsz, L, D), x.dtype, dev)
    if return_final_state and hT is None:
        hT = torch.empty((Bsz, D, N), dtype=torch.float32, device=dev)
    if hT is not None:
        _need(hT, "hT", (Bsz, D, N), torch.float32, dev)
    if D_skip is not None:
        _need(D_skip, "D_skip", (D,), torch.float32, dev)
    if z is not None:
        _need(z, "z", (Bsz, L, D), x.dtype, dev)
    with torch.cuda.device(dev):
        if gated or zoh:
            flags = (FLAG_SOFTPLUS if delta_softplus else 0) | (FLAG_ZOH if zoh else 0)
            rc = lib().selscan_fwd_ex(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D_skip),
                                      _ptr(z), _ptr(y), Bsz, L, D, N, code, flags,
                                      _ptr(h0), _ptr(hT), _stream_ptr(stream))
        else:
            rc = lib().selscan_fwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(y),
                                   Bsz, L, D, N, code, int(bool(delta_softplus)), _ptr(h0), _ptr(hT),
                                   _stream_ptr(stream))
    _check(rc)
    if check:
        check_device_error(stream)
    return (y, hT) if (return_final_state or hT is not None) else y


def selscan_bwd(x, delta, A, B, C, dy, delta_softplus: bool = False, h0=None, dhT=None,
                want_dh0: bool = True, stream=None, check: bool = False, D_skip=None, z=None):
    """Backward pass of the forward scan (fp32; see ``include/selscan.h``):
    gradients of a loss with respect to x, delta, A, B, C and h0, given dy
    (Bsz, L, D) = dLoss/dy and dhT (Bsz, D, N) = dLoss/dhT or None. Device
    float32 tensors only. Returns a dict with dx, ddelta (Bsz, L, D), dA
    (D, N), dB, dC (Bsz, L, N) and, when ``want_dh0``, dh0 (Bsz, D, N).
    With ``D_skip`` (D,) and/or ``z`` (like x), dy is the gradient of the
    block's output (scan + D_skip x) silu(z) (``selscan_bwd_gated``), and the
    dict adds dD_skip and/or dz.
    """
    import torch
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("selscan_bwd takes device tensors")
    Bsz, L, D = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    f = torch.float32
    for t, name, shape in ((x, "x", (Bsz, L, D)), (delta, "delta", (Bsz, L, D)), (A, "A", (D, N)),
                           (B, "B", (Bsz, L, N)), (C, "C", (Bsz, L, N)), (dy, "dy", (Bsz, L, D))):
        _need(t, name, shape, f, dev)
    if h0 is not None:
        _need(h0, "h0", (Bsz, D, N), f, dev)
    if dhT is not None:
        _need(dhT, "dhT", (Bsz, D, N), f, dev)
    if D_skip is not None:
        _need(D_skip, "D_skip", (D,), f, dev)
    if z is not None:
        _need(z, "z", (Bsz, L, D), f, dev)
    g = dict(dx=torch.empty((Bsz, L, D), dtype=f, device=dev), ddelta=torch.empty((Bsz, L, D), dtype=f, device=dev),
             dA=torch.empty((D, N), dtype=f, device=dev), dB=torch.empty((Bsz, L, N), dtype=f, device=dev),
             dC=torch.empty((Bsz, L, N), dtype=f, device=dev))
    if want_dh0:
        g["dh0"] = torch.empty((Bsz, D, N), dtype=f, device=dev)
    if D_skip is not None:
        g["dD_skip"] = torch.empty((D,), dtype=f, device=dev)
    if z is not None:
        g["dz"] = torch.empty((Bsz, L, D), dtype=f, device=dev)
    with torch.cuda.device(dev):
        if D_skip is None and z is None:
            rc = lib().selscan_bwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(h0), _ptr(dy), _ptr(dhT),
                                   _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
                                   _ptr(g.get("dh0")), Bsz, L, D, N, int(bool(delta_softplus)), _stream_ptr(stream))
        else:
            rc = lib().selscan_bwd_gated(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D_skip), _ptr(z),
                                         _ptr(h0), _ptr(dy), _ptr(dhT), _ptr(g["dx"]), _ptr(g["ddelta"]),
                                         _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g.get("dD_skip")),
                                         _ptr(g.get("dz")), _ptr(g.get("dh0")), Bsz, L, D, N,
                                         int(bool(delta_softplus)), _stream_ptr(stream))
    _check(rc)
    if check:
        check_device_error(stream)
    return g


_autograd_fn = None


def _selective_scan_fn():
    """The autograd Function behind ``selective_scan`` (built on first use, so
    importing the binding does not import torch)."""
    global _autograd_fn
    if _autograd_fn is None:
        import torch

        class SelectiveScan(torch.autograd.Function):
            @staticmethod
            def forward(ctx, x, delta, A, B, C, h0, delta_softplus, check, D_skip, z):
                y, hT = selscan_fwd(x, delta, A, B, C, delta_softplus, h0=h0, return_final_state=True,
                                    check=check, D_skip=D_skip, z=z)
                ctx.save_for_backward(x, delta, A, B, C, h0, D_skip, z)
                ctx.delta_softplus = delta_softplus
                ctx.check = check
                return y, hT

            @staticmethod
            def backward(ctx, dy, dhT):
                x, delta, A, B, C, h0, D_skip, z = ctx.saved_tensors
                want_dh0 = h0 is not None and ctx.needs_input_grad[5]
                g = selscan_bwd(x, delta, A, B, C, dy.contiguous(), ctx.delta_softplus, h0=h0,
                                dhT=None if dhT is None else dhT.contiguous(), want_dh0=want_dh0,
                                check=ctx.check, D_skip=D_skip, z=z)
                return (g["dx"], g["ddelta"], g["dA"], g["dB"], g["dC"], g.get("dh0"), None, None,
                        g.get("dD_skip"), g.get("dz"))

        _autograd_fn = SelectiveScan
    return _autograd_fn


def selective_scan(x, delta, A, B, C, delta_softplus: bool = False, h0=None, check: bool = False,
                   D_skip=None, z=None):
    """The forward scan as a differentiable torch operation: returns (y, hT),
    and ``backward`` runs ``selscan_bwd`` (the states are recomputed, not
    stored). Device float32 tensors; h0 (Bsz, D, N) or None; ``D_skip`` (D,)
    and ``z`` (like x) make y the block's output (scan + D_skip x) silu(z),
    differentiable in both. ``check`` makes the forward and the backward wait
    for their kernels and raise if a wait inside one ran out."""
    return _selective_scan_fn().apply(x, delta, A, B, C, h0, bool(delta_softplus), bool(check), D_skip, z)


def selscan_fwd_noalloc(x, delta, A, B, C, y, delta_softplus: bool = False, h0=None, hT=None,
                        stream=None, check: bool = False):
    """selscan_fwd without any allocation, for callers that cannot allocate
    device memory (another allocator owns it, or allocation latency is not
    allowed); see ``include/selscan.h``. Device tensors only, with the outputs
    ``y`` (and ``hT`` if wanted) supplied by the caller. Calls that may overlap
    on the GPU share one scratch array and must be ordered."""
    import torch
    dev = x.device
    Bsz, L, D = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    code = _dtype_code(x)
    for t, name, shape, dt in ((x, "x", (Bsz, L, D), x.dtype), (delta, "delta", (Bsz, L, D), x.dtype),
                               (A, "A", (D, N), torch.float32), (B, "B", (Bsz, L, N), x.dtype),
                               (C, "C", (Bsz, L, N), x.dtype), (y, "y", (Bsz, L, D), x.dtype)):
        _need(t, name, shape, dt, dev)
    for t, name in ((h0, "h0"), (hT, "hT")):
        if t is not None:
            _need(t, name, (Bsz, D, N), torch.float32, dev)
    with torch.cuda.device(dev):
        rc = lib().selscan_fwd_noalloc(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(y),
                                       Bsz, L, D, N, code, int(bool(delta_softplus)), _ptr(h0), _ptr(hT),
                                       _stream_ptr(stream))
    _check(rc)
    if check:
        check_device_error(stream)
    return y


def selscan_step(state, x, delta, A, B, C, y=None, stream=None, D_skip=None, z=None,
                 zoh: bool = False):
    """One decode step (see ``include/selscan.h``): ``state`` (Bsz, D, N)
    float32 is updated in place; returns y (Bsz, D) float32. delta is used
    as given (no softplus). ``D_skip`` (D,) and ``z`` (Bsz, D) add the
    block's skip and gate; ``zoh`` selects the zero-order-hold discretisation
    (selscan_step_ex; device tensors only)."""
    import torch
    gated = D_skip is not None or z is not None
    if state.device.type == "cpu":
        if gated or zoh:
            raise ValueError("D_skip / z / zoh are supported for device tensors only")
        return _step_host(state, x, delta, A, B, C, y)
    dev = state.device
    Bsz, D, N = state.shape
    f = torch.float32
    _need(state, "state", (Bsz, D, N), f, dev)
    _need(x, "x", (Bsz, D), f, dev)
    _need(delta, "delta", (Bsz, D), f, dev)
    _need(A, "A", (D, N), f, dev)
    _need(B, "B", (Bsz, N), f, dev)
    _need(C, "C", (Bsz, N), f, dev)
    if y is None:
        y = torch.empty((Bsz, D), dtype=f, device=dev)
    else:
        _need(y, "y", (Bsz, D), f, dev)
    if D_skip is not None:
        _need(D_skip, "D_skip", (D,), f, dev)
    if z is not None:
        _need(z, "z", (Bsz, D), f, dev)
    with torch.cuda.device(dev):
        if gated or zoh:
            rc = lib().selscan_step_ex(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                       _ptr(D_skip), _ptr(z), _ptr(y), Bsz, D, N, FLAG_ZOH if zoh else 0,
                                       _stream_ptr(stream))
        else:
            rc = lib().selscan_step(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                    _ptr(y), Bsz, D, N, _stream_ptr(stream))
    _check(rc)
    return y


def conv1d(x, w, bias=None, silu: bool = True, state_in=None, return_state: bool = False, out=None,
           state_out=None, stream=None):
    """Causal depthwise convolution and SiLU in front of the scan (see
    ``include/selscan.h``, selscan_conv1d): x (Bsz, L, D) float32 or
    bfloat16, w (D, K) float32, bias (D,) or None, state_in (Bsz, D, K-1)
    float32 or None. Returns out (like x), or (out, state_out) with the last
    K-1 inputs when ``return_state``. Device tensors only."""
    import torch
    dev = x.device
    Bsz, L, D = x.shape
    K = w.shape[1] if w.dim() == 2 else -1
    code = _dtype_code(x)
    _need(x, "x", (Bsz, L, D), x.dtype, dev)
    _need(w, "w", (D, K), torch.float32, dev)
    if bias is not None:
        _need(bias, "bias", (D,), torch.float32, dev)
    if state_in is not None:
        _need(state_in, "state_in", (Bsz, D, K - 1), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    else:
        _need(out, "out", (Bsz, L, D), x.dtype, dev)
    if return_state and state_out is None:
        state_out = torch.empty((Bsz, D, K - 1), dtype=torch.float32, device=dev)
    if state_out is not None:
        _need(state_out, "state_out", (Bsz, D, K - 1), torch.float32, dev)
    with torch.cuda.device(dev):
        rc = lib().selscan_conv1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), Bsz, L, D, K, code,
                                  int(bool(silu)), _ptr(state_in), _ptr(state_out), _stream_ptr(stream))
    _check(rc)
    return (out, state_out) if (return_state or state_out is not None) else out


def conv1d_step(conv_state, x, w, bias=None, silu: bool = True, out=None, stream=None):
    """One decode step of conv1d (selscan_conv1d_step): conv_state
    (Bsz, D, K-1) float32 is updated in place; returns out (Bsz, D)."""
    import torch
    dev = x.device
    Bsz, D = x.shape
    K = w.shape[1] if w.dim() == 2 else -1
    f = torch.float32
    _need(x, "x", (Bsz, D), f, dev)
    _need(w, "w", (D, K), f, dev)
    _need(conv_state, "conv_state", (Bsz, D, K - 1), f, dev)
    if bias is not None:
        _need(bias, "bias", (D,), f, dev)
    if out is None:
        out = torch.empty((Bsz, D), dtype=f, device=dev)
    else:
        _need(out, "out", (Bsz, D), f, dev)
    with torch.cuda.device(dev):
        rc = lib().selscan_conv1d_step(_ptr(conv_state) if K > 1 else None, _ptr(x), _ptr(w), _ptr(bias),
                                       _ptr(out), Bsz, D, K, int(bool(silu)), _stream_ptr(stream))
    _check(rc)
    return out


def ssd_fwd(x, dt, A, B, C, dt_softplus: bool = True, h0=None, return_final_state: bool = False, y=None,
            hT=None, stream=None, check: bool = False):
    """Mamba-2 SSD forward (selscan_ssd_fwd): x (Bsz, L, H, P) float32 or
    bfloat16, dt (Bsz, L, H) float32, A (H,) float32, B, C (Bsz, L, N) like
    x, h0 (Bsz, H, N, P) float32 or None. Returns y (like x), or (y, hT)
    when ``return_final_state``. Device tensors only."""
    import torch
    dev = x.device
    Bsz, L, H, P = x.shape
    N = B.shape[2] if B.dim() == 3 else -1
    code = _dtype_code(x)
    f = torch.float32
    _need(x, "x", (Bsz, L, H, P), x.dtype, dev)
    _need(dt, "dt", (Bsz, L, H), f, dev)
    _need(A, "A", (H,), f, dev)
    _need(B, "B", (Bsz, L, N), x.dtype, dev)
    _need(C, "C", (Bsz, L, N), x.dtype, dev)
    if h0 is not None:
        _need(h0, "h0", (Bsz, H, N, P), f, dev)
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", (Bsz, L, H, P), x.dtype, dev)
    if return_final_state and hT is None:
        hT = torch.empty((Bsz, H, N, P), dtype=f, device=dev)
    if hT is not None:
        _need(hT, "hT", (Bsz, H, N, P), f, dev)
    with torch.cuda.device(dev):
        rc = lib().selscan_ssd_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(y), _ptr(h0), _ptr(hT),
                                   Bsz, L, H, P, N, code, int(bool(dt_softplus)), _stream_ptr(stream))
    _check(rc)
    if check:
        check_device_error(stream)
    return (y, hT) if (return_final_state or hT is not None) else y


# ---- host tensors: copy in, run on the current device, copy out ------------

def _to_dev(t, dev):
    return None if t is None else t.to(dev, non_blocking=True)


def _fwd_host(x, delta, A, B, C, delta_softplus, h0, return_final_state, y, hT, D_skip=None, z=None,
              zoh=False):
    """Host tensors: one selscan_fwd_host (or, with the skip, gate or
    zero-order hold, selscan_fwd_host_ex) call: the library pipelines the
    copies in, the scan and the copies out on the current device. Returns
    once the outputs are in host memory. Page-locked tensors let the copies
    overlap the scan."""
    import torch
    Bsz, L, D = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    code = _dtype_code(x)
    cpu = torch.device("cpu")
    for t, name, shape, dt in ((x, "x", (Bsz, L, D), x.dtype), (delta, "delta", (Bsz, L, D), x.dtype),
                               (A, "A", (D, N), torch.float32), (B, "B", (Bsz, L, N), x.dtype),
                               (C, "C", (Bsz, L, N), x.dtype)):
        _need(t, name, shape, dt, cpu)
    if h0 is not None:
        _need(h0, "h0", (Bsz, D, N), torch.float32, cpu)
    want_state = return_final_state or hT is not None
    if y is None:
        y = torch.empty((Bsz, L, D), dtype=x.dtype, pin_memory=True)
    else:
        _need(y, "y", (Bsz, L, D), x.dtype, cpu)
    if want_state and hT is None:
        hT = torch.empty((Bsz, D, N), dtype=torch.float32, pin_memory=True)
    if hT is not None:
        _need(hT, "hT", (Bsz, D, N), torch.float32, cpu)
    if D_skip is not None:
        _need(D_skip, "D_skip", (D,), torch.float32, cpu)
    if z is not None:
        _need(z, "z", (Bsz, L, D), x.dtype, cpu)
    if D_skip is not None or z is not None or zoh:
        flags = (FLAG_SOFTPLUS if delta_softplus else 0) | (FLAG_ZOH if zoh else 0)
        rc = lib().selscan_fwd_host_ex(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D_skip), _ptr(z),
                                       _ptr(y), Bsz, L, D, N, code, flags, _ptr(h0), _ptr(hT), _stream_ptr(None))
    else:
        rc = lib().selscan_fwd_host(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(y),
                                    Bsz, L, D, N, code, int(bool(delta_softplus)), _ptr(h0), _ptr(hT),
                                    _stream_ptr(None))
    _check(rc)
    return (y, hT) if want_state else y


def _step_host(state, x, delta, A, B, C, y):
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    sd, xd, dd, Ad, Bd, Cd = (_to_dev(t, dev) for t in (state, x, delta, A, B, C))
    yd = selscan_step(sd, xd, dd, Ad, Bd, Cd)
    if y is None:
        y = torch.empty(yd.shape, dtype=yd.dtype, pin_memory=True)
    y.copy_(yd, non_blocking=True)
    state.copy_(sd, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    return y
