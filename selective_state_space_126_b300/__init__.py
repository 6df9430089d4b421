"""B300-native selective state space (S6) scan and decode step.

A thin ctypes binding over ``libssm.so`` (C ABI in ``include/ssm.h``).  The
functions here only marshal torch tensors into the C argument structs; every
step of the scan and of the decode update runs in the library's CUDA
kernels.  There is no CPU fallback: if ``libssm.so`` is missing or no CUDA
device is present, the calls raise.

Public API (same names as the C entry points):
  ssm_scan_fwd(u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, h0=None, ...)
  ssm_state_update(state, u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, ...)
  ssm_scan_bwd(u, delta, A, Bm, Cm, dy, Dskip=None, z=None, delta_bias=None, h0=None, dh_last=None, ...)
  ssm_causal_conv1d_fwd(x, weight, bias=None, x_hist=None, silu=True, ...)
  ssm_scan_workspace_size(...), ssm_status_string(code), ssm_version()
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssm.so")

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_WORKSPACE = range(6)
SSM_F32, SSM_BF16 = 0, 1
SSM_SCAN_FORCE_GENERIC, SSM_SCAN_FORCE_TILED, SSM_SCAN_FORCE_CHUNKED, SSM_SCAN_FORCE_WARPSCAN = 0x1, 0x2, 0x4, 0x8
SSM_DISC_EULER, SSM_DISC_ZOH = 0, 1
PATH_NAMES = {0: "generic", 1: "tiled", 2: "chunked", 3: "warpscan", 4: "split"}

# every symbol include/ssm.h declares
EXPORTED_SYMBOLS = ["ssm_scan_workspace_size", "ssm_scan_fwd", "ssm_state_update", "ssm_status_string",
                    "ssm_last_error_detail", "ssm_get_device_status", "ssm_scan_plan_path", "ssm_version",
                    "ssm_abi_sizeof", "ssm_scan_fwd_noalloc", "ssm_causal_conv1d_fwd",
                    "ssm_scan_bwd_workspace_size", "ssm_scan_bwd", "ssm_probe_sfu", "ssm_ssd_fwd",
                    "ssm_ssd_plan_path"]

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


class ScanArgs(ctypes.Structure):
    """Mirror of ssm_scan_args_t."""
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64), ("dstate", _i64),
        ("io_dtype", ctypes.c_int), ("delta_softplus", ctypes.c_int32),
        ("u", _vp), ("delta", _vp), ("z", _vp), ("Bm", _vp), ("Cm", _vp),
        ("A", _vp), ("Dskip", _vp), ("delta_bias", _vp), ("h0", _vp), ("h_last", _vp), ("y", _vp),
        ("stride_u", _i64 * 3), ("stride_delta", _i64 * 3), ("stride_z", _i64 * 3), ("stride_y", _i64 * 3),
        ("stride_B", _i64 * 3), ("stride_C", _i64 * 3), ("stride_A", _i64 * 2),
        ("stride_h0", _i64 * 3), ("stride_h_last", _i64 * 3),
        ("flags", ctypes.c_int32), ("discretization", ctypes.c_int32), ("chunk_len", _i64),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("A_imag", _vp),
    ]


class SsdArgs(ctypes.Structure):
    """Mirror of ssm_ssd_args_t."""
    _fields_ = [
        ("batch", _i64), ("nheads", _i64), ("headdim", _i64), ("seqlen", _i64), ("dstate", _i64),
        ("io_dtype", ctypes.c_int), ("delta_softplus", ctypes.c_int32),
        ("x", _vp), ("delta", _vp), ("z", _vp), ("Bm", _vp), ("Cm", _vp),
        ("A", _vp), ("Dskip", _vp), ("delta_bias", _vp), ("h0", _vp), ("h_last", _vp), ("y", _vp),
        ("stride_x", _i64 * 3), ("stride_z", _i64 * 3), ("stride_y", _i64 * 3), ("stride_delta", _i64 * 3),
        ("stride_B", _i64 * 3), ("stride_C", _i64 * 3), ("stride_h0", _i64 * 4), ("stride_h_last", _i64 * 4),
        ("flags", ctypes.c_int32), ("reserved0", ctypes.c_int32),
    ]


class StepArgs(ctypes.Structure):
    """Mirror of ssm_step_args_t."""
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("dstate", _i64),
        ("io_dtype", ctypes.c_int), ("delta_softplus", ctypes.c_int32),
        ("state", _vp), ("u", _vp), ("delta", _vp), ("z", _vp), ("Bm", _vp), ("Cm", _vp),
        ("A", _vp), ("Dskip", _vp), ("delta_bias", _vp), ("y", _vp),
        ("stride_state", _i64 * 3), ("stride_u", _i64 * 2), ("stride_delta", _i64 * 2),
        ("stride_z", _i64 * 2), ("stride_y", _i64 * 2), ("stride_B", _i64 * 2), ("stride_C", _i64 * 2),
        ("stride_A", _i64 * 2), ("discretization", ctypes.c_int32), ("reserved0", ctypes.c_int32),
    ]


class ConvArgs(ctypes.Structure):
    """Mirror of ssm_conv_args_t."""
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64),
        ("width", ctypes.c_int32), ("io_dtype", ctypes.c_int), ("silu", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("x", _vp), ("weight", _vp), ("bias", _vp), ("x_hist", _vp), ("out", _vp),
        ("stride_x", _i64 * 3), ("stride_out", _i64 * 3), ("stride_weight", _i64 * 2),
        ("stride_x_hist", _i64 * 3),
    ]


class BwdArgs(ctypes.Structure):
    """Mirror of ssm_scan_bwd_args_t."""
    _fields_ = [
        ("fwd", ScanArgs),
        ("dy", _vp), ("dh_last", _vp),
        ("du", _vp), ("ddelta", _vp), ("dz", _vp),
        ("dA", _vp), ("dB", _vp), ("dC", _vp), ("dDskip", _vp), ("ddelta_bias", _vp), ("dh0", _vp),
        ("stride_dy", _i64 * 3), ("stride_du", _i64 * 3), ("stride_ddelta", _i64 * 3), ("stride_dz", _i64 * 3),
        ("stride_dB", _i64 * 3), ("stride_dC", _i64 * 3), ("stride_dh_last", _i64 * 3), ("stride_dh0", _i64 * 3),
    ]


class SsmError(RuntimeError):
    def __init__(self, code, detail=""):
        self.code = code
        super().__init__(f"{status_name(code)}: {detail}" if detail else status_name(code))


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libssm.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with `python -m selective_state_space_126_b300.build`")
        lib = ctypes.CDLL(path)
        lib.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanArgs), ctypes.POINTER(ctypes.c_size_t)]
        lib.ssm_scan_workspace_size.restype = ctypes.c_int
        lib.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanArgs), _vp]
        lib.ssm_scan_fwd.restype = ctypes.c_int
        lib.ssm_state_update.argtypes = [ctypes.POINTER(StepArgs), _vp]
        lib.ssm_state_update.restype = ctypes.c_int
        lib.ssm_status_string.argtypes = [ctypes.c_int]
        lib.ssm_status_string.restype = ctypes.c_char_p
        lib.ssm_last_error_detail.argtypes = []
        lib.ssm_last_error_detail.restype = ctypes.c_char_p
        lib.ssm_get_device_status.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        lib.ssm_get_device_status.restype = ctypes.c_int
        lib.ssm_scan_plan_path.argtypes = [ctypes.POINTER(ScanArgs)]
        lib.ssm_scan_plan_path.restype = ctypes.c_int
        lib.ssm_version.argtypes = []
        lib.ssm_version.restype = ctypes.c_int
        lib.ssm_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ScanArgs), _vp]
        lib.ssm_scan_fwd_noalloc.restype = ctypes.c_int
        lib.ssm_abi_sizeof.argtypes = [ctypes.c_int]
        lib.ssm_abi_sizeof.restype = ctypes.c_size_t
        lib.ssm_causal_conv1d_fwd.argtypes = [ctypes.POINTER(ConvArgs), _vp]
        lib.ssm_causal_conv1d_fwd.restype = ctypes.c_int
        lib.ssm_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(BwdArgs), ctypes.POINTER(ctypes.c_size_t)]
        lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_int
        lib.ssm_scan_bwd.argtypes = [ctypes.POINTER(BwdArgs), _vp]
        lib.ssm_scan_bwd.restype = ctypes.c_int
        lib.ssm_probe_sfu.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp]
        lib.ssm_probe_sfu.restype = ctypes.c_int
        lib.ssm_ssd_fwd.argtypes = [ctypes.POINTER(SsdArgs), _vp]
        lib.ssm_ssd_fwd.restype = ctypes.c_int
        lib.ssm_ssd_plan_path.argtypes = [ctypes.POINTER(SsdArgs)]
        lib.ssm_ssd_plan_path.restype = ctypes.c_int
        if (lib.ssm_abi_sizeof(0) != ctypes.sizeof(ScanArgs) or lib.ssm_abi_sizeof(1) != ctypes.sizeof(StepArgs)
                or lib.ssm_abi_sizeof(2) != ctypes.sizeof(ConvArgs) or lib.ssm_abi_sizeof(3) != ctypes.sizeof(BwdArgs)
                or lib.ssm_abi_sizeof(4) != ctypes.sizeof(SsdArgs)):
            raise ImportError("libssm.so argument structs do not match this binding")
        if path == LIB_PATH:
            _lib = lib
        return lib


def status_name(code: int) -> str:
    try:
        return load_library().ssm_status_string(int(code)).decode()
    except ImportError:
        return f"status {code}"


def ssm_status_string(code: int) -> str:
    return status_name(code)


def ssm_version() -> int:
    return int(load_library().ssm_version())


def _check(code: int):
    if code != SSM_OK:
        raise SsmError(code, load_library().ssm_last_error_detail().decode())


# ---------------------------------------------------------------------------
# torch marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _io_dtype(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported I/O dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _strides(t, rank, dims=None):
    if t is None:
        return [0] * rank
    s = list(t.stride())
    if dims is not None and t.dim() == rank - 1:   # broadcast over a missing batch dimension
        s = [0] + s
    elif dims is not None and t.dim() == rank and t.shape[0] == 1:   # a batch of one is broadcast
        s[0] = 0
    if len(s) != rank:
        raise ValueError(f"expected a {rank}-d tensor, got shape {tuple(t.shape)}")
    return s


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _f32(t, name):
    torch = _torch()
    if t is None:
        return None
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t


def _state_strides(t):
    """Strides of a (B, D, N) state tensor in floats: a complex tensor holds (re, im) float pairs."""
    if t is None:
        return [0, 0, 0]
    s = _strides(t, 3)
    return [2 * v for v in s] if t.is_complex() else s


def make_scan_args(u, delta, A, Bm, Cm, y, Dskip=None, z=None, delta_bias=None, h0=None, h_last=None,
                   delta_softplus=True, flags=0, chunk_len=0, workspace=None,
                   discretization=SSM_DISC_EULER, A_imag=None) -> ScanArgs:
    """Fill an ssm_scan_args_t from torch tensors (no copies, strides passed through).  With A_imag (the
    imaginary part of a complex A, strides of A) h0 / h_last are complex64 tensors."""
    Bsz, D, L = u.shape
    N = A.shape[1]
    a = ScanArgs()
    a.batch, a.dim, a.seqlen, a.dstate = Bsz, D, L, N
    a.io_dtype = _io_dtype(u)
    a.delta_softplus = 1 if delta_softplus else 0
    a.u, a.delta, a.z, a.Bm, a.Cm = _ptr(u), _ptr(delta), _ptr(z), _ptr(Bm), _ptr(Cm)
    a.A, a.Dskip, a.delta_bias = _ptr(A), _ptr(Dskip), _ptr(delta_bias)
    a.h0, a.h_last, a.y = _ptr(h0), _ptr(h_last), _ptr(y)
    a.stride_u[:] = _strides(u, 3)
    a.stride_delta[:] = _strides(delta, 3)
    a.stride_z[:] = _strides(z, 3)
    a.stride_y[:] = _strides(y, 3)
    a.stride_B[:] = _strides(Bm, 3, dims="b")
    a.stride_C[:] = _strides(Cm, 3, dims="b")
    a.stride_A[:] = _strides(A, 2)
    a.stride_h0[:] = _state_strides(h0)
    a.stride_h_last[:] = _state_strides(h_last)
    a.A_imag = _ptr(A_imag)
    if A_imag is not None and tuple(A_imag.stride()) != tuple(A.stride()):
        raise ValueError("A_imag must have the strides of A")
    a.flags = int(flags)
    a.discretization = int(discretization)
    a.chunk_len = int(chunk_len)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def ssm_scan_workspace_size(args: ScanArgs) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().ssm_scan_workspace_size(ctypes.byref(args), ctypes.byref(n)))
    return int(n.value)


def ssm_scan_plan_path(args: ScanArgs) -> str:
    return PATH_NAMES.get(int(load_library().ssm_scan_plan_path(ctypes.byref(args))), "invalid")


def ssm_scan_fwd(u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, h0=None, delta_softplus=True,
                 y=None, return_last_state=False, h_last=None, workspace=None, flags=0, chunk_len=0,
                 stream=None, discretization=SSM_DISC_EULER):
    """Selective-scan forward pass on the GPU (``discretization``: SSM_DISC_EULER or SSM_DISC_ZOH).

    u, delta, z: (B, D, L); Bm, Cm: (B, N, L) or (N, L) (shared across the batch);
    A: (D, N) fp32, or complex64 for a complex diagonal (S4D-Lin); Dskip, delta_bias: (D,) fp32;
    h0: (B, D, N) fp32 (complex64 with a complex A).
    I/O tensors are float32 or bfloat16 (all the same dtype), on one CUDA device.
    Returns y (B, D, L) in the I/O dtype, and h_last (B, D, N) fp32 (complex64 with a complex A) if
    requested.
    """
    torch = _torch()
    lib = load_library()
    for name, t in (("u", u), ("delta", delta), ("Bm", Bm), ("Cm", Cm), ("z", z)):
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    A_imag = None
    cplx = A.is_complex()
    if cplx:
        if A.dtype != torch.complex64:
            raise ValueError("a complex A must be complex64")
        A, A_imag = A.real.contiguous(), A.imag.contiguous()
        if h0 is not None and h0.dtype != torch.complex64:
            raise ValueError("with a complex A, h0 must be complex64")
    _f32(A, "A"); _f32(Dskip, "Dskip"); _f32(delta_bias, "delta_bias")
    if not cplx:
        _f32(h0, "h0")
    if Dskip is not None:
        Dskip = Dskip.contiguous()
    if delta_bias is not None:
        delta_bias = delta_bias.contiguous()
    if y is None:
        y = torch.empty(u.shape, dtype=u.dtype, device=u.device)
    if return_last_state and h_last is None:
        h_last = torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.complex64 if cplx else torch.float32,
                             device=u.device)
    args = make_scan_args(u, delta, A, Bm, Cm, y, Dskip, z, delta_bias, h0, h_last, delta_softplus, flags,
                          chunk_len, None, discretization, A_imag)
    need = ssm_scan_workspace_size(args)
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=u.device)
        args.workspace = workspace.data_ptr()
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.ssm_scan_fwd(ctypes.byref(args), _vp(_stream_handle(stream))))
    return (y, h_last) if return_last_state else y


def make_step_args(state, u, delta, A, Bm, Cm, y, Dskip=None, z=None, delta_bias=None,
                   delta_softplus=True, discretization=SSM_DISC_EULER) -> StepArgs:
    Bsz, D, N = state.shape
    a = StepArgs()
    a.batch, a.dim, a.dstate = Bsz, D, N
    a.io_dtype = _io_dtype(u)
    a.delta_softplus = 1 if delta_softplus else 0
    a.state, a.u, a.delta, a.z, a.Bm, a.Cm = _ptr(state), _ptr(u), _ptr(delta), _ptr(z), _ptr(Bm), _ptr(Cm)
    a.A, a.Dskip, a.delta_bias, a.y = _ptr(A), _ptr(Dskip), _ptr(delta_bias), _ptr(y)
    a.stride_state[:] = _strides(state, 3)
    a.stride_u[:] = _strides(u, 2)
    a.stride_delta[:] = _strides(delta, 2)
    a.stride_z[:] = _strides(z, 2)
    a.stride_y[:] = _strides(y, 2)
    a.stride_B[:] = _strides(Bm, 2)
    a.stride_C[:] = _strides(Cm, 2)
    a.stride_A[:] = _strides(A, 2)
    a.discretization = int(discretization)
    return a


def ssm_state_update(state, u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, delta_softplus=True,
                     y=None, stream=None, discretization=SSM_DISC_EULER):
    """One decode step: ``state`` (B, D, N) fp32 is updated in place; returns y (B, D)."""
    torch = _torch()
    lib = load_library()
    _f32(state, "state"); _f32(A, "A"); _f32(Dskip, "Dskip"); _f32(delta_bias, "delta_bias")
    if Dskip is not None:
        Dskip = Dskip.contiguous()
    if delta_bias is not None:
        delta_bias = delta_bias.contiguous()
    if y is None:
        y = torch.empty(u.shape, dtype=u.dtype, device=u.device)
    args = make_step_args(state, u, delta, A, Bm, Cm, y, Dskip, z, delta_bias, delta_softplus, discretization)
    _check(lib.ssm_state_update(ctypes.byref(args), _vp(_stream_handle(stream))))
    return y


SSM_BWD_SEGMENT = 8


def make_bwd_args(fwd: ScanArgs, dy, grads: dict, dh_last=None) -> BwdArgs:
    """Fill an ssm_scan_bwd_args_t: ``fwd`` from make_scan_args (its y may be None), ``grads`` a dict of
    output tensors du, ddelta, dz, dA, dB, dC, dDskip, ddelta_bias, dh0 (missing keys = NULL)."""
    a = BwdArgs()
    a.fwd = fwd
    a.dy, a.dh_last = _ptr(dy), _ptr(dh_last)
    a.stride_dy[:] = _strides(dy, 3)
    a.stride_dh_last[:] = _strides(dh_last, 3)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dDskip", "ddelta_bias", "dh0"):
        setattr(a, k, _ptr(grads.get(k)))
    for k in ("du", "ddelta", "dz", "dh0"):
        getattr(a, "stride_" + k)[:] = _strides(grads.get(k), 3)
    for k in ("dB", "dC"):
        getattr(a, "stride_" + k)[:] = _strides(grads.get(k), 3, dims="b")
    return a


def ssm_scan_bwd(u, delta, A, Bm, Cm, dy, Dskip=None, z=None, delta_bias=None, h0=None, delta_softplus=True,
                 dh_last=None, return_dh0=True, workspace=None, stream=None, discretization=SSM_DISC_EULER):
    """Gradients of ssm_scan_fwd (Euler or exact-ZOH input term, ``discretization``) for an upstream
    gradient ``dy`` (B, D, L) of y (and ``dh_last`` (B, D, N) fp32 of the final state, optional).

    Returns a dict: du, ddelta (and dz if z is given) in the I/O dtype, (B, D, L); dA (D, N); dB, dC
    fp32 shaped like Bm, Cm ((N, L) when they are shared across the batch); dDskip (D,) if Dskip is
    given; ddelta_bias (D,) if delta_bias is given; dh0 (B, D, N) if ``return_dh0``.
    """
    torch = _torch()
    lib = load_library()
    for name, t in (("u", u), ("delta", delta), ("Bm", Bm), ("Cm", Cm), ("z", z), ("dy", dy)):
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    if dy.dtype != u.dtype:
        raise TypeError("dy must have u's dtype")
    _f32(A, "A"); _f32(Dskip, "Dskip"); _f32(delta_bias, "delta_bias"); _f32(h0, "h0"); _f32(dh_last, "dh_last")
    if Dskip is not None:
        Dskip = Dskip.contiguous()
    if delta_bias is not None:
        delta_bias = delta_bias.contiguous()
    Bsz, D, L = u.shape
    N = A.shape[1]
    dev = u.device
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dA": torch.empty((D, N), dtype=torch.float32, device=dev),
         "dB": torch.empty(tuple(Bm.shape), dtype=torch.float32, device=dev),
         "dC": torch.empty(tuple(Cm.shape), dtype=torch.float32, device=dev)}
    if z is not None:
        g["dz"] = torch.empty_like(u)
    if Dskip is not None:
        g["dDskip"] = torch.empty(D, dtype=torch.float32, device=dev)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty(D, dtype=torch.float32, device=dev)
    if return_dh0:
        g["dh0"] = torch.empty((Bsz, D, N), dtype=torch.float32, device=dev)
    fwd = make_scan_args(u, delta, A, Bm, Cm, None, Dskip, z, delta_bias, h0, None, delta_softplus,
                         discretization=discretization)
    args = make_bwd_args(fwd, dy, g, dh_last)
    need = ctypes.c_size_t(0)
    _check(lib.ssm_scan_bwd_workspace_size(ctypes.byref(args), ctypes.byref(need)))
    if need.value > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need.value:
            workspace = torch.empty(need.value, dtype=torch.uint8, device=dev)
        args.fwd.workspace = workspace.data_ptr()
        args.fwd.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.ssm_scan_bwd(ctypes.byref(args), _vp(_stream_handle(stream))))
    return g


def make_conv_args(x, weight, out, bias=None, x_hist=None, silu=True) -> ConvArgs:
    """Fill an ssm_conv_args_t from torch tensors (no copies, strides passed through)."""
    Bsz, D, L = x.shape
    a = ConvArgs()
    a.batch, a.dim, a.seqlen, a.width = Bsz, D, L, weight.shape[1]
    a.io_dtype = _io_dtype(x)
    a.silu = 1 if silu else 0
    a.x, a.weight, a.bias, a.x_hist, a.out = _ptr(x), _ptr(weight), _ptr(bias), _ptr(x_hist), _ptr(out)
    a.stride_x[:] = _strides(x, 3)
    a.stride_out[:] = _strides(out, 3)
    a.stride_weight[:] = _strides(weight, 2)
    a.stride_x_hist[:] = _strides(x_hist, 3)
    return a


def ssm_causal_conv1d_fwd(x, weight, bias=None, x_hist=None, silu=True, out=None, stream=None):
    """Causal depthwise convolution along time, then SiLU if ``silu``.

    x: (B, D, L) float32 or bfloat16; weight: (D, W) fp32, tap W-1 on the current step;
    bias: (D,) fp32; x_hist: (B, D, W-1) in x's dtype, the inputs before t = 0 (zero if None).
    Returns out (B, D, L) in x's dtype.
    """
    torch = _torch()
    lib = load_library()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    _f32(weight, "weight"); _f32(bias, "bias")
    if bias is not None:
        bias = bias.contiguous()
    if x_hist is not None and x_hist.dtype != x.dtype:
        raise TypeError("x_hist must have x's dtype")
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    args = make_conv_args(x, weight, out, bias, x_hist, silu)
    _check(lib.ssm_causal_conv1d_fwd(ctypes.byref(args), _vp(_stream_handle(stream))))
    return out


def ssm_get_device_status(clear=True, stream=None) -> int:
    code = ctypes.c_int(0)
    _check(load_library().ssm_get_device_status(_vp(_stream_handle(stream)), int(bool(clear)),
                                                 ctypes.byref(code)))
    return int(code.value)


# Bytes of the static scratch array ssm_scan_fwd_noalloc keeps its chunk records in.
SSM_NOALLOC_SCRATCH_BYTES = 8 << 20


def ssm_scan_fwd_noalloc(u, delta, A, Bm, Cm, y, Dskip=None, z=None, delta_bias=None, h0=None, h_last=None,
                         delta_softplus=True, chunk_len=0, stream=None, discretization=SSM_DISC_EULER):
    """The chunked scan without a caller workspace, for callers that cannot allocate.

    The caller passes every input and the outputs (``y`` and optionally
    ``h_last``); the chunk records live in a scratch array the library holds
    statically on each GPU (SSM_NOALLOC_SCRATCH_BYTES).  Nothing is allocated
    here or in the library.  Calls on one device share that array: do not let
    two of them overlap on the GPU.
    """
    args = make_scan_args(u, delta, A, Bm, Cm, y, Dskip, z, delta_bias, h0, h_last, delta_softplus,
                          SSM_SCAN_FORCE_CHUNKED, chunk_len, None, discretization)
    _check(load_library().ssm_scan_fwd_noalloc(ctypes.byref(args), _vp(_stream_handle(stream))))
    return y


SSM_SSD_FORCE_GENERIC = 0x1


def make_ssd_args(x, delta, A, Bm, Cm, y, Dskip=None, z=None, delta_bias=None, h0=None, h_last=None,
                  delta_softplus=True, flags=0) -> SsdArgs:
    """Fill an ssm_ssd_args_t from torch tensors: x, z, y (B, H*P, L); delta (B, H, L); Bm, Cm (B, L, N);
    A, Dskip, delta_bias (H,); h0, h_last (B, H, P, N)."""
    Bsz, H, L = delta.shape
    D = x.shape[1]
    N = Bm.shape[-1]
    a = SsdArgs()
    a.batch, a.nheads, a.headdim, a.seqlen, a.dstate = Bsz, H, D // H, L, N
    a.io_dtype = _io_dtype(x)
    a.delta_softplus = 1 if delta_softplus else 0
    a.x, a.delta, a.z, a.Bm, a.Cm = _ptr(x), _ptr(delta), _ptr(z), _ptr(Bm), _ptr(Cm)
    a.A, a.Dskip, a.delta_bias, a.h0, a.h_last, a.y = _ptr(A), _ptr(Dskip), _ptr(delta_bias), _ptr(h0), _ptr(h_last), _ptr(y)
    a.stride_x[:] = _strides(x, 3)
    a.stride_z[:] = _strides(z, 3)
    a.stride_y[:] = _strides(y, 3)
    a.stride_delta[:] = _strides(delta, 3)
    a.stride_B[:] = _strides(Bm, 3)
    a.stride_C[:] = _strides(Cm, 3)
    a.stride_h0[:] = _strides(h0, 4)
    a.stride_h_last[:] = _strides(h_last, 4)
    a.flags = int(flags)
    return a


def ssm_ssd_plan_path(args: SsdArgs) -> str:
    return {1: "tensor_core", 0: "generic"}.get(int(load_library().ssm_ssd_plan_path(ctypes.byref(args))), "invalid")


def ssm_ssd_fwd(x, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, h0=None, delta_softplus=True,
                y=None, return_last_state=False, h_last=None, flags=0, stream=None):
    """Mamba-2 SSD layer on the GPU: x, z (B, H*P, L); delta (B, H, L); Bm, Cm (B, L, N); A, Dskip,
    delta_bias (H,) fp32; h0 (B, H, P, N) fp32.  Returns y (B, H*P, L) in the I/O dtype, and h_last
    (B, H, P, N) fp32 if requested."""
    torch = _torch()
    lib = load_library()
    for name, t in (("x", x), ("delta", delta), ("Bm", Bm), ("Cm", Cm), ("z", z)):
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    _f32(A, "A"); _f32(Dskip, "Dskip"); _f32(delta_bias, "delta_bias"); _f32(h0, "h0")
    A = A.contiguous()
    Dskip = Dskip.contiguous() if Dskip is not None else None
    delta_bias = delta_bias.contiguous() if delta_bias is not None else None
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    Bsz, H, L = delta.shape
    if return_last_state and h_last is None:
        h_last = torch.empty((Bsz, H, x.shape[1] // H, Bm.shape[-1]), dtype=torch.float32, device=x.device)
    args = make_ssd_args(x, delta, A, Bm, Cm, y, Dskip, z, delta_bias, h0, h_last, delta_softplus, flags)
    _check(lib.ssm_ssd_fwd(ctypes.byref(args), _vp(_stream_handle(stream))))
    return (y, h_last) if return_last_state else y
