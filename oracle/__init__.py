"""fp64 CPU oracle for the selective state space (S6) scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never imports it and shares
no code with it.

The arithmetic lives in ``ssm_oracle.c`` (plain C, fp64, one pthread per
block of channels).  This module only compiles it with gcc and marshals numpy
arrays.  See the header of ``ssm_oracle.c`` for the passages each step
follows.

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: hand-worked examples, the convolution form of the LTI
case, Theorem 1's gated RNN, brute-force unrolled sums, the tree-order
evaluation of the associative combine, and the reset / ignore limits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")

DISC_EULER = 0
DISC_ZOH = 1
ORDER_SEQUENTIAL = 0
ORDER_TREE = 1

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared object with gcc (IEEE fp64, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-D_GNU_SOURCE", src, "-o", out, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build(path: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Load (compiling if stale) the oracle library. ``path`` loads another build of it."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build(_LIB_PATH):
                compile_oracle()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_selective_scan.restype = ctypes.c_int
    lib.oracle_selective_scan.argtypes = [i64, i64, i64, i64] + [dp] * 9 + [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, ctypes.c_int]
    lib.oracle_state_update.restype = ctypes.c_int
    lib.oracle_state_update.argtypes = [i64, i64, i64, dp] + [dp] * 8 + [
        ctypes.c_int, ctypes.c_int, dp]
    lib.oracle_selective_scan_bwd.restype = ctypes.c_int
    lib.oracle_selective_scan_bwd.argtypes = [i64, i64, i64, i64] + [dp] * 9 + [ctypes.c_int] + [dp] * 11 + \
        [ctypes.c_int]
    lib.oracle_causal_conv1d.restype = ctypes.c_int
    lib.oracle_causal_conv1d.argtypes = [i64, i64, i64, i64] + [dp] * 4 + [ctypes.c_int, dp]
    lib.oracle_selective_scan_complex.restype = ctypes.c_int
    lib.oracle_selective_scan_complex.argtypes = [i64, i64, i64, i64] + [dp] * 10 + [ctypes.c_int, dp, dp]
    lib.oracle_ssd_scan.restype = ctypes.c_int
    lib.oracle_ssd_scan.argtypes = [i64] * 5 + [dp] * 9 + [ctypes.c_int, dp, dp]
    lib.oracle_default_threads.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    return lib


def _f64(a, shape=None):
    if a is None:
        return None
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and arr.shape != tuple(shape):
        arr = np.ascontiguousarray(np.broadcast_to(arr, shape))
    return arr


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return int(load().oracle_default_threads())


def selective_scan(u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, h0=None,
                   delta_softplus=True, disc=DISC_EULER, order=ORDER_SEQUENTIAL,
                   return_last_state=False, nthreads=0, lib=None):
    """fp64 selective scan.

    u, delta, z: (B, D, L); Bm, Cm: (B, N, L) (a leading batch of 1 is broadcast);
    A: (D, N); Dskip, delta_bias: (D,); h0: (B, D, N).
    Returns y (B, D, L) float64, and h_last (B, D, N) if ``return_last_state``.
    """
    lib = lib or load()
    u = _f64(u)
    Bsz, D, L = u.shape
    A = _f64(A)
    N = A.shape[1]
    delta = _f64(delta, (Bsz, D, L))
    z = _f64(z, (Bsz, D, L))
    Bm = _f64(Bm, (Bsz, N, L))
    Cm = _f64(Cm, (Bsz, N, L))
    Dskip = _f64(Dskip, (D,))
    delta_bias = _f64(delta_bias, (D,))
    h0 = _f64(h0, (Bsz, D, N))
    y = np.empty((Bsz, D, L), dtype=np.float64)
    h_last = np.empty((Bsz, D, N), dtype=np.float64) if return_last_state else None
    rc = lib.oracle_selective_scan(Bsz, D, L, N, _ptr(u), _ptr(delta), _ptr(z), _ptr(Bm),
                                   _ptr(Cm), _ptr(A), _ptr(Dskip), _ptr(delta_bias), _ptr(h0),
                                   int(bool(delta_softplus)), int(disc), int(order), _ptr(y),
                                   _ptr(h_last), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_selective_scan failed")
    return (y, h_last) if return_last_state else y


def selective_scan_complex(u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None, h0=None,
                           delta_softplus=True, return_last_state=False, lib=None):
    """fp64 selective scan with a complex diagonal A (S4D-Lin): complex state, real input term,
    y = Re(C . h) + D u (then the gate).

    A: complex (D, N); h0: complex (B, D, N) or None; other arguments as for selective_scan.
    Returns y (B, D, L) float64, and the complex h_last (B, D, N) if ``return_last_state``.
    """
    lib = lib or load()
    u = _f64(u)
    Bsz, D, L = u.shape
    A = np.asarray(A, dtype=np.complex128)
    N = A.shape[1]
    A_re = np.ascontiguousarray(A.real)
    A_im = np.ascontiguousarray(A.imag)
    delta = _f64(delta, (Bsz, D, L))
    z = _f64(z, (Bsz, D, L))
    Bm = _f64(Bm, (Bsz, N, L))
    Cm = _f64(Cm, (Bsz, N, L))
    Dskip = _f64(Dskip, (D,))
    delta_bias = _f64(delta_bias, (D,))
    h0c = None
    if h0 is not None:
        h0c = np.ascontiguousarray(np.broadcast_to(np.asarray(h0, dtype=np.complex128), (Bsz, D, N)))
    y = np.empty((Bsz, D, L), dtype=np.float64)
    h_last = np.empty((Bsz, D, N), dtype=np.complex128) if return_last_state else None
    cp = lambda a: None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.oracle_selective_scan_complex(Bsz, D, L, N, _ptr(u), _ptr(delta), _ptr(z), _ptr(Bm), _ptr(Cm),
                                           _ptr(A_re), _ptr(A_im), _ptr(Dskip), _ptr(delta_bias), cp(h0c),
                                           int(bool(delta_softplus)), _ptr(y), cp(h_last))
    if rc != 0:
        raise RuntimeError("oracle_selective_scan_complex failed")
    return (y, h_last) if return_last_state else y


def ssd_scan(x, delta, a, Bm, Cm, Dskip=None, z=None, delta_bias=None, h0=None, delta_softplus=True,
             return_last_state=False, lib=None):
    """fp64 Mamba-2 SSD layer (scalar A per head, B / C shared by the heads).

    x, z: (B, H*P, L); delta: (B, H, L); a, Dskip, delta_bias: (H,); Bm, Cm: (B, L, N);
    h0: (B, H, P, N).  Returns y (B, H*P, L), and h_last (B, H, P, N) if ``return_last_state``.
    """
    lib = lib or load()
    delta = _f64(delta)
    Bsz, H, L = delta.shape
    x = _f64(x)
    P = x.shape[1] // H
    Bm = _f64(Bm)
    N = Bm.shape[2]
    Cm = _f64(Cm, (Bsz, L, N))
    z = _f64(z, x.shape)
    a = _f64(a, (H,))
    Dskip = _f64(Dskip, (H,))
    delta_bias = _f64(delta_bias, (H,))
    h0 = _f64(h0, (Bsz, H, P, N))
    y = np.empty(x.shape, dtype=np.float64)
    h_last = np.empty((Bsz, H, P, N), dtype=np.float64) if return_last_state else None
    rc = lib.oracle_ssd_scan(Bsz, H, P, L, N, _ptr(x), _ptr(delta), _ptr(z), _ptr(Bm), _ptr(Cm), _ptr(a),
                             _ptr(Dskip), _ptr(delta_bias), _ptr(h0), int(bool(delta_softplus)), _ptr(y),
                             _ptr(h_last))
    if rc != 0:
        raise RuntimeError("oracle_ssd_scan failed")
    return (y, h_last) if return_last_state else y


def s4d_lin(D, N):
    """The S4D-Lin initialisation of a complex diagonal A: A[d, n] = -1/2 + n i ("gitcode",
    section 3.6, initialisation)."""
    return np.broadcast_to(-0.5 + 1j * np.arange(N, dtype=np.float64), (D, N)).copy()


def state_update(state, u, delta, A, Bm, Cm, Dskip=None, z=None, delta_bias=None,
                 delta_softplus=True, disc=DISC_EULER, lib=None):
    """One fp64 decode step. state (B, D, N); u, delta, z (B, D); Bm, Cm (B, N).

    Returns (new_state, y); the input ``state`` is not modified.
    """
    lib = lib or load()
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    Bsz, D, N = st.shape
    u = _f64(u, (Bsz, D))
    delta = _f64(delta, (Bsz, D))
    z = _f64(z, (Bsz, D))
    Bm = _f64(Bm, (Bsz, N))
    Cm = _f64(Cm, (Bsz, N))
    A = _f64(A, (D, N))
    Dskip = _f64(Dskip, (D,))
    delta_bias = _f64(delta_bias, (D,))
    y = np.empty((Bsz, D), dtype=np.float64)
    rc = lib.oracle_state_update(Bsz, D, N, _ptr(st), _ptr(u), _ptr(delta), _ptr(z), _ptr(Bm),
                                 _ptr(Cm), _ptr(A), _ptr(Dskip), _ptr(delta_bias),
                                 int(bool(delta_softplus)), int(disc), _ptr(y))
    if rc != 0:
        raise RuntimeError("oracle_state_update failed")
    return st, y


def causal_conv1d(x, w, bias=None, x_hist=None, silu=True, lib=None):
    """fp64 causal depthwise convolution along time, then SiLU if ``silu``.

    x: (B, D, L); w: (D, W), tap W-1 on the current step; bias: (D,);
    x_hist: (B, D, W-1), the inputs before t = 0 (oldest first), zero if None.
    Returns out (B, D, L) float64.
    """
    lib = lib or load()
    x = _f64(x)
    Bsz, D, L = x.shape
    w = _f64(w)
    W = w.shape[1]
    bias = _f64(bias, (D,))
    x_hist = _f64(x_hist, (Bsz, D, W - 1)) if W > 1 else None
    out = np.empty((Bsz, D, L), dtype=np.float64)
    rc = lib.oracle_causal_conv1d(Bsz, D, L, W, _ptr(x), _ptr(w), _ptr(bias), _ptr(x_hist),
                                  int(bool(silu)), _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_causal_conv1d failed")
    return out


def selective_scan_bwd(u, delta, A, Bm, Cm, dy, Dskip=None, z=None, delta_bias=None, h0=None,
                       delta_softplus=True, dh_last=None, disc=DISC_EULER, lib=None):
    """fp64 gradients of the selective scan (Euler or exact-ZOH input term, ``disc``) for an upstream
    gradient dy (B, D, L) of y and, optionally, dh_last (B, D, N) of the final state.

    Returns a dict with du, ddelta (B, D, L); dz (B, D, L) if z is given; dBm, dCm shaped like the
    given Bm, Cm (a leading batch of 1 gets the sum over the batch); dA (D, N); dDskip (D,) if Dskip is
    given; ddelta_bias (D,); dh0 (B, D, N).
    """
    lib = lib or load()
    u = _f64(u)
    Bsz, D, L = u.shape
    A = _f64(A)
    N = A.shape[1]
    bc_shared = np.asarray(Bm).shape[0] == 1 and Bsz != 1
    delta = _f64(delta, (Bsz, D, L))
    z = _f64(z, (Bsz, D, L))
    Bm = _f64(Bm, (Bsz, N, L))
    Cm = _f64(Cm, (Bsz, N, L))
    Dskip = _f64(Dskip, (D,))
    delta_bias = _f64(delta_bias, (D,))
    h0 = _f64(h0, (Bsz, D, N))
    dy = _f64(dy, (Bsz, D, L))
    dh_last = _f64(dh_last, (Bsz, D, N))
    out = {k: np.empty(s, dtype=np.float64) for k, s in (
        ("du", (Bsz, D, L)), ("ddelta", (Bsz, D, L)), ("dBm", (Bsz, N, L)), ("dCm", (Bsz, N, L)),
        ("dA", (D, N)), ("ddelta_bias", (D,)), ("dh0", (Bsz, D, N)))}
    out["dz"] = np.empty((Bsz, D, L)) if z is not None else None
    out["dDskip"] = np.empty(D) if Dskip is not None else None
    rc = lib.oracle_selective_scan_bwd(Bsz, D, L, N, _ptr(u), _ptr(delta), _ptr(z), _ptr(Bm), _ptr(Cm),
                                       _ptr(A), _ptr(Dskip), _ptr(delta_bias), _ptr(h0),
                                       int(bool(delta_softplus)), _ptr(dy), _ptr(dh_last),
                                       _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dz"]), _ptr(out["dBm"]),
                                       _ptr(out["dCm"]), _ptr(out["dA"]), _ptr(out["dDskip"]),
                                       _ptr(out["ddelta_bias"]), _ptr(out["dh0"]), int(disc))
    if rc != 0:
        raise RuntimeError("oracle_selective_scan_bwd failed")
    if bc_shared:
        out["dBm"] = out["dBm"].sum(axis=0, keepdims=True)
        out["dCm"] = out["dCm"].sum(axis=0, keepdims=True)
    return out
