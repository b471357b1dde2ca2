"""fp64 CPU oracle for the SSD sequence-mixing forward pass.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
in ``ssd_sequence_mixing_fwd_b300``.

Two independent evaluations of the same map live here:

* :func:`recurrence` -- the C library ``ssd_oracle.c``: the token-by-token
  recurrence h_t = a_t h_{t-1} + B_t x_t^T, y_t = C_t^T h_t (+ D x_t), in fp64
  (Structured State Space Duality, "The recurrence as one matrix").
* :mod:`oracle.brute` -- numpy fp64: the materialised lower-triangular matrix
  M of the same page and section, and the masked-attention form of the
  scalar case.  It pins the recurrence on tiny inputs.
* :func:`recurrence_bwd` -- the C library's reverse mode of the same
  recurrence (the gradients of sum y*dy + sum final_state*dfinal), pinned by
  central finite differences of the dense form of :mod:`oracle.brute`.
"""
import ctypes
import os
import threading

import numpy as np

from . import build as _build

_lib = None
_lock = threading.Lock()

A_SCALAR = 0
A_DIAGONAL = 1


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            lib.ssd_oracle_fwd.restype = ctypes.c_int
            lib.ssd_oracle_fwd.argtypes = (
                [ctypes.c_int64] * 6 + [ctypes.c_int]
                + [ctypes.c_void_p] * 7
                + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]
                + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int])
            lib.ssd_oracle_bwd.restype = ctypes.c_int
            lib.ssd_oracle_bwd.argtypes = (
                [ctypes.c_int64] * 6 + [ctypes.c_int]
                + [ctypes.c_void_p] * 16 + [ctypes.c_int, ctypes.c_int])
            lib.ssd_oracle_threads.restype = ctypes.c_int
            lib.ssd_oracle_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _f32(a):
    """Host fp32 contiguous copy (bf16 values are exact in fp32)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def threads_used(nthreads=None):
    """Number of OpenMP threads the oracle runs with for this request."""
    return _load().ssd_oracle_threads(int(nthreads or 0))


def recurrence(x, dt, A, B, C, D=None, init_state=None, streams=None, t_end=None,
               nthreads=None, plant=0):
    """Token-by-token fp64 recurrence.

    Shapes: x (b,T,H,P), dt (b,T,H), A (H) scalar or (H,N) diagonal,
    B and C (b,T,G,N), D (H) or None, init_state (b,H,N,P) or None.

    With ``streams=None`` returns ``(y, final_state)`` with y (b,T,H,P) and
    final_state (b,H,N,P), both fp64.  With a list of stream ids
    (``bi*H + h``) returns y (n_streams, t_end, P) and final_state
    (n_streams, N, P) for those streams only; ``t_end`` truncates the
    sequence (the state returned is the state after token ``t_end - 1``).
    """
    x, dt, A, B, C = (_f32(v) for v in (x, dt, A, B, C))
    D, init_state = _f32(D), _f32(init_state)
    nb, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    a_mode = A_SCALAR if A.ndim == 1 else A_DIAGONAL
    assert dt.shape == (nb, T, H) and B.shape == C.shape == (nb, T, G, N)
    assert A.shape == ((H,) if a_mode == A_SCALAR else (H, N))
    if D is not None:
        assert D.shape == (H,)
    if init_state is not None:
        assert init_state.shape == (nb, H, N, P)
    t_end = T if t_end is None else int(t_end)
    sel = None
    if streams is not None:
        sel = np.ascontiguousarray(np.asarray(streams, dtype=np.int64))
        ns = sel.shape[0]
    else:
        ns = nb * H
    y = np.zeros((ns, t_end, P), dtype=np.float64)
    fin = np.zeros((ns, N, P), dtype=np.float64)
    rc = _load().ssd_oracle_fwd(
        nb, T, H, P, N, G, a_mode,
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
        _ptr(sel), ns, t_end, _ptr(y), _ptr(fin), int(nthreads or 0), int(plant))
    if rc != 0:
        raise ValueError("ssd_oracle_fwd rejected its arguments (status %d)" % rc)
    if streams is None:
        y = y.reshape(nb, H, t_end, P).transpose(0, 2, 1, 3).copy()
        fin = fin.reshape(nb, H, N, P)
    return y, fin


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def recurrence_bwd(x, dt, A, B, C, D=None, init_state=None, dy=None, dfinal=None, nthreads=None, plant=0):
    """fp64 gradients of L = sum y*dy + sum final_state*dfinal (the reverse mode of the recurrence).

    Inputs as for :func:`recurrence` (whole tensors), ``dy`` (b,T,H,P) and ``dfinal``
    (b,H,N,P) or None.  Returns a dict with dx, ddt, dA, dB, dC, dD (None without D) and
    dinit, fp64, in the layouts of the corresponding inputs.
    """
    x, dt, A, B, C = (_f32(v) for v in (x, dt, A, B, C))
    D, init_state = _f32(D), _f32(init_state)
    dy, dfinal = _f64(dy), _f64(dfinal)
    nb, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    a_mode = A_SCALAR if A.ndim == 1 else A_DIAGONAL
    assert dy is not None and dy.shape == x.shape
    if dfinal is not None:
        assert dfinal.shape == (nb, H, N, P)
    out = dict(dx=np.zeros((nb, T, H, P)), ddt=np.zeros((nb, T, H)), dA=np.zeros(A.shape),
               dB=np.zeros((nb, T, G, N)), dC=np.zeros((nb, T, G, N)),
               dD=np.zeros((H,)) if D is not None else None, dinit=np.zeros((nb, H, N, P)))
    rc = _load().ssd_oracle_bwd(
        nb, T, H, P, N, G, a_mode,
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state), _ptr(dy), _ptr(dfinal),
        _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
        _ptr(out["dD"]), _ptr(out["dinit"]), int(nthreads or 0), int(plant))
    if rc != 0:
        raise ValueError("ssd_oracle_bwd rejected its arguments (status %d)" % rc)
    return out
