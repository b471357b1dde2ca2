"""B300 (sm_103a) forward pass of the SSD chunked scan (Mamba-2 sequence mixing).

A thin Python binding over the C ABI of ``libssd_b300.so`` (``include/ssd.h``):
argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; PyTorch supplies device memory and the current stream.
There is no CPU or PyTorch fallback: if the library is missing, the calls raise.

    y, final_state = ssd_fwd(x, dt, A, B, C, D=None, init_state=None, chunk_Q=256)

Shapes: x (b,T,H,P) bf16|fp32, dt (b,T,H) fp32, A (H) or (H,N) fp32,
B and C (b,T,G,N) same dtype as x, D (H) fp32, init_state (b,H,N,P) fp32.
"""
import ctypes
import os
import threading

from . import inputs  # noqa: F401  (seeded workload definitions)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd_b300.so")

# Mirrors of include/ssd.h
SSD_OK = 0
SSD_ERR_INVALID_ARG = 1
SSD_ERR_UNSUPPORTED = 2
SSD_ERR_ALIGNMENT = 3
SSD_ERR_WORKSPACE = 4
SSD_ERR_CUDA = 5
SSD_ERR_TIMEOUT = 6
SSD_ERR_DEVICE = 7
SSD_ERR_SCRATCH_LIMIT = 8
SSD_NOALLOC_SCRATCH_BYTES = 64 << 20
SSD_A_SCALAR = 0
SSD_A_DIAGONAL = 1
SSD_DTYPE_BF16 = 0
SSD_DTYPE_F32 = 1
SSD_PATH_AUTO = 0
SSD_PATH_GENERIC = 1
SSD_PATH_TCGEN05 = 2
_PATHS = {"auto": SSD_PATH_AUTO, "generic": SSD_PATH_GENERIC, "tcgen05": SSD_PATH_TCGEN05}

# Every symbol include/ssd.h declares.
EXPORTED = ("ssd_fwd_workspace_size", "ssd_fwd_path", "ssd_fwd", "ssd_check_device_status",
            "ssd_status_string", "ssd_abi_version", "ssd_debug_set_wait",
            "ssd_debug_set_kernel_events", "ssd_launch_count", "ssd_fwd_noalloc", "ssd_last_cuda_error",
            "ssd_scan", "ssd_decode_step", "ssd_bwd_workspace_size", "ssd_bwd")


class ssd_dims(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("P", ctypes.c_int64), ("N", ctypes.c_int64), ("G", ctypes.c_int64),
                ("Q", ctypes.c_int64), ("a_mode", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("path", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class SSDError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        msg = "%s: %s (status %d)" % (what or "ssd", ssd_status_string(status), status)
        if status == SSD_ERR_CUDA:
            msg += ": " + ssd_last_cuda_error()
        super().__init__(msg)


_lib = None
_lock = threading.Lock()


def load_library(path=LIB_PATH):
    """Load libssd_b300.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError("libssd_b300.so is not built (%s); run __graft_entry__.build()" % path)
            lib = ctypes.CDLL(path)
            vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
            P_dims = ctypes.POINTER(ssd_dims)
            lib.ssd_fwd_workspace_size.argtypes = [P_dims, ctypes.POINTER(sz)]
            lib.ssd_fwd_path.argtypes = [P_dims, ctypes.POINTER(ctypes.c_int32)]
            lib.ssd_fwd.argtypes = [P_dims] + [vp] * 9 + [vp, sz, vp]
            lib.ssd_fwd_noalloc.argtypes = [P_dims] + [vp] * 9 + [vp]
            lib.ssd_scan.argtypes = [P_dims] + [vp] * 9 + [vp]
            lib.ssd_decode_step.argtypes = [P_dims] + [vp] * 8 + [vp]
            lib.ssd_bwd_workspace_size.argtypes = [P_dims, ctypes.POINTER(sz)]
            lib.ssd_bwd.argtypes = [P_dims] + [vp] * 16 + [vp, sz, vp]
            lib.ssd_check_device_status.argtypes = [vp, sz, vp]
            lib.ssd_status_string.argtypes = [ctypes.c_int]
            lib.ssd_status_string.restype = ctypes.c_char_p
            lib.ssd_last_cuda_error.argtypes = []
            lib.ssd_last_cuda_error.restype = ctypes.c_char_p
            lib.ssd_abi_version.argtypes = []
            lib.ssd_debug_set_wait.argtypes = [i64, i64]
            lib.ssd_debug_set_kernel_events.argtypes = [vp, vp]
            lib.ssd_launch_count.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
            for name in ("ssd_fwd_workspace_size", "ssd_fwd_path", "ssd_fwd",
                         "ssd_check_device_status", "ssd_abi_version", "ssd_debug_set_wait",
                         "ssd_debug_set_kernel_events", "ssd_launch_count", "ssd_fwd_noalloc",
                         "ssd_scan", "ssd_decode_step", "ssd_bwd_workspace_size", "ssd_bwd"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def ssd_status_string(status):
    try:
        return load_library().ssd_status_string(int(status)).decode()
    except RuntimeError:
        return "status %d" % status


def ssd_last_cuda_error():
    """Text of the last CUDA error the library ran into."""
    try:
        return load_library().ssd_last_cuda_error().decode()
    except RuntimeError:
        return "library not loaded"


def ssd_abi_version():
    return load_library().ssd_abi_version()


def make_dims(b, T, H, P, N, G, Q, a_mode="scalar", dtype="bf16", path="auto"):
    return ssd_dims(b, T, H, P, N, G, Q,
                    SSD_A_SCALAR if a_mode == "scalar" else SSD_A_DIAGONAL,
                    SSD_DTYPE_BF16 if dtype == "bf16" else SSD_DTYPE_F32,
                    _PATHS[path], 0)


def ssd_fwd_workspace_size(dims):
    n = ctypes.c_size_t(0)
    st = load_library().ssd_fwd_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    if st != SSD_OK:
        raise SSDError(st, "ssd_fwd_workspace_size")
    return n.value


def ssd_fwd_path(dims):
    out = ctypes.c_int32(0)
    st = load_library().ssd_fwd_path(ctypes.byref(dims), ctypes.byref(out))
    if st != SSD_OK:
        raise SSDError(st, "ssd_fwd_path")
    return {SSD_PATH_GENERIC: "generic", SSD_PATH_TCGEN05: "tcgen05"}[out.value]


def ssd_check_device_status(workspace, stream=None):
    """Synchronise ``stream`` and return (and clear) the workspace's device status."""
    import torch
    s = torch.cuda.current_stream(workspace.device) if stream is None else stream
    return load_library().ssd_check_device_status(
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), ctypes.c_void_p(s.cuda_stream))


def ssd_debug_set_wait(spin_limit=0, withhold_chunk=-1):
    return load_library().ssd_debug_set_wait(int(spin_limit), int(withhold_chunk))


def ssd_debug_set_kernel_events(start_event=None, stop_event=None):
    """Bracket the dominant kernel of later calls with these torch.cuda.Events."""
    a = None if start_event is None else ctypes.c_void_p(start_event.cuda_event)
    b = None if stop_event is None else ctypes.c_void_p(stop_event.cuda_event)
    return load_library().ssd_debug_set_kernel_events(a, b)


def ssd_launch_count():
    n = ctypes.c_uint64(0)
    load_library().ssd_launch_count(ctypes.byref(n))
    return n.value


_NO_WORKSPACE = object()     # marshal without a workspace (entry points that take none)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _marshal(x, dt, A, B, C, D, init_state, chunk_Q, return_final_state, path, y, final_state,
             workspace, stream):
    """Checks the tensors, allocates missing outputs, and builds the C ABI arguments."""
    import torch
    for name, t in (("x", x), ("dt", dt), ("A", A), ("B", B), ("C", C), ("D", D),
                    ("init_state", init_state)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if x.dtype not in (torch.bfloat16, torch.float32) or B.dtype != x.dtype or C.dtype != x.dtype:
        raise ValueError("x, B, C must share dtype bf16 or fp32")
    for name, t in (("dt", dt), ("A", A), ("D", D), ("init_state", init_state)):
        if t is not None and t.dtype != torch.float32:
            raise ValueError("%s must be float32" % name)
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dims = make_dims(b, T, H, P, N, G, chunk_Q, "scalar" if A.dim() == 1 else "diagonal",
                     "bf16" if x.dtype == torch.bfloat16 else "f32", path)
    if tuple(dt.shape) != (b, T, H) or tuple(B.shape) != tuple(C.shape) or B.shape[:2] != x.shape[:2]:
        raise ValueError("shape mismatch among x, dt, B, C")
    if tuple(A.shape) not in ((H,), (H, N)):
        raise ValueError("A must be (H) or (H,N)")
    if D is not None and tuple(D.shape) != (H,):
        raise ValueError("D must be (H)")
    if init_state is not None and tuple(init_state.shape) != (b, H, N, P):
        raise ValueError("init_state must be (b,H,N,P)")
    dev = x.device
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, N, P), device=dev, dtype=torch.float32)
    if workspace is _NO_WORKSPACE:
        workspace = None
    elif workspace is None:
        workspace = torch.empty(max(ssd_fwd_workspace_size(dims), 256), device=dev, dtype=torch.uint8)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    args = (ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
            _ptr(y), _ptr(final_state), _ptr(workspace), 0 if workspace is None else workspace.numel(),
            ctypes.c_void_p(s.cuda_stream))
    return dims, args, y, final_state, workspace, s


def ssd_fwd(x, dt, A, B, C, D=None, init_state=None, chunk_Q=256, return_final_state=True,
            path="auto", y=None, final_state=None, workspace=None, stream=None, check=False):
    """SSD chunked-scan forward on the GPU.  Returns ``(y, final_state)``.

    ``y``, ``final_state`` and ``workspace`` may be passed preallocated
    (workspace: uint8 CUDA tensor of at least ``ssd_fwd_workspace_size``
    bytes).

    The call is asynchronous.  Errors the kernels find on the device -- a
    bounded wait between blocks that ran out (SSD_ERR_TIMEOUT; the kernel then
    continues with a zero state) or an operand outside the fused path's fp16
    range (SSD_ERR_DEVICE) -- leave y and final_state invalid WITHOUT raising,
    unless ``check=True`` (which synchronises and raises) or the caller reads
    the status with ``ssd_check_device_status(workspace)`` afterwards.
    """
    dims, args, y, final_state, workspace, s = _marshal(
        x, dt, A, B, C, D, init_state, chunk_Q, return_final_state, path, y, final_state, workspace, stream)
    st = load_library().ssd_fwd(*args)
    if st != SSD_OK:
        raise SSDError(st, "ssd_fwd")
    if check:
        st = ssd_check_device_status(workspace, s)
        if st != SSD_OK:
            raise SSDError(st, "ssd_fwd (device)")
    return y, final_state


def fwd(x, dt, A, B, C, D=None, init_state=None, chunk=256, return_final_state=True, **kw):
    """``ssd_fwd`` under its short name: ``(y, final_state)`` for chunk length ``chunk``
    (``final_state`` is None unless ``return_final_state``).  Raises :class:`SSDError`."""
    return ssd_fwd(x, dt, A, B, C, D, init_state, chunk_Q=chunk, return_final_state=return_final_state, **kw)


def ssd_scan(x, dt, A, B, C, D=None, init_state=None, return_final_state=True, y=None, final_state=None,
             stream=None):
    """The same map as :func:`ssd_fwd`, evaluated by the linear recurrence token by token on CUDA
    cores (no workspace).  Returns ``(y, final_state)``."""
    dims, args, y, final_state, _, s = _marshal(
        x, dt, A, B, C, D, init_state, 256, return_final_state, "auto", y, final_state, _NO_WORKSPACE, stream)
    st = load_library().ssd_scan(*(args[:10] + args[12:]))
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan")
    return y, final_state


def ssd_decode_step(x, dt, A, B, C, D, state, y=None, stream=None):
    """One generated token: x (b,1,H,P), dt (b,1,H), B and C (b,1,G,N); ``state`` (b,H,N,P) fp32 is
    updated in place.  Returns y (b,1,H,P)."""
    import torch
    if state is None or state.dtype != torch.float32 or not state.is_cuda or not state.is_contiguous():
        raise ValueError("state must be a contiguous float32 CUDA tensor")
    if x.shape[1] != 1:
        raise ValueError("a decode step takes one token (x of shape (b,1,H,P))")
    dims, args, y, _, _, s = _marshal(
        x, dt, A, B, C, D, state, 256, False, "auto", y, None, _NO_WORKSPACE, stream)
    st = load_library().ssd_decode_step(args[0], *args[1:7], _ptr(state), args[8], args[12])
    if st != SSD_OK:
        raise SSDError(st, "ssd_decode_step")
    return y


def ssd_bwd_workspace_size(dims):
    n = ctypes.c_size_t(0)
    st = load_library().ssd_bwd_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    if st != SSD_OK:
        raise SSDError(st, "ssd_bwd_workspace_size")
    return n.value


def ssd_bwd(x, dt, A, B, C, D=None, init_state=None, dy=None, dfinal=None, want_dD=True, want_dinit=True,
            workspace=None, stream=None, path="auto"):
    """Gradients of ``sum y*dy + sum final_state*dfinal`` for the map :func:`ssd_fwd` computes.

    Returns a dict with dx (like x), ddt (b,T,H) fp32, dA (like A) fp32, dB and dC (like B) in
    the io dtype, dD (H) fp32 (None unless ``want_dD``) and dinit (b,H,N,P) fp32 (None unless
    ``want_dinit``).  ``dy`` has x's shape and dtype; ``dfinal`` is (b,H,N,P) fp32 or None.
    ``path``: "auto" (the chunked path where it applies) or "generic" (the token recurrence).
    Asynchronous on the current stream."""
    import torch
    if dy is None or dy.shape != x.shape or dy.dtype != x.dtype or not dy.is_cuda or not dy.is_contiguous():
        raise ValueError("dy must be a contiguous CUDA tensor with x's shape and dtype")
    if dfinal is not None and (dfinal.dtype != torch.float32 or not dfinal.is_cuda or not dfinal.is_contiguous()):
        raise ValueError("dfinal must be a contiguous float32 CUDA tensor")
    dims, args, _, _, _, s = _marshal(x, dt, A, B, C, D, init_state, 256, False, path, x, None,
                                      _NO_WORKSPACE, stream)
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if dfinal is not None and tuple(dfinal.shape) != (b, H, N, P):
        raise ValueError("dfinal must be (b,H,N,P)")
    dev = x.device
    out = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dA=torch.empty_like(A),
               dB=torch.empty_like(B), dC=torch.empty_like(C),
               dD=torch.empty((H,), device=dev, dtype=torch.float32) if want_dD else None,
               dinit=torch.empty((b, H, N, P), device=dev, dtype=torch.float32) if want_dinit else None)
    if workspace is None:
        workspace = torch.empty(max(ssd_bwd_workspace_size(dims), 256), device=dev, dtype=torch.uint8)
    st = load_library().ssd_bwd(args[0], *args[1:8], _ptr(dy), _ptr(dfinal), _ptr(out["dx"]), _ptr(out["ddt"]),
                                _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                                _ptr(out["dinit"]), _ptr(workspace), workspace.numel(),
                                ctypes.c_void_p(s.cuda_stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_bwd")
    return out


class PreparedCall:
    """One ssd_fwd call with its arguments checked and marshalled once.

    For loops that run the same problem on the same buffers (serving steps,
    benchmarks): each call of the object only crosses the C ABI, so the GPU
    is not left idle while Python rebuilds arguments.  The tensors passed in
    (and the outputs/workspace it allocates) must stay alive and in place;
    their contents may change between calls.

        run = PreparedCall(x, dt, A, B, C, D, chunk_Q=256)
        y, final_state = run()
    """

    def __init__(self, x, dt, A, B, C, D=None, init_state=None, chunk_Q=256, return_final_state=True,
                 path="auto", y=None, final_state=None, workspace=None, stream=None):
        self._keep = (x, dt, A, B, C, D, init_state)
        (self.dims, self._args, self.y, self.final_state, self.workspace,
         self.stream) = _marshal(x, dt, A, B, C, D, init_state, chunk_Q, return_final_state, path, y,
                                 final_state, workspace, stream)
        self._fn = load_library().ssd_fwd

    def __call__(self):
        st = self._fn(*self._args)
        if st != SSD_OK:
            raise SSDError(st, "ssd_fwd")
        return self.y, self.final_state

    def check(self):
        """Synchronise the stream and raise on a device-side error of the last call."""
        st = ssd_check_device_status(self.workspace, self.stream)
        if st != SSD_OK:
            raise SSDError(st, "ssd_fwd (device)")
