"""The allocation-free entry point ssd_fwd_noalloc, checked through the C ABI.

ssd_fwd_noalloc is for callers that may not allocate device memory
themselves (for example a plug-in whose host application owns the whole
device-memory budget, or a latency-bound loop where cudaMalloc's possible
device synchronisation is not allowed).  It uses a fixed scratch array inside
the library instead of a caller workspace.  These tests compare it with the
ordinary entry point ssd_fwd on three calls in a row, the last two of the
same shape with different inputs (the array keeps the previous call's
contents, so a call must not depend on them), and check that a problem too large for the array is refused before
any GPU work.  The file sorts last so that a stop-at-first-failure run has
already run every other test when it gets here.
"""
import ctypes

import numpy as np
import pytest
import torch

import ssd_sequence_mixing_fwd_b300 as ssd
from ssd_sequence_mixing_fwd_b300 import _build
from ssd_sequence_mixing_fwd_b300.inputs import Workload, make_inputs

TOL = 2e-3


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, w, d, y, fin, stream):
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, w.a_mode, w.dtype)
    return lib.ssd_fwd_noalloc(ctypes.byref(dims), _vp(d["x"]), _vp(d["dt"]), _vp(d["A"]), _vp(d["B"]),
                               _vp(d["C"]), _vp(d["D"]), _vp(d["init_state"]), _vp(y), _vp(fin),
                               ctypes.c_void_p(stream.cuda_stream))


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_noalloc_rejects_problem_larger_than_its_scratch():
    _build.build()
    lib = ssd.load_library()
    # 2.7B layer shape: chunk states alone are 335 MB > 64 MiB
    dims = ssd.make_dims(4, 8192, 80, 64, 128, 1, 256)
    fake = [ctypes.c_void_p((1 << 22) + 4096 * i) for i in range(9)]
    st = lib.ssd_fwd_noalloc(ctypes.byref(dims), *fake, None)
    assert st == ssd.SSD_ERR_SCRATCH_LIMIT
    assert "scratch" in ssd.ssd_status_string(st)


@pytest.mark.gpu
def test_noalloc_matches_ssd_fwd_on_calls_in_a_row(cuda_device):
    lib = ssd.load_library()
    stream = torch.cuda.current_stream(cuda_device)
    # the second and third calls have the same shape with different inputs: the array still
    # holds the second call's chunk states when the third one starts
    cases = [
        Workload("na1", b=2, T=1000, H=4, P=64, N=128, G=2, Q=128, D="normal", init_std=0.1, seed=901),
        Workload("na2", b=1, T=777, H=6, P=64, N=64, G=3, Q=256, a_mode="diagonal", D="none",
                 init_std=0.2, seed=902),
        Workload("na3", b=1, T=777, H=6, P=64, N=64, G=3, Q=256, a_mode="diagonal", D="none",
                 init_std=0.2, seed=903),
    ]
    for w in cases:
        d = {k: (None if v is None else v.to(cuda_device)) for k, v in make_inputs(w).items()}
        y_ref, f_ref = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                                   chunk_Q=w.Q, check=True)
        y = torch.full_like(d["x"], float("nan"))
        fin = torch.full((w.b, w.H, w.N, w.P), float("nan"), device=cuda_device)
        assert _noalloc(lib, w, d, y, fin, stream) == ssd.SSD_OK
        torch.cuda.synchronize(cuda_device)
        assert torch.isfinite(y.float()).all() and torch.isfinite(fin).all()
        assert _rel(y, y_ref) <= TOL
        assert _rel(fin, f_ref) <= TOL
