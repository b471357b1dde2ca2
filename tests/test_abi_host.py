"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The library must load, export every function include/ssd.h declares, and
reject bad arguments before touching the GPU.
"""
import ctypes
import os
import re

import pytest

import ssd_sequence_mixing_fwd_b300 as ssd
from ssd_sequence_mixing_fwd_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ssd.load_library()


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            names += re.findall(r"^SSD_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "ssd_fwd" in names and len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    for n in ssd.EXPORTED:
        assert n in names


def test_abi_version_and_status_strings(lib):
    assert ssd.ssd_abi_version() == 1
    for st in range(0, 8):
        assert isinstance(ssd.ssd_status_string(st), str)
    assert ssd.ssd_status_string(99) == "unknown status"


def dims(**kw):
    base = dict(b=2, T=1000, H=4, P=64, N=128, G=2, Q=128)
    base.update(kw)
    return ssd.make_dims(**base)


def test_workspace_size_matches_layout(lib):
    d = dims()
    n = ssd.ssd_fwd_workspace_size(dims(path="generic"))
    nc = (1000 + 127) // 128
    states = 2 * 4 * nc * 128 * 64 * 4
    assert n >= states and n < states + 4096 + 2 * 4 * nc * 4 + 256
    assert ssd.ssd_fwd_workspace_size(d) > 0


@pytest.mark.parametrize("bad", [
    dict(H=3, G=2),          # H % G != 0
    dict(Q=96),              # chunk length not supported
    dict(Q=0),
    dict(T=-1),
    dict(b=-2),
    dict(P=0),
    dict(N=0),
    dict(G=0),
])
def test_invalid_dims_rejected(lib, bad):
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_fwd_workspace_size(dims(**bad))
    assert e.value.status == ssd.SSD_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(P=48), dict(P=512), dict(N=300), dict(N=256, P=128)])
def test_unsupported_dims_rejected(lib, bad):
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_fwd_workspace_size(dims(**bad))
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED


def test_bad_mode_values_rejected(lib):
    for field, val in (("a_mode", 5), ("io_dtype", 9), ("path", 7), ("reserved", 1)):
        d = dims()
        setattr(d, field, val)
        n = ctypes.c_size_t(0)
        assert lib.ssd_fwd_workspace_size(ctypes.byref(d), ctypes.byref(n)) == ssd.SSD_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected_before_any_launch(lib):
    d = dims(path="generic")
    ws = ctypes.c_void_p(1 << 20)
    args = [ctypes.c_void_p((1 << 21) + 4096 * i) for i in range(9)]
    # required pointer missing
    a = list(args)
    a[0] = None
    assert lib.ssd_fwd(ctypes.byref(d), *a, ws, 1 << 40, None) == ssd.SSD_ERR_INVALID_ARG
    # misaligned x
    a = list(args)
    a[0] = ctypes.c_void_p((1 << 21) + 2)
    assert lib.ssd_fwd(ctypes.byref(d), *a, ws, 1 << 40, None) == ssd.SSD_ERR_ALIGNMENT
    # workspace too small / missing
    assert lib.ssd_fwd(ctypes.byref(d), *args, ws, 16, None) == ssd.SSD_ERR_WORKSPACE
    assert lib.ssd_fwd(ctypes.byref(d), *args, None, 1 << 40, None) == ssd.SSD_ERR_WORKSPACE
    # y aliasing x
    a = list(args)
    a[7] = a[0]
    assert lib.ssd_fwd(ctypes.byref(d), *a, ws, 1 << 40, None) == ssd.SSD_ERR_INVALID_ARG


def test_path_query(lib):
    assert ssd.ssd_fwd_path(dims(path="generic")) == "generic"
    assert ssd.ssd_fwd_path(dims(dtype="f32")) in ("generic", "tcgen05")


def test_diagonal_path_selection(lib):
    # diagonal A runs on tcgen05 for bf16 io with N = P = 64 (any Q, G, T); otherwise generic
    assert ssd.ssd_fwd_path(dims(a_mode="diagonal", N=64)) == "tcgen05"
    assert ssd.ssd_fwd_path(dims(a_mode="diagonal", N=64, Q=64, G=1, T=1)) == "tcgen05"
    assert ssd.ssd_fwd_path(dims(a_mode="diagonal", N=128)) == "generic"
    assert ssd.ssd_fwd_path(dims(a_mode="diagonal", N=64, P=32)) == "generic"
    assert ssd.ssd_fwd_path(dims(a_mode="diagonal", N=64, dtype="f32")) == "generic"
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_fwd_workspace_size(dims(a_mode="diagonal", N=128, path="tcgen05"))
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    # its workspace is the status block alone
    assert ssd.ssd_fwd_workspace_size(dims(a_mode="diagonal", N=64, path="tcgen05")) == 256


@pytest.mark.parametrize("big", [dict(H=70000, G=70000), dict(b=70000)], ids=["H_over_grid_y", "b_over_grid_z"])
def test_dims_beyond_launch_limits_rejected_before_enqueue(lib, big):
    # The generic path's grids put H and b on grid dimensions y and z (at most 65535 each):
    # such dims are refused at validation, before anything is enqueued.
    for a_mode in ("scalar", "diagonal"):
        d = dims(path="generic", a_mode=a_mode, **big)
        with pytest.raises(ssd.SSDError) as e:
            ssd.ssd_fwd_workspace_size(d)
        assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    # diagonal A at N = 128 has no tcgen05 path, so AUTO has nothing to fall back to either
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_fwd_workspace_size(dims(a_mode="diagonal", **big))
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    # and ssd_fwd itself returns the same status without touching the (fake) device pointers
    d = dims(path="generic", **big)
    args = [ctypes.c_void_p((1 << 21) + 4096 * i) for i in range(9)]
    assert lib.ssd_fwd(ctypes.byref(d), *args, ctypes.c_void_p(1 << 20), 1 << 40, None) == ssd.SSD_ERR_UNSUPPORTED


def test_fused_path_index_limit(lib):
    # blocks x b x H must stay below 2^31 on the fused path (32-bit item and head numbers)
    d = dims(b=64, T=1 << 24, H=4096, G=4096, path="tcgen05")
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_fwd_workspace_size(d)
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED


def test_scan_and_decode_reject_bad_arguments_before_any_launch(lib):
    args = [ctypes.c_void_p((1 << 21) + 4096 * i) for i in range(9)]
    # decode: exactly one token, and a state
    d = dims(T=5)
    assert lib.ssd_decode_step(ctypes.byref(d), *args[:6], args[6], args[7], None) == ssd.SSD_ERR_INVALID_ARG
    d = dims(T=1)
    assert lib.ssd_decode_step(ctypes.byref(d), *args[:6], None, args[7], None) == ssd.SSD_ERR_INVALID_ARG
    # scan: no path selection, aligned pointers, invalid dims
    assert lib.ssd_scan(ctypes.byref(dims(path="generic")), *args, None) == ssd.SSD_ERR_INVALID_ARG
    a = list(args)
    a[0] = ctypes.c_void_p((1 << 21) + 1)                # odd address for bf16 x
    assert lib.ssd_scan(ctypes.byref(dims()), *a, None) == ssd.SSD_ERR_ALIGNMENT
    a = list(args)
    a[1] = ctypes.c_void_p((1 << 21) + 4096 + 2)         # dt not 4-byte aligned
    assert lib.ssd_scan(ctypes.byref(dims()), *a, None) == ssd.SSD_ERR_ALIGNMENT
    assert lib.ssd_scan(ctypes.byref(dims(Q=96)), *args, None) == ssd.SSD_ERR_INVALID_ARG


def test_backward_argument_checks_enqueue_nothing(lib):
    # every refusal happens before any CUDA call, so fake device addresses are safe here
    vp = lambda i: ctypes.c_void_p((1 << 21) + 4096 * i)
    args = [vp(i) for i in range(16)]
    d = dims(path="auto")
    ws_ok = (vp(40), 1 << 40)
    bad = list(args)
    bad[7] = None                                                    # dy missing
    assert lib.ssd_bwd(ctypes.byref(d), *bad, *ws_ok, None) == ssd.SSD_ERR_INVALID_ARG
    bad = list(args)
    bad[0] = ctypes.c_void_p((1 << 21) + 8)                          # x not 16-byte aligned
    assert lib.ssd_bwd(ctypes.byref(d), *bad, *ws_ok, None) == ssd.SSD_ERR_ALIGNMENT
    assert lib.ssd_bwd(ctypes.byref(d), *args, vp(40), 256, None) == ssd.SSD_ERR_WORKSPACE
    d2 = dims(path="tcgen05")
    assert lib.ssd_bwd(ctypes.byref(d2), *args, *ws_ok, None) == ssd.SSD_ERR_UNSUPPORTED
    d3 = dims(P=256, N=64)
    n = ctypes.c_size_t(0)
    assert lib.ssd_bwd_workspace_size(ctypes.byref(d3), ctypes.byref(n)) == ssd.SSD_ERR_UNSUPPORTED


def a256(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("kw", [dict(b=2, T=100, H=4, P=64, N=128), dict(b=1, T=64, H=2, P=64, N=64),
                                dict(b=3, T=1, H=6, P=64, N=128, G=3), dict(b=1, T=100, H=4, P=64, N=256),
                                dict(b=1, T=100, H=4, P=128, N=64), dict(b=2, T=70, H=2, P=128, N=128)])
def test_backward_workspace_of_the_chunked_path(lib, kw):
    # scalar A at P 64 / 128, N 64 / 128 / 256 on Q-token chunks (Q = 64; 32 at N 256 and at
    # P = N = 128): states and
    # adjoints (b H ceil(T/Q) N P fp32 each), the chunk sums, per-head dB and dC (b T H N fp32
    # each), C B^T per chunk and group (b ceil(T/Q) G Q Q fp32), every region rounded up to 256
    # bytes
    d = dims(path="auto", **kw)
    b, T, H, P, N = kw["b"], kw["T"], kw["H"], kw["P"], kw["N"]
    G = kw.get("G", 2)
    Q = 32 if N > 128 or (P == 128 and N == 128) else 64
    nc = -(-T // Q)
    want = 256 + a256(4 * b * H * nc) + a256(4 * b * H * nc * N * P) * 2 + a256(4 * b * T * H * N) * 2
    want += a256(4 * b * nc * G * Q * Q)
    assert ssd.ssd_bwd_workspace_size(d) == want


def test_backward_workspace_of_the_recurrence_path(lib):
    # diagonal A (and other head dims): checkpoints b H ceil(N / (1024 / P)) ceil(T / 8) x 4 KB and
    # three b T H N fp32 arrays plus the b T H P dx accumulator
    for kw in (dict(b=2, T=100, H=4, P=64, N=64, a_mode="diagonal"), dict(b=1, T=33, H=2, P=32, N=16)):
        d = dims(path="auto", **kw)
        b, T, H, P, N = kw["b"], kw["T"], kw["H"], kw["P"], kw["N"]
        nsl = -(-N // (1024 // P))
        want = 256 + a256(4 * b * H * nsl * -(-T // 8) * 1024)
        want = a256(want + 4 * b * T * H * N)
        want = a256(want + 4 * b * T * H * N)
        want = a256(want + 4 * b * T * H * N)
        want = a256(want + 4 * b * T * H * P)
        assert ssd.ssd_bwd_workspace_size(d) == want
