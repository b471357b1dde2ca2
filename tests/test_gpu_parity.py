"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (whole-tensor relative L2 error, fp64 on the host):
  bf16 x/B/C: 2e-3 on y and on final_state; fp32 x/B/C: 1e-5.
Every bf16 case is also run with D absent, so the skip term cannot hide an
error in the SSM part; the per-(batch, head) worst case is bounded too.
Full-size workloads are compared on the whole tensor as well.
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_sequence_mixing_fwd_b300 as ssd
from ssd_sequence_mixing_fwd_b300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f32": 1e-5}
HEAD_TOL = {"bf16": 4e-3, "f32": 3e-5}


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def available_paths(w):
    out = []
    for path in ("generic", "tcgen05"):
        try:
            ssd.ssd_fwd_path(ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, w.a_mode, w.dtype, path))
            out.append(path)
        except ssd.SSDError:
            pass
    return out


def gpu_run(inp, Q, path="auto", drop_D=False, want_final=True):
    dev = torch.device("cuda:0")
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    if drop_D:
        d["D"] = None
    y, fin = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                         chunk_Q=Q, path=path, return_final_state=want_final, check=True)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), (None if fin is None else fin.cpu().numpy())


def compare(w, inp, y, fin, streams=None, drop_D=False, tol=None):
    tol = TOL[w.dtype] if tol is None else tol
    D = None if drop_D else inp["D"]
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D,
                               inp["init_state"], streams=streams)
    H = w.H
    if streams is None:
        yg, fg = y, fin
        per_head = [rel(yg[bi, :, h], yr[bi, :, h]) for bi in range(w.b) for h in range(H)]
    else:
        yg = np.stack([y[s // H, :, s % H] for s in streams])
        fg = None if fin is None else np.stack([fin[s // H, s % H] for s in streams])
        per_head = [rel(yg[i], yr[i]) for i in range(len(streams))]
    e_y = rel(yg, yr)
    assert np.isfinite(yg).all()
    assert e_y <= tol, "y relL2 %.3g > %.3g" % (e_y, tol)
    assert max(per_head) <= HEAD_TOL[w.dtype] * (tol / TOL[w.dtype]), "worst head %.3g" % max(per_head)
    if fg is not None:
        e_f = rel(fg, fr)
        assert e_f <= tol, "final_state relL2 %.3g > %.3g" % (e_f, tol)
    return e_y


SMALL = [
    # name, workload: several chunks and a ragged tail
    ("ragged_T1000_G2", Workload("t", b=2, T=1000, H=4, P=64, N=128, G=2, Q=128, D="normal",
                                 init_std=0.1, seed=11)),
    ("q256_T700", Workload("t", b=1, T=700, H=6, P=64, N=128, G=1, Q=256, D="normal", seed=12)),
    ("q64_N64", Workload("t", b=2, T=333, H=4, P=64, N=64, G=4, Q=64, D="none", seed=13)),
    ("n256_q128", Workload("t", b=1, T=520, H=8, P=64, N=256, G=8, Q=128, D="none", init_std=0.1,
                           seed=14)),
    ("diag_small", Workload("t", b=2, T=300, H=4, P=64, N=64, G=1, Q=64, a_mode="diagonal",
                            D="normal", init_std=0.1, seed=15)),
    ("f32_small", Workload("t", b=1, T=200, H=3, P=16, N=16, G=1, Q=64, dtype="f32", D="ones",
                           seed=16)),
    ("f32_P32_diag", Workload("t", b=1, T=150, H=2, P=32, N=8, G=2, Q=128, dtype="f32",
                              a_mode="diagonal", D="none", init_std=0.3, seed=17)),
]


@pytest.mark.parametrize("name,w", SMALL, ids=[s[0] for s in SMALL])
def test_small_cases_all_paths(name, w, cuda_device):
    inp = make_inputs(w)
    for path in available_paths(w):
        y, fin = gpu_run(inp, w.Q, path)
        compare(w, inp, y, fin)
        if w.D != "none" and w.dtype == "bf16":
            y0, f0 = gpu_run(inp, w.Q, path, drop_D=True)
            compare(w, inp, y0, f0, drop_D=True)


@pytest.mark.parametrize("dt_scale,dtype", [(1.0, "f32"), (1.0, "bf16"), (25.0, "bf16")],
                         ids=["f32_split_tiles", "bf16_split_tiles", "bf16_large_decay_direct_tiles"])
def test_diagonal_a_split_decay_tiles(dt_scale, dtype, cuda_device):
    # The generic diagonal-A output kernel splits each tile's decay e^{A_n (cum_i - cum_j)}
    # into a row and a column factor; a tile on the diagonal falls back to one exponential
    # per (i, j, n) when the factors would leave fp32 range (dt scaled up 25x forces that).
    # N = 50 puts the transposed factor buffer on a non-16-byte offset before its alignment.
    w = Workload("t", b=2, T=200, H=3, P=64, N=50, G=1, Q=128, a_mode="diagonal", dtype=dtype,
                 D="normal", init_std=0.1, seed=31)
    inp = make_inputs(w)
    inp["dt"] = inp["dt"] * dt_scale
    y, fin = gpu_run(inp, w.Q, "generic")
    compare(w, inp, y, fin)


@pytest.mark.parametrize("name", ["tiny_fp32", "mamba2_130m", "diag_a"])
def test_workload_full_parity(name, cuda_device):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    y, fin = gpu_run(inp, w.Q)
    compare(w, inp, y, fin)
    if w.D != "none" and w.dtype == "bf16":
        y0, f0 = gpu_run(inp, w.Q, drop_D=True)
        compare(w, inp, y0, f0, drop_D=True)


@pytest.mark.parametrize("name", ["mamba2_2p7b", "long_seq"])
def test_workload_full_size_whole_tensor(name, cuda_device):
    """Full-size call in the configuration the benchmark times, checked on every (batch, head)
    stream over the whole sequence against the oracle (with and without D), including the
    per-(batch, head) worst case."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    y, fin = gpu_run(inp, w.Q)
    compare(w, inp, y, fin)
    if w.D != "none":
        y0, f0 = gpu_run(inp, w.Q, drop_D=True)
        compare(w, inp, y0, f0, drop_D=True)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 129, 255, 257, 3 * 128 + 17])
def test_sequence_length_edges(T, cuda_device):
    w = Workload("t", b=2, T=T, H=4, P=64, N=128, G=2, Q=128, D="normal", init_std=0.2, seed=T)
    inp = make_inputs(w)
    for Q in (64, 128, 256):
        for path in available_paths(w.with_(Q=Q)):
            y, fin = gpu_run(inp, Q, path)
            compare(w, inp, y, fin)


def test_chunk_length_invariance(cuda_device):
    """The chunked algorithm is exact for every Q: all Q agree with the oracle and each other."""
    w = Workload("t", b=2, T=1024, H=4, P=64, N=128, G=1, Q=64, D="none", seed=21)
    inp = make_inputs(w)
    ys = {}
    for Q in (64, 128, 256):
        y, fin = gpu_run(inp, Q)
        compare(w, inp, y, fin)
        ys[Q] = y
    assert rel(ys[64], ys[256]) < 3e-3


def test_empty_problems(cuda_device):
    dev = cuda_device
    for b, T in ((0, 16), (2, 0)):
        x = torch.zeros((b, T, 4, 64), device=dev, dtype=torch.bfloat16)
        Bm = torch.zeros((b, T, 1, 128), device=dev, dtype=torch.bfloat16)
        dt = torch.zeros((b, T, 4), device=dev)
        A = -torch.ones(4, device=dev)
        h0 = torch.randn((b, 4, 128, 64), device=dev)
        y, fin = ssd.ssd_fwd(x, dt, A, Bm, Bm.clone(), None, h0, chunk_Q=128, check=True)
        assert y.shape == x.shape
        assert torch.equal(fin, h0)
        y, fin = ssd.ssd_fwd(x, dt, A, Bm, Bm.clone(), None, None, chunk_Q=128, check=True)
        assert fin.abs().sum().item() == 0


def test_closed_forms_through_gpu(cuda_device):
    """a == 1 and a == 0 (the oracle is pinned to both closed forms)."""
    w = Workload("t", b=1, T=600, H=4, P=64, N=128, G=1, Q=128, D="normal", seed=31)
    inp = make_inputs(w)
    inp1 = dict(inp, A=torch.zeros_like(inp["A"]))
    y, fin = gpu_run(inp1, w.Q)
    compare(w, inp1, y, fin)
    inp0 = dict(inp, A=torch.full_like(inp["A"], -1e4), dt=torch.ones_like(inp["dt"]))
    y, fin = gpu_run(inp0, w.Q)
    compare(w, inp0, y, fin)


def test_final_state_optional_and_init_state(cuda_device):
    w = Workload("t", b=2, T=400, H=4, P=64, N=128, G=2, Q=128, D="none", init_std=0.5, seed=41)
    inp = make_inputs(w)
    y, fin = gpu_run(inp, w.Q, want_final=False)
    assert fin is None
    compare(w, inp, y, None)


def test_split_sequence_composition_gpu(cuda_device):
    """fwd(x[:T1]) then fwd(x[T1:]) from its final state equals fwd(x)."""
    w = Workload("t", b=2, T=768, H=4, P=64, N=128, G=1, Q=128, D="normal", seed=51)
    inp = make_inputs(w)
    y, fin = gpu_run(inp, w.Q)
    T1 = 256
    first = {k: (v[:, :T1].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    y1, f1 = gpu_run(first, w.Q)
    second = {k: (v[:, T1:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    second["init_state"] = torch.from_numpy(f1)
    y2, f2 = gpu_run(second, w.Q)
    assert rel(np.concatenate([y1, y2], axis=1), y) < 3e-3
    assert rel(f2, fin) < 1e-3
    # each part against the oracle run over the whole sequence
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])
    assert rel(np.concatenate([y1, y2], axis=1), yr) <= 2e-3
    assert rel(f2, fr) <= 2e-3


def test_short_name_fwd_matches_ssd_fwd(cuda_device):
    # ssd.fwd is ssd_fwd under its short name: the same kernels, bit for bit
    w = Workload("t", b=1, T=300, H=4, P=64, N=128, G=2, Q=128, D="normal", init_std=0.1, seed=931)
    d = {k: (None if v is None else v.to(cuda_device)) for k, v in make_inputs(w).items()}
    y1, f1 = ssd.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk=w.Q)
    y2, f2 = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk_Q=w.Q)
    y3, f3 = ssd.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk=w.Q,
                     return_final_state=False)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2) and torch.equal(y1, y3) and f3 is None
