"""The linear form (ssd_scan) and the decode step (ssd_decode_step), through the C ABI.

ssd_scan evaluates the same map as ssd_fwd by the recurrence itself, token by
token (Structured State Space Duality, "The recurrence as one matrix"), so it
is checked against the same fp64 oracle and tolerances (relative L2 on the
whole tensor: 2e-3 for bf16 inputs, 1e-5 for fp32).  A decode step is the
T = 1 case with the state updated in place; a prompt run through ssd_fwd and
continued token by token must match the oracle run over the whole sequence.
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_sequence_mixing_fwd_b300 as ssd
from ssd_sequence_mixing_fwd_b300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f32": 1e-5}


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def _dev(inp, dev):
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


def check(w, inp, y, fin):
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])
    yg = y.float().cpu().numpy()
    assert np.isfinite(yg).all()
    assert rel(yg, yr) <= TOL[w.dtype], rel(yg, yr)
    assert rel(fin.cpu().numpy(), fr) <= TOL[w.dtype]
    per_head = [rel(yg[b, :, h], yr[b, :, h]) for b in range(w.b) for h in range(w.H)]
    assert max(per_head) <= 2 * TOL[w.dtype]


SMALL = [
    Workload("s1", b=2, T=300, H=4, P=64, N=128, G=2, Q=128, D="normal", init_std=0.1, seed=501),
    Workload("s2", b=1, T=77, H=3, P=16, N=16, G=1, Q=64, dtype="f32", D="ones", seed=502),
    Workload("s3", b=2, T=129, H=4, P=64, N=64, G=1, Q=64, a_mode="diagonal", D="none", init_std=0.2, seed=503),
    Workload("s4", b=1, T=200, H=2, P=32, N=8, G=2, Q=128, dtype="f32", a_mode="diagonal", D="normal",
             init_std=0.3, seed=504),
    Workload("s5", b=1, T=64, H=8, P=64, N=256, G=8, Q=128, D="none", init_std=0.1, seed=505),
    Workload("s6", b=1, T=33, H=2, P=256, N=64, G=1, Q=256, D="normal", seed=506),
    # bf16 with a 16-wide state at P 64 (the bench's state-16 comparison runs this configuration)
    Workload("s7", b=2, T=180, H=4, P=64, N=16, G=1, Q=64, D="normal", seed=507),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_scan_matches_oracle_small(w, cuda_device):
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    y, fin = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    torch.cuda.synchronize()
    check(w, inp, y, fin)


@pytest.mark.parametrize("name", ["tiny_fp32", "mamba2_130m", "diag_a", "mamba2_2p7b"])
def test_scan_matches_oracle_workloads(name, cuda_device):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    y, fin = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    torch.cuda.synchronize()
    check(w, inp, y, fin)


def test_scan_state_in_place(cuda_device):
    w = Workload("t", b=2, T=100, H=4, P=64, N=128, G=1, Q=128, D="normal", init_std=0.5, seed=511)
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    state = d["init_state"].clone()
    y, fin = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], state, final_state=state)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    check(w, inp, y, fin)


@pytest.mark.parametrize("w", [
    Workload("d1", b=2, T=300, H=8, P=64, N=128, G=1, Q=128, D="normal", init_std=0.1, seed=521),
    Workload("d2", b=1, T=200, H=4, P=64, N=64, G=2, Q=64, a_mode="diagonal", D="none", seed=522),
    Workload("d3", b=1, T=150, H=2, P=16, N=16, G=1, Q=64, dtype="f32", D="ones", seed=523),
], ids=["scalar_fused_prefill", "diagonal", "fp32"])
def test_prefill_then_decode_matches_whole_sequence(w, cuda_device):
    """ssd_fwd over a prompt, then one ssd_decode_step per further token from its final state."""
    inp = make_inputs(w)
    T0, K = w.T - 12, 12
    d = _dev(inp, cuda_device)
    pre = {k: (v[:, :T0].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    y0, state = ssd.ssd_fwd(pre["x"], pre["dt"], pre["A"], pre["B"], pre["C"], pre["D"], pre["init_state"],
                            chunk_Q=w.Q, check=True)
    ys = [y0]
    for t in range(T0, T0 + K):
        ys.append(ssd.ssd_decode_step(d["x"][:, t:t + 1].contiguous(), d["dt"][:, t:t + 1].contiguous(), d["A"],
                                      d["B"][:, t:t + 1].contiguous(), d["C"][:, t:t + 1].contiguous(), d["D"],
                                      state))
    torch.cuda.synchronize()
    check(w, inp, torch.cat(ys, dim=1), state)


def test_decode_step_rejects_more_than_one_token(cuda_device):
    w = Workload("t", b=1, T=2, H=2, P=64, N=128, G=1, Q=128, D="none", seed=531)
    d = _dev(make_inputs(w), cuda_device)
    state = torch.zeros((1, 2, 128, 64), device=cuda_device)
    with pytest.raises(ValueError):
        ssd.ssd_decode_step(d["x"], d["dt"], d["A"], d["B"], d["C"], None, state)
    lib = ssd.load_library()
    dims = ssd.make_dims(1, 2, 2, 64, 128, 1, 128)
    import ctypes
    fake = [ctypes.c_void_p(d[k].data_ptr()) for k in ("x", "dt", "A", "B", "C")]
    st = lib.ssd_decode_step(ctypes.byref(dims), *fake, None, ctypes.c_void_p(state.data_ptr()),
                             ctypes.c_void_p(state.data_ptr() + 4096), None)
    assert st == ssd.SSD_ERR_INVALID_ARG


@pytest.mark.parametrize("aligned", [True, False], ids=["one_token_kernel", "unaligned_state_fallback"])
@pytest.mark.parametrize("a_mode", ["scalar", "diagonal"])
def test_decode_steps_both_state_alignments(aligned, a_mode, cuda_device):
    """Decode steps on a 16-byte aligned state (the one-token kernel) and on a state that starts 4
    bytes into its buffer (the general kernel), against the oracle over the whole sequence."""
    w = Workload("t", b=3, T=20, H=4, P=32, N=64 if a_mode == "diagonal" else 48, G=2, Q=64, a_mode=a_mode,
                 D="normal", init_std=0.2, seed=541)
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    n = w.b * w.H * w.N * w.P
    buf = torch.empty(n + 4, device=cuda_device, dtype=torch.float32)
    state = buf[:n] if aligned else buf[1:n + 1]
    state.view(w.b, w.H, w.N, w.P).copy_(d["init_state"])
    st4 = state.view(w.b, w.H, w.N, w.P)
    ys = []
    for t in range(w.T):
        ys.append(ssd.ssd_decode_step(d["x"][:, t:t + 1].contiguous(), d["dt"][:, t:t + 1].contiguous(), d["A"],
                                      d["B"][:, t:t + 1].contiguous(), d["C"][:, t:t + 1].contiguous(), d["D"], st4))
    torch.cuda.synchronize()
    check(w, inp, torch.cat(ys, dim=1), st4)
