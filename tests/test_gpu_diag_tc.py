"""GPU parity of the diagonal-A tcgen05 path (through the C ABI) against the fp64 oracle.

The kernel splits every decay exp(A_n (Dt_i - Dt_j)) at a reference token
between i and j, so that the fp16 operands carry factors <= 1; the pairs inside
one 16-token group are summed in fp32 on the CUDA cores, with one exponential
per term when the split factors could leave fp32 range.  These cases cover:
ragged lengths around the 128-token block and the 16-token group, several
B/C groups, D and init_state present or absent, more sequences than SMs (the
persistent loop over sequences), large decays that force the direct form, and
per-(batch, head) worst cases.  Tolerance: relative L2 2e-3 (bf16 io).
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_sequence_mixing_fwd_b300 as ssd
from ssd_sequence_mixing_fwd_b300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3
HEAD_TOL = 4e-3


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def run_tc(inp, w, dev, drop_D=False):
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    if drop_D:
        d["D"] = None
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, a_mode="diagonal", path="tcgen05")
    ws = torch.empty(ssd.ssd_fwd_workspace_size(dims), device=dev, dtype=torch.uint8)
    y, fin = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk_Q=w.Q,
                         path="tcgen05", workspace=ws)
    st = ssd.ssd_check_device_status(ws)
    assert st == ssd.SSD_OK, ssd.ssd_status_string(st)
    return y.float().cpu().numpy(), fin.cpu().numpy()


def check(w, inp, y, fin, drop_D=False):
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                               None if drop_D else inp["D"], inp["init_state"])
    assert np.isfinite(y).all() and np.isfinite(fin).all()
    e_y, e_f = rel(y, yr), rel(fin, fr)
    assert e_y <= TOL, "y relL2 %.3g" % e_y
    assert e_f <= TOL, "final_state relL2 %.3g" % e_f
    worst = max(rel(y[bi, :, h], yr[bi, :, h]) for bi in range(w.b) for h in range(w.H))
    assert worst <= HEAD_TOL, "worst head %.3g" % worst
    return e_y


CASES = [
    ("T1", Workload("t", b=1, T=1, H=2, P=64, N=64, G=1, Q=64, a_mode="diagonal", D="normal",
                    init_std=0.3, seed=601)),
    ("T15_group_tail", Workload("t", b=2, T=15, H=2, P=64, N=64, G=2, Q=64, a_mode="diagonal",
                                D="none", init_std=0.2, seed=602)),
    ("T128_one_block", Workload("t", b=1, T=128, H=4, P=64, N=64, G=1, Q=128, a_mode="diagonal",
                                D="normal", seed=603)),
    ("T129", Workload("t", b=2, T=129, H=4, P=64, N=64, G=4, Q=64, a_mode="diagonal", D="none",
                      init_std=0.1, seed=604)),
    ("T1000_G2", Workload("t", b=2, T=1000, H=6, P=64, N=64, G=2, Q=256, a_mode="diagonal",
                          D="normal", init_std=0.1, seed=605)),
    ("more_sequences_than_SMs", Workload("t", b=5, T=200, H=32, P=64, N=64, G=1, Q=64,
                                         a_mode="diagonal", D="normal", init_std=0.1, seed=606)),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_diagonal_tcgen05_small(name, w, cuda_device):
    assert ssd.ssd_fwd_path(ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, a_mode="diagonal")) == "tcgen05"
    inp = make_inputs(w)
    y, fin = run_tc(inp, w, cuda_device)
    check(w, inp, y, fin)
    if w.D != "none":
        y0, f0 = run_tc(inp, w, cuda_device, drop_D=True)
        check(w, inp, y0, f0, drop_D=True)


@pytest.mark.parametrize("dt_scale", [0.05, 4.0, 25.0], ids=["small_decay", "large_decay", "direct_groups"])
def test_diagonal_tcgen05_decay_range(dt_scale, cuda_device):
    # dt x 25 puts |A| x (half a group's Dt range) beyond the split's fp32 range for most
    # groups, so their in-group pairs take the direct form; dt x 0.05 keeps the state long-lived.
    w = Workload("t", b=2, T=300, H=4, P=64, N=64, G=1, Q=128, a_mode="diagonal", D="normal",
                 init_std=0.1, seed=611)
    inp = make_inputs(w)
    inp["dt"] = inp["dt"] * dt_scale
    y, fin = run_tc(inp, w, cuda_device)
    check(w, inp, y, fin)


def test_diagonal_workload_on_tcgen05_matches_generic(cuda_device):
    """The full diagonal-A workload: tcgen05 against the oracle on the whole tensor, and
    against the fp32 generic path."""
    w = WORKLOADS["diag_a"]
    assert ssd.ssd_fwd_path(ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, a_mode="diagonal")) == "tcgen05"
    inp = make_inputs(w)
    y, fin = run_tc(inp, w, cuda_device)
    check(w, inp, y, fin)
    d = {k: (None if v is None else v.to(cuda_device)) for k, v in inp.items()}
    yg, fg = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk_Q=w.Q,
                         path="generic", check=True)
    assert rel(y, yg.float().cpu().numpy()) < 3e-3
