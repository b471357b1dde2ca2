"""GPU tests specific to the fused tcgen05 path (through the C ABI).

* failure detection: a block whose item withholds its state makes the next
  block's bounded wait run out; the call reports SSD_ERR_TIMEOUT through
  ssd_check_device_status, and the context stays usable (the next call is
  correct).  Nothing faults or hangs: the wait has an iteration limit.
* the fused path agrees with the generic CUDA-core path on the same inputs.
* heads-per-item edge: one head per B/C group (G == H).
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_sequence_mixing_fwd_b300 as ssd
from ssd_sequence_mixing_fwd_b300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _dev(inp, dev):
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


def _fused_ok(w):
    try:
        return ssd.ssd_fwd_path(ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, w.a_mode, w.dtype,
                                              "tcgen05")) == "tcgen05"
    except ssd.SSDError:
        return False


@pytest.mark.parametrize("N", [128, 256], ids=["n128_issuer_publishes", "n256_warps_publish"])
def test_withheld_state_reports_timeout_and_context_survives(N, cuda_device):
    # N = 128 publishes a block's state through the group's issuer warp; N = 256 has
    # every warp publish its own rows of each half: both must time out cleanly
    w = Workload("t", b=1, T=768, H=4, P=64, N=N, G=1, Q=128, D="none", seed=61)
    assert _fused_ok(w)
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q)
    ws = torch.empty(ssd.ssd_fwd_workspace_size(dims), device=cuda_device, dtype=torch.uint8)
    try:
        ssd.ssd_debug_set_wait(spin_limit=20000, withhold_chunk=2)
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], None, None, chunk_Q=w.Q, path="tcgen05",
                    workspace=ws)
        st = ssd.ssd_check_device_status(ws)
    finally:
        ssd.ssd_debug_set_wait(0, -1)
    assert st == ssd.SSD_ERR_TIMEOUT
    # the status word is cleared by the check, and the next call is correct
    assert ssd.ssd_check_device_status(ws) == ssd.SSD_OK
    y, fin = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], None, None, chunk_Q=w.Q, path="tcgen05",
                         workspace=ws, check=True)
    torch.cuda.synchronize()
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], None, None)
    assert rel(y.float().cpu().numpy(), yr) <= 2e-3
    assert rel(fin.cpu().numpy(), fr) <= 2e-3


@pytest.mark.parametrize("w", [
    Workload("t", b=3, T=1536, H=8, P=64, N=128, G=2, Q=256, D="normal", init_std=0.3, seed=71),
    Workload("t", b=1, T=640, H=3, P=64, N=128, G=3, Q=128, D="none", init_std=0.1, seed=72),
    Workload("t", b=2, T=130, H=10, P=64, N=128, G=1, Q=128, D="normal", seed=73),
    # 2 * 64 blocks * 2 head groups = 256 work items: several per CTA
    Workload("t", b=2, T=8192, H=16, P=64, N=128, G=2, Q=256, D="normal", init_std=0.1, seed=74),
    # odd heads per item (k = 5): consecutive items start on alternating math groups
    Workload("t", b=3, T=4000, H=10, P=64, N=128, G=2, Q=128, D="none", seed=75),
    # N = 256 (one math group, one C/B stage, two state accumulators): 4 heads per group
    Workload("t", b=1, T=1500, H=8, P=64, N=256, G=2, Q=128, D="normal", init_std=0.1, seed=76),
    # N = 256 with several items per CTA, k = 3 (dt by thread loads), Q = 256
    Workload("t", b=2, T=9000, H=6, P=64, N=256, G=2, Q=256, D="none", init_std=0.1, seed=77),
], ids=["k4_g2", "one_head_per_group", "k5_ragged130", "many_items_per_cta", "odd_k_many_items",
        "n256_k4", "n256_many_items_k3"])
def test_fused_matches_generic_and_oracle(w, cuda_device):
    assert _fused_ok(w)
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    out = {}
    for path in ("generic", "tcgen05"):
        y, fin = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk_Q=w.Q,
                             path=path, check=True)
        torch.cuda.synchronize()
        out[path] = (y.float().cpu().numpy(), fin.cpu().numpy())
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])
    for path, (y, fin) in out.items():
        assert rel(y, yr) <= 2e-3, path
        assert rel(fin, fr) <= 2e-3, path
    assert rel(out["tcgen05"][0], out["generic"][0]) <= 2e-3


def test_fused_repeated_calls_same_workspace(cuda_device):
    """The ticket and flags are reset by every call: back-to-back calls agree."""
    w = Workload("t", b=2, T=1024, H=8, P=64, N=128, G=1, Q=256, D="normal", seed=81)
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q)
    ws = torch.empty(ssd.ssd_fwd_workspace_size(dims), device=cuda_device, dtype=torch.uint8)
    ys = []
    for _ in range(3):
        y, _ = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, chunk_Q=w.Q, workspace=ws,
                           check=True)
        ys.append(y.clone())
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_prepared_call_matches_ssd_fwd(cuda_device):
    """PreparedCall marshals once; after the inputs change in place it still computes the new result."""
    w = Workload("t", b=2, T=512, H=8, P=64, N=128, G=1, Q=256, D="normal", seed=91)
    inp = make_inputs(w)
    d = _dev(inp, cuda_device)
    run = ssd.PreparedCall(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, chunk_Q=w.Q)
    y1, f1 = run()
    run.check()
    yr, fr = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, chunk_Q=w.Q, check=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, yr) and torch.equal(f1, fr)
    inp2 = make_inputs(w.with_(seed=92))
    for k in ("x", "dt", "B", "C"):
        d[k].copy_(inp2[k].to(cuda_device))
    y2, f2 = run()
    run.check()
    yo, fo = oracle.recurrence(inp2["x"], inp2["dt"], inp["A"], inp2["B"], inp2["C"], inp["D"], None)
    assert rel(y2.float().cpu().numpy(), yo) <= 2e-3
    assert rel(f2.cpu().numpy(), fo) <= 2e-3
