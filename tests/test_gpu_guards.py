"""GPU checks of the guards around the computation (through the C ABI).

* fp16 range: the tcgen05 paths' matrix operands are fp16; inputs (or states)
  beyond +-65504 must give either the oracle's answer or SSD_ERR_DEVICE from
  the device status -- never a silent inf/NaN with SSD_OK.
* canaries: output and workspace buffers padded with sentinels on both sides;
  ragged-T calls on both paths must leave the padding untouched (a stand-in
  for a memory checker, which this GPU pool does not offer).
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


def _run(d, w, path, workspace=None, y=None, fin=None):
    return ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk_Q=w.Q,
                       path=path, workspace=workspace, y=y, final_state=fin)


BIG = [("x", 1e5), ("B", 1e5), ("C", 1e5), ("init_state", 1e5)]


@pytest.mark.parametrize("what,val", BIG, ids=[b[0] for b in BIG])
@pytest.mark.parametrize("path", ["tcgen05", "generic"])
@pytest.mark.parametrize("a_mode", ["scalar", "diagonal"])
def test_out_of_fp16_range_is_reported_or_correct(what, val, path, a_mode, cuda_device):
    w = Workload("t", b=1, T=300, H=4, P=64, N=128 if a_mode == "scalar" else 64, G=1, Q=128,
                 a_mode=a_mode, D="none", init_std=0.1, seed=301)
    inp = make_inputs(w)
    t = inp[what].clone()
    flat = t.view(-1)
    flat[[3, 777, flat.numel() // 2]] = val         # a few huge entries
    inp[what] = t
    d = {k: (None if v is None else v.to(cuda_device)) for k, v in inp.items()}
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, a_mode=w.a_mode, path=path)
    ws = torch.empty(ssd.ssd_fwd_workspace_size(dims), device=cuda_device, dtype=torch.uint8)
    y, fin = _run(d, w, path, workspace=ws)
    st = ssd.ssd_check_device_status(ws)
    if st == ssd.SSD_ERR_DEVICE:
        assert path == "tcgen05", "the fp32 generic path has no fp16 range limit"
        return
    assert st == ssd.SSD_OK
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], None, inp["init_state"])
    yg = y.float().cpu().numpy()
    assert np.isfinite(yg).all() and np.isfinite(fin.cpu().numpy()).all()
    assert rel(yg, yr) <= 2e-3 and rel(fin.cpu().numpy(), fr) <= 2e-3


def _padded(shape, dtype, dev, pad, fill):
    n = int(np.prod(shape))
    big = torch.full((n + 2 * pad,), fill, dtype=dtype, device=dev)
    return big, big[pad:pad + n].view(shape)


@pytest.mark.parametrize("T", [77, 300, 1000])
@pytest.mark.parametrize("path", ["tcgen05", "generic"])
@pytest.mark.parametrize("a_mode", ["scalar", "diagonal"])
def test_ragged_calls_stay_inside_their_buffers(T, path, a_mode, cuda_device):
    w = Workload("t", b=2, T=T, H=4, P=64, N=128 if a_mode == "scalar" else 64, G=2, Q=128,
                 a_mode=a_mode, D="normal", init_std=0.1, seed=400 + T)
    inp = make_inputs(w)
    d = {k: (None if v is None else v.to(cuda_device)) for k, v in inp.items()}
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, a_mode=w.a_mode, path=path)
    need = ssd.ssd_fwd_workspace_size(dims)
    pad = 4096                                        # elements; keeps every view 16-byte aligned
    y_big, y = _padded((w.b, w.T, w.H, w.P), torch.bfloat16, cuda_device, pad, 7.0)
    f_big, fin = _padded((w.b, w.H, w.N, w.P), torch.float32, cuda_device, pad, 7.0)
    w_big = torch.full((need + 2 * pad,), 0xA5, dtype=torch.uint8, device=cuda_device)
    ws = w_big[pad:pad + need]
    for _ in range(2):
        _run(d, w, path, workspace=ws, y=y, fin=fin)
        assert ssd.ssd_check_device_status(ws) == ssd.SSD_OK
    torch.cuda.synchronize()
    for big, n in ((y_big, y.numel()), (f_big, fin.numel()), (w_big, need)):
        head, tail = big[:pad], big[pad + n:]
        ref = big.new_full((pad,), 7.0 if big.dtype != torch.uint8 else 0xA5)
        assert torch.equal(head, ref) and torch.equal(tail, ref), "write outside a buffer"
    yr, fr = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"])
    assert rel(y.float().cpu().numpy(), yr) <= 2e-3 and rel(fin.cpu().numpy(), fr) <= 2e-3
