"""GPU parity of the backward pass (``ssd_bwd``, through the C ABI) against the fp64 backward oracle.

Every gradient -- dx, ddt, dA, dB, dC, dD, dinit -- is compared on the whole
tensor (relative L2).  Tolerances: fp32 io 1e-5 (fp32 arithmetic throughout);
bf16 io 2e-3 (dx, dB and dC are rounded to bf16 on output; the fp32 outputs
ddt, dA, dD and dinit are held to 1e-4).  Cases cover both A modes, D and the
initial state present or absent, dfinal present or absent, several B/C
groups, ragged lengths around the 8-token checkpoint blocks of the recurrence
path and the 64-token chunks of the chunked path (scalar A at P 64, N 64 or
128), a state dimension that does not fill its last slice of rows, and the
head dims each path takes.
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
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def cotangents(w, seed, with_dfinal):
    g = torch.Generator().manual_seed(seed)
    io = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dy = torch.randn((w.b, w.T, w.H, w.P), generator=g).to(io)
    df = torch.randn((w.b, w.H, w.N, w.P), generator=g) if with_dfinal else None
    return dy, df


def run_and_check(w, seed=0, with_dfinal=True, drop_D=False, dt_scale=1.0, device="cuda:0"):
    inp = make_inputs(w)
    inp["dt"] = inp["dt"] * dt_scale
    if drop_D:
        inp["D"] = None
    dy, df = cotangents(w, 100 + seed, with_dfinal)
    d = {k: (None if v is None else v.to(device)) for k, v in inp.items()}
    got = ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], dy.to(device),
                      None if df is None else df.to(device), want_dD=inp["D"] is not None)
    torch.cuda.synchronize()
    ref = oracle.recurrence_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init_state"],
                                dy.double().numpy(), None if df is None else df.double().numpy())
    io_tol = 2e-3 if w.dtype == "bf16" else 1e-5
    f32_tol = 1e-4 if w.dtype == "bf16" else 1e-5
    errs = {}
    for k, tol in (("dx", io_tol), ("dB", io_tol), ("dC", io_tol), ("ddt", f32_tol), ("dA", f32_tol),
                   ("dD", f32_tol), ("dinit", f32_tol)):
        if ref[k] is None:
            continue
        g = got[k].float().cpu().numpy()
        assert np.isfinite(g).all(), k
        errs[k] = rel(g, ref[k])
        assert errs[k] <= tol, "%s relL2 %.3g > %.3g" % (k, errs[k], tol)
    return errs


CASES = [
    ("scalar_bf16", Workload("t", b=2, T=100, H=4, P=64, N=128, G=2, Q=128, D="normal", init_std=0.1, seed=701)),
    ("diag_bf16", Workload("t", b=2, T=77, H=4, P=64, N=64, G=1, Q=64, a_mode="diagonal", D="none",
                           init_std=0.2, seed=702)),
    ("scalar_f32", Workload("t", b=1, T=130, H=3, P=16, N=16, G=1, Q=64, dtype="f32", D="ones", seed=703)),
    ("diag_f32_N50", Workload("t", b=2, T=65, H=2, P=32, N=50, G=2, Q=128, dtype="f32", a_mode="diagonal",
                              D="normal", init_std=0.3, seed=704)),
    ("scalar_bf16_P128_N128", Workload("t", b=1, T=40, H=2, P=128, N=128, G=1, Q=128, D="normal", seed=705)),
    ("scalar_f32_P4_T1", Workload("t", b=3, T=1, H=2, P=4, N=8, G=1, Q=64, dtype="f32", D="normal",
                                  init_std=0.5, seed=706)),
    ("scalar_bf16_T32", Workload("t", b=1, T=32, H=2, P=64, N=128, G=1, Q=128, D="none", seed=707)),
    # the chunked path (scalar A, P 64, N 64 or 128): 64-token chunks, ragged tails, one-token
    # sequences, fp32 io at 1e-5, two B/C groups
    ("chunked_f32_N64_G2", Workload("t", b=2, T=150, H=4, P=64, N=64, G=2, Q=64, dtype="f32", D="normal",
                                    init_std=0.2, seed=721)),
    ("chunked_f32_N128_T65", Workload("t", b=1, T=65, H=2, P=64, N=128, G=1, Q=128, dtype="f32", D="ones",
                                      init_std=0.3, seed=722)),
    ("chunked_bf16_N64_T1", Workload("t", b=3, T=1, H=2, P=64, N=64, G=1, Q=64, D="normal", init_std=0.5,
                                     seed=723)),
    ("chunked_bf16_N128_G2_T200", Workload("t", b=2, T=200, H=6, P=64, N=128, G=2, Q=256, D="none",
                                           init_std=0.1, seed=724)),
    # the long-sequence head dims (N 256, one head per B/C group): the chunked path on 32-token chunks
    ("chunked_bf16_N256_G8", Workload("t", b=1, T=150, H=8, P=64, N=256, G=8, Q=128, D="none", init_std=0.1,
                                      seed=725)),
    ("chunked_f32_N256_G2", Workload("t", b=2, T=77, H=4, P=64, N=256, G=2, Q=128, dtype="f32", D="normal",
                                     init_std=0.2, seed=726)),
    # P 128: 64-token chunks at N 64, 32-token chunks at N 128
    ("chunked_f32_P128_N64", Workload("t", b=2, T=90, H=2, P=128, N=64, G=1, Q=64, dtype="f32", D="normal",
                                      init_std=0.2, seed=728)),
    ("chunked_bf16_P128_N128_G2", Workload("t", b=1, T=170, H=4, P=128, N=128, G=2, Q=128, D="none",
                                           init_std=0.1, seed=729)),
    # the recurrence path at N 256 (P 32 is outside the chunked path)
    ("scalar_bf16_P32_N256", Workload("t", b=1, T=90, H=2, P=32, N=256, G=1, Q=128, D="normal", seed=727)),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_backward_small(name, w, cuda_device):
    run_and_check(w, seed=1)
    run_and_check(w, seed=2, with_dfinal=False, drop_D=w.D != "none")


def test_backward_large_decay_and_long(cuda_device):
    # dt scaled up (states forget within a few tokens) and a 1000-token sequence (31 checkpoints)
    w = Workload("t", b=1, T=1000, H=2, P=64, N=128, G=1, Q=128, D="normal", init_std=0.1, seed=711)
    run_and_check(w, seed=3, dt_scale=10.0)
    run_and_check(w, seed=4)


def test_backward_at_the_2p7b_head_dims(cuda_device):
    """A medium case at the 2.7B layer's head dims (N 128, P 64, 8 heads per group)."""
    w = Workload("t", b=1, T=512, H=8, P=64, N=128, G=1, Q=256, D="normal", seed=712)
    run_and_check(w, seed=5)


def test_backward_empty_and_rejections(cuda_device):
    dev = cuda_device
    x = torch.zeros((2, 0, 4, 64), device=dev, dtype=torch.bfloat16)
    Bm = torch.zeros((2, 0, 1, 128), device=dev, dtype=torch.bfloat16)
    dt = torch.zeros((2, 0, 4), device=dev)
    A = -torch.ones(4, device=dev)
    df = torch.randn((2, 4, 128, 64), device=dev)
    g = ssd.ssd_bwd(x, dt, A, Bm, Bm.clone(), None, None, x.clone(), df)
    torch.cuda.synchronize()
    assert torch.equal(g["dinit"], df) and torch.count_nonzero(g["dA"]) == 0
    # head dims above 128 and the tcgen05 path are not taken
    for kw in (dict(P=256, N=64), dict(P=64, N=128, path="tcgen05")):
        d = ssd.make_dims(1, 64, 2, kw["P"], kw["N"], 1, 128, path=kw.get("path", "auto"))
        with pytest.raises(ssd.SSDError) as e:
            ssd.ssd_bwd_workspace_size(d)
        assert e.value.status == ssd.SSD_ERR_UNSUPPORTED


def test_backward_at_the_2p7b_bench_shape(cuda_device):
    """The bench's backward call at the full 2.7B shape (b4 T8192 H80 P64 N128 G1), checked on two
    whole heads: every batch row's dx, ddt and dinit of the head, and the head's dA and dD (sums
    over all batch rows and tokens), against the fp64 backward oracle run on that head alone (with
    one B/C group, a head's gradients depend on its own inputs and the shared B and C only).

    dA = sum_k dt_k rc_k and dD = sum dy x are sums of 32768 (and 2M) terms of both signs; for head
    0 here |dA| = 0.53 while sum_k |dt_k rc_k| = 8.7e3.  A sum of terms that each carry a few fp32
    rounding errors is only held to about eps_32 * sum |terms| (the forward error bound of
    summation), so these two scalars get 1e-4 relative plus 2 eps_32 sum |terms|, the terms taken
    from the oracle (dt ddt / A for dA, dy x for dD)."""
    from ssd_sequence_mixing_fwd_b300.inputs import WORKLOADS
    w = WORKLOADS["mamba2_2p7b"]
    inp = make_inputs(w)
    dy, df = cotangents(w, 4242, True)
    d = {k: (None if v is None else v.to(cuda_device)) for k, v in inp.items()}
    got = ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], dy.to(cuda_device),
                      df.to(cuda_device))
    torch.cuda.synchronize()
    got = {k: (None if v is None else v.float().cpu().numpy()) for k, v in got.items()}
    for h in (0, 57):
        sl = lambda t: None if t is None else t[:, :, h:h + 1].contiguous()
        ref = oracle.recurrence_bwd(sl(inp["x"]), sl(inp["dt"]), inp["A"][h:h + 1], inp["B"], inp["C"],
                                    None if inp["D"] is None else inp["D"][h:h + 1],
                                    None if inp["init_state"] is None else inp["init_state"][:, h:h + 1],
                                    dy[:, :, h:h + 1].double().numpy(), df[:, h:h + 1].double().numpy())
        assert rel(got["dx"][:, :, h], ref["dx"][:, :, 0]) <= 2e-3
        assert rel(got["ddt"][:, :, h], ref["ddt"][:, :, 0]) <= 1e-4
        assert rel(got["dinit"][:, h], ref["dinit"][:, 0]) <= 1e-4
        eps = 2.0 ** -24
        dt_h = inp["dt"][:, :, h].double().numpy()
        terms_a = np.abs(dt_h * ref["ddt"][:, :, 0] / float(inp["A"][h])).sum()
        assert abs(got["dA"][h] - ref["dA"][0]) <= 1e-4 * abs(ref["dA"][0]) + 2 * eps * terms_a
        if ref["dD"] is not None:
            terms_d = np.abs(dy[:, :, h].double().numpy() * inp["x"][:, :, h].double().numpy()).sum()
            assert abs(got["dD"][h] - ref["dD"][0]) <= 1e-4 * abs(ref["dD"][0]) + 2 * eps * terms_d


@pytest.mark.parametrize("dtype,tol", [("f32", 1e-5), ("bf16", 1e-4)])
def test_chunked_and_recurrence_paths_agree(dtype, tol, cuda_device):
    """The chunked backward (path "auto") and the token recurrence (path "generic") are two
    different evaluations of the same gradients: on the same inputs they agree with each other,
    every output, at the fp32 arithmetic's accuracy (io rounding aside)."""
    w = Workload("t", b=2, T=150, H=4, P=64, N=128, G=2, Q=128, dtype=dtype, D="normal", init_std=0.2,
                 seed=731)
    inp = make_inputs(w)
    dy, df = cotangents(w, 9, True)
    d = {k: (None if v is None else v.to(cuda_device)) for k, v in inp.items()}
    args = (d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], dy.to(cuda_device),
            df.to(cuda_device))
    a = ssd.ssd_bwd(*args, path="auto")
    r = ssd.ssd_bwd(*args, path="generic")
    torch.cuda.synchronize()
    dims = ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, dtype=dtype)
    assert ssd.ssd_bwd_workspace_size(dims) != ssd.ssd_bwd_workspace_size(
        ssd.make_dims(w.b, w.T, w.H, w.P, w.N, w.G, w.Q, dtype=dtype, path="generic"))   # two layouts
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        ga, gr = a[k].float().cpu().numpy(), r[k].float().cpu().numpy()
        lim = 2e-3 if (dtype == "bf16" and k in ("dx", "dB", "dC")) else tol
        assert rel(ga, gr) <= lim, (k, rel(ga, gr))
