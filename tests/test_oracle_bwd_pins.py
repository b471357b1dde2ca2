"""Pins of the fp64 backward oracle (``oracle.recurrence_bwd``), CPU only.

The backward oracle is the reverse mode of the token recurrence.  It is pinned
here against something it shares nothing with: central finite differences, in
fp64, of the loss L = sum y*dy + sum final_state*dfinal evaluated through the
dense lower-triangular matrix of Structured State Space Duality, "The
recurrence as one matrix" (``oracle.brute``), for every entry of every
gradient, in both A modes, with and without D and the initial state, with one
and with two B/C groups.  Deliberately wrong variants of the backward (a
dropped decay factor, a wrong order of operations, a missing skip term, the
state used in place of the adjoint) must fail the same comparison.
"""
import numpy as np
import pytest

import oracle
from oracle import brute


def make_case(rng, nb=2, T=5, H=2, P=3, N=2, G=1, diagonal=False, with_D=True, with_init=True, with_dfinal=True):
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    c = dict(x=f(nb, T, H, P), B=f(nb, T, G, N) * 0.7, C=f(nb, T, G, N) * 0.7,
             dt=(np.log1p(np.exp(f(nb, T, H) - 1.0))).astype(np.float32),
             A=(-np.exp(rng.uniform(0, np.log(4), (H, N) if diagonal else (H,)))).astype(np.float32),
             D=f(H) if with_D else None, init=f(nb, H, N, P) if with_init else None)
    c["dy"] = rng.standard_normal((nb, T, H, P))
    c["dfinal"] = rng.standard_normal((nb, H, N, P)) if with_dfinal else None
    return c


def loss_dense(c, x, dt, A, B, C, D, init):
    """L through brute.dense_M / apply_M / final_state_from_M, fp64."""
    nb, T, H, P = x.shape
    G = B.shape[2]
    hpg = H // G
    total = 0.0
    for bi in range(nb):
        for h in range(H):
            g = h // hpg
            a = np.exp(dt[bi, :, h][:, None] * A[h][None, :]) if A.ndim == 2 else np.exp(dt[bi, :, h] * A[h])
            h0 = None if init is None else init[bi, h]
            M = brute.dense_M(a, B[bi, :, g], C[bi, :, g])
            y = brute.apply_M(M, x[bi, :, h], a, C[bi, :, g], h0, None if D is None else D[h])
            total += float(np.sum(y * c["dy"][bi, :, h]))
            if c["dfinal"] is not None:
                fin = brute.final_state_from_M(x[bi, :, h], a, B[bi, :, g], h0)
                total += float(np.sum(fin * c["dfinal"][bi, h]))
    return total


def fd_grads(c, eps=1e-6):
    base = {k: (None if c[k] is None else c[k].astype(np.float64)) for k in ("x", "dt", "A", "B", "C", "D", "init")}
    out = {}
    for k, arr in base.items():
        if arr is None:
            out[k] = None
            continue
        g = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = loss_dense(c, **base)
            flat[i] = old - eps
            lm = loss_dense(c, **base)
            flat[i] = old
            g.reshape(-1)[i] = (lp - lm) / (2 * eps)
        out[k] = g
    return out


def oracle_grads(c, plant=0):
    return oracle.recurrence_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init"], c["dy"], c["dfinal"],
                                 plant=plant)


PAIRS = [("dx", "x"), ("ddt", "dt"), ("dA", "A"), ("dB", "B"), ("dC", "C"), ("dD", "D"), ("dinit", "init")]


def compare(og, fd, tol=1e-6):
    worst = 0.0
    for ok, fk in PAIRS:
        if fd[fk] is None:
            continue
        a, b = og[ok], fd[fk]
        err = np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))
        worst = max(worst, err)
        assert err <= tol, "%s: max error %.3g" % (ok, err)
    return worst


CASES = [
    dict(diagonal=False), dict(diagonal=True), dict(diagonal=False, G=2, H=4),
    dict(diagonal=True, G=2, H=4, with_D=False), dict(diagonal=False, with_init=False, with_dfinal=False),
    dict(diagonal=True, with_init=False, with_dfinal=True, T=7),
]


@pytest.mark.parametrize("kw", CASES, ids=["scalar", "diagonal", "scalar_G2", "diagonal_G2_noD",
                                           "scalar_no_init_no_dfinal", "diagonal_T7"])
def test_backward_oracle_matches_finite_differences_of_dense_form(kw):
    rng = np.random.default_rng(7 + len(str(kw)))
    c = make_case(rng, **kw)
    compare(oracle_grads(c), fd_grads(c))


@pytest.mark.parametrize("plant", [1, 2, 3, 4])
def test_planted_backward_mistakes_are_caught(plant):
    rng = np.random.default_rng(99)
    c = make_case(rng, diagonal=True)
    fd = fd_grads(c)
    with pytest.raises(AssertionError):
        compare(oracle_grads(c, plant=plant), fd)


def test_skip_and_initial_state_gradients_closed_form():
    # dD_h = sum over batch rows and tokens of dy . x (y gains D_h x); with every decay 0
    # (dt -> large, A < 0) the initial state only reaches y_0 and final_state only sees the
    # last token, so dinit = 0 and dx_{T-1} = B_{T-1}^T (C_{T-1} dy_{T-1}^T + dfinal) + D dy.
    rng = np.random.default_rng(5)
    c = make_case(rng, diagonal=False)
    c["dt"] = np.full_like(c["dt"], 80.0)
    g = oracle_grads(c)
    np.testing.assert_allclose(g["dD"], np.einsum("bthp,bthp->h", c["dy"], c["x"].astype(np.float64)), rtol=1e-12)
    assert np.max(np.abs(g["dinit"])) < 1e-20
    nb, T, H, P = c["x"].shape
    for bi in range(nb):
        for h in range(H):
            gT = np.outer(c["C"][bi, T - 1, 0], c["dy"][bi, T - 1, h]) + c["dfinal"][bi, h]
            want = c["B"][bi, T - 1, 0].astype(np.float64) @ gT + c["D"][h] * c["dy"][bi, T - 1, h]
            np.testing.assert_allclose(g["dx"][bi, T - 1, h], want, rtol=1e-10, atol=1e-12)
