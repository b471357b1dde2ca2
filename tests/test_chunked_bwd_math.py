"""The chunked backward's algebra, restated in fp64 numpy and pinned to the backward oracle (CPU).

The GPU's scalar-A backward evaluates the chunked algorithm (Structured State Space Duality, "The
chunked algorithm takes both") in reverse, chunk by chunk: the state entering every chunk, the
adjoint at every chunk's end (a reverse scan), then per chunk the dense products of the quadratic
form and the rank-N terms, and the gradient with respect to the in-chunk prefix sums in the
cancellation-free form

    rc_k = e^{cum_Q} <g, h> + sum_{j<k} w_j v_j + sum_{i>=k, j<k} K_ij + sum_{i>=k} e_i u_i.

This file restates that algebra in plain fp64 numpy (no GPU, nothing shared with the kernels)
and checks it against the token-recurrence oracle to rounding, on ragged chunks, several B/C
groups and chunk lengths, with and without D, init_state and dfinal.  A wrong term (a dropped
decay, a missing straddle block) fails it.
"""
import numpy as np
import pytest

import oracle


def chunked_bwd(x, dt, A, B, C, D, init, dy, dfinal, Q, drop=None):
    nb, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    x, B, C, dt = (np.asarray(v, np.float64) for v in (x, B, C, dt))
    nc = -(-T // Q)
    out = dict(dx=np.zeros_like(x), ddt=np.zeros_like(dt), dA=np.zeros(H), dB=np.zeros_like(B), dC=np.zeros_like(C),
               dD=np.zeros(H) if D is not None else None, dinit=np.zeros((nb, H, N, P)))

    def chunk(a, bi, c, hh, width):
        t0 = c * Q
        L = min(Q, T - t0)
        m = np.zeros((Q, width))
        m[:L] = a[bi, t0:t0 + L, hh]
        return m, L

    for bi in range(nb):
        for h in range(H):
            g = h // hpg
            cums = []
            for c in range(nc):
                t0 = c * Q
                L = min(Q, T - t0)
                cum = np.zeros(Q)
                cum[:L] = np.cumsum(dt[bi, t0:t0 + L, h] * A[h])
                cum[L:] = cum[L - 1]
                cums.append(cum)
            # the state entering every chunk
            hs = []
            hc = np.zeros((N, P)) if init is None else np.asarray(init[bi, h], np.float64)
            for c in range(nc):
                Xc, _ = chunk(x, bi, c, h, P)
                Bc, _ = chunk(B, bi, c, g, N)
                hs.append(hc)
                w = np.exp(cums[c][-1] - cums[c])
                hc = np.exp(cums[c][-1]) * hc + Bc.T @ (w[:, None] * Xc)
            # the adjoint at every chunk's end: a reverse scan over chunks
            gs = [None] * nc
            gc = np.zeros((N, P)) if dfinal is None else np.asarray(dfinal[bi, h], np.float64)
            for c in range(nc - 1, -1, -1):
                Cc, _ = chunk(C, bi, c, g, N)
                dYc, _ = chunk(dy, bi, c, h, P)
                gs[c] = gc
                gc = np.exp(cums[c][-1]) * gc + Cc.T @ (np.exp(cums[c])[:, None] * dYc)
            out["dinit"][bi, h] = gc
            for c in range(nc):
                t0 = c * Q
                cum = cums[c]
                Xc, L = chunk(x, bi, c, h, P)
                dYc, _ = chunk(dy, bi, c, h, P)
                Bc, _ = chunk(B, bi, c, g, N)
                Cc, _ = chunk(C, bi, c, g, N)
                hp, gcc = hs[c], gs[c]
                Lm = np.tril(np.exp(np.minimum(cum[:, None] - cum[None, :], 0.0)))
                if drop == "mask":
                    Lm = np.tril(np.ones((Q, Q)))
                CB = Cc @ Bc.T
                S, Gm = Lm * CB, Lm * (dYc @ Xc.T)
                w, e = np.exp(cum[-1] - cum), np.exp(cum)
                Bg, dYh = Bc @ gcc, dYc @ hp.T
                out["dx"][bi, t0:t0 + L, h] = (S.T @ dYc + w[:, None] * Bg + (0 if D is None else D[h]) * dYc)[:L]
                out["dC"][bi, t0:t0 + L, g] += (Gm @ Bc + e[:, None] * dYh)[:L]
                out["dB"][bi, t0:t0 + L, g] += (Gm.T @ Cc + w[:, None] * (Xc @ gcc.T))[:L]
                K = Gm * CB
                v = np.sum(Bg * Xc, 1)
                u = np.sum(Cc * dYh, 1)
                E = np.exp(cum[-1]) * np.sum(gcc * hp)
                rc = np.array([E + np.sum((w * v)[:k]) + (0.0 if drop == "straddle" else K[k:, :k].sum())
                               + np.sum((e * u)[k:]) for k in range(Q)])
                out["ddt"][bi, t0:t0 + L, h] = A[h] * rc[:L]
                out["dA"][h] += np.sum(dt[bi, t0:t0 + L, h] * rc[:L])
                if D is not None:
                    out["dD"][h] += np.sum(dYc * Xc)
    return out


def case(rng, nb, T, H, P, N, G, with_D, with_init, with_dfinal):
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    return dict(x=f(nb, T, H, P), B=f(nb, T, G, N) * 0.5, C=f(nb, T, G, N) * 0.5,
                dt=np.log1p(np.exp(f(nb, T, H) - 1.0)).astype(np.float32),
                A=(-np.exp(rng.uniform(0, np.log(4), H))).astype(np.float32),
                D=f(H) if with_D else None, init=f(nb, H, N, P) if with_init else None,
                dy=rng.standard_normal((nb, T, H, P)), dfinal=rng.standard_normal((nb, H, N, P)) if with_dfinal else None)


def compare(got, ref):
    worst = 0.0
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        if ref[k] is None:
            continue
        worst = max(worst, float(np.abs(got[k] - ref[k]).max() / max(1e-30, np.abs(ref[k]).max())))
    return worst


@pytest.mark.parametrize("shape", [(2, 100, 4, 8, 6, 2, 16, True, True, True), (1, 37, 2, 4, 5, 1, 8, False, False, True),
                                   (2, 64, 2, 8, 8, 1, 64, True, True, False), (1, 130, 3, 4, 4, 3, 32, True, False, False)],
                         ids=["G2_Q16", "ragged_Q8", "Q64_one_chunk", "G3_Q32"])
def test_chunked_backward_algebra_equals_the_recurrence(shape):
    nb, T, H, P, N, G, Q, wD, wI, wF = shape
    c = case(np.random.default_rng(T + Q), nb, T, H, P, N, G, wD, wI, wF)
    ref = oracle.recurrence_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init"], c["dy"], c["dfinal"])
    got = chunked_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init"], c["dy"], c["dfinal"], Q)
    assert compare(got, ref) < 1e-12


@pytest.mark.parametrize("drop", ["mask", "straddle"])
def test_a_wrong_term_is_caught(drop):
    c = case(np.random.default_rng(5), 1, 40, 2, 4, 4, 1, True, True, True)
    ref = oracle.recurrence_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init"], c["dy"], c["dfinal"])
    got = chunked_bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init"], c["dy"], c["dfinal"], 16, drop=drop)
    assert compare(got, ref) > 1e-3
