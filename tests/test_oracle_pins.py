"""Pins for the fp64 oracle, checked against things other than itself.

Each test compares the token-by-token recurrence (oracle.recurrence, C) with
an independent statement of the same map: the materialised matrix M and the
masked-attention form (Structured State Space Duality, "The recurrence as one
matrix"), hand-worked examples, closed forms, the diagonal-as-sum-of-scalar
structure ("What the duality gives up"), the rank bound on off-diagonal blocks
("When it breaks") and algebraic invariants.  ``test_planted_mistakes_are_caught``
plants typical mistakes in the oracle and checks that these pins fail.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_case(rng, nb=2, T=37, H=4, P=3, N=5, G=2, diagonal=False, with_D=True,
              with_init=True, dt_scale=1.0):
    x = rng.standard_normal((nb, T, H, P)).astype(np.float32)
    B = (rng.standard_normal((nb, T, G, N)) / np.sqrt(N)).astype(np.float32)
    C = (rng.standard_normal((nb, T, G, N)) / np.sqrt(N)).astype(np.float32)
    dt = (np.log1p(np.exp(rng.standard_normal((nb, T, H)) - 2.0)) * dt_scale).astype(np.float32)
    A = -np.exp(rng.uniform(0, np.log(16), (H, N) if diagonal else (H,))).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32) if with_D else None
    h0 = (0.3 * rng.standard_normal((nb, H, N, P))).astype(np.float32) if with_init else None
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D, init_state=h0)


def brute_all(c):
    """y and final state for every stream through the dense matrix M."""
    x, dt, A, B, C, D, h0 = (c[k] for k in ("x", "dt", "A", "B", "C", "D", "init_state"))
    nb, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((nb, T, H, P))
    fin = np.zeros((nb, H, N, P))
    for bi in range(nb):
        for h in range(H):
            g = h // (H // G)
            Ah = A[h].astype(np.float64)
            a = np.exp(dt[bi, :, h].astype(np.float64)[:, None] * Ah[None, :]) if A.ndim == 2 \
                else np.exp(dt[bi, :, h].astype(np.float64) * float(Ah))
            Bs, Cs = B[bi, :, g].astype(np.float64), C[bi, :, g].astype(np.float64)
            M = brute.dense_M(a, Bs, Cs)
            hh = None if h0 is None else h0[bi, h].astype(np.float64)
            y[bi, :, h] = brute.apply_M(M, x[bi, :, h], a, Cs, hh, None if D is None else D[h])
            fin[bi, h] = brute.final_state_from_M(x[bi, :, h], a, Bs, hh)
    return y, fin


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("diagonal", [False, True])
@pytest.mark.parametrize("with_init", [False, True])
@pytest.mark.parametrize("with_D", [False, True])
def test_recurrence_equals_dense_M(diagonal, with_init, with_D):
    rng = np.random.default_rng(10 + 4 * diagonal + 2 * with_init + with_D)
    c = rand_case(rng, diagonal=diagonal, with_D=with_D, with_init=with_init)
    y, fin = oracle.recurrence(**c)
    yb, fb = brute_all(c)
    assert rel(y, yb) < 1e-12
    assert rel(fin, fb) < 1e-12


@pytest.mark.parametrize("seed", range(4))
def test_recurrence_equals_dense_M_random_shapes(seed):
    rng = np.random.default_rng(100 + seed)
    G = int(rng.integers(1, 3))
    H = G * int(rng.integers(1, 3))
    c = rand_case(rng, nb=int(rng.integers(1, 3)), T=int(rng.integers(1, 90)), H=H,
                  P=int(rng.integers(1, 6)), N=int(rng.integers(1, 7)), G=G,
                  diagonal=bool(seed % 2))
    y, fin = oracle.recurrence(**c)
    yb, fb = brute_all(c)
    assert rel(y, yb) < 1e-12
    assert rel(fin, fb) < 1e-12


def test_recurrence_equals_dense_M_tiny_workload_shape():
    """The shape of the tiny fp32 workload (T=256, N=16, P=16) through dense M."""
    rng = np.random.default_rng(7)
    c = rand_case(rng, nb=1, T=256, H=2, P=16, N=16, G=1, with_init=False)
    y, fin = oracle.recurrence(**c)
    yb, fb = brute_all(c)
    assert rel(y, yb) < 1e-12
    assert rel(fin, fb) < 1e-12


def test_scalar_case_is_masked_linear_attention():
    """Scalar-identity SSM == (L o C B^T) X with L_ij = prod_{k=j+1..i} a_k."""
    rng = np.random.default_rng(3)
    c = rand_case(rng, nb=1, T=120, H=3, P=4, N=6, G=1, with_init=False)
    y, _ = oracle.recurrence(**c)
    for h in range(3):
        a = np.exp(c["dt"][0, :, h].astype(np.float64) * float(c["A"][h]))
        ya = brute.masked_attention(c["x"][0, :, h], a, c["B"][0, :, 0], c["C"][0, :, 0], c["D"][h])
        assert rel(y[0, :, h], ya) < 1e-12


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = v.split()
    return vals


@pytest.mark.parametrize("name", ["tiny_scalar_T3.txt", "tiny_diagonal_T3.txt"])
def test_hand_worked_examples(name):
    g = _read_golden(name)
    dims = {k: int(g[k][0]) for k in ("b", "T", "H", "P", "N", "G")}
    nb, T, H, P, N, G = (dims[k] for k in ("b", "T", "H", "P", "N", "G"))
    f = lambda k, shape: np.array([float(v) for v in g[k]], dtype=np.float32).reshape(shape)
    A = f("A", (H,) if g["a_mode"][0] == "scalar" else (H, N))
    y, fin = oracle.recurrence(f("x", (nb, T, H, P)), f("dt", (nb, T, H)), A,
                               f("B", (nb, T, G, N)), f("C", (nb, T, G, N)), f("D", (H,)),
                               f("init_state", (nb, H, N, P)))
    np.testing.assert_allclose(y.ravel(), [float(v) for v in g["y"]], rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(fin.ravel(), [float(v) for v in g["final_state"]], rtol=1e-7, atol=1e-8)


def test_closed_form_no_decay_is_cumulative_sum():
    """a == 1 (A = 0): y_t = C_t^T (h_{-1} + sum_{j<=t} B_j x_j^T) + D x_t."""
    rng = np.random.default_rng(5)
    c = rand_case(rng, nb=2, T=50, H=2, P=3, N=4, G=1)
    c["A"] = np.zeros_like(c["A"])
    y, fin = oracle.recurrence(**c)
    x, B, C, h0 = (c[k].astype(np.float64) for k in ("x", "B", "C", "init_state"))
    outer = np.einsum("btn,bthp->bthnp", B[:, :, 0], x)
    S = np.cumsum(outer, axis=1) + h0[:, None]
    yc = np.einsum("btn,bthnp->bthp", C[:, :, 0], S) + c["D"][None, None, :, None] * x
    assert rel(y, yc) < 1e-13
    assert rel(fin, S[:, -1]) < 1e-13


@pytest.mark.parametrize("diagonal", [False, True])
def test_closed_form_full_decay_is_diagonal_readout(diagonal):
    """a == 0 (A = -1e4, dt = 1): y_t = (C_t . B_t) x_t + D x_t; h_T = B_{T-1} x_{T-1}^T."""
    rng = np.random.default_rng(6)
    c = rand_case(rng, nb=2, T=40, H=2, P=3, N=4, G=1, diagonal=diagonal)
    c["A"] = np.full_like(c["A"], -1e4)
    c["dt"] = np.ones_like(c["dt"])
    y, fin = oracle.recurrence(**c)
    x, B, C = (c[k].astype(np.float64) for k in ("x", "B", "C"))
    cb = np.einsum("btn,btn->bt", C[:, :, 0], B[:, :, 0])
    yc = cb[:, :, None, None] * x + c["D"][None, None, :, None] * x
    assert rel(y, yc) < 1e-13
    fc = np.einsum("bn,bhp->bhnp", B[:, -1, 0], x[:, -1])
    assert rel(fin, fc) < 1e-13


def test_diagonal_is_sum_of_scalar_state_dims():
    """A diagonal SSM with N state dims == sum of N scalar SSMs with one state dim each."""
    rng = np.random.default_rng(8)
    c = rand_case(rng, nb=2, T=60, H=4, P=3, N=5, G=2, diagonal=True)
    y, fin = oracle.recurrence(**c)
    ysum = np.zeros_like(y)
    for n in range(5):
        cn = dict(c)
        cn["A"] = np.ascontiguousarray(c["A"][:, n])
        cn["B"] = np.ascontiguousarray(c["B"][..., n:n + 1])
        cn["C"] = np.ascontiguousarray(c["C"][..., n:n + 1])
        cn["D"] = None
        cn["init_state"] = np.ascontiguousarray(c["init_state"][:, :, n:n + 1])
        yn, fn = oracle.recurrence(**cn)
        ysum += yn
        assert rel(fin[:, :, n:n + 1], fn) < 1e-13
    ysum += c["D"][None, None, :, None] * c["x"].astype(np.float64)
    assert rel(y, ysum) < 1e-12


def test_diagonal_with_constant_decay_equals_scalar():
    rng = np.random.default_rng(9)
    c = rand_case(rng, nb=2, T=70, H=4, P=3, N=5, G=2)
    y, fin = oracle.recurrence(**c)
    cd = dict(c)
    cd["A"] = np.ascontiguousarray(np.repeat(c["A"][:, None], 5, axis=1))
    yd, fd = oracle.recurrence(**cd)
    assert rel(yd, y) < 1e-14 and rel(fd, fin) < 1e-14


@pytest.mark.parametrize("diagonal", [False, True])
def test_split_sequence_composition(diagonal):
    """Running T1 tokens, then the rest from the returned state, equals one run."""
    rng = np.random.default_rng(11)
    c = rand_case(rng, nb=2, T=90, H=4, P=3, N=5, G=2, diagonal=diagonal)
    y, fin = oracle.recurrence(**c)
    T1 = 33
    c1 = {k: (v[:, :T1].copy() if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    y1, f1 = oracle.recurrence(**c1)
    c2 = {k: (v[:, T1:].copy() if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    c2["init_state"] = f1.astype(np.float32)
    y2, f2 = oracle.recurrence(**c2)
    assert rel(y1, y[:, :T1]) < 1e-14
    # the handed-over state is rounded to fp32, so allow fp32-level differences
    assert rel(y2, y[:, T1:]) < 1e-6
    assert rel(f2, fin) < 1e-6


def test_linearity_and_skip_term():
    rng = np.random.default_rng(12)
    c = rand_case(rng, with_init=False)
    y1, _ = oracle.recurrence(**c)
    c2 = dict(c)
    c2["x"] = (2.0 * c["x"]).astype(np.float32)          # exact scaling by 2
    y2, _ = oracle.recurrence(**c2)
    assert rel(y2, 2.0 * y1) < 1e-15
    c0 = dict(c)
    c0["D"] = None
    y0, _ = oracle.recurrence(**c0)
    dx = c["D"][None, None, :, None].astype(np.float64) * c["x"].astype(np.float64)
    assert rel(y1 - y0, dx) < 1e-12


def test_group_map_and_head_independence():
    """G = H equals running each head alone; heads of one group share its B, C."""
    rng = np.random.default_rng(13)
    H, G = 4, 2
    c = rand_case(rng, nb=1, T=30, H=H, G=G)
    y, fin = oracle.recurrence(**c)
    for h in range(H):
        g = h // (H // G)
        ch = dict(x=c["x"][:, :, h:h + 1].copy(), dt=c["dt"][:, :, h:h + 1].copy(),
                  A=c["A"][h:h + 1].copy(), B=c["B"][:, :, g:g + 1].copy(),
                  C=c["C"][:, :, g:g + 1].copy(), D=c["D"][h:h + 1].copy(),
                  init_state=c["init_state"][:, h:h + 1].copy())
        yh, fh = oracle.recurrence(**ch)
        assert rel(yh[:, :, 0], y[:, :, h]) < 1e-15
        assert rel(fh[:, 0], fin[:, h]) < 1e-15
    # G = 1 equals G = H with B, C broadcast to every head
    c1 = rand_case(rng, nb=1, T=30, H=3, G=1)
    y1, _ = oracle.recurrence(**c1)
    cH = dict(c1)
    cH["B"] = np.ascontiguousarray(np.repeat(c1["B"], 3, axis=2))
    cH["C"] = np.ascontiguousarray(np.repeat(c1["C"], 3, axis=2))
    yH, _ = oracle.recurrence(**cH)
    assert rel(yH, y1) < 1e-15


def test_stream_subset_and_truncation_match_full_run():
    rng = np.random.default_rng(14)
    c = rand_case(rng, nb=2, T=40, H=4)
    y, fin = oracle.recurrence(**c)
    streams = [5, 0, 7]
    ys, fs = oracle.recurrence(**c, streams=streams, t_end=25)
    for i, s in enumerate(streams):
        bi, h = divmod(s, 4)
        assert np.array_equal(ys[i], y[bi, :25, h])
    cf = {k: (v[:, :25].copy() if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    _, ff = oracle.recurrence(**cf)
    for i, s in enumerate(streams):
        bi, h = divmod(s, 4)
        assert np.array_equal(fs[i], ff[bi, h])


def test_off_diagonal_blocks_have_rank_at_most_N():
    """Off-diagonal blocks of M factor through the N-dim state: rank <= N."""
    rng = np.random.default_rng(15)
    T, N = 64, 4
    B = rng.standard_normal((T, N))
    C = rng.standard_normal((T, N))
    a = np.exp(-0.05 * rng.random(T))
    M = brute.dense_M(a, B, C)
    for split in (16, 32, 48):
        blk = M[split:, :split]
        s = np.linalg.svd(blk, compute_uv=False)
        assert np.sum(s > 1e-10 * s[0]) <= N
    diag_blk = M[:32, :32]
    assert np.linalg.matrix_rank(diag_blk) > N         # the diagonal blocks are not low rank


PLANTS = {
    1: "readout before update",
    2: "initial state not decayed",
    3: "skip term dropped",
    4: "group map h mod G",
    5: "decay applied after the input",
    6: "B and C swapped",
    7: "diagonal: one decay for every n",
    8: "decay of the previous token",
    9: "state index transposed in the readout",
}


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_planted_mistakes_are_caught(plant):
    """Each planted mistake in the oracle breaks the dense-M pin by a wide margin."""
    rng = np.random.default_rng(200 + plant)
    c = rand_case(rng, nb=1, T=24, H=4, P=4, N=4, G=2, diagonal=(plant == 7))
    yb, fb = brute_all(c)
    y, fin = oracle.recurrence(**c, plant=plant)
    err = max(rel(y, yb), rel(fin, fb))
    assert err > 1e-3, "planted mistake '%s' went unnoticed (err %g)" % (PLANTS[plant], err)
    y0, f0 = oracle.recurrence(**c, plant=0)
    assert max(rel(y0, yb), rel(f0, fb)) < 1e-12


def test_oracle_reports_threads():
    assert oracle.threads_used(2) == 2


@pytest.mark.parametrize("name", ["tiny_scalar_T3.txt", "tiny_diagonal_T3.txt"])
def test_brute_force_forms_match_hand_worked_examples(name):
    """Pins the dense-M and masked-attention code itself to the hand-worked values."""
    g = _read_golden(name)
    N = int(g["N"][0])
    vals = lambda k: np.array([float(v) for v in g[k]])
    x, dt, A = vals("x").reshape(3, 1), vals("dt"), vals("A").astype(np.float32).astype(np.float64)
    B, C = vals("B").reshape(3, N), vals("C").reshape(3, N)
    a = np.exp(dt[:, None] * A[None, :]) if g["a_mode"][0] == "diagonal" else np.exp(dt * A[0])
    M = brute.dense_M(a, B, C)
    y = brute.apply_M(M, x, a, C, vals("init_state").reshape(N, 1), float(g["D"][0]))
    np.testing.assert_allclose(y.ravel(), vals("y"), rtol=1e-7, atol=1e-8)
    h = brute.final_state_from_M(x, a, B, vals("init_state").reshape(N, 1))
    np.testing.assert_allclose(h.ravel(), vals("final_state"), rtol=1e-7, atol=1e-8)
    if g["a_mode"][0] == "scalar":
        # with zero initial state the single-mask form gives y minus the decayed-h0 term
        y0 = brute.apply_M(M, x, a, C, None, float(g["D"][0]))
        ya = brute.masked_attention(x, a, B, C, float(g["D"][0]))
        np.testing.assert_allclose(ya, y0, rtol=1e-14, atol=1e-14)
