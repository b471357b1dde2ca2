"""Brute-force fp64 evaluations of the SSD map on tiny inputs (numpy).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  These pin the recurrence
oracle; they are written from the matrix view of the pages and share nothing
with the recurrence code or the CUDA path.

* :func:`dense_M` builds the lower-triangular matrix of Structured State Space
  Duality, "The recurrence as one matrix":
  M[i, j] = C_i^T (Abar_i ... Abar_{j+1}) B_j for i >= j, else 0, with
  Abar_k = diag(a_k) (a_k a scalar times the identity in the scalar case).
* :func:`masked_attention` is the scalar case written as the same page says it
  collapses: a 1-semiseparable decay mask L[i, j] = prod_{k=j+1..i} a_k applied
  to the query-key products C_i^T B_j, then multiplied by X
  (also "On Structured State-Space Duality", abstract).

Both take fp64 numpy arrays for one (batch, head) stream: x (T,P), a (T,) or
(T,N) per-token decays, B and C (T,N), h0 (N,P) or None, D scalar or None.
"""
import numpy as np


def decay_products(a):
    """L[..., i, j] = prod_{k=j+1}^{i} a_k for i >= j, 0 above the diagonal.

    ``a`` is (T,) or (T, N); the result is (T, T) or (N, T, T).  Built row by
    row from L[i, j] = a_i * L[i-1, j] and L[i, i] = 1 (the empty product).
    """
    a = np.asarray(a, dtype=np.float64)
    per_n = a.ndim == 2
    T = a.shape[0]
    cols = a.T if per_n else a[None, :]          # (N or 1, T)
    L = np.zeros((cols.shape[0], T, T), dtype=np.float64)
    for i in range(T):
        if i > 0:
            L[:, i, :i] = cols[:, i:i + 1] * L[:, i - 1, :i]
        L[:, i, i] = 1.0
    return L if per_n else L[0]


def prefix_products(a):
    """q[i] = prod_{k=0}^{i} a_k, shape like ``a`` (the decay applied to h_{-1})."""
    a = np.asarray(a, dtype=np.float64)
    q = np.empty_like(a)
    run = np.ones(a.shape[1:], dtype=np.float64)
    for i in range(a.shape[0]):
        run = run * a[i]
        q[i] = run
    return q


def dense_M(a, B, C):
    """The T x T matrix M with M[i, j] = sum_n C[i,n] (prod_{k=j+1}^{i} a_k[n]) B[j,n]."""
    B = np.asarray(B, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    T, N = B.shape
    if a.ndim == 1:
        a = np.repeat(a[:, None], N, axis=1)
    L = decay_products(a)                      # (N, T, T)
    M = np.zeros((T, T), dtype=np.float64)
    for n in range(N):
        M += np.outer(C[:, n], B[:, n]) * L[n]
    return M


def apply_M(M, x, a, C, h0=None, D=None):
    """y = M x + C_i^T diag(prod_{k<=i} a_k) h0 + D x for one stream."""
    x = np.asarray(x, dtype=np.float64)
    y = M @ x
    if h0 is not None:
        a = np.asarray(a, dtype=np.float64)
        C = np.asarray(C, dtype=np.float64)
        q = prefix_products(a if a.ndim == 2 else np.repeat(a[:, None], C.shape[1], axis=1))
        y = y + (C * q) @ np.asarray(h0, dtype=np.float64)
    if D is not None:
        y = y + float(D) * x
    return y


def final_state_from_M(x, a, B, h0=None):
    """h_{T-1} = sum_j diag(prod_{k=j+1}^{T-1} a_k) B_j x_j^T (+ decayed h0)."""
    x = np.asarray(x, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    T, N = B.shape
    if a.ndim == 1:
        a = np.repeat(a[:, None], N, axis=1)
    L = decay_products(a)                      # (N, T, T); last row is the decay to the end
    w = L[:, T - 1, :].T                       # (T, N): prod_{k=j+1}^{T-1} a_k[n]
    h = (B * w).T @ x
    if h0 is not None:
        h = h + prefix_products(a)[T - 1][:, None] * np.asarray(h0, dtype=np.float64)
    return h


def masked_attention(x, a, B, C, D=None):
    """Scalar case only: y = (L o (C B^T)) x + D x with L the 1-semiseparable mask."""
    a = np.asarray(a, dtype=np.float64)
    assert a.ndim == 1, "the single-mask form exists for the scalar case only"
    L = decay_products(a)
    S = L * (np.asarray(C, dtype=np.float64) @ np.asarray(B, dtype=np.float64).T)
    y = S @ np.asarray(x, dtype=np.float64)
    if D is not None:
        y = y + float(D) * np.asarray(x, dtype=np.float64)
    return y
