"""Seeded synthetic inputs for the SSD forward pass.

This module holds the workload shapes and the seeded input recipe only; it
contains none of the method's arithmetic.  Both the CUDA path's tests/bench and
the fp64 oracle draw their inputs from here, so they see identical bits.

Recipe (the Mamba-2 layer distributions):
  x ~ N(0,1); B, C ~ N(0,1)/sqrt(N); cast to the io dtype (bf16 or fp32)
  dt = softplus(N(0,1) - 2)                     fp32, shape (b,T,H)
  A  = -exp(U(0, ln 16))                        fp32, (H) scalar or (H,N) diagonal
  D  = 1, N(0,1) or absent                      fp32, (H)
  init_state = 0 or N(0, std^2)                 fp32, (b,H,N,P)
All draws are made on the host in fp32 from one ``torch.Generator`` seeded per
workload, in the fixed order x, B, C, dt, A, D, init_state, then cast.
"""
from dataclasses import dataclass, field, replace
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    T: int
    H: int
    P: int
    N: int
    G: int
    Q: int
    a_mode: str = "scalar"          # "scalar": A (H); "diagonal": A (H,N)
    dtype: str = "bf16"             # io dtype of x, B, C, y
    D: str = "normal"               # "ones", "normal" or "none"
    init_std: float = 0.0           # 0 -> zero initial state
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.b * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the throughput and parity targets are quoted on.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", b=1, T=256, H=2, P=16, N=16, G=1, Q=64,
                          dtype="f32", D="ones", seed=1001,
                          note="scalar-A tiny, all fp32"),
    "mamba2_130m": Workload("mamba2_130m", b=8, T=2048, H=24, P=64, N=128, G=1, Q=256,
                            D="normal", seed=1002, note="Mamba-2 130M layer shape"),
    "mamba2_2p7b": Workload("mamba2_2p7b", b=4, T=8192, H=80, P=64, N=128, G=1, Q=256,
                            D="normal", seed=1003, note="Mamba-2 2.7B layer shape"),
    "long_seq": Workload("long_seq", b=1, T=131072, H=32, P=64, N=256, G=8, Q=128,
                         D="none", init_std=0.1, seed=1004, note="scalar-A long sequence"),
    "diag_a": Workload("diag_a", b=4, T=4096, H=32, P=64, N=64, G=1, Q=64,
                       a_mode="diagonal", D="none", seed=1005,
                       note="general diagonal A, one decay per state dim"),
}

WORKLOAD_ORDER = ["tiny_fp32", "mamba2_130m", "mamba2_2p7b", "long_seq", "diag_a"]


def torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def make_inputs(w: Workload, device="cpu", seed=None):
    """Draw the seeded inputs of workload ``w`` (host draw, then moved to ``device``).

    Returns a dict with x, dt, A, B, C, D (or None), init_state (or None).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    f32 = torch.float32
    x = torch.randn((w.b, w.T, w.H, w.P), generator=g, dtype=f32)
    Bm = torch.randn((w.b, w.T, w.G, w.N), generator=g, dtype=f32) / math.sqrt(w.N)
    Cm = torch.randn((w.b, w.T, w.G, w.N), generator=g, dtype=f32) / math.sqrt(w.N)
    dt = torch.nn.functional.softplus(torch.randn((w.b, w.T, w.H), generator=g, dtype=f32) - 2.0)
    a_shape = (w.H,) if w.a_mode == "scalar" else (w.H, w.N)
    A = -torch.exp(torch.rand(a_shape, generator=g, dtype=f32) * math.log(16.0))
    if w.D == "ones":
        D = torch.ones((w.H,), dtype=f32)
    elif w.D == "normal":
        D = torch.randn((w.H,), generator=g, dtype=f32)
    else:
        D = None
    init = None
    if w.init_std > 0:
        init = torch.randn((w.b, w.H, w.N, w.P), generator=g, dtype=f32) * w.init_std
    io = torch_dtype(w)
    out = dict(x=x.to(io), dt=dt, A=A, B=Bm.to(io), C=Cm.to(io), D=D, init_state=init)
    if device != "cpu":
        out = {k: (None if v is None else v.to(device)) for k, v in out.items()}
    return out


def algorithmic_bytes(w: Workload, final_state=True) -> int:
    """Inputs read once plus outputs written once (the HBM floor of one call)."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.b * w.T
    by = tok * w.H * w.P * e * 2                 # x in, y out
    by += tok * w.G * w.N * e * 2                # B, C
    by += tok * w.H * 4                          # dt
    by += (w.H if w.a_mode == "scalar" else w.H * w.N) * 4
    by += w.H * 4 if w.D != "none" else 0
    st = w.b * w.H * w.N * w.P * 4
    by += st if w.init_std > 0 else 0
    by += st if final_state else 0
    return by


def algorithmic_bytes_bwd(w: Workload) -> int:
    """HBM floor of one backward call: x, dy, B, C, dt (and init_state, dfinal) read once; dx, dB,
    dC, ddt (and dinit) written once; dA and dD are negligible."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.b * w.T
    by = tok * w.H * w.P * e * 3                 # x, dy in; dx out
    by += tok * w.G * w.N * e * 4                # B, C in; dB, dC out
    by += tok * w.H * 4 * 2                      # dt in, ddt out
    st = w.b * w.H * w.N * w.P * 4
    by += st * (2 if w.init_std > 0 else 1) + st  # init (if any), dfinal in; dinit out
    return by


def _bwd_grad_floats(N: int, P: int, Q: int) -> int:
    return 8 + 2 * Q * (P + 1) + 2 * Q * (N + 1) + 2 * N * (P + 1) + 3 * Q * (Q + 1) + 5 * Q


def bwd_chunk_len(w: Workload) -> int:
    """Tokens per chunk of the chunked backward: 64 where its product kernel's shared memory
    (227 KB) fits, else 32; 0 where neither fits."""
    for Q in (64, 32):
        if _bwd_grad_floats(w.N, w.P, Q) <= 227 * 1024 // 4:
            return Q
    return 0


def bwd_chunked_applies(w: Workload) -> bool:
    """Whether ssd_bwd takes its chunked path (scalar A, P 64 or 128, N 64, 128 or 256, and a
    chunk length whose product kernel fits) for ``w``."""
    return w.a_mode == "scalar" and w.P in (64, 128) and w.N in (64, 128, 256) and bwd_chunk_len(w) > 0


def algorithmic_flops_bwd(w: Workload, Q: int = None) -> float:
    """Causal work of the chunked backward on Q-token chunks (every product a multiply-add
    pair): per chunk and head, dY X^T, S^T dY, G B and G^T C on the causal triangle
    (Q^2 N + Q^2 P) and the five rank-N products B g, dY h^T, X g^T, C^T (e o dY) and the
    chunk state B^T (w o X) (5 Q N P); per chunk and B/C group, C B^T (Q^2 N / 2)."""
    Q = bwd_chunk_len(w) if Q is None else Q
    nc = -(-w.T // Q)
    per_head = Q * Q * w.N + Q * Q * w.P + 5 * Q * w.N * w.P
    per_group = 0.5 * Q * Q * w.N
    return 2.0 * nc * w.b * (per_head * w.H + per_group * w.G)


def algorithmic_flops(w: Workload) -> float:
    """Causal tensor-core work of the chunked algorithm (elementwise work excluded).

    Per chunk of Q tokens: C B^T once per (batch, group) -- per head in the
    diagonal variant -- over the causal triangle (2*tri*N), the masked product
    with X per head (2*tri*P), the chunk state B^T (decay o X) per head (2*Q*N*P)
    and the output C h_prev per head (2*Q*N*P); tri = Q(Q+1)/2.
    """
    nc_full, rem = divmod(w.T, w.Q)
    chunks = [w.Q] * nc_full + ([rem] if rem else [])
    f = 0.0
    for q in chunks:
        tri = q * (q + 1) / 2
        cb_units = w.G if w.a_mode == "scalar" else w.H
        f += w.b * cb_units * 2 * tri * w.N
        f += w.b * w.H * (2 * tri * w.P + 4 * q * w.N * w.P)
    return f
