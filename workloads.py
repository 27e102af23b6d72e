"""Seeded synthetic inputs for the selective scan and the pscan primitive.

This module is the only code shared by the CUDA path's tests/benchmark and the
oracle.  It draws random numbers and rounds them to the I/O dtype; it holds
none of the scan's arithmetic.

Every tensor is drawn on the CPU from a ``torch.Generator`` seeded per
workload, in the fixed order u, delta-normal, A-uniform (where the recipe has
one), B, C, D, h0.  delta is softplus of a normal draw (the recipe names the
positive step size that way; the scan itself takes delta as given).  For
bf16 I/O, u, delta, B and C are drawn in fp32 and rounded to bf16
(round-to-nearest-even); A, D and h0 stay fp32.

The five named workloads are the selective-scan shapes of the pages'
discussion (dim 512 at L = 8192; d_model 2048 at L = 2048 with N = 16; a long
sequence with state carry; a wide state with a scalar decay per channel):

==========  ===========================  =====  =========================  ====
name        batch, dim, L, N             I/O    delta = softplus(N(mu,s))  seed
==========  ===========================  =====  =========================  ====
tiny        1, 4, 64, 4                  fp32   mu=-2, s=0.5               0
dim512      1, 512, 8192, 16             fp32   mu=-2, s=0.5               1
bf16_2k     4, 2048, 2048, 16            bf16   mu=-3, s=1                 2
long64k     1, 1536, 65536, 16 (+h0)     fp32   mu=-4, s=0.5               3
wide64      8, 1024, 4096, 64 (scalar A) bf16   mu=-2, s=1                 4
==========  ===========================  =====  =========================  ====

A[d,n] = -(n+1) except bf16_2k (-(n+1)*U(0.5,1.5), drawn per (d,n)) and
wide64 (a_d = -U(1,16) drawn per d, the same for every n).  u, B, C, D ~
N(0,1); h0 ~ N(0, 0.1^2) for long64k, absent (zeros) elsewhere.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    dim: int
    L: int
    N: int
    dtype: str            # "f32" or "bf16" (I/O type of u, delta, B, C, out)
    delta_mu: float
    delta_sigma: float
    A_kind: str           # "s4d" -(n+1) | "s4d_jitter" -(n+1)U(.5,1.5) | "scalar" -U(1,16)
    h0_std: float         # 0 -> no h0
    seed: int

    @property
    def channels(self) -> int:
        return self.batch * self.dim

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.L * self.N

    def scaled(self, *, batch=None, dim=None, L=None, N=None, name=None):
        """The same recipe at other sizes (for oracle-sized parity cases)."""
        return replace(self, batch=batch or self.batch, dim=dim or self.dim,
                       L=L or self.L, N=N or self.N,
                       name=name or f"{self.name}@{batch or self.batch}x"
                       f"{dim or self.dim}x{L or self.L}x{N or self.N}")


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 64, 4, "f32", -2.0, 0.5, "s4d", 0.0, 0),
    "dim512": Workload("dim512", 1, 512, 8192, 16, "f32", -2.0, 0.5, "s4d", 0.0, 1),
    "bf16_2k": Workload("bf16_2k", 4, 2048, 2048, 16, "bf16", -3.0, 1.0,
                        "s4d_jitter", 0.0, 2),
    "long64k": Workload("long64k", 1, 1536, 65536, 16, "f32", -4.0, 0.5, "s4d", 0.1, 3),
    "wide64": Workload("wide64", 8, 1024, 4096, 64, "bf16", -2.0, 1.0, "scalar", 0.0, 4),
}
ORDER = ["tiny", "dim512", "bf16_2k", "long64k", "wide64"]


def io_dtype(dtype: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def make_inputs(w: Workload, seed: int | None = None):
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with u, delta [batch, dim, L]; A [dim, N] fp32;
    B, C [batch, N, L]; D [dim] fp32; h0 [batch, dim, N] fp32 or None.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shp = (w.batch, w.dim, w.L)
    u = torch.randn(shp, generator=g, dtype=torch.float32)
    z = torch.randn(shp, generator=g, dtype=torch.float32)
    delta = F.softplus(z * w.delta_sigma + w.delta_mu)
    n1 = torch.arange(1, w.N + 1, dtype=torch.float32)
    if w.A_kind == "s4d":
        A = (-n1).repeat(w.dim, 1)
    elif w.A_kind == "s4d_jitter":
        jit = torch.rand((w.dim, w.N), generator=g, dtype=torch.float32) + 0.5
        A = -n1[None, :] * jit
    elif w.A_kind == "scalar":
        a_d = -(torch.rand((w.dim, 1), generator=g, dtype=torch.float32) * 15.0 + 1.0)
        A = a_d.expand(w.dim, w.N).contiguous()
    else:
        raise ValueError(f"unknown A recipe {w.A_kind!r}")
    B = torch.randn((w.batch, w.N, w.L), generator=g, dtype=torch.float32)
    C = torch.randn((w.batch, w.N, w.L), generator=g, dtype=torch.float32)
    D = torch.randn((w.dim,), generator=g, dtype=torch.float32)
    h0 = None
    if w.h0_std > 0:
        h0 = torch.randn((w.batch, w.dim, w.N), generator=g,
                         dtype=torch.float32) * w.h0_std
    dt = io_dtype(w.dtype)
    return {
        "u": u.to(dt).contiguous(), "delta": delta.to(dt).contiguous(),
        "A": A.contiguous(), "B": B.to(dt).contiguous(), "C": C.to(dt).contiguous(),
        "D": D.contiguous(), "h0": None if h0 is None else h0.contiguous(),
    }


def make_option_inputs(w: Workload):
    """Inputs of the scan's options for workload ``w`` (a generator of its own,
    seeded ``w.seed + 100``, so the plain inputs stay as they are): the raw
    delta before softplus ~ N(delta_mu, delta_sigma) in the I/O dtype (its
    softplus has the plain recipe's distribution), a per-channel delta bias
    ~ N(0, 0.1^2) float32, and the gate z ~ N(0, 1) in the I/O dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 100)
    shp = (w.batch, w.dim, w.L)
    raw = torch.randn(shp, generator=g, dtype=torch.float32) * w.delta_sigma + w.delta_mu
    bias = torch.randn((w.dim,), generator=g, dtype=torch.float32) * 0.1
    z = torch.randn(shp, generator=g, dtype=torch.float32)
    dt = io_dtype(w.dtype)
    return {"delta_raw": raw.to(dt).contiguous(), "delta_bias": bias.contiguous(),
            "z": z.to(dt).contiguous()}


@dataclass(frozen=True)
class PscanWorkload:
    name: str
    rows: int
    len: int
    seed: int


# The pscan(deltaA, BX) primitive over rows of a materialised scan: decay
# a = exp(-softplus(N(-2, 0.5)) * (r % 16 + 1)) in (0, 1), b ~ N(0, 1), h0 ~ N(0, 1).
PSCAN_WORKLOADS = {
    "pscan_8k": PscanWorkload("pscan_8k", 8192, 8192, 11),
    "pscan_small": PscanWorkload("pscan_small", 37, 1000, 12),
}


def make_pscan_inputs(w: PscanWorkload):
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    z = torch.randn((w.rows, w.len), generator=g, dtype=torch.float32)
    rate = (torch.arange(w.rows, dtype=torch.float32) % 16 + 1.0)[:, None]
    a = torch.exp(-F.softplus(z * 0.5 - 2.0) * rate)
    b = torch.randn((w.rows, w.len), generator=g, dtype=torch.float32)
    h0 = torch.randn((w.rows,), generator=g, dtype=torch.float32)
    return {"a": a.contiguous(), "b": b.contiguous(), "h0": h0.contiguous()}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    N: int
    dtype: str
    seed: int


# One decode step for a batch of 256 sequences of a d_inner = 5120 layer (the
# channel count of a 2.8B-parameter Mamba) with N = 16: bf16 activations, an
# fp32 state cache of 256*5120*16 floats.  Same distributions as the dim512
# recipe; the cached state ~ N(0, 0.5^2).
DECODE_WORKLOAD = DecodeWorkload("decode_b256_d5120", 256, 5120, 16, "bf16", 21)


def make_decode_inputs(w: DecodeWorkload):
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    u = torch.randn((w.batch, w.dim), generator=g, dtype=torch.float32)
    z = torch.randn((w.batch, w.dim), generator=g, dtype=torch.float32)
    delta = F.softplus(z * 0.5 - 2.0)
    A = (-torch.arange(1, w.N + 1, dtype=torch.float32)).repeat(w.dim, 1)
    B = torch.randn((w.batch, w.N), generator=g, dtype=torch.float32)
    C = torch.randn((w.batch, w.N), generator=g, dtype=torch.float32)
    D = torch.randn((w.dim,), generator=g, dtype=torch.float32)
    state = torch.randn((w.batch, w.dim, w.N), generator=g, dtype=torch.float32) * 0.5
    dt = io_dtype(w.dtype)
    return {"u": u.to(dt).contiguous(), "delta": delta.to(dt).contiguous(), "A": A.contiguous(),
            "B": B.to(dt).contiguous(), "C": C.to(dt).contiguous(), "D": D.contiguous(),
            "state": state.contiguous()}
