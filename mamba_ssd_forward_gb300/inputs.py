"""Seeded synthetic inputs and the named workloads.

This module holds no arithmetic of the method: it only draws random tensors
with the value distributions below and rounds them to the storage dtype.
Both the CUDA path and the float64 oracle consume what it returns.

Value distributions (every workload):
    x, B, C ~ N(0, 1)
    dt      = exp(U(ln 1e-3, ln 1e-1))          (so dt > 0)
    A       = -exp(U(ln 1, ln 16))              (so A < 0, a_t = A dt < 0)
    D       ~ N(0, 1)
    h0      ~ N(0, 0.1^2) when the workload has an initial state, else none

Draw order is fixed -- x, dt, A, B, C, D, h0 -- from one CPU
``torch.Generator`` seeded with ``seed``, in float64.  x, dt, B and C are
then rounded to the I/O dtype (bf16 or fp32); A, D and h0 to fp32, which is
what the library takes for them.  The oracle receives the rounded values
upcast exactly to float64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str          # "fp32" or "bf16": storage type of x, dt, B, C, y
    has_h0: bool

    @property
    def nchunks(self) -> int:
        return (self.seqlen + self.chunk - 1) // self.chunk

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The four named layer shapes and the shape sweep.
TINY = Workload("tiny_fp32_b1_L256_h2_P16_S16_T64", 1, 256, 2, 16, 16, 1, 64, "fp32", False)
MAMBA2_130M = Workload("mamba2_130m_layer_b4_L2048_h24_P64_S128_T256_bf16",
                       4, 2048, 24, 64, 128, 1, 256, "bf16", False)
MAMBA2_2P7B = Workload("mamba2_2p7b_layer_b2_L4096_h80_P64_S128_T256_bf16_h0",
                       2, 4096, 80, 64, 128, 1, 256, "bf16", True)
LONG_32K = Workload("long_context_b1_L32768_h48_P64_S256_g8_T256_bf16",
                    1, 32768, 48, 64, 256, 8, 256, "bf16", False)

NAMED = [TINY, MAMBA2_130M, MAMBA2_2P7B, LONG_32K]


def sweep() -> list[Workload]:
    """batch 2, nheads 32, P 64, ngroups 1, nonzero h0; S x L x T x dtype."""
    out = []
    for dtype in ("fp32", "bf16"):
        for S in (64, 128, 256):
            for L in (1024, 4096, 16384, 4000):
                for T in (128, 256):
                    out.append(Workload(f"sweep_{dtype}_S{S}_L{L}_T{T}", 2, L, 32, 64, S, 1, T, dtype, True))
    return out


def torch_dtype(name: str) -> torch.dtype:
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw one seeded input set for workload ``w`` on the CPU.

    Returns a dict of CPU tensors: x, dt, B, C in the I/O dtype, A, D in
    fp32 and h0 in fp32 (or None)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    b, L, nh, P, S, ng = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    f64 = torch.float64

    def uniform(shape, lo, hi):
        return lo + (hi - lo) * torch.rand(shape, generator=g, dtype=f64)

    x = torch.randn((b, L, nh, P), generator=g, dtype=f64)
    dt = torch.exp(uniform((b, L, nh), math.log(1e-3), math.log(1e-1)))
    A = -torch.exp(uniform((nh,), math.log(1.0), math.log(16.0)))
    B = torch.randn((b, L, ng, S), generator=g, dtype=f64)
    C = torch.randn((b, L, ng, S), generator=g, dtype=f64)
    D = torch.randn((nh,), generator=g, dtype=f64)
    h0 = 0.1 * torch.randn((b, nh, P, S), generator=g, dtype=f64) if w.has_h0 else None

    io = torch_dtype(w.dtype)
    return {
        "x": x.to(io), "dt": dt.to(io), "A": A.float(),
        "B": B.to(io), "C": C.to(io), "D": D.float(),
        "h0": None if h0 is None else h0.float(),
    }
