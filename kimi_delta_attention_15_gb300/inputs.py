"""Seeded synthetic workloads for the KDA gated delta rule (K = V = 128).

This module only draws random numbers and shapes tensors. It holds none of
the method's arithmetic, so both the fp64 oracle tests and the CUDA path can
use it without sharing any computation.

Workloads follow the shapes admitted by the flashinfer ``kda_backward`` page
("Supported contract"): fixed B=1,T=17,H=1; packed lengths [17,33,65] at H=4;
fixed B=1,T=4096,H=32; fixed B=1,T=8192,H=96; packed lengths
[1300,547,2048,963,271,3063] at H=96. Extra admitted shapes (B=1,T=17,H=16;
B=1,T=1024,H=4; eight packed sequences of 1024 at H=96) are listed too.

Layouts (packed, B=1; H counts value heads, q and k hold H / groups heads):
  q, k              [T, H / groups, 128]  bf16
  g_raw, do         [T, H, 128]  bf16
  v                 [T, H, 128]  bf16
  beta_raw          [T, H]       bf16
  A_log             [H]          fp32   log(U[1,16])
  dt_bias           [H, 128]     fp32   0.1 * N(0,1)
  h0, dhT           [N, H, 128, 128] fp32 value-first, or None (= zero)
  cu_seqlens        [N + 1]      int64

Draw order is fixed: q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, do, dhT,
all in fp32 from one CPU ``torch.Generator`` seeded with ``seed``; token
tensors are then rounded to bf16. The same seed gives the same tensors on
every machine.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

D = 128            # key and value head dimension
BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple          # per-sequence token counts (packed when len > 1)
    H: int
    g_std: float = 1.0      # std of g_raw
    h0: bool = False        # draw h0 ~ 0.1 N(0,1)
    dhT: bool = False       # draw dhT ~ 0.1 N(0,1)
    packed: bool = False    # inputs given as packed varlen with offsets
    groups: int = 1         # value heads per query/key head (q, k: H // groups heads)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def token_heads(self) -> int:
        return self.T * self.H


# The five workloads the method is measured and checked on, in order.
WORKLOADS = [
    Workload("fixed_T17_H1", (17,), 1),
    Workload("varlen_17_33_65_H4", (17, 33, 65), 4, h0=True, dhT=True, packed=True),
    Workload("fixed_T4096_H32", (4096,), 32, g_std=2.0),
    Workload("fixed_T8192_H96", (8192,), 96),
    Workload("varlen_6seq_T8192_H96", (1300, 547, 2048, 963, 271, 3063), 96,
             h0=True, dhT=True, packed=True),
]

# Further shapes admitted on the flashinfer page (parity cases only).
EXTRA_WORKLOADS = [
    Workload("fixed_T17_H16", (17,), 16),
    Workload("fixed_T1024_H4", (1024,), 4),
    Workload("varlen_8x1024_H96", (1024,) * 8, 96, h0=True, dhT=True, packed=True),
]

HEADLINE = 3   # index of fixed_T8192_H96 in WORKLOADS


def custom(lengths, H, g_std=1.0, h0=False, dhT=False, name=None, groups=1) -> Workload:
    """A workload of arbitrary packed lengths (tests of edge cases)."""
    lengths = tuple(int(x) for x in lengths)
    tag = f"_G{groups}" if groups > 1 else ""
    return Workload(name or f"custom_{'_'.join(map(str, lengths))}_H{H}{tag}", lengths, H,
                    g_std=g_std, h0=h0, dhT=dhT, packed=len(lengths) > 1, groups=groups)


def cu_seqlens(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int64)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw the seeded inputs of workload ``w`` as CPU tensors."""
    if seed is None:
        idx = WORKLOADS.index(w) if w in WORKLOADS else 0
        seed = BASE_SEED + idx
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    T, H, N = w.T, w.H, w.N

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    Hqk = H // w.groups          # grouped value heads: fewer query/key heads
    q = randn(T, Hqk, D)
    k = randn(T, Hqk, D)
    v = randn(T, H, D)
    g_raw = randn(T, H, D) * w.g_std
    beta_raw = randn(T, H)
    A_log = torch.log(torch.rand(H, generator=gen, dtype=torch.float32) * 15.0 + 1.0)
    dt_bias = randn(H, D) * 0.1
    h0 = randn(N, H, D, D) * 0.1 if w.h0 else None
    do = randn(T, H, D)
    dhT = randn(N, H, D, D) * 0.1 if w.dhT else None
    bf = torch.bfloat16
    return dict(
        q=q.to(bf), k=k.to(bf), v=v.to(bf), g_raw=g_raw.to(bf), beta_raw=beta_raw.to(bf),
        A_log=A_log, dt_bias=dt_bias, h0=h0, do=do.to(bf), dhT=dhT,
        cu_seqlens=cu_seqlens(w.lengths), lengths=list(w.lengths), H=H, T=T, N=N,
    )
