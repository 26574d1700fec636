"""Seeded synthetic inputs for the SSD forward, shaped like the Mamba-2 layers.

This module only draws random numbers and fixes shapes; it holds none of the
layer's arithmetic.  It is the one module that both the CUDA-side harness and
the CPU oracle's tests read their inputs from.

Distributions: x, B, C ~ N(0, 1); dt = exp(U(ln lo, ln hi)) per (batch, token,
head) (a positive step size, as produced upstream by a softplus); A_h =
-exp(U(0, ln 16)) (negative, so every decay factor is in (0, 1)); D_h ~ N(0, 1);
init_state ~ N(0, 1) where a workload carries state in.  Draw order: x, B, C,
dt, A, D, init_state, all from one CPU ``torch.Generator``.  For bf16 workloads
x, B and C are rounded to bf16 before either side sees them.

The 2.7B-shaped layer (d_model 2560, expand 2 -> d_inner 5120 = 80 heads x
headdim 64, state 64) follows the model configuration printed in
"Mamba-2架构深度解析" §3.1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

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
    dtype: str                 # "f32" or "bf16": element type of x, B, C, y
    dt_range: tuple = (1e-3, 1e-1)
    with_init: bool = False
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


WORKLOADS = [
    Workload("tiny_f32_b1_L256_H4_P16_N16", 1, 256, 4, 16, 16, 1, 64, "f32", seed=20260,
             note="small fp32 case for full element-by-element parity"),
    Workload("mamba2_2p7b_b2_L2048_H80_P64_N64", 2, 2048, 80, 64, 64, 1, 128, "bf16", seed=20261,
             note="Mamba-2 2.7B-shaped SSD layer (d_inner 5120), headline workload"),
    Workload("state128_b1_L8192_H80_P64_N128", 1, 8192, 80, 64, 128, 1, 256, "bf16", seed=20262,
             note="larger-state layer"),
    Workload("long_b1_L131072_H24_P64_N256", 1, 131072, 24, 64, 256, 1, 256, "bf16",
             dt_range=(1e-4, 1e-2), seed=20263,
             note="long sequence, big state; decay spans many chunks"),
    Workload("grouped_b16_L4096_H32_P128_N128_G8", 16, 4096, 32, 128, 128, 8, 128, "bf16",
             with_init=True, seed=20264,
             note="grouped B/C (4 heads per group) with state carried in and out"),
]

HEADLINE = WORKLOADS[1]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def make_inputs(batch, seqlen, nheads, headdim, dstate, ngroups, dtype="bf16", seed=0,
                dt_range=(1e-3, 1e-1), with_init=False, with_D=True):
    """Draw one seeded input set on the CPU.

    Returns a dict with x [b,L,H,P], dt [b,L,H] fp32, A [H] fp32, B, C [b,L,G,N],
    D [H] fp32 (or None), init_state [b,H,P,N] fp32 (or None).  x, B, C have the
    requested element type (already rounded for bf16).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    el = torch_dtype(dtype)
    x = torch.randn(batch, seqlen, nheads, headdim, generator=g, dtype=torch.float32).to(el)
    B = torch.randn(batch, seqlen, ngroups, dstate, generator=g, dtype=torch.float32).to(el)
    C = torch.randn(batch, seqlen, ngroups, dstate, generator=g, dtype=torch.float32).to(el)
    lo, hi = math.log(dt_range[0]), math.log(dt_range[1])
    dt = torch.exp(torch.empty(batch, seqlen, nheads, dtype=torch.float32).uniform_(lo, hi, generator=g))
    A = -torch.exp(torch.empty(nheads, dtype=torch.float32).uniform_(0.0, math.log(16.0), generator=g))
    D = torch.randn(nheads, generator=g, dtype=torch.float32)
    init = (torch.randn(batch, nheads, headdim, dstate, generator=g, dtype=torch.float32)
            if with_init else None)
    return {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D if with_D else None,
            "init_state": init}


def make_varlen_inputs(lengths, nheads, headdim, dstate, ngroups, dtype="bf16", seed=0,
                       dt_range=(1e-3, 1e-1), with_init=False, with_D=True):
    """Draw one seeded packed input set on the CPU: the sequences of ``lengths``
    back to back along one token dimension.

    Returns the dict of ``make_inputs`` with the batch dimension dropped (x
    [T,H,P], dt [T,H], B, C [T,G,N]; init_state [nseq,H,P,N] or None) plus
    ``cu_seqlens`` (a list of nseq + 1 offsets).
    """
    lengths = [int(v) for v in lengths]
    T = sum(lengths)
    d = make_inputs(1, T, nheads, headdim, dstate, ngroups, dtype, seed, dt_range, False, with_D)
    out = {k: (v[0] if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    if with_init:
        g = torch.Generator(device="cpu")
        g.manual_seed(int(seed) + 1)
        out["init_state"] = torch.randn(len(lengths), nheads, headdim, dstate, generator=g, dtype=torch.float32)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    out["cu_seqlens"] = cu
    return out


def varlen_lengths(total, nseq, seed, min_len=1):
    """Seeded mix of nseq sequence lengths summing to total: lengths drawn
    log-uniformly (short and long sequences together), then rescaled."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    w = torch.exp(torch.empty(nseq, dtype=torch.float64).uniform_(0.0, math.log(64.0), generator=g))
    raw = (w / w.sum() * (total - nseq * min_len)).floor().long() + min_len
    raw[-1] += total - int(raw.sum())
    return [int(v) for v in raw]


def workload_inputs(w: Workload):
    return make_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.dtype,
                       w.seed, w.dt_range, w.with_init)


def sample_rows(w_or_dims, count: int, seed: int = 7):
    """Seeded sample of flat row ids (b*H + h)*P + p, always including the
    first and last row and at least one row of every group."""
    if isinstance(w_or_dims, Workload):
        b, H, P, G = w_or_dims.batch, w_or_dims.nheads, w_or_dims.headdim, w_or_dims.ngroups
    else:
        b, H, P, G = w_or_dims
    total = b * H * P
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    rows = set([0, total - 1])
    hpg = H // G
    for grp in range(G):
        h = grp * hpg + int(torch.randint(0, hpg, (1,), generator=g))
        bb = int(torch.randint(0, b, (1,), generator=g))
        p = int(torch.randint(0, P, (1,), generator=g))
        rows.add((bb * H + h) * P + p)
    while len(rows) < min(count, total):
        rows.add(int(torch.randint(0, total, (1,), generator=g)))
    return sorted(rows)


def make_cotangents(batch, seqlen, nheads, headdim, dstate, dtype="bf16", seed=0, with_dfinal=True):
    """Draw the incoming gradients of a backward: dy [b,L,H,P] ~ N(0, 1) in the
    element type of x (rounded to bf16 for bf16 workloads) and dfinal
    [b,H,P,N] ~ N(0, 1) fp32 (or None).  One CPU generator, draw order dy, dfinal."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    dy = torch.randn(batch, seqlen, nheads, headdim, generator=g, dtype=torch.float32).to(torch_dtype(dtype))
    dfinal = (torch.randn(batch, nheads, headdim, dstate, generator=g, dtype=torch.float32)
              if with_dfinal else None)
    return dy, dfinal
