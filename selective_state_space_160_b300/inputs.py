"""Seeded synthetic inputs for the selective scan, shared by the tests, the bench
and the CPU oracle.

This module holds only the input recipe (random draws, bf16 rounding and the
parameter initialisation); none of the scan's arithmetic lives here.

Recipe (one numpy ``Generator(Philox(seed))`` per problem, draws in this order):
  u, z, B, C, dy, x      ~ N(0, 1)
  delta (raw pre-activation) ~ 0.5 * N(0, 1)
  dt ~ log-uniform[1e-3, 1e-1] per channel (per head for SSD);
  delta_bias = log(expm1(dt)), the inverse softplus, so softplus(bias) = dt
  A[d, n] = -(n + 1)   (S4D-real style initialisation: bqwf survey sec. 2.1 and
                        the study note "Mamba — 选择性状态空间模型" both name
                        HiPPO-style initialisation of A)
  A_h ~ -U[1, 16]      (SSD, one scalar per head)
  D = 1
bf16 inputs are rounded once (round-to-nearest-even) on the host; the GPU gets
the bf16 bit patterns and the oracle the same rounded values.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 160_000


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    lsb = (b >> 16) & 1
    r = ((b + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)).astype(np.uint32)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint32(0x7FC00000)
    return r.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns (uint16) of bf16-representable float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def _normal(g, shape, scale=1.0):
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)).astype(np.float32)


def s6_inputs(batch, dim, seqlen, dstate, seed=SEED_BASE, bf16=False, with_z=True,
              with_D=True, with_bias=True, with_dy=False):
    """Inputs of one S6 problem as float32 numpy arrays (bf16-rounded when bf16)."""
    g = _rng(seed)
    rnd = bf16_round if bf16 else (lambda a: a)
    out = {}
    out["u"] = rnd(_normal(g, (batch, dim, seqlen)))
    out["delta"] = rnd(_normal(g, (batch, dim, seqlen), 0.5))
    z = rnd(_normal(g, (batch, dim, seqlen)))
    out["z"] = z if with_z else None
    out["B"] = rnd(_normal(g, (batch, dstate, seqlen)))
    out["C"] = rnd(_normal(g, (batch, dstate, seqlen)))
    dt = np.exp(g.uniform(np.log(1e-3), np.log(1e-1), size=dim))
    out["delta_bias"] = np.log(np.expm1(dt)).astype(np.float32) if with_bias else None
    out["A"] = np.tile(-np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))
    out["D"] = np.ones(dim, np.float32) if with_D else None
    if with_dy:
        out["dy"] = rnd(_normal(g, (batch, dim, seqlen)))
    return out


def ssd_inputs(batch, seqlen, nheads, headdim, dstate, ngroups=1, seed=SEED_BASE,
               bf16=True, with_z=False, with_D=True, with_bias=True, with_dy=False):
    """Inputs of one SSD (scalar-A, multi-head) problem as float32 numpy arrays
    (with_dy: also an upstream gradient dy shaped like x, drawn last)."""
    g = _rng(seed)
    rnd = bf16_round if bf16 else (lambda a: a)
    out = {}
    out["x"] = rnd(_normal(g, (batch, seqlen, nheads, headdim)))
    out["delta"] = rnd(_normal(g, (batch, seqlen, nheads), 0.5))
    z = rnd(_normal(g, (batch, seqlen, nheads, headdim)))
    out["z"] = z if with_z else None
    out["B"] = rnd(_normal(g, (batch, seqlen, ngroups, dstate)))
    out["C"] = rnd(_normal(g, (batch, seqlen, ngroups, dstate)))
    dt = np.exp(g.uniform(np.log(1e-3), np.log(1e-1), size=nheads))
    out["delta_bias"] = np.log(np.expm1(dt)).astype(np.float32) if with_bias else None
    out["A"] = (-g.uniform(1.0, 16.0, size=nheads)).astype(np.float32)
    out["D"] = np.ones(nheads, np.float32) if with_D else None
    if with_dy:
        out["dy"] = rnd(_normal(g, (batch, seqlen, nheads, headdim)))
    return out


def s6_inputs_torch(batch, dim, seqlen, dstate, seed=SEED_BASE, bf16=False, device="cuda",
                    with_dy=False):
    """Device-side generator for workloads too large to draw on the host
    (the 2^20-step sequence).  Same distributions, drawn by torch's Philox
    generator on the device; the oracle receives copies of sampled rows."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt_ = torch.bfloat16 if bf16 else torch.float32

    def normal(shape, scale=1.0):
        t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        return t.to(dt_)

    out = {}
    out["u"] = normal((batch, dim, seqlen))
    out["delta"] = normal((batch, dim, seqlen), 0.5)
    out["z"] = normal((batch, dim, seqlen))
    out["B"] = normal((batch, dstate, seqlen))
    out["C"] = normal((batch, dstate, seqlen))
    hg = _rng(seed)
    dt = np.exp(hg.uniform(np.log(1e-3), np.log(1e-1), size=dim))
    out["delta_bias"] = torch.from_numpy(np.log(np.expm1(dt)).astype(np.float32)).to(device)
    out["A"] = (-torch.arange(1, dstate + 1, dtype=torch.float32, device=device)).repeat(dim, 1).contiguous()
    out["D"] = torch.ones(dim, dtype=torch.float32, device=device)
    if with_dy:
        out["dy"] = normal((batch, dim, seqlen))
    return out


def conv_taps(dim, width, seed=SEED_BASE):
    """Causal conv1d front-end parameters: weight [dim, width] with unit-variance
    outputs for unit-variance inputs, and a small bias [dim] (float32)."""
    g = _rng(seed)
    w = (_normal(g, (dim, width)) / np.float32(np.sqrt(width))).astype(np.float32)
    b = _normal(g, (dim,), 0.1)
    return w, b
