"""Seeded synthetic inputs for the selective scan.

This module only draws random numbers and lays them out; it holds none of the
scan's arithmetic.  It serves both the CUDA path and the float64 oracle, which
receive identical stored values.

Recipe (shapes of Mamba layers; no trained weights, no dataset):
  x, z         ~ N(0, 1)                      (batch, L, D)
  delta_raw    ~ N(0, 1)                      (batch, L, D)
  dt_d         ~ U[0.001, 0.1]  per channel;  delta_bias = log(expm1(dt_d)),
               the value whose softplus is dt_d (Mamba's step-size init)
  A            = -exp(N(0, variance 0.5)) per (d, n), or S4D-real -(n+1)
  B, C         ~ N(0, 1) per (b, t, n)  (time-varying, shared by channels), or
               ~ N(0, variance 1/N) per (d, n) for the LTI workload
  D            ~ N(0, 1) per channel
  h_init       ~ N(0, 1) per (b, d, n) for the recurrent step workload
Block prologue (``make_conv``, its own generator seeded with seed + 7919):
  conv taps    ~ U[-1/2, 1/2] per (d, k), k = 0..3  (uniform in +-1/sqrt(width))
  conv bias    ~ U[-1/2, 1/2] per channel
  history      ~ N(0, 1) per (b, d, 3), the inputs before the sequence
Draw order: x, delta_raw, dt, A, B, C, D, z, h_init, from numpy's PCG64 seeded
with the workload's seed.
Mamba-2 SSD layer (``make_ssd``; the same distributions with the decay, the step
and D per head):
  x, z         ~ N(0, 1)                      (batch, L, H, P)
  dt_raw       ~ N(0, 1)                      (batch, L, H)
  dt_h         ~ U[0.001, 0.1] per head;  dt_bias = log(expm1(dt_h))
  A            = -exp(N(0, variance 0.5)) per head
  B, C         ~ N(0, 1) per (b, t, group, n)
  D            ~ N(0, 1) per head;  h_init ~ N(0, 1) per (b, h, p, n)
  draw order x, dt_raw, dt, A, B, C, D, z, h_init.  bf16 inputs are the fp32 draws rounded to nearest
even bfloat16 and are carried as raw uint16 bit patterns; A, D, delta_bias and
h_init stay fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest-even bfloat16; return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_u.size, step):
        v = flat_u[i:i + step]
        r = ((v >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
        flat_o[i:i + step] = ((v + r) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    io: str                      # "f32" or "bf16": x, delta, z, time-varying B, C, out
    x: np.ndarray
    delta: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: Optional[np.ndarray]
    z: Optional[np.ndarray]
    delta_bias: Optional[np.ndarray]
    h0: Optional[np.ndarray]
    delta_softplus: bool = True
    per_channel_bc: bool = False
    seed: int = 0
    recipe: dict = field(default_factory=dict)

    @property
    def tokens_channels(self) -> int:
        return self.batch * self.seqlen * self.dim

    @property
    def element_updates(self) -> int:
        return self.tokens_channels * self.dstate

    def algorithmic_bytes(self) -> int:
        """Minimum bytes moved: every input read once, every output written once."""
        e = 2 if self.io == "bf16" else 4
        tc = self.tokens_channels
        per_td = 2 + (1 if self.z is not None else 0) + 1      # x, delta, [z], out
        nbytes = tc * per_td * e
        if self.per_channel_bc:
            nbytes += 2 * self.dim * self.dstate * 4
        else:
            nbytes += 2 * self.batch * self.seqlen * self.dstate * e
        nbytes += self.dim * self.dstate * 4                      # A
        nbytes += self.dim * 4 * ((self.D is not None) + (self.delta_bias is not None))
        state = self.batch * self.dim * self.dstate * 4
        nbytes += state * (2 if self.h0 is not None else 1)       # final_state (+ h_init)
        return int(nbytes)


def make_workload(name: str, batch: int, seqlen: int, dim: int, dstate: int, *,
                  io: str = "f32", seed: int = 0, a_init: str = "random",
                  gate: bool = True, lti: bool = False, state_in: bool = False,
                  with_D: bool = True, with_bias: bool = True) -> Workload:
    """Draw one workload following the module recipe."""
    assert io in ("f32", "bf16")
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = (batch, seqlen, dim)
    x = rng.standard_normal(shp, dtype=np.float32)
    delta_raw = None if lti else rng.standard_normal(shp, dtype=np.float32)
    dt = rng.uniform(0.001, 0.1, size=dim)
    if a_init == "random":
        A = -np.exp(rng.normal(0.0, np.sqrt(0.5), size=(dim, dstate)))
    elif a_init == "s4d_real":
        A = -np.tile(np.arange(1, dstate + 1, dtype=np.float64), (dim, 1))
    else:
        raise ValueError(a_init)
    A = A.astype(np.float32)
    if lti:
        B = rng.normal(0.0, np.sqrt(1.0 / dstate), size=(dim, dstate)).astype(np.float32)
        C = rng.normal(0.0, np.sqrt(1.0 / dstate), size=(dim, dstate)).astype(np.float32)
    else:
        B = rng.standard_normal((batch, seqlen, dstate), dtype=np.float32)
        C = rng.standard_normal((batch, seqlen, dstate), dtype=np.float32)
    D = rng.standard_normal(dim, dtype=np.float32) if with_D else None
    z = rng.standard_normal(shp, dtype=np.float32) if gate else None
    h0 = rng.standard_normal((batch, dim, dstate), dtype=np.float32) if state_in else None

    if lti:
        # constant step per channel, passed as delta with softplus off and no bias
        delta = np.broadcast_to(dt.astype(np.float32), shp).copy()
        bias = None
        softplus = False
    else:
        delta = delta_raw
        bias = np.log(np.expm1(dt)).astype(np.float32) if with_bias else None
        softplus = True

    if io == "bf16":
        x = f32_to_bf16_bits(x)
        delta = f32_to_bf16_bits(delta)
        z = None if z is None else f32_to_bf16_bits(z)
        if not lti:
            B, C = f32_to_bf16_bits(B), f32_to_bf16_bits(C)
    return Workload(name=name, batch=batch, seqlen=seqlen, dim=dim, dstate=dstate,
                    io=io, x=x, delta=delta, A=A, B=B, C=C, D=D, z=z,
                    delta_bias=bias, h0=h0, delta_softplus=softplus,
                    per_channel_bc=lti, seed=seed,
                    recipe=dict(a_init=a_init, gate=gate, lti=lti, state_in=state_in,
                                with_D=with_D, with_bias=with_bias))


# The five scan workloads and the recurrent-step workload (sizes from the
# Mamba-shaped layers they stand for), plus a shortened long-context case for
# profiler captures.
CONFIGS = {
    "tiny_f32": dict(batch=1, seqlen=256, dim=16, dstate=4, io="f32", seed=0,
                     a_init="random", gate=True),
    "lti_f32": dict(batch=2, seqlen=2048, dim=64, dstate=16, io="f32", seed=1,
                    a_init="s4d_real", gate=False, lti=True, with_bias=False),
    "mamba130m_f32": dict(batch=8, seqlen=2048, dim=1536, dstate=16, io="f32", seed=2,
                          a_init="s4d_real", gate=True),
    "mamba1p4b_bf16": dict(batch=4, seqlen=4096, dim=4096, dstate=16, io="bf16", seed=3,
                           a_init="random", gate=True),
    "long_bf16": dict(batch=1, seqlen=131072, dim=2560, dstate=16, io="bf16", seed=4,
                      a_init="random", gate=True),
    "step_bf16": dict(batch=256, seqlen=1, dim=2560, dstate=16, io="bf16", seed=5,
                      a_init="random", gate=True, state_in=True),
    # the long-context layer cut to 16384 steps (inputs 252 MB, still larger than L2):
    # the size used for full profiler captures, which replay each launch ~40 times
    "long_bf16_16k": dict(batch=1, seqlen=16384, dim=2560, dstate=16, io="bf16", seed=4,
                          a_init="random", gate=True),
}


@dataclass
class ConvPrologue:
    w: np.ndarray                # (dim, 4) fp32, tap k multiplies the input k steps back
    b: Optional[np.ndarray]      # (dim,) fp32
    hist: Optional[np.ndarray]   # (batch, dim, 3) fp32, oldest first


def make_conv(w: Workload, *, with_bias: bool = True, hist: bool = False, width: int = 4) -> ConvPrologue:
    """Draw the block prologue's taps, bias and input history for a workload."""
    rng = np.random.Generator(np.random.PCG64(w.seed + 7919))
    bound = 1.0 / np.sqrt(width)
    taps = rng.uniform(-bound, bound, size=(w.dim, width)).astype(np.float32)
    bias = rng.uniform(-bound, bound, size=w.dim).astype(np.float32)
    h = rng.standard_normal((w.batch, w.dim, width - 1), dtype=np.float32)
    return ConvPrologue(taps, bias if with_bias else None, h if hist else None)


def config(name: str) -> Workload:
    return make_workload(name, **CONFIGS[name])


@dataclass
class SsdWorkload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    io: str
    x: np.ndarray                 # (batch, L, H, P)
    dt: np.ndarray                # (batch, L, H), raw step before bias and softplus
    A: np.ndarray                 # (H,) fp32, one decay rate per head
    B: np.ndarray                 # (batch, L, G, N)
    C: np.ndarray                 # (batch, L, G, N)
    D: Optional[np.ndarray]       # (H,) fp32
    z: Optional[np.ndarray]       # (batch, L, H, P)
    dt_bias: Optional[np.ndarray]  # (H,) fp32
    h0: Optional[np.ndarray]      # (batch, H, P, N) fp32
    dt_softplus: bool = True
    seed: int = 0

    @property
    def tokens_channels(self) -> int:
        return self.batch * self.seqlen * self.nheads * self.headdim


def make_ssd(name: str, batch: int, seqlen: int, nheads: int, headdim: int, dstate: int, *,
             ngroups: int = 1, io: str = "bf16", seed: int = 0, gate: bool = True,
             state_in: bool = False, with_D: bool = True, with_bias: bool = True) -> SsdWorkload:
    """Draw one Mamba-2 SSD workload following the module recipe."""
    assert io == "bf16" and nheads % ngroups == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = (batch, seqlen, nheads, headdim)
    x = rng.standard_normal(shp, dtype=np.float32)
    dt_raw = rng.standard_normal((batch, seqlen, nheads), dtype=np.float32)
    dt = rng.uniform(0.001, 0.1, size=nheads)
    A = (-np.exp(rng.normal(0.0, np.sqrt(0.5), size=nheads))).astype(np.float32)
    B = rng.standard_normal((batch, seqlen, ngroups, dstate), dtype=np.float32)
    C = rng.standard_normal((batch, seqlen, ngroups, dstate), dtype=np.float32)
    D = rng.standard_normal(nheads, dtype=np.float32) if with_D else None
    z = rng.standard_normal(shp, dtype=np.float32) if gate else None
    h0 = (rng.standard_normal((batch, nheads, headdim, dstate), dtype=np.float32)
          if state_in else None)
    bias = np.log(np.expm1(dt)).astype(np.float32) if with_bias else None
    return SsdWorkload(name=name, batch=batch, seqlen=seqlen, nheads=nheads, headdim=headdim,
                       ngroups=ngroups, dstate=dstate, io=io, x=f32_to_bf16_bits(x),
                       dt=f32_to_bf16_bits(dt_raw), A=A, B=f32_to_bf16_bits(B),
                       C=f32_to_bf16_bits(C), D=D,
                       z=None if z is None else f32_to_bf16_bits(z), dt_bias=bias, h0=h0,
                       seed=seed)


# Mamba-2-shaped SSD layers: 2.7B-like (d_inner 5120 = 80 heads of 64, N 128, one
# group) and the same width with N 256 (the state size the pages give for Mamba-2).
SSD_CONFIGS = {
    "ssd_tiny": dict(batch=1, seqlen=200, nheads=4, headdim=64, dstate=64, seed=20),
    "mamba2_2p7b_bf16": dict(batch=4, seqlen=4096, nheads=80, headdim=64, dstate=128, seed=21),
    "mamba2_n256_bf16": dict(batch=4, seqlen=4096, nheads=80, headdim=64, dstate=256, seed=22),
}
