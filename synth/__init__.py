"""Seeded synthetic inputs for the state-passing mixer forward and decode update.

This module is shared by the GPU path's tests and benchmark and by the CPU
oracle's tests.  It holds none of the method's arithmetic: it only draws
random numbers, rounds each one once to the storage type of the run and lays
the arrays out.  Nothing here computes a convolution, a decay, a state or an
output.

Storage types
-------------
* ``"f32"`` arrays are ``numpy.float32``.
* ``"bf16"`` arrays are ``numpy.uint16`` holding bfloat16 bit patterns
  (float64 draw -> float32 round-to-nearest-even -> bfloat16
  round-to-nearest-even).  ``Arr.f64()`` gives the exact float64 value of every
  element, which is what the oracle consumes.

Distributions (one recipe for every workload; shapes vary)
----------------------------------------------------------
x ~ N(0,1); B, C ~ N(0,1); dt = softplus(N(0,1) - 2) (already positive);
A_h ~ -U(0.01, 1) one value per head; conv weight w ~ N(0, 0.5) (variance
0.5); conv bias = 0.1 for every channel; optional Gaussian initial states
h0 ~ N(0, 0.1^2) (fp32) and conv state ~ N(0, 1) (activation type).
Full Mamba-2 wiring: xBC and z ~ N(0,1), dt_raw ~ N(0,1) - 2 (before its bias
and softplus), dt_bias ~ U(-0.5, 0.5) and D_skip ~ U(0.5, 1.5) per head, conv
weight ~ N(0, 0.5) and bias 0.1 over every xBC channel.
Decode pools: conv pool ~ N(0,1), SSM pool ~ N(0, 0.1^2), slot map = the
first Bz entries of a random permutation of the pool rows, cache_seqlens ~
integers uniform on [0, 10000).

Layouts (row-major, last index fastest)
---------------------------------------
x, u, y: [Bz, L, H*P];  B, C: [Bz, L, G, N];  dt: [Bz, L, H];  A: [H];
w: [D, K];  bias: [D];  conv state: [Bz, D, K-1] oldest -> newest;
SSM state: [Bz, H, P, N];  conv pool: [pool, D, S_len];  SSM pool:
[pool, H, P, N].
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "Arr", "f32", "bf16", "rng", "MixerShape", "DecodeShape", "WORKLOADS",
    "DECODE", "mixer_params", "mixer_segment", "mixer_initial_states",
    "decode_inputs", "bf16_bits_from_f32", "bf16_bits_to_f64", "mamba2_inputs",
]


# ----------------------------------------------------------------------------
# storage types
# ----------------------------------------------------------------------------

def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    is_nan = np.isnan(a)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    r[is_nan] = 0x7FC0
    return r


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 bit patterns."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Arr:
    """An array as it is stored in memory: ``data`` and its storage ``dtype``."""

    data: np.ndarray
    dtype: str  # "f32" | "bf16" | "i32"

    @property
    def shape(self):
        return self.data.shape

    def f64(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f64(self.data)
        return self.data.astype(np.float64)

    @property
    def nbytes(self) -> int:
        return int(self.data.nbytes)


def f32(v: np.ndarray) -> Arr:
    return Arr(np.ascontiguousarray(v, dtype=np.float32), "f32")


def bf16(v: np.ndarray) -> Arr:
    return Arr(bf16_bits_from_f32(np.asarray(v, dtype=np.float32)), "bf16")


def store(v: np.ndarray, dtype: str) -> Arr:
    return bf16(v) if dtype == "bf16" else f32(v)


def rng(seed: int, name: str, part: int = 0) -> np.random.Generator:
    """Independent stream per (seed, tensor name, part) so that a segment or a
    slice can be drawn without drawing the rest."""
    return np.random.default_rng([int(seed), zlib.crc32(name.encode()), int(part)])


# ----------------------------------------------------------------------------
# workload shapes
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class MixerShape:
    """A prefill / streaming workload: ``segments`` tokens per call, the state
    of one call passed to the next."""

    name: str
    dtype: str            # activation storage type: "f32" or "bf16"
    Bz: int
    segments: tuple       # tokens per consecutive call
    H: int
    P: int
    N: int
    G: int = 1
    K: int = 4
    gaussian_init: bool = False   # h0 ~ N(0, .1^2), conv state ~ N(0, 1)
    seed: int = 0

    @property
    def D(self) -> int:
        return self.H * self.P

    @property
    def L(self) -> int:
        return int(sum(self.segments))

    def with_(self, **kw) -> "MixerShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    """A continuous-batching decode update over a circular conv-state pool."""

    name: str
    dtype: str
    Bz: int          # active requests
    pool: int        # pool rows
    L_new: int
    H: int
    P: int
    N: int
    G: int = 1
    K: int = 4
    S_len: int = 4
    max_seqlen: int = 10000
    seed: int = 0

    @property
    def D(self) -> int:
        return self.H * self.P

    def with_(self, **kw) -> "DecodeShape":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny fp32 check, three Mamba-2-like prefill /
# streaming layers (370M-, 1.3B- and 780M-like) and a continuous-batching
# decode update.  Seeds are 1000 + workload number.
WORKLOADS: Dict[str, MixerShape] = {
    "tiny_f32": MixerShape("tiny_f32", "f32", Bz=1, segments=(32, 32), H=2, P=4,
                           N=8, seed=1001),
    "m370m_2k": MixerShape("m370m_2k", "bf16", Bz=8, segments=(1024, 1024), H=32,
                           P=64, N=128, seed=1002),
    "m1p3b_8k": MixerShape("m1p3b_8k", "bf16", Bz=4, segments=(8192,), H=64,
                           P=64, N=128, gaussian_init=True, seed=1003),
    "m780m_128k": MixerShape("m780m_128k", "bf16", Bz=1, segments=(2048,) * 64,
                             H=48, P=64, N=128, seed=1004),
}

DECODE: Dict[str, DecodeShape] = {
    "decode_256x1": DecodeShape("decode_256x1", "bf16", Bz=256, pool=512, L_new=1,
                                H=64, P=64, N=128, seed=1005),
    "decode_256x4": DecodeShape("decode_256x4", "bf16", Bz=256, pool=512, L_new=4,
                                H=64, P=64, N=128, seed=1005),
}


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------

def _softplus(v: np.ndarray) -> np.ndarray:
    # input preparation: the method takes dt already positive
    return np.logaddexp(0.0, v)


def mixer_params(s: MixerShape) -> Dict[str, Arr]:
    """Per-layer parameters: A [H] (fp32, < 0), conv w [D, K], bias [D]."""
    A = -rng(s.seed, "A").uniform(0.01, 1.0, size=s.H)
    w = rng(s.seed, "w").normal(0.0, np.sqrt(0.5), size=(s.D, s.K))
    bias = np.full(s.D, 0.1)
    return {"A": f32(A), "w": f32(w), "bias": f32(bias)}


def mixer_segment(s: MixerShape, seg: int, Bz: Optional[slice] = None) -> Dict[str, Arr]:
    """Inputs of segment ``seg``: x [Bz, Ls, D], dt [Bz, Ls, H], B, C [Bz, Ls, G, N]."""
    Ls = s.segments[seg]
    x = rng(s.seed, "x", seg).standard_normal((s.Bz, Ls, s.D))
    dt = _softplus(rng(s.seed, "dt", seg).standard_normal((s.Bz, Ls, s.H)) - 2.0)
    B = rng(s.seed, "B", seg).standard_normal((s.Bz, Ls, s.G, s.N))
    C = rng(s.seed, "C", seg).standard_normal((s.Bz, Ls, s.G, s.N))
    out = {"x": store(x, s.dtype), "dt": store(dt, s.dtype),
           "B": store(B, s.dtype), "C": store(C, s.dtype)}
    if Bz is not None:
        out = {k: Arr(np.ascontiguousarray(v.data[Bz]), v.dtype) for k, v in out.items()}
    return out


def mixer_initial_states(s: MixerShape) -> Dict[str, Arr]:
    """Conv state [Bz, D, K-1] (activation type) and h0 [Bz, H, P, N] (fp32)."""
    if s.gaussian_init:
        S = rng(s.seed, "conv_state").standard_normal((s.Bz, s.D, s.K - 1))
        h0 = rng(s.seed, "h0").normal(0.0, 0.1, size=(s.Bz, s.H, s.P, s.N))
    else:
        S = np.zeros((s.Bz, s.D, s.K - 1))
        h0 = np.zeros((s.Bz, s.H, s.P, s.N))
    return {"conv_state": store(S, s.dtype), "h0": f32(h0)}


def decode_inputs(s: DecodeShape) -> Dict[str, Arr]:
    """Pools, slot map, lengths and the new tokens of one decode call."""
    conv_pool = rng(s.seed, "conv_pool").standard_normal((s.pool, s.D, s.S_len))
    ssm_pool = rng(s.seed, "ssm_pool").normal(0.0, 0.1, size=(s.pool, s.H, s.P, s.N))
    idx = rng(s.seed, "conv_state_indices").permutation(s.pool)[: s.Bz]
    seqlens = rng(s.seed, "cache_seqlens").integers(0, s.max_seqlen, size=s.Bz)
    x = rng(s.seed, "x_new", s.L_new).standard_normal((s.Bz, s.L_new, s.D))
    dt = _softplus(rng(s.seed, "dt_new", s.L_new).standard_normal((s.Bz, s.L_new, s.H)) - 2.0)
    B = rng(s.seed, "B_new", s.L_new).standard_normal((s.Bz, s.L_new, s.G, s.N))
    C = rng(s.seed, "C_new", s.L_new).standard_normal((s.Bz, s.L_new, s.G, s.N))
    A = -rng(s.seed, "A").uniform(0.01, 1.0, size=s.H)
    w = rng(s.seed, "w").normal(0.0, np.sqrt(0.5), size=(s.D, s.K))
    return {
        "conv_pool": store(conv_pool, s.dtype),
        "ssm_pool": f32(ssm_pool),
        "conv_state_indices": Arr(idx.astype(np.int32), "i32"),
        "cache_seqlens": Arr(seqlens.astype(np.int32), "i32"),
        "x": store(x, s.dtype), "dt": store(dt, s.dtype),
        "B": store(B, s.dtype), "C": store(C, s.dtype),
        "A": f32(A), "w": f32(w), "bias": f32(np.full(s.D, 0.1)),
    }


def shrink(s, **kw):
    """Same recipe at other sizes (tests use this for oracle-sized cases)."""
    return s.with_(**kw)


def mamba2_inputs(s: MixerShape, seg: int = 0, Bz: Optional[slice] = None) -> Dict[str, Arr]:
    """Inputs of segment ``seg`` of the full Mamba-2 wiring for the shape of
    ``s`` (its segment lengths, H, P, N, G, K, dtype): xBC [Bz, Ls, D + 2 G N],
    z [Bz, Ls, D], dt_raw [Bz, Ls, H]; and, independent of the segment,
    dt_bias, A, D_skip [H], conv w [D + 2 G N, K], bias [D + 2 G N], conv state
    [Bz, D + 2 G N, K-1] and h0 [Bz, H, P, N] (zeros unless s.gaussian_init)."""
    Ls = s.segments[seg]
    Dt = s.D + 2 * s.G * s.N
    xBC = rng(s.seed, "m2_xBC", seg).standard_normal((s.Bz, Ls, Dt))
    z = rng(s.seed, "m2_z", seg).standard_normal((s.Bz, Ls, s.D))
    dt_raw = rng(s.seed, "m2_dt", seg).standard_normal((s.Bz, Ls, s.H)) - 2.0
    out = {"xBC": store(xBC, s.dtype), "z": store(z, s.dtype), "dt_raw": store(dt_raw, s.dtype)}
    if Bz is not None:
        out = {k: Arr(np.ascontiguousarray(v.data[Bz]), v.dtype) for k, v in out.items()}
    nb = s.Bz if Bz is None else len(range(*Bz.indices(s.Bz)))
    rows = slice(0, s.Bz) if Bz is None else Bz
    if s.gaussian_init:
        S = rng(s.seed, "m2_conv_state").standard_normal((s.Bz, Dt, s.K - 1))[rows]
        h0 = rng(s.seed, "m2_h0").normal(0.0, 0.1, size=(s.Bz, s.H, s.P, s.N))[rows]
    else:
        S = np.zeros((nb, Dt, s.K - 1))
        h0 = np.zeros((nb, s.H, s.P, s.N))
    out.update({
        "dt_bias": f32(rng(s.seed, "m2_dt_bias").uniform(-0.5, 0.5, s.H)),
        "A": f32(-rng(s.seed, "A").uniform(0.01, 1.0, size=s.H)),
        "D_skip": f32(rng(s.seed, "m2_D").uniform(0.5, 1.5, s.H)),
        "w": f32(rng(s.seed, "m2_w").normal(0.0, np.sqrt(0.5), size=(Dt, s.K))),
        "bias": f32(np.full(Dt, 0.1)),
        "conv_state": store(S, s.dtype),
        "h0": f32(h0),
    })
    return out
