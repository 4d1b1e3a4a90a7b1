"""Seeded synthetic inputs for LSH attention, shared by the tests and the benchmark.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no hashing, sorting, attention or combination), so both
the CUDA path and the oracle can consume what it produces.

Workloads stand in for the pages' imagenet64 / enwik8 experiments, which are not
available here: image-shaped (L = 64*64*3), long-text-shaped (L = 64K) and a
length sweep at a fixed token count, with the head counts of the Reformer
experiments (8 heads, batch 8).

Recipe for the "clustered" shared-QK projection: per (batch, head) draw K unit
centres u_k = g / |g| with g ~ N(0, I_d); each token picks k uniformly and gets
x = u_k * |h| + 0.3 * n with h, n ~ N(0, I_d) independent.  The cosine between
x and its centre is then about 0.96, the "near" vector of the Reformer glossary
page's hashing example.  Values v and the random rotations R are i.i.d. N(0, 1).
bf16 (fp16) workloads are rounded to bf16 (fp16) with round-to-nearest-even once, here,
and both sides receive exactly those values.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    dtype: str          # "f32", "bf16" or "f16"
    n_buckets: int
    n_rounds: int
    chunk: int
    causal: bool
    clusters: int       # 0 = i.i.d. Gaussian qk
    seed: int
    noise: float = 0.3

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.L

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _sweep():
    out = {}
    for i, L in enumerate([1024, 2048, 4096, 8192, 16384, 32768]):
        for R in (1, 2, 4, 8):
            name = f"sweep_B{131072 // L}_H8_L{L}_d64_R{R}"
            out[name] = Workload(name, 131072 // L, 8, L, 64, "bf16", L // 64, R, 64, True,
                                 L // 64, 1000 + 100 * (i + 1) + R)
    return out


#: The workloads, named by what they are.
WORKLOADS = {
    "gauss_f32_B1_H1_L1024_d64": Workload(
        "gauss_f32_B1_H1_L1024_d64", 1, 1, 1024, 64, "f32", 32, 1, 32, True, 0, 1001),
    "clustered_B8_H8_L4096_d64_R4": Workload(
        "clustered_B8_H8_L4096_d64_R4", 8, 8, 4096, 64, "bf16", 64, 4, 64, True, 64, 1002),
    "image_B8_H8_L12288_d128_R8": Workload(
        "image_B8_H8_L12288_d128_R8", 8, 8, 12288, 128, "bf16", 192, 8, 64, True, 256, 1003),
    "long_B1_H8_L65536_d128_R8": Workload(
        "long_B1_H8_L65536_d128_R8", 1, 8, 65536, 128, "bf16", 1024, 8, 64, True, 1024, 1004),
    **_sweep(),
}

WORKLOADS["long_f16_B1_H8_L65536_d128_R8"] = WORKLOADS["long_B1_H8_L65536_d128_R8"].replace(
    name="long_f16_B1_H8_L65536_d128_R8", dtype="f16")

WORKLOADS["long_chunk32_B1_H8_L65536_d128_R8"] = WORKLOADS["long_B1_H8_L65536_d128_R8"].replace(
    name="long_chunk32_B1_H8_L65536_d128_R8", chunk=32)

WORKLOADS["long_chunk128_B1_H8_L65536_d128_R8"] = WORKLOADS["long_B1_H8_L65536_d128_R8"].replace(
    name="long_chunk128_B1_H8_L65536_d128_R8", chunk=128)

#: The headline workload: L = 64K, 8 rounds.
HEADLINE = "long_B1_H8_L65536_d128_R8"


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def round_f16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest fp16 value (ties to even); returns float32."""
    return np.asarray(a, np.float32).astype(np.float16).astype(np.float32)


def _gauss(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def clustered(rng: np.random.Generator, n_heads: int, L: int, d: int, K: int,
              noise: float) -> np.ndarray:
    """[n_heads, L, d] float32 drawn from the clustered recipe in the module docstring."""
    out = np.empty((n_heads, L, d), np.float32)
    for h in range(n_heads):
        g = _gauss(rng, (K, d))
        u = g / np.linalg.norm(g, axis=1, keepdims=True)
        k = rng.integers(0, K, size=L)
        hn = np.linalg.norm(_gauss(rng, (L, d)), axis=1, keepdims=True)
        out[h] = u[k] * hn + noise * _gauss(rng, (L, d))
    return out


def make_inputs(w: Workload, seed: int | None = None):
    """qk, v [B, H, L, d] and R [n_rounds, d, n_buckets/2] as float32 numpy arrays.

    For bf16 workloads every value is already a bf16 value.
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    n_heads = w.B * w.H
    if w.clusters > 0:
        qk = clustered(rng, n_heads, w.L, w.d, w.clusters, w.noise)
    else:
        qk = _gauss(rng, (n_heads, w.L, w.d))
    v = _gauss(rng, (n_heads, w.L, w.d))
    R = _gauss(rng, (w.n_rounds, w.d, w.n_buckets // 2))
    qk = qk.reshape(w.B, w.H, w.L, w.d)
    v = v.reshape(w.B, w.H, w.L, w.d)
    if w.dtype == "bf16":
        qk, v, R = round_bf16(qk), round_bf16(v), round_bf16(R)
    elif w.dtype == "f16":
        qk, v, R = round_f16(qk), round_f16(v), round_f16(R)
    return qk, v, R


@dataclasses.dataclass(frozen=True)
class BlockWorkload:
    """One reversible residual block around the LSH attention: residual stream
    [B, L, d_model] split into heads of d = d_model / heads, feed-forward width d_ff run
    over chunks of ff_chunk positions."""
    name: str
    B: int
    L: int
    d_model: int
    heads: int
    d_ff: int
    n_buckets: int
    n_rounds: int
    chunk: int
    causal: bool
    ff_chunk: int
    seed: int

    @property
    def d(self) -> int:
        return self.d_model // self.heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def tokens(self) -> int:
        return self.B * self.L


#: The reversible block at the long-text shape: 8 heads of 128 (d_model 1024), a
#: feed-forward four times as wide, run over chunks of 8192 positions.
BLOCK_LONG = BlockWorkload("block_B1_L65536_dm1024_H8_ff4096_R8", 1, 65536, 1024, 8, 4096,
                           1024, 8, 64, True, 8192, 1005)


def make_block_inputs(w: BlockWorkload, seed: int | None = None) -> dict:
    """Inputs of one reversible block as float32 numpy arrays: the two halves of the
    residual stream x1, x2 ~ N(0, 1) [B, L, d_model]; weights [out][in] drawn N(0, 1/fan_in)
    and rounded to bf16 (Wqk, Wv, Wo [d_model, d_model], W1 [d_ff, d_model], W2
    [d_model, d_ff]); biases b1 [d_ff], b2 [d_model] ~ N(0, 0.01), float32; rotations
    R ~ N(0, 1) [n_rounds, d, n_buckets/2], rounded to bf16."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    shape = (w.B, w.L, w.d_model)

    def lin(o, i):
        return round_bf16(_gauss(rng, (o, i)) / np.float32(math.sqrt(i)))

    out = dict(x1=_gauss(rng, shape), x2=_gauss(rng, shape))
    out.update(Wqk=lin(w.d_model, w.d_model), Wv=lin(w.d_model, w.d_model),
               Wo=lin(w.d_model, w.d_model), W1=lin(w.d_ff, w.d_model),
               b1=np.float32(0.1) * _gauss(rng, (w.d_ff,)), W2=lin(w.d_model, w.d_ff),
               b2=np.float32(0.1) * _gauss(rng, (w.d_model,)),
               R=round_bf16(_gauss(rng, (w.n_rounds, w.d, w.n_buckets // 2))))
    return out


def synthetic_buckets(rng: np.random.Generator, n_segments: int, L: int, n_buckets: int,
                      alpha: float = 1.0) -> np.ndarray:
    """int32 [n_segments, L] bucket ids with uneven occupancy (Dirichlet(alpha) weights)."""
    out = np.empty((n_segments, L), np.int32)
    for s in range(n_segments):
        w = rng.dirichlet(np.full(n_buckets, alpha))
        out[s] = rng.choice(n_buckets, size=L, p=w).astype(np.int32)
    return out


def synthetic_round_outputs(rng: np.random.Generator, n_segments: int, L: int, d: int,
                            self_fraction: float = 0.02):
    """Per-round outputs o_r [n_segments, L, d] ~ N(0,1) and lse_r [n_segments, L].

    lse_r ~ N(1, 2); a fraction of rows carries the self-only value -1e5.
    """
    o = _gauss(rng, (n_segments, L, d))
    lse = (1.0 + 2.0 * _gauss(rng, (n_segments, L))).astype(np.float32)
    mask = rng.random((n_segments, L)) < self_fraction
    lse[mask] = -1.0e5
    return o, lse
