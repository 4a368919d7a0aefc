"""Seeded synthetic workloads shaped like the pages' EXL3 MoE layers.

Nothing here computes any part of the layer.  Every array is drawn from numpy's
PCG64 (``numpy.random.default_rng``) with a seed tuple that names what is drawn,
so a projection, a residual stage or a router batch can be regenerated on its
own (the oracle only needs the experts a token touches).

Recipe (shapes from the pages' GLM-5.2 and RED-SNOW layers, values synthetic):

* trellis words: uniform random 32-bit words, ``[in/16, out/16, 8*K]`` per
  projection (16x16 tiles, ``K`` bits per weight);
* ``suh`` / ``svh``: uniform random +-1 in fp16;
* ``scale``: fp16(U[0.5, 1.5] / sqrt(in)) per output channel;
* activations ``x``: N(0, 1) rounded to the activation dtype;
* router: logits N(0, 1) (+ an optional Zipf bias), softmax over all experts,
  top-k by probability (ties to the lower id), weights = those probabilities,
  not renormalised, rounded to the route-weight dtype.

Tokens are drawn as a prefix of one stream, so token ``t`` of an ``M=8`` batch
is token ``t`` of the ``M=128`` batch with the same seed (used by the
row-invariance tests).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "CB_MUL1", "CB_MCG", "CB_3INST", "CB_NAMES", "GATE", "UP", "DOWN",
    "Projection", "MoESpec", "MoEWorkload", "LinearWorkload",
    "config", "round_to_bf16_bits", "bf16_bits_to_f64", "act_to_f64",
    "rw_to_f64", "make_projection", "trellis_words_per_tile",
]

CB_MUL1, CB_MCG, CB_3INST = 0, 1, 2
CB_NAMES = {CB_MUL1: "mul1", CB_MCG: "mcg", CB_3INST: "3inst"}
GATE, UP, DOWN = 0, 1, 2


def trellis_words_per_tile(K: int) -> int:
    """32-bit words holding one 16x16 tile of K-bit codes (256*K bits)."""
    return 8 * K


def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def act_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def rw_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return act_to_f64(a, dtype)


def _round_act(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16_bits(a.astype(np.float32))
    if dtype == "f16":
        return a.astype(np.float16)
    if dtype == "f32":
        return a.astype(np.float32)
    raise ValueError(dtype)


@dataclass
class Projection:
    """One EXL3 projection: trellis codes plus rotation signs and scale."""
    trellis: np.ndarray  # uint32 [in/16, out/16, 8K]
    suh: np.ndarray      # float16 [in]
    svh: np.ndarray      # float16 [out]
    scale: np.ndarray    # float16 [out]
    K: int
    codebook: int

    @property
    def in_features(self) -> int:
        return self.trellis.shape[0] * 16

    @property
    def out_features(self) -> int:
        return self.trellis.shape[1] * 16


def _random_words(rng: np.random.Generator, n: int) -> np.ndarray:
    return np.frombuffer(rng.bytes(4 * n), dtype="<u4").copy()


def make_projection(seed, in_f: int, out_f: int, K: int, cb: int) -> Projection:
    assert in_f % 16 == 0 and out_f % 16 == 0 and 1 <= K <= 8
    rng = np.random.default_rng(seed)
    words = _random_words(rng, (in_f // 16) * (out_f // 16) * 8 * K)
    trellis = words.reshape(in_f // 16, out_f // 16, 8 * K)
    suh = (rng.integers(0, 2, size=in_f) * 2 - 1).astype(np.float16)
    svh = (rng.integers(0, 2, size=out_f) * 2 - 1).astype(np.float16)
    scale = (rng.uniform(0.5, 1.5, size=out_f) / math.sqrt(in_f)).astype(np.float16)
    return Projection(trellis, suh, svh, scale, K, cb)


def make_residual_trellis(seed, in_f: int, out_f: int, K: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return _random_words(rng, (in_f // 16) * (out_f // 16) * 8 * K).reshape(
        in_f // 16, out_f // 16, 8 * K)


@dataclass
class MoESpec:
    name: str
    hidden: int
    inter: int
    E: int
    topk: int
    M: int
    act: str            # "f16" | "bf16"
    ids_dtype: str      # "i32" | "i64"
    rw_dtype: str       # "f16" | "bf16" | "f32"
    K: np.ndarray       # int [E], width of every projection of expert e
    cb: np.ndarray      # int [E], codebook of every projection of expert e
    seed: int
    capacity: int = 512
    zipf_s: float = 0.0
    # additive residual stages (stage 0 is the base and is implicit)
    residual_K: list = field(default_factory=list)       # one K per residual stage
    residual_zero_frac: float = 0.5
    residual_alpha: tuple = (0.05, 0.2)

    @property
    def routes(self) -> int:
        return self.M * self.topk

    @property
    def num_stages(self) -> int:
        return 1 + len(self.residual_K)

    def proj_shape(self, p: int):
        return (self.hidden, self.inter) if p in (GATE, UP) else (self.inter, self.hidden)


def config(idx: int, M: int | None = None) -> MoESpec:
    """The five workload configurations (seed = config index)."""
    if idx == 0:
        E = 8
        return MoESpec("tiny", 512, 256, E, 2, M or 16, "f16", "i32", "f16",
                       np.full(E, 4), np.full(E, CB_MCG), seed=0)
    if idx == 1:
        E = 192
        return MoESpec("decode", 5120, 1536, E, 8, M or 1, "bf16", "i32", "bf16",
                       np.full(E, 3), np.full(E, CB_MCG), seed=1)
    if idx == 2:
        E = 288
        K = np.random.default_rng([2, 13]).integers(4, 9, size=E)
        cb = np.where(np.arange(E) % 2 == 0, CB_3INST, CB_MUL1)
        return MoESpec("mixed", 4096, 1408, E, 8, M or 64, "f16", "i64", "f16",
                       K, cb, seed=2)
    if idx == 3:
        E = 192
        K = np.random.default_rng([3, 13]).integers(3, 5, size=E)
        return MoESpec("prefill", 5120, 1536, E, 8, M or 3072, "bf16", "i32", "bf16",
                       K, np.full(E, CB_MCG), seed=3, capacity=512, zipf_s=1.2)
    if idx == 4:
        E = 288
        return MoESpec("additive", 4096, 1408, E, 8, M or 512, "f16", "i64", "f32",
                       np.full(E, 3), np.full(E, CB_MCG), seed=4, residual_K=[2])
    raise ValueError(idx)


class MoEWorkload:
    """Inputs of one MoE layer call.  Expert projections are generated lazily."""

    def __init__(self, spec: MoESpec):
        self.spec = spec
        s = spec
        rng_x = np.random.default_rng([s.seed, 10])
        self.x = _round_act(rng_x.standard_normal((s.M, s.hidden)), s.act)
        rng_r = np.random.default_rng([s.seed, 11])
        logits = rng_r.standard_normal((s.M, s.E))
        if s.zipf_s:
            rank = np.random.default_rng([s.seed, 12]).permutation(s.E) + 1
            logits = logits + (-s.zipf_s * np.log(rank))[None, :]
        z = logits - logits.max(axis=1, keepdims=True)
        prob = np.exp(z)
        prob /= prob.sum(axis=1, keepdims=True)
        order = np.argsort(-prob, axis=1, kind="stable")[:, : s.topk]
        self.ids = order.astype(np.int32 if s.ids_dtype == "i32" else np.int64)
        self.rw = _round_act(np.take_along_axis(prob, order, axis=1), s.rw_dtype)
        self._cache = {}
        # residual stage tables (stage-major [S-1][E][3])
        nres = len(s.residual_K)
        if nres:
            rng_a = np.random.default_rng([s.seed, 14])
            zero = rng_a.random((nres, s.E, 3)) < s.residual_zero_frac
            alpha = rng_a.uniform(*s.residual_alpha, size=(nres, s.E, 3))
            self.alpha = np.where(zero, 0.0, alpha).astype(np.float32)
        else:
            self.alpha = np.zeros((0, s.E, 3), np.float32)

    def projection(self, e: int, p: int, cache: bool = False) -> Projection:
        key = (e, p)
        if key in self._cache:
            return self._cache[key]
        s = self.spec
        in_f, out_f = s.proj_shape(p)
        pr = make_projection([s.seed, 1, e, p], in_f, out_f, int(s.K[e]), int(s.cb[e]))
        if cache:
            self._cache[key] = pr
        return pr

    def residual(self, stage: int, e: int, p: int):
        """Residual trellis of stage ``stage`` (1-based) or None where alpha is 0."""
        s = self.spec
        if self.alpha[stage - 1, e, p] == 0.0:
            return None
        in_f, out_f = s.proj_shape(p)
        return make_residual_trellis([s.seed, 2, stage, e, p], in_f, out_f,
                                     int(s.residual_K[stage - 1]))


class LinearWorkload:
    """Inputs of one ``exl3_linear`` call."""

    def __init__(self, M: int, in_f: int, out_f: int, K: int, cb: int, act: str,
                 seed: int):
        self.M, self.act = M, act
        self.proj = make_projection([seed, 20], in_f, out_f, K, cb)
        rng = np.random.default_rng([seed, 21])
        self.x = _round_act(rng.standard_normal((M, in_f)), act)
