"""Seeded synthetic inputs for the MoE layer (shared by tests, smoke and bench).

This module draws random numbers and lays them out in the packed storage
format; it holds none of the layer's arithmetic.  Distributions follow the
workloads the layer is specified on:

* router logits ~ N(0, 1) in fp32, optionally +bias on a set of "hot" experts
  (the TP4 shard shape with skewed segment lengths);
* activations x ~ N(0, 1), rounded to fp16;
* weight codes q and zero points z uniform over {0..15}: a uniformly random
  32-bit word is exactly eight independent uniform 4-bit codes, so packed
  words are drawn directly;
* group scales s ~ U[0.002, 0.02], rounded to fp16.

Packed layouts (little-endian words, row-major):
  W13 qweight u32 [E][2I][H/8], scales f16 [E][2I][H/32], qzeros u32 [E][2I/8][H/32]
  W2  qweight u32 [E][H][I/8],  scales f16 [E][H][I/32],  qzeros u32 [E][H/8][I/32]
Element (n, kk) of a matrix W[N][K]: q = nibble kk%8 of qweight[n][kk/8]
(bits 4*(kk%8)..+3), z = nibble n%8 of qzeros[n/8][kk/32], s = scales[n][kk/32].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class MoEShape:
    T: int
    H: int
    I: int
    E: int
    k: int

    @property
    def P(self) -> int:
        return self.T * self.k


@dataclass
class Workload:
    name: str
    shape: MoEShape
    seed: int = 0
    hot_experts: tuple = ()
    hot_bias: float = 0.0
    extra: dict = field(default_factory=dict)


# The workloads the layer is specified on.
TINY = Workload("tiny_T4_H256_I64_E16_k2", MoEShape(4, 256, 64, 16, 2))
QWEN_C1 = Workload("qwen4exp_decode_T1_H2560_I640_E512_k10", MoEShape(1, 2560, 640, 512, 10))
QWEN_C2 = Workload("qwen4exp_decode_T2_H2560_I640_E512_k10", MoEShape(2, 2560, 640, 512, 10))
QWEN_C4 = Workload("qwen4exp_decode_T4_H2560_I640_E512_k10", MoEShape(4, 2560, 640, 512, 10))
QWEN_C8 = Workload("qwen4exp_decode_T8_H2560_I640_E512_k10", MoEShape(8, 2560, 640, 512, 10))
_HOT = tuple(range(16))
TP4_C2 = Workload("tp4shard_decode_T2_H2560_I160_E512_k10_hot16", MoEShape(2, 2560, 160, 512, 10),
                  hot_experts=_HOT, hot_bias=2.0)
TP4_C4 = Workload("tp4shard_decode_T4_H2560_I160_E512_k10_hot16", MoEShape(4, 2560, 160, 512, 10),
                  hot_experts=_HOT, hot_bias=2.0)
TP4_C8 = Workload("tp4shard_decode_T8_H2560_I160_E512_k10_hot16", MoEShape(8, 2560, 160, 512, 10),
                  hot_experts=_HOT, hot_bias=2.0)
PREFILL = Workload("qwen4exp_prefill_T4096_H2560_I640_E512_k10", MoEShape(4096, 2560, 640, 512, 10))

ALL = {w.name: w for w in (TINY, QWEN_C1, QWEN_C2, QWEN_C4, QWEN_C8,
                           TP4_C2, TP4_C4, TP4_C8, PREFILL)}


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag])))


def _scales(rng: np.random.Generator, shape) -> np.ndarray:
    u = rng.random(shape, dtype=np.float32)
    return (np.float32(0.002) + np.float32(0.018) * u).astype(np.float16)


def _words(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint32)


def make_weights(E: int, H: int, I: int, seed: int = 0):
    """(w13, w2), each a tuple (qweight u32, scales f16, qzeros u32)."""
    if H % 32 or I % 32:
        raise ValueError("H and I must be multiples of 32")
    G_h, G_i = H // 32, I // 32
    w13 = (_words(_rng(seed, 11), (E, 2 * I, H // 8)),
           _scales(_rng(seed, 12), (E, 2 * I, G_h)),
           _words(_rng(seed, 13), (E, 2 * I // 8, G_h)))
    w2 = (_words(_rng(seed, 21), (E, H, I // 8)),
          _scales(_rng(seed, 22), (E, H, G_i)),
          _words(_rng(seed, 23), (E, H // 8, G_i)))
    return w13, w2


def make_weights_nvfp4(E: int, H: int, I: int, seed: int = 0):
    """(w13, w2) in the NVFP4 layout, each a tuple (codes u32 [E][N][K/8],
    bscale u8 [E][N][K/16], gscale f32 [E]).  Codes: uniformly random words
    (eight independent E2M1 codes, both signs); block scales: FP8 E4M3 bytes
    drawn uniformly from 0x30-0x3F (0.5 to 1.875); per-expert scales
    ~ U[0.005, 0.02], so weights span the same range as the W4A16 ones."""
    if H % 32 or I % 32:
        raise ValueError("H and I must be multiples of 32")

    def mat(tag, N, K):
        codes = _words(_rng(seed, tag), (E, N, K // 8))
        bs = _rng(seed, tag + 1).integers(0x30, 0x40, size=(E, N, K // 16), dtype=np.uint8)
        gs = (np.float32(0.005) + np.float32(0.015) * _rng(seed, tag + 2).random(E, dtype=np.float32))
        return codes, bs, gs.astype(np.float32)
    return mat(31, 2 * I, H), mat(41, H, I)


def make_activations(T: int, H: int, E: int, seed: int = 0, hot_experts=(), hot_bias=0.0):
    """(logits f32 [T,E], x f16 [T,H])."""
    logits = _rng(seed, 1).standard_normal((T, E), dtype=np.float32)
    if len(hot_experts):
        logits[:, list(hot_experts)] += np.float32(hot_bias)
    x = _rng(seed, 2).standard_normal((T, H), dtype=np.float32).astype(np.float16)
    return logits, x


def make_workload(w: Workload, seed: int | None = None):
    """(logits, x, w13, w2) for a named workload."""
    s = w.seed if seed is None else seed
    sh = w.shape
    logits, x = make_activations(sh.T, sh.H, sh.E, s, w.hot_experts, w.hot_bias)
    w13, w2 = make_weights(sh.E, sh.H, sh.I, s)
    return logits, x, w13, w2


def make_router(E: int, H: int, seed: int = 0) -> np.ndarray:
    """Router matrix w_router f16 [E, H] ~ N(0, 1/H): with x ~ N(0, 1) the
    logits x . w_router[e] have unit variance, like the logits drawn above."""
    w = _rng(seed, 51).standard_normal((E, H), dtype=np.float32) / np.float32(np.sqrt(H))
    return w.astype(np.float16)


def make_awq_layer(E: int, K: int, N: int, seed: int = 0, tag: int = 61):
    """A stack of E AWQ GEMM-layout layers with input size K and output size
    N: (qweight u32 [E][K][N/8], qzeros u32 [E][K/32][N/8], scales f16
    [E][K/32][N]); codes and zeros uniformly random words, scales as above."""
    if K % 32 or N % 8:
        raise ValueError("K must be a multiple of 32 and N of 8")
    return (_words(_rng(seed, tag), (E, K, N // 8)),
            _words(_rng(seed, tag + 1), (E, K // 32, N // 8)),
            _scales(_rng(seed, tag + 2), (E, K // 32, N)))


def random_topk_ids(T: int, E: int, k: int, seed: int = 0) -> np.ndarray:
    """k distinct expert ids per token, uniformly at random (for testing the
    grouping step on its own)."""
    rng = _rng(seed, 3)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


def bytes_per_expert_nvfp4(H: int, I: int) -> dict:
    """Bytes of one expert's NVFP4 weights (codes + E4M3 block scales +
    the fp32 per-expert scale)."""
    def mat(N, K):
        return N * K // 2 + N * (K // 16) + 4
    return {"w13": mat(2 * I, H), "w2": mat(H, I)}


def bytes_per_expert(H: int, I: int) -> dict:
    """Packed bytes of one expert's weights (qweight + scales + qzeros)."""
    def mat(N, K):
        return N * K // 2 + N * (K // 32) * 2 + (N // 8) * (K // 32) * 4
    return {"w13": mat(2 * I, H), "w2": mat(H, I)}
