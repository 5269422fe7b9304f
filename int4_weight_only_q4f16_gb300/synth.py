"""Seeded synthetic inputs for the q4f16_1 projections.

This module is shared by the tests, the benchmark and the CPU oracle's
callers. It draws random inputs only; it holds none of the method's
arithmetic (no nibble unpacking, no dequantization, no dot products).

Distributions (the q4f16_1 format of MLC, described on the Zero-TVM docs
page, section "Q4F16 quantization format"):

* packed codes: every uint32 word is drawn uniformly from [0, 2**32), so each
  of its eight 4-bit codes is an independent uniform draw from {0..15};
* group scales: one f16 per 32 weights along K, ``f16(|N(0, 0.02)|)``;
* activations: ``f16(N(0, 1))``;
* MoE routing: per token, ``top_k`` distinct experts drawn uniformly without
  replacement, and router weights = softmax of ``top_k`` N(0, 1) logits
  (stored as float32).

Every tensor gets its own stream, derived from (master seed, tag, index), so
a tensor does not change when another one is added or resized.
"""
from __future__ import annotations

import zlib

import numpy as np

MASTER_SEED = 20260730

# Weight shapes of the projections, from the Zero-TVM docs page (section
# "Q4F16 quantization format", Phi-3-mini weight table) and the Qwen3-4B /
# MoE shapes of the workloads; (name, N rows, K reduction).
PHI3_LAYER = (("qkv", 9216, 3072), ("o", 3072, 3072),
              ("gate_up", 16384, 3072), ("down", 3072, 8192))
PHI3_LM_HEAD = ("lm_head", 32064, 3072)
PHI3_LAYERS = 32

QWEN3_4B_LAYER = (("qkv", 6144, 2560), ("o", 2560, 4096),
                  ("gate_up", 19456, 2560), ("down", 2560, 9728))
QWEN3_4B_LAYERS = 36

MOE_EXPERTS = 128
MOE_TOP_K = 8
MOE_GATE_UP = (1024, 2048)   # N2 = 2*I rows, K
MOE_DOWN = (2048, 512)       # N, K


def rng_for(tag: str, *index: int, seed: int = MASTER_SEED) -> np.random.Generator:
    """Independent PCG64 stream for tensor ``tag`` at ``index``."""
    key = [seed, zlib.crc32(tag.encode())] + [int(i) & 0xFFFFFFFF for i in index]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def packed_codes(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """Uniform random packed words, shape [N, K/8] uint32 (8 codes per word)."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    n = N * (K // 8)                      # even: K/8 is a multiple of 4
    raw = rng.bit_generator.random_raw(n // 2)
    return raw.astype("<u8", copy=False).view("<u4").astype(np.uint32, copy=False).reshape(N, K // 8)


def group_scales(rng: np.random.Generator, N: int, K: int, sigma: float = 0.02,
                 signed: bool = False) -> np.ndarray:
    """f16(|N(0, sigma)|) (signed: f16(N(0, sigma))), shape [N, K/32] float16."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    g = rng.standard_normal((N, K // 32), dtype=np.float32) * np.float32(sigma)
    return (g if signed else np.abs(g)).astype(np.float16)


def activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """f16(N(0, 1)), shape [M, K] float16."""
    return rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)


def routing(rng: np.random.Generator, T: int, E: int, top_k: int):
    """Expert ids [T, top_k] int32 (distinct per token) and router weights
    [T, top_k] float32 = softmax of top_k N(0, 1) logits."""
    if top_k > E:
        raise ValueError("top_k > number of experts")
    ids = np.empty((T, top_k), dtype=np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=top_k, replace=False)
    logits = rng.standard_normal((T, top_k))
    ex = np.exp(logits - logits.max(axis=1, keepdims=True))
    r = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, r


def weight(tag: str, N: int, K: int, *index: int, seed: int = MASTER_SEED, sigma: float = 0.02,
           signed: bool = False):
    """(packed codes, scales) of one q4f16_1 matrix."""
    rng = rng_for(tag, *index, seed=seed)
    return packed_codes(rng, N, K), group_scales(rng, N, K, sigma, signed)


def unit_gain_sigma(K: int, gate_up: bool = False) -> float:
    """Scale sigma for which a projection with signed scales (N(0, sigma))
    keeps the size of its input x: uniform codes give E[(q - 7)^2] = 21.5
    and E[s^2] = sigma^2, so E[y^2] = K * 21.5 * sigma^2 * E[x^2]; the fused
    silu(g) * u output has mean square 1 when g and u have standard
    deviation ~1.27 (so gate_up rows take 1.27 times the sigma). Chained
    synthetic stacks use it in place of the norms a real decode step applies
    between projections. (With the default positive scales, (q - 7) s has
    mean 0.5 E[s]: every output shares a term in sum(x) that grows ~5x per
    3072-wide projection, and f16 overflows within a few layers.)"""
    return float((21.5 * K) ** -0.5) * (1.27 if gate_up else 1.0)
