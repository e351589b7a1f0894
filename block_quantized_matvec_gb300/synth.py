"""Seeded synthetic inputs shaped like the matrices the MMVQ pages measure.

This module only draws random bytes and numbers; it holds none of the
method's arithmetic (no decode, no quantisation, no dot products).  Both the
CUDA path and the CPU oracle consume exactly the arrays made here.

Weight bytes follow the block sizes of the K-quant formats named in the pages
("Strata" PR #2340, "Q6_K six-bit offset", and PR #2207's Q6_K/Q4_K
dense_bench table), with the field distributions of the synthetic workload:

* Q6_K, 210 B per 256 weights: ql[128] and qh[64] uniform bytes (so every
  6-bit code q in 0..63 is uniform), scales[16] int8 uniform in [-32, 31],
  d = fp16(uniform[1e-3, 1e-2]).
* Q4_K, 144 B per 256 weights: d, dmin = fp16(uniform[1e-3, 1e-2]),
  scales[12] uniform bytes, qs[128] uniform bytes.  Every bit of the 12-byte
  packed scale field feeds exactly one 6-bit scale or min, so uniform bytes
  give 16 independent values uniform on 0..63, which is the stated
  distribution without any packing code here.
* Activations: fp32 N(0, 1), one row per column, ``[ncols][K]``.
* Routing: each token picks ``k`` distinct experts uniformly
  (a partial Fisher-Yates shuffle via ``Generator.permutation``).
* Draft-head rows: ``n`` distinct row ids drawn uniformly, in draw order.

Seeds: weights 1, activations 2, routing 3, draft rows 4, each offset by a
caller-chosen salt so that different matrices of one workload differ.
"""
from __future__ import annotations

import numpy as np

Q6_K_BLOCK_BYTES = 210
Q4_K_BLOCK_BYTES = 144
Q8_1_BLOCK_BYTES = 36
QK_K = 256
QK8_1 = 32

SEED_WEIGHTS = 1
SEED_ACTIVATIONS = 2
SEED_ROUTING = 3
SEED_DRAFT_ROWS = 4


def _rng(seed: int, salt: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(salt)])


def _fp16_uniform(rng: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    """n fp16 values drawn uniform in [lo, hi], returned as raw little-endian bytes."""
    v = rng.uniform(lo, hi, size=n).astype(np.float16)
    return v.view(np.uint8).reshape(n, 2)


def q6_k_weights(rows: int, K: int, salt: int = 0, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """Q6_K weight matrix as GGUF-ordered blocks, shape ``[rows, K//256, 210]`` uint8."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    n = rows * nb
    rng = _rng(seed, salt)
    w = np.empty((n, Q6_K_BLOCK_BYTES), dtype=np.uint8)
    w[:, 0:192] = rng.integers(0, 256, size=(n, 192), dtype=np.uint8)        # ql | qh
    w[:, 192:208] = rng.integers(-32, 32, size=(n, 16), dtype=np.int8).view(np.uint8)
    w[:, 208:210] = _fp16_uniform(rng, n, 1e-3, 1e-2)
    return w.reshape(rows, nb, Q6_K_BLOCK_BYTES)


def q4_k_weights(rows: int, K: int, salt: int = 0, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """Q4_K weight matrix as GGUF-ordered blocks, shape ``[rows, K//256, 144]`` uint8."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    n = rows * nb
    rng = _rng(seed, salt)
    w = np.empty((n, Q4_K_BLOCK_BYTES), dtype=np.uint8)
    w[:, 0:2] = _fp16_uniform(rng, n, 1e-3, 1e-2)                            # d
    w[:, 2:4] = _fp16_uniform(rng, n, 1e-3, 1e-2)                            # dmin
    w[:, 4:144] = rng.integers(0, 256, size=(n, 140), dtype=np.uint8)        # scales | qs
    return w.reshape(rows, nb, Q4_K_BLOCK_BYTES)


def q5_k_weights(rows: int, K: int, salt: int = 0, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """Q5_K weight matrix as GGUF-ordered blocks, shape ``[rows, K//256, 176]`` uint8:
    fp16 d and dmin uniform in [1e-3, 1e-2], every other byte (scales, qh, qs) uniform."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    n = rows * nb
    rng = _rng(seed, 5000 + salt)
    w = np.empty((n, 176), dtype=np.uint8)
    w[:, 0:2] = _fp16_uniform(rng, n, 1e-3, 1e-2)                            # d
    w[:, 2:4] = _fp16_uniform(rng, n, 1e-3, 1e-2)                            # dmin
    w[:, 4:176] = rng.integers(0, 256, size=(n, 172), dtype=np.uint8)        # scales | qh | qs
    return w.reshape(rows, nb, 176)


def expert_weights(kind: str, n_experts: int, rows: int, K: int, salt: int = 0,
                   seed: int = SEED_WEIGHTS) -> np.ndarray:
    """Stacked per-expert matrices ``[n_experts, rows, K//256, block]``."""
    gen = {"q4_k": q4_k_weights, "q6_k": q6_k_weights}[kind]
    w = gen(n_experts * rows, K, salt=salt, seed=seed)
    return w.reshape(n_experts, rows, K // QK_K, w.shape[-1])


def activations(K: int, ncols: int, salt: int = 0, seed: int = SEED_ACTIVATIONS) -> np.ndarray:
    """fp32 activations ``[ncols, K]`` drawn N(0, 1)."""
    rng = _rng(seed, salt)
    return rng.standard_normal(size=(ncols, K), dtype=np.float32)


def moe_hidden(H: int, T: int, salt: int = 0, seed: int = SEED_ACTIVATIONS) -> np.ndarray:
    """Hidden states entering an expert layer, ``[T, H]``: N(0, 1) scaled by 2^-6
    (exact), so that with the synthetic expert weights (whose values run a
    hundred times larger than trained ones) SiLU(gate)*up stays well inside
    the fp16 range of the Q8_1 scale and sum fields."""
    return activations(H, T, salt=salt, seed=seed) * np.float32(1.0 / 64.0)


def routing(T: int, k: int = 8, n_experts: int = 256, salt: int = 0,
            seed: int = SEED_ROUTING) -> np.ndarray:
    """Top-k expert ids per token, ``[T, k]`` int32, distinct within a token."""
    if k > n_experts:
        raise ValueError("k must not exceed n_experts")
    rng = _rng(seed, salt)
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = rng.permutation(n_experts)[:k]
    return out


def draft_rows(n: int, rows: int, salt: int = 0, seed: int = SEED_DRAFT_ROWS) -> np.ndarray:
    """``n`` distinct row ids in ``[0, rows)``, in draw order, int32."""
    rng = _rng(seed, salt)
    return rng.choice(rows, size=n, replace=False).astype(np.int32)


def gate_up(n: int, F: int, salt: int = 0, seed: int = SEED_ACTIVATIONS) -> np.ndarray:
    """fp32 gate|up rows ``[n, 2F]`` drawn N(0, 1), for exercising SiLU-mul on its own."""
    rng = _rng(seed, 1000 + salt)
    return rng.standard_normal(size=(n, 2 * F), dtype=np.float32)
