"""Byte accounting for the weight-bandwidth metric.

The pages quote MMVQ speed as the matrix's weight bytes over the call time,
with the weights read once for all activation columns ("Strata" PR #2207,
Summary and mmvq_bench table; PR #1774, "How it was checked": "the weight
bytes of the matrix ... over that time").  Grouped expert calls count the
bytes of the distinct experts actually read.
"""
from __future__ import annotations

BYTES_PER_256 = {"q6_k": 210, "q6_k_planar": 210, "q6_k_planar_draft": 210, "q4_k": 144,
                 "q4_k_planar": 144, "q5_k": 176, "q5_k_planar": 176, "iq3_s": 110}
Q8_1_BYTES_PER_32 = 36


def weight_bytes(fmt: str, rows: int, K: int) -> int:
    """Bytes of a rows x K matrix in format ``fmt`` (K a multiple of 256)."""
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    return rows * (K // 256) * BYTES_PER_256[fmt]


def call_bytes(fmt: str, rows: int, K: int, ncols: int) -> int:
    """Algorithmic bytes one dense call moves: weights once, Q8_1 columns in, fp32 y out."""
    return weight_bytes(fmt, rows, K) + ncols * (K // 32) * Q8_1_BYTES_PER_32 + ncols * rows * 4


def gbps(nbytes: float, seconds: float) -> float:
    return nbytes / seconds / 1e9


def moe_step_bytes(distinct_experts: int, hidden: int, ffn: int, fmt: str = "q4_k") -> int:
    """Weight bytes one MoE step reads: every distinct routed expert's gate|up
    (2*ffn x hidden) and down (hidden x ffn) matrices, once."""
    return distinct_experts * (weight_bytes(fmt, 2 * ffn, hidden) + weight_bytes(fmt, hidden, ffn))
