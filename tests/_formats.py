"""Test-side encoders for the block formats: the inverse direction of the
oracle's decoders, written independently from the format descriptions, so
that a round trip through them pins the oracle's field placement.

Q6_K (GGUF arrangement, "Strata" PR #2340 "Q6_K six-bit offset"): weight n of
a 256-block sits in half h = n // 128, quarter r = (n % 128) // 32 and
position l = n % 32; its low 4 bits go to ql[64h + 32*(r % 2) + l] (low
nibble for r < 2, high nibble for r >= 2) and its high 2 bits to
qh[32h + l] at bit 2r.  Scale index n // 16, block layout
ql[128] | qh[64] | int8 scales[16] | fp16 d.

Q5_K (GGUF arrangement): d | dmin | the Q4_K scale bytes | qh[32] | qs[128];
weight n = 32j + l (sub-block j) keeps its low 4 bits where Q4_K would and
its fifth bit in bit j of qh[l].

Q4_K (GGUF arrangement): d | dmin | 12 packed scale bytes | qs[128]; the
scales of sub-blocks 0-3 and mins of 0-3 take the low 6 bits of bytes 0-3 and
4-7; sub-blocks 4-7 keep their low 4 bits of scale and min in bytes 8-11
(scale low nibble, min high nibble) and their top 2 bits in the top 2 bits of
bytes 0-3 (scale) and 4-7 (min).  Weight n: chunk c = n // 64, the low nibble
of qs[32c + n % 32] when (n % 64) < 32, else the high nibble.
"""
import numpy as np


def f16_bytes(v) -> np.ndarray:
    return np.array([v], dtype=np.float16).view(np.uint8)


def f16_value(b: np.ndarray) -> float:
    return float(np.ascontiguousarray(b[:2]).view(np.float16)[0])


def encode_q6_k(q: np.ndarray, sc: np.ndarray, d) -> np.ndarray:
    """q: 256 codes in 0..63, sc: 16 int8, d: float (stored as fp16)."""
    q = np.asarray(q, dtype=np.int64)
    n = np.arange(256)
    h, r, l = n // 128, (n % 128) // 32, n % 32
    ql = np.zeros(128, dtype=np.int64)
    qh = np.zeros(64, dtype=np.int64)
    np.add.at(ql, 64 * h + 32 * (r % 2) + l, (q & 15) << (4 * (r // 2)))
    np.add.at(qh, 32 * h + l, (q >> 4) << (2 * r))
    out = np.zeros(210, dtype=np.uint8)
    out[0:128] = ql
    out[128:192] = qh
    out[192:208] = np.asarray(sc, dtype=np.int8).view(np.uint8)
    out[208:210] = f16_bytes(d)
    return out


def encode_q4_k(q: np.ndarray, sc: np.ndarray, m: np.ndarray, d, dmin) -> np.ndarray:
    """q: 256 codes in 0..15; sc, m: 8 values in 0..63."""
    q = np.asarray(q, dtype=np.int64)
    sc = np.asarray(sc, dtype=np.int64)
    m = np.asarray(m, dtype=np.int64)
    s = np.zeros(12, dtype=np.int64)
    s[0:4] = sc[0:4] | ((sc[4:8] >> 4) << 6)
    s[4:8] = m[0:4] | ((m[4:8] >> 4) << 6)
    s[8:12] = (sc[4:8] & 15) | ((m[4:8] & 15) << 4)
    n = np.arange(256)
    qs = np.zeros(128, dtype=np.int64)
    np.add.at(qs, 32 * (n // 64) + n % 32, q << (4 * ((n % 64) // 32)))
    out = np.zeros(144, dtype=np.uint8)
    out[0:2] = f16_bytes(d)
    out[2:4] = f16_bytes(dmin)
    out[4:16] = s
    out[16:144] = qs
    return out


def _pack_scales_mins(sc, m) -> np.ndarray:
    sc = np.asarray(sc, dtype=np.int64)
    m = np.asarray(m, dtype=np.int64)
    s = np.zeros(12, dtype=np.int64)
    s[0:4] = sc[0:4] | ((sc[4:8] >> 4) << 6)
    s[4:8] = m[0:4] | ((m[4:8] >> 4) << 6)
    s[8:12] = (sc[4:8] & 15) | ((m[4:8] & 15) << 4)
    return s


def encode_q5_k(q: np.ndarray, sc: np.ndarray, m: np.ndarray, d, dmin) -> np.ndarray:
    """q: 256 codes in 0..31; sc, m: 8 values in 0..63."""
    q = np.asarray(q, dtype=np.int64)
    n = np.arange(256)
    j, l = n // 32, n % 32
    qs = np.zeros(128, dtype=np.int64)
    np.add.at(qs, 32 * (j // 2) + l, (q & 15) << (4 * (j % 2)))
    qh = np.zeros(32, dtype=np.int64)
    np.add.at(qh, l, (q >> 4) << j)
    out = np.zeros(176, dtype=np.uint8)
    out[0:2] = f16_bytes(d)
    out[2:4] = f16_bytes(dmin)
    out[4:16] = _pack_scales_mins(sc, m)
    out[16:48] = qh
    out[48:176] = qs
    return out


def q8_1_fields(xq: np.ndarray):
    """Q8_1 bytes [..., 36] -> (d fp64 [...], s fp64 [...], q int64 [..., 32])."""
    xq = np.ascontiguousarray(xq)
    d = xq[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    s = xq[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    q = xq[..., 4:36].view(np.int8).astype(np.int64)
    return d, s, q
