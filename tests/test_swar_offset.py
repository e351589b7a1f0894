"""The Q6_K kernels' 6-bit offset as SWAR ("Strata" PR #2340: the Q6_K
decode subtracts 32 from four packed 6-bit codes in one 32-bit operation
instead of byte by byte).

The kernel helper q6_minus_32 (csrc/common.cuh) maps a word of four codes
0..63 to the four int8 values code - 32.  This test reads its three
constants from the source and checks the identity against per-byte
subtraction over every one of the 64^4 packed words, so a changed constant
or a borrow that crosses a byte boundary fails here, on the CPU.  (The GPU
parity tests check the same decode end to end through the per-block sums.)
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "block_quantized_matvec_gb300", "csrc",
                   "common.cuh")


def _kernel_constants():
    text = open(SRC).read()
    m = re.search(r"int q6_minus_32\(uint32_t v\) \{\s*return \(int\)\(\(\(v \| (0x[0-9a-fA-F]+)u\) - "
                  r"(0x[0-9a-fA-F]+)u\) \^ (0x[0-9a-fA-F]+)u\);", text)
    assert m, "q6_minus_32 not found in the form ((v | A) - B) ^ C"
    return tuple(np.uint32(int(g, 16)) for g in m.groups())


def test_swar_offset_equals_per_byte_subtraction_on_every_packed_word():
    a, b, c = _kernel_constants()
    codes = np.arange(64, dtype=np.uint32)
    # every word of four 6-bit codes, byte i holding code_i
    w = (codes[:, None, None, None] | (codes[None, :, None, None] << 8) |
         (codes[None, None, :, None] << 16) | (codes[None, None, None, :] << 24)).reshape(-1)
    assert w.size == 64 ** 4
    got = ((w | a) - b) ^ c                                  # uint32 wrap-around, as on the GPU
    got_bytes = got.view(np.uint8).reshape(-1, 4).view(np.int8)
    want = w.view(np.uint8).reshape(-1, 4).astype(np.int16) - 32
    assert np.array_equal(got_bytes.astype(np.int16), want)
    # the result spans exactly -32..31 in every byte
    assert got_bytes.min() == -32 and got_bytes.max() == 31


def test_the_check_catches_a_wrong_constant():
    # a subtrahend off by one in one byte, a mask that misses the guard bit,
    # or no final flip: each breaks the identity on some of these words
    a, b, c = _kernel_constants()
    codes = np.arange(64, dtype=np.uint32)
    w = (codes[:, None] | (codes[None, :] << 8)).reshape(-1) | np.uint32(0x1f1f0000)
    want = w.view(np.uint8).reshape(-1, 4).astype(np.int16) - 32
    for a2, b2, c2 in ((a, b + np.uint32(1), c), (np.uint32(0x40404040), b, c), (a, b, np.uint32(0))):
        got = (((w | a2) - b2) ^ c2).view(np.uint8).reshape(-1, 4).view(np.int8).astype(np.int16)
        assert not np.array_equal(got, want)
