"""The arithmetic the MXFP4 GEMMs decode with, checked on the CPU against the
oracle's E2M1 values (the GPU tests check the kernels themselves, bit for
bit, against the bf16 GEMMs on the dequantized weights).

The library stores a feature's codes along K eight to a little-endian 32-bit
word: k = 8i + 2j at bits 4j .. 4j + 3 and k = 8i + 2j + 1 at bits
16 + 4j .. 19 + 4j (include/moe_prefill.h).  The decode takes pair j with
one mask, one multiply by 2^(6 - 4j) + 2^(12 - 4j) (after a shift right by
8 for j = 2, 3) and one mask, which places a code's magnitude bits at bf16
bits 8..6 and its sign at bit 15: the bf16 value is value(code) x 2^-126 for
all 16 codes.  One bf16 multiply by 2^(S-1) then gives value(code) x
2^(S-127), exactly while S <= 128 (2^(S-1) is a finite bf16 value).
"""
import struct

import oracle


def bf16_value(h: int) -> float:
    return struct.unpack(">f", struct.pack(">I", (h & 0xFFFF) << 16))[0]


def word_of(codes):
    """Eight codes (k = 0..7) -> the library's 32-bit code word."""
    w = 0
    for i, c in enumerate(codes):
        w |= c << (4 * (i >> 1) + 16 * (i & 1))
    return w


def pair_bits(w: int, j: int) -> int:
    """The decode's bf16 pair for pair j of a code word (low half: even k)."""
    x = w >> 8 if j & 2 else w
    if j & 1:
        t = (x & 0x00F000F0) * 0x104
    else:
        t = (x & 0x000F000F) * 0x1040
    return t & 0x81C081C0


def test_bit_placement_reads_value_times_2_to_minus_126_for_every_code():
    for c_even in range(16):
        for c_odd in range(16):
            for j in range(4):
                codes = [0] * 8
                codes[2 * j], codes[2 * j + 1] = c_even, c_odd
                u = pair_bits(word_of(codes), j)
                assert bf16_value(u) * 2.0 ** 126 == oracle.e2m1_value(c_even)
                assert bf16_value(u >> 16) * 2.0 ** 126 == oracle.e2m1_value(c_odd)
                # the sign of a zero code survives (-0 stays -0)
                if c_even == 8:
                    assert u & 0x8000


def test_pairs_of_one_word_do_not_disturb_each_other():
    # every word of a few code patterns: each pair decodes from its own bits only
    patterns = [[15] * 8, [7, 8, 1, 9, 6, 14, 0, 15], [i * 2 + 1 for i in range(8)]]
    for codes in patterns:
        w = word_of(codes)
        for j in range(4):
            u = pair_bits(w, j)
            assert bf16_value(u) * 2.0 ** 126 == oracle.e2m1_value(codes[2 * j])
            assert bf16_value(u >> 16) * 2.0 ** 126 == oracle.e2m1_value(codes[2 * j + 1])


def test_scale_multiply_is_exact_up_to_s_128():
    for S in range(0, 129):
        scale_bits = (S + 126) << 7          # bf16 2^(S-1), a normal value
        scale = bf16_value(scale_bits)
        assert scale == 2.0 ** (S - 1)
        for c in range(16):
            u = pair_bits(word_of([c] + [0] * 7), 0)
            prod = bf16_value(u) * scale     # exact in fp64
            want = oracle.e2m1_value(c) * 2.0 ** (S - 127)
            assert prod == want
            # and a bf16 value (at most 2 significant bits, exponent in range)
            if prod != 0:
                assert bf16_value(struct.unpack(">I", struct.pack(">f", prod))[0] >> 16) == prod
    # S = 129 would need 2^128, which bf16 cannot hold: such blocks take the
    # decode's fp32 path
    assert (129 + 126) << 7 == 0x7F80  # the bf16 infinity pattern
