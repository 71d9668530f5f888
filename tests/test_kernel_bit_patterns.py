"""The coarse kernels' word-level dequantisation, checked on the CPU against the oracle's packing.

Both kernels read the packed head (the page's quarter-split int2 byte, or half-split int4 byte)
32 bits at a time. For a word t holding bytes b0..b3 of row positions 4w..4w+3, and plane p
(weight shift s = 2p for int2, 4p for int4), they rely on:

* warp-MMA pass: the two 16-bit halves of t & (code mask << s) are the f16 values
  code(b0, p) 2^(s - 24) and code(b2, p) 2^(s - 24) (f16 subnormals), and the same AND of t >> 8
  gives code(b1, p) and code(b3, p);
* tensor-core pass (int2): the halves of (t & (0x0003 << 2p, twice)) | 0x3C00 3C00 are
  1 + code 4^p 2^-10;

where code(b, p) is the weight at hidden index p * RB + b (RB = packed bytes per row). Here the
words come from oracle.quantize_pack and the codes from oracle.unpack_codes.
"""
import numpy as np
import pytest

import oracle
from bit_draft_lm_gb300 import synth


def _halves_f16(v: np.ndarray):
    lo = (v & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    hi = (v >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    return lo, hi


@pytest.mark.parametrize("bits,G", [(2, 128), (2, 64), (4, 128)])
def test_word_ops_recover_the_oracles_codes(bits, G):
    N, K = 16, 2048
    w = synth.make_workload(1, K, N, 7 + bits, plant=False)
    packed, _, _ = oracle.quantize_pack(w.W, G, bits)
    codes = oracle.unpack_codes(packed, K, bits).astype(np.float64)
    RB = K * bits // 8
    P = 8 // bits
    cmask = (1 << bits) - 1
    t = np.ascontiguousarray(packed).view("<u4").astype(np.uint64)  # [N, RB / 4]
    b = 4 * np.arange(RB // 4)
    for p in range(P):
        s = bits * p
        mask = ((cmask << s) | (cmask << (s + 16)))
        c = [codes[:, p * RB + b + j] for j in range(4)]  # bytes b0..b3 of every word
        even_lo, even_hi = _halves_f16(t & mask)
        odd_lo, odd_hi = _halves_f16((t >> 8) & mask)
        unit = 2.0 ** (s - 24)
        assert np.array_equal(even_lo, c[0] * unit) and np.array_equal(even_hi, c[2] * unit)
        assert np.array_equal(odd_lo, c[1] * unit) and np.array_equal(odd_hi, c[3] * unit)
        if bits == 2:
            one = 0x3C003C00
            e_lo, e_hi = _halves_f16((t & mask) | one)
            o_lo, o_hi = _halves_f16(((t >> 8) & mask) | one)
            f = 4.0 ** p / 1024.0
            assert np.array_equal(e_lo, 1 + c[0] * f) and np.array_equal(e_hi, 1 + c[2] * f)
            assert np.array_equal(o_lo, 1 + c[1] * f) and np.array_equal(o_hi, 1 + c[3] * f)


def test_every_byte_value():
    # all 256 byte values in every byte slot of a word, int2: the masks separate the planes
    for v in range(256):
        for slot in range(4):
            t = np.array([v << (8 * slot)], dtype=np.uint64)
            for p in range(4):
                code = (v >> (2 * p)) & 3
                mask = (3 << 2 * p) | (3 << (2 * p + 16))
                src = t if slot % 2 == 0 else t >> 8
                lo, hi = _halves_f16(src & mask)
                want = code * 2.0 ** (2 * p - 24)
                got = lo[0] if slot < 2 else hi[0]
                other = hi[0] if slot < 2 else lo[0]
                assert got == want and other == 0.0
