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


@pytest.mark.parametrize("bits,G", [(2, 128), (2, 64), (4, 128), (4, 64)])
def test_warp_mma_scaling_constants_match_the_oracle(bits, G):
    """The warp-MMA pass's operands and scale factors, composed in fp64: A = code 2^(s - 24) (the
    f16 subnormals above), B = f16(x 2^(15 - E - s)) with E from the largest |x| of the warp's
    strip (64 packed bytes of every plane), and each partial times S_g 2^(E + 9 - log2 L)
    (L = 4 for int2, 16 for int4), plus the zero-point part sum_g (S - ZS) XS: that is the page's
    coarse value (the oracle's), so the exponent offsets are right."""
    M, K, N = 3, 2048, 64
    w = synth.make_workload(M, K, N, 51 + bits + G, plant=False)
    packed, S, ZS = oracle.quantize_pack(w.W, G, bits)
    codes = oracle.unpack_codes(packed, K, bits).astype(np.float64)      # [N, K]
    Sv = synth.bf16_value(S).astype(np.float64)
    ZSv = synth.bf16_value(ZS).astype(np.float64)
    x = synth.bf16_value(w.x).astype(np.float64)
    RB = K * bits // 8
    k = np.arange(K)
    plane, byte = k // RB, k % RB
    shift = bits * plane
    strip = byte // 64
    logL = 2 if bits == 2 else 4
    A = codes * 2.0 ** (shift - 24)                                      # [N, K]
    c = np.zeros((M, N))
    for m in range(M):
        E = np.zeros(K, dtype=np.int64)
        for j in range(RB // 64):
            sel = strip == j
            mx = int(np.max(w.x[m][sel] & 0x7FFF))
            E[sel] = min(max((mx >> 7) - 126, -100), 100)
        B = np.float16(x[m] * 2.0 ** (15 - E - shift)).astype(np.float64)
        c[m] = (A * B * 2.0 ** (E + 9 - logL) * np.repeat(Sv, G, axis=1)).sum(axis=1)
    XS = x.reshape(M, K // G, G).sum(axis=2)
    c += XS @ (Sv - ZSv).T
    ref = oracle.coarse(w.x, packed, S, ZS, G, bits)
    scale = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    assert np.max(np.abs(c - ref) / scale) < 1e-9
