"""The tensor-core pass's dequantisation arithmetic (csrc/coarse_tc.cu), emulated step by step in
IEEE half precision on the CPU.

Per row the kernel takes e from the row's largest scale (S_max 2^e in [8, 16)); per code c of
plane p it forms r = 1 + c 4^p 2^-10 (the code put into the mantissa of 1.0), the multiplier
M = f16(S 2^(e + 10 - 2p)), and one fused multiply-add r M - M rounded once to f16. The claims
pinned here: the result is exactly c S 2^e whenever S 2^e >= 2^-17 (so for every scale of at
least 2^-20 of the row's largest), and below that it is off by less than one f16 subnormal step.
"""
import numpy as np
import pytest


def _bf16_bits(v: float) -> int:
    b = int(np.float32(v).view(np.uint32))
    return (b + 0x7FFF + ((b >> 16) & 1)) >> 16


def _scale_exponent(max_bits: int) -> int:
    """The kernel's e from the bf16 magnitude bits of the row's largest scale."""
    return 130 - (max_bits >> 7) if max_bits else 0


def _dequant(c: int, p: int, s_scaled: float) -> float:
    """c S 2^e as the kernel computes it, given s_scaled = S 2^e (a bf16 value times 2^e)."""
    r = np.float16(1.0 + c * 4.0 ** p / 1024.0)
    m = np.float16(np.float32(s_scaled) * np.float32(2.0 ** (10 - 2 * p)))  # __float2half_rn
    # the FMA: r m is exact in binary64 (two 11-bit significands), then one rounding to f16
    return float(np.float16(float(r) * float(m) - float(m)))


def _binade(x: int):
    """Every bf16 value in [2^x, 2^(x+1)): 128 mantissas."""
    return [(1 + k / 128) * 2.0 ** x for k in range(128)]


def test_scale_exponent_puts_the_largest_scale_in_8_16():
    for x in range(-60, 60):
        for s in _binade(x)[::7]:
            e = _scale_exponent(_bf16_bits(s) & 0x7FFF)
            assert 8.0 <= s * 2.0 ** e < 16.0, (s, e)
    assert _scale_exponent(0) == 0  # an all-zero row


@pytest.mark.parametrize("x", range(-17, 4))
def test_exact_from_2_to_the_minus_17(x):
    for s in _binade(x):
        for p in range(4):
            for c in range(4):
                assert _dequant(c, p, s) == c * s, (s, p, c)


def test_inexact_below_but_within_one_subnormal_step():
    inexact = 0
    for x in range(-40, -17):
        for s in _binade(x):
            for p in range(4):
                for c in range(4):
                    err = abs(_dequant(c, p, s) - c * s)
                    assert err < 2.0 ** -24
                    inexact += err > 0
    assert inexact > 0  # the threshold is real: the claim above is the boundary


def test_ratio_bound_holds_for_any_largest_scale():
    # whatever the mantissa of the row's largest scale, a scale at 2^-20 of it stays exact
    rng = np.random.default_rng(0)
    for _ in range(200):
        smax = float(np.float32(rng.uniform(1e-6, 1e2)))
        smax_b = _bf16_bits(smax) & 0x7FFF
        smax = float(np.uint32(smax_b << 16).view(np.float32))
        e = _scale_exponent(smax_b)
        for k in range(128):
            s = float(np.uint32((_bf16_bits(smax * 2.0 ** -20 * (1 + k / 128))) << 16)
                      .view(np.float32))
            if s < smax * 2.0 ** -20:
                continue
            for p in range(4):
                for c in range(4):
                    assert _dequant(c, p, s * 2.0 ** e) == c * s * 2.0 ** e


def test_fold_formula_matches_the_oracle():
    """The whole pass's arithmetic, with the kernel's operands: A = c S 2^e (exact, above), B = the
    f16 x 2^(15 - E_m), D = sum A B (here in fp64), then the fold D 2^(E_m - e - 17) plus the
    zero-point part sum_g (S - ZS) XS. That must be the page's coarse value (the oracle's), so the
    exponent offsets are right."""
    import oracle
    from bit_draft_lm_gb300 import synth
    M, K, N, G = 3, 1024, 64, 128
    w = synth.make_workload(M, K, N, 41, plant=False)
    packed, S, ZS = oracle.quantize_pack(w.W, G, 2)
    codes = oracle.unpack_codes(packed, K, 2).astype(np.float64)          # [N, K]
    Sv = synth.bf16_value(S).astype(np.float64)                          # [N, K/G]
    ZSv = synth.bf16_value(ZS).astype(np.float64)
    x = synth.bf16_value(w.x).astype(np.float64)                         # [M, K]
    e = np.array([_scale_exponent(int(np.max(S[n] & 0x7FFF))) for n in range(N)])
    A = codes * np.repeat(Sv, G, axis=1) * (2.0 ** e)[:, None]
    Em = np.array([(int(np.max(w.x[m] & 0x7FFF)) >> 7) - 126 for m in range(M)])
    B = np.stack([np.float16(x[m] * 2.0 ** (15 - Em[m])).astype(np.float64) for m in range(M)])
    D = B @ A.T                                                          # [M, N]
    XS = x.reshape(M, K // G, G).sum(axis=2)                             # [M, K/G]
    c = D * 2.0 ** (Em[:, None] - e[None, :] - 17) + XS @ (Sv - ZSv).T
    ref = oracle.coarse(w.x, packed, S, ZS, G, 2)
    scale = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    assert np.max(np.abs(c - ref) / scale) < 1e-9
