"""The hidden states' f16 operand in both coarse kernels, emulated in IEEE half precision on the CPU.

Each kernel takes e from the largest |x| of a row (the tensor-core pass) or of a warp's strip of
a row (the warp-MMA pass): e = bf16 exponent field - 126, so max |x| lies in [2^(e-1), 2^e),
clamped to [-100, 100]. It converts x * 2^(15 - e - shift) to f16 with round-to-nearest, where
shift is 0 in the tensor-core pass and the plane's weight shift in the warp-MMA pass (2p for
int2, 4p for int4). The claims pinned here: the f16 value is exact whenever it is at least 2^-17,
so for every element of at least 2^(shift - 31) of the largest; below that it is off by less
than one f16 subnormal step; nothing overflows.
"""
import numpy as np
import pytest


def _bits(v: float) -> int:
    b = int(np.float32(v).view(np.uint32))
    return (b + 0x7FFF + ((b >> 16) & 1)) >> 16  # bf16 round-to-nearest-even


def _val(bits: int) -> float:
    return float(np.uint32(bits << 16).view(np.float32))


def _exponent(max_bits: int) -> int:
    e = (max_bits >> 7) - 126
    return -100 if e < -100 else (100 if e > 100 else e)


def _to_f16(x: float, e: int, shift: int) -> float:
    return float(np.float16(np.float32(x) * np.float32(2.0 ** (15 - e - shift))))


SHIFTS = [0, 2, 4, 6]


@pytest.mark.parametrize("shift", SHIFTS)
def test_exact_above_threshold_and_no_overflow(shift):
    rng = np.random.default_rng(shift)
    for _ in range(40):
        xmax = _val(_bits(float(rng.uniform(0.5, 1.0)) * 2.0 ** int(rng.integers(-40, 40))))
        e = _exponent(_bits(xmax) & 0x7FFF)
        assert 2.0 ** (e - 1) <= xmax < 2.0 ** e
        scale = 2.0 ** (15 - e - shift)
        # every bf16 value from the threshold up to the largest
        for k in range(0, 31 - shift + 1):
            for m in range(128):
                x = _val(_bits(xmax * 2.0 ** -k * (1 + m / 128) / 2))
                if x > xmax or x < xmax * 2.0 ** (shift - 31):
                    continue
                for sgn in (1.0, -1.0):
                    got = _to_f16(sgn * x, e, shift)
                    assert got == sgn * x * scale, (x, e, shift)
                    assert abs(got) < 65504.0


@pytest.mark.parametrize("shift", SHIFTS)
def test_below_threshold_within_one_subnormal_step(shift):
    inexact = 0
    e = 3  # max |x| in [4, 8)
    scale = 2.0 ** (15 - e - shift)
    for x_exp in range(e - 45, e - 31 + shift):
        for m in range(128):
            x = (1 + m / 128) * 2.0 ** x_exp
            err = abs(_to_f16(x, e, shift) - x * scale)
            assert err < 2.0 ** -24
            inexact += err > 0
    assert inexact > 0  # the threshold is the boundary


def test_zero_and_tiny_rows():
    assert _exponent(0) == -100  # an all-zero row: e clamped, every x is 0
    assert _to_f16(0.0, -100, 0) == 0.0
    tiny = _val(0x0001)  # the smallest bf16 subnormal as the largest |x|
    e = _exponent(0x0001)
    assert e == -100 and _to_f16(tiny, e, 0) > 0.0
