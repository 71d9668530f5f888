"""Seeded synthetic inputs for the int2 draft head.

This module only draws random numbers and encodes them as bf16 bit patterns. It holds none of
the head's arithmetic (no quantisation, no projection, no selection), so the CPU oracle and the
CUDA path can both be fed from it without sharing any of the method's code.

Recipe (numpy ``default_rng(seed)``, float64 draws, one bf16 round-to-nearest-even cast):

* hidden states ``x[M, K]``: z ~ N(0, 1) per row; for the vocabulary-scale workloads each row is
  RMS-normalised, ``x = z / sqrt(mean(z**2))`` (the draft head sees the output of the final
  RMS-norm; no gamma), the small workload keeps z as drawn.
* head weight ``W[N, K]`` (vocab rows, the lm_head layout): ``0.02 * exp(0.3 * u_n) * z_nk`` with
  u, z ~ N(0, 1), i.e. lognormal(sigma 0.3) row norms, or plain ``0.02 * z`` for the small
  workload.
* 16 planted vocab rows (chosen by the seed) are scaled by 3 before the cast, and oriented so that
  their logit against hidden row 0 is non-negative.
* 4 near-tie pairs (a, b), a planted: row b copies row a except at ``k* = argmax_k |x[0, k]|``,
  where it is moved by about ``1e-3 / x[0, k*]`` (at least one bf16 step), so the exact logits of
  a and b against hidden row 0 differ by about 1e-3. Two pairs share a 64-row block, two sit in
  neighbouring blocks.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Tuple

import numpy as np

BLOCK_ROWS = 64          # width of one candidate block (vocab rows)
N_PLANTED = 16
N_PAIRS = 4
TIE_GAP = 1e-3


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), round to nearest, ties to even, in one step.

    frexp gives a in [0.5, 1) * 2**e; the bf16 significand has 8 bits, so the value rounds to
    rint(m * 256) / 256 * 2**e exactly in float64 (rint is ties-to-even); the result is then
    representable in bf16 and float32, so the float32 view's top half is the encoding.
    """
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)
    r = np.ldexp(np.rint(m * 256.0), e - 8)
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Workload:
    name: str
    M: int
    K: int
    N: int
    seed: int
    x: np.ndarray            # uint16 [M, K] bf16 bits
    W: np.ndarray            # uint16 [N, K] bf16 bits
    planted: np.ndarray      # int64 [16] planted vocab rows
    pairs: np.ndarray        # int64 [4, 2] near-tie pairs (a, b)
    kstar: int               # column where each pair differs


def _pick_pairs(rng: np.random.Generator, N: int, planted: np.ndarray) -> np.ndarray:
    taken = set(int(p) for p in planted)
    pairs = []
    for i in range(N_PAIRS):
        a = int(planted[i])
        blk = a // BLOCK_ROWS
        for _ in range(1000):
            if i < 2:      # same 64-row block
                lo = blk * BLOCK_ROWS
                hi = min(lo + BLOCK_ROWS, N)
                b = int(rng.integers(lo, hi))
            else:          # neighbouring block
                nb = blk + 1 if (blk + 1) * BLOCK_ROWS < N else blk - 1
                lo = nb * BLOCK_ROWS
                hi = min(lo + BLOCK_ROWS, N)
                b = int(rng.integers(lo, hi))
            if b not in taken:
                break
        else:  # pragma: no cover - only for absurdly small N
            raise ValueError("cannot place near-tie pair")
        taken.add(b)
        pairs.append((a, b))
    return np.asarray(pairs, dtype=np.int64)


def make_workload(M: int, K: int, N: int, seed: int, rms_norm: bool = True,
                  lognormal_rows: bool = True, name: str = "", plant: bool = True) -> Workload:
    """Draw one workload; see the module docstring for the recipe. ``plant=False`` skips the
    planted rows and near-tie pairs (for very small N)."""
    if not plant:
        rng = np.random.default_rng(seed)
        z = rng.standard_normal((M, K))
        if rms_norm:
            z = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True))
        scale = 0.02 * (np.exp(0.3 * rng.standard_normal(N)) if lognormal_rows else np.ones(N))
        W = bf16_bits(rng.standard_normal((N, K)) * scale[:, None])
        return Workload(name or f"M{M}_K{K}_N{N}_s{seed}_plain", M, K, N, seed, bf16_bits(z), W,
                        np.zeros(0, dtype=np.int64), np.zeros((0, 2), dtype=np.int64), 0)
    if N < 2 * BLOCK_ROWS or N < N_PLANTED + N_PAIRS:
        raise ValueError("N too small for the planting recipe")
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((M, K))
    if rms_norm:
        z = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    x = bf16_bits(z)
    row_scale = 0.02 * (np.exp(0.3 * rng.standard_normal(N)) if lognormal_rows else np.ones(N))
    planted = np.sort(rng.choice(N, size=N_PLANTED, replace=False)).astype(np.int64)
    row_scale[planted] *= 3.0
    pairs = _pick_pairs(rng, N, planted)
    tie_sign = rng.choice([-1.0, 1.0], size=N_PAIRS)

    W = np.empty((N, K), dtype=np.uint16)
    chunk = 8192
    for r0 in range(0, N, chunk):
        r1 = min(r0 + chunk, N)
        W[r0:r1] = bf16_bits(rng.standard_normal((r1 - r0, K)) * row_scale[r0:r1, None])

    x0 = bf16_value(x[0])
    for p in planted:                      # orient planted rows towards hidden row 0
        if float(np.dot(bf16_value(W[p]), x0)) < 0.0:
            W[p] ^= np.uint16(0x8000)      # exact sign flip of every element
    kstar = int(np.argmax(np.abs(x0)))
    for (a, b), s in zip(pairs, tie_sign):
        W[b] = W[a]
        wa = bf16_value(W[a, kstar])
        target = wa + s * TIE_GAP / x0[kstar]
        nb = bf16_bits(np.float64(target))
        if int(nb) == int(W[a, kstar]):    # at least one bf16 step away from row a
            nb = _bf16_step(W[a, kstar], s * x0[kstar] > 0)
        W[b, kstar] = nb
    return Workload(name or f"M{M}_K{K}_N{N}_s{seed}", M, K, N, seed, x, W, planted, pairs, kstar)


def _bf16_step(bits: np.uint16, up: bool) -> np.uint16:
    """The bf16 neighbour of `bits` one step towards +inf (up) or -inf."""
    b = int(bits)
    neg = bool(b & 0x8000)
    mag = b & 0x7FFF
    if up != neg:          # moving away from zero in magnitude
        mag += 1
    elif mag == 0:         # crossing zero
        neg = not neg
        mag = 1
    else:
        mag -= 1
    return np.uint16((0x8000 if neg else 0) | mag)


# Named workloads: the small draft head and the vocabulary-scale draft head at three row counts,
# the 4-bit comparison and the group-64 ablation.
WORKLOADS: Dict[str, Tuple[int, int, int, int, bool]] = {
    # name: (M, K, N, seed, vocabulary-scale distributions)
    "tiny_m1_k1024_n8192": (1, 1024, 8192, 0, False),
    "head_m1_k5120_n124160": (1, 5120, 124160, 1, True),
    "head_m8_k5120_n124160": (8, 5120, 124160, 2, True),
    "head_m72_k5120_n124160": (72, 5120, 124160, 3, True),
    "head_m8_k5120_n124160_ablation": (8, 5120, 124160, 4, True),
}

_CACHE: Dict[str, Workload] = {}


def named(name: str) -> Workload:
    """Draw (and memoise in this process) one of the named workloads."""
    if name not in _CACHE:
        M, K, N, seed, big = WORKLOADS[name]
        _CACHE[name] = make_workload(M, K, N, seed, rms_norm=big, lognormal_rows=big, name=name)
    return _CACHE[name]


def hidden_rows(M: int, K: int, seed: int, rms_norm: bool = True) -> np.ndarray:
    """M fresh hidden rows (bf16 bits [M, K]) by the recipe above: z ~ N(0, 1), RMS-normalised
    unless ``rms_norm`` is False. Used with a cached head to draw more rows without redrawing W."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((M, K))
    if rms_norm:
        z = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    return bf16_bits(z)


RECALL_HEAD = "head_m1_k5120_n124160"
RECALL_ROWS, RECALL_SEED = 64, 7


def recall_rows(w: Workload) -> np.ndarray:
    """The hidden rows of the recall report on head ``w``: its own row 0 (the planted rows and
    near-tie pairs face it), then RECALL_ROWS - 1 fresh rows of seed RECALL_SEED."""
    x = hidden_rows(RECALL_ROWS, w.K, RECALL_SEED)
    x[0] = w.x[0]
    return x


def wide_range_rows(M: int, K: int, seed: int) -> np.ndarray:
    """Hidden rows with an extreme dynamic range (bf16 bits [M, K]), to exercise the kernels'
    per-row power-of-two scaling of x: row 0 is 2^-20 z with two spikes of +-2^12; row 1 is
    2^-20 z alone (a tiny maximum); row 2 mixes 2^-20 z and z halves (a spike-free wide range);
    further rows are plain RMS-normalised draws."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((M, K))
    z = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    if M > 0:
        z[0] *= 2.0 ** -20
        i, j = rng.choice(K, 2, replace=False)
        z[0, i], z[0, j] = 2.0 ** 12, -(2.0 ** 12)
    if M > 1:
        z[1] *= 2.0 ** -20
    if M > 2:
        z[2, : K // 2] *= 2.0 ** -20
    return bf16_bits(z)


def wide_scale_range_head(W: np.ndarray, G: int, seed: int) -> np.ndarray:
    """A head whose scale groups span a wide range within each row (bf16 bits [N, K] in and out):
    every G-wide group of a row is multiplied by 2^-k, k drawn per (row, group) from
    {0, 0, 0, 8, 16, 22, 26, 30}; row 0 keeps one group at full size and shrinks every other by
    2^-30, and row 1 is shrunk by 2^-30 as a whole. Powers of two keep every bf16 exact."""
    rng = np.random.default_rng(seed)
    N, K = W.shape
    kg = rng.choice(np.array([0, 0, 0, 8, 16, 22, 26, 30]), size=(N, K // G))
    if N > 0:
        kg[0] = 30
        kg[0, rng.integers(K // G)] = 0
    if N > 1:
        kg[1] = 30
    f = np.repeat(np.ldexp(1.0, -kg), G, axis=1)
    return bf16_bits(bf16_value(W) * f)


def fp8_head(W: np.ndarray):
    """An FP8 per-channel head built from a bf16 head (bit patterns uint16 [N, K]): the fp32
    row scale max|W[n]| / 448 and the e4m3 bytes of W / scale (round to nearest even, the
    float8_e4m3fn conversion). Returns (W8 uint8 [N, K], scale float32 [N])."""
    import torch
    w = torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).view(torch.bfloat16).float()
    scale = (w.abs().amax(dim=1) / 448.0).clamp(min=1e-12)
    w8 = (w / scale[:, None]).to(torch.float8_e4m3fn)
    return w8.view(torch.uint8).numpy().copy(), scale.numpy().astype(np.float32)
