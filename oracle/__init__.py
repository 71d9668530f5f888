"""CPU oracle for the low-bit draft head -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. It wraps ``oracle.c`` (plain C, fp32 quantiser as the page states it, fp64 for
everything after it) through ctypes and shares no code with the CUDA library.

Every function takes and returns numpy arrays; bf16 tensors are carried as their uint16 bit
patterns. Functions and the passages they follow (page "radiance_drafthead.py"):

* ``quantize_pack``   -- the load-time quantiser: asymmetric min/max codes per (row, group),
                         quarter-split int2 / half-split int4 packing, S and ZS premultiplied.
* ``unpack_codes``    -- the packing read back (module docstring, on the quarter-split packing).
* ``coarse``          -- the int2 coarse kernel: ``sum_gi S*P_gi - ZS*XS_gi`` in fp64.
* ``coarse_dequant``  -- the same value as a dot with dequantised weights (fold self-check).
* ``block_topk``      -- the block candidate emission: top-KCAND per 64-row block.
* ``global_topr``     -- the head application's RERANK best block candidates.
* ``rerank``          -- the exact rerank: exact logits of the selected rows.
* ``argmax``          -- the argmax the caller takes.
* ``exact_logits``    -- brute force over every vocab row.
* ``topk_only``       -- the top-K-only output: every logit -inf, then the rerank's exact logits,
                         rounded to bf16, at the reranked ids.
* ``e4m3_decode``     -- the exact rerank on the FP8 head: the exact bit decode of an e4m3 byte.
* ``quantize_pack_fp8`` -- the load-time quantiser on the FP8 head: the e4m3 values times the fp32
                         per-row scale, then the same quantiser.
* ``rerank_fp8``      -- the exact rerank with FP8 rows: sum_k x_k * e4m3(W8[n,k]) * scale[n].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

BLOCK = 64


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/liboracle.so (strict IEEE: no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB: another build of oracle.c, for the pin tests' planted-mistake (mutant)
        # check; normally unset
        path = os.environ.get("ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        sigs = {
            "orc_quantize_pack": [P, I64, I64, I, I, P, P, P, I],
            "orc_quantize_pack_f32": [P, I64, I64, I, I, P, P, P, I],
            "orc_unpack_codes": [P, I64, I64, I, P],
            "orc_coarse": [P, I64, I64, P, P, P, I64, I, I, P, I],
            "orc_coarse_dequant": [P, I64, I64, P, P, P, I64, I, I, P, I],
            "orc_block_topk": [P, I64, I64, I, P, P],
            "orc_global_topr": [P, P, I64, I64, I, P, P],
            "orc_rerank": [P, I64, I64, P, I64, P, I, P],
            "orc_argmax": [P, P, I64, I, P],
            "orc_exact_logits": [P, I64, I64, P, I64, P, I],
        }
        for name, args in sigs.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    """Host threads the oracle uses (all cores this process may run on)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (status {rc})")


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def quantize_pack(W: np.ndarray, G: int = 128, bits: int = 2, nthreads: int | None = None):
    """W: uint16 [N, K] bf16 bits -> (packed uint8 [N, K*bits/8], S uint16 [N, K/G], ZS ditto)."""
    W = _u16(W)
    N, K = W.shape
    packed = np.empty((N, K * bits // 8), dtype=np.uint8)
    S = np.empty((N, K // G), dtype=np.uint16)
    ZS = np.empty((N, K // G), dtype=np.uint16)
    _check(_load().orc_quantize_pack(_p(W), N, K, G, bits, _p(packed), _p(S), _p(ZS),
                                     nthreads or threads()), "quantize_pack")
    return packed, S, ZS


def unpack_codes(packed: np.ndarray, K: int, bits: int = 2) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    codes = np.empty((N, K), dtype=np.uint8)
    _check(_load().orc_unpack_codes(_p(packed), N, K, bits, _p(codes)), "unpack_codes")
    return codes


def _coarse(fn, x, packed, S, ZS, G, bits, nthreads):
    x = _u16(x)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    S, ZS = _u16(S), _u16(ZS)
    M, K = x.shape
    N = packed.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    _check(fn(_p(x), M, K, _p(packed), _p(S), _p(ZS), N, G, bits, _p(out),
              nthreads or threads()), "coarse")
    return out


def coarse(x, packed, S, ZS, G: int = 128, bits: int = 2, nthreads: int | None = None):
    """fp64 coarse values c[M, N]."""
    return _coarse(_load().orc_coarse, x, packed, S, ZS, G, bits, nthreads)


def coarse_dequant(x, packed, S, ZS, G: int = 128, bits: int = 2, nthreads: int | None = None):
    """fp64 coarse values via explicit dequantised weights (self-check form)."""
    return _coarse(_load().orc_coarse_dequant, x, packed, S, ZS, G, bits, nthreads)


def block_topk(c: np.ndarray, kcand: int):
    """c fp64 [M, N] -> (cand_val fp64 [M, nblk*kcand], cand_id int32 [M, nblk*kcand])."""
    c = np.ascontiguousarray(c, dtype=np.float64)
    M, N = c.shape
    nblk = (N + BLOCK - 1) // BLOCK
    val = np.empty((M, nblk * kcand), dtype=np.float64)
    ids = np.empty((M, nblk * kcand), dtype=np.int32)
    _check(_load().orc_block_topk(_p(c), M, N, kcand, _p(val), _p(ids)), "block_topk")
    return val, ids


def global_topr(cand_val: np.ndarray, cand_id: np.ndarray, R: int):
    """-> (rr_id int32 [M, R], rr_coarse fp64 [M, R]) in descending coarse order."""
    cand_val = np.ascontiguousarray(cand_val, dtype=np.float64)
    cand_id = np.ascontiguousarray(cand_id, dtype=np.int32)
    M, ncand = cand_val.shape
    rr = np.empty((M, R), dtype=np.int32)
    rv = np.empty((M, R), dtype=np.float64)
    _check(_load().orc_global_topr(_p(cand_val), _p(cand_id), M, ncand, R, _p(rr), _p(rv)),
           "global_topr")
    return rr, rv


def rerank(x, W, ids):
    """Exact fp64 logits e[M, R] of rows ids[M, R]."""
    x, W = _u16(x), _u16(W)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    M, K = x.shape
    N = W.shape[0]
    R = ids.shape[1]
    e = np.empty((M, R), dtype=np.float64)
    _check(_load().orc_rerank(_p(x), M, K, _p(W), N, _p(ids), R, _p(e)), "rerank")
    return e


def argmax(e, ids):
    e = np.ascontiguousarray(e, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    M, R = e.shape
    out = np.empty(M, dtype=np.int32)
    _check(_load().orc_argmax(_p(e), _p(ids), M, R, _p(out)), "argmax")
    return out


def exact_logits(x, W, nthreads: int | None = None):
    x, W = _u16(x), _u16(W)
    M, K = x.shape
    N = W.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    _check(_load().orc_exact_logits(_p(x), M, K, _p(W), N, _p(out), nthreads or threads()),
           "exact_logits")
    return out


def head(x, packed, S, ZS, W, G=128, bits=2, kcand=8, R=16, nthreads=None):
    """The whole path for one batch: coarse -> block top-K -> global top-R -> rerank -> argmax."""
    c = coarse(x, packed, S, ZS, G, bits, nthreads)
    cv, ci = block_topk(c, kcand)
    rr, rc = global_topr(cv, ci, R)
    e = rerank(x, W, rr)
    am = argmax(e, rr)
    return {"coarse": c, "cand_val": cv, "cand_id": ci, "rr_id": rr, "rr_coarse": rc,
            "rr_logit": e, "argmax": am}


def bf16_rne(v: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def topk_only(rr_id: np.ndarray, rr_logit: np.ndarray, N: int) -> np.ndarray:
    """bf16 bits [M, N]: -inf (0xFF80) everywhere, then bf16(rr_logit[m, j]) at rr_id[m, j] --
    the logits a top-K caller ranks (page: the top-K-only output)."""
    M, R = rr_id.shape
    y = np.full((M, N), 0xFF80, dtype=np.uint16)
    for m in range(M):
        for j in range(R):
            n = int(rr_id[m, j])
            if 0 <= n < N:
                y[m, n] = bf16_rne(np.float32(rr_logit[m, j]).reshape(1))[0]
    return y


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """e4m3 bytes -> float64, the page's bit decode: exponent e = (b >> 3) & 15, mantissa
    m = b & 7; e == 0: m * 2^-9, else (1 + m/8) * 2^(e - 7); bit 7 the sign."""
    b = np.asarray(b, dtype=np.int64)
    e = (b >> 3) & 15
    m = (b & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m * 0.125) * np.exp2((e - 7).astype(np.float64)))
    return np.where((b & 128) != 0, -mag, mag)


def quantize_pack_fp8(W8: np.ndarray, scale: np.ndarray, G: int = 128, bits: int = 2,
                      nthreads: int | None = None):
    """W8 uint8 [N, K] e4m3 rows, scale fp32 [N] -> (packed, S, ZS) of the values
    fp32(e4m3(W8)) * fp32(scale) (one IEEE single multiply)."""
    W8 = np.ascontiguousarray(W8, dtype=np.uint8)
    N, K = W8.shape
    Wf = np.ascontiguousarray(e4m3_decode(W8).astype(np.float32) *
                              np.asarray(scale, dtype=np.float32)[:, None])
    per = 8 // bits
    packed = np.empty((N, K // per), dtype=np.uint8)
    S = np.empty((N, K // G), dtype=np.uint16)
    ZS = np.empty((N, K // G), dtype=np.uint16)
    _check(_load().orc_quantize_pack_f32(_p(Wf), N, K, G, bits, _p(packed), _p(S), _p(ZS),
                                         nthreads or threads()), "quantize_pack_f32")
    return packed, S, ZS


def bf16_bits_to_f64(u: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rerank_fp8(x, W8, scale, ids):
    """Exact logits against FP8 rows: e[m, j] = sum_k x[m, k] * e4m3(W8[n, k]) * scale[n]
    (fp64), n = ids[m, j]; -inf for ids outside [0, N)."""
    xf = bf16_bits_to_f64(np.asarray(x))
    M, R = ids.shape
    N = W8.shape[0]
    e = np.full((M, R), -np.inf)
    for m in range(M):
        for j in range(R):
            n = int(ids[m, j])
            if 0 <= n < N:
                e[m, j] = float(np.dot(xf[m], e4m3_decode(W8[n])) * float(scale[n]))
    return e
