"""The oracle's pins catch planted mistakes (CPU only).

Each case below plants one plausible mistake (a dropped term, a wrong sign, a wrong index or
layout, a swapped operand, a wrong tie-break or rounding) in a copy of the oracle and runs
tests/test_oracle_pins.py against it: every mutant must fail at least one pin.
- C mutants of oracle/oracle.c are built with the oracle's own compiler flags and loaded through
  the ORACLE_LIB hook.
- Python mutants of oracle/__init__.py (the e4m3 decode, the FP8 quantiser's input, the FP8
  rerank, bf16 rounding, the top-K logits) are loaded as the `oracle` module through the
  ORACLE_PY hook of tests/conftest.py.
The unmodified sources pass the pins (the pin file itself runs in this suite, and a fresh build
of the unmodified C source is checked below).
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("levels: 2^bits instead of 2^bits - 1",
     "float sc = (hi - lo) / lv;", "float sc = (hi - lo) / (lv + 1.0f);"),
    ("zero point: sign of lo",
     "float zp = rintf(-lo / sc);", "float zp = rintf(lo / sc);"),
    ("code: zero point subtracted",
     "float r = rintf(v / sc + zp);", "float r = rintf(v / sc - zp);"),
    ("code: rounding half away from zero",
     "float r = rintf(v / sc + zp);", "float r = roundf(v / sc + zp);"),
    ("S: bias factor dropped",
     "float s4 = bias * sc;", "float s4 = sc;"),
    ("ZS: zero-point term subtracted",
     "c->ZS[n * ng + gi] = float_to_bf16(s4 + zs);", "c->ZS[n * ng + gi] = float_to_bf16(s4 - zs);"),
    ("bf16 store: truncation instead of round-to-nearest-even",
     "u += 0x7fffu + lsb;", "u += 0u * lsb;"),
    ("int2 packing: quarters 1 and 2 swapped",
     "(q[Q + j] << 2) | (q[2 * Q + j] << 4)", "(q[2 * Q + j] << 2) | (q[Q + j] << 4)"),
    ("int4 packing: nibbles swapped",
     "out[j] = (uint8_t)(q[j] | (q[H + j] << 4));", "out[j] = (uint8_t)(q[H + j] | (q[j] << 4));"),
    ("unpack: interleaved instead of quarter-split",
     "return (row[k % Q] >> (2 * (int)(k / Q))) & 3;", "return (row[k / 4] >> (2 * (int)(k % 4))) & 3;"),
    ("coarse: zero-point term dropped",
     "acc += s * pg - zs * xs;", "acc += s * pg;"),
    ("coarse: the 1 of 1 + v/beta dropped",
     "d[k] = 1.0 + (double)v[k] / beta;", "d[k] = (double)v[k] / beta;"),
    ("selection: equal values to the highest id",
     "return (x->id > y->id) - (x->id < y->id);", "return (x->id < y->id) - (x->id > y->id);"),
    ("block top-K: empty slots get id 0",
     "cand_id[o] = s < cnt ? buf[s].id : -1;", "cand_id[o] = s < cnt ? buf[s].id : 0;"),
    ("rerank: row offset without the K stride",
     "exact_dot(x + m * K, W + (int64_t)n * K, K)", "exact_dot(x + m * K, W + (int64_t)n, K)"),
    ("argmax: equal logits to the highest id",
     "ids[m * R + j] < ids[m * R + best]", "ids[m * R + j] > ids[m * R + best]"),
]


PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")

# (name, text in oracle/__init__.py, replacement)
PY_MUTANTS = [
    ("e4m3: subnormal step 2^-10",
     "m * 2.0 ** -9, (1.0", "m * 2.0 ** -10, (1.0"),
    ("e4m3: exponent bias 8",
     "np.exp2((e - 7).astype(np.float64))", "np.exp2((e - 8).astype(np.float64))"),
    ("e4m3: sign from bit 6",
     "np.where((b & 128) != 0, -mag, mag)", "np.where((b & 64) != 0, -mag, mag)"),
    ("bf16 rounding: ties away from zero",
     "((u + 0x7FFF + ((u >> 16) & 1)) >> 16)", "((u + 0x8000) >> 16)"),
    ("top-K logits: +inf fill",
     "y = np.full((M, N), 0xFF80, dtype=np.uint16)", "y = np.full((M, N), 0x7F80, dtype=np.uint16)"),
    ("FP8 quantiser: row scale not applied",
     "e4m3_decode(W8).astype(np.float32) *\n                              np.asarray(scale, dtype=np.float32)[:, None]",
     "e4m3_decode(W8).astype(np.float32) *\n                              np.float32(1.0)"),
    ("FP8 rerank: row scale dropped",
     "e4m3_decode(W8[n])) * float(scale[n]))", "e4m3_decode(W8[n])))"),
]


def _build(src_text, out):
    c = out + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-pthread", "-o", out, c, "-lm"])


def _pins_fail(lib_path, py_path=None):
    env = dict(os.environ, ORACLE_LIB=lib_path) if lib_path else dict(os.environ)
    if py_path:
        env["ORACLE_PY"] = py_path
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode != 0, r.stdout[-400:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    src = open(SRC).read()
    libs = []
    for i, (name, old, new) in enumerate(MUTANTS):
        assert src.count(old) == 1, f"mutation site not unique or missing: {name}"
        out = str(tmp_path / f"mutant{i}.so")
        _build(src.replace(old, new), out)
        libs.append(out)
    with ThreadPoolExecutor(max_workers=4) as pool:
        results = list(pool.map(_pins_fail, libs))
    survived = [(name, tail) for (name, _, _), (failed, tail) in zip(MUTANTS, results)
                if not failed]
    assert not survived, "mutants the pins did not catch: " + "; ".join(n for n, _ in survived)


def test_unmodified_copy_passes_the_pins(tmp_path):
    """The hook itself: the pins pass on a fresh build of the unmodified source."""
    out = str(tmp_path / "same.so")
    _build(open(SRC).read(), out)
    failed, tail = _pins_fail(out)
    assert not failed, tail


def test_every_planted_python_mistake_fails_a_pin(tmp_path):
    src = open(PY_SRC).read()
    c_src = open(SRC).read()
    paths = []
    for i, (name, old, new) in enumerate(PY_MUTANTS):
        old, new = old.replace("\\n", "\n"), new.replace("\\n", "\n")
        assert src.count(old) == 1, f"mutation site not unique or missing: {name}"
        d = tmp_path / f"pymut{i}"
        d.mkdir()
        (d / "__init__.py").write_text(src.replace(old, new))
        (d / "oracle.c").write_text(c_src)  # the mutant package builds its own library copy
        paths.append(str(d / "__init__.py"))
    with ThreadPoolExecutor(max_workers=4) as pool:
        results = list(pool.map(lambda p: _pins_fail(None, p), paths))
    survived = [name for (name, _, _), (failed, _) in zip(PY_MUTANTS, results) if not failed]
    assert not survived, "mutants the pins did not catch: " + "; ".join(survived)
