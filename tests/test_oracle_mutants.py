"""The oracle's pins catch planted mistakes (CPU only).

Each case below plants one plausible mistake in a copy of oracle/oracle.c (a dropped term, a
wrong sign, a wrong index or layout, a swapped operand, a wrong tie-break or rounding), builds it
with the oracle's own compiler flags and runs tests/test_oracle_pins.py against it through the
ORACLE_LIB hook: every mutant must fail at least one pin. The unmodified source passes them (the
pin file itself runs in this suite).
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


def _build(src_text, out):
    c = out + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-pthread", "-o", out, c, "-lm"])


def _pins_fail(lib_path):
    env = dict(os.environ, ORACLE_LIB=lib_path)
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
