"""Writes tests/golden/recall_k5120_n124160_m64.json: the recall of the method on the
vocabulary-scale synthetic head, computed by the oracle alone.

The page "radiance_drafthead.py" (module docstring, the paragraphs on accuracy from reranking and
on KCAND as the lever) claims that the int2 head with KCAND=8 and an exact rerank returns the
exact bf16 argmax on every row, while a 4-bit head at KCAND=1 misses some rows (a winner that
shares a 64-row block with a stronger coarse value is never a candidate). Its rows are captured
draft-head inputs, which are not available; these synthetic rows stand in for them.

Workload: the head the bench times (synth workload head_m1_k5120_n124160: K=5120, N=124160,
seed 1, lognormal row norms, planted rows and near-tie pairs facing its hidden row 0) and 64
hidden rows: that row 0, then 63 RMS-normalised rows of seed 7 (synth.hidden_rows).

For each configuration (int2 G=128 KCAND=8, int4 G=128 KCAND=1, int2 G=64 KCAND=8; RERANK=16,
the three the bench times; then the two levers the page names, KCAND and RERANK, moved one at a
time on the int2 and int4 heads) the oracle's method (quantise, coarse, block top-KCAND, global
top-R, exact rerank, argmax) is compared with the brute-force exact argmax over all N rows. A row
is a miss when the two differ.
Stored per row: the exact argmax and the gap between the two largest exact logits; per
configuration: the method's argmax, the gap between its two largest reranked logits (a row whose
gap is within 1e-4 of the top is a tie, and the GPU may pick either), and every miss with its
exact-logit gap (exact logit of the true argmax minus that of the method's choice).

Run: python tests/golden/make_recall.py   (a few minutes of host time; calls only oracle/)
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from bit_draft_lm_gb300 import synth  # noqa: E402

OUT = os.path.join(HERE, "recall_k5120_n124160_m64.json")
HEAD, ROWS, ROW_SEED = synth.RECALL_HEAD, synth.RECALL_ROWS, synth.RECALL_SEED
CONFIGS = [  # name, bits, G, KCAND, RERANK
    ("int2_g128_kcand8", 2, 128, 8, 16),
    ("int4_g128_kcand1", 4, 128, 1, 16),
    ("int2_g64_kcand8", 2, 64, 8, 16),
    # the levers
    ("int2_g128_kcand1", 2, 128, 1, 16),
    ("int2_g128_kcand8_r64", 2, 128, 8, 64),
    ("int2_g128_kcand16_r64", 2, 128, 16, 64),
    ("int2_g128_kcand8_r256", 2, 128, 8, 256),
    ("int4_g128_kcand8", 4, 128, 8, 16),
]


def workload():
    w = synth.named(HEAD)
    return w, synth.recall_rows(w)


def top2_gap(v):
    s = np.sort(v[np.isfinite(v)])[::-1]
    return float(s[0] - s[1]) if s.size > 1 else float("inf")


def main():
    t0 = time.time()
    w, x = workload()
    exact = oracle.exact_logits(x, w.W)
    ex_am = np.argmax(exact, axis=1)  # first occurrence: the lowest id on equal logits
    out = {
        "about": "recall of the method vs the brute-force exact argmax, oracle only "
                 "(tests/golden/make_recall.py)",
        "head": HEAD, "K": w.K, "N": w.N, "rows": ROWS, "row_seed": ROW_SEED,
        "row0": "the head's own hidden row 0",
        "exact_argmax": ex_am.tolist(),
        "exact_top2_gap": [top2_gap(exact[m]) for m in range(ROWS)],
        "exact_top": [float(exact[m, ex_am[m]]) for m in range(ROWS)],
        "configs": {},
    }
    coarse = {}
    for name, bits, G, kcand, R in CONFIGS:
        if (bits, G) not in coarse:
            packed, S, ZS = oracle.quantize_pack(w.W, G, bits)
            coarse[(bits, G)] = oracle.coarse(x, packed, S, ZS, G, bits)
        c = coarse[(bits, G)]
        # the method's steps after the coarse pass, as oracle.head takes them
        cv, ci = oracle.block_topk(c, kcand)
        rr, _ = oracle.global_topr(cv, ci, R)
        e = oracle.rerank(x, w.W, rr)
        am = oracle.argmax(e, rr)
        misses = []
        for m in range(ROWS):
            if am[m] != ex_am[m]:
                misses.append({"row": m, "exact_id": int(ex_am[m]), "method_id": int(am[m]),
                               "gap": float(exact[m, ex_am[m]] - exact[m, am[m]]),
                               "exact_in_rerank": bool(ex_am[m] in rr[m])})
        out["configs"][name] = {
            "bits": bits, "G": G, "kcand": kcand, "rerank": R,
            "method_argmax": [int(v) for v in am],
            "method_top2_gap": [top2_gap(e[m]) for m in range(ROWS)],
            "misses": misses,
        }
        print(f"{name}: {len(misses)} misses of {ROWS} rows", flush=True)
    with open(OUT, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(f"wrote {OUT} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
