"""Recall of the method on the vocabulary-scale synthetic head, on the GPU.

The page "radiance_drafthead.py" (module docstring: accuracy from reranking, KCAND as the lever)
claims its int2 head with KCAND=8 and an exact rerank matches the exact argmax on every captured
row, against misses for a 4-bit head at KCAND=1. Recall is a property of the method, not of the
kernels: on the rows of tests/golden/recall_k5120_n124160_m64.json (written from the oracle alone
by tests/golden/make_recall.py) the GPU path must miss exactly the rows the oracle's method
misses, and return the oracle method's argmax on every row that is not a tie among its reranked
logits. The misses themselves (which rows, their exact-logit gaps) are the report.
"""
import json
import os

import numpy as np
import pytest
import torch

from bit_draft_lm_gb300 import build as dh_build
from bit_draft_lm_gb300 import drafthead as dh
from bit_draft_lm_gb300 import synth

from _parity import dev_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "recall_k5120_n124160_m64.json")


@pytest.fixture(scope="module")
def setup():
    dh_build.build()
    dh.lib()
    with open(GOLDEN) as f:
        gold = json.load(f)
    w = synth.named(gold["head"])
    x = synth.recall_rows(w)
    return gold, dev_bf16(w.W), dev_bf16(x)


def _gpu_argmax(x, W, bits, G, kcand, R, batch):
    quant = dh.dh_quantize_pack_int2 if bits == 2 else dh.dh_quantize_pack_int4
    packed, S, ZS = quant(W, G)
    out = []
    for m0 in range(0, x.shape[0], batch):
        xb = x[m0:m0 + batch]
        ws = dh.new_workspace(xb.shape[0], W.shape[0], W.shape[1], kcand, R)
        rr, rl, am, _, _ = dh.dh_draft_head_argmax(xb, packed, S, ZS, W, G, bits, kcand, R,
                                                   workspace=ws)
        torch.cuda.synchronize()
        assert dh.dh_workspace_status(ws) == 0
        out.append(am.cpu().numpy())
    return np.concatenate(out)


@pytest.mark.parametrize("name,batch", [
    ("int2_g128_kcand8", 8),    # the warp-MMA kernel, in the bench's 8-row calls
    ("int2_g128_kcand8", 64),   # the tensor-core pass, all rows at once
    ("int4_g128_kcand1", 8),
    ("int2_g64_kcand8", 8),
    ("int2_g128_kcand8_r64", 8),   # RERANK > 32: the one-CTA rerank kernel
    ("int2_g128_kcand8_r256", 8),
])
def test_gpu_misses_equal_oracle_method_misses(setup, name, batch):
    gold, W, x = setup
    cfg = gold["configs"][name]
    am = _gpu_argmax(x, W, cfg["bits"], cfg["G"], cfg["kcand"], cfg["rerank"], batch)
    ex = np.asarray(gold["exact_argmax"])
    method = np.asarray(cfg["method_argmax"])
    top = np.abs(np.asarray(gold["exact_top"]))
    tie = np.asarray(cfg["method_top2_gap"]) <= 1e-4 * top
    assert np.array_equal(am[~tie], method[~tie])
    gpu_miss = set(np.nonzero(am != ex)[0].tolist()) - set(np.nonzero(tie)[0].tolist())
    oracle_miss = {d["row"] for d in cfg["misses"]} - set(np.nonzero(tie)[0].tolist())
    assert gpu_miss == oracle_miss
    print(f"{name} (batch {batch}): {len(gpu_miss)} misses of {len(ex)} rows "
          f"{sorted(gpu_miss)}; oracle method {sorted(oracle_miss)}")
