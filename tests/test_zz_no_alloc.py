"""dh_draft_head_rerank_argmax_noalloc, the rerank + argmax entry point for callers that cannot
allocate device memory (a plug-in handed only its input and output buffers, code inside another
framework's memory pool): instead of a caller workspace it uses a fixed scratch array among the
library's device globals. Through the C ABI, its outputs must agree with those of
dh_draft_head_rerank_argmax (which takes a caller workspace) on two calls in a row, the second
with different sizes and candidates so that nothing left in the shared scratch by the first call
can pass for a result.

This file is named to be collected last: if it fails, a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_draft_lm_gb300 import build as dh_build
from bit_draft_lm_gb300 import drafthead as dh
from bit_draft_lm_gb300 import synth

from _parity import bf16_to_f64, dev_bf16, near_tie_rows, RERANK_ABS, RERANK_RTOL


@pytest.fixture(scope="module")
def lib():
    dh_build.build()
    return dh.lib()


def test_noalloc_rejects_out_of_range_sizes_on_host(lib):
    """M = 0 is refused before any CUDA call (the fake addresses are never touched)."""
    A16 = 0x10000
    rc = lib.dh_draft_head_rerank_argmax_noalloc(A16, 0, 1024, A16, 8192, A16, A16, 64, 16,
                                                 A16, A16, A16, None, None)
    assert rc == dh.DH_ERR_SHAPE
    assert "out of range" in dh.dh_last_error()


def _inputs(M, K, N, ncand, seed):
    rng = np.random.default_rng(seed)
    w = synth.make_workload(M, K, N, seed, plant=False)
    val = rng.standard_normal((M, ncand)).astype(np.float32)
    ids = np.stack([rng.choice(N, ncand, replace=False) for _ in range(M)]).astype(np.int32)
    val[:, -2:] = -np.inf  # empty slots, as short blocks leave them
    ids[:, -2:] = -1
    return (w, dev_bf16(w.x), dev_bf16(w.W), torch.from_numpy(val).cuda(),
            torch.from_numpy(ids).cuda())


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point(lib):
    # two calls in a row: the first larger, the second with other sizes and candidates
    for M, K, N, ncand, R, seed in ((8, 5120, 20000, 15520, 16, 60), (3, 1024, 8192, 1000, 32, 61)):
        w, x, W, cv, ci = _inputs(M, K, N, ncand, seed)
        ws = dh.new_workspace(M, N, K, 1, R)
        rr0, rl0, am0 = dh.dh_draft_head_rerank_argmax(x, W, cv, ci, R, workspace=ws)
        rr1, rl1, am1 = dh.dh_draft_head_rerank_argmax_noalloc(x, W, cv, ci, R)
        torch.cuda.synchronize()
        rr0, rr1 = rr0.cpu().numpy(), rr1.cpu().numpy()
        rl0 = rl0.cpu().numpy().astype(np.float64)
        rl1 = rl1.cpu().numpy().astype(np.float64)
        assert np.array_equal(rr1, rr0)
        fin = np.isfinite(rl0)
        assert np.array_equal(np.isfinite(rl1), fin)
        # the rerank tolerance of the parity tests, around the workspace entry point's values
        xf, Wf = bf16_to_f64(w.x), bf16_to_f64(w.W)
        absdot = np.array([[np.abs(xf[m] * Wf[n]).sum() if n >= 0 else 0.0 for n in rr0[m]]
                           for m in range(M)])
        tol = RERANK_RTOL * np.abs(np.where(fin, rl0, 0.0)) + RERANK_ABS * absdot
        assert np.all(np.abs(rl1[fin] - rl0[fin]) <= tol[fin])
        ok = ~near_tie_rows(rl0)
        assert np.array_equal(am1.cpu().numpy()[ok], am0.cpu().numpy()[ok])
