"""Test-side comparison helpers for GPU-vs-oracle parity (tolerances of the draft head).

Tolerances (per hidden row m; c = oracle coarse value, e = oracle exact logit):
  coarse:   |c_gpu - c| <= 2e-3 * max(|c|, rms_n c[m, :])
  rerank:   |e_gpu - e| <= 1e-4 * |e| + 1e-6 * sum_k |x_k W_nk|
  argmax:   equal on every row whose two largest exact reranked logits differ by more than
            1e-4 * |top|.
Candidate ids must match exactly except where the oracle's own coarse values of the two ids
are within the coarse tolerance of each other (an fp32 accumulation-order tie).
"""
import numpy as np
import torch

COARSE_RTOL = 2e-3
RERANK_RTOL = 1e-4
RERANK_ABS = 1e-6


def dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def coarse_tol(c: np.ndarray) -> np.ndarray:
    rms = np.sqrt(np.mean(c * c, axis=1, keepdims=True))
    return COARSE_RTOL * np.maximum(np.abs(c), rms)


def check_block_candidates(c, o_val, o_id, g_val, g_id, kcand):
    """Returns the number of slots whose id differs from the oracle's (all of them near-ties)."""
    M, N = c.shape
    tol = coarse_tol(c)
    nblk = (N + 63) // 64
    g_val = np.asarray(g_val, dtype=np.float64)
    mism = 0
    for m in range(M):
        gi = g_id[m].reshape(nblk, kcand)
        oi = o_id[m].reshape(nblk, kcand)
        gv = g_val[m].reshape(nblk, kcand)
        valid = gi >= 0
        assert np.array_equal(valid, oi >= 0), f"row {m}: padding slots differ"
        assert np.all(np.isneginf(gv[~valid]))
        blk = np.arange(nblk)[:, None]
        assert np.all((gi[valid] // 64) == np.broadcast_to(blk, gi.shape)[valid]), "id outside block"
        ids = np.where(valid, gi, 0)
        cg = c[m, ids]
        tg = tol[m, ids]
        assert np.all(np.abs(gv[valid] - cg[valid]) <= tg[valid]), \
            f"row {m}: coarse value off by {np.max(np.abs(gv[valid] - cg[valid]) / tg[valid]):.3g} tol"
        for b in range(nblk):
            row = gi[b][valid[b]]
            assert len(set(row.tolist())) == len(row), "duplicate id in a block"
        diff = (gi != oi) & valid
        if diff.any():
            co = c[m, np.where(valid, oi, 0)]
            to = tol[m, np.where(valid, oi, 0)]
            assert np.all(np.abs(cg[diff] - co[diff]) <= np.maximum(tg[diff], to[diff])), \
                f"row {m}: candidate differs beyond a near-tie"
            mism += int(diff.sum())
    return mism


def ambiguous_slots(c, kcand):
    """How many (row, block, slot) selections the coarse tolerance leaves open: slot s of a block
    (s < kcand, the oracle's values sorted descending) can hold another id only if its value is
    within the tolerance of its neighbour above or below. An upper bound on the near-tie swaps,
    whatever the data (a row whose values are all near-ties at its own scale has many)."""
    M, N = c.shape
    tol = coarse_tol(c)
    n = 0
    for m in range(M):
        for b0 in range(0, N, 64):
            v = c[m, b0:b0 + 64]
            t = tol[m, b0:b0 + 64]
            o = np.argsort(-v, kind="stable")
            vs, ts = v[o], t[o]
            gap = vs[:-1] - vs[1:]
            close = gap <= np.maximum(ts[:-1], ts[1:])  # pair (s, s + 1) is a near-tie
            k = min(kcand, v.size)
            for s in range(k):
                if (s > 0 and close[s - 1]) or (s < close.size and close[s]):
                    n += 1
    return n


def rerank_tol(x_u16, W_u16, ids, e):
    x = bf16_to_f64(x_u16)
    tol = np.empty_like(e)
    for m in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            n = ids[m, j]
            s = np.abs(x[m] * bf16_to_f64(W_u16[n])).sum() if n >= 0 else 0.0
            tol[m, j] = RERANK_RTOL * abs(e[m, j]) + RERANK_ABS * s if np.isfinite(e[m, j]) else 0
    return tol


def near_tie_rows(e):
    """Rows whose two largest exact reranked logits are within 1e-4 * |top|."""
    s = np.sort(np.where(np.isfinite(e), e, -np.inf), axis=1)[:, ::-1]
    if s.shape[1] < 2:
        return np.zeros(s.shape[0], dtype=bool)
    return (s[:, 0] - s[:, 1]) <= RERANK_RTOL * np.abs(s[:, 0])
