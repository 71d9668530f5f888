"""Vocabulary-sharded argmax merge: the head's vocab rows split across ranks at 64-row block
boundaries, each rank running the path on its rows, one MAX all-reduce of one int64 key per
hidden row merging the ranks' answers.

CPU (no GPU): the partition, the key order and decode through the library's host routines, and
the exchange itself on two gloo ranks fed by the oracle's per-shard results. GPU: two shards of
one head on one device through the library's kernels, merged, against the unsharded call and the
oracle.

The expected merge is the definition: over the union of the shards' reranked slots, the largest
fp32 logit, equal logits going to the lowest vocab id.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from bit_draft_lm_gb300 import build as dh_build
from bit_draft_lm_gb300 import drafthead as dh
from bit_draft_lm_gb300 import synth


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dh_build.build()
    dh.lib()


def _expected(parts):
    """parts: [(rr_id global int array [M, R], logit float32 [M, R])] -> (id [M], logit [M])."""
    ids = np.concatenate([p[0] for p in parts], axis=1)
    lg = np.concatenate([p[1] for p in parts], axis=1).astype(np.float32)
    M = ids.shape[0]
    out_id = np.full(M, -1, dtype=np.int64)
    out_l = np.full(M, -np.inf, dtype=np.float32)
    for m in range(M):
        best = None
        for n, v in zip(ids[m], lg[m]):
            if n < 0:
                continue
            if best is None or v > best[1] or (v == best[1] and n < best[0]):
                best = (int(n), v)
        if best is not None:
            out_id[m], out_l[m] = best
    return out_id, out_l


@pytest.mark.parametrize("N,world", [(124160, 2), (124160, 8), (8232, 3), (70, 2), (64, 4)])
def test_vocab_shard_partition(N, world):
    """Shards cover [0, N) once, in rank order, and start on 64-row block boundaries."""
    edges = [dh.vocab_shard(N, world, r) for r in range(world)]
    assert edges[0][0] == 0 and edges[-1][1] == N
    for (a0, a1), (b0, b1) in zip(edges, edges[1:]):
        assert a1 == b0
    for n0, n1 in edges:
        assert n0 % 64 == 0 and n0 <= n1
    sizes = [(n1 - n0 + 63) // 64 for n0, n1 in edges]
    assert max(sizes) - min(sizes) <= 1 or N < 64 * world


def test_shard_keys_order_and_decode_host():
    """Keys order as (logit, then lower id) under signed int64 comparison; decode returns the
    winner; +0 and -0 tie; -inf is a value; an empty row decodes to (-1, -inf)."""
    rng = np.random.default_rng(150)
    M, R = 64, 8
    logit = rng.standard_normal((M, R)).astype(np.float32)
    logit[0, :] = 0.5                     # a row of equal logits: the lowest id wins
    logit[1, 0], logit[1, 1] = 0.0, -0.0  # +0 and -0 compare equal
    logit[1, 2:] = -1.0
    logit[2, :] = -np.inf                 # all -inf: still the lowest id
    ids = np.stack([rng.choice(100000, R, replace=False) for _ in range(M)]).astype(np.int32)
    ids[3, :] = -1                        # no candidate at all
    ids[4, 3] = -1                        # one empty slot
    off = 777
    keys = dh.dh_argmax_shard_keys(torch.from_numpy(ids), torch.from_numpy(logit), off)
    am, lv = dh.dh_argmax_merge(keys.view(1, -1))
    e_id, e_l = _expected([(np.where(ids >= 0, ids + off, -1), logit)])
    assert np.array_equal(am.numpy(), e_id) and np.array_equal(lv.numpy(), e_l)
    assert am[3] == -1 and np.isneginf(lv[3].item())
    assert am[1] == min(ids[1, 0], ids[1, 1]) + off
    # the order itself: for random pairs, key comparison == (logit, -id) comparison
    a = torch.from_numpy(rng.standard_normal((200, 1)).astype(np.float32))
    a[::7] = a[1::7][: a[::7].shape[0]]  # some equal logits
    n = torch.from_numpy(rng.integers(0, 2 ** 31 - 1, size=(200, 1)).astype(np.int32))
    k = dh.dh_argmax_shard_keys(n, a, 0).numpy()
    for i in range(0, 200, 2):
        want = (a[i, 0] > a[i + 1, 0]) or (a[i, 0] == a[i + 1, 0] and n[i, 0] < n[i + 1, 0])
        if a[i, 0] == a[i + 1, 0] and n[i, 0] == n[i + 1, 0]:
            continue
        assert (k[i] > k[i + 1]) == bool(want)


def test_merge_host_over_gathered_shards():
    """dh_argmax_merge over P gathered key rows equals the definition over the union."""
    rng = np.random.default_rng(151)
    M, R, P = 16, 4, 5
    parts, keys = [], []
    for p in range(P):
        lg = np.round(rng.standard_normal((M, R)) * 4).astype(np.float32) / 4  # many ties
        ids = rng.integers(0, 1000, size=(M, R)).astype(np.int32)
        off = 1000 * p
        parts.append((ids + off, lg))
        keys.append(dh.dh_argmax_shard_keys(torch.from_numpy(ids), torch.from_numpy(lg), off))
    am, lv = dh.dh_argmax_merge(torch.stack(keys))
    e_id, e_l = _expected(parts)
    assert np.array_equal(am.numpy(), e_id) and np.array_equal(lv.numpy(), e_l)


def _shard_results(w, n0, n1, G, bits, kcand, R):
    """The oracle's path on rows [n0, n1) of the head: (rr_id shard-local, rr_logit fp32)."""
    Ws = np.ascontiguousarray(w.W[n0:n1])
    packed, S, ZS = oracle.quantize_pack(Ws, G, bits)
    h = oracle.head(w.x, packed, S, ZS, Ws, G=G, bits=bits, kcand=kcand, R=R)
    return h["rr_id"].astype(np.int32), h["rr_logit"].astype(np.float32)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_rank(rank, world, port, q):
    import torch.distributed as dist
    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                world_size=world)
        w = synth.make_workload(4, 1024, 8232, 152, plant=True)
        n0, n1 = dh.vocab_shard(w.N, world, rank)
        rr, lg = _shard_results(w, n0, n1, 128, 2, 8, 16)
        am, lv = dh.merge_argmax_across_ranks(torch.from_numpy(rr), torch.from_numpy(lg), n0)
        q.put((rank, am.numpy().tolist(), lv.numpy().tolist(), None))
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, None, repr(e)))


def test_gloo_two_rank_exchange():
    """Two gloo ranks, each with its shard's results from the oracle: after the exchange both hold
    the argmax over the union of their reranked slots. That union holds the unsharded method's
    top-R, so its winner's exact logit is at least the unsharded winner's (equal ids wherever the
    unsharded method found the exact argmax), and the planted row's winner is the brute-force
    exact argmax."""
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, am, lv, err in got:
        assert err is None, f"rank {rank}: {err}"
    w = synth.make_workload(4, 1024, 8232, 152, plant=True)
    parts = []
    for r in range(world):
        n0, n1 = dh.vocab_shard(w.N, world, r)
        rr, lg = _shard_results(w, n0, n1, 128, 2, 8, 16)
        parts.append((np.where(rr >= 0, rr + n0, -1), lg))
    e_id, e_l = _expected(parts)
    for rank, am, lv, _ in got:
        assert am == e_id.tolist() and np.array_equal(np.float32(lv), e_l)
    # unsharded: the method's argmax over the whole head, and the exact argmax of row 0
    packed, S, ZS = oracle.quantize_pack(w.W, 128, 2)
    full = oracle.head(w.x, packed, S, ZS, w.W, G=128, bits=2, kcand=8, R=16)
    exact = oracle.exact_logits(w.x, w.W)
    ex_am = np.argmax(exact, axis=1)
    for m in range(w.M):
        assert exact[m, e_id[m]] >= exact[m, full["argmax"][m]]
        if full["argmax"][m] == ex_am[m]:
            assert e_id[m] == ex_am[m]
    assert e_id[0] == ex_am[0]


@pytest.mark.gpu
@pytest.mark.parametrize("M,K,N,world,bits,kcand", [(4, 1024, 8232, 2, 2, 8),
                                                    (3, 5120, 124160, 2, 2, 8),
                                                    (20, 2048, 20000, 3, 2, 8),
                                                    (8, 1024, 9000, 2, 4, 1)])
def test_shard_then_merge_on_one_gpu(M, K, N, world, bits, kcand):
    """The head split into `world` 64-aligned row shards on one GPU: each shard runs
    dh_draft_head_argmax on its slices of packed, S, ZS and W, its keys come from
    dh_argmax_shard_keys, and dh_argmax_merge over the gathered keys must equal the definition
    over the shards' reranked slots, and the unsharded call's argmax wherever that call's winner
    is also the exact winner of the union."""
    G, R = 128, 16
    if (K, N) == (5120, 124160):
        w0 = synth.named("head_m8_k5120_n124160")
        w = synth.Workload(w0.name, M, K, N, w0.seed, np.ascontiguousarray(w0.x[:M]), w0.W,
                           w0.planted, w0.pairs, w0.kstar)
    else:
        w = synth.make_workload(M, K, N, 153 + M, plant=True)
    W = torch.from_numpy(np.ascontiguousarray(w.W).view(np.int16)).cuda().view(torch.bfloat16)
    x = torch.from_numpy(np.ascontiguousarray(w.x).view(np.int16)).cuda().view(torch.bfloat16)
    quant = dh.dh_quantize_pack_int2 if bits == 2 else dh.dh_quantize_pack_int4
    packed, S, ZS = quant(W, G)
    keys, parts = [], []
    for r in range(world):
        n0, n1 = dh.vocab_shard(N, world, r)
        rr, rl, am, _, _ = dh.dh_draft_head_argmax(x, packed[n0:n1], S[n0:n1], ZS[n0:n1],
                                                   W[n0:n1], G, bits, kcand, R)
        keys.append(dh.dh_argmax_shard_keys(rr, rl, n0))
        rrh = rr.cpu().numpy()
        parts.append((np.where(rrh >= 0, rrh + n0, -1), rl.cpu().numpy()))
    g_id, g_l = dh.dh_argmax_merge(torch.stack(keys))
    torch.cuda.synchronize()
    e_id, e_l = _expected(parts)
    assert np.array_equal(g_id.cpu().numpy(), e_id)
    assert np.array_equal(g_l.cpu().numpy(), e_l)
    # against the unsharded call and the oracle's unsharded method
    rr, rl, am, _, _ = dh.dh_draft_head_argmax(x, packed, S, ZS, W, G, bits, kcand, R)
    torch.cuda.synchronize()
    ex = oracle.rerank(w.x, w.W, np.where(e_id[:, None] >= 0, e_id[:, None], -1).astype(np.int32))
    ue = oracle.rerank(w.x, w.W, am.cpu().numpy()[:, None].astype(np.int32))
    for m in range(M):
        # the union holds the unsharded top-R, so its exact winner is at least as good
        assert ex[m, 0] >= ue[m, 0] - 1e-4 * abs(ue[m, 0]) - 1e-6
        if int(am[m]) != int(e_id[m]):
            print(f"row {m}: sharded {int(e_id[m])} ({ex[m, 0]:.6f}) vs unsharded "
                  f"{int(am[m])} ({ue[m, 0]:.6f})")
