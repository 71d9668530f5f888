"""Pins of the CPU oracle against what the page and the mathematics fix (no GPU).

Each test ties one oracle step to something other than the oracle itself: hand-worked values
(tests/golden), the page's own bit-pattern dequant, closed forms, brute force on tiny inputs,
and the page's stated sizes. Page: "radiance_drafthead.py" (module docstring, the load-time
quantiser, the int2 coarse kernel, the block candidate emission, the exact rerank and the head
application).
"""
import os

import numpy as np
import pytest

import oracle
from bit_draft_lm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases(fname):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key in ("S", "ZS"):
                cur[key] = [int(v, 16) for v in vals]
            elif key == "w":
                cur[key] = [float(v) for v in vals]
            else:
                cur[key] = [int(v) for v in vals]
    return cases


def _bf16(vals):
    """Exact small values -> bf16 bits (they are exactly representable by construction)."""
    a = np.asarray(vals, dtype=np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), a)
    return bits


@pytest.mark.parametrize("fname,bits", [("quantize_int2_small.txt", 2),
                                        ("quantize_int4_small.txt", 4)])
def test_quantizer_hand_worked(fname, bits):
    """Quantiser + packing + premultiplied scales against hand-worked groups (golden files)."""
    for case in _cases(fname):
        K, G = case["K"][0], case["G"][0]
        W = _bf16(case["w"]).reshape(1, K)
        packed, S, ZS = oracle.quantize_pack(W, G=G, bits=bits, nthreads=1)
        assert packed[0].tolist() == case["bytes"], case["name"]
        assert S[0].tolist() == case["S"], case["name"]
        assert ZS[0].tolist() == case["ZS"], case["name"]
        assert oracle.unpack_codes(packed, K, bits)[0].tolist() == case["codes"], case["name"]


def _page_pattern(b, q):
    """The page's hoisted dequant: 0x3F80 | ((b << (5-2q)) & 0x60) for q < 3, else
    0x3F80 | ((b >> 1) & 0x60), read as bf16 (docstring, 'Bit-pattern dequant, hoisted')."""
    b = np.asarray(b, dtype=np.uint16)
    if q < 3:
        bits = ((b << (5 - 2 * q)) & 0x60) | 0x3F80
    else:
        bits = ((b >> 1) & 0x60) | 0x3F80
    return synth.bf16_value(bits.astype(np.uint16))


def test_dequant_pattern_matches_unpack_all_bytes():
    """For every byte and quarter, the page's bit pattern reads as 1 + v/4 with v the code the
    oracle unpacks from that quarter of the byte (quarter-split layout)."""
    K = 4 * 256                      # Q = 256: byte j of the row is j, so every byte value occurs
    packed = np.arange(256, dtype=np.uint8).reshape(1, 256)
    codes = oracle.unpack_codes(packed, K, 2)[0]
    for q in range(4):
        v = codes[q * 256:(q + 1) * 256].astype(np.float64)
        d = _page_pattern(np.arange(256), q)
        assert np.array_equal(d, 1.0 + v / 4.0), q
        # the page's equivalence: (b << (5-2q)) & 0x60 == ((b >> 2q) & 3) << 5
        b = np.arange(256, dtype=np.uint16)
        alt = synth.bf16_value(((((b >> (2 * q)) & 3) << 5) | 0x3F80).astype(np.uint16))
        assert np.array_equal(d, alt)


def test_int4_pattern_matches_unpack_all_bytes():
    """4-bit: 0x3F80 | (nibble << 3) reads as 1 + v/16 (the '16 for the 4-bit path (v << 3)'
    premultiplier), half-split layout: low nibble is k = j, high nibble k = K/2 + j."""
    K = 2 * 256
    packed = np.arange(256, dtype=np.uint8).reshape(1, 256)
    codes = oracle.unpack_codes(packed, K, 4)[0]
    b = np.arange(256, dtype=np.uint16)
    for h in range(2):
        nib = (b >> (4 * h)) & 15
        d = synth.bf16_value(((nib << 3) | 0x3F80).astype(np.uint16))
        assert np.array_equal(d, 1.0 + codes[h * 256:(h + 1) * 256] / 16.0)


def test_pack_roundtrip_random_codes():
    """Codes chosen at random, realised as exactly-quantisable weights, come back unchanged."""
    rng = np.random.default_rng(11)
    for bits, K, G in ((2, 1024, 128), (2, 512, 64), (4, 512, 128)):
        lv = (1 << bits) - 1
        N = 8
        codes = rng.integers(0, lv + 1, size=(N, K))
        codes[:, ::G] = 0          # every group holds the lowest and highest code
        codes[:, 1::G] = lv
        zp = rng.integers(0, lv + 1, size=(N, K // G))
        sc = 2.0 ** rng.integers(-8, -4, size=(N, K // G))
        w = (codes - np.repeat(zp, G, axis=1)) * np.repeat(sc, G, axis=1)
        packed, S, ZS = oracle.quantize_pack(synth.bf16_bits(w), G=G, bits=bits, nthreads=2)
        assert np.array_equal(oracle.unpack_codes(packed, K, bits), codes)
    packed, _, _ = oracle.quantize_pack(np.zeros((2, 512), dtype=np.uint16), G=128, bits=2)
    assert np.all(packed == 0)


def _exact_grid_weight(rng, N, K, G, bits):
    """Weights that the quantiser represents exactly: group values (q - zp) * sc with sc a power
    of two and codes 0 and lv present, so sc, zp, S and ZS are all exact."""
    lv = (1 << bits) - 1
    codes = rng.integers(0, lv + 1, size=(N, K))
    codes[:, ::G] = 0
    codes[:, 1::G] = lv
    zp = rng.integers(0, lv + 1, size=(N, K // G))
    sc = 2.0 ** rng.integers(-9, -5, size=(N, K // G))
    return synth.bf16_bits((codes - np.repeat(zp, G, axis=1)) * np.repeat(sc, G, axis=1))


@pytest.mark.parametrize("bits,G", [(2, 128), (2, 64), (4, 128)])
def test_coarse_equals_brute_force_on_exact_grid(bits, G):
    """When every weight is exactly representable, the coarse value must equal the brute-force
    exact logit x . W (the fold adds no approximation of its own)."""
    rng = np.random.default_rng(5 + bits + G)
    N, K, M = 96, 1024, 3
    W = _exact_grid_weight(rng, N, K, G, bits)
    x = synth.bf16_bits(rng.standard_normal((M, K)))
    packed, S, ZS = oracle.quantize_pack(W, G=G, bits=bits)
    c = oracle.coarse(x, packed, S, ZS, G=G, bits=bits)
    e = oracle.exact_logits(x, W)
    np.testing.assert_allclose(c, e, rtol=0, atol=1e-12 * np.abs(e).max())


def test_fold_identity_dequant_form():
    """sum_k x (1 + v/4) folded with S and ZS equals the dot with dequantised weights
    (S/4) v - (ZS - S): the accumulator identity of the docstring."""
    w = synth.named("tiny_m1_k1024_n8192")
    rng = np.random.default_rng(3)
    x = synth.bf16_bits(rng.standard_normal((4, w.K)))
    packed, S, ZS = oracle.quantize_pack(w.W[:512], 128, 2)
    c1 = oracle.coarse(x, packed, S, ZS)
    c2 = oracle.coarse_dequant(x, packed, S, ZS)
    np.testing.assert_allclose(c1, c2, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("bits", [2, 4])
def test_one_hot_closed_form(bits):
    """x = e_k: c[n] = S[n, g(k)] (1 + v_k/beta) - ZS[n, g(k)], with v_k decoded from the packed
    byte by the page's bit pattern (not by the oracle's unpacking)."""
    w = synth.named("tiny_m1_k1024_n8192")
    N, K, G = 256, w.K, 128
    packed, S, ZS = oracle.quantize_pack(w.W[:N], G, bits)
    Sv, ZSv = synth.bf16_value(S), synth.bf16_value(ZS)
    for k in (0, 1, 255, 256, 511, 700, 1023):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80                       # 1.0
        c = oracle.coarse(x, packed, S, ZS, G, bits)[0]
        if bits == 2:
            Q = K // 4
            d = _page_pattern(packed[:, k % Q], k // Q)
        else:
            H = K // 2
            nib = (packed[:, k % H].astype(np.uint16) >> (4 * (k // H))) & 15
            d = synth.bf16_value(((nib << 3) | 0x3F80).astype(np.uint16))
        g = k // G
        np.testing.assert_array_equal(c, Sv[:, g] * d - ZSv[:, g])


def test_quantizer_error_bound_and_ranges():
    """Codes lie in [0, 3] and reconstruction error is within about one step when the group
    straddles zero: |w - (S/4)(q - zp)| <= 1.01 sc (sc from S, zp from ZS - S)."""
    w = synth.named("tiny_m1_k1024_n8192")
    W = w.W[:300]
    packed, S, ZS = oracle.quantize_pack(W, 128, 2)
    codes = oracle.unpack_codes(packed, w.K, 2).astype(np.float64)
    assert codes.min() >= 0 and codes.max() <= 3
    sc = synth.bf16_value(S) / 4.0
    zp = np.rint((synth.bf16_value(ZS) - synth.bf16_value(S)) / sc)
    wv = synth.bf16_value(W)
    rec = np.repeat(sc, 128, axis=1) * (codes - np.repeat(zp, 128, axis=1))
    err = np.abs(wv - rec)
    assert np.all(err <= 1.01 * np.repeat(sc, 128, axis=1) + 1e-12)


def test_constant_group_follows_formula():
    """hi == lo: sc clamps to 1e-8 and every code is 0 for a zero group (literal formula)."""
    W = np.zeros((1, 512), dtype=np.uint16)
    packed, S, ZS = oracle.quantize_pack(W, 128, 2)
    assert np.all(packed == 0)
    four_e8 = np.float32(4.0) * np.float32(1e-8)
    expect = synth.bf16_bits(np.float64(four_e8))
    assert np.all(S == expect) and np.all(ZS == expect)


def test_stored_sizes_match_page():
    """Stored bytes per vocab row x 124160 rows: 0.167 GiB/rank of int2 head, 152 MiB of packed
    int2, against 1.18 GiB for the bf16 head (docstring; 'on its 152 MiB of int2')."""
    W = np.zeros((4, 5120), dtype=np.uint16)
    packed, S, ZS = oracle.quantize_pack(W, 128, 2)
    per_row = packed[0].nbytes + S[0].nbytes + ZS[0].nbytes
    N = 124160
    assert per_row * N == 178_790_400
    assert round(per_row * N / 2 ** 30, 3) == 0.167
    assert round(packed[0].nbytes * N / 2 ** 20) == 152
    assert round(5120 * 2 * N / 2 ** 30, 2) == 1.18


def _brute_block_topk(c, kcand):
    M, N = c.shape
    nblk = (N + 63) // 64
    val = np.full((M, nblk * kcand), -np.inf)
    ids = np.full((M, nblk * kcand), -1, dtype=np.int64)
    for m in range(M):
        for b in range(nblk):
            cols = list(range(64 * b, min(64 * b + 64, N)))
            order = sorted(cols, key=lambda n: (-c[m, n], n))[:kcand]
            for s, n in enumerate(order):
                val[m, b * kcand + s] = c[m, n]
                ids[m, b * kcand + s] = n
    return val, ids


@pytest.mark.parametrize("N,kcand", [(640, 8), (700, 8), (130, 1), (64, 64), (200, 3),
                                     (70, 8), (130, 4)])  # last block shorter than KCAND
def test_block_topk_brute_force(N, kcand):
    """Block top-KCAND by successive max-and-mask (the block candidate emission) == sorting each 64-row block by
    (value desc, id asc); short last block padded with (-inf, -1); ties present."""
    rng = np.random.default_rng(N + kcand)
    c = np.round(rng.standard_normal((3, N)) * 4) / 4     # many exact ties
    v, i = oracle.block_topk(c, kcand)
    bv, bi = _brute_block_topk(c, kcand)
    assert np.array_equal(i, bi)
    assert np.array_equal(v, bv)


def test_global_topr_brute_force():
    rng = np.random.default_rng(9)
    M, ncand, R = 4, 1000, 16
    val = np.round(rng.standard_normal((M, ncand)) * 3) / 3
    ids = np.stack([rng.permutation(5000)[:ncand] for _ in range(M)]).astype(np.int32)
    rr, rv = oracle.global_topr(val, ids, R)
    for m in range(M):
        order = sorted(range(ncand), key=lambda j: (-val[m, j], ids[m, j]))[:R]
        assert rr[m].tolist() == [int(ids[m, j]) for j in order]
        assert rv[m].tolist() == [float(val[m, j]) for j in order]


def test_rerank_one_hot_and_full_row_identity():
    """One-hot x gives e = W[n, k] exactly; a reranked value equals the full-row exact logit of
    the same row (candidate-only scoring is the dense score at that position)."""
    w = synth.named("tiny_m1_k1024_n8192")
    ids = np.array([[5, 77, 8191, 0]], dtype=np.int32)
    x = np.zeros((1, w.K), dtype=np.uint16)
    x[0, 300] = 0x3F80
    e = oracle.rerank(x, w.W, ids)
    np.testing.assert_array_equal(e[0], synth.bf16_value(w.W[ids[0], 300]))
    e2 = oracle.rerank(w.x, w.W, ids)
    full = oracle.exact_logits(w.x, w.W)
    np.testing.assert_array_equal(e2[0], full[0, ids[0]])


def test_argmax_ties_to_lowest_id():
    e = np.array([[1.0, 3.0, 3.0, 2.0], [0.5, 0.5, 0.5, 0.5]])
    ids = np.array([[10, 40, 30, 20], [9, 7, 8, 6]], dtype=np.int32)
    assert oracle.argmax(e, ids).tolist() == [30, 6]
    e = np.array([[-np.inf, 1.0]])
    assert oracle.argmax(e, np.array([[-1, 4]], dtype=np.int32)).tolist() == [4]


def test_kcand_recall_claim_small_workload():
    """The page's claim (KCAND=8 + rerank recovers the exact bf16 argmax): on the small planted
    workload the method's argmax equals the brute-force argmax of the exact logits, and the
    near-tie pair at the top is resolved to the right member."""
    w = synth.named("tiny_m1_k1024_n8192")
    packed, S, ZS = oracle.quantize_pack(w.W, 128, 2)
    r = oracle.head(w.x, packed, S, ZS, w.W, kcand=8, R=16)
    ex = oracle.exact_logits(w.x, w.W)
    assert r["argmax"][0] == int(np.argmax(ex[0]))
    # the winner is a member of a near-tie pair whose partner is also in the reranked set
    pair = [p for p in w.pairs if r["argmax"][0] in p]
    assert pair and all(int(n) in r["rr_id"][0] for n in pair[0])


def test_unreranked_coarse_is_not_exact():
    """Without the rerank the coarse argmax is off on this workload (why the rerank exists)."""
    w = synth.named("tiny_m1_k1024_n8192")
    packed, S, ZS = oracle.quantize_pack(w.W, 128, 2)
    c = oracle.coarse(w.x, packed, S, ZS)
    ex = oracle.exact_logits(w.x, w.W)
    assert int(np.argmax(c[0])) != int(np.argmax(ex[0]))


def test_topk_only_oracle():
    """topk_only (the page's y.fill_(-inf) + scatter of bf16 exact logits): bf16 rounding is
    round-to-nearest-even (checked against torch's own conversion, an independent
    implementation, and on hand-picked ties); every entry but the R reranked ones is -inf."""
    import torch
    v = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 3.0e-3, -7.123e4],
                 dtype=np.float32)
    got = oracle.bf16_rne(v)
    assert got[0] == 0x3F80 and got[1] == 0x3F80 and got[2] == 0x3F82 and got[3] == 0xC020
    rng = np.random.default_rng(7)
    r = (rng.standard_normal(4096) * 10.0 ** rng.integers(-6, 6, 4096)).astype(np.float32)
    ref = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(r), ref)
    M, R, N = 3, 16, 1000
    ids = np.stack([rng.choice(N, R, replace=False) for _ in range(M)]).astype(np.int32)
    lg = rng.standard_normal((M, R)).astype(np.float32)
    y = oracle.topk_only(ids, lg, N)
    assert y.shape == (M, N)
    for m in range(M):
        fin = np.flatnonzero(y[m] != 0xFF80)
        assert np.array_equal(np.sort(fin), np.sort(ids[m]))
        assert np.array_equal(y[m, ids[m]], oracle.bf16_rne(lg[m]))


def test_e4m3_decode_matches_torch():
    """The page's e4m3 bit decode (oracle) equals torch's float8_e4m3fn conversion (an
    independent implementation) on every byte that is not a NaN."""
    import torch
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = oracle.e4m3_decode(b)
    ok = ~np.isnan(ref)
    assert ok.sum() == 254
    assert np.array_equal(dec[ok], ref[ok])


def test_fp8_quantiser_and_rerank_pins():
    """FP8 head: with a row scale of 1, quantising the scaled e4m3 values (fp32 rows) gives the
    same bytes as quantising the same values stored as bf16 (every e4m3 value is a bf16 value),
    so the fp32 path is pinned to the bf16 quantiser; a power-of-two row scale scales S and ZS
    exactly and leaves the codes; the FP8 rerank of a one-hot x is e4m3(w) * scale exactly."""
    rng = np.random.default_rng(11)
    N, K, G = 6, 512, 128
    W8 = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    W8[(W8 & 0x7F) == 0x7F] = 0x3C  # no NaN bytes
    one = np.ones(N, dtype=np.float32)
    p8, S8, Z8 = oracle.quantize_pack_fp8(W8, one, G)
    Wb = oracle.bf16_rne(oracle.e4m3_decode(W8).astype(np.float32))
    pb, Sb, Zb = oracle.quantize_pack(Wb, G, 2)
    assert np.array_equal(p8, pb) and np.array_equal(S8, Sb) and np.array_equal(Z8, Zb)
    p4, S4, Z4 = oracle.quantize_pack_fp8(W8, one * 0.25, G)
    assert np.array_equal(p4, p8)
    assert np.array_equal(oracle.bf16_bits_to_f64(S4), oracle.bf16_bits_to_f64(S8) * 0.25)
    assert np.array_equal(oracle.bf16_bits_to_f64(Z4), oracle.bf16_bits_to_f64(Z8) * 0.25)
    scale = rng.uniform(0.001, 0.01, N).astype(np.float32)
    k = 77
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, k] = 0x3F80  # 1.0
    ids = np.arange(N, dtype=np.int32)[None, :]
    e = oracle.rerank_fp8(x, W8, scale, ids)
    assert np.array_equal(e[0], oracle.e4m3_decode(W8[:, k]) * scale.astype(np.float64))
