"""Pins of the float64 oracle to things other than itself (CPU only).

Each test names what fixes the expected value: a number printed on the pages
(fixtures under tests/golden/, each with its citation), exact arithmetic in
high-precision decimal, a closed form, an independent library routine
(numpy's fp16, torch's bf16, scipy's softmax / logsumexp), or an invariant
that the derivations prove (any split with any merge equals the unsplit
result).
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f32(a):
    return np.asarray(a, dtype=np.float32)


# ---------------------------------------------------------------- decoders

def test_f16_decoder_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode_elements(bits.view(np.float16), "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode_elements(bits.view(np.int16), "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------- worked example: x=[1,2,.5]

def test_online_softmax_worked_example():
    g = _golden("online_softmax_example.json")
    tol = 0.5 * 10 ** -g["decimals"] + 1e-9
    m, dn, ms, ds = oracle.online_softmax(g["x"])
    assert np.allclose(ms, g["m_steps"], atol=tol, rtol=0)
    assert np.allclose(ds, g["d_steps"], atol=tol, rtol=0)
    assert m == 2.0
    assert abs(dn - g["d_steps"][-1]) <= tol
    # softmax via the recurrence's final state, as the page does
    sm = [math.exp(x - m) / dn for x in g["x"]]
    assert np.allclose(sm, g["softmax"], atol=tol, rtol=0)


def test_attention_reproduces_worked_softmax():
    """q=[1,0,0], K_j=[x_j,0,0], V=I, scale 1 => out = softmax(x), lse = ln sum e^x."""
    g = _golden("online_softmax_example.json")
    tol = 0.5 * 10 ** -g["decimals"] + 1e-9
    x = g["x"]
    q = _f32([[[1, 0, 0]]])
    K = _f32([[[[xi, 0, 0] for xi in x]]])
    V = _f32(np.eye(3))[None, None]
    out, lse = oracle.attention(q, K, V, scale=1.0)
    assert np.allclose(out[0, 0], g["softmax"], atol=tol, rtol=0)
    # sum_exp printed to 3 decimals: ln is pinned to within that rounding
    assert abs(math.exp(lse[0, 0]) - g["sum_exp"]) <= 0.5e-3 + 1e-9
    # every split count and both merges reproduce it
    for P in (1, 2, 3, 4):
        o, m, l, s = oracle.split_partials(q, K, V, P, scale=1.0)
        for got in (oracle.combine_mlo(o, m, l), oracle.combine_lse(o, s),
                    oracle.merge_lse_sequential(o, s), oracle.merge_mlo_tree(o, m, l)):
            assert np.allclose(got[0], out, atol=1e-15, rtol=0)
            assert np.allclose(got[1], lse, atol=1e-15, rtol=0)


# ------------------------------------------- worked example: 3-token tile

def _tile_case():
    g = _golden("tile_incremental_example.json")
    q = _f32(g["q"])[None, None]
    K = _f32(g["K"])[None, None]
    V = _f32(g["V"])[None, None]
    return g, q, K, V


def test_tile_example_scores_and_direct_form():
    g, q, K, V = _tile_case()
    # P=3 puts one token in each split: m of a one-token split is its score
    o, m, l, s = oracle.split_partials(q, K, V, 3, scale=g["scale"])
    assert np.allclose(m[0, 0], g["scores"], atol=0.5e-4, rtol=0)
    assert np.allclose(l[0, 0], 1.0, atol=0, rtol=0)
    # P=1: the whole tile in the direct form of §2.4.1
    o1, m1, l1, _ = oracle.split_partials(q, K, V, 1, scale=g["scale"])
    assert abs(m1[0, 0, 0] - g["m_steps"][-1]) <= 0.5e-4
    assert abs(l1[0, 0, 0] - g["l_steps"][-1]) <= 0.5e-4
    assert np.allclose(o1[0, 0, 0], g["o_steps"][-1], atol=0.5e-3 + 1e-9, rtol=0)
    # the three exp terms the page sums for l
    terms = np.exp(m[0, 0] - m1[0, 0, 0])
    assert np.allclose(terms, g["direct_terms"], atol=0.5e-3 + 1e-9, rtol=0)


def test_tile_example_incremental_step_table():
    g, q, K, V = _tile_case()
    # exact scores (float32 inputs widened), then the per-token recurrence
    qd = q[0, 0].astype(np.float64)
    s = np.array([g["scale"] * float(np.dot(qd, k.astype(np.float64))) for k in K[0, 0]])
    m, l, o, ms, ls, os_ = oracle.tile_incremental(s, V[0, 0].astype(np.float64))
    assert np.allclose(ms, g["m_steps"], atol=0.5e-4, rtol=0)
    assert np.allclose(ls, g["l_steps"], atol=0.5e-4, rtol=0)
    assert np.allclose(os_, g["o_steps"], atol=0.5e-3 + 1e-9, rtol=0)
    # incremental == direct (the page states they differ by < 1e-15)
    o1, m1, l1, _ = oracle.split_partials(q, K, V, 1, scale=g["scale"])
    assert abs(m - m1[0, 0, 0]) == 0.0
    assert abs(l - l1[0, 0, 0]) < 1e-15
    assert np.allclose(o, o1[0, 0, 0], atol=1e-15, rtol=0)
    # the 2-token prefix row is itself a partial: split {1,2} + {3} merged
    o2, m2, l2, s2 = oracle.split_partials(q, K, V, 2, scale=g["scale"])
    assert abs(l2[0, 0, 0] - g["l_steps"][1]) <= 0.5e-4
    assert np.allclose(o2[0, 0, 0], g["o_steps"][1], atol=0.5e-3 + 1e-9, rtol=0)
    out, lse = oracle.attention(q, K, V, scale=g["scale"])
    mo, ml = oracle.combine_mlo(o2, m2, l2)
    assert np.allclose(mo, out, atol=1e-15, rtol=0)
    assert abs(ml[0, 0] - lse[0, 0]) < 1e-15
    assert np.allclose(out[0, 0], g["o_steps"][-1], atol=0.5e-3 + 1e-9, rtol=0)


def test_rescale_example():
    """Tile 1 = {5, 3}, tile 2 = {8}: the s=3 token's weight, locally and globally."""
    g = _golden("rescale_example.json")
    q = _f32([[[1, 0, 0]]])
    K = _f32([[[[g["m1"], 0, 0], [g["s"], 0, 0], [g["m2"], 0, 0]]]])
    V = _f32(np.eye(3))[None, None]
    o, m, l, s = oracle.split_partials(q, K, V, 2, scale=1.0)
    assert m[0, 0, 0] == g["m1"] and m[0, 0, 1] == g["m2"]
    # o is normalised: o * l recovers the local weights exp(s_j - m1)
    local = o[0, 0, 0, 1] * l[0, 0, 0]
    assert abs(local - g["local"]) <= 0.5e-3
    out, lse = oracle.attention(q, K, V, scale=1.0)
    mg = max(g["m1"], g["m2"])
    glob = out[0, 0, 1] * math.exp(lse[0, 0] - mg)  # weight * l_global
    assert abs(glob - g["global"]) <= 0.5e-5
    assert abs(math.exp(g["m1"] - mg) - g["shift"]) <= 0.5e-4


# ---------------------------------------- exact brute force (Decimal, no shift)

def _decimal_attention(q, K, V, scale):
    """Textbook softmax attention, no max shift, in 50-digit decimal arithmetic."""
    getcontext().prec = 50
    sc = Decimal(float(scale))
    s = [sc * sum(Decimal(float(a)) * Decimal(float(b)) for a, b in zip(q, k)) for k in K]
    e = [x.exp() for x in s]
    tot = sum(e)
    out = [float(sum(ej * Decimal(float(vj[i])) for ej, vj in zip(e, V)) / tot)
           for i in range(len(V[0]))]
    return out, float(tot.ln())


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_bruteforce_decimal(dtype):
    rng = np.random.default_rng(1234)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    for trial in range(12):
        n = int(rng.integers(1, 9))
        d = int(rng.integers(1, 7))
        q = torch.from_numpy(rng.normal(size=(1, 1, d)) * 2).to(tdt)
        K = torch.from_numpy(rng.normal(size=(1, 1, n, d)) * 2).to(tdt)
        V = torch.from_numpy(rng.normal(size=(1, 1, n, d))).to(tdt)
        scale = 1.0 / math.sqrt(d)
        out, lse = oracle.attention(q, K, V, scale=scale)
        qd = q.double().numpy()[0, 0]
        Kd = K.double().numpy()[0, 0]
        Vd = V.double().numpy()[0, 0]
        ref_o, ref_l = _decimal_attention(qd, Kd, Vd, scale)
        assert np.allclose(out[0, 0], ref_o, atol=1e-14, rtol=1e-13), (trial, n, d)
        assert abs(lse[0, 0] - ref_l) <= 1e-13 * max(1.0, abs(ref_l)), (trial, n, d)


# ------------------------------------------------------------ closed forms

def test_special_cases():
    rng = np.random.default_rng(7)
    d, n = 8, 13
    V = _f32(rng.normal(size=(1, 1, n, d)))
    K = _f32(rng.normal(size=(1, 1, n, d)))
    # q = 0: uniform weights => mean of V rows, lse = ln n
    out, lse = oracle.attention(_f32(np.zeros((1, 1, d))), K, V)
    assert np.allclose(out[0, 0], V[0, 0].astype(np.float64).mean(axis=0), atol=1e-15)
    assert abs(lse[0, 0] - math.log(n)) < 1e-15
    # one token: out = V_0 exactly, lse = s_0
    q = _f32(rng.normal(size=(1, 1, d)))
    out, lse = oracle.attention(q, K, V, lens=[1])
    assert np.array_equal(out[0, 0], V[0, 0, 0].astype(np.float64))
    s0 = float(np.dot(q[0, 0].astype(np.float64), K[0, 0, 0].astype(np.float64))) / math.sqrt(d)
    assert abs(lse[0, 0] - s0) < 1e-15
    # constant V rows: out = that row whatever the scores
    Vc = np.broadcast_to(V[:, :, :1, :], V.shape).copy()
    out, _ = oracle.attention(q, K * 30, Vc)
    assert np.allclose(out[0, 0], Vc[0, 0, 0].astype(np.float64), atol=1e-15, rtol=1e-15)
    # one dominating score: out = that V row (others underflow), lse = that score
    Kd = np.zeros((1, 1, n, d), np.float32)
    Kd[0, 0, 5, 0] = 1.0e4
    qd = np.zeros((1, 1, d), np.float32)
    qd[0, 0, 0] = 1.0
    out, lse = oracle.attention(qd, Kd, V, scale=1.0)
    assert np.array_equal(out[0, 0], V[0, 0, 5].astype(np.float64))
    assert lse[0, 0] == 1.0e4
    # empty sequence: out = 0, lse = -inf; its splits are all empty
    out, lse = oracle.attention(q, K, V, lens=[0])
    assert np.array_equal(out[0, 0], np.zeros(d)) and lse[0, 0] == -math.inf
    o, m, l, s = oracle.split_partials(q, K, V, 3, lens=[0])
    assert np.all(l == 0) and np.all(m == -math.inf) and np.all(s == -math.inf)
    for got in (oracle.combine_mlo(o, m, l), oracle.combine_lse(o, s),
                oracle.merge_lse_sequential(o, s), oracle.merge_mlo_tree(o, m, l)):
        assert np.array_equal(got[0][0, 0], np.zeros(d)) and got[1][0, 0] == -math.inf


def test_shift_invariance_of_scores():
    """Adding c to every score leaves out unchanged and adds c to lse."""
    rng = np.random.default_rng(11)
    d, n = 4, 9
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 1.0
    K = _f32(rng.integers(-8, 8, size=(1, 1, n, d)))
    V = _f32(rng.normal(size=(1, 1, n, d)))
    out, lse = oracle.attention(q, K, V, scale=1.0)
    K2 = K.copy()
    K2[..., 0] += 64.0  # exact in fp32: every score moves by exactly 64
    out2, lse2 = oracle.attention(q, K2, V, scale=1.0)
    assert np.allclose(out2, out, atol=1e-15, rtol=1e-14)
    assert abs(lse2[0, 0] - (lse[0, 0] + 64.0)) < 1e-12


def test_matches_scipy_softmax_and_logsumexp():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    B, H, N, d = 2, 3, 200, 16
    q = _f32(rng.normal(size=(B, H, d)))
    K = _f32(rng.normal(size=(B, H, N, d)) * 3)
    V = _f32(rng.normal(size=(B, H, N, d)))
    lens = [200, 77]
    out, lse = oracle.attention(q, K, V, lens=lens)
    for b in range(B):
        n = lens[b]
        for h in range(H):
            s = (K[b, h, :n].astype(np.float64) @ q[b, h].astype(np.float64)) / math.sqrt(d)
            ref = sp.softmax(s) @ V[b, h, :n].astype(np.float64)
            assert np.allclose(out[b, h], ref, atol=1e-13, rtol=0)
            assert abs(lse[b, h] - sp.logsumexp(s)) < 1e-12


# ----------------------------------------------------- partition & invariants

def test_partition_rule():
    """chunk = ceil(n/P); split p = [p*chunk, min((p+1)*chunk, n)), empty past n."""
    n, d = 10, 2
    q = _f32([[[1.0, 0.0]]])
    K = _f32([[[[j, 0.0] for j in range(n)]]])  # score of token j is exactly j
    V = _f32(np.ones((1, 1, n, d)))
    for P, bounds in [(4, [(0, 3), (3, 6), (6, 9), (9, 10)]),
                      (3, [(0, 4), (4, 8), (8, 10)]),
                      (11, [(j, j + 1) for j in range(10)] + [(10, 10)]),
                      (1, [(0, 10)])]:
        o, m, l, s = oracle.split_partials(q, K, V, P, scale=1.0)
        for p, (lo, hi) in enumerate(bounds):
            if lo >= hi:
                assert m[0, 0, p] == -math.inf and l[0, 0, p] == 0.0
                continue
            assert m[0, 0, p] == hi - 1
            ref_l = sum(math.exp(j - (hi - 1)) for j in range(lo, hi))
            assert abs(l[0, 0, p] - ref_l) < 1e-15
            assert abs(s[0, 0, p] - (m[0, 0, p] + math.log(l[0, 0, p]))) < 1e-15


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_merge_invariants(dtype):
    """Any split count with any merge equals unsplit attention (the equivalence
    theorems of both derivations), including ragged lengths and empty splits."""
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    g = torch.Generator().manual_seed(5)
    B, H, N, d = 3, 2, 37, 8
    q = torch.randn(B, H, d, generator=g).to(tdt)
    K = (torch.randn(B, H, N, d, generator=g) * 4).to(tdt)
    V = torch.randn(B, H, N, d, generator=g).to(tdt)
    lens = [37, 5, 1]
    out, lse = oracle.attention(q, K, V, lens=lens)
    for P in (1, 2, 3, 7, N, N + 5):
        o, m, l, s = oracle.split_partials(q, K, V, P, lens=lens)
        # S = m + ln l wherever the split is non-empty
        ne = l > 0
        assert np.allclose(s[ne], m[ne] + np.log(l[ne]), atol=1e-15, rtol=0)
        for got in (oracle.combine_mlo(o, m, l), oracle.combine_lse(o, s),
                    oracle.merge_lse_sequential(o, s), oracle.merge_mlo_tree(o, m, l)):
            assert np.allclose(got[0], out, atol=1e-12, rtol=0), P
            assert np.allclose(got[1], lse, atol=1e-12, rtol=0), P


def test_merge_order_and_token_permutation():
    """(+) is associative/commutative: reversed partials merge to the same result;
    permuting tokens (K and V rows together) leaves out and lse unchanged."""
    g = torch.Generator().manual_seed(9)
    B, H, N, d = 1, 4, 50, 16
    q = torch.randn(B, H, d, generator=g)
    K = torch.randn(B, H, N, d, generator=g) * 3
    V = torch.randn(B, H, N, d, generator=g)
    out, lse = oracle.attention(q, K, V)
    o, m, l, s = oracle.split_partials(q, K, V, 6)
    rev = (o[:, :, ::-1], m[:, :, ::-1], l[:, :, ::-1], s[:, :, ::-1])
    for got in (oracle.combine_mlo(rev[0], rev[1], rev[2]), oracle.merge_lse_sequential(rev[0], rev[3]),
                oracle.merge_mlo_tree(rev[0], rev[1], rev[2])):
        assert np.allclose(got[0], out, atol=1e-12) and np.allclose(got[1], lse, atol=1e-12)
    perm = torch.randperm(N, generator=g)
    out_p, lse_p = oracle.attention(q, K[:, :, perm], V[:, :, perm])
    assert np.allclose(out_p, out, atol=1e-13) and np.allclose(lse_p, lse, atol=1e-13)


def test_merges_of_synthetic_partials_agree():
    """The four merges agree on arbitrary partial sets (not only on ones that
    came from a split), with wide m ranges and empty entries."""
    rng = np.random.default_rng(21)
    rows, P, d = 40, 9, 5
    o = rng.normal(size=(rows, P, d))
    m = rng.normal(size=(rows, P)) * 30
    l = rng.uniform(1.0, 50.0, size=(rows, P))
    empty = rng.random((rows, P)) < 0.3
    o[empty] = 0.0
    m[empty] = -np.inf
    l[empty] = 0.0
    s = np.where(empty, -np.inf, m + np.log(np.where(empty, 1.0, l)))
    a = oracle.combine_mlo(o, m, l)
    for got in (oracle.combine_lse(o, s), oracle.merge_lse_sequential(o, s),
                oracle.merge_mlo_tree(o, m, l)):
        fin = np.isfinite(a[1])
        assert np.allclose(got[0], a[0], atol=1e-12)
        assert np.allclose(got[1][fin], a[1][fin], atol=1e-12)
        assert np.array_equal(np.isfinite(got[1]), fin)
    # closed form for one row: out = sum_p e^{S_p} o_p / sum_p e^{S_p}
    r = int(np.argmax((~empty).sum(1)))
    w = np.where(empty[r], 0.0, np.exp(s[r] - np.max(s[r])))
    assert np.allclose(a[0][r], (w[:, None] * o[r]).sum(0) / w.sum(), atol=1e-13)


# ------------------------------------------------------------ paged KV cache

def _paged_from_contiguous(K, V, lens, page_size, rng, extra_pages=3):
    """Scatter contiguous [B,H,N,d] K/V into shuffled pages [P,H,ps,d] with a
    block table; unused pages and rows are NaN (never to be read)."""
    B, H, N, d = K.shape
    maxp = -(-N // page_size)
    num_pages = B * maxp + extra_pages
    perm = rng.permutation(num_pages)[: B * maxp].reshape(B, maxp).astype(np.int32)
    Kp = np.full((num_pages, H, page_size, d), np.nan, dtype=K.dtype)
    Vp = np.full((num_pages, H, page_size, d), np.nan, dtype=V.dtype)
    for b in range(B):
        for j in range(maxp):
            lo, hi = j * page_size, min((j + 1) * page_size, int(lens[b]))
            if lo >= hi:
                continue
            Kp[perm[b, j], :, : hi - lo] = K[b, :, lo:hi]
            Vp[perm[b, j], :, : hi - lo] = V[b, :, lo:hi]
    return Kp, Vp, perm


@pytest.mark.parametrize("page_size", [1, 3, 16, 37])
def test_paged_oracle_equals_contiguous_on_gathered_rows(page_size):
    rng = np.random.default_rng(page_size)
    B, H, N, d = 3, 2, 75, 8
    q = _f32(rng.normal(size=(B, H, d)))
    K = _f32(rng.normal(size=(B, H, N, d)) * 3)
    V = _f32(rng.normal(size=(B, H, N, d)))
    lens = np.array([75, 0, 41], np.int32)
    Kp, Vp, table = _paged_from_contiguous(K, V, lens, page_size, rng)
    out, lse = oracle.attention(q, K, V, lens=lens)
    pout, plse = oracle.attention_paged(q, Kp, Vp, table, lens)
    # same rows, same loop order: identical results
    assert np.array_equal(pout, out)
    assert np.array_equal(plse, lse)
    assert np.all(np.isfinite(pout))  # no NaN page or row was read


def test_paged_oracle_single_page_per_sequence_is_contiguous():
    rng = np.random.default_rng(0)
    B, H, N, d = 2, 3, 20, 4
    q = _f32(rng.normal(size=(B, H, d)))
    K = _f32(rng.normal(size=(B, H, N, d)))
    V = _f32(rng.normal(size=(B, H, N, d)))
    # page b holds sequence b whole: the paged layout of one page per sequence
    Kp = np.ascontiguousarray(K)
    Vp = np.ascontiguousarray(V)
    table = np.arange(B, dtype=np.int32).reshape(B, 1)
    lens = np.array([20, 7], np.int32)
    out, lse = oracle.attention(q, K, V, lens=lens)
    pout, plse = oracle.attention_paged(q, Kp, Vp, table, lens)
    assert np.array_equal(pout, out) and np.array_equal(plse, lse)


def test_paged_oracle_rejects_bad_table_entries():
    q = _f32(np.zeros((1, 1, 4)))
    Kp = _f32(np.zeros((2, 1, 4, 4)))
    with pytest.raises(RuntimeError):
        oracle.attention_paged(q, Kp, Kp, np.array([[0, 2]], np.int32), [5])
    with pytest.raises(RuntimeError):
        oracle.attention_paged(q, Kp, Kp, np.array([[-1, 0]], np.int32), [2])
    # an entry past the sequence's last page is never used
    out, _ = oracle.attention_paged(q, Kp, Kp, np.array([[1, 99]], np.int32), [4])
    assert np.all(out == 0)


# ------------------------------------------------------------ FP8 (E4M3) KV cache

def test_e4m3_decoder_exhaustive_vs_torch():
    bits = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_elements(bits, "e4m3")
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _fp8_case(rng, B=2, H=3, N=40, d=16, pow2=True):
    q = _f32(rng.normal(size=(B, H, d)))
    kb = rng.integers(0, 256, size=(B, H, N, d), dtype=np.uint8)
    vb = rng.integers(0, 256, size=(B, H, N, d), dtype=np.uint8)
    # keep the draws finite and moderate: no NaN codes, exponents <= 9
    kb[(kb & 0x7F) >= 0x50] &= 0xC7
    vb[(vb & 0x7F) >= 0x50] &= 0xC7
    if pow2:
        ks = (2.0 ** rng.integers(-6, -2, size=(B, H))).astype(np.float32)
        vs = (2.0 ** rng.integers(-3, 2, size=(B, H))).astype(np.float32)
    else:
        ks = rng.uniform(0.01, 0.2, size=(B, H)).astype(np.float32)
        vs = rng.uniform(0.1, 3.0, size=(B, H)).astype(np.float32)
    return q, kb, vb, ks, vs


def test_fp8_oracle_equals_contiguous_on_exact_dequantised_values():
    rng = np.random.default_rng(2)
    q, kb, vb, ks, vs = _fp8_case(rng)
    lens = np.array([40, 17], np.int32)
    K = (oracle.decode_elements(kb, "e4m3") * ks[:, :, None, None]).astype(np.float32)
    V = (oracle.decode_elements(vb, "e4m3") * vs[:, :, None, None]).astype(np.float32)
    # power-of-two scales: every dequantised value is exact in float32
    assert np.array_equal(K.astype(np.float64), oracle.decode_elements(kb, "e4m3") * ks[:, :, None, None])
    out, lse = oracle.attention(q, K, V, lens=lens)
    fout, flse = oracle.attention_fp8(q, kb, vb, ks, vs, lens=lens)
    assert np.array_equal(fout, out) and np.array_equal(flse, lse)


def test_fp8_oracle_against_numpy_float64():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(4)
    q, kb, vb, ks, vs = _fp8_case(rng, pow2=False)
    lens = np.array([40, 29], np.int32)
    fout, flse = oracle.attention_fp8(q, kb, vb, ks, vs, lens=lens)
    Kd = oracle.decode_elements(kb, "e4m3") * ks[:, :, None, None].astype(np.float64)
    Vd = oracle.decode_elements(vb, "e4m3") * vs[:, :, None, None].astype(np.float64)
    for b in range(2):
        for h in range(3):
            n = lens[b]
            s = Kd[b, h, :n] @ q[b, h].astype(np.float64) / np.sqrt(q.shape[-1])
            assert np.allclose(fout[b, h], sp.softmax(s) @ Vd[b, h, :n], atol=1e-13, rtol=0)
            assert abs(flse[b, h] - sp.logsumexp(s)) < 1e-12
    # out is linear in v_scale: doubling it doubles out exactly
    fout2, flse2 = oracle.attention_fp8(q, kb, vb, ks, vs * 2, lens=lens)
    assert np.array_equal(fout2, 2 * fout) and np.array_equal(flse2, flse)


# ------------------------------------------------------ grouped-query attention

@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_gqa_oracle_equals_mha_on_repeated_kv_heads(G):
    """GQA with group size G equals multi-head attention with each K/V head
    repeated G times (numpy repeat), bit for bit; G = 1 is plain MHA."""
    rng = np.random.default_rng(G)
    B, Hkv, N, d = 2, 3, 50, 16
    q = _f32(rng.normal(size=(B, Hkv * G, d)))
    K = _f32(rng.normal(size=(B, Hkv, N, d)) * 2)
    V = _f32(rng.normal(size=(B, Hkv, N, d)))
    lens = np.array([50, 23], np.int32)
    gout, glse = oracle.attention_gqa(q, K, V, lens=lens)
    Kr = np.repeat(K, G, axis=1)
    Vr = np.repeat(V, G, axis=1)
    out, lse = oracle.attention(q, Kr, Vr, lens=lens)
    assert np.array_equal(gout, out) and np.array_equal(glse, lse)
    with pytest.raises(ValueError):
        oracle.attention_gqa(q[:, :-1] if G > 1 else q, K[:, :2] if G == 1 else K, V)
