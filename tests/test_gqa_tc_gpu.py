"""Grouped-query decode with large groups (MQA / GQA with at least 17 query
heads per K/V head): the tcgen05 kernel, whose products run on the
fifth-generation tensor cores with TMEM accumulators, against the float64
GQA oracle ("从第一性原理推导 Flash Attention" §8).

Covers groups from 17 to 256 (two slices of 128), head dims 64 and 128,
bf16 and f16, the automatic decomposition and explicit splits, lengths 0,
shorter than one 64-token chunk and ragged, peaked scores (the lazy
rescale of the O rows in TMEM), one long sequence cut into many pieces
(the last arriver's merge in one batch and, past 64 pieces, in batches
whose results are written back as partials), and both output dtypes.
Padding rows are NaN.
"""
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import random_case
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}
DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _gqa_case(B, Hq, Hkv, N, d, dtype, lens, seed, k_scale=1.0):
    _, k, v, lt = random_case(B, Hkv, N, d, dtype, lens=lens, seed=seed, k_scale=k_scale)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, d, generator=g).to(DT[dtype])
    return q, k, v, lt


def _run(q, k, v, lt, dtype, num_splits=0):
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    out, lse = fd.decode_gqa(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), num_splits=num_splits,
                             out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)
    out16, _ = fd.decode_gqa(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), num_splits=num_splits,
                             out_dtype=DT[dtype])
    check_out(out16, ref_out, dtype)
    assert fd.device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [17, 32, 33, 48, 64, 128])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_large_groups_match_oracle(dtype, d, G, num_splits):
    Hkv = 2
    q, k, v, lt = _gqa_case(3, Hkv * G, Hkv, 700, d, dtype, [700, 0, 13], seed=G + d)
    _run(q, k, v, lt, dtype, num_splits)


@pytest.mark.parametrize("G", [40, 200, 256])
def test_groups_in_slices_and_uneven(G):
    """G = 40 (one slice, rows past 40 idle), 200 (two slices of 100) and 256
    (two full slices) on one K/V head, ragged lengths."""
    q, k, v, lt = _gqa_case(4, G, 1, 1500, 128, "bf16", [1500, 64, 65, 1], seed=G)
    _run(q, k, v, lt, "bf16")


def test_peaked_scores_rescale_o_in_tmem():
    """K scaled by 8 over 20K tokens: the running max grows by more than the
    lazy-rescale threshold many times, so the O rows in TMEM are rescaled."""
    q, k, v, lt = _gqa_case(2, 64, 1, 20000, 128, "bf16", [20000, 9001], seed=5, k_scale=8.0)
    _run(q, k, v, lt, "bf16")


@pytest.mark.parametrize("G,d", [(64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("num_splits", [0, 40, 100])
def test_long_sequence_many_pieces(G, d, num_splits):
    """One long sequence: cut into one piece per CTA (automatic: 152 pieces,
    three merge batches), into 40 explicit splits (one batch) and into 100
    (two batches).  The last arriver is at its last segment, so it stages
    the pieces in its idle ring: blocks of 16 heads (40 pieces of 64 heads)
    down to one head per block (64 pieces of 128 heads at d = 128)."""
    q, k, v, lt = _gqa_case(1, G, 1, 150000 if G == 64 else 60000, d, "bf16", None, seed=11 + G + d)
    _run(q, k, v, lt, "bf16", num_splits)


def test_many_short_sequences():
    """96 sequences of 1..300 tokens on 2 K/V heads with G = 64: many
    segments per CTA, most shorter than a chunk."""
    lens = [(37 * i) % 301 for i in range(96)]
    q, k, v, lt = _gqa_case(96, 128, 2, 300, 128, "f16", lens, seed=3)
    _run(q, k, v, lt, "f16")


def test_alternating_queries_reuse_the_workspace():
    """Two query sets in turn, eight launches through the same workspace,
    with 152 pieces merged in three batches: the last arriver reads the
    other pieces' partials and its own intermediate batches back from the
    workspace, so a read that saw the previous launch's data (the same
    slots, the other query set) would show against each set's oracle."""
    _, k, v, lt = random_case(1, 1, 60000, 128, "bf16", lens=None, seed=21)
    qs = [torch.randn(1, 128, 128, generator=torch.Generator().manual_seed(s)).to(torch.bfloat16) for s in (1, 2)]
    refs = [oracle.attention_gqa(q, k, v, lens=lt) for q in qs]
    kd, vd, ld = k.to(DEV), v.to(DEV), lt.to(DEV)
    for r in range(8):
        i = r % 2
        od = torch.float32 if r < 4 else torch.bfloat16
        out, lse = fd.decode_gqa(qs[i].to(DEV), kd, vd, ld, out_dtype=od)
        check_out(out, refs[i][0], "bf16")
        check_lse(lse, refs[i][1], "bf16")
    assert fd.device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_start_charge_empty_pieces(d):
    """Sequences of 1, 2 and 5000 tokens: the automatic decomposition charges
    every sequence a start cost in the space the CTAs divide, so the short
    sequences' spans are mostly charge, and a dozen CTAs each hold an empty
    piece (no tokens) of the same sequence next to the one that holds its
    tokens; the merge gives the empty pieces weight 0."""
    q, k, v, lt = _gqa_case(3, 64, 1, 5000, d, "bf16", [1, 2, 5000], seed=31 + d)
    _run(q, k, v, lt, "bf16")
