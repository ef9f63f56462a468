"""Grouped-query decode over an E4M3 KV cache on the FP8 tcgen05 kernel
(head dim 128; contiguous caches and pages of a multiple of 128 tokens)
against the float64 FP8 oracle on repeated K/V heads ("从第一性原理推导 Flash
Attention" §6.2 and §8).

The kernel splits q and P into three E4M3 parts and runs both products in
FP8 from the staged cache bytes; the cases here aim at its own machinery:
many segments per CTA (short sequences: the softmax groups hand each
segment's result to the epilogue warps through a double staging buffer),
one long sequence cut into more than 64 pieces (the last arriver's merge in
batches), more than 1024 sequences (the split decomposition), the lazy
rescale of the O^T columns (peaked scores, and scores that grow along the
sequence), slices of up to 8 query heads (G = 24 and 40), large pages in a
shuffled pool, q far from 1, and both output dtypes.
"""
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import quantize_e4m3, random_case, to_paged_bytes
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _case(B, Hkv, G, N, lens, seed, k_scale=1.0, q_scale=1.0, qdt=torch.bfloat16):
    _, k, v, lt = random_case(B, Hkv, N, 128, "bf16", lens=lens, seed=seed, k_scale=k_scale, nan_pad=False)
    q = (torch.randn(B, Hkv * G, 128, generator=torch.Generator().manual_seed(seed + 7)) * q_scale).to(qdt)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    return q, k8, v8, ks, vs, lt


def _reference(q, k8, v8, ks, vs, G, lens):
    rep = lambda t: t.repeat_interleave(G, dim=1)   # noqa: E731
    return oracle.attention_fp8(q, rep(k8), rep(v8), rep(ks), rep(vs), lens=lens)


def _check(q, k8, v8, ks, vs, lt, G, num_splits=0, out_dtype=torch.float32):
    ref_out, ref_lse = _reference(q, k8, v8, ks, vs, G, lt)
    out, lse = fd.decode_gqa_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV), lt.to(DEV),
                                 num_splits=num_splits, out_dtype=out_dtype)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    assert fd.device_status() == 0
    return out, lse


def test_many_short_sequences():
    """200 sequences of 0..400 tokens on 2 K/V heads, G = 8: every CTA runs
    several segments, most shorter than one 128-token chunk."""
    lens = [(53 * i) % 401 for i in range(200)]
    _check(*_case(200, 2, 8, 400, lens, seed=1), G=8)


@pytest.mark.parametrize("num_splits", [0, 90])
def test_long_sequence_many_pieces(num_splits):
    """One 100K-token sequence, G = 4: cut into one piece per CTA (152) or
    into 90 explicit splits; the last arriver merges them in batches of 64."""
    _check(*_case(1, 1, 4, 100000, None, seed=2), G=4, num_splits=num_splits)


def test_more_than_1024_sequences():
    """1100 sequences (past the balanced decomposition's prefix-sum limit):
    the split decomposition, one piece per sequence and K/V head."""
    lens = [1 + (97 * i) % 300 for i in range(1100)]
    _check(*_case(1100, 1, 2, 300, lens, seed=3), G=2)


@pytest.mark.parametrize("k_scale", [8.0, 30.0])
def test_peaked_scores(k_scale):
    """K scaled up: the reference max of a softmax group moves many times by
    more than the lazy threshold, so the O^T columns in TMEM are rescaled."""
    _check(*_case(2, 2, 8, 20000, [20000, 7777], seed=4, k_scale=k_scale), G=8)


def test_scores_growing_along_the_sequence():
    """K grows with the token index, so nearly every chunk raises the max."""
    q, k8, v8, ks, vs, lt = _case(1, 1, 8, 8192, None, seed=5)
    ramp = torch.linspace(0.1, 6.0, 8192)[None, None, :, None]
    _, k, _, _ = random_case(1, 1, 8192, 128, "bf16", lens=None, seed=5, nan_pad=False)
    k8, ks = quantize_e4m3((k.float() * ramp).to(torch.bfloat16))
    _check(q, k8, v8, ks, vs, lt, G=8)


@pytest.mark.parametrize("G", [3, 5, 24, 40])
def test_group_sizes_and_slices(G):
    """Groups that leave part-columns idle (3, 5) and groups served as slices
    of at most 8 heads (24: three slices, 40: five)."""
    _check(*_case(3, 2, G, 900, [900, 129, 128], seed=G), G=G)


@pytest.mark.parametrize("qdt,q_scale", [(torch.float32, 1e-3), (torch.float32, 3e4), (torch.float16, 1.0)])
def test_q_magnitudes(qdt, q_scale):
    """q far below and above 1 (each head is brought to amax in [128, 256)
    by a power of two before its parts are taken).  K is scaled by the
    inverse, so that the scores stay near 1: the test is about q's range,
    and with scores near 1e5 no 12-bit q could hold lse to 1e-3."""
    _check(*_case(2, 2, 8, 1000, [1000, 500], seed=6, q_scale=q_scale, k_scale=1.0 / q_scale, qdt=qdt), G=8)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_16bit_outputs(out_dtype):
    _check(*_case(2, 2, 8, 700, [700, 300], seed=7), G=8, out_dtype=out_dtype)


@pytest.mark.parametrize("page_size", [128, 256])
def test_large_pages_equal_contiguous(page_size):
    """Pages of 128 and 256 tokens in a shuffled pool run the same kernel on
    the same chunks as the contiguous cache: bit-identical results."""
    q, k8, v8, ks, vs, lt = _case(4, 2, 8, 1024, [1024, 1, 300, 777], seed=8)
    cout, clse = _check(q, k8, v8, ks, vs, lt, G=8)
    kp, table = to_paged_bytes(k8, page_size, seed=page_size)
    vp, _ = to_paged_bytes(v8, page_size, seed=page_size)
    out, lse = fd.decode_gqa_paged_fp8(q.to(DEV), kp.to(DEV), vp.to(DEV), ks.to(DEV), vs.to(DEV), table.to(DEV),
                                       lt.to(DEV), out_dtype=torch.float32)
    assert torch.equal(out, cout) and torch.equal(lse, clse)
    assert fd.device_status() == 0


def test_start_charge_empty_pieces():
    """Sequences of 1, 2 and 3000 tokens with 4 K/V heads: the start charge
    per sequence makes most of the short sequences' spans empty pieces."""
    _check(*_case(3, 4, 8, 3000, [1, 2, 3000], seed=9), G=8)
