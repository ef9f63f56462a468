"""Decompositions that give a CTA many segments, and (b, h) sequences cut into
many pieces, on the GPU against the float64 oracle.

- Many short sequences: each CTA of the balanced decomposition walks tens of
  (b, h) segments, more than the split kernel keeps in flight between its
  streaming warps and its merge warp (4 buffers for 16-bit K/V, 2 for FP8),
  so the buffers are reused many times over.
- Explicit split counts with many items per CTA (DECOMP_SPLITS).
- GQA sequences cut into more pieces than the last arriver stages in shared
  memory (64), and into fewer, with both decompositions.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import quantize_e4m3, random_case
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _short_lengths(B, lo, hi, seed):
    g = np.random.default_rng(seed)
    lens = g.integers(lo, hi + 1, size=B)
    lens[::17] = 0          # some empty sequences among them
    return [int(x) for x in lens]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("num_splits", [0, 7])
def test_many_short_sequences(dtype, num_splits):
    """256 x 16 short (b, h) rows: tens of segments per CTA."""
    B, H, N, d = 256, 16, 48, 128
    q, k, v, lt = random_case(B, H, N, d, dtype, lens=_short_lengths(B, 1, N, 3), seed=11)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), num_splits=num_splits,
                         out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)


def test_many_short_sequences_fp8():
    """The FP8 kernel keeps 2 segment buffers: the same many-segment walk."""
    B, H, N, d = 192, 16, 64, 128
    q, k, v, lt = random_case(B, H, N, d, "bf16", lens=_short_lengths(B, 1, N, 4), seed=12,
                              nan_pad=False)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = oracle.attention_fp8(q, k8, v8, ks, vs, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_fp8(q.to(dev), k8.to(dev), v8.to(dev), ks.to(dev), vs.to(dev), lt.to(dev),
                             out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_split_items_many_per_cta():
    """16 x 32 rows x 9 splits = 4608 items: ~30 split items per CTA."""
    B, H, N, d = 16, 32, 1500, 64
    q, k, v, lt = random_case(B, H, N, d, "bf16", lens="ragged", seed=13)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), num_splits=9,
                         out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def _gqa_case(B, Hq, Hkv, N, d, lens, seed):
    _, k, v, lt = random_case(B, Hkv, N, d, "bf16", lens=lens, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    return q, k, v, lt


@pytest.mark.parametrize("num_splits", [0, 40, 100])
def test_gqa_sequence_in_many_pieces(num_splits):
    """One (b, kv head) of 150K tokens: the balanced decomposition cuts it
    into one piece per CTA (more than 64), explicit splits into 40 or 100."""
    q, k, v, lt = _gqa_case(1, 8, 1, 150000, 128, None, seed=21)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), num_splits=num_splits,
                             out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_gqa_sixteen_heads_in_many_pieces():
    """G = 16 (two column tiles of heads) across many CTAs, ragged lengths."""
    q, k, v, lt = _gqa_case(2, 32, 2, 40000, 64, [40000, 12345], seed=22)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
