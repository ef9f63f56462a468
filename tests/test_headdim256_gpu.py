"""Head dim 256 (16-bit and E4M3 K/V) through every entry point of the split
kernel, against the float64 oracle: fused decode with both decompositions,
the two-call path with both merges, the paged and FP8 caches, the no-alloc
entry point, and many short sequences (the merge warp's segment buffers
hold 256-element rows); and grouped-query decode at d = 256 (G <= 8),
contiguous and paged."""
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import quantize_e4m3, random_case, to_paged
from parity_util import check_lse, check_out, to_np

pytestmark = pytest.mark.gpu

D = 256
DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fused_d256(dtype, num_splits):
    q, k, v, lt = random_case(3, 5, 900, D, dtype, lens=[900, 0, 457], seed=num_splits + 1)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    out, lse = fd.decode(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), num_splits=num_splits,
                         out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)


def test_split_and_both_combines_d256():
    q, k, v, lt = random_case(2, 4, 1000, D, "bf16", lens=[1000, 333], seed=7)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    o, m, l, s = fd.decode_split(q.to(DEV), k.to(DEV), v.to(DEV), 5, seqlens=lt.to(DEV))
    ro, _, _, rs = oracle.split_partials(q, k, v, 5, lens=lt)
    assert float(abs(to_np(o) - ro).max()) <= 2e-3
    for out, lse in (fd.combine_mlo(o, m, l, out_dtype=torch.float32),
                     fd.combine_lse(o, s, out_dtype=torch.float32)):
        check_out(out, ref_out, "bf16")
        check_lse(lse, ref_lse, "bf16")


@pytest.mark.parametrize("page_size", [16, 100])
def test_paged_d256(page_size):
    q, k, v, lt = random_case(3, 4, 700, D, "f16", lens=[700, 0, 333], seed=page_size)
    kp, vp, table = to_paged(k, v, page_size, seed=page_size)
    ref_out, ref_lse = oracle.attention_paged(q, kp, vp, table, lt)
    qd, ld = q.to(DEV), lt.to(DEV)
    out, lse = fd.decode_paged(qd, kp.to(DEV), vp.to(DEV), table.to(DEV), ld, out_dtype=torch.float32)
    check_out(out, ref_out, "f16")
    check_lse(lse, ref_lse, "f16")
    cout, clse = fd.decode(qd, k.to(DEV), v.to(DEV), ld, out_dtype=torch.float32)
    assert torch.equal(out, cout) and torch.equal(lse, clse)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_fp8_d256(num_splits):
    q, k, v, lt = random_case(2, 6, 800, D, "bf16", lens=[800, 271], seed=11, nan_pad=False)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = oracle.attention_fp8(q, k8, v8, ks, vs, lens=lt)
    out, lse = fd.decode_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV), lt.to(DEV),
                             num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_noalloc_d256():
    q, k, v, lt = random_case(2, 8, 1500, D, "bf16", lens=[1500, 64], seed=13)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    out, lse = fd.decode_noalloc(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_many_short_sequences_d256():
    """192 x 8 short rows: tens of segments per CTA through the merge warp's
    4 segment buffers of 256-element rows."""
    g = torch.Generator().manual_seed(3)
    lens = torch.randint(0, 80, (192,), generator=g).tolist()
    q, k, v, lt = random_case(192, 8, 80, D, "bf16", lens=lens, seed=14)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    out, lse = fd.decode(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def _gqa_case(B, Hq, Hkv, N, dtype, lens, seed):
    _, k, v, lt = random_case(B, Hkv, N, D, dtype, lens=lens, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, D, generator=g).to({"bf16": torch.bfloat16, "f16": torch.float16}[dtype])
    return q, k, v, lt


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_gqa_d256(dtype, G, num_splits):
    """The tensor-core kernel at d = 256 (4 warps, G <= 8), contiguous and in
    16- and 64-token pages."""
    q, k, v, lt = _gqa_case(3, 2 * G, 2, 700, dtype, [700, 0, 333], seed=G + num_splits)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    qd, ld = q.to(DEV), lt.to(DEV)
    out, lse = fd.decode_gqa(qd, k.to(DEV), v.to(DEV), ld, num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)
    for ps in (16, 64):
        kp, vp, table = to_paged(k, v, ps, seed=ps)
        pout, plse = fd.decode_gqa_paged(qd, kp.to(DEV), vp.to(DEV), table.to(DEV), ld,
                                         num_splits=num_splits, out_dtype=torch.float32)
        check_out(pout, ref_out, dtype)
        check_lse(plse, ref_lse, dtype)


def test_gqa_d256_long_sequence_in_many_pieces():
    """One 100K-token sequence (G = 8): one piece per CTA, merged by the last."""
    q, k, v, lt = _gqa_case(1, 8, 1, 100000, "bf16", None, seed=31)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    out, lse = fd.decode_gqa(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_gqa_d256_group_of_one():
    q, k, v, lt = random_case(2, 4, 300, D, "bf16", lens=[300, 9], seed=15)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    out, lse = fd.decode_gqa(q.to(DEV), k.to(DEV), v.to(DEV), lt.to(DEV), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")      # G = 1 is fd_decode
