"""Grouped-query decode over a paged KV cache on the GPU (fd_decode_gqa_paged):
against the float64 GQA oracle on the contiguous rows, and against
fd_decode_gqa on the same rows laid out contiguously: bit for bit when the
page size is a multiple of 32 (the kernel walks the same chunks of logical
tokens; only the rows' addresses differ), within fp32 rounding for 16-token
pages (a chunk that starts inside its aligned 32-token block has its tokens
split between the two warps differently).  Pages are in a seeded random
order; unused pages and rows past each length are NaN, so a row read past a
chunk's valid tokens shows up."""
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import make_inputs, random_case, to_paged
from split_kv_fd_gb300.workloads import WORKLOADS
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _same_as_contiguous(page_size, out, lse, cout, clse):
    if page_size % 32 == 0:
        assert torch.equal(out, cout) and torch.equal(lse, clse)
    else:
        assert float((out - cout).abs().max()) <= 2e-5
        fin = torch.isfinite(clse)
        assert torch.equal(torch.isfinite(lse), fin)
        assert float((lse[fin] - clse[fin]).abs().max()) <= 2e-5


def _case(B, Hq, Hkv, N, d, dtype, lens, seed):
    _, k, v, lt = random_case(B, Hkv, N, d, dtype, lens=lens, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, d, generator=g).to(DT[dtype])
    return q, k, v, lt


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64)])
@pytest.mark.parametrize("G", [2, 8, 16])
@pytest.mark.parametrize("page_size", [16, 32, 64, 160])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_gqa_paged_matches_oracle_and_contiguous(dtype, d, G, page_size, num_splits):
    Hkv = 2
    q, k, v, lt = _case(3, G * Hkv, Hkv, 700, d, dtype, [700, 0, 333], seed=page_size + G)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    kp, vp, table = to_paged(k, v, page_size, seed=page_size)
    dev = torch.device("cuda")
    qd, kd, vd, ld = (t.to(dev) for t in (q, k, v, lt))
    out, lse = fd.decode_gqa_paged(qd, kp.to(dev), vp.to(dev), table.to(dev), ld, num_splits=num_splits,
                                   out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)
    cout, clse = fd.decode_gqa(qd, kd, vd, ld, num_splits=num_splits, out_dtype=torch.float32)
    _same_as_contiguous(page_size, out, lse, cout, clse)


def test_gqa_paged_group_of_one_is_paged_decode():
    q, k, v, lt = random_case(2, 4, 300, 128, "bf16", lens=[300, 77], seed=9)
    kp, vp, table = to_paged(k, v, 64, seed=2)
    dev = torch.device("cuda")
    args = (q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lt.to(dev))
    out, lse = fd.decode_gqa_paged(*args, out_dtype=torch.float32)
    pout, plse = fd.decode_paged(*args, out_dtype=torch.float32)
    assert torch.equal(out, pout) and torch.equal(lse, plse)


@pytest.mark.parametrize("page_size", [8, 48])
def test_gqa_paged_rejects_other_page_sizes(page_size):
    q, k, v, lt = _case(1, 8, 2, 96, 128, "bf16", None, seed=4)
    kp, vp, table = to_paged(k, v, page_size, seed=1)
    dev = torch.device("cuda")
    with pytest.raises(fd.FDError) as e:
        fd.decode_gqa_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lt.to(dev))
    assert e.value.status == 2   # FD_ERR_UNSUPPORTED: 16 or a multiple of 32 tokens


@pytest.mark.parametrize("num_splits", [0, 5, 40])
def test_gqa_paged16_chunks_starting_mid_page(num_splits):
    """16-token pages with segment starts at every offset in a page: many
    short ragged sequences and explicit splits put chunk starts anywhere in
    the aligned 32-token block, so rows before a chunk's first token are
    masked as well as rows after its last."""
    B, Hkv, G, N, d = 24, 2, 8, 150, 128
    g = torch.Generator().manual_seed(17)
    lens = torch.randint(0, N + 1, (B,), generator=g).tolist()
    q, k, v, lt = _case(B, G * Hkv, Hkv, N, d, "bf16", lens, seed=18)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    kp, vp, table = to_paged(k, v, 16, seed=19)
    dev = torch.device("cuda")
    qd, ld = q.to(dev), lt.to(dev)
    out, lse = fd.decode_gqa_paged(qd, kp.to(dev), vp.to(dev), table.to(dev), ld, num_splits=num_splits,
                                   out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    cout, clse = fd.decode_gqa(qd, k.to(dev), v.to(dev), ld, num_splits=num_splits,
                               out_dtype=torch.float32)
    _same_as_contiguous(16, out, lse, cout, clse)


def test_gqa_paged_bad_table_entry_is_reported_not_dereferenced():
    dev = torch.device("cuda")
    q, k, v, lt = _case(2, 16, 2, 256, 128, "bf16", [256, 256], seed=5)
    kp, vp, table = to_paged(k, v, 32, seed=1)
    bad = table.clone()
    bad[1, 2] = 10 ** 6       # names no page
    bad[0, 0] = -5
    fd.decode_gqa_paged(q.to(dev), kp.to(dev), vp.to(dev), bad.to(dev), lt.to(dev))
    assert fd.device_status(reset=True) == 7   # FD_ERR_BAD_PAGE, then cleared
    assert fd.device_status() == 0
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    out, lse = fd.decode_gqa_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lt.to(dev),
                                   out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    assert fd.device_status() == 0


@pytest.mark.slow
def test_gqa_paged_full_size_equals_contiguous():
    """The benchmarked GQA workload (1 GiB of K/V, G = 8) in 16-, 64- and
    256-token pages, automatic decomposition."""
    w = WORKLOADS["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"]
    q, k, v, lens = make_inputs(w, device="cuda")
    cout, clse = fd.decode_gqa(q, k, v, lens, scale=w.scale, out_dtype=torch.float32)
    for ps in (16, 64, 256):
        kp, vp, table = to_paged(k, v, ps, seed=ps)
        out, lse = fd.decode_gqa_paged(q, kp, vp, table, lens, scale=w.scale, out_dtype=torch.float32)
        _same_as_contiguous(ps, out, lse, cout, clse)
        del kp, vp
        torch.cuda.empty_cache()
