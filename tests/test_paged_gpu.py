"""Paged KV cache on the GPU: fd_decode_paged against the float64 paged
oracle, and bit-for-bit against fd_decode on the same rows laid out
contiguously (the kernel walks logical tokens, so the arithmetic is the same
whatever the page order).  Unused pages and rows past each length are NaN.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import make_inputs, random_case, to_paged
from split_kv_fd_gb300.workloads import WORKLOADS
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 128), ("f32", 64), ("bf16", 64)])
@pytest.mark.parametrize("page_size", [1, 3, 16, 64, 100])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_paged_matches_oracle_and_contiguous(dtype, d, page_size, num_splits):
    q, k, v, lt = random_case(3, 4, 700, d, dtype, lens=[700, 0, 333], seed=page_size + d)
    kp, vp, table = to_paged(k, v, page_size, seed=page_size)
    ref_out, ref_lse = oracle.attention_paged(q, kp, vp, table, lt)
    dev = torch.device("cuda")
    qd, kd, vd, ld = (t.to(dev) for t in (q, k, v, lt))
    kpd, vpd, td = kp.to(dev), vp.to(dev), table.to(dev)
    out, lse = fd.decode_paged(qd, kpd, vpd, td, ld, num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)
    cout, clse = fd.decode(qd, kd, vd, ld, num_splits=num_splits, out_dtype=torch.float32)
    assert torch.equal(out, cout) and torch.equal(lse, clse)


def test_paged_full_size_equals_contiguous():
    """The benchmark workload (4 GiB of K/V) paged in 16- and 128-token pages."""
    w = WORKLOADS["decode_b8_h32_n32k_d128_bf16"]
    q, k, v, lens = make_inputs(w, device="cuda")
    cout, clse = fd.decode(q, k, v, lens, scale=w.scale)
    for ps in (16, 128):
        kp, vp, table = to_paged(k, v, ps, seed=ps)
        out, lse = fd.decode_paged(q, kp, vp, table, lens, scale=w.scale)
        assert torch.equal(out, cout) and torch.equal(lse, clse), ps
        del kp, vp
        torch.cuda.empty_cache()


def test_bad_table_entry_is_reported_not_dereferenced():
    dev = torch.device("cuda")
    q, k, v, lt = random_case(2, 2, 64, 128, "bf16", lens=[64, 64], seed=3)
    kp, vp, table = to_paged(k, v, 16, seed=1)
    table = table.clone()
    table[1, 2] = 10 ** 6     # names no page
    table[0, 0] = -5
    out, lse = fd.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lt.to(dev))
    assert fd.device_status(reset=True) == 7   # FD_ERR_BAD_PAGE, then cleared
    assert fd.device_status() == 0
    # with a valid table the same call is clean and correct
    kp2, vp2, table2 = to_paged(k, v, 16, seed=1)
    ref_out, ref_lse = oracle.attention_paged(q, kp2, vp2, table2, lt)
    out, lse = fd.decode_paged(q.to(dev), kp2.to(dev), vp2.to(dev), table2.to(dev), lt.to(dev),
                               out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    assert fd.device_status() == 0
