"""fd_merge_lse, the associative (+) of the LSE form, on the GPU: against the
oracle's sequential fold, and as the merge step of a decode whose sequence is
sharded into token ranges (one fd_decode per range, as a sequence-sharded
multi-GPU decode would run, here on one GPU), in sequential and tree order."""
import math

import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import random_case
from parity_util import check_lse, check_out, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def test_merge_matches_oracle_fold_with_empty_rows():
    g = torch.Generator().manual_seed(3)
    rows, d = 301, 128
    o = torch.randn(2, rows, d, generator=g)
    s = torch.randn(2, rows, generator=g) * 30
    s[0, :20] = -math.inf      # empty on one side
    s[1, 10:30] = -math.inf    # rows 10..19 empty on both sides
    o[0, :20] = 0
    o[1, 10:30] = 0
    dev = torch.device("cuda")
    out, lse = fd.merge_lse(o[0].to(dev), s[0].to(dev), o[1].to(dev), s[1].to(dev))
    ro, rl = oracle.merge_lse_sequential(o.permute(1, 0, 2).double().numpy(),
                                         s.permute(1, 0).double().numpy())
    check_out(out, ro, "f32")
    got = to_np(lse)
    assert np.array_equal(np.isfinite(got), np.isfinite(rl))
    fin = np.isfinite(rl)
    assert np.max(np.abs(got[fin] - rl[fin]) / np.maximum(1, np.abs(rl[fin]))) <= 1e-6
    assert np.all(to_np(out)[10:20] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sequence_sharded_decode_folds_to_unsplit(dtype):
    B, H, N, d = 3, 8, 3000, 128
    q, k, v, lt = random_case(B, H, N, d, dtype, lens=[3000, 1200, 5], seed=9)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    dev = torch.device("cuda")
    qd = q.to(dev)
    bounds = [0, 1000, 2100, 3000]
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        ks = k[:, :, a:b].contiguous().to(dev)
        vs = v[:, :, a:b].contiguous().to(dev)
        ls = torch.clamp(lt - a, 0, b - a).to(torch.int32).to(dev)
        parts.append(fd.decode(qd, ks, vs, ls, out_dtype=torch.float32))
    # sequential, in place into the first shard's buffers
    o, s = parts[0][0].clone(), parts[0][1].clone()
    for po, ps in parts[1:]:
        fd.merge_lse(o, s, po, ps, out=o, lse=s)
    check_out(o, ref_out, dtype)
    check_lse(s, ref_lse, dtype)
    # a tree in another order: (p2 (+) p0) (+) p1
    t_o, t_s = fd.merge_lse(parts[2][0], parts[2][1], parts[0][0], parts[0][1])
    t_o, t_s = fd.merge_lse(t_o, t_s, parts[1][0], parts[1][1])
    check_out(t_o, ref_out, dtype)
    check_lse(t_s, ref_lse, dtype)
