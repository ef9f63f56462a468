"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small cases span several chunks, several CTAs per sequence and ragged tails;
inputs are seeded (split_kv_fd_gb300.inputs) and the padding past every
sequence's length is NaN, so any out-of-range read fails the test.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import random_case
from parity_util import check_lse, check_out, to_np

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _case(B, H, N, d, dtype, lens, seed, k_scale=1.0):
    q, k, v, lt = random_case(B, H, N, d, dtype, lens=lens, seed=seed, k_scale=k_scale)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    dev = torch.device("cuda")
    return (q.to(dev), k.to(dev), v.to(dev), lt.to(dev)), (q, k, v, lt), ref_out, ref_lse


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("num_splits", [0, 1, 3, 7])
def test_fused_decode_matrix(dtype, d, num_splits):
    (q, k, v, lt), _, ref_out, ref_lse = _case(3, 5, 700, d, dtype, [700, 0, 333], seed=d + 3)
    out, lse = fd.decode(q, k, v, lt, num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)
    if dtype != "f32":  # the storage dtype as output: adds its own rounding
        out16, lse16 = fd.decode(q, k, v, lt, num_splits=num_splits, out_dtype=DT[dtype])
        check_out(out16, ref_out, dtype)
        check_lse(lse16, ref_lse, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("P", [1, 2, 5, 64, 1003])
def test_split_partials_match_oracle_tiles(dtype, P):
    (q, k, v, lt), (qc, kc, vc, lc), _, _ = _case(2, 3, 1000, 128, dtype, [1000, 517], seed=P)
    o, m, l, s = fd.decode_split(q, k, v, P, seqlens=lt)
    ro, rm, rl, rs = oracle.split_partials(qc, kc, vc, P, lens=lc)
    empty = rl == 0
    gm, gl, gs = to_np(m), to_np(l), to_np(s)
    assert np.all(gl[empty] == 0) and np.all(gm[empty] == -np.inf) and np.all(gs[empty] == -np.inf)
    assert np.all(to_np(o)[empty] == 0)
    ne = ~empty
    tol_o = 1e-5 if dtype == "f32" else 2e-3
    assert np.max(np.abs(to_np(o)[ne] - ro[ne])) <= tol_o
    assert np.max(np.abs(gm[ne] - rm[ne]) / np.maximum(1, np.abs(rm[ne]))) <= 1e-5
    assert np.max(np.abs(gl[ne] - rl[ne]) / rl[ne]) <= 1e-5
    assert np.max(np.abs(gs[ne] - rs[ne])) <= (1e-5 if dtype == "f32" else 1e-3)


@pytest.mark.parametrize("form", ["mlo", "lse"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_combine_on_synthetic_partials(form, out_dtype):
    """Combine kernels against the oracle's merges on arbitrary partials with
    wide m ranges and empty splits (including all-empty rows)."""
    g = torch.Generator().manual_seed(17)
    B, H, P, d = 3, 7, 37, 128
    o = torch.randn(B, H, P, d, generator=g)
    m = torch.randn(B, H, P, generator=g) * 40
    l = torch.rand(B, H, P, generator=g) * 100 + 1
    empty = torch.rand(B, H, P, generator=g) < 0.3
    empty[1, 2, :] = True
    o[empty] = 0
    m[empty] = -math.inf
    l[empty] = 0
    s = torch.where(empty, torch.tensor(-math.inf), m + torch.log(torch.where(empty, torch.ones_like(l), l)))
    dev = torch.device("cuda")
    if form == "mlo":
        out, lse = fd.combine_mlo(o.to(dev), m.to(dev), l.to(dev), out_dtype=out_dtype)
        ro, rl = oracle.combine_mlo(o.double().numpy(), m.double().numpy(), l.double().numpy())
    else:
        out, lse = fd.combine_lse(o.to(dev), s.to(dev), out_dtype=out_dtype)
        ro, rl = oracle.combine_lse(o.double().numpy(), s.double().numpy())
    check_out(out, ro, "f32" if out_dtype == torch.float32 else "bf16")
    fin = np.isfinite(rl)
    got = to_np(lse)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.max(np.abs(got[fin] - rl[fin]) / np.maximum(1, np.abs(rl[fin]))) <= 1e-6
    assert np.all(to_np(out)[1, 2] == 0)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_split_then_both_combines(dtype):
    (q, k, v, lt), _, ref_out, ref_lse = _case(4, 4, 2049, 128, dtype, "ragged", seed=11)
    for P in (1, 4, 33):
        o, m, l, s = fd.decode_split(q, k, v, P, seqlens=lt)
        for out, lse in (fd.combine_mlo(o, m, l), fd.combine_lse(o, s)):
            check_out(out, ref_out, dtype)
            check_lse(lse, ref_lse, dtype)


def test_split_invariance_across_decompositions():
    (q, k, v, lt), _, ref_out, ref_lse = _case(2, 8, 5000, 128, "bf16", [5000, 4097], seed=5,
                                               k_scale=8.0)
    outs = []
    for ns in (0, 1, 2, 3, 16, 129, 5000):
        out, lse = fd.decode(q, k, v, lt, num_splits=ns, out_dtype=torch.float32)
        check_out(out, ref_out, "bf16")
        check_lse(lse, ref_lse, "bf16")
        outs.append(to_np(out))
    spread = max(np.max(np.abs(a - outs[0])) for a in outs)
    assert spread <= 1e-4


def test_repeat_calls_are_deterministic_and_reuse_workspace():
    (q, k, v, lt), _, ref_out, ref_lse = _case(3, 16, 3000, 128, "bf16", "ragged", seed=8)
    ws = fd.new_workspace(3, 16, 3000, 128, 0)
    first = None
    for _ in range(5):
        out, lse = fd.decode(q, k, v, lt, workspace=ws, out_dtype=torch.float32)
        if first is None:
            first = (out.clone(), lse.clone())
            check_out(out, ref_out, "bf16")
            check_lse(lse, ref_lse, "bf16")
        else:
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1])


def test_edge_shapes():
    dev = torch.device("cuda")
    # a single token, d=64
    (q, k, v, lt), _, ro, rl = _case(1, 1, 1, 64, "f32", None, seed=2)
    out, lse = fd.decode(q, k, v, lt)
    check_out(out, ro, "f32")
    check_lse(lse, rl, "f32")
    # fewer tokens than CTAs, many heads of length 0..5
    (q, k, v, lt), _, ro, rl = _case(6, 3, 5, 128, "bf16", [0, 1, 2, 3, 4, 5], seed=3)
    for ns in (0, 2, 9):
        out, lse = fd.decode(q, k, v, lt, num_splits=ns, out_dtype=torch.float32)
        check_out(out, ro, "bf16")
        check_lse(lse, rl, "bf16")
    # N = 0: every sequence empty
    q = torch.randn(2, 3, 128, device=dev, dtype=torch.bfloat16)
    kv = torch.empty(2, 3, 0, 128, device=dev, dtype=torch.bfloat16)
    for ns in (0, 1, 4):
        out, lse = fd.decode(q, kv, kv, None, num_splits=ns, out_dtype=torch.float32)
        assert torch.all(out == 0) and torch.all(lse == -math.inf)
    # B*H == 0: nothing to do
    z = torch.empty(0, 4, 128, device=dev, dtype=torch.bfloat16)
    out, lse = fd.decode(z, torch.empty(0, 4, 8, 128, device=dev, dtype=torch.bfloat16),
                         torch.empty(0, 4, 8, 128, device=dev, dtype=torch.bfloat16))
    assert out.numel() == 0
    # lengths beyond N are clamped to N
    (q, k, v, lt), (qc, kc, vc, _), _, _ = _case(2, 2, 300, 128, "bf16", [300, 300], seed=4)
    ro, rl = oracle.attention(qc, kc, vc, lens=[300, 300])
    out, lse = fd.decode(q, k, v, torch.tensor([10 ** 6, 300], dtype=torch.int32, device=dev),
                         out_dtype=torch.float32)
    check_out(out, ro, "bf16")
    check_lse(lse, rl, "bf16")
    # no seqlens tensor: all N
    out, lse = fd.decode(q, k, v, None, out_dtype=torch.float32)
    check_out(out, ro, "bf16")


def test_large_batch_uses_split_decomposition():
    """B above the balanced decomposition's limit (1024) falls back to splits."""
    (q, k, v, lt), _, ro, rl = _case(1100, 1, 40, 64, "bf16", "ragged", seed=6)
    out, lse = fd.decode(q, k, v, lt, out_dtype=torch.float32)
    check_out(out, ro, "bf16")
    check_lse(lse, rl, "bf16")


def test_output_canaries_untouched():
    (q, k, v, lt), _, ro, rl = _case(2, 4, 900, 128, "bf16", [900, 13], seed=12)
    dev = torch.device("cuda")
    guard = 4096
    out_buf = torch.full((guard * 2 + 2 * 4 * 128,), 7.0, device=dev, dtype=torch.float32)
    lse_buf = torch.full((guard * 2 + 2 * 4,), 7.0, device=dev, dtype=torch.float32)
    out = out_buf[guard:guard + 2 * 4 * 128].view(2, 4, 128)
    lse = lse_buf[guard:guard + 8].view(2, 4)
    fd.decode(q, k, v, lt, out=out, lse=lse)
    check_out(out, ro, "bf16")
    check_lse(lse, rl, "bf16")
    assert torch.all(out_buf[:guard] == 7) and torch.all(out_buf[-guard:] == 7)
    assert torch.all(lse_buf[:guard] == 7) and torch.all(lse_buf[-guard:] == 7)


def test_host_side_errors():
    dev = torch.device("cuda")
    lib = fd.load()
    q = torch.randn(1, 1, 128, device=dev, dtype=torch.bfloat16)
    k = torch.randn(1, 1, 64, 128, device=dev, dtype=torch.bfloat16)
    out = torch.empty(1, 1, 128, device=dev, dtype=torch.bfloat16)
    ws = fd.new_workspace(1, 1, 64, 128)
    nbytes = ws.numel()
    import ctypes
    P = ctypes.c_void_p
    # misaligned K
    st = lib.fd_decode(P(q.data_ptr()), P(k.data_ptr() + 2), P(k.data_ptr()), None, 1, 1, 32, 128, 2, 0,
                       1.0, P(out.data_ptr()), 2, None, P(ws.data_ptr()), nbytes, None)
    assert st == 1
    # unsupported head dim
    st = lib.fd_decode(P(q.data_ptr()), P(k.data_ptr()), P(k.data_ptr()), None, 1, 1, 64, 96, 2, 0,
                       1.0, P(out.data_ptr()), 2, None, P(ws.data_ptr()), nbytes, None)
    assert st == 2
    # workspace too small
    st = lib.fd_decode(P(q.data_ptr()), P(k.data_ptr()), P(k.data_ptr()), None, 1, 1, 64, 128, 2, 0,
                       1.0, P(out.data_ptr()), 2, None, P(ws.data_ptr()), 16, None)
    assert st == 3
    with pytest.raises(ValueError):
        fd.decode(q.cpu(), k.cpu(), k.cpu())
    with pytest.raises(fd.FDError):
        fd.decode_split(q, k, k, 0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("num_splits", [0, 3])
def test_workspace_needs_no_initialisation(num_splits):
    """A workspace full of garbage (here 0xFF bytes) gives the same result:
    the call clears the arrival counters it uses."""
    (q, k, v, lt), _, ro, rl = _case(2, 6, 1500, 128, "bf16", [1500, 700], seed=21)
    ws = fd.new_workspace(2, 6, 1500, 128, num_splits)
    ws.fill_(255)
    out, lse = fd.decode(q, k, v, lt, num_splits=num_splits, workspace=ws, out_dtype=torch.float32)
    check_out(out, ro, "bf16")
    check_lse(lse, rl, "bf16")
