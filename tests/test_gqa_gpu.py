"""Grouped-query decode on the GPU (fd_decode_gqa, tensor-core path for
G >= 2, in slices of at most 16 query heads) against the float64 GQA oracle.  Lengths include 0, shorter than
one chunk, and ragged tails; padding rows are NaN."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import random_case
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


def _gqa_case(B, Hq, Hkv, N, d, dtype, lens, seed, k_scale=1.0):
    # K/V with Hkv heads; q drawn separately with Hq heads
    _, k, v, lt = random_case(B, Hkv, N, d, dtype, lens=lens, seed=seed, k_scale=k_scale)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, d, generator=g).to(DT[dtype])
    return q, k, v, lt


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [2, 4, 8, 16])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_gqa_matches_oracle(dtype, d, G, num_splits):
    Hkv = 2
    q, k, v, lt = _gqa_case(3, Hkv * G, Hkv, 700, d, dtype, [700, 0, 13], seed=G + d)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), num_splits=num_splits,
                             out_dtype=torch.float32)
    check_out(out, ref_out, dtype)
    check_lse(lse, ref_lse, dtype)
    out16, _ = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), num_splits=num_splits,
                             out_dtype=DT[dtype])
    check_out(out16, ref_out, dtype)


def test_gqa_peaked_scores_and_long_sequences():
    """K scaled by 8 (near one-hot attention) over 20K tokens, G = 8."""
    q, k, v, lt = _gqa_case(2, 32, 4, 20000, 128, "bf16", [20000, 7777], seed=5, k_scale=8.0)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_gqa_group_of_one_is_decode_and_errors():
    dev = torch.device("cuda")
    q, k, v, lt = _gqa_case(2, 4, 4, 300, 128, "bf16", [300, 100], seed=2)
    a = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev))
    b = fd.decode(q.to(dev), k.to(dev), v.to(dev), lt.to(dev))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    # f32 with G > 1 is not supported (the tensor cores take 16-bit operands)
    qf = torch.randn(1, 4, 64, device=dev)
    kf = torch.randn(1, 2, 64, 64, device=dev)
    with pytest.raises(fd.FDError):
        fd.decode_gqa(qf, kf, kf)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16",
                                  "decode_gqa_b2_hq64_hkv8_n32k_d128_bf16",
                                  "decode_gqa_b8_hq16_hkv8_n32k_d256_bf16",
                                  "decode_mqa_b32_hq64_hkv1_n32k_d128_bf16"])
def test_gqa_benchmark_workloads_sampled(name):
    """The benchmarked GQA workloads at full size, in the launch the benchmark
    times (automatic decomposition, the workload's own output dtype, and f32):
    sampled query rows against the oracle, each row computed one by one as
    plain attention of that query head over its K/V head (h // G); every
    output finite and inside the range of its V column."""
    from split_kv_fd_gb300.inputs import make_inputs
    from split_kv_fd_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    G = w.H // w.kv_heads
    q, k, v, lens = make_inputs(w, device="cuda")
    rng = np.random.default_rng(5)
    # the first and last query heads of the first K/V head and the first of
    # the second (when there is one)
    rows = {(0, 0), (w.B - 1, w.H - 1), (0, G - 1), (w.B - 1, min(G, w.H - 1))}
    while len(rows) < 12:
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.H))))
    rows = sorted(rows)
    ref_o, ref_s = [], []
    for b, h in rows:
        o, s = oracle.attention(q[b:b + 1, h:h + 1].cpu(), k[b:b + 1, h // G:h // G + 1].cpu(),
                                v[b:b + 1, h // G:h // G + 1].cpu(), scale=w.scale)
        ref_o.append(o[0, 0])
        ref_s.append(s[0, 0])
    ref_o, ref_s = np.stack(ref_o), np.array(ref_s)
    bi = torch.tensor([r[0] for r in rows])
    hi = torch.tensor([r[1] for r in rows])
    for odt in (DT[w.out_dtype], torch.float32):
        out, lse = fd.decode_gqa(q, k, v, lens, scale=w.scale, out_dtype=odt)
        eo = check_out(out[bi, hi], ref_o, w.dtype, what=f"{name} {odt} out")
        el = check_lse(lse[bi, hi], ref_s, w.dtype, what=f"{name} {odt} lse")
        print(f"PARITY {name} out={odt} rows={len(rows)} max_err_out={eo:.3e} max_err_lse={el:.3e}")
        assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
    # every query row is a convex combination of its K/V head's V rows
    for b in range(w.B):
        vb = v[b].float()                                  # [Hkv, N, d]
        lo = vb.amin(dim=1).repeat_interleave(G, dim=0) - 1e-3
        hi_ = vb.amax(dim=1).repeat_interleave(G, dim=0) + 1e-3
        assert bool(torch.all(out[b] >= lo)) and bool(torch.all(out[b] <= hi_)), f"batch {b}"
        del vb
    del q, k, v
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("d,G,Hkv", [(128, 17, 2), (128, 24, 2), (128, 32, 1), (64, 48, 1), (128, 64, 1),
                                     (256, 12, 2), (256, 32, 1)])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_gqa_large_groups_and_mqa(d, G, Hkv, num_splits):
    """More query heads per K/V head than one warp holds (16; 8 at d = 256):
    the heads are served as slices of at most that many, each reading the
    same K/V rows.  Hkv = 1 is MQA.  Contiguous and in 16- and 64-token
    pages, lengths 700/0/333."""
    from split_kv_fd_gb300.inputs import to_paged
    q, k, v, lt = _gqa_case(3, G * Hkv, Hkv, 700, d, "bf16", [700, 0, 333], seed=G + d + num_splits)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    qd, ld = q.to(dev), lt.to(dev)
    out, lse = fd.decode_gqa(qd, k.to(dev), v.to(dev), ld, num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    for ps in (16, 64):
        kp, vp, table = to_paged(k, v, ps, seed=ps)
        pout, plse = fd.decode_gqa_paged(qd, kp.to(dev), vp.to(dev), table.to(dev), ld,
                                         num_splits=num_splits, out_dtype=torch.float32)
        check_out(pout, ref_out, "bf16")
        check_lse(plse, ref_lse, "bf16")


def test_mqa_long_sequence_many_pieces():
    """MQA, 64 query heads on one K/V head of 100K tokens: four slices of 16
    heads, each cut into pieces across the CTAs and merged by the last."""
    q, k, v, lt = _gqa_case(1, 64, 1, 100000, 128, "bf16", None, seed=41)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


@pytest.mark.parametrize("G", [8, 24])
def test_gqa_more_sequences_than_the_balanced_limit(G):
    """1100 sequences (more than the balanced decomposition's 1024): the
    automatic split count, with and without slices of the query heads."""
    B, Hkv, N, d = 1100, 2, 96, 64
    g = torch.Generator().manual_seed(G)
    lens = torch.randint(0, N + 1, (B,), generator=g).tolist()
    q, k, v, lt = _gqa_case(B, G * Hkv, Hkv, N, d, "bf16", lens, seed=50 + G)
    ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_gqa(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
