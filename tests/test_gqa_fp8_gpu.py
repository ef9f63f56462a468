"""Grouped-query decode over an E4M3 KV cache (fd_decode_gqa_fp8) against the
float64 oracle.  The reference is the FP8 oracle of one-query-per-head
decode on the K/V heads and scales repeated G times (data movement only:
query head h reads K/V head h / G)."""
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import make_inputs, quantize_e4m3, random_case, to_paged_bytes
from split_kv_fd_gb300.workloads import WORKLOADS
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
QT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _reference(q, k8, v8, ks, vs, G, lens):
    rep = lambda t: t.repeat_interleave(G, dim=1)   # noqa: E731
    return oracle.attention_fp8(q, rep(k8), rep(v8), rep(ks), rep(vs), lens=lens)


@pytest.mark.parametrize("qdt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("G", [2, 8, 16, 24])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_gqa_fp8_matches_oracle(qdt, d, G, num_splits):
    Hkv = 2
    _, k, v, lt = random_case(3, Hkv, 700, d, "bf16", lens=[700, 0, 333], seed=G + d, nan_pad=False)
    q = torch.randn(3, G * Hkv, d, generator=torch.Generator().manual_seed(G)).to(QT[qdt])
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = _reference(q, k8, v8, ks, vs, G, lt)
    out, lse = fd.decode_gqa_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV), lt.to(DEV),
                                 num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_gqa_fp8_peaked_scores_and_many_pieces():
    """K scaled by 8 (peaked softmax) over 60K tokens, one sequence cut into
    one piece per CTA; G = 8."""
    _, k, v, lt = random_case(1, 1, 60000, 128, "bf16", lens=None, seed=5, k_scale=8.0, nan_pad=False)
    q = torch.randn(1, 8, 128, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = _reference(q, k8, v8, ks, vs, 8, lt)
    out, lse = fd.decode_gqa_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV), lt.to(DEV),
                                 out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")


def test_gqa_fp8_group_of_one_and_limits():
    _, k, v, lt = random_case(2, 4, 300, 128, "bf16", lens=[300, 9], seed=7, nan_pad=False)
    q = torch.randn(2, 4, 128).to(torch.bfloat16)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    args = (q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV), lt.to(DEV))
    a = fd.decode_gqa_fp8(*args)
    b = fd.decode_fp8(*args)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])    # G = 1 is fd_decode_fp8
    _, k2, v2, l2 = random_case(1, 1, 64, 96, "bf16", lens=None, seed=8, nan_pad=False)
    k82, ks2 = quantize_e4m3(k2)
    with pytest.raises(fd.FDError) as e:
        fd.decode_gqa_fp8(torch.randn(1, 4, 96, device=DEV).to(torch.bfloat16), k82.to(DEV), k82.to(DEV),
                          ks2.to(DEV), ks2.to(DEV), l2.to(DEV))
    assert e.value.status == 2   # d = 96: FD_ERR_UNSUPPORTED


@pytest.mark.slow
def test_gqa_fp8_benchmark_workload_sampled():
    """The 1 GiB GQA workload stored as E4M3, automatic decomposition, in the
    launch the benchmark times; sampled rows against the oracle."""
    import numpy as np
    w = WORKLOADS["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"]
    G = w.H // w.kv_heads
    q, k, v, lens = make_inputs(w, device="cuda")
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    del k, v
    out, lse = fd.decode_gqa_fp8(q, k8, v8, ks, vs, lens, scale=w.scale, out_dtype=torch.float32)
    rng = np.random.default_rng(9)
    for _ in range(8):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.H))
        kv = h // G
        ro, rs = oracle.attention_fp8(q[b:b + 1, h:h + 1].cpu(), k8[b:b + 1, kv:kv + 1].cpu(),
                                      v8[b:b + 1, kv:kv + 1].cpu(), ks[b:b + 1, kv:kv + 1].cpu(),
                                      vs[b:b + 1, kv:kv + 1].cpu(), scale=w.scale)
        check_out(out[b:b + 1, h:h + 1], ro, "bf16")
        check_lse(lse[b:b + 1, h:h + 1], rs, "bf16")
    assert bool(torch.isfinite(out).all())


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_paged_gqa_fp8_matches_oracle(d, G, page_size, num_splits):
    Hkv = 2
    _, k, v, lt = random_case(3, Hkv, 700, d, "bf16", lens=[700, 0, 333], seed=G + page_size + d,
                              nan_pad=False)
    q = torch.randn(3, G * Hkv, d, generator=torch.Generator().manual_seed(G + 1)).to(torch.bfloat16)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = _reference(q, k8, v8, ks, vs, G, lt)
    kp, table = to_paged_bytes(k8, page_size, seed=page_size)
    vp, _ = to_paged_bytes(v8, page_size, seed=page_size)
    out, lse = fd.decode_gqa_paged_fp8(q.to(DEV), kp.to(DEV), vp.to(DEV), ks.to(DEV), vs.to(DEV),
                                       table.to(DEV), lt.to(DEV), num_splits=num_splits,
                                       out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    # the same cache contiguous
    if G > 1:
        cout, clse = fd.decode_gqa_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV), lt.to(DEV),
                                       num_splits=num_splits, out_dtype=torch.float32)
        # the same kernel on the same chunks: at d = 128 the tcgen05 kernel
        # (128-token chunks) serves contiguous caches and pages of a
        # multiple of 128 tokens, the mma.sync kernel smaller pages
        if page_size % (128 if d == 128 else 32) == 0:
            assert torch.equal(out, cout) and torch.equal(lse, clse)


def test_paged_gqa_fp8_limits_and_bad_entries():
    _, k, v, lt = random_case(2, 2, 256, 128, "bf16", lens=[256, 256], seed=3, nan_pad=False)
    q = torch.randn(2, 16, 128).to(torch.bfloat16)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    kp, table = to_paged_bytes(k8, 32, seed=1)
    vp, _ = to_paged_bytes(v8, 32, seed=1)
    bad = table.clone()
    bad[1, 2] = 10 ** 6
    fd.decode_gqa_paged_fp8(q.to(DEV), kp.to(DEV), vp.to(DEV), ks.to(DEV), vs.to(DEV), bad.to(DEV), lt.to(DEV))
    assert fd.device_status(reset=True) == 7   # FD_ERR_BAD_PAGE, then cleared
    kp8, t8 = to_paged_bytes(k8, 8, seed=1)
    with pytest.raises(fd.FDError) as e:
        fd.decode_gqa_paged_fp8(q.to(DEV), kp8.to(DEV), kp8.to(DEV), ks.to(DEV), vs.to(DEV), t8.to(DEV),
                                lt.to(DEV))
    assert e.value.status == 2   # 8-token pages: FD_ERR_UNSUPPORTED
    assert fd.device_status() == 0


@pytest.mark.slow
def test_paged_gqa_fp8_full_size_equals_contiguous():
    """The 1 GiB GQA workload stored as E4M3 in shuffled 128-token pages:
    bit-identical to the contiguous E4M3 kernel (the same kernel and chunks)."""
    w = WORKLOADS["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"]
    q, k, v, lens = make_inputs(w, device="cuda")
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    del k, v
    cout, clse = fd.decode_gqa_fp8(q, k8, v8, ks, vs, lens, scale=w.scale, out_dtype=torch.float32)
    kp, table = to_paged_bytes(k8, 128, seed=5)
    vp, _ = to_paged_bytes(v8, 128, seed=5)
    del k8, v8
    out, lse = fd.decode_gqa_paged_fp8(q, kp, vp, ks, vs, table, lens, scale=w.scale, out_dtype=torch.float32)
    assert torch.equal(out, cout) and torch.equal(lse, clse)


@pytest.mark.slow
@pytest.mark.parametrize("name,page_size", [("decode_gqa_b8_hq16_hkv8_n32k_d256_bf16", 0),
                                            ("decode_gqa_b8_hq16_hkv8_n32k_d256_bf16", 16),
                                            ("decode_gqa_b16_hq64_hkv8_n32k_d64_bf16", 16),
                                            ("decode_gqa_b16_hq64_hkv8_n32k_d64_bf16", 64)])
def test_gqa_fp8_full_size_head_dims(name, page_size):
    """The 2 GiB head-dim-256 (G = 2) and 1 GiB head-dim-64 (G = 8) GQA
    workloads stored as E4M3, contiguous or in shuffled pages, automatic
    decomposition: sampled rows against the oracle; 64-token pages are
    bit-identical to the contiguous kernel (the same chunks)."""
    import numpy as np
    w = WORKLOADS[name]
    G = w.H // w.kv_heads
    q, k, v, lens = make_inputs(w, device="cuda")
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    del k, v
    cout, clse = fd.decode_gqa_fp8(q, k8, v8, ks, vs, lens, scale=w.scale, out_dtype=torch.float32)
    out, lse = cout, clse
    if page_size:
        kp, table = to_paged_bytes(k8, page_size, seed=5)
        vp, _ = to_paged_bytes(v8, page_size, seed=5)
        out, lse = fd.decode_gqa_paged_fp8(q, kp, vp, ks, vs, table, lens, scale=w.scale,
                                           out_dtype=torch.float32)
        del kp, vp
        if page_size % 32 == 0:
            assert torch.equal(out, cout) and torch.equal(lse, clse)
    rng = np.random.default_rng(13)
    for _ in range(8):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.H))
        kv = h // G
        ro, rs = oracle.attention_fp8(q[b:b + 1, h:h + 1].cpu(), k8[b:b + 1, kv:kv + 1].cpu(),
                                      v8[b:b + 1, kv:kv + 1].cpu(), ks[b:b + 1, kv:kv + 1].cpu(),
                                      vs[b:b + 1, kv:kv + 1].cpu(), scale=w.scale)
        check_out(out[b:b + 1, h:h + 1], ro, "bf16")
        check_lse(lse[b:b + 1, h:h + 1], rs, "bf16")
    assert bool(torch.isfinite(out).all())
    assert fd.device_status() == 0


@pytest.mark.parametrize("qdt", ["f32", "bf16"])
@pytest.mark.parametrize("d,page_size", [(64, 0), (128, 0), (256, 0), (64, 16), (128, 16), (128, 64),
                                         (256, 32)])
def test_gqa_fp8_q_beyond_f16_range(qdt, d, page_size):
    """q far outside f16's range (|q| up to ~1e6 > 65504), which the E4M3
    products take in f16: each head's q is brought into range by a power of
    two and its scores scaled back, so the result is the oracle's.  K is
    scaled down so that the scores stay moderate (the test is about q's
    range, not about scores of 1e6: with |q| ~ 1e6 and K ~ 1e-6 the scores
    have a standard deviation ~1, where the f16 rounding of q, 2^-12
    relative, stays within the tolerance)."""
    Hkv, G, B = 2, 8, 2
    _, k, v, lt = random_case(B, Hkv, 500, d, "bf16", lens=[500, 77], seed=3, nan_pad=False)
    g = torch.Generator().manual_seed(11)
    mag = torch.tensor([1.0, 3.0, 1e3, 7e4, 1e5, 3e5, 1e6, 2.5e5] * Hkv)   # per query head
    q = (torch.randn(B, G * Hkv, d, generator=g) * mag[None, :, None]).to(QT[qdt])
    assert float(q.float().abs().max()) > 65504
    k = (k.float() * 1e-6).to(torch.bfloat16)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = _reference(q, k8, v8, ks, vs, G, lt)
    args = (q.to(DEV), None, None, ks.to(DEV), vs.to(DEV))
    if page_size:
        kp, table = to_paged_bytes(k8, page_size, seed=page_size)
        vp, _ = to_paged_bytes(v8, page_size, seed=page_size)
        out, lse = fd.decode_gqa_paged_fp8(args[0], kp.to(DEV), vp.to(DEV), args[3], args[4], table.to(DEV),
                                           lt.to(DEV), out_dtype=torch.float32)
    else:
        out, lse = fd.decode_gqa_fp8(args[0], k8.to(DEV), v8.to(DEV), args[3], args[4], lt.to(DEV),
                                     out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    assert fd.device_status() == 0
