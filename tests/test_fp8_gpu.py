"""FP8 (E4M3) KV cache on the GPU: fd_decode_fp8 against the float64 FP8
oracle, which reads the same bytes and scales.  Tolerances as for 16-bit
inputs (2e-3 on out, 1e-3 on lse; float32 accumulation)."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import make_inputs, quantize_e4m3, random_case
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


@pytest.mark.parametrize("qdt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_fp8_matches_oracle(qdt, d, num_splits):
    q, k, v, lt = random_case(3, 4, 900, d, "f32", lens=[900, 0, 333], seed=d + num_splits,
                              k_scale=3.0)
    q = q.to({"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[qdt])
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    ref_out, ref_lse = oracle.attention_fp8(q, k8, v8, ks, vs, lens=lt)
    dev = torch.device("cuda")
    out, lse = fd.decode_fp8(q.to(dev), k8.to(dev), v8.to(dev), ks.to(dev), vs.to(dev),
                             seqlens=lt.to(dev), num_splits=num_splits, out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    # the bf16 output carries its own final rounding on top
    out16, _ = fd.decode_fp8(q.to(dev), k8.to(dev), v8.to(dev), ks.to(dev), vs.to(dev),
                             seqlens=lt.to(dev), num_splits=num_splits, out_dtype=torch.bfloat16)
    check_out(out16, ref_out, "bf16")


def test_fp8_full_size_sampled():
    """The benchmark workload stored in E4M3 (2 GiB of K/V), sampled rows."""
    w = WORKLOADS["decode_b8_h32_n32k_d128_bf16"]
    q, k, v, lens = make_inputs(w, device="cuda")
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    del k, v
    torch.cuda.empty_cache()
    out, lse = fd.decode_fp8(q, k8, v8, ks, vs, seqlens=lens, scale=w.scale, out_dtype=torch.float32)
    rows = [(0, 0), (3, 17), (7, 31), (5, 2)]
    for b, h in rows:
        ro, rl = oracle.attention_fp8(q[b:b + 1, h:h + 1].cpu(), k8[b:b + 1, h:h + 1].cpu(),
                                      v8[b:b + 1, h:h + 1].cpu(), ks[b:b + 1, h:h + 1].cpu(),
                                      vs[b:b + 1, h:h + 1].cpu(), scale=w.scale)
        check_out(out[b:b + 1, h:h + 1], ro, "bf16")
        check_lse(lse[b:b + 1, h:h + 1], rl, "bf16")
    assert bool(torch.isfinite(out).all())
