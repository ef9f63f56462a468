"""Parity on the five named workloads, in the launch configuration the
benchmark times (fused decode, automatic decomposition, default stream).

All five are compared element by element, on every (b, h) row, with the
float64 oracle: the two small workloads through every path and both output
dtypes, the three large ones (2-16 GiB of KV) through the fused call (the
benchmarked configuration) and the two-call path with both merges.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import make_inputs
from split_kv_fd_gb300.workloads import WORKLOADS
from parity_util import check_lse, check_out, to_np

pytestmark = pytest.mark.gpu

OUT_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["decode_b1_h1_n1k_d64_f32_p4", "decode_b1_h8_n4k_d128_f16_p4"])
def test_small_workloads_elementwise(name):
    w = WORKLOADS[name]
    q, k, v, lens = make_inputs(w, device="cuda")
    qc, kc, vc, lc = (t.cpu() for t in (q, k, v, lens))
    ref_out, ref_lse = oracle.attention(qc, kc, vc, lens=lc, scale=w.scale)
    # fused, the workload's split count, its own output dtype and float32
    for odt in {OUT_DT[w.out_dtype], torch.float32}:
        out, lse = fd.decode(q, k, v, lens, num_splits=w.num_splits, scale=w.scale, out_dtype=odt)
        eo = check_out(out, ref_out, w.dtype)
        el = check_lse(lse, ref_lse, w.dtype)
        print(f"PARITY {name} fused_P{w.num_splits}_{str(odt)[6:]} all elements "
              f"max_err_out={eo:.3e} max_err_lse={el:.3e}")
    # automatic decomposition
    out, lse = fd.decode(q, k, v, lens, scale=w.scale, out_dtype=torch.float32)
    check_out(out, ref_out, w.dtype)
    check_lse(lse, ref_lse, w.dtype)
    # two-call path, both merges, against the oracle's per-split partials too
    o, m, l, s = fd.decode_split(q, k, v, w.num_splits, seqlens=lens, scale=w.scale)
    ro, rm, rl, rs = oracle.split_partials(qc, kc, vc, w.num_splits, lens=lc, scale=w.scale)
    assert np.max(np.abs(to_np(o) - ro)) <= (1e-5 if w.dtype == "f32" else 2e-3)
    assert np.max(np.abs(to_np(s) - rs)) <= (1e-5 if w.dtype == "f32" else 1e-3)
    for out, lse in (fd.combine_mlo(o, m, l, out_dtype=OUT_DT[w.out_dtype]),
                     fd.combine_lse(o, s, out_dtype=OUT_DT[w.out_dtype])):
        check_out(out, ref_out, w.dtype)
        check_lse(lse, ref_lse, w.dtype)


def _oracle_all_rows(w, q, k, v, lens):
    """The oracle over every (b, h) row of a full-size workload.

    The K/V bits are copied to the host as they are (padding included; the
    oracle reads only the first lens[b] rows) and the float64 C oracle runs
    threaded over all rows.
    """
    return oracle.attention(q.cpu(), k.cpu(), v.cpu(), lens=lens.cpu(), scale=w.scale)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_b8_h32_n32k_d128_bf16", "decode_b1_h32_n128k_d128_bf16_k8",
                                  "decode_ragged_b16_h32_n64k_d128_bf16"])
def test_large_workloads_every_row(name):
    """Every element of every (b, h) row against the float64 oracle.

    Split + merge equals unsplit attention on every row ("FlashDecoding 数学
    推导" §2.6, "...传统 m/l/o 方法与 LSE 方法" §2.3.6), whatever the
    decomposition cuts; so each path below is compared with the oracle
    directly, never with another CUDA path.
    """
    w = WORKLOADS[name]
    q, k, v, lens = make_inputs(w, device="cuda")
    ref_out, ref_lse = _oracle_all_rows(w, q, k, v, lens)
    rows = w.B * w.H

    results = {}
    # the benchmarked configuration: fused, automatic decomposition, the
    # workload's own output dtype; then the strict bound with a float32 output
    results[f"fused_auto_{w.out_dtype}"] = fd.decode(q, k, v, lens, scale=w.scale,
                                                     out_dtype=OUT_DT[w.out_dtype])
    results["fused_auto_f32"] = fd.decode(q, k, v, lens, scale=w.scale, out_dtype=torch.float32)
    # the two-call path with both merges, each with both output dtypes
    P = fd.auto_num_splits(w.B, w.H, w.N, w.d)
    o, m, l, s = fd.decode_split(q, k, v, P, seqlens=lens, scale=w.scale)
    for odt in (w.out_dtype, "f32"):
        results[f"split{P}_mlo_{odt}"] = fd.combine_mlo(o, m, l, out_dtype=OUT_DT[odt])
        results[f"split{P}_lse_{odt}"] = fd.combine_lse(o, s, out_dtype=OUT_DT[odt])
    del o, m, l, s
    for key, (out, lse) in results.items():
        eo = check_out(out, ref_out, w.dtype, what=f"{key} out")
        el = check_lse(lse, ref_lse, w.dtype, what=f"{key} lse")
        print(f"PARITY {name} {key} rows={rows}/{rows} all elements "
              f"max_err_out={eo:.3e} max_err_lse={el:.3e}")
    del q, k, v, results
    _free()
