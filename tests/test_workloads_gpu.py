"""Parity on the five named workloads, in the launch configuration the
benchmark times (fused decode, automatic decomposition, default stream).

The two small workloads are compared element by element with the oracle.
The three large ones (2-16 GiB of KV) are compared on a seeded sample of
(b, h) rows, which the oracle computes one by one, and on properties that
hold at any size: every output is finite, every output element lies within
the range of its V column (a softmax average is a convex combination), and
the fused path agrees with the two-call path on every row.
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


def _sample_rows(w, lens, n=12, seed=0):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (w.B - 1, w.H - 1)}
    if w.ragged:  # the shortest and the longest sequence
        lo, hi = int(np.argmin(lens)), int(np.argmax(lens))
        rows |= {(lo, 0), (hi, w.H - 1)}
    while len(rows) < n:
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.H))))
    return sorted(rows)


def _oracle_rows(w, q, k, v, lens, rows):
    """Oracle on the sampled rows only (each row copied to the host)."""
    outs, lses = [], []
    for b, h in rows:
        n = int(lens[b])
        qs = q[b:b + 1, h:h + 1].cpu()
        ks = k[b:b + 1, h:h + 1, :n].cpu()
        vs = v[b:b + 1, h:h + 1, :n].cpu()
        o, s = oracle.attention(qs, ks, vs, scale=w.scale)
        outs.append(o[0, 0])
        lses.append(s[0, 0])
    return np.stack(outs), np.array(lses)


def _convex_bounds_ok(v, lens, out):
    """Each output element lies within [min_j V_j, max_j V_j] of its column."""
    for b in range(v.shape[0]):
        n = int(lens[b])
        vb = v[b, :, :n].float()
        lo = vb.amin(dim=1) - 1e-3
        hi = vb.amax(dim=1) + 1e-3
        ob = out[b].float()
        assert bool(torch.all(ob >= lo)) and bool(torch.all(ob <= hi)), f"row {b} outside hull"
        del vb


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_b8_h32_n32k_d128_bf16", "decode_b1_h32_n128k_d128_bf16_k8",
                                  "decode_ragged_b16_h32_n64k_d128_bf16"])
def test_large_workloads_sampled(name):
    w = WORKLOADS[name]
    q, k, v, lens = make_inputs(w, device="cuda")
    lens_h = lens.cpu().numpy()
    rows = _sample_rows(w, lens_h)
    ref_out, ref_lse = _oracle_rows(w, q, k, v, lens_h, rows)
    bi = torch.tensor([r[0] for r in rows])
    hi = torch.tensor([r[1] for r in rows])

    results = {}
    # the benchmarked configuration: fused, automatic decomposition
    out, lse = fd.decode(q, k, v, lens, scale=w.scale, out_dtype=OUT_DT[w.out_dtype])
    results["fused_auto"] = (out, lse)
    out32, lse32 = fd.decode(q, k, v, lens, scale=w.scale, out_dtype=torch.float32)
    results["fused_auto_f32"] = (out32, lse32)
    # the two-call path with both merges
    P = fd.auto_num_splits(w.B, w.H, w.N, w.d)
    o, m, l, s = fd.decode_split(q, k, v, P, seqlens=lens, scale=w.scale)
    results["split_mlo"] = fd.combine_mlo(o, m, l, out_dtype=torch.float32)
    results["split_lse"] = fd.combine_lse(o, s, out_dtype=torch.float32)
    del o, m, l, s
    for key, (out, lse) in results.items():
        so = out[bi, hi]
        sl = lse[bi, hi]
        eo = check_out(so, ref_out, w.dtype, what=f"{key} out")
        el = check_lse(sl, ref_lse, w.dtype, what=f"{key} lse")
        print(f"PARITY {name} {key} rows={len(rows)} max_err_out={eo:.3e} max_err_lse={el:.3e}")
        assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all()), key
    # properties over every row
    _convex_bounds_ok(v, lens_h, results["fused_auto_f32"][0])
    a, b = results["fused_auto_f32"][0], results["split_mlo"][0]
    assert float((a - b).abs().max()) <= 2e-3
    del q, k, v
    _free()
