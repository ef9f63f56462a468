"""A seeded sweep of random shapes through every decode entry point against
the float64 oracle: batch, heads, group size (1 to 40), head dim (64, 128,
256), K/V dtype, page size, split count and ragged lengths (empty ones
included) drawn per case, so the combinations the targeted tests do not
name get exercised too.  Each case is small enough for the oracle to run in
well under a second."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import quantize_e4m3, random_case, to_paged, to_paged_bytes
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
TD = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _draw(seed):
    r = np.random.default_rng(seed)
    d = int(r.choice([64, 128, 256]))
    kind = str(r.choice(["mha", "paged", "fp8", "gqa", "gqa_paged", "gqa_fp8", "gqa_paged_fp8"]))
    if kind == "gqa_fp8":
        d = int(r.choice([64, 128]))
    elif kind == "gqa_paged_fp8":
        d = 128
    dtype = str(r.choice(["f16", "bf16"] if (kind.startswith("gqa") or d == 256) else ["f32", "f16", "bf16"]))
    if kind == "fp8":
        dtype = str(r.choice(["f16", "bf16"]))
    B = int(r.integers(1, 6))
    Hkv = int(r.integers(1, 5))
    G = int(r.choice([1, 2, 3, 5, 8, 12, 16, 20, 40])) if kind.startswith("gqa") else 1
    N = int(r.integers(1, 1500))
    lens = [int(x) for x in r.integers(0, N + 1, size=B)]
    if r.random() < 0.5:
        lens[int(r.integers(B))] = N
    num_splits = int(r.choice([0, 0, 1, 2, 7, 33]))
    page = 0
    if kind == "paged":
        page = int(r.choice([1, 7, 16, 64, 200]))
    elif kind in ("gqa_paged", "gqa_paged_fp8"):
        page = int(r.choice([16, 32, 64, 96]))
    return dict(d=d, kind=kind, dtype=dtype, B=B, Hkv=Hkv, G=G, N=N, lens=lens, num_splits=num_splits,
                page=page)


@pytest.mark.parametrize("seed", range(100))
def test_random_case(seed):
    c = _draw(1000 + seed)
    B, Hkv, G, N, d, dtype = c["B"], c["Hkv"], c["G"], c["N"], c["d"], c["dtype"]
    kind, ns = c["kind"], c["num_splits"]
    _, k, v, lt = random_case(B, Hkv, N, d, dtype, lens=c["lens"], seed=seed)
    q = torch.randn(B, Hkv * G, d, generator=torch.Generator().manual_seed(seed + 7)).to(TD[dtype])
    ld = lt.to(DEV)
    if kind in ("fp8", "gqa_fp8", "gqa_paged_fp8"):
        k8, ks = quantize_e4m3(k.nan_to_num(0.0))
        v8, vs = quantize_e4m3(v.nan_to_num(0.0))
        rep = lambda x: x.repeat_interleave(G, dim=1)   # noqa: E731  query head h reads K/V head h / G
        ref_out, ref_lse = oracle.attention_fp8(q, rep(k8), rep(v8), rep(ks), rep(vs), lens=lt)
        args = (ks.to(DEV), vs.to(DEV))
        if kind == "fp8":
            out, lse = fd.decode_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), *args, ld, num_splits=ns,
                                     out_dtype=torch.float32)
        elif kind == "gqa_fp8":
            out, lse = fd.decode_gqa_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), *args, ld, num_splits=ns,
                                         out_dtype=torch.float32)
        else:
            kp, table = to_paged_bytes(k8, c["page"], seed=seed)
            vp, _ = to_paged_bytes(v8, c["page"], seed=seed)
            out, lse = fd.decode_gqa_paged_fp8(q.to(DEV), kp.to(DEV), vp.to(DEV), *args, table.to(DEV), ld,
                                               num_splits=ns, out_dtype=torch.float32)
    elif kind in ("gqa", "gqa_paged"):
        ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=lt)
        if kind == "gqa":
            out, lse = fd.decode_gqa(q.to(DEV), k.to(DEV), v.to(DEV), ld, num_splits=ns,
                                     out_dtype=torch.float32)
        else:
            kp, vp, table = to_paged(k, v, c["page"], seed=seed)
            out, lse = fd.decode_gqa_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), ld,
                                           num_splits=ns, out_dtype=torch.float32)
    elif kind == "paged":
        kp, vp, table = to_paged(k, v, c["page"], seed=seed)
        ref_out, ref_lse = oracle.attention_paged(q, kp, vp, table, lt)
        out, lse = fd.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), ld, num_splits=ns,
                                   out_dtype=torch.float32)
    else:
        ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
        out, lse = fd.decode(q.to(DEV), k.to(DEV), v.to(DEV), ld, num_splits=ns, out_dtype=torch.float32)
    what = f"seed {seed}: {c}"
    check_out(out, ref_out, dtype, what=what)
    check_lse(lse, ref_lse, dtype, what=what)
