"""fd_decode_noalloc, the entry point for callers that cannot allocate device
memory (a serving engine whose memory pool owns the GPU, a runtime plugin
given only pointers and a stream): it must give fd_decode's results with
its scratch taken from the library's static device array.

Called through the C ABI directly and through the binding's
decode_noalloc.  This file is collected last so that a
run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process (it builds and loads the library
itself).
"""
import ctypes

import numpy as np
import pytest
import torch

import split_kv_fd_gb300 as fd
from split_kv_fd_gb300 import fd as fdmod
from split_kv_fd_gb300.inputs import random_case
from parity_util import OUT_TOL, LSE_TOL, to_np

pytestmark = pytest.mark.gpu

DT = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
FD_ERR_SCRATCH_TOO_SMALL = 6


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    lib = fdmod.load()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fd_decode_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, I, P, P]
    lib.fd_decode_noalloc.restype = I
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, q, k, v, lens, num_splits, out, lse):
    B, H, N, d = k.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fd_decode_noalloc(_p(q), _p(k), _p(v), _p(lens), B, H, N, d, DT[q.dtype],
                                 num_splits, float(d) ** -0.5, _p(out), DT[out.dtype], _p(lse),
                                 stream)


def _close(a, b, dtype_name):
    ga, gb = to_np(a), to_np(b)
    return np.max(np.abs(ga - gb)) <= OUT_TOL[dtype_name]


CASES = [
    # (B, H, N, d, dtype, lens, num_splits)
    (3, 8, 3000, 128, "bf16", "ragged", 0),
    (2, 4, 1000, 64, "f32", [1000, 377], 3),
    (1, 32, 20000, 128, "f16", None, 0),
]


def test_noalloc_matches_fd_decode_on_consecutive_calls(lib):
    dev = torch.device("cuda")
    results = []
    for B, H, N, d, dt, lens, ns in CASES:
        q, k, v, lt = (t.to(dev) for t in random_case(B, H, N, d, dt, lens=lens, seed=B + N))
        ref_out, ref_lse = fd.decode(q, k, v, lt, num_splits=ns, out_dtype=torch.float32)
        results.append(((q, k, v, lt, ns), ref_out, ref_lse, dt))
    # two calls in a row on each case, then the cases again interleaved: each
    # call must not depend on what the previous one left in the shared array
    order = [0, 0, 1, 1, 2, 2, 0, 2, 1]
    for i in order:
        (q, k, v, lt, ns), ref_out, ref_lse, dt = results[i]
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _noalloc(lib, q, k, v, lt, ns, out, lse)
        assert st == 0, fdmod.status_str(st)
        torch.cuda.synchronize()
        assert _close(out, ref_out, dt), f"case {i}: out differs from fd_decode"
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        assert float((lse[fin] - ref_lse[fin]).abs().max()) <= LSE_TOL[dt]
    assert fd.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    dev = torch.device("cuda")
    # B*H*P*(d+2)*4 bytes of partials is far above 1 MiB here
    B, H, N, d, P = 4, 64, 64, 128, 64
    q = torch.zeros(B, H, d, device=dev, dtype=torch.bfloat16)
    k = torch.zeros(B, H, N, d, device=dev, dtype=torch.bfloat16)
    out = torch.zeros(B, H, d, device=dev, dtype=torch.bfloat16)
    st = _noalloc(lib, q, k, k, None, P, out, None)
    assert st == FD_ERR_SCRATCH_TOO_SMALL
    assert "FD_NOALLOC_SCRATCH_BYTES" in fdmod.status_str(st)
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched


def _documented_need(B, H, N, d, num_splits, sms):
    """The scratch bytes the header documents for fd_decode_noalloc (each
    term rounded up to 256 bytes)."""
    r = lambda x: -(-x // 256) * 256  # noqa: E731
    if num_splits == 0 and B <= 1024:
        return r(2 * sms * d * 4) + r(2 * sms * 2 * 4) + r(4 * B * H)
    P = num_splits or fd.auto_num_splits(B, H, N, d, torch.bfloat16)
    return r(B * H * P * d * 4) + r(B * H * P * 2 * 4) + r(4 * B * H)


@pytest.mark.parametrize("B,H,N,num_splits", [(1024, 1, 64, 0), (1025, 1, 64, 0), (2048, 1, 64, 0),
                                              (2048, 1, 300, 0), (64, 4, 5000, 7)])
def test_noalloc_limit_is_the_documented_one(lib, B, H, N, num_splits):
    """Above B = 1024 the automatic mode switches to split counts, whose
    partials grow with B*H*P: the status follows the documented bound on
    either side of it, and a call within it matches fd_decode."""
    dev = torch.device("cuda")
    d = 128
    need = _documented_need(B, H, N, d, num_splits, fd.num_sms())
    q, k, v, lt = (t.to(dev) for t in random_case(B, H, N, d, "bf16", lens="ragged", seed=B + N))
    out = torch.zeros(B, H, d, device=dev, dtype=torch.float32)
    lse = torch.zeros(B, H, device=dev, dtype=torch.float32)
    st = _noalloc(lib, q, k, v, lt, num_splits, out, lse)
    if need > 1 << 20:
        assert st == FD_ERR_SCRATCH_TOO_SMALL, (need, fdmod.status_str(st))
        return
    assert st == 0, (need, fdmod.status_str(st))
    ref_out, ref_lse = fd.decode(q, k, v, lt, num_splits=num_splits, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert _close(out, ref_out, "bf16")
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), fin)
    assert float((lse[fin] - ref_lse[fin]).abs().max()) <= LSE_TOL["bf16"]


def test_binding_decode_noalloc_matches_oracle(lib):
    """The Python binding's decode_noalloc against the float64 oracle, and its
    error for a problem beyond the scratch."""
    import oracle
    from parity_util import check_lse, check_out
    dev = torch.device("cuda")
    q, k, v, lt = random_case(3, 8, 2500, 128, "bf16", lens=[2500, 1, 0], seed=77)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    out, lse = fd.decode_noalloc(q.to(dev), k.to(dev), v.to(dev), lt.to(dev), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    qb = torch.zeros(4, 64, 128, device=dev, dtype=torch.bfloat16)
    kb = torch.zeros(4, 64, 64, 128, device=dev, dtype=torch.bfloat16)
    with pytest.raises(fd.FDError) as e:
        fd.decode_noalloc(qb, kb, kb, num_splits=64)
    assert e.value.status == FD_ERR_SCRATCH_TOO_SMALL
