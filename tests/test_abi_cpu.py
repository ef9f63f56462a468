"""The C-ABI library without a GPU: it loads, exports every symbol that
include/fd.h declares, and rejects bad arguments on the host before any
CUDA call.  Also checks the seeded input generator (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import split_kv_fd_gb300 as fd
from split_kv_fd_gb300 import fd as fdmod
from split_kv_fd_gb300.inputs import make_inputs, random_case
from split_kv_fd_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F32, F16, BF16, E4M3 = 0, 1, 2, 3   # fd_dtype


@pytest.fixture(scope="module")
def lib():
    return fdmod.load(build_if_missing=True)


def _declared():
    src = open(os.path.join(ROOT, "include", "fd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert set(names) == set(fdmod.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.fd_version() >= 100


def test_status_strings(lib):
    for code, name in fdmod.STATUS_NAMES.items():
        assert lib.fd_status_str(code).decode().startswith(name)
    assert lib.fd_status_str(99).decode() == "FD_UNKNOWN_STATUS"


def test_host_rejects_bad_arguments_without_cuda(lib):
    P = ctypes.c_void_p
    dummy = P(4096)  # aligned, never dereferenced: the checks fail first
    # negative sizes
    assert lib.fd_decode(dummy, dummy, dummy, None, -1, 1, 8, 128, 2, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 1
    # unsupported head dim / dtype (256 needs 16-bit or E4M3 K/V)
    assert lib.fd_decode(dummy, dummy, dummy, None, 1, 1, 8, 96, 2, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 2
    assert lib.fd_decode(dummy, dummy, dummy, None, 1, 1, 8, 256, 0, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 2
    assert lib.fd_decode(dummy, dummy, dummy, None, 1, 1, 8, 512, 2, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 2
    assert lib.fd_decode(dummy, dummy, dummy, None, 1, 1, 8, 128, 7, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 2
    # null and misaligned pointers
    assert lib.fd_decode(None, dummy, dummy, None, 1, 1, 8, 128, 2, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 1
    assert lib.fd_decode(dummy, P(4098), dummy, None, 1, 1, 8, 128, 2, 0, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 1
    # negative split count; split path needs >= 1
    assert lib.fd_decode(dummy, dummy, dummy, None, 1, 1, 8, 128, 2, -1, 1.0, dummy, 2, None,
                         dummy, 1 << 20, None) == 1
    assert lib.fd_decode_split(dummy, dummy, dummy, None, 1, 1, 8, 128, 2, 0, 1.0, dummy, dummy,
                               dummy, None, None) == 1
    # combine: P out of range, unsupported d
    assert lib.fd_combine_mlo(dummy, dummy, dummy, 1, 1, 0, 128, dummy, 0, None, None) == 1
    assert lib.fd_combine_lse(dummy, dummy, 1, 1, 4, 80, dummy, 0, None, None) == 2
    # an empty problem is a no-op
    assert lib.fd_decode(None, None, None, None, 0, 4, 8, 128, 2, 0, 1.0, None, 2, None,
                         None, 0, None) == 0


def _fill(bh, P, G):
    items = bh * P
    return items / (G * -(-items // G))


def test_auto_num_splits_rule(lib):
    # >= 4 work items per SM, never splits under 256 tokens, >= 1; among
    # counts up to 4x that minimum, the best fill of the last wave of CTAs
    assert lib.fd_auto_num_splits(8, 32, 32768, 128, BF16, 152) == 7      # 1792 items: 11.8 per CTA
    assert lib.fd_auto_num_splits(16, 32, 65536, 128, BF16, 152) == 5     # 2560 items: 16.8 per CTA
    assert lib.fd_auto_num_splits(1, 32, 131072, 128, BF16, 152) == 19    # 608 items: exactly 4 per CTA
    assert lib.fd_auto_num_splits(1, 1, 1024, 64, F32, 152) == 4
    assert lib.fd_auto_num_splits(1, 1, 100, 64, F32, 152) == 1
    assert lib.fd_auto_num_splits(0, 1, 100, 64, F32, 152) == 1
    assert lib.fd_auto_num_splits(1, 1, 100, 64, F32, 0) == -1
    assert lib.fd_auto_num_splits(1, 1, 100, 64, 9, 152) == -1       # unknown storage type
    # the same rule for every storage type (fd_workspace_size takes none)
    for dt in (F32, F16, BF16, E4M3):
        assert lib.fd_auto_num_splits(8, 32, 32768, 128, dt, 152) == 7
    # the chosen count never fills worse than the minimum one, nor splits
    # below 256 tokens
    for B, H, N in [(8, 32, 32768), (3, 7, 50000), (2, 8, 32768), (64, 8, 4096), (1, 5, 9000)]:
        bh = B * H
        lo = max(1, min(-(-4 * 152 // bh), max(1, N // 256)))
        P = lib.fd_auto_num_splits(B, H, N, 128, BF16, 152)
        assert lo <= P <= max(lo, 4 * lo)
        assert P == 1 or N // P >= 256
        assert _fill(bh, P, 152) >= _fill(bh, lo, 152)


def test_input_generator_is_seeded_and_pads_with_nan():
    w = WORKLOADS["decode_b1_h1_n1k_d64_f32_p4"]
    a = make_inputs(w)
    b = make_inputs(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q, k, v, lens = random_case(3, 2, 50, 64, "bf16", lens=[50, 7, 0], seed=1)
    assert lens.tolist() == [50, 7, 0]
    assert torch.isnan(k[1, :, 7:].float()).all() and torch.isfinite(k[1, :, :7].float()).all()
    assert torch.isnan(v[2].float()).all() and torch.isfinite(k[0].float()).all()
    # K draws scaled by k_scale
    w4 = WORKLOADS["decode_b1_h32_n128k_d128_bf16_k8"]
    assert w4.k_scale == 8.0 and w4.scale == pytest.approx(1 / np.sqrt(128))


def test_binding_refuses_cpu_tensors():
    q = torch.zeros(1, 1, 64)
    k = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        fd.decode(q, k, k)


def test_library_has_no_unresolved_symbols_of_its_own():
    """Every undefined dynamic symbol comes from another library (versioned,
    e.g. libcudart's or libc's) or is weak: a symbol of this library that the
    link left undefined would only fail when the library is loaded."""
    import shutil
    import subprocess
    from split_kv_fd_gb300 import _build_lib as bl
    if not shutil.which("nm"):
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--undefined-only", bl.LIB], capture_output=True, text=True,
                         check=True).stdout.split("\n")
    own = [l.split()[-1] for l in out if l.strip() and l.split()[0] == "U" and "@" not in l]
    assert own == [], own


def test_other_entry_points_reject_bad_arguments_without_cuda(lib):
    """GQA, FP8, paged, no-alloc and merge entry points check their arguments
    on the host before any CUDA call (1 = invalid, 2 = unsupported, 0 = an
    empty problem, nothing launched)."""
    P = ctypes.c_void_p
    dm = P(4096)
    MB = 1 << 20

    def gqa(B, Hq, Hkv, N, d, dt=2, q=dm, ns=0):
        return lib.fd_decode_gqa(q, dm, dm, None, B, Hq, Hkv, N, d, dt, ns, 1.0, dm, 2, None, dm,
                                 MB, None)
    assert gqa(1, 6, 4, 64, 128) == 1            # Hq not a multiple of Hkv
    assert gqa(1, 8, 0, 64, 128) == 1            # no K/V heads
    assert gqa(1, 16, 2, 64, 128, dt=0) == 2     # G > 1 needs 16-bit K/V
    assert gqa(1, 16, 2, 64, 96) == 2            # head dim
    assert gqa(1, 8, 8, 64, 96) == 2             # G = 1 goes to fd_decode's checks
    # 2^31 K/V rows in all is no limit (copies address (row in block, block)):
    # only the null q is refused here
    assert gqa(1, 16, 2, 1 << 30, 128, q=None) == 1
    assert gqa(1, 16, 2, 64, 128, q=None) == 1
    assert gqa(1, 16, 2, 64, 128, ns=-2) == 1
    assert gqa(0, 16, 2, 64, 128, q=None) == 0   # empty

    def fp8(B=1, H=2, N=64, d=128, qdt=2, ks=dm, q=dm):
        return lib.fd_decode_fp8(q, qdt, dm, dm, ks, dm, None, B, H, N, d, 0, 1.0, dm, 2, None, dm,
                                 MB, None)
    assert fp8(ks=None) == 1                     # scales are required
    assert fp8(qdt=3) == 2                       # q stays 16/32-bit
    assert fp8(d=80) == 2
    assert fp8(q=P(4100)) == 1                   # misaligned q
    assert fp8(B=0, q=None, ks=None) == 0

    def paged(B=1, H=2, d=128, ps=16, mp=4, npg=8, lens=dm, table=dm):
        return lib.fd_decode_paged(dm, dm, dm, table, lens, B, H, d, ps, mp, npg, 2, 0, 1.0, dm, 2,
                                   None, dm, MB, None)
    assert paged(ps=0) == 1                      # page size >= 1
    assert paged(ps=1 << 16, mp=1 << 16) == 1    # pages x size beyond int32 tokens
    assert paged(mp=-1) == 1
    assert paged(lens=None) == 1                 # lengths are required
    assert paged(npg=0) == 1                     # a table needs pages to name
    assert paged(table=P(4098)) == 1             # misaligned block table
    assert paged(d=72) == 2
    assert paged(B=0, lens=None, table=None) == 0

    def noalloc(B=1, H=2, N=64, d=128, q=dm, dt=2):
        return lib.fd_decode_noalloc(q, dm, dm, None, B, H, N, d, dt, 0, 1.0, dm, 2, None, None)
    assert noalloc(d=96) == 2
    assert noalloc(dt=3) == 2                    # E4M3 K/V has its own entry point
    assert noalloc(q=None) == 1
    assert noalloc(B=0, q=None) == 0

    def merge(rows=4, d=128, oa=dm):
        return lib.fd_merge_lse(oa, dm, dm, dm, rows, d, dm, dm, None)
    assert merge(rows=-1) == 1
    assert merge(d=6) == 1                       # d a multiple of 4
    assert merge(oa=None) == 1
    assert merge(oa=P(4104)) == 1                # o rows 16-byte aligned
    assert merge(rows=0, oa=None) == 0

    def gqa_paged(B=1, Hq=16, Hkv=2, d=128, ps=64, mp=4, npg=8, dt=2, lens=dm, table=dm):
        return lib.fd_decode_gqa_paged(dm, dm, dm, table, lens, B, Hq, Hkv, d, ps, mp, npg, dt, 0, 1.0,
                                       dm, 2, None, dm, MB, None)
    assert gqa_paged(Hq=6, Hkv=4) == 1            # Hq not a multiple of Hkv
    assert gqa_paged(ps=0) == 1
    assert gqa_paged(ps=8) == 2                   # pages of 16 or a multiple of 32 tokens
    assert gqa_paged(ps=48) == 2
    assert gqa_paged(dt=0) == 2                   # 16-bit K/V only
    assert gqa_paged(npg=1 << 28, Hkv=8) == 2     # 2^31 (page, K/V head) blocks: past 32-bit coordinates
    # a serving-size pool (2^20 pages x 8 heads x 256 tokens = 2^31 rows) is
    # accepted: only the missing lengths are refused here
    assert gqa_paged(npg=1 << 20, Hkv=8, ps=256, lens=None) == 1
    assert gqa_paged(lens=None) == 1
    assert gqa_paged(npg=0) == 1
    assert gqa_paged(table=P(4098)) == 1
    assert gqa_paged(Hq=2, d=96) == 2             # G = 1 goes to fd_decode_paged's checks
    assert gqa_paged(B=0, lens=None, table=None) == 0

    def gqa_fp8(B=1, Hq=16, Hkv=2, N=64, d=128, qdt=2, ks=dm, q=dm):
        return lib.fd_decode_gqa_fp8(q, qdt, dm, dm, ks, dm, None, B, Hq, Hkv, N, d, 0, 1.0, dm, 2, None, dm,
                                     MB, None)
    assert gqa_fp8(Hq=6, Hkv=4) == 1             # Hq not a multiple of Hkv
    assert gqa_fp8(ks=None) == 1                 # scales are required
    assert gqa_fp8(d=96) == 2                    # head dims 64, 128 and 256
    assert gqa_fp8(qdt=3) == 2                   # q stays 16/32-bit
    assert gqa_fp8(q=P(4100)) == 1
    assert gqa_fp8(B=0, q=None, ks=None) == 0

    def gqa_paged_fp8(B=1, Hq=16, Hkv=2, d=128, ps=64, npg=8, ks=dm):
        return lib.fd_decode_gqa_paged_fp8(dm, 2, dm, dm, ks, dm, dm, dm, B, Hq, Hkv, d, ps, 4, npg, 0, 1.0, dm,
                                           2, None, dm, MB, None)
    assert gqa_paged_fp8(d=96) == 2              # paged E4M3: d 64, 128 or 256
    assert gqa_paged_fp8(ps=48) == 2
    assert gqa_paged_fp8(ks=None) == 1
    assert gqa_paged_fp8(Hq=6, Hkv=4) == 1
    assert gqa_paged_fp8(B=0) == 0
    assert gqa_paged_fp8(npg=1 << 28, Hkv=8) == 2   # 2^31 (page, K/V head) blocks
    assert gqa_paged_fp8(npg=1 << 20, Hkv=8, ps=256, ks=None) == 1

    assert lib.fd_workspace_size_gqa(1, 6, 4, 64, 128, 0) == 0
    assert lib.fd_combine_mlo(dm, dm, dm, 1, 1, 4, 80, dm, 0, None, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the answer without a GPU")
def test_valid_call_without_a_gpu_reports_a_cuda_error(lib):
    """Arguments that pass every host check reach the first CUDA call, which
    fails without a device: the call returns FD_ERR_CUDA and launches nothing."""
    P = ctypes.c_void_p
    dm = P(4096)
    assert lib.fd_decode(dm, dm, dm, None, 1, 1, 8, 128, 2, 0, 1.0, dm, 2, None, P(1 << 20),
                         1 << 20, None) == 4
    # caches of 2^31 rows and more pass every host check of the grouped-query
    # entry points (contiguous, and a 2^20-page pool of 256-token pages)
    assert lib.fd_decode_gqa(dm, dm, dm, None, 2, 16, 2, 1 << 30, 128, 2, 0, 1.0, dm, 2, None,
                             P(1 << 20), 1 << 20, None) == 4
    assert lib.fd_decode_gqa_paged(dm, dm, dm, dm, dm, 1, 16, 8, 128, 256, 4, 1 << 20, 2, 0, 1.0, dm, 2,
                                   None, P(1 << 20), 1 << 20, None) == 4
    assert lib.fd_decode_gqa_paged_fp8(dm, 2, dm, dm, dm, dm, dm, dm, 1, 16, 8, 128, 256, 4, 1 << 20, 0,
                                       1.0, dm, 2, None, P(1 << 20), 1 << 20, None) == 4
    # E4M3 grouped-query decode at head dims 64 and 256, paged (16-token
    # pages) and contiguous
    for d in (64, 256):
        assert lib.fd_decode_gqa_paged_fp8(dm, 2, dm, dm, dm, dm, dm, dm, 1, 16, 2, d, 16, 4, 8, 0, 1.0, dm, 2,
                                           None, P(1 << 20), 1 << 20, None) == 4
        assert lib.fd_decode_gqa_fp8(dm, 2, dm, dm, dm, dm, None, 1, 16, 2, 64, d, 0, 1.0, dm, 2, None,
                                     P(1 << 20), 1 << 20, None) == 4
    assert lib.fd_num_sms() <= 0
