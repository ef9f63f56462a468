"""The entry points inside CUDA graphs, as a serving loop runs them: each call
is captured once on a side stream (the counter clear becomes a memset node,
the kernel a kernel node), then the graph is replayed after new inputs, new
lengths or a new block table were written into the captured buffers, and
every replay is compared with the float64 oracle on those inputs."""
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import random_case, to_paged
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


def _capture(call):
    """Run `call(stream)` once eagerly on a side stream, then capture it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("num_splits", [0, 3])
def test_decode_graph_replays_on_new_inputs(num_splits):
    B, H, N, d = 4, 8, 3000, 128
    q, k, v, lt = random_case(B, H, N, d, "bf16", lens=[3000, 1, 0, 1234], seed=61)
    qd, kd, vd, ld = (t.to(DEV) for t in (q, k, v, lt))
    out = torch.empty(B, H, d, device=DEV)
    lse = torch.empty(B, H, device=DEV)
    ws = fd.new_workspace(B, H, N, d, num_splits, device=DEV)
    g = _capture(lambda s: fd.decode(qd, kd, vd, ld, num_splits=num_splits, out=out, lse=lse,
                                     workspace=ws, stream=s))
    for seed, lens in ((62, [17, 3000, 2999, 0]), (63, [3000, 3000, 64, 5])):
        q2, k2, v2, l2 = random_case(B, H, N, d, "bf16", lens=lens, seed=seed)
        qd.copy_(q2)
        kd.copy_(k2)
        vd.copy_(v2)
        ld.copy_(l2)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.attention(q2, k2, v2, lens=l2)
        check_out(out, ref_out, "bf16")
        check_lse(lse, ref_lse, "bf16")


def test_paged_gqa_graph_replays_on_a_new_block_table():
    """GQA (G = 4) over 16-token pages: the replay reads whatever table and
    lengths the buffers hold, so a serving loop can remap pages between
    steps without capturing again."""
    B, Hkv, G, N, d = 3, 2, 4, 640, 128
    # every row is real data: the replays change the lengths
    _, k, v, lt = random_case(B, Hkv, N, d, "bf16", lens=[640, 333, 0], seed=71, nan_pad=False)
    q = torch.randn(B, G * Hkv, d, generator=torch.Generator().manual_seed(72)).to(torch.bfloat16)
    kp, vp, table = to_paged(k, v, 16, seed=1)
    qd, ld = q.to(DEV), lt.to(DEV)
    kpd, vpd, td = kp.to(DEV), vp.to(DEV), table.to(DEV)
    out = torch.empty(B, G * Hkv, d, device=DEV)
    lse = torch.empty(B, G * Hkv, device=DEV)
    ws = torch.empty(max(256, fd.workspace_size_gqa(B, G * Hkv, Hkv, N, d)), dtype=torch.uint8, device=DEV)
    g = _capture(lambda s: fd.decode_gqa_paged(qd, kpd, vpd, td, ld, out=out, lse=lse, workspace=ws,
                                               stream=s))
    for seed, lens in ((2, [640, 333, 0]), (3, [1, 640, 500])):
        # the same contiguous rows laid out in another page order
        kp2, vp2, table2 = to_paged(k, v, 16, seed=seed)
        kpd.copy_(kp2)
        vpd.copy_(vp2)
        td.copy_(table2)
        ld.copy_(torch.tensor(lens, dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.attention_gqa(q, k, v, lens=torch.tensor(lens, dtype=torch.int32))
        check_out(out, ref_out, "bf16")
        check_lse(lse, ref_lse, "bf16")


def test_split_and_combine_graph():
    """The two-kernel form, both launches in one graph."""
    B, H, N, d, P = 2, 4, 2000, 64, 5
    q, k, v, lt = random_case(B, H, N, d, "f16", lens=[2000, 777], seed=81)
    qd, kd, vd, ld = (t.to(DEV) for t in (q, k, v, lt))
    o_p = torch.empty(B, H, P, d, device=DEV)
    m_p = torch.empty(B, H, P, device=DEV)
    l_p = torch.empty(B, H, P, device=DEV)
    s_p = torch.empty(B, H, P, device=DEV)
    out = torch.empty(B, H, d, device=DEV)
    lse = torch.empty(B, H, device=DEV)
    lib = fd.load()

    def call(s):
        st = lib.fd_decode_split(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), ld.data_ptr(), B, H, N, d, 1, P,
                                 d ** -0.5, o_p.data_ptr(), m_p.data_ptr(), l_p.data_ptr(), s_p.data_ptr(),
                                 s.cuda_stream)
        assert st == 0
        fd.combine_lse(o_p, s_p, out=out, lse=lse, stream=s)
    g = _capture(call)
    q2, k2, v2, _ = random_case(B, H, N, d, "f16", lens=[2000, 777], seed=82)
    qd.copy_(q2)
    kd.copy_(k2)
    vd.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention(q2, k2, v2, lens=lt)
    check_out(out, ref_out, "f16")
    check_lse(lse, ref_lse, "f16")


def test_paged_gqa_fp8_graph_replays_on_a_new_block_table():
    """E4M3 pages, G = 8, 16-token pages: the captured launch holds the page
    pools' tensor maps (by value, as kernel parameters); the replay reads
    whatever table, lengths and page contents the captured buffers hold."""
    from split_kv_fd_gb300.inputs import quantize_e4m3, to_paged_bytes
    B, Hkv, G, N, d = 3, 2, 8, 640, 128
    _, k, v, lt = random_case(B, Hkv, N, d, "bf16", lens=[640, 333, 0], seed=91, nan_pad=False)
    q = torch.randn(B, G * Hkv, d, generator=torch.Generator().manual_seed(92)).to(torch.bfloat16)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    kp, table = to_paged_bytes(k8, 16, seed=1)
    vp, _ = to_paged_bytes(v8, 16, seed=1)
    qd, ld = q.to(DEV), lt.to(DEV)
    kpd, vpd, td, ksd, vsd = kp.to(DEV), vp.to(DEV), table.to(DEV), ks.to(DEV), vs.to(DEV)
    out = torch.empty(B, G * Hkv, d, device=DEV)
    lse = torch.empty(B, G * Hkv, device=DEV)
    ws = torch.empty(max(256, fd.workspace_size_gqa(B, G * Hkv, Hkv, N, d)), dtype=torch.uint8, device=DEV)
    g = _capture(lambda s: fd.decode_gqa_paged_fp8(qd, kpd, vpd, ksd, vsd, td, ld, out=out, lse=lse,
                                                   workspace=ws, stream=s))
    rep = lambda x: x.repeat_interleave(G, dim=1)   # noqa: E731
    for seed, lens in ((2, [640, 333, 0]), (3, [1, 640, 500])):
        kp2, table2 = to_paged_bytes(k8, 16, seed=seed)
        vp2, _ = to_paged_bytes(v8, 16, seed=seed)
        kpd.copy_(kp2)
        vpd.copy_(vp2)
        td.copy_(table2)
        l2 = torch.tensor(lens, dtype=torch.int32)
        ld.copy_(l2)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.attention_fp8(q, rep(k8), rep(v8), rep(ks), rep(vs), lens=l2)
        check_out(out, ref_out, "bf16")
        check_lse(lse, ref_lse, "bf16")
