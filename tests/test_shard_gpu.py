"""Sequence-sharded decode on the GPU, against the float64 oracle's unsplit
attention.

Every run here has one GPU, so the W ranks' local decodes run one after
another in this process, each on its own copy of its shard of K/V (as a
rank would hold it), and the exchange is the copy of each rank's partial
into the gathered buffers; the fold is the module's tree of fd_merge_lse
launches.  ``decode_sharded`` itself (local decode, NCCL all-gather, fold)
runs in a one-rank NCCL process group.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300 import shard
from split_kv_fd_gb300.inputs import random_case
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

OUT_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    yield
    assert fd.device_status() == 0


@pytest.mark.parametrize("W", [2, 3, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_w_rank_split_folds_to_unsplit(W, dtype):
    B, H, N, d = 4, 8, 5000, 128 if dtype != "f32" else 64
    # lengths that leave some ranks empty for some sequences, and one empty sequence
    lens = [5000, 1900, 333, 0]
    q, k, v, lt = random_case(B, H, N, d, dtype, lens=lens, seed=W * 7 + len(dtype))
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    dev = torch.device("cuda")
    qd = q.to(dev)
    o_all = torch.empty((W, B, H, d), dtype=torch.float32, device=dev)
    s_all = torch.empty((W, B, H), dtype=torch.float32, device=dev)
    for r, (lo, hi) in enumerate(shard.shard_bounds(N, W)):
        ks = k[:, :, lo:hi].contiguous().to(dev)
        vs = v[:, :, lo:hi].contiguous().to(dev)
        ls = shard.local_lengths(lt, lo, hi).to(dev)
        o_r, s_r = fd.decode(qd, ks, vs, ls, out_dtype=torch.float32)
        o_all[r].copy_(o_r)
        s_all[r].copy_(s_r)
    out, lse = shard.fold_tree(o_all, s_all)
    check_out(out, ref_out, dtype, what=f"W={W} out")
    check_lse(lse, ref_lse, dtype, what=f"W={W} lse")


_CHILD = r"""
import os, sys, torch, torch.distributed as dist
sys.path.insert(0, os.environ["FD_ROOT"])
import numpy as np
import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300 import shard
from split_kv_fd_gb300.inputs import random_case
sys.path.insert(0, os.path.join(os.environ["FD_ROOT"], "tests"))
from parity_util import check_lse, check_out
torch.cuda.set_device(0)
dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
try:
    fd.load()
    q, k, v, lt = random_case(2, 8, 3000, 128, "bf16", lens=[3000, 17], seed=5)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lt)
    lo, hi = shard.shard_bounds(3000, 1)[0]
    dev = torch.device("cuda", 0)
    out, lse = shard.decode_sharded(q.to(dev), k.to(dev), v.to(dev),
                                    shard.local_lengths(lt, lo, hi).to(dev))
    torch.cuda.synchronize()
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    assert fd.device_status() == 0
    print("SHARDED_OK")
finally:
    dist.destroy_process_group()
"""


@pytest.mark.timeout(300)
def test_decode_sharded_through_nccl_one_rank():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    env = dict(os.environ, FD_ROOT=root, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
               NCCL_NVLS_ENABLE="0")
    r = subprocess.run([sys.executable, "-c", _CHILD], env=env, capture_output=True, text=True,
                       timeout=240)
    assert r.returncode == 0 and "SHARDED_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
