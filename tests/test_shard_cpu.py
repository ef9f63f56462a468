"""Sequence-sharded decode, host side (no GPU): the token partition over the
ranks, the exchange of partials over a real process group (gloo, world
sizes 2 and 3, one process per rank) and the tree fold's order.

Each rank's local partial comes from the float64 oracle on its shard, and
the fold is the oracle's sequential (+) ("...传统 m/l/o 方法与 LSE 方法"
§3.2.1 stage 2) or the module's tree with an oracle merge; both must equal
the oracle's unsplit attention on the whole sequence ("...LSE 方法" §2.3.6).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from split_kv_fd_gb300 import shard
from split_kv_fd_gb300.inputs import random_case


def test_shard_bounds_cover_every_position_once():
    for N in (0, 1, 5, 1000, 4097):
        for W in (1, 2, 3, 4, 7, 8, 16):
            b = shard.shard_bounds(N, W)
            assert len(b) == W
            assert b[0][0] == 0 and b[-1][1] == N
            for (lo, hi), (lo2, _) in zip(b, b[1:]):
                assert lo <= hi == lo2
            c = -(-N // W) if N else 0
            assert all(hi - lo <= c for lo, hi in b)
    with pytest.raises(ValueError):
        shard.shard_bounds(10, 0)


def test_local_lengths_add_up():
    lens = [0, 1, 999, 1000, 1001, 2500, 4096]
    for W in (1, 2, 3, 5, 8):
        parts = [shard.local_lengths(lens, lo, hi) for lo, hi in shard.shard_bounds(4096, W)]
        assert all(p.dtype == torch.int32 for p in parts)
        assert torch.equal(sum(p.to(torch.int64) for p in parts), torch.tensor(lens))
        for (lo, hi), p in zip(shard.shard_bounds(4096, W), parts):
            assert int(p.min()) >= 0 and int(p.max()) <= hi - lo


def _oracle_merge(oa, sa, ob, sb, out, lse):
    """One (+) of two float32 partial sets by the oracle's sequential fold."""
    o = np.stack([oa.double().numpy(), ob.double().numpy()], axis=-2)
    s = np.stack([sa.double().numpy(), sb.double().numpy()], axis=-1)
    ro, rl = oracle.merge_lse_sequential(o, s)
    out.copy_(torch.from_numpy(ro))
    lse.copy_(torch.from_numpy(rl))


def _case():
    B, H, N, d = 3, 4, 700, 64
    q, k, v, lt = random_case(B, H, N, d, "bf16", lens=[700, 230, 0], seed=21)
    return q, k, v, lt, N


def _local_partial(q, k, v, lt, lo, hi):
    ls = shard.local_lengths(lt, lo, hi)
    o, s = oracle.attention(q, k[:, :, lo:hi].contiguous(), v[:, :, lo:hi].contiguous(), lens=ls)
    return torch.from_numpy(o).float(), torch.from_numpy(s).float()


def _check(o, s, ref_o, ref_s):
    o, s = o.double().numpy(), s.double().numpy()
    assert np.max(np.abs(o - ref_o)) <= 1e-5
    fin = np.isfinite(ref_s)
    assert np.array_equal(np.isfinite(s), fin)
    assert np.all(s[~fin] == -np.inf) and np.all(o[~fin] == 0)
    assert np.max(np.abs(s[fin] - ref_s[fin]) / np.maximum(1, np.abs(ref_s[fin]))) <= 1e-6


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8])
def test_fold_tree_equals_unsplit(W):
    """The tree order of fold_tree, every rank's partial computed here."""
    q, k, v, lt, N = _case()
    ref_o, ref_s = oracle.attention(q, k, v, lens=lt)
    parts = [_local_partial(q, k, v, lt, lo, hi) for lo, hi in shard.shard_bounds(N, W)]
    o_all = torch.stack([p[0] for p in parts])
    s_all = torch.stack([p[1] for p in parts])
    # the oracle's own sequential fold over the W partials
    so, ss = oracle.merge_lse_sequential(o_all.permute(1, 2, 0, 3).double().numpy(),
                                         s_all.permute(1, 2, 0).double().numpy())
    _check(torch.from_numpy(so), torch.from_numpy(ss), ref_o, ref_s)
    o, s = shard.fold_tree(o_all, s_all, merge=_oracle_merge)
    _check(o, s, ref_o, ref_s)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, lt, N = _case()
        lo, hi = shard.shard_bounds(N, world)[rank]
        # this rank holds only its own tokens
        o_loc, s_loc = _local_partial(q, k, v, lt, lo, hi)
        o_all, s_all = shard.exchange(o_loc, s_loc)
        # every rank's slot holds that rank's partial
        for r, (a, b) in enumerate(shard.shard_bounds(N, world)):
            eo, es = _local_partial(q, k, v, lt, a, b)
            assert torch.equal(o_all[r], eo) and torch.equal(s_all[r], es)
        ref_o, ref_s = oracle.attention(q, k, v, lens=lt)
        so, ss = oracle.merge_lse_sequential(o_all.permute(1, 2, 0, 3).double().numpy(),
                                             s_all.permute(1, 2, 0).double().numpy())
        _check(torch.from_numpy(so), torch.from_numpy(ss), ref_o, ref_s)
        o, s = shard.fold_tree(o_all, s_all, merge=_oracle_merge)
        _check(o, s, ref_o, ref_s)
        queue.put((rank, "ok"))
    except Exception as e:  # report to the parent instead of hanging it
        queue.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
@pytest.mark.parametrize("world", [2, 3])
def test_exchange_and_fold_over_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(150)
    got = dict(queue.get(timeout=5) for _ in range(world))
    assert got == {r: "ok" for r in range(world)}, got
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
