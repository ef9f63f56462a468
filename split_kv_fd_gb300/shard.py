"""Sequence-sharded decode: every sequence's KV cache spread over the ranks
of a process group by token position, and the merge of the partial results
the ranks exchange.

This is the multi-device form of the split the pages derive: tiles of the
sequence processed apart and merged exactly, with the tiles on different
devices ("FlashDecoding 数学推导：传统 m/l/o 方法与 LSE 方法" §3.1.3, tiles on
several streams reduced pairwise in a tree; §5.4, the LSE form for settings
where communication is the limit, such as ring attention; "从第一性原理推导
Flash Attention" §8, ring attention).

The three steps, on every rank r of W:

1. Local decode.  Rank r holds tokens [lo_r, hi_r) of every sequence
   (``shard_bounds``: W contiguous ranges of ceil(N / W) positions, the
   partition of "adv04: Flash-Decoding" §4 applied to the ranks) as its own
   K/V [B, H, hi_r - lo_r, d] with its own lengths (``local_lengths``).  It
   runs ``fd.decode`` on them with a float32 output and lse: one normalised
   partial (o_r, S_r) per (b, h), S_r = -inf where it holds no token.
2. Exchange (``exchange``).  An all-gather of (o_r, S_r), (d + 1) floats per
   (b, h), into buffers [W, B, H, d] and [W, B, H] that the rank owns.  No
   kernel ever reads another device's memory: the collective library moves
   the bytes, and every merge below reads local buffers only.
3. Fold (``fold_tree``).  The W partials merge with the associative (+) of
   the LSE form ("...LSE 方法" §2.3.5, in the safe two-term form of its
   §3.2.1), pairwise in a tree: ceil(log2 W) rounds of ``fd.merge_lse``, in
   place in the gathered buffers.  Every rank ends with the unsplit result.

The collective is torch.distributed's (NCCL between GPUs; gloo on the host,
which the CPU tests use).  The arithmetic of steps 1 and 3 runs in the
library's kernels.
"""
from __future__ import annotations

import torch


def shard_bounds(N: int, world: int) -> list[tuple[int, int]]:
    """Token range [lo_r, hi_r) of every rank: ranges of c = ceil(N / world)
    positions, the last ones shorter or empty when world does not divide N."""
    if world < 1 or N < 0:
        raise ValueError("world >= 1 and N >= 0 required")
    c = -(-N // world) if N else 0
    return [(min(r * c, N), min((r + 1) * c, N)) for r in range(world)]


def local_lengths(lens, lo: int, hi: int) -> torch.Tensor:
    """The tokens of each sequence that fall in [lo, hi): clamp(len - lo, 0,
    hi - lo), as a host int32 tensor.  ``lens`` are the global lengths on the
    host (a list, a numpy array or a CPU tensor); a serving system keeps
    them there, beside the block tables."""
    t = torch.as_tensor(lens, dtype=torch.int64)
    if t.is_cuda:
        raise ValueError("local_lengths works on host lengths")
    return torch.clamp(t - lo, min=0, max=max(0, hi - lo)).to(torch.int32)


def exchange(o_local: torch.Tensor, lse_local: torch.Tensor, group=None, o_all=None, lse_all=None):
    """All-gather every rank's partial (o [B, H, d], lse [B, H], float32) into
    this rank's buffers o_all [W, B, H, d] and lse_all [W, B, H] (allocated
    when not given), rank r's partial at index r.  Returns ``(o_all, lse_all)``.
    """
    import torch.distributed as dist
    W = dist.get_world_size(group)
    if o_local.dtype != torch.float32 or lse_local.dtype != torch.float32:
        raise ValueError("partials must be float32")
    if lse_local.shape != o_local.shape[:-1]:
        raise ValueError("shapes: o [..., d], lse [...]")
    if o_all is None:
        o_all = torch.empty((W,) + tuple(o_local.shape), dtype=torch.float32, device=o_local.device)
    if lse_all is None:
        lse_all = torch.empty((W,) + tuple(lse_local.shape), dtype=torch.float32,
                              device=lse_local.device)
    if o_all.shape != (W,) + tuple(o_local.shape) or lse_all.shape != (W,) + tuple(lse_local.shape):
        raise ValueError("o_all / lse_all must be [W, ...] of the local shapes")
    # gather straight into the views of the rank's own buffers
    dist.all_gather(list(o_all.unbind(0)), o_local.contiguous(), group=group)
    dist.all_gather(list(lse_all.unbind(0)), lse_local.contiguous(), group=group)
    return o_all, lse_all


def fold_tree(o_all: torch.Tensor, lse_all: torch.Tensor, merge=None):
    """Fold W partials with (+) pairwise: in round k, index i (a multiple of
    2^(k+1)) absorbs index i + 2^k, in place.  Returns views of index 0
    ``(o [B, H, d], lse [B, H])``.  ``merge(o_a, s_a, o_b, s_b, out=, lse=)``
    defaults to the library's ``fd.merge_lse``."""
    if merge is None:
        from . import fd
        merge = fd.merge_lse
    W = o_all.shape[0]
    if lse_all.shape[0] != W:
        raise ValueError("o_all and lse_all must hold the same number of partials")
    step = 1
    while step < W:
        for i in range(0, W - step, 2 * step):
            merge(o_all[i], lse_all[i], o_all[i + step], lse_all[i + step],
                  out=o_all[i], lse=lse_all[i])
        step *= 2
    return o_all[0], lse_all[0]


def decode_sharded(q, k_local, v_local, local_lens, group=None, scale=None, workspace=None,
                   o_all=None, lse_all=None):
    """Sequence-sharded decode on one rank: local ``fd.decode`` (float32 out
    and lse), all-gather of the partials, tree fold, all on the current
    stream.  Every rank returns the unsplit ``(out [B, H, d], lse [B, H])``
    in float32.

    q [B, H, d] (the same on every rank); k_local / v_local [B, H, n_r, d]
    this rank's tokens of every sequence; local_lens [B] int32 on the device
    (``local_lengths`` of the global lengths).  All tensors on this rank's
    GPU.
    """
    from . import fd
    out, lse = fd.decode(q, k_local, v_local, local_lens, scale=scale, out_dtype=torch.float32,
                         workspace=workspace)
    o_all, lse_all = exchange(out, lse, group=group, o_all=o_all, lse_all=lse_all)
    return fold_tree(o_all, lse_all)
