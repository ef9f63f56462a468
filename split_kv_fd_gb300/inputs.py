"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no arithmetic of the method: it only draws numbers.

Recipe (one ``torch.Generator`` on the target device, seeded with the
workload's seed; draws in this order):
  1. lengths: ``randint(1, N + 1, (B,))`` if the workload is ragged, else N;
  2. q: float32 N(0, 1), shape [B, H, d];
  3. K: float32 N(0, 1) * k_scale, shape [B, Hkv, N, d] (Hkv = H unless the
     workload is grouped-query), drawn in chunks of the flattened tensor;
  4. V: float32 N(0, 1), shape [B, Hkv, N, d], drawn the same way;
each cast to the storage dtype with round-to-nearest-even.  Rows past a
sequence's length are filled with NaN, so a read past the end shows up as a
NaN in the result.
"""
from __future__ import annotations

import torch

from .workloads import Workload

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _fill_normal(t: torch.Tensor, g: torch.Generator, factor: float, chunk: int) -> None:
    flat = t.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=g, device=t.device, dtype=torch.float32)
        if factor != 1.0:
            x.mul_(factor)
        flat[s:e].copy_(x)


def make_lengths(w: Workload, device="cpu", seed: int | None = None) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    if w.ragged:
        return torch.randint(1, w.N + 1, (w.B,), generator=g, device=device).to(torch.int32)
    return torch.full((w.B,), w.N, dtype=torch.int32, device=device)


def make_inputs(w: Workload, device="cpu", seed: int | None = None,
                nan_pad: bool = True, chunk: int = 1 << 26):
    """Return ``(q, K, V, lens)`` for workload ``w`` on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    dt = TORCH_DTYPES[w.dtype]
    if w.ragged:
        lens = torch.randint(1, w.N + 1, (w.B,), generator=g, device=device).to(torch.int32)
    else:
        lens = torch.full((w.B,), w.N, dtype=torch.int32, device=device)
    q = torch.empty((w.B, w.H, w.d), dtype=dt, device=device)
    k = torch.empty((w.B, w.kv_heads, w.N, w.d), dtype=dt, device=device)
    v = torch.empty((w.B, w.kv_heads, w.N, w.d), dtype=dt, device=device)
    _fill_normal(q, g, 1.0, chunk)
    _fill_normal(k, g, w.k_scale, chunk)
    _fill_normal(v, g, 1.0, chunk)
    if nan_pad and w.ragged:
        for b, n in enumerate(lens.tolist()):
            if n < w.N:
                k[b, :, n:, :] = float("nan")
                v[b, :, n:, :] = float("nan")
    return q, k, v, lens


def random_case(B, H, N, d, dtype="bf16", lens=None, seed=0, device="cpu",
                k_scale=1.0, nan_pad=True):
    """A small seeded case with explicit shapes (for parity and edge tests).

    ``lens``: None (all N), an int list of length B, or "ragged" (drawn
    uniformly from [0, N] so that empty sequences occur).
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = TORCH_DTYPES[dtype]
    if lens is None:
        lt = torch.full((B,), N, dtype=torch.int32, device=device)
    elif isinstance(lens, str) and lens == "ragged":
        lt = torch.randint(0, N + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        lt = torch.tensor(list(lens), dtype=torch.int32, device=device)
    q = torch.empty((B, H, d), dtype=dt, device=device)
    k = torch.empty((B, H, N, d), dtype=dt, device=device)
    v = torch.empty((B, H, N, d), dtype=dt, device=device)
    _fill_normal(q, g, 1.0, 1 << 24)
    _fill_normal(k, g, k_scale, 1 << 24)
    _fill_normal(v, g, 1.0, 1 << 24)
    if nan_pad:
        for b, n in enumerate(lt.tolist()):
            if n < N:
                k[b, :, n:, :] = float("nan")
                v[b, :, n:, :] = float("nan")
    return q, k, v, lt


def to_paged(k: torch.Tensor, v: torch.Tensor, page_size: int, seed: int = 0,
             extra_pages: int = 3):
    """Lay a contiguous [B,H,N,d] cache out as pages [num_pages, H, page_size, d]
    in a seeded random page order, with the block table [B, ceil(N/page_size)].

    Every page that holds no token and every row past N is NaN.  This only
    moves numbers (no arithmetic of the method).
    """
    B, H, N, d = k.shape
    maxp = -(-N // page_size)
    npad = maxp * page_size
    num_pages = B * maxp + extra_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[: B * maxp].to(k.device)
    table = perm.view(B, maxp).to(torch.int32).contiguous()

    def scatter(x):
        if npad != N:
            x = torch.cat([x, torch.full((B, H, npad - N, d), float("nan"), dtype=x.dtype,
                                         device=x.device)], dim=2)
        pages = torch.full((num_pages, H, page_size, d), float("nan"), dtype=x.dtype,
                           device=x.device)
        src = x.view(B, H, maxp, page_size, d).permute(0, 2, 1, 3, 4).reshape(B * maxp, H,
                                                                             page_size, d)
        pages[perm] = src
        return pages

    return scatter(k), scatter(v), table


E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor):
    """Per-(b,h) symmetric E4M3 storage of a [B,H,N,d] cache (input
    preparation for the FP8 path, not part of the attention): scale = amax /
    448 over the finite rows of (b, h) (1 if there are none), bytes = E4M3
    round-to-nearest-even of x / scale.  NaN rows (past a sequence's length)
    stay NaN.  Returns ``(x_e4m3 [B,H,N,d] float8_e4m3fn, scale [B,H] float32)``.
    """
    B, H, N, d = x.shape
    out = torch.empty((B, H, N, d), dtype=torch.float8_e4m3fn, device=x.device)
    scale = torch.empty((B, H), dtype=torch.float32, device=x.device)
    for b in range(B):  # one sequence at a time bounds the float32 temporaries
        xb = x[b].float()
        amax = torch.nan_to_num(xb, nan=0.0).abs().amax(dim=(1, 2))
        sb = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        scale[b] = sb
        out[b] = (xb / sb[:, None, None]).to(torch.float8_e4m3fn)
    return out, scale


def to_paged_bytes(x8: torch.Tensor, page_size: int, seed: int = 0, extra_pages: int = 3):
    """An E4M3 cache [B,H,N,d] (torch.float8_e4m3fn) laid out as pages
    [num_pages, H, page_size, d] in the seeded page order of to_paged, with the
    block table [B, ceil(N/page_size)].  Unused pages and rows past N hold
    0x7F (an E4M3 NaN).  This only moves bytes."""
    B, H, N, d = x8.shape
    maxp = -(-N // page_size)
    num_pages = B * maxp + extra_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[: B * maxp].to(x8.device)
    u = x8.view(torch.uint8)
    if maxp * page_size != N:
        u = torch.cat([u, torch.full((B, H, maxp * page_size - N, d), 0x7F, dtype=torch.uint8,
                                     device=x8.device)], dim=2)
    pages = torch.full((num_pages, H, page_size, d), 0x7F, dtype=torch.uint8, device=x8.device)
    pages[perm] = u.view(B, H, maxp, page_size, d).permute(0, 2, 1, 3, 4).reshape(B * maxp, H, page_size, d)
    return pages.view(torch.float8_e4m3fn), perm.view(B, maxp).to(torch.int32).contiguous()
