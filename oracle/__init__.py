"""Float64 CPU oracle for split-KV decode attention (FlashDecoding).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the
``split_kv_fd_gb300`` package and its CUDA library) never imports this
module, and this module never imports the product path.

The arithmetic lives in ``fd_oracle.c`` (plain C, IEEE double, index-order
loops); this file only compiles it with gcc and marshals numpy arrays.  Each
function names the passage of the pages it follows; see the C file header
for the page titles.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against values printed on the pages, closed forms, exact high-precision brute
force, scipy, and split/merge invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfd_oracle.so")

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fd_oracle.c into a shared library (gcc, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I, I64, D = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.or_attention.argtypes = [P, P, P, P, I, I, I, I, I, D, P, P, I]
        lib.or_attention.restype = I
        lib.or_split_partials.argtypes = [P, P, P, P, I, I, I, I, I, D, I, P, P, P, P, I]
        lib.or_split_partials.restype = I
        lib.or_combine_mlo.argtypes = [P, P, P, I64, I, I, P, P]
        lib.or_combine_mlo.restype = None
        lib.or_combine_lse.argtypes = [P, P, I64, I, I, P, P]
        lib.or_combine_lse.restype = None
        lib.or_merge_lse_sequential.argtypes = [P, P, I64, I, I, P, P]
        lib.or_merge_lse_sequential.restype = None
        lib.or_merge_mlo_tree.argtypes = [P, P, P, I64, I, I, P, P]
        lib.or_merge_mlo_tree.restype = I
        lib.or_online_softmax.argtypes = [P, I, P, P, P, P]
        lib.or_online_softmax.restype = None
        lib.or_tile_incremental.argtypes = [P, P, I, I, P, P, P, P, P, P]
        lib.or_tile_incremental.restype = None
        lib.or_attention_paged.argtypes = [P, P, P, P, P, I, I, I, I, I, I64, I, D, P, P, I]
        lib.or_attention_paged.restype = I
        lib.or_attention_fp8.argtypes = [P, I, P, P, P, P, P, I, I, I, I, D, P, P, I]
        lib.or_attention_fp8.restype = I
        lib.or_attention_gqa.argtypes = [P, P, P, P, I, I, I, I, I, I, D, P, P, I]
        lib.or_attention_gqa.restype = I
        lib.or_decode.argtypes = [I, P, P, I64]
        lib.or_decode.restype = None
        lib.or_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_double.restype = D
        lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_double.restype = D
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_bits(x, dtype: str | None = None):
    """Return ``(contiguous numpy array holding the raw element bits, dtype)``.

    Accepts numpy arrays (float32 / float16, or uint16/int16 with
    ``dtype='bf16'``) and CPU torch tensors (float32 / float16 / bfloat16).
    """
    if hasattr(x, "detach"):  # torch tensor: read its bits, no conversion
        import torch  # local import: only tensors need it
        x = x.detach().contiguous()
        if x.dtype == torch.float32:
            return np.ascontiguousarray(x.numpy()), "f32"
        if x.dtype == torch.float16:
            return np.ascontiguousarray(x.numpy()), "f16"
        if x.dtype == torch.bfloat16:
            return np.ascontiguousarray(x.view(torch.int16).numpy()), "bf16"
        raise TypeError(f"unsupported tensor dtype {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, "f32"
    if x.dtype == np.float16:
        return x, "f16"
    if x.dtype in (np.uint16, np.int16) and dtype == "bf16":
        return x, "bf16"
    raise TypeError(f"unsupported array dtype {x.dtype} (tag {dtype})")


def _inputs(q, k, v, lens, dtype):
    qb, dq = as_bits(q, dtype)
    kb, dk = as_bits(k, dtype)
    vb, dv = as_bits(v, dtype)
    if not (dq == dk == dv):
        raise TypeError("q, K and V must share one dtype")
    if kb.ndim != 4 or vb.shape != kb.shape or qb.shape != kb.shape[:2] + kb.shape[3:]:
        raise ValueError(f"shapes q{qb.shape} K{kb.shape} V{vb.shape}")
    B, H, N, d = kb.shape
    lb = None
    if lens is not None:
        if hasattr(lens, "detach"):
            lens = lens.detach().cpu().numpy()
        lb = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
        if lb.shape != (B,):
            raise ValueError("lens must have shape [B]")
    return qb, kb, vb, lb, (B, H, N, d), DTYPE_CODES[dq]


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attention(q, k, v, lens=None, scale=None, dtype=None, nthreads=None):
    """Full unsplit attention in float64.  Returns ``(out [B,H,d], lse [B,H])``.

    out = softmax(scale * q K^T) V and lse = ln sum_j exp(scale * q.K_j)
    per (b, h) over the first ``lens[b]`` tokens; defined in
    "FlashDecoding 数学推导" §2.1.1 and "...传统 m/l/o 方法与 LSE 方法"
    §2.1.1 / §2.3.2.  ``scale`` defaults to 1/sqrt(d).
    """
    lib = _load()
    qb, kb, vb, lb, (B, H, N, d), code = _inputs(q, k, v, lens, dtype)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((B, H, d), np.float64)
    lse = np.empty((B, H), np.float64)
    rc = lib.or_attention(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(lb), B, H, N, d, code,
                          float(scale), _ptr(out), _ptr(lse),
                          int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("or_attention failed")
    return out, lse


def attention_paged(q, k_pages, v_pages, block_table, lens, scale=None, dtype=None,
                    nthreads=None):
    """Full attention over a paged KV cache, in float64.  Returns ``(out, lse)``.

    k_pages / v_pages [num_pages, H, page_size, d]; block_table [B, max_pages]
    int32; lens [B].  Logical token t of sequence b is row t % page_size of
    physical page block_table[b, t // page_size] (the block-table
    indirection of "adv04: Flash-Decoding" §5 and "从第一性原理推导 Flash
    Attention" §7.1).
    """
    lib = _load()
    qb, dq = as_bits(q, dtype)
    kb, dk = as_bits(k_pages, dtype)
    vb, dv = as_bits(v_pages, dtype)
    if not (dq == dk == dv):
        raise TypeError("q, K and V must share one dtype")
    num_pages, H, ps, d = kb.shape
    B = qb.shape[0]
    if qb.shape != (B, H, d) or vb.shape != kb.shape:
        raise ValueError("shapes")
    if hasattr(block_table, "detach"):
        block_table = block_table.detach().cpu().numpy()
    if hasattr(lens, "detach"):
        lens = lens.detach().cpu().numpy()
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    lb = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    maxp = bt.shape[1] if bt.ndim == 2 else 0
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((B, H, d), np.float64)
    lse = np.empty((B, H), np.float64)
    rc = lib.or_attention_paged(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(lb), B, H, d, ps,
                                maxp, num_pages, DTYPE_CODES[dq], float(scale), _ptr(out),
                                _ptr(lse), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("or_attention_paged failed (bad arguments or block-table entry)")
    return out, lse


def attention_gqa(q, k, v, lens=None, scale=None, dtype=None, nthreads=None):
    """Grouped-query attention in float64 ("从第一性原理推导 Flash Attention" §8).

    q [B, Hq, d]; k, v [B, Hkv, N, d] with Hq a multiple of Hkv; query head h
    uses K/V head h // (Hq // Hkv).  Returns ``(out [B,Hq,d], lse [B,Hq])``.
    """
    lib = _load()
    qb, dq = as_bits(q, dtype)
    kb, dk = as_bits(k, dtype)
    vb, dv = as_bits(v, dtype)
    if not (dq == dk == dv):
        raise TypeError("q, K and V must share one dtype")
    B, Hkv, N, d = kb.shape
    Hq = qb.shape[1]
    if qb.shape != (B, Hq, d) or vb.shape != kb.shape or Hq % Hkv:
        raise ValueError("shapes: q [B,Hq,d], K/V [B,Hkv,N,d], Hq % Hkv == 0")
    lb = None
    if lens is not None:
        if hasattr(lens, "detach"):
            lens = lens.detach().cpu().numpy()
        lb = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    rc = lib.or_attention_gqa(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(lb), B, Hq, Hkv, N, d,
                              DTYPE_CODES[dq], float(scale), _ptr(out), _ptr(lse),
                              int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("or_attention_gqa failed")
    return out, lse


def _e4m3_bits(x):
    if hasattr(x, "detach"):
        import torch
        x = x.detach().contiguous()
        if x.dtype == torch.float8_e4m3fn:
            x = x.view(torch.uint8)
        return np.ascontiguousarray(x.numpy().astype(np.uint8, copy=False))
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint8))


def attention_fp8(q, k, v, k_scale, v_scale, lens=None, scale=None, nthreads=None):
    """Full attention over an E4M3 KV cache with per-(b,h) scales, in float64.

    k, v: [B,H,N,d] E4M3 bytes (uint8 arrays or torch float8_e4m3fn / uint8
    tensors); k_scale, v_scale: [B,H] float32; the value of an element is
    scale[b,h] * e4m3(byte).  q: float32 / float16 / bfloat16 [B,H,d].
    Returns ``(out, lse)``.
    """
    lib = _load()
    qb, dq = as_bits(q)
    kb, vb = _e4m3_bits(k), _e4m3_bits(v)
    B, H, N, d = kb.shape
    if qb.shape != (B, H, d) or vb.shape != kb.shape:
        raise ValueError("shapes")
    ks = _f32_arr(k_scale).reshape(B * H)
    vs = _f32_arr(v_scale).reshape(B * H)
    lb = None
    if lens is not None:
        if hasattr(lens, "detach"):
            lens = lens.detach().cpu().numpy()
        lb = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((B, H, d), np.float64)
    lse = np.empty((B, H), np.float64)
    rc = lib.or_attention_fp8(_ptr(qb), DTYPE_CODES[dq], _ptr(kb), _ptr(vb), _ptr(ks), _ptr(vs),
                              _ptr(lb), B, H, N, d, float(scale), _ptr(out), _ptr(lse),
                              int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("or_attention_fp8 failed")
    return out, lse


def _f32_arr(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def split_partials(q, k, v, P, lens=None, scale=None, dtype=None, nthreads=None):
    """Per-split (o, m, l, S) in the partition of "adv04: Flash-Decoding" §4.

    Returns ``(o [B,H,P,d], m [B,H,P], l [B,H,P], S [B,H,P])`` with o
    normalised per split ("FlashDecoding 数学推导" §2.4.1 direct form) and
    S = m + ln l.  Empty splits are (0, -inf, 0, -inf).
    """
    lib = _load()
    qb, kb, vb, lb, (B, H, N, d), code = _inputs(q, k, v, lens, dtype)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((B, H, P, d), np.float64)
    m = np.empty((B, H, P), np.float64)
    l = np.empty((B, H, P), np.float64)
    s = np.empty((B, H, P), np.float64)
    rc = lib.or_split_partials(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(lb), B, H, N, d, code,
                               float(scale), int(P), _ptr(o), _ptr(m), _ptr(l), _ptr(s),
                               int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("or_split_partials failed")
    return o, m, l, s


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _rows(o_part):
    *lead, P, d = o_part.shape
    rows = int(np.prod(lead)) if lead else 1
    return tuple(lead), rows, P, d


def combine_mlo(o_part, m_part, l_part):
    """m/l/o merge ("FlashDecoding 数学推导" §2.4.2).  Returns (out, lse)."""
    o_part, m_part, l_part = _f64(o_part), _f64(m_part), _f64(l_part)
    lead, rows, P, d = _rows(o_part)
    out = np.empty(lead + (d,), np.float64)
    lse = np.empty(lead, np.float64)
    _load().or_combine_mlo(_ptr(o_part), _ptr(m_part), _ptr(l_part), rows, P, d,
                           _ptr(out), _ptr(lse))
    return out, lse


def combine_lse(o_part, s_part):
    """LSE merge ("...传统 m/l/o 方法与 LSE 方法" §2.3.4).  Returns (out, lse)."""
    o_part, s_part = _f64(o_part), _f64(s_part)
    lead, rows, P, d = _rows(o_part)
    out = np.empty(lead + (d,), np.float64)
    lse = np.empty(lead, np.float64)
    _load().or_combine_lse(_ptr(o_part), _ptr(s_part), rows, P, d, _ptr(out), _ptr(lse))
    return out, lse


def merge_lse_sequential(o_part, s_part):
    """Sequential safe two-term (+) fold ("...LSE 方法" §3.2.1 stage 2)."""
    o_part, s_part = _f64(o_part), _f64(s_part)
    lead, rows, P, d = _rows(o_part)
    out = np.empty(lead + (d,), np.float64)
    lse = np.empty(lead, np.float64)
    _load().or_merge_lse_sequential(_ptr(o_part), _ptr(s_part), rows, P, d,
                                    _ptr(out), _ptr(lse))
    return out, lse


def merge_mlo_tree(o_part, m_part, l_part):
    """Pairwise tree reduction of (O, M, L) ("...LSE 方法" §3.1.3)."""
    o_part, m_part, l_part = _f64(o_part), _f64(m_part), _f64(l_part)
    lead, rows, P, d = _rows(o_part)
    out = np.empty(lead + (d,), np.float64)
    lse = np.empty(lead, np.float64)
    rc = _load().or_merge_mlo_tree(_ptr(o_part), _ptr(m_part), _ptr(l_part), rows, P, d,
                                   _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError("or_merge_mlo_tree failed")
    return out, lse


def online_softmax(x):
    """(m, d) recurrence ("FlashDecoding 数学推导" §2.3.2) with its step states."""
    x = _f64(x)
    n = x.shape[0]
    ms = np.empty(n, np.float64)
    ds = np.empty(n, np.float64)
    m = ctypes.c_double()
    dd = ctypes.c_double()
    _load().or_online_softmax(_ptr(x), n, _ptr(ms), _ptr(ds), ctypes.byref(m), ctypes.byref(dd))
    return m.value, dd.value, ms, ds


def tile_incremental(s, V):
    """Per-token m/l/o update ("FlashDecoding 数学推导" §2.4.1 增量更新).

    Returns ``(m, l, o, m_steps, l_steps, o_steps)``.
    """
    s, V = _f64(s), _f64(V)
    n, d = V.shape
    ms = np.empty(n, np.float64)
    ls = np.empty(n, np.float64)
    os_ = np.empty((n, d), np.float64)
    o = np.empty(d, np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    _load().or_tile_incremental(_ptr(s), _ptr(V), n, d, _ptr(ms), _ptr(ls), _ptr(os_),
                                ctypes.byref(m), ctypes.byref(l), _ptr(o))
    return m.value, l.value, o, ms, ls, os_


def decode_elements(bits, dtype: str):
    """Widen raw fp16/bf16/fp32 element bits to float64 with the oracle's decoders."""
    bits = np.ascontiguousarray(bits)
    out = np.empty(bits.shape, np.float64)
    _load().or_decode(DTYPE_CODES[dtype], _ptr(bits), _ptr(out), bits.size)
    return out
