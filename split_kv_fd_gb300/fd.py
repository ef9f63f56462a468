"""Python binding of the C ABI in include/fd.h (ctypes; marshalling only).

Every function takes CUDA torch tensors, checks that their dtype, shape,
contiguity and device fit the C call, passes raw device pointers and the
current CUDA stream, and turns a non-OK status into an exception.  All the
arithmetic runs in the CUDA kernels of ``libfd.so``; there is no fallback:
if the library is missing or no GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build_lib

FD_OK = 0
STATUS_NAMES = {0: "FD_OK", 1: "FD_ERR_INVALID_ARG", 2: "FD_ERR_UNSUPPORTED",
                3: "FD_ERR_WORKSPACE", 4: "FD_ERR_CUDA", 5: "FD_ERR_DEVICE_TIMEOUT",
                6: "FD_ERR_SCRATCH_TOO_SMALL", 7: "FD_ERR_BAD_PAGE"}

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# every symbol include/fd.h declares
EXPORTS = ["fd_status_str", "fd_version", "fd_num_sms", "fd_auto_num_splits",
           "fd_workspace_size", "fd_decode", "fd_decode_split", "fd_combine_mlo",
           "fd_combine_lse", "fd_device_status", "fd_decode_noalloc", "fd_decode_paged",
           "fd_decode_fp8", "fd_merge_lse", "fd_decode_gqa", "fd_workspace_size_gqa",
           "fd_selftest_wait_timeout", "fd_decode_gqa_paged", "fd_decode_gqa_fp8",
           "fd_decode_gqa_paged_fp8"]

_lock = threading.Lock()
_lib = None


class FDError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}")


def library_path() -> str:
    return _build_lib.LIB


def load(build_if_missing: bool = False):
    """Load libfd.so (no GPU needed).  Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing and _build_lib.is_stale():
            _build_lib.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fd_status_str.argtypes = [I]
        lib.fd_status_str.restype = ctypes.c_char_p
        lib.fd_version.argtypes = []
        lib.fd_version.restype = I
        lib.fd_num_sms.argtypes = []
        lib.fd_num_sms.restype = I
        lib.fd_auto_num_splits.argtypes = [I, I, I, I, I, I]
        lib.fd_auto_num_splits.restype = I
        lib.fd_workspace_size.argtypes = [I, I, I, I, I]
        lib.fd_workspace_size.restype = S
        lib.fd_decode.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, I, P, P, S, P]
        lib.fd_decode.restype = I
        lib.fd_decode_split.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, P]
        lib.fd_decode_split.restype = I
        lib.fd_combine_mlo.argtypes = [P, P, P, I, I, I, I, P, I, P, P]
        lib.fd_combine_mlo.restype = I
        lib.fd_combine_lse.argtypes = [P, P, I, I, I, I, P, I, P, P]
        lib.fd_combine_lse.restype = I
        lib.fd_decode_paged.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_longlong, I, I, F, P, I,
                                        P, P, S, P]
        lib.fd_decode_paged.restype = I
        lib.fd_decode_fp8.argtypes = [P, I, P, P, P, P, P, I, I, I, I, I, F, P, I, P, P, S, P]
        lib.fd_decode_fp8.restype = I
        lib.fd_merge_lse.argtypes = [P, P, P, P, I, I, P, P, P]
        lib.fd_merge_lse.restype = I
        lib.fd_decode_gqa.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P, I, P, P, S, P]
        lib.fd_decode_gqa.restype = I
        lib.fd_workspace_size_gqa.argtypes = [I, I, I, I, I, I]
        lib.fd_workspace_size_gqa.restype = S
        lib.fd_device_status.argtypes = [I]
        lib.fd_device_status.restype = I
        lib.fd_selftest_wait_timeout.argtypes = [P]
        lib.fd_selftest_wait_timeout.restype = I
        lib.fd_decode_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, I, P, P]
        lib.fd_decode_noalloc.restype = I
        lib.fd_decode_gqa_paged.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_longlong, I, I,
                                            F, P, I, P, P, S, P]
        lib.fd_decode_gqa_paged.restype = I
        lib.fd_decode_gqa_fp8.argtypes = [P, I, P, P, P, P, P, I, I, I, I, I, I, F, P, I, P, P, S, P]
        lib.fd_decode_gqa_fp8.restype = I
        lib.fd_decode_gqa_paged_fp8.argtypes = [P, I, P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_longlong, I,
                                                F, P, I, P, P, S, P]
        lib.fd_decode_gqa_paged_fp8.restype = I
        _lib = lib
        return lib


def status_str(status: int) -> str:
    try:
        return load().fd_status_str(int(status)).decode()
    except Exception:  # pragma: no cover - library not loadable
        return STATUS_NAMES.get(status, str(status))


def _check(status: int, what: str) -> None:
    if status != FD_OK:
        raise FDError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the library has no CPU path)")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _check_qkv(q, k, v, seqlens):
    _need_cuda(q, k, v, seqlens)
    if q.dtype not in DTYPE_CODE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, K, V must share one dtype among float32/float16/bfloat16")
    if k.dim() != 4 or v.shape != k.shape or q.shape != (k.shape[0], k.shape[1], k.shape[3]):
        raise ValueError(f"shapes: q{tuple(q.shape)} must be [B,H,d], K/V{tuple(k.shape)} [B,H,N,d]")
    if seqlens is not None and (seqlens.dtype != torch.int32 or seqlens.shape != (k.shape[0],)):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    B, H, N, d = k.shape
    return B, H, N, d


def num_sms() -> int:
    return load().fd_num_sms()


KV_DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, "f32": 0, "f16": 1,
                 "bf16": 2, "e4m3": 3}


def auto_num_splits(B, H, N, d, dtype=torch.bfloat16, sm_count=None) -> int:
    """fd_auto_num_splits: the split count of the two-call path for this
    shape and K/V storage type (a torch dtype, or "f32"/"f16"/"bf16"/"e4m3")."""
    sm = num_sms() if sm_count is None else sm_count
    return load().fd_auto_num_splits(B, H, N, d, KV_DTYPE_CODE[dtype], sm)


def workspace_size(B, H, N, d, num_splits=0) -> int:
    return load().fd_workspace_size(B, H, N, d, num_splits)


def new_workspace(B, H, N, d, num_splits=0, device=None) -> torch.Tensor:
    """A workspace for fd_decode (reusable across calls on one stream)."""
    n = workspace_size(B, H, N, d, num_splits)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


_ws_cache: dict = {}


def _cached_workspace(device, nbytes):
    key = (device.index if device.index is not None else torch.cuda.current_device())
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def decode(q, k, v, seqlens=None, num_splits=0, scale=None, out_dtype=None, out=None,
           lse=None, return_lse=True, workspace=None, stream=None):
    """Fused split-KV decode attention (fd_decode).  Returns ``(out, lse)``.

    q [B,H,d], k/v [B,H,N,d] on one CUDA device; ``seqlens`` int32 [B] or
    None; ``num_splits`` 0 = automatic.  ``workspace`` defaults to a cached
    buffer per device (calls that overlap on the GPU need their own
    workspaces).
    """
    B, H, N, d = _check_qkv(q, k, v, seqlens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, d), dtype=odt, device=q.device)
    _need_cuda(out, lse)
    if out.dtype not in DTYPE_CODE or out.shape != (B, H, d):
        raise ValueError("out must be [B,H,d] float32/float16/bfloat16")
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (B, H)):
        raise ValueError("lse must be float32 [B,H]")
    lib = load()
    need = lib.fd_workspace_size(B, H, N, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    _need_cuda(workspace)
    st = lib.fd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(seqlens), B, H, N, d, DTYPE_CODE[q.dtype],
                       int(num_splits), float(scale), _ptr(out), DTYPE_CODE[out.dtype], _ptr(lse),
                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                       _stream(q, stream))
    _check(st, "fd_decode")
    return out, lse



def decode_noalloc(q, k, v, seqlens=None, num_splits=0, scale=None, out_dtype=None, out=None,
                   lse=None, return_lse=True, stream=None):
    """fd_decode on the library's own device scratch (fd_decode_noalloc).
    Returns ``(out, lse)``.

    The C call allocates nothing.  This wrapper allocates only what the
    caller leaves out: pass ``out`` (and ``lse``, or ``return_lse=False``)
    for a call that allocates no device memory at all.  Calls on one device
    share the scratch, so they must not overlap on the GPU; problems whose
    partials exceed the scratch raise FD_ERR_SCRATCH_TOO_SMALL."""
    B, H, N, d = _check_qkv(q, k, v, seqlens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, d), dtype=odt, device=q.device)
    _need_cuda(out, lse)
    if out.dtype not in DTYPE_CODE or out.shape != (B, H, d):
        raise ValueError("out must be [B,H,d] float32/float16/bfloat16")
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (B, H)):
        raise ValueError("lse must be float32 [B,H]")
    st = load().fd_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(seqlens), B, H, N, d,
                                  DTYPE_CODE[q.dtype], int(num_splits), float(scale), _ptr(out),
                                  DTYPE_CODE[out.dtype], _ptr(lse), _stream(q, stream))
    _check(st, "fd_decode_noalloc")
    return out, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, num_splits=0, scale=None,
                 out_dtype=None, out=None, lse=None, return_lse=True, workspace=None, stream=None):
    """fd_decode over a paged KV cache (fd_decode_paged).  Returns ``(out, lse)``.

    q [B,H,d]; k_pages/v_pages [num_pages, H, page_size, d]; block_table
    [B, max_pages] int32; seqlens [B] int32 (required).
    """
    _need_cuda(q, k_pages, v_pages, block_table, seqlens)
    if q.dtype not in DTYPE_CODE or k_pages.dtype != q.dtype or v_pages.dtype != q.dtype:
        raise ValueError("q, K, V must share one dtype among float32/float16/bfloat16")
    if k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages/v_pages must be [num_pages, H, page_size, d]")
    num_pages, H, page_size, d = k_pages.shape
    B = q.shape[0]
    if q.shape != (B, H, d):
        raise ValueError("q must be [B,H,d] with H, d of the pages")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seqlens.dtype != torch.int32 or seqlens.shape != (B,):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    max_pages = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, d), dtype=odt, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    lib = load()
    need = lib.fd_workspace_size(B, H, max_pages * page_size, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    st = lib.fd_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens),
                             B, H, d, page_size, max_pages, num_pages, DTYPE_CODE[q.dtype],
                             int(num_splits), float(scale), _ptr(out), DTYPE_CODE[out.dtype],
                             _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(q, stream))
    _check(st, "fd_decode_paged")
    return out, lse


def decode_gqa(q, k, v, seqlens=None, num_splits=0, scale=None, out_dtype=None, out=None,
               lse=None, return_lse=True, workspace=None, stream=None):
    """Grouped-query decode (fd_decode_gqa).  Returns ``(out, lse)``.

    q [B, Hq, d]; k, v [B, Hkv, N, d] with Hq a multiple of Hkv.
    """
    _need_cuda(q, k, v, seqlens)
    if q.dtype not in DTYPE_CODE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, K, V must share one dtype among float32/float16/bfloat16")
    if k.dim() != 4 or v.shape != k.shape or q.dim() != 3 or q.shape[0] != k.shape[0] \
            or q.shape[2] != k.shape[3] or q.shape[1] % k.shape[1]:
        raise ValueError("shapes: q [B,Hq,d], k/v [B,Hkv,N,d], Hq % Hkv == 0")
    B, Hkv, N, d = k.shape
    Hq = q.shape[1]
    if seqlens is not None and (seqlens.dtype != torch.int32 or seqlens.shape != (B,)):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, d), dtype=odt, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    lib = load()
    need = lib.fd_workspace_size_gqa(B, Hq, Hkv, N, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    st = lib.fd_decode_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(seqlens), B, Hq, Hkv, N, d,
                           DTYPE_CODE[q.dtype], int(num_splits), float(scale), _ptr(out),
                           DTYPE_CODE[out.dtype], _ptr(lse), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(q, stream))
    _check(st, "fd_decode_gqa")
    return out, lse



def decode_gqa_paged(q, k_pages, v_pages, block_table, seqlens, num_splits=0, scale=None,
                     out_dtype=None, out=None, lse=None, return_lse=True, workspace=None, stream=None):
    """Grouped-query decode over a paged KV cache (fd_decode_gqa_paged).
    Returns ``(out, lse)``.

    q [B, Hq, d]; k_pages/v_pages [num_pages, Hkv, page_size, d] with Hq a
    multiple of Hkv and page_size 16 or a multiple of 32; block_table [B,
    max_pages] int32; seqlens [B] int32 (required).
    """
    _need_cuda(q, k_pages, v_pages, block_table, seqlens)
    if q.dtype not in DTYPE_CODE or k_pages.dtype != q.dtype or v_pages.dtype != q.dtype:
        raise ValueError("q, K, V must share one dtype among float32/float16/bfloat16")
    if k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages/v_pages must be [num_pages, Hkv, page_size, d]")
    num_pages, Hkv, page_size, d = k_pages.shape
    B, Hq = q.shape[0], q.shape[1]
    if q.dim() != 3 or q.shape[2] != d or Hq % Hkv:
        raise ValueError("q must be [B, Hq, d] with Hq a multiple of the pages' Hkv")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seqlens.dtype != torch.int32 or seqlens.shape != (B,):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    max_pages = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, d), dtype=odt, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    lib = load()
    need = lib.fd_workspace_size_gqa(B, Hq, Hkv, max_pages * page_size, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    st = lib.fd_decode_gqa_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                 _ptr(seqlens), B, Hq, Hkv, d, page_size, max_pages, num_pages,
                                 DTYPE_CODE[q.dtype], int(num_splits), float(scale), _ptr(out),
                                 DTYPE_CODE[out.dtype], _ptr(lse), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(q, stream))
    _check(st, "fd_decode_gqa_paged")
    return out, lse


def workspace_size_gqa(B, Hq, Hkv, N, d, num_splits=0) -> int:
    return load().fd_workspace_size_gqa(B, Hq, Hkv, N, d, num_splits)


def decode_fp8(q, k, v, k_scale, v_scale, seqlens=None, num_splits=0, scale=None, out_dtype=None,
               out=None, lse=None, return_lse=True, workspace=None, stream=None):
    """fd_decode over an E4M3 KV cache with per-(b,h) scales (fd_decode_fp8).

    k, v: [B,H,N,d] torch.float8_e4m3fn (or uint8 holding E4M3 bytes);
    k_scale, v_scale: float32 [B,H]; q: float32/float16/bfloat16 [B,H,d].
    Returns ``(out, lse)``.
    """
    _need_cuda(q, k, v, k_scale, v_scale, seqlens)
    if q.dtype not in DTYPE_CODE:
        raise ValueError("q must be float32, float16 or bfloat16")
    if k.dtype not in (torch.float8_e4m3fn, torch.uint8) or v.dtype != k.dtype:
        raise ValueError("k, v must be float8_e4m3fn (or uint8 E4M3 bytes)")
    if k.dim() != 4 or v.shape != k.shape or q.shape != (k.shape[0], k.shape[1], k.shape[3]):
        raise ValueError("shapes: q [B,H,d], k/v [B,H,N,d]")
    B, H, N, d = k.shape
    for t in (k_scale, v_scale):
        if t.dtype != torch.float32 or t.shape != (B, H):
            raise ValueError("k_scale/v_scale must be float32 [B,H]")
    if seqlens is not None and (seqlens.dtype != torch.int32 or seqlens.shape != (B,)):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, d), dtype=odt, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    lib = load()
    need = lib.fd_workspace_size(B, H, N, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    st = lib.fd_decode_fp8(_ptr(q), DTYPE_CODE[q.dtype], _ptr(k), _ptr(v), _ptr(k_scale),
                           _ptr(v_scale), _ptr(seqlens), B, H, N, d, int(num_splits), float(scale),
                           _ptr(out), DTYPE_CODE[out.dtype], _ptr(lse), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(q, stream))
    _check(st, "fd_decode_fp8")
    return out, lse



def decode_gqa_fp8(q, k, v, k_scale, v_scale, seqlens=None, num_splits=0, scale=None, out_dtype=None,
                   out=None, lse=None, return_lse=True, workspace=None, stream=None):
    """Grouped-query decode over an E4M3 KV cache (fd_decode_gqa_fp8).

    q: float32/float16/bfloat16 [B, Hq, d]; k, v: [B, Hkv, N, d]
    torch.float8_e4m3fn (or uint8 E4M3 bytes) with Hq a multiple of Hkv, d
    64, 128 or 256; k_scale, v_scale: float32 [B, Hkv].  Returns ``(out, lse)``.
    """
    _need_cuda(q, k, v, k_scale, v_scale, seqlens)
    if q.dtype not in DTYPE_CODE:
        raise ValueError("q must be float32, float16 or bfloat16")
    if k.dtype not in (torch.float8_e4m3fn, torch.uint8) or v.dtype != k.dtype:
        raise ValueError("k, v must be float8_e4m3fn (or uint8 E4M3 bytes)")
    if k.dim() != 4 or v.shape != k.shape or q.dim() != 3 or q.shape[0] != k.shape[0] \
            or q.shape[2] != k.shape[3] or q.shape[1] % k.shape[1]:
        raise ValueError("shapes: q [B,Hq,d], k/v [B,Hkv,N,d], Hq % Hkv == 0")
    B, Hkv, N, d = k.shape
    Hq = q.shape[1]
    for t in (k_scale, v_scale):
        if t.dtype != torch.float32 or t.shape != (B, Hkv):
            raise ValueError("k_scale/v_scale must be float32 [B,Hkv]")
    if seqlens is not None and (seqlens.dtype != torch.int32 or seqlens.shape != (B,)):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, d), dtype=odt, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    lib = load()
    need = lib.fd_workspace_size_gqa(B, Hq, Hkv, N, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    st = lib.fd_decode_gqa_fp8(_ptr(q), DTYPE_CODE[q.dtype], _ptr(k), _ptr(v), _ptr(k_scale),
                               _ptr(v_scale), _ptr(seqlens), B, Hq, Hkv, N, d, int(num_splits),
                               float(scale), _ptr(out), DTYPE_CODE[out.dtype], _ptr(lse),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(q, stream))
    _check(st, "fd_decode_gqa_fp8")
    return out, lse



def decode_gqa_paged_fp8(q, k_pages, v_pages, k_scale, v_scale, block_table, seqlens, num_splits=0,
                         scale=None, out_dtype=None, out=None, lse=None, return_lse=True, workspace=None,
                         stream=None):
    """Grouped-query decode over a paged E4M3 KV cache (fd_decode_gqa_paged_fp8).

    q: float32/float16/bfloat16 [B, Hq, d]; k_pages/v_pages [num_pages, Hkv,
    page_size, d] torch.float8_e4m3fn (or uint8 E4M3 bytes), d 64, 128 or
    256, page_size 16 or a multiple of 32; k_scale, v_scale float32 [B, Hkv]; block_table int32
    [B, max_pages]; seqlens int32 [B].  Returns ``(out, lse)``.
    """
    _need_cuda(q, k_pages, v_pages, k_scale, v_scale, block_table, seqlens)
    if q.dtype not in DTYPE_CODE:
        raise ValueError("q must be float32, float16 or bfloat16")
    if k_pages.dtype not in (torch.float8_e4m3fn, torch.uint8) or v_pages.dtype != k_pages.dtype:
        raise ValueError("pages must be float8_e4m3fn (or uint8 E4M3 bytes)")
    if k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages/v_pages must be [num_pages, Hkv, page_size, d]")
    num_pages, Hkv, page_size, d = k_pages.shape
    B, Hq = q.shape[0], q.shape[1]
    if q.dim() != 3 or q.shape[2] != d or Hq % Hkv:
        raise ValueError("q must be [B, Hq, d] with Hq a multiple of the pages' Hkv")
    for t in (k_scale, v_scale):
        if t.dtype != torch.float32 or t.shape != (B, Hkv):
            raise ValueError("k_scale/v_scale must be float32 [B,Hkv]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seqlens.dtype != torch.int32 or seqlens.shape != (B,):
        raise ValueError("seqlens must be an int32 tensor of shape [B]")
    max_pages = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, d), dtype=odt, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    lib = load()
    need = lib.fd_workspace_size_gqa(B, Hq, Hkv, max_pages * page_size, d, int(num_splits))
    if workspace is None:
        workspace = _cached_workspace(q.device, need)
    st = lib.fd_decode_gqa_paged_fp8(_ptr(q), DTYPE_CODE[q.dtype], _ptr(k_pages), _ptr(v_pages),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seqlens), B, Hq,
                                     Hkv, d, page_size, max_pages, num_pages, int(num_splits), float(scale),
                                     _ptr(out), DTYPE_CODE[out.dtype], _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(q, stream))
    _check(st, "fd_decode_gqa_paged_fp8")
    return out, lse


def decode_split(q, k, v, num_splits, seqlens=None, scale=None, stream=None, o_part=None,
                 m_part=None, l_part=None, lse_part=None):
    """Stage 1 alone (fd_decode_split).  Returns ``(o_part, m_part, l_part, lse_part)``.

    The partial buffers may be passed in (float32, [B,H,P,d] and [B,H,P]);
    those not given are allocated."""
    B, H, N, d = _check_qkv(q, k, v, seqlens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    P = int(num_splits)
    dev = q.device
    if o_part is None:
        o_part = torch.empty((B, H, P, d), dtype=torch.float32, device=dev)
    for t in (m_part, l_part, lse_part):
        if t is not None and (t.shape != (B, H, P) or t.dtype != torch.float32
                              or not t.is_contiguous()):
            raise ValueError("m_part / l_part / lse_part must be contiguous float32 [B,H,P]")
    if o_part.shape != (B, H, P, d) or o_part.dtype != torch.float32 or not o_part.is_contiguous():
        raise ValueError("o_part must be contiguous float32 [B,H,P,d]")
    if m_part is None:
        m_part = torch.empty((B, H, P), dtype=torch.float32, device=dev)
    if l_part is None:
        l_part = torch.empty((B, H, P), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, H, P), dtype=torch.float32, device=dev)
    _need_cuda(o_part, m_part, l_part, lse_part)
    st = load().fd_decode_split(_ptr(q), _ptr(k), _ptr(v), _ptr(seqlens), B, H, N, d,
                                DTYPE_CODE[q.dtype], P, float(scale), _ptr(o_part), _ptr(m_part),
                                _ptr(l_part), _ptr(lse_part), _stream(q, stream))
    _check(st, "fd_decode_split")
    return o_part, m_part, l_part, lse_part


def _combine_out(o_part, out_dtype, out, lse, return_lse):
    B, H, P, d = o_part.shape
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype or torch.float32, device=o_part.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=o_part.device)
    _need_cuda(out, lse)
    return B, H, P, d, out, lse


def combine_mlo(o_part, m_part, l_part, out_dtype=None, out=None, lse=None, return_lse=True,
                stream=None):
    """Stage 2, m/l/o merge (fd_combine_mlo).  Returns ``(out, lse)``."""
    _need_cuda(o_part, m_part, l_part)
    B, H, P, d, out, lse = _combine_out(o_part, out_dtype, out, lse, return_lse)
    for t in (o_part, m_part, l_part):
        if t.dtype != torch.float32:
            raise ValueError("partials must be float32")
    if m_part.shape != (B, H, P) or l_part.shape != (B, H, P):
        raise ValueError("m_part/l_part must be [B,H,P]")
    st = load().fd_combine_mlo(_ptr(o_part), _ptr(m_part), _ptr(l_part), B, H, P, d, _ptr(out),
                               DTYPE_CODE[out.dtype], _ptr(lse), _stream(o_part, stream))
    _check(st, "fd_combine_mlo")
    return out, lse


def combine_lse(o_part, lse_part, out_dtype=None, out=None, lse=None, return_lse=True,
                stream=None):
    """Stage 2, LSE merge (fd_combine_lse).  Returns ``(out, lse)``."""
    _need_cuda(o_part, lse_part)
    B, H, P, d, out, lse = _combine_out(o_part, out_dtype, out, lse, return_lse)
    for t in (o_part, lse_part):
        if t.dtype != torch.float32:
            raise ValueError("partials must be float32")
    if lse_part.shape != (B, H, P):
        raise ValueError("lse_part must be [B,H,P]")
    st = load().fd_combine_lse(_ptr(o_part), _ptr(lse_part), B, H, P, d, _ptr(out),
                               DTYPE_CODE[out.dtype], _ptr(lse), _stream(o_part, stream))
    _check(st, "fd_combine_lse")
    return out, lse


def merge_lse(o_a, lse_a, o_b, lse_b, out=None, lse=None, stream=None):
    """(o_a, lse_a) (+) (o_b, lse_b) row by row (fd_merge_lse).  Returns ``(out, lse)``.

    o_*: float32 [..., d]; lse_*: float32 [...] (same leading shape).  ``out``
    / ``lse`` may be ``o_a`` / ``lse_a`` for an in-place fold.
    """
    _need_cuda(o_a, lse_a, o_b, lse_b)
    for t in (o_a, lse_a, o_b, lse_b):
        if t.dtype != torch.float32:
            raise ValueError("partials must be float32")
    if o_b.shape != o_a.shape or lse_a.shape != o_a.shape[:-1] or lse_b.shape != lse_a.shape:
        raise ValueError("shapes: o [..., d], lse [...]")
    d = o_a.shape[-1]
    rows = lse_a.numel()
    if out is None:
        out = torch.empty_like(o_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    _need_cuda(out, lse)
    st = load().fd_merge_lse(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, d, _ptr(out),
                             _ptr(lse), _stream(o_a, stream))
    _check(st, "fd_merge_lse")
    return out, lse


def selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self-test (fd_selftest_wait_timeout): a kernel
    whose wait nothing completes gives up after the kernels' wait limit (1 s)
    and records FD_ERR_DEVICE_TIMEOUT, read back by device_status()."""
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = load().fd_selftest_wait_timeout(ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise FDError(rc, "fd_selftest_wait_timeout")


def device_status(reset: bool = True) -> int:
    """FD_OK, or FD_ERR_DEVICE_TIMEOUT if a kernel gave up waiting (synchronises)."""
    return load().fd_device_status(1 if reset else 0)
