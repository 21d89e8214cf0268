"""Python binding of libattn45.so (the GB300 fused exact attention forward).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/attn45.h``. PyTorch is used for
device memory and streams. There is no CPU fallback: if the library is not
built or the device is not a GB300, calls raise.

Functions carry the C names:

* ``attn_fwd(q, k, v, causal=False, scale=None, out=None, lse=None)``
* ``attn_fwd_varlen(q, k, v, cu_seqlens, causal=False, ...)``
* ``attn_fp8_prepass(q, k, v, mode="block", rotate=True, hadamard_seed=0)``
* ``attn_fwd_fp8(pre, causal=False, scale=None, ...)``
* ``attn_fwd_fp8_auto(q, k, v, workspace=None, ...)``
* ``attn_decode(q, k_cache, v_cache, seqlens, num_splits=0, ...)``
* ``attn_combine(o_parts, lse_parts, dtype=torch.bfloat16)``
* ``attn_bwd(q, k, v, o, lse, dout, causal=False, ...)``
* ``attn_fp8_prepass_varlen(q, k, v, cu_seqlens, ...)``, ``attn_fwd_fp8_varlen(pre, ...)``
* ``attn_get_device_error()``, ``attn_set_wait_timeout_ns(ns)``

``capi()`` returns the raw ctypes handle (pointer-and-size arguments).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

__all__ = [
    "AttnError", "capi", "library_path",
    "attn_fwd", "attn_fwd_varlen", "attn_fp8_prepass", "attn_fwd_fp8", "attn_fwd_fp8_auto",
    "attn_fp8_workspace_size", "attn_fp8_vt_ld", "attn_get_device_error", "attn_set_wait_timeout_ns",
    "attn_debug_timeout_probe", "attn_decode", "attn_decode_num_splits", "attn_decode_workspace_size",
    "attn_combine", "attn_bwd", "attn_bwd_workspace_size", "attn_fp8_varlen_tmax", "attn_fp8_prepass_varlen",
    "attn_fwd_fp8_varlen", "EXPORTED_SYMBOLS",
]

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
_DTYPE = {torch.bfloat16: 0, torch.float16: 1}
_FP8_MODE = {"tensor": 0, "block": 1}

# Every function include/attn45.h declares.
EXPORTED_SYMBOLS = (
    "attn_fwd", "attn_fwd_varlen", "attn_fp8_vt_ld", "attn_fp8_prepass", "attn_fwd_fp8",
    "attn_fp8_workspace_size", "attn_fwd_fp8_auto", "attn_fwd_fp8_auto_noalloc", "attn_get_device_error",
    "attn_set_wait_timeout_ns", "attn_debug_timeout_probe", "attn_status_string", "attn_last_error_message",
    "attn_version", "attn_decode", "attn_decode_num_splits", "attn_decode_workspace_size", "attn_combine",
    "attn_bwd", "attn_bwd_workspace_size", "attn_fp8_varlen_tmax", "attn_fp8_prepass_varlen", "attn_fwd_fp8_varlen",
)


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def capi(build_if_missing: bool = True):
    """Load libattn45.so (compiling it first if absent) and declare signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise AttnError(ATTN_ERR_UNSUPPORTED, f"{path} is not built")
            path = _build.build()
        lib = ctypes.CDLL(path)
        P, I, F, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
        sig = {
            "attn_fwd": ([P, P, P, P, P, I, I, I, I, I, I, F, I, P], I),
            "attn_fwd_varlen": ([P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P], I),
            "attn_fp8_vt_ld": ([I], I),
            "attn_fp8_prepass": ([P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, U64, P], I),
            "attn_fwd_fp8": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P], I),
            "attn_fp8_workspace_size": ([I, I, I, I, I, I], SZ),
            "attn_fwd_fp8_auto": ([P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, I, I, U64, P], I),
            "attn_fwd_fp8_auto_noalloc": ([P, P, P, P, P, I, I, I, I, I, I, F, I, I, U64, P], I),
            "attn_get_device_error": ([P], I),
            "attn_set_wait_timeout_ns": ([U64], I),
            "attn_debug_timeout_probe": ([U64, P], I),
            "attn_status_string": ([I], ctypes.c_char_p),
            "attn_last_error_message": ([], ctypes.c_char_p),
            "attn_version": ([], I),
            "attn_decode": ([P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, I, P], I),
            "attn_decode_num_splits": ([I, I, I], I),
            "attn_decode_workspace_size": ([I, I, I, I], SZ),
            "attn_combine": ([P, P, P, P, I, I, I, I, P], I),
            "attn_bwd": ([P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, I, P], I),
            "attn_bwd_workspace_size": ([I, I, I, I], SZ),
            "attn_fp8_varlen_tmax": ([I, I], I),
            "attn_fp8_prepass_varlen": ([P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, U64, P], I),
            "attn_fwd_fp8_varlen": ([P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int):
    if rc != ATTN_OK:
        lib = capi()
        raise AttnError(rc, lib.attn_last_error_message().decode())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise AttnError(ATTN_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise AttnError(ATTN_ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise AttnError(ATTN_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise AttnError(ATTN_ERR_INVALID_ARG, f"{name} must have {ndim} dims")


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None):
    """O, LSE for q [B,N,H,d], k/v [B,N,Hkv,d] (bf16 or fp16)."""
    _need(q, "q", ndim=4)
    _need(k, "k", q.dtype, 4)
    _need(v, "v", q.dtype, 4)
    if q.dtype not in _DTYPE:
        raise AttnError(ATTN_ERR_INVALID_ARG, "q must be bf16 or fp16")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise AttnError(ATTN_ERR_INVALID_ARG, "k and v must be [B,N,Hkv,d] matching q")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", q.dtype, 4)
    _need(lse, "lse", torch.float32, 3)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(capi().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d, int(bool(causal)),
                           scale, _DTYPE[q.dtype], _stream(stream)))
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens, causal: bool = False, scale: float | None = None, out=None, lse=None,
                    max_seqlen: int = 0, stream=None):
    """O, LSE for packed q [T,H,d], k/v [T,Hkv,d] with int32 cu_seqlens [nseq+1] on the device."""
    _need(q, "q", ndim=3)
    _need(k, "k", q.dtype, 3)
    _need(v, "v", q.dtype, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if q.dtype not in _DTYPE:
        raise AttnError(ATTN_ERR_INVALID_ARG, "q must be bf16 or fp16")
    T, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise AttnError(ATTN_ERR_INVALID_ARG, "k and v must be [T,Hkv,d] matching q")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nseq = cu_seqlens.numel() - 1
    _check(capi().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens), nseq,
                                  int(max_seqlen), T, H, Hkv, d, int(bool(causal)), scale, _DTYPE[q.dtype],
                                  _stream(stream)))
    return out, lse


def attn_fp8_vt_ld(N: int) -> int:
    return int(capi().attn_fp8_vt_ld(N))


def attn_fp8_workspace_size(B, H, Hkv, N, d, mode: str = "block") -> int:
    return int(capi().attn_fp8_workspace_size(B, H, Hkv, N, d, _FP8_MODE[mode]))


def attn_fp8_prepass(q, k, v, mode: str = "block", rotate: bool = True, hadamard_seed: int = 0, stream=None):
    """e4m3 codes and fp32 scales for bf16 q/k/v [B,N,H(kv),d]; returns a dict."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    dev = q.device
    ld = attn_fp8_vt_ld(N)
    nb = (N + 127) // 128
    u8 = torch.uint8
    pre = {
        "q8": torch.empty((B, N, H, d), dtype=u8, device=dev),
        "k8": torch.empty((B, N, Hkv, d), dtype=u8, device=dev),
        "vt8": torch.empty((B, Hkv, d, ld), dtype=u8, device=dev),
        "sq": torch.empty((B, H, nb) if mode == "block" else (1,), dtype=torch.float32, device=dev),
        "sk": torch.empty((B, Hkv, nb) if mode == "block" else (1,), dtype=torch.float32, device=dev),
        "sv": torch.empty((B, Hkv, d) if mode == "block" else (1,), dtype=torch.float32, device=dev),
        "mode": mode, "rotate": rotate, "seed": hadamard_seed,
    }
    _check(capi().attn_fp8_prepass(_ptr(q), _ptr(k), _ptr(v), _ptr(pre["q8"]), _ptr(pre["k8"]), _ptr(pre["vt8"]),
                                   _ptr(pre["sq"]), _ptr(pre["sk"]), _ptr(pre["sv"]), B, H, Hkv, N, d,
                                   _FP8_MODE[mode], int(bool(rotate)), int(hadamard_seed), _stream(stream)))
    return pre


def attn_fwd_fp8(pre: dict, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None):
    """O (bf16) and LSE from attn_fp8_prepass outputs."""
    q8, k8 = pre["q8"], pre["k8"]
    B, N, H, d = q8.shape
    Hkv = k8.shape[2]
    out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(capi().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(pre["vt8"]), _ptr(pre["sq"]), _ptr(pre["sk"]),
                               _ptr(pre["sv"]), _ptr(out), _ptr(lse), B, H, Hkv, N, d, int(bool(causal)), scale,
                               _FP8_MODE[pre["mode"]], _stream(stream)))
    return out, lse


def attn_fwd_fp8_auto(q, k, v, causal: bool = False, scale: float | None = None, mode: str = "block",
                      rotate: bool = True, hadamard_seed: int = 0, workspace=None, out=None, lse=None, stream=None):
    """Pre-pass + FP8 forward in one call; ``workspace`` is a uint8 CUDA tensor."""
    _need(q, "q", torch.bfloat16, 4)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    need = attn_fp8_workspace_size(B, H, Hkv, N, d, mode)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(capi().attn_fwd_fp8_auto(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), B, H, Hkv, N, d,
                                    int(bool(causal)), scale, _FP8_MODE[mode], int(bool(rotate)),
                                    int(hadamard_seed), _stream(stream)))
    return out, lse


def attn_decode_num_splits(B: int, Hkv: int, Nmax: int) -> int:
    return int(capi().attn_decode_num_splits(B, Hkv, Nmax))


def attn_decode_workspace_size(B: int, H: int, d: int, num_splits: int) -> int:
    return int(capi().attn_decode_workspace_size(B, H, d, num_splits))


def attn_decode(q, k_cache, v_cache, seqlens, num_splits: int = 0, scale: float | None = None, workspace=None,
                out=None, lse=None, stream=None):
    """Split-KV decode: q [B,H,d], caches [B,Nmax,Hkv,d], int32 seqlens [B] on the device -> O [B,H,d], lse [B,H]."""
    _need(q, "q", ndim=3)
    _need(k_cache, "k_cache", q.dtype, 4)
    _need(v_cache, "v_cache", q.dtype, 4)
    _need(seqlens, "seqlens", torch.int32, 1)
    if q.dtype not in _DTYPE:
        raise AttnError(ATTN_ERR_INVALID_ARG, "q must be bf16 or fp16")
    B, H, d = q.shape
    Nmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Nmax, Hkv, d) or v_cache.shape != k_cache.shape or seqlens.numel() != B:
        raise AttnError(ATTN_ERR_INVALID_ARG, "caches must be [B,Nmax,Hkv,d] and seqlens [B]")
    if num_splits <= 0:
        num_splits = attn_decode_num_splits(B, Hkv, Nmax)
    need = attn_decode_workspace_size(B, H, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(capi().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(out), _ptr(lse),
                              _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, Hkv, Nmax, d,
                              num_splits, scale, _DTYPE[q.dtype], _stream(stream)))
    return out, lse


def attn_combine(o_parts, lse_parts, dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """Merge fp32 partials o_parts [S, rows..., d], lse_parts [S, rows...] -> O (dtype), lse."""
    _need(o_parts, "o_parts", torch.float32)
    _need(lse_parts, "lse_parts", torch.float32)
    S, d = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel()
    if lse_parts.shape[0] != S or o_parts.numel() != S * rows * d:
        raise AttnError(ATTN_ERR_INVALID_ARG, "o_parts must be [S, rows..., d] matching lse_parts [S, rows...]")
    out = torch.empty(o_parts.shape[1:], dtype=dtype, device=o_parts.device) if out is None else out
    lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device) if lse is None else lse
    _check(capi().attn_combine(_ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse), S, rows, d, _DTYPE[dtype],
                               _stream(stream)))
    return out, lse


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(capi().attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, workspace=None, dq=None,
             dk=None, dv=None, stream=None):
    """dQ, dK, dV of sum(dout * o) for the forward attn_fwd(q, k, v) that returned (o, lse)."""
    _need(q, "q", ndim=4)
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need(t, name, q.dtype, 4)
    _need(lse, "lse", torch.float32, 3)
    if q.dtype not in _DTYPE:
        raise AttnError(ATTN_ERR_INVALID_ARG, "q must be bf16 or fp16")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise AttnError(ATTN_ERR_INVALID_ARG, "shapes must match the forward's (BSHD)")
    need = attn_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(capi().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, Hkv, N, d,
                           int(bool(causal)), scale, _DTYPE[q.dtype], _stream(stream)))
    return dq, dk, dv


def attn_fp8_varlen_tmax(total: int, nseq: int) -> int:
    return int(capi().attn_fp8_varlen_tmax(total, nseq))


def attn_fp8_prepass_varlen(q, k, v, cu_seqlens, mode: str = "block", rotate: bool = True, hadamard_seed: int = 0,
                            stream=None):
    """e4m3 codes and scales of packed bf16 q [T,H,d], k/v [T,Hkv,d] (int32 cu_seqlens on the device); a dict."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, H, d = q.shape
    Hkv = k.shape[1]
    nseq = cu_seqlens.numel() - 1
    tmax = attn_fp8_varlen_tmax(T, nseq)
    dev = q.device
    u8 = torch.uint8
    blk = mode == "block"
    pre = {
        "q8": torch.empty((T, H, d), dtype=u8, device=dev),
        "k8": torch.empty((T, Hkv, d), dtype=u8, device=dev),
        "vt8": torch.empty((Hkv, d, 128 * tmax), dtype=u8, device=dev),   # columns past the last block unused
        "sq": torch.empty((H, tmax) if blk else (1,), dtype=torch.float32, device=dev),
        "sk": torch.empty((Hkv, tmax) if blk else (1,), dtype=torch.float32, device=dev),
        "sv": torch.empty((nseq, Hkv, d) if blk else (1,), dtype=torch.float32, device=dev),
        "blk_off": torch.empty((nseq + 1,), dtype=torch.int32, device=dev),
        "cu_seqlens": cu_seqlens, "tmax": tmax, "mode": mode, "rotate": rotate, "seed": hadamard_seed,
    }
    _check(capi().attn_fp8_prepass_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(pre["q8"]),
                                          _ptr(pre["k8"]), _ptr(pre["vt8"]), _ptr(pre["sq"]), _ptr(pre["sk"]),
                                          _ptr(pre["sv"]), _ptr(pre["blk_off"]), nseq, T, H, Hkv, d, _FP8_MODE[mode],
                                          int(bool(rotate)), int(hadamard_seed), _stream(stream)))
    return pre


def attn_fwd_fp8_varlen(pre: dict, causal: bool = False, scale: float | None = None, out=None, lse=None,
                        stream=None):
    """O [T,H,d] (bf16) and lse [H,T] from attn_fp8_prepass_varlen outputs."""
    q8, k8 = pre["q8"], pre["k8"]
    T, H, d = q8.shape
    Hkv = k8.shape[1]
    cu = pre["cu_seqlens"]
    nseq = cu.numel() - 1
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((H, T), dtype=torch.float32, device=q8.device) if lse is None else lse
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(capi().attn_fwd_fp8_varlen(_ptr(q8), _ptr(k8), _ptr(pre["vt8"]), _ptr(pre["sq"]), _ptr(pre["sk"]),
                                      _ptr(pre["sv"]), _ptr(pre["blk_off"]), _ptr(cu), _ptr(out), _ptr(lse), nseq, T,
                                      H, Hkv, d, int(bool(causal)), scale, _FP8_MODE[pre["mode"]], _stream(stream)))
    return out, lse


def attn_get_device_error(stream=None) -> int:
    """Synchronise ``stream`` and return the device error status (clears it)."""
    return int(capi().attn_get_device_error(_stream(stream)))


def attn_set_wait_timeout_ns(ns: int):
    _check(capi().attn_set_wait_timeout_ns(int(ns)))


def attn_debug_timeout_probe(ns: int, stream=None):
    _check(capi().attn_debug_timeout_probe(int(ns), _stream(stream)))
