"""ctypes binding over libfa_gb300.so (C ABI declared in include/fa.h).

The ``fa_*`` functions mirror the C entry points one to one (pointers as
Python ints, streams as ints).  ``prefill`` / ``decode`` are the two calls of
the flash-attention-cuda README's usage section, taking torch tensors: they
only check and marshal arguments, allocate the output, and call the library.
Every step of the computation runs in the library's CUDA kernels; if the
library is missing this module raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

FA_F16, FA_BF16, FA_F32 = 0, 1, 2
FA_FLAG_NONE, FA_FLAG_NO_CAUSAL_SKIP = 0, 1
FA_FLAG_SCHEDULE_UNITS, FA_FLAG_SCHEDULE_STREAM_K = 2, 4
FA_BWD_FLAG_NONE, FA_BWD_RECOMPUTE_DQ = 0, 1
FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_SHAPE", 3: "FA_ERR_HEAD_DIM",
    4: "FA_ERR_DTYPE", 5: "FA_ERR_ALIGN", 6: "FA_ERR_SCALE", 7: "FA_ERR_ARCH",
    8: "FA_ERR_WORKSPACE", 9: "FA_ERR_CUDA", 10: "FA_ERR_WATCHDOG",
    11: "FA_ERR_SEQ_LEN", 12: "FA_ERR_ALIAS", 13: "FA_ERR_SPLITS",
}
(FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEAD_DIM, FA_ERR_DTYPE, FA_ERR_ALIGN, FA_ERR_SCALE, FA_ERR_ARCH,
 FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_WATCHDOG, FA_ERR_SEQ_LEN, FA_ERR_ALIAS,
 FA_ERR_SPLITS) = range(1, 14)

_lock = threading.Lock()
_lib = None

_vp, _i, _f, _u, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint, ctypes.c_size_t
_SIGNATURES = {
    "fa_prefill": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_prefill_ex": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_prefill_gqa": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _u, _vp]),
    "fa_prefill_host": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _u, _vp]),
    "fa_prefill_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                               _f, _i, _i, _u, _vp]),
    "fa_prefill_lse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _u,
                            _vp]),
    "fa_prefill_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                 _i, _f, _i, _i, _vp]),
    "fa_prefill_backward_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                    _i, _f, _i, _i, _u, _vp]),
    "fa_prefill_plan": (_i, [_i, _i, _i, _i, _i, _u, _i, _vp, _vp, _i]),
    "fa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp]),
    "fa_decode_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _sz, _vp]),
    "fa_decode_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _sz,
                           _vp]),
    "fa_decode_gqa_choose_splits": (_i, [_i, _i, _i, _i, _i]),
    "fa_decode_splits_for_sms": (_i, [_i, _i, _i, _i, _i]),
    "fa_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp]),
    "fa_decode_noalloc_max_bytes": (_sz, []),
    "fa_decode_choose_splits": (_i, [_i, _i, _i, _i]),
    "fa_decode_chunk_len": (_i, [_i, _i]),
    "fa_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_last_cuda_error": (_i, []),
    "fa_device_status": (_i, [_i]),
    "fa_watchdog_selftest": (_i, [ctypes.c_longlong, _vp, _vp]),
    "fa_pool_stats": (_i, [_vp, _i]),
    "fa_read_probe": (_i, [_vp, _sz, _vp, _vp]),
    "fa_version": (_i, []),
}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({status_string(status)})")


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load libfa_gb300.so (building it first only if asked)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(
                        f"{path} is missing: build it with attention_forward_prefill_gb300.build"
                        ".build() (there is no CPU fallback)")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


# ---------------------------------------------------------------- raw C ABI
def fa_prefill(q, k, v, out, B, H, N, d, causal, scale, stream=0) -> int:
    return load().fa_prefill(q, k, v, out, B, H, N, d, int(causal), float(scale), stream)


def fa_prefill_ex(q, k, v, out, B, H, N, d, causal, scale, in_dtype, out_dtype,
                  stream=0) -> int:
    return load().fa_prefill_ex(q, k, v, out, B, H, N, d, int(causal), float(scale),
                                in_dtype, out_dtype, stream)


def fa_prefill_gqa(q, k, v, out, B, Hq, Hkv, Nq, Nk, d, causal, scale, in_dtype, out_dtype,
                   flags=0, stream=0) -> int:
    return load().fa_prefill_gqa(q, k, v, out, B, Hq, Hkv, Nq, Nk, d, int(causal), float(scale),
                                 in_dtype, out_dtype, flags, stream)


def fa_prefill_host(q, k, v, out, B, Hq, Hkv, Nq, Nk, d, causal, scale, in_dtype, out_dtype,
                    flags=0, stream=0) -> int:
    return load().fa_prefill_host(q, k, v, out, B, Hq, Hkv, Nq, Nk, d, int(causal), float(scale),
                                  in_dtype, out_dtype, flags, stream)


def fa_prefill_varlen(q, k, v, out, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q, total_k,
                      max_seqlen_q, max_seqlen_k, d, causal, scale, in_dtype, out_dtype, flags=0,
                      stream=0) -> int:
    return load().fa_prefill_varlen(q, k, v, out, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q,
                                    total_k, max_seqlen_q, max_seqlen_k, d, int(causal),
                                    float(scale), in_dtype, out_dtype, flags, stream)


def fa_prefill_lse(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, in_dtype, out_dtype,
                   flags=0, stream=0) -> int:
    return load().fa_prefill_lse(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, d, int(causal),
                                 float(scale), in_dtype, out_dtype, flags, stream)


def fa_prefill_backward(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                        in_dtype, grad_dtype, stream=0) -> int:
    return load().fa_prefill_backward(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, N, d,
                                      int(causal), float(scale), in_dtype, grad_dtype, stream)


def fa_prefill_backward_ex(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                           in_dtype, grad_dtype, flags=0, stream=0) -> int:
    return load().fa_prefill_backward_ex(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, N, d,
                                         int(causal), float(scale), in_dtype, grad_dtype, flags,
                                         stream)


def fa_prefill_plan(B, Hq, Nq, Nk, causal, flags=0, num_sms=0, max_items=192):
    """The prefill schedule as (status, info[9], items[n][5]) -- host arithmetic only."""
    info = (ctypes.c_longlong * 9)()
    items = (ctypes.c_longlong * (5 * max_items))()
    rc = load().fa_prefill_plan(B, Hq, Nq, Nk, int(causal), flags, num_sms, info, items, max_items)
    n = int(info[5]) if rc == FA_OK else 0
    rows = [tuple(int(items[5 * i + c]) for c in range(5)) for i in range(min(n, max_items))]
    return rc, [int(x) for x in info], rows


def fa_decode(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d, scale, stream=0) -> int:
    return load().fa_decode(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d,
                            float(scale), stream)


def fa_decode_ex(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d, scale, in_dtype,
                 out_dtype, num_splits=0, workspace=None, workspace_bytes=0, stream=0) -> int:
    return load().fa_decode_ex(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d,
                               float(scale), in_dtype, out_dtype, num_splits, workspace,
                               workspace_bytes, stream)


def fa_decode_gqa(q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, max_len, d, scale, in_dtype,
                  out_dtype, num_splits=0, workspace=None, workspace_bytes=0, stream=0) -> int:
    return load().fa_decode_gqa(q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, max_len, d,
                                float(scale), in_dtype, out_dtype, num_splits, workspace,
                                workspace_bytes, stream)


def fa_decode_gqa_choose_splits(B, Hq, Hkv, max_len, device=-1) -> int:
    return load().fa_decode_gqa_choose_splits(B, Hq, Hkv, max_len, device)


def fa_decode_splits_for_sms(B, Hq, Hkv, max_len, num_sms) -> int:
    return load().fa_decode_splits_for_sms(B, Hq, Hkv, max_len, num_sms)


def fa_decode_noalloc(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d, scale, in_dtype,
                      out_dtype, num_splits=0, stream=0) -> int:
    """Decode with the library's static scratch: allocates no device memory."""
    return load().fa_decode_noalloc(q, k_cache, v_cache, seq_lens, out, B, H, max_len, d,
                                    float(scale), in_dtype, out_dtype, num_splits, stream)


def fa_decode_noalloc_max_bytes() -> int:
    return load().fa_decode_noalloc_max_bytes()


def fa_decode_choose_splits(B, H, max_len, device=-1) -> int:
    return load().fa_decode_choose_splits(B, H, max_len, device)


def fa_decode_chunk_len(max_len, num_splits) -> int:
    return load().fa_decode_chunk_len(max_len, num_splits)


def fa_decode_workspace_bytes(B, H, max_len, d, num_splits) -> int:
    return load().fa_decode_workspace_bytes(B, H, max_len, d, num_splits)


def status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


def fa_last_cuda_error() -> int:
    return load().fa_last_cuda_error()


def fa_device_status(reset: bool = False) -> int:
    return load().fa_device_status(int(reset))


def fa_version() -> int:
    return load().fa_version()


def fa_watchdog_selftest(limit_ns, result, stream=0) -> int:
    return load().fa_watchdog_selftest(int(limit_ns), result, stream)


def fa_pool_stats(reset_high: bool = False):
    """(status, [reserved, reserved_high, used, used_high]) of the library's scratch pool."""
    out = (ctypes.c_longlong * 4)()
    rc = load().fa_pool_stats(out, int(reset_high))
    return rc, [int(x) for x in out]


def fa_read_probe(src, nbytes, xor_out, stream=0) -> int:
    return load().fa_read_probe(src, nbytes, xor_out, stream)


# ---------------------------------------------------------------- torch calls
def _torch():
    import torch
    return torch


def dtype_code(dt) -> int:
    torch = _torch()
    if dt == torch.float16:
        return FA_F16
    if dt == torch.bfloat16:
        return FA_BF16
    if dt == torch.float32:
        return FA_F32
    raise TypeError(f"unsupported dtype {dt}")


def _check_cuda(name, t, shape=None, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _stream_handle(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def prefill(q, k, v, causal: bool = False, scale: float | None = None, out_dtype=None,
            flags: int = 0, out=None, sync: bool = True):
    """out = softmax(scale * q k^T [causal]) v for q [B, Hq, Nq, d] and k, v
    [B, Hkv, Nk, d] (fp16/bf16; Hq a multiple of Hkv; causal queries are the
    last Nq positions).

    CUDA inputs run on the current stream and return a CUDA tensor.  Host
    inputs go through fa_prefill_host (copies in, compute and copies out
    pipelined over chunks of heads) on the current stream and return the host
    result (pinned when q is).  With sync (the default) the call waits for the
    stream first; with sync=False it returns at once, like the C call, and the
    result is ready, and the host tensors free to reuse, once the stream has
    passed the call.
    """
    torch = _torch()
    if not q.is_cuda:
        return _prefill_host(torch, q, k, v, causal, scale, out_dtype, flags, out, sync)
    B, Hq, Nq, d = q.shape
    _check_cuda("q", q)
    _check_cuda("k", k, None, q.dtype)
    if k.dim() != 4 or k.shape[0] != B or k.shape[3] != d:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [{B}, Hkv, Nk, {d}]")
    Hkv, Nk = k.shape[1], k.shape[2]
    _check_cuda("v", v, k.shape, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    else:
        _check_cuda("out", out, q.shape, out_dtype)
    rc = fa_prefill_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv, Nq,
                        Nk, d, causal, scale, dtype_code(q.dtype), dtype_code(out_dtype), flags,
                        _stream_handle(q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_prefill_gqa")
    return out


def _check_host(name, t, shape=None, dtype=None):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor when q is")
    if t.dtype not in (_torch().float16, _torch().bfloat16) and name != "out":
        raise ValueError(f"{name} must be float16 or bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _prefill_host(torch, q, k, v, causal, scale, out_dtype, flags, out, sync=True):
    B, Hq, Nq, d = q.shape
    _check_host("q", q)
    _check_host("k", k, None, q.dtype)
    if k.dim() != 4 or k.shape[0] != B or k.shape[3] != d:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [{B}, Hkv, Nk, {d}]")
    Hkv, Nk = k.shape[1], k.shape[2]
    _check_host("v", v, k.shape, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, pin_memory=q.is_pinned())
    else:
        _check_host("out", out, q.shape, out_dtype)
    stream = torch.cuda.current_stream()
    rc = fa_prefill_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv, Nq,
                         Nk, d, causal, scale, dtype_code(q.dtype), dtype_code(out_dtype), flags,
                         stream.cuda_stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_prefill_host")
    if sync:
        stream.synchronize()
    return out


def prefill_with_lse(q, k, v, causal: bool = False, scale: float | None = None, flags: int = 0):
    """Forward for training: returns (out, lse) with out in q's dtype and lse
    fp32 [B, Hq, Nq] (natural-log row log-sum-exp of the visible scores)."""
    torch = _torch()
    B, Hq, Nq, d = q.shape
    _check_cuda("q", q)
    _check_cuda("k", k, None, q.dtype)
    Hkv, Nk = k.shape[1], k.shape[2]
    _check_cuda("v", v, k.shape, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    rc = fa_prefill_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                        Hq, Hkv, Nq, Nk, d, causal, scale, dtype_code(q.dtype), dtype_code(q.dtype),
                        flags, _stream_handle(q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_prefill_lse")
    return out, lse


def prefill_backward(q, k, v, out, dout, lse, causal: bool = False, scale: float | None = None,
                     grad_dtype=None, flags: int = 0):
    """(dq, dk, dv) for square prefill with q, out, dout [B, H, N, d] and k, v
    [B, Hkv, N, d], from the forward's out and lse; dk, dv have k's shape.
    flags: FA_BWD_* bits (FA_BWD_RECOMPUTE_DQ)."""
    torch = _torch()
    B, H, N, d = q.shape
    for name, t in (("q", q), ("out", out), ("dout", dout)):
        _check_cuda(name, t, q.shape, q.dtype)
    _check_cuda("k", k, None, q.dtype)
    if k.dim() != 4 or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [{B}, Hkv, {N}, {d}]")
    _check_cuda("v", v, k.shape, q.dtype)
    Hkv = k.shape[1]
    _check_cuda("lse", lse, (B, H, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    grad_dtype = q.dtype if grad_dtype is None else grad_dtype
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk, dv = (torch.empty(k.shape, dtype=grad_dtype, device=q.device) for _ in range(2))
    rc = fa_prefill_backward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, Hkv, N, d, causal, scale, dtype_code(q.dtype),
                                dtype_code(grad_dtype), flags, _stream_handle(q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_prefill_backward_ex")
    return dq, dk, dv


def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                   causal: bool = False, scale: float | None = None, out_dtype=None,
                   flags: int = 0, out=None):
    """Packed variable-length prefill: q [total_q, Hq, d], k, v [total_k, Hkv, d],
    cu_seqlens_* int32 [B + 1] on the same device.  Returns [total_q, Hq, d]."""
    torch = _torch()
    _check_cuda("q", q)
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q and k must be [tokens, heads, d]")
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    _check_cuda("k", k, (total_k, Hkv, d), q.dtype)
    _check_cuda("v", v, k.shape, q.dtype)
    B = cu_seqlens_q.shape[0] - 1
    _check_cuda("cu_seqlens_q", cu_seqlens_q, (B + 1,), torch.int32)
    _check_cuda("cu_seqlens_k", cu_seqlens_k, (B + 1,), torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    else:
        _check_cuda("out", out, q.shape, out_dtype)
    rc = fa_prefill_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, Hq, Hkv, total_q,
                           total_k, int(max_seqlen_q), int(max_seqlen_k), d, causal, scale,
                           dtype_code(q.dtype), dtype_code(out_dtype), flags,
                           _stream_handle(q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_prefill_varlen")
    return out


def decode(q, k_cache, v_cache, seq_lens, scale: float | None = None, out_dtype=None,
           num_splits: int = 0, workspace=None, out=None):
    """One query row per (b, h) over the first seq_lens[b] rows of the cache.

    q: [B, Hq, 1, d]; caches: [B, Hkv, max_len, d] with Hkv dividing Hq (query
    head h reads cache head h // (Hq // Hkv)); seq_lens: int32 [B] on the same
    device.  Returns [B, Hq, 1, d].
    """
    torch = _torch()
    B, Hkv, max_len, d = k_cache.shape
    _check_cuda("k_cache", k_cache)
    _check_cuda("v_cache", v_cache, k_cache.shape, k_cache.dtype)
    _check_cuda("q", q, None, k_cache.dtype)
    if q.dim() != 4 or q.shape[0] != B or q.shape[2] != 1 or q.shape[3] != d:
        raise ValueError(f"q has shape {tuple(q.shape)}, expected [{B}, Hq, 1, {d}]")
    Hq = q.shape[1]
    _check_cuda("seq_lens", seq_lens, (B,), torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((B, Hq, 1, d), dtype=out_dtype, device=q.device)
    else:
        _check_cuda("out", out, (B, Hq, 1, d), out_dtype)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _check_cuda("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = fa_decode_gqa(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seq_lens.data_ptr(),
                       out.data_ptr(), B, Hq, Hkv, max_len, d, scale, dtype_code(q.dtype),
                       dtype_code(out_dtype), num_splits, ws_ptr, ws_bytes,
                       _stream_handle(q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_decode_gqa")
    return out
