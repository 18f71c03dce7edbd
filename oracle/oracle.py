"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this module.  The product path (the CUDA
library ``libfa_gb300.so`` and its Python binding) never imports it, and the
two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain C, IEEE double); this file
builds that library with gcc on first use, converts the fp16 / bf16 input bit
patterns to exact doubles, and loops over (batch, head).  It computes the
textbook definition of scaled-dot-product attention described in the
flash-attention-cuda README ("What is Attention?", "The Problem", and the
causal row of the "Kernel design" table): explicit scores, max-subtracted
softmax, weighted sum of the value rows.

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            lib.oracle_attention_head.argtypes = [
                dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                ctypes.c_int, ctypes.c_double, lp, ctypes.c_long, dp]
            lib.oracle_attention_head.restype = ctypes.c_int
            lib.oracle_decode_head.argtypes = [
                dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                ctypes.c_double, dp]
            lib.oracle_decode_head.restype = ctypes.c_int
            lib.oracle_lse_head.argtypes = [dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_double, dp]
            lib.oracle_lse_head.restype = ctypes.c_int
            lib.oracle_backward_head.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                 dp, dp, dp]
            lib.oracle_backward_head.restype = ctypes.c_int
            _lib = lib
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


# --------------------------------------------------------------------------
# Exact decoding of the 16-bit input formats into float64.
# --------------------------------------------------------------------------
def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> exact float64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values.

    bfloat16 is the upper half of an IEEE binary32, so shifting the pattern
    left by 16 bits gives the binary32 with the same value.
    """
    b32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b32.view(np.float32).astype(np.float64)


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f16_bits_to_f64(bits)
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    raise ValueError(f"unknown 16-bit dtype {dtype!r}")


# --------------------------------------------------------------------------
# Prefill (batched, multi-head) and decode.
# --------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
              scale: float, rows=None, threads: int = 1) -> np.ndarray:
    """O = softmax(scale * Q K^T [causal mask]) V for every (batch, head).

    q: float64 [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d] (or [N, d] for one head).
    Grouped heads: Hq must be a multiple of Hkv, and query head h reads key /
    value head h // (Hq // Hkv) -- the result equals repeating every key /
    value head Hq // Hkv times in place, the host-side repeat that the
    flash-attention-cuda README's "Future work" (kernel-side GQA) refers to.
    Causal with Nq != Nk: query i sees key j iff j <= i + (Nk - Nq).
    rows: None (all rows) or a sequence of query indices, the same for every
    head; the result then has shape [B, Hq, len(rows), d].
    threads: heads are independent, so they may be spread over host threads.
    """
    single = q.ndim == 2
    if single:
        q, k, v = q[None, None], k[None, None], v[None, None]
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, H, n_q, d = q.shape
    h_kv, n_k = k.shape[1], k.shape[2]
    if H % h_kv != 0 or v.shape[:3] != k.shape[:3] or k.shape[0] != B:
        raise ValueError("bad shapes: q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] with Hkv | Hq")
    group = H // h_kv
    if rows is None:
        row_arr = None
        n_rows = n_q
    else:
        row_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.int_)
        n_rows = len(row_arr)
    out = np.zeros((B, H, n_rows, d), dtype=np.float64)
    lib = _load()
    rows_ptr = (row_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
                if row_arr is not None else None)

    def one(bh):
        b, h = divmod(bh, H)
        o = np.zeros((n_rows, d), dtype=np.float64)
        hk = h // group
        rc = lib.oracle_attention_head(
            _dptr(q[b, h]), _dptr(k[b, hk]), _dptr(v[b, hk]), _dptr(o),
            n_q, n_k, d, int(bool(causal)), float(scale), rows_ptr, n_rows, None)
        if rc != 0:
            raise RuntimeError("oracle_attention_head failed")
        out[b, h] = o

    if threads > 1 and B * H > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(B * H)))
    else:
        for bh in range(B * H):
            one(bh)
    return out[0, 0] if single else out


def attention_varlen(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens_q,
                     cu_seqlens_k, causal: bool, scale: float, threads: int = 1) -> np.ndarray:
    """Packed variable-length batch: sequence b owns query tokens
    [cu_q[b], cu_q[b+1]) and key tokens [cu_k[b], cu_k[b+1]).

    q: float64 [total_q, Hq, d]; k, v: [total_k, Hkv, d]; returns [total_q, Hq, d].
    Each sequence is an independent problem with its own lengths (causal
    alignment and grouped heads as in ``attention``); sequences never see
    each other's keys.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    if len(cq) != len(ck) or cq[0] != 0 or ck[0] != 0:
        raise ValueError("cu_seqlens must start at 0 and have B + 1 entries each")
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(len(cq) - 1):
        if cq[b + 1] == cq[b]:
            continue
        qs = q[cq[b]:cq[b + 1]].transpose(1, 0, 2)[None]      # [1, Hq, nq, d]
        ks = k[ck[b]:ck[b + 1]].transpose(1, 0, 2)[None]
        vs = v[ck[b]:ck[b + 1]].transpose(1, 0, 2)[None]
        if ks.shape[2] == 0:
            continue                                           # no keys: zero rows
        o = attention(qs, ks, vs, causal, scale, threads=threads)
        out[cq[b]:cq[b + 1]] = o[0].transpose(1, 0, 2)
    return out


def attention_weights(q: np.ndarray, k: np.ndarray, causal: bool, scale: float,
                      rows=None) -> np.ndarray:
    """The softmax weight rows P[i, :] of one head (zero where masked)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    n_q, d = q.shape
    n_k = k.shape[0]
    if rows is None:
        rows = np.arange(n_q)
    row_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.int_)
    n_rows = len(row_arr)
    v = np.zeros((n_k, d), dtype=np.float64)
    o = np.zeros((n_rows, d), dtype=np.float64)
    p = np.zeros((n_rows, n_k), dtype=np.float64)
    rc = _load().oracle_attention_head(
        _dptr(q), _dptr(k), _dptr(v), _dptr(o), n_q, n_k, d, int(bool(causal)),
        float(scale), row_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
        n_rows, _dptr(p))
    if rc != 0:
        raise RuntimeError("oracle_attention_head failed")
    return p


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
           seq_lens, scale: float, threads: int = 1) -> np.ndarray:
    """Decode: each (b, h) query row attends over cache rows [0, seq_lens[b]).

    q: [B, Hq, 1, d] (or [B, Hq, d]); caches: [B, Hkv, max_len, d] with Hkv | Hq
    (query head h reads cache head h // (Hq // Hkv)); returns [B, Hq, 1, d].
    """
    k_cache = np.ascontiguousarray(k_cache, dtype=np.float64)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.float64)
    B, h_kv, max_len, d = k_cache.shape
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(B, -1, d)
    H = q.shape[1]
    if H % h_kv != 0 or v_cache.shape != k_cache.shape:
        raise ValueError("bad shapes: q [B,Hq,1,d], caches [B,Hkv,L,d] with Hkv | Hq")
    group = H // h_kv
    lens = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
    out = np.zeros((B, H, 1, d), dtype=np.float64)
    lib = _load()

    def one(bh):
        b, h = divmod(bh, H)
        hk = h // group
        o = np.zeros(d, dtype=np.float64)
        rc = lib.oracle_decode_head(_dptr(q[b, h]), _dptr(k_cache[b, hk]),
                                    _dptr(v_cache[b, hk]), int(lens[b]), max_len,
                                    d, float(scale), _dptr(o))
        if rc != 0:
            raise RuntimeError("oracle_decode_head failed")
        out[b, h, 0] = o

    if threads > 1 and B * H > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(B * H)))
    else:
        for bh in range(B * H):
            one(bh)
    return out


# --------------------------------------------------------------------------
# Training: the log-sum-exp of the forward, and the backward pass.
# --------------------------------------------------------------------------
def attention_lse(q: np.ndarray, k: np.ndarray, causal: bool, scale: float) -> np.ndarray:
    """lse[b, h, i] = log sum_{j visible} exp(scale * q_i . k_j); -inf for an empty row.

    q: [B, H, Nq, d]; k: [B, H, Nk, d].
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    B, H, n_q, d = q.shape
    n_k = k.shape[2]
    out = np.zeros((B, H, n_q), dtype=np.float64)
    lib = _load()
    for b in range(B):
        for h in range(H):
            o = np.zeros(n_q, dtype=np.float64)
            if lib.oracle_lse_head(_dptr(q[b, h]), _dptr(k[b, h]), n_q, n_k, d,
                                   int(bool(causal)), float(scale), _dptr(o)) != 0:
                raise RuntimeError("oracle_lse_head failed")
            out[b, h] = o
    return out


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                       causal: bool, scale: float, threads: int = 1):
    """(dQ, dK, dV) of O = softmax(scale Q K^T [mask]) V for the upstream gradient dO.

    q, dout: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d] (float64), Hkv | Hq with
    query head h reading key/value head h // (Hq // Hkv) as in ``attention``;
    the gradient of a shared key/value head is the sum over the query heads
    that read it (the chain rule through the repeat).  Causal alignment as in
    ``attention``.  Heads are independent and may be spread over threads.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    dout = np.ascontiguousarray(dout, dtype=np.float64)
    B, H, n_q, d = q.shape
    h_kv, n_k = k.shape[1], k.shape[2]
    if H % h_kv != 0:
        raise ValueError("Hkv must divide Hq")
    group = H // h_kv
    dq = np.zeros_like(q)
    dk_h = np.zeros((B, H, n_k, d))   # per query head, summed into the shared heads below
    dv_h = np.zeros((B, H, n_k, d))
    lib = _load()

    def one(bh):
        b, h = divmod(bh, H)
        hk = h // group
        a, bb, c = np.zeros((n_q, d)), np.zeros((n_k, d)), np.zeros((n_k, d))
        if lib.oracle_backward_head(_dptr(q[b, h]), _dptr(k[b, hk]), _dptr(v[b, hk]),
                                    _dptr(dout[b, h]), n_q, n_k, d, int(bool(causal)),
                                    float(scale), _dptr(a), _dptr(bb), _dptr(c)) != 0:
            raise RuntimeError("oracle_backward_head failed")
        dq[b, h], dk_h[b, h], dv_h[b, h] = a, bb, c

    if threads > 1 and B * H > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(B * H)))
    else:
        for bh in range(B * H):
            one(bh)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(H):          # in query-head order
        dk[:, h // group] += dk_h[:, h]
        dv[:, h // group] += dv_h[:, h]
    return dq, dk, dv
