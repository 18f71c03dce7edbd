"""fp64 model of the *method* (tiled online softmax, split merges) -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module.  It is not the oracle: the oracle
(``attn_oracle.c``) is the plain definition with explicit score rows.  This
module restates, in float64 numpy, the recurrence that the fused kernels run,
so that a CPU test can show -- before any GPU number is trusted -- that the
recurrence reaches the same answer as the definition:

* flash-attention-cuda README, "What is Flash Attention?": the score table is
  never held whole; keys are visited block after block while each row keeps a
  running maximum and a running sum;
* same README, "Kernel design" table, online-softmax row: m and l are running
  per-row values, and the output accumulator is rescaled when the maximum
  moves.  Here the rescale is *lazy*: the reference maximum m_ref only moves
  (and O, l are multiplied by alpha = 2^(m_ref_old - m_ref_new)) when a block's
  maximum exceeds m_ref by more than tau (log2 units); otherwise the stale
  m_ref is kept, which leaves O / l unchanged mathematically.  tau = 0 is the
  eager form;
* same README, "What did I implement?" and the split-K / two-pass-merge rows of
  "Kernel design": a long key range is cut into chunks, each chunk produces a
  partial (m_s, l_s, acc_s), and the partials are merged exactly by
  M = max_s m_s, O = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s.
  The prefill schedule that cuts a query tile's key range between two workers
  uses the same merge.

It also models the rounding points of the tensor-core path (the weights p
rounded to the 16-bit input type before the P.V product, l summed over the
rounded weights, the output rounded to nearest even), which predicts how large
the GPU's deviation from the oracle should be.

All scores live in the log2 domain: t = s * scale * log2(e), p = 2^(t - m_ref).
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


# --------------------------------------------------------------- rounding
def round_to(x: np.ndarray, dtype: str | None) -> np.ndarray:
    """Round float64 values to the nearest value of ``dtype`` (ties to even).

    dtype: None (keep fp64), "f32", "f16" or "bf16".  fp16 / fp32 rounding is
    numpy's IEEE conversion.  bf16 is the upper half of a binary32: the value is
    first rounded to binary32, then the low 16 bits are rounded away to even.
    """
    if dtype is None:
        return np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
        lsb = (b >> np.uint64(16)) & np.uint64(1)
        b = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16) << np.uint64(16)
        return (b.astype(np.uint32)).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# ------------------------------------------------------- blockwise recurrence
def _visible(n_q: int, n_k: int, causal: bool, causal_offset: int):
    """Boolean [n_q, n_k]: key j visible to query i (causal: j <= i + offset)."""
    if not causal:
        return np.ones((n_q, n_k), dtype=bool)
    i = np.arange(n_q)[:, None]
    j = np.arange(n_k)[None, :]
    return j <= i + causal_offset


def partial_over_keys(q, k, v, scale, visible, j_begin, j_end, block=128, tau=8.0,
                      p_dtype=None, l_from_rounded=True):
    """Run the online recurrence for every query row over keys [j_begin, j_end).

    q: [n_q, d]; k, v: [n_k, d]; visible: bool [n_q, n_k].
    Returns the unnormalised state (o, m_ref, l): o [n_q, d] and m_ref, l [n_q],
    with m_ref = -inf and l = 0 for a row that saw no visible key.
    p_dtype: None for exact fp64 weights, else the 16-bit type the weights are
    rounded to before they enter P.V; l sums the rounded weights unless
    l_from_rounded is False (then l sums the unrounded ones).
    """
    n_q, d = q.shape
    c = scale * LOG2E
    o = np.zeros((n_q, d))
    m_ref = np.full(n_q, -np.inf)
    l = np.zeros(n_q)
    for j0 in range(j_begin, j_end, block):
        j1 = min(j0 + block, j_end)
        t = (q @ k[j0:j1].T) * c                       # [n_q, bj] block of scaled scores
        t = np.where(visible[:, j0:j1], t, -np.inf)
        m_blk = t.max(axis=1)
        empty = np.isinf(m_ref)                        # nothing accumulated yet
        move = (m_blk > m_ref + tau) | (empty & ~np.isinf(m_blk))
        m_new = np.where(move, m_blk, m_ref)
        with np.errstate(invalid="ignore"):
            alpha = np.where(empty, 0.0, np.where(move, np.exp2(m_ref - m_new), 1.0))
            o *= alpha[:, None]
            l *= alpha
            m_ref = m_new
            p_exact = np.where(np.isinf(t), 0.0, np.exp2(t - m_ref[:, None]))
        p = round_to(p_exact, p_dtype)
        l += (p if l_from_rounded else p_exact).sum(axis=1)
        o += p @ v[j0:j1]
    return o, m_ref, l


def merge_partials(parts):
    """Exact merge of partial states [(o, m_ref, l), ...] in the given order.

    M = max m; w_s = 2^(m_s - M) (0 for a part that saw nothing);
    returns (sum_s w_s o_s, M, sum_s w_s l_s).
    """
    ms = np.stack([p[1] for p in parts])               # [S, n_q]
    big = ms.max(axis=0)
    o = np.zeros_like(parts[0][0])
    l = np.zeros_like(parts[0][2])
    for (o_s, m_s, l_s) in parts:
        with np.errstate(invalid="ignore"):
            w = np.where(np.isinf(m_s), 0.0, np.exp2(m_s - big))
        o += w[:, None] * o_s
        l += w * l_s
    return o, big, l


def finish(o, l, out_dtype=None):
    """O = o / l (a row with l = 0 saw no key and is zero), rounded to out_dtype."""
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return round_to(out, out_dtype)


def tiled_attention(q, k, v, causal, scale, block=128, tau=8.0, cuts=(), causal_offset=None,
                    p_dtype=None, out_dtype=None, l_from_rounded=True):
    """One head by the tiled method.

    cuts: key indices at which the key range is cut into separately computed
    partials that are merged afterwards (the split-K / cut-unit schedules).
    causal_offset: key j is visible to query i iff j <= i + offset; default
    n_k - n_q (bottom-right alignment, 0 for square problems).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, n_k = q.shape[0], k.shape[0]
    off = (n_k - n_q) if causal_offset is None else causal_offset
    vis = _visible(n_q, n_k, causal, off)
    bounds = [0, *sorted(c for c in cuts if 0 < c < n_k), n_k]
    parts = [partial_over_keys(q, k, v, scale, vis, a, b, block, tau, p_dtype, l_from_rounded)
             for a, b in zip(bounds[:-1], bounds[1:])]
    o, _, l = merge_partials(parts) if len(parts) > 1 else parts[0]
    return finish(o, l, out_dtype)


def split_decode(q, k_cache, v_cache, seq_len, scale, chunk, tau=8.0, p_dtype=None,
                 out_dtype=None):
    """Decode of one (b, h) row by split-K: chunks of ``chunk`` cache rows, then the merge."""
    n = int(min(max(seq_len, 0), k_cache.shape[0]))
    q = np.asarray(q, dtype=np.float64).reshape(1, -1)
    if n == 0:
        return np.zeros(q.shape[1])
    cuts = list(range(chunk, n, chunk))
    return tiled_attention(q, k_cache[:n], v_cache[:n], False, scale, block=chunk, tau=tau,
                           cuts=cuts, p_dtype=p_dtype, out_dtype=out_dtype)[0]


# ------------------------------------------------------------- backward model
def backward_with_rounding(q, k, v, dout, causal, scale, p_dtype):
    """Gradients computed with the backward kernels' rounding points, in fp64.

    The forward (``tiled_attention`` with 16-bit weights) gives the output O,
    rounded to p_dtype as a training step stores it, and the row log-sum-exp
    lse = log(l) + m over the rounded weights it normalised by.  The backward
    recomputes P = exp(s - lse), forms dP = dO V^T and D = rowsum(dO * O16),
    dS = P (dP - D), and feeds the tensor-core products with 16-bit P and dS:
    dV = P16^T dO, dK = scale dS16^T Q, dQ = scale dS16 K.
    Returns (dq, dk, dv).  Square problems, one head: q, k, v, dout [N, d].
    """
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    n = q.shape[0]
    vis = _visible(n, n, causal, 0)
    o, m_ref, l = partial_over_keys(q, k, v, scale, vis, 0, n, 128, 8.0, p_dtype)
    o16 = round_to(o / l[:, None], p_dtype)
    lse = (m_ref + np.log2(l)) * math.log(2.0)
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    p = np.exp(s - lse[:, None])
    dp = dout @ v.T
    dsum = (dout * o16).sum(axis=1)
    ds = p * (dp - dsum[:, None])
    p16, ds16 = round_to(p, p_dtype), round_to(ds, p_dtype)
    return scale * ds16 @ k, scale * ds16.T @ q, p16.T @ dout
