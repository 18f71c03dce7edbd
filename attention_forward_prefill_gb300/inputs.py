"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws numbers: it holds none of the attention arithmetic, so
the oracle and the CUDA path can both be fed from it without sharing any part
of the method.  Everything is counter-based and pure numpy, so the same seed
gives the same bits on x86 and Arm hosts and under any torch version.

Recipe (the workloads the pages describe; no dataset is involved):
  * uniform: SplitMix64 of (seed + (i + 1) * 0x9E3779B97F4A7C15), top 53 bits;
  * normal:  Box-Muller on consecutive uniform pairs (cos and sin branches);
  * 16-bit:  value -> binary32 (round to nearest even) -> fp16 or bf16
             (round to nearest even); fp16 via numpy's correctly rounded cast;
  * outlier keys: per (batch, head), round(0.01 * N) distinct rows chosen by a
    seeded partial Fisher-Yates shuffle are multiplied by 20 before rounding;
  * decode lengths: seq_len_b = 1 + (u64 mod max_len), exactly uniform on
    [1, max_len] when max_len is a power of two.
Seeds: 0xFA000000 + 16 * config_id + tensor_id, tensor ids Q=0, K=1, V=2,
outlier rows=3, seq_lens=4.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_OUTLIER, TENSOR_SEQLEN = 0, 1, 2, 3, 4


def seed_for(config_id: int, tensor_id: int) -> int:
    return 0xFA000000 + 16 * int(config_id) + int(tensor_id)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the counter-based SplitMix64 stream."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def normal_f64_range(seed: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 (start even) of the seeded N(0, 1) stream."""
    if start % 2:
        raise ValueError("a range of the normal stream starts at an even index")
    out = np.empty(count, dtype=np.float64)
    n_pairs = (count + 1) // 2
    p0 = start // 2
    done = 0
    while done < n_pairs:
        m = min(_CHUNK, n_pairs - done)
        z = splitmix64(seed, 2 * (p0 + done), 2 * m)
        top = (z >> np.uint64(11)).astype(np.float64)
        u1 = (top[0::2] + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = top[1::2] * (2.0 ** -53)          # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * math.pi * u2
        pair = np.empty(2 * m, dtype=np.float64)
        pair[0::2] = r * np.cos(t)
        pair[1::2] = r * np.sin(t)
        lo = 2 * done
        hi = min(count, lo + 2 * m)
        out[lo:hi] = pair[: hi - lo]
        done += m
    return out


def normal_f64(seed: int, count: int) -> np.ndarray:
    """count i.i.d. N(0, 1) draws (float64) from the seeded stream."""
    return normal_f64_range(seed, 0, count)


def _blocks(n: int, threads: int, block: int):
    """Even-aligned [lo, hi) blocks covering [0, n)."""
    block = max(2, (block // 2) * 2)
    return [(lo, min(n, lo + block)) for lo in range(0, n, block)] if threads > 1 else [(0, n)]


def f64_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16).view(np.uint16)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    b = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f64_to_f16_bits(x)
    if dtype == "bf16":
        return f64_to_bf16_bits(x)
    raise ValueError(f"unknown 16-bit dtype {dtype!r}")


def normal_bits(shape, seed: int, dtype: str, threads: int = 1) -> np.ndarray:
    """i.i.d. N(0,1) values rounded to fp16/bf16, as uint16 bit patterns.

    threads > 1 fills blocks of the same stream on host threads (numpy
    releases the GIL): the bits do not depend on the thread count.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(b):
        lo, hi = b
        out[lo:hi] = to_bits(normal_f64_range(seed, lo, hi - lo), dtype)

    blocks = _blocks(n, threads, 1 << 22)
    if len(blocks) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, blocks))
    else:
        fill(blocks[0])
    return out.reshape(shape)


def outlier_rows(seed: int, n_rows: int, count: int) -> np.ndarray:
    """count distinct indices in [0, n_rows): seeded partial Fisher-Yates."""
    perm = np.arange(n_rows, dtype=np.int64)
    z = splitmix64(seed, 0, count)
    for i in range(count):
        j = i + int(z[i] % np.uint64(n_rows - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:count])


def keys_with_outliers(shape, seed_k: int, seed_rows: int, dtype: str,
                       fraction: float = 0.01, factor: float = 20.0, threads: int = 1):
    """N(0,1) keys where round(fraction*N) rows per (b, h) are scaled by factor.

    The draw is scaled before it is rounded to 16 bits.  Heads are generated
    one by one (on host threads when threads > 1; the bits are the same).
    Returns (bits [B,H,N,d], rows [B*H, count]).
    """
    B, H, N, d = shape
    out = np.empty((B * H, N, d), dtype=np.uint16)
    count = int(round(fraction * N))
    rows = np.zeros((B * H, count), dtype=np.int64)
    head = N * d

    def one(bh):
        x = normal_f64_range(seed_k, bh * head, head).reshape(N, d)
        if count:
            r = outlier_rows(seed_rows + (bh << 32), N, count)
            rows[bh] = r
            x[r, :] *= factor
        out[bh] = to_bits(x, dtype)

    if threads > 1 and B * H > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(B * H)))
    else:
        for bh in range(B * H):
            one(bh)
    return out.reshape(shape), rows


def seq_lens(seed: int, batch: int, max_len: int) -> np.ndarray:
    """Per-sequence lengths uniform on [1, max_len] (int32)."""
    z = splitmix64(seed, 0, batch)
    return (np.uint64(1) + (z % np.uint64(max_len))).astype(np.int32)
