"""The prefill schedule on the host (no GPU): the library's planner, read
through fa_prefill_plan, against a Python restatement of what every CTA of the
kernel then does -- which key tiles of which unit it runs, which partial slot
it writes -- and of what the fixup kernel reads back.  For every shape: each
unit's query tiles are finished exactly once, either whole in one CTA or from
pieces that tile their key range without gaps or overlaps, and every slot the
fixup reads is one a piece wrote for that unit.
"""
import bisect
import random

import pytest

from attention_forward_prefill_gb300 import binding, build

R, BM = 256, 128


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def kv_tiles(causal, no_skip, nq, nk, row0):
    # key tiles a 128-row query tile at row0 needs; queries are the last nq positions
    if row0 >= nq:
        return 0
    tk = (nk + 127) // 128
    if not causal or no_skip:
        return tk
    last = min(row0 + 127, nq - 1) + nk - nq
    return 0 if last < 0 else min(tk, last // 128 + 1)


def check_pairs(Nq):
    # The kernel's pairing: unit i of a head holds 128-row tiles i and T - 1 - i
    # (the latter absent when it is i itself), i < ceil(T / 2) = the units per head.
    T = (Nq + BM - 1) // BM
    seen = []
    for i in range((Nq + R - 1) // R):
        seen.append(i)
        if T - 1 - i > i:
            seen.append(T - 1 - i)
    assert sorted(seen) == list(range(T)), (Nq, seen)


def check_plan(B, H, Nq, Nk, causal, no_skip, sms, flags):
    rc, info, items = binding.fa_prefill_plan(B, H, Nq, Nk, causal, flags, sms)
    assert rc == 0
    stream_k, G, W, HT, n_qb, n_split, dp_full, s0, paired = info
    assert n_qb == (Nq + R - 1) // R and len(items) == n_split
    n_units = B * H * n_qb
    if not stream_k:
        assert G == min(n_units, sms) and n_split == 0
        forced_sk = bool(flags & binding.FA_FLAG_SCHEDULE_STREAM_K) and not (flags & binding.FA_FLAG_SCHEDULE_UNITS)
        assert paired == int(bool(causal) and not no_skip and n_units <= sms and not forced_sk)
        if paired:
            check_pairs(Nq)
        return False
    assert paired == 0
    assert G == min(sms, 192)
    cost = [max(kv_tiles(causal, no_skip, Nq, Nk, qb * R), kv_tiles(causal, no_skip, Nq, Nk, qb * R + BM))
            for qb in range(n_qb)]
    pre = [0]
    for c in cost:
        assert c >= 1
        pre.append(pre[-1] + c)
    assert HT == pre[-1] and W == B * H * HT
    if causal:
        assert dp_full == 0 and s0 == 0
    else:                                    # whole units first, then the cut ranges
        assert dp_full == n_units // G and s0 == dp_full * G * cost[0]
    fs = lambda c: s0 + c * (W - s0) // G
    writes, whole = {}, set()
    for c in range(G):                       # the kernel's per-CTA walk
        for kk in range(dp_full):
            u = c + kk * G
            for t in range(2):
                if kv_tiles(causal, no_skip, Nq, Nk, (u % n_qb) * R + t * BM) > 0:
                    whole.add((u, t))
        s, e, seg = fs(c), fs(c + 1), dp_full
        while s < e:
            bh, rem = divmod(s, HT)
            qb = bisect.bisect_right(pre, rem) - 1
            j0 = rem - pre[qb]
            j1 = min(cost[qb], j0 + (e - s))
            s += j1 - j0
            u = bh * n_qb + qb
            partial = not (j0 == 0 and j1 == cost[qb])
            for t in range(2):
                nt = min(kv_tiles(causal, no_skip, Nq, Nk, qb * R + t * BM), j1)
                if nt <= j0:
                    continue
                if partial:
                    key = (c, 0 if seg == dp_full else 1, t)
                    assert key not in writes
                    writes[key] = (u, j0, nt)
                else:
                    whole.add((u, t))
            seg += 1
    cut = set()
    for (u, cf, cl, ucost, us) in items:     # the fixup's reads
        cut.add(u)
        qb = u % n_qb
        assert ucost == cost[qb] and us == (u // n_qb) * HT + pre[qb]
        for t in range(2):
            if qb * R + t * BM >= Nq:
                continue
            nt = kv_tiles(causal, no_skip, Nq, Nk, qb * R + t * BM)
            spans = []
            for c in range(cf, cl + 1):
                if fs(c + 1) <= fs(c):
                    continue
                jf = max(fs(c) - us, 0)
                if jf < nt:
                    w = writes.get((c, 0 if fs(c) >= us else 1, t))
                    assert w is not None and w[0] == u
                    spans.append(w[1:])
            pos = 0
            for a, b in sorted(spans):
                assert a == pos
                pos = b
            assert pos == nt
    for u in range(n_units):
        qb = u % n_qb
        for t in range(2):
            if kv_tiles(causal, no_skip, Nq, Nk, qb * R + t * BM) > 0:
                assert ((u, t) in whole) != (u in cut)
    return True


FIXED = [(1, 16, 8192, 8192, 0), (1, 16, 16384, 16384, 1), (1, 12, 2048, 2048, 1), (8, 32, 8192, 8192, 1),
         (1, 24, 8192, 8192, 0), (2, 5, 4100, 4100, 0), (1, 4, 700, 1500, 1), (1, 2, 300, 300, 1)]


@pytest.mark.parametrize("shape", FIXED)
@pytest.mark.parametrize("flags", [0, 4])
def test_fixed_shapes(lib, shape, flags):
    B, H, Nq, Nk, causal = shape
    check_plan(B, H, Nq, Nk, causal, 0, 152, flags)


def test_random_shapes_forced_stream_k(lib):
    rng = random.Random(7)
    taken = 0
    for _ in range(250):
        B, H = rng.randint(1, 3), rng.randint(1, 6)
        Nq = rng.randint(1, 3000)
        no_skip = rng.random() < 0.2
        Nk = rng.randint(1, 4000) if no_skip else rng.randint(Nq, 4000)
        sms = rng.choice([152, 148, 7, 1, 192, 300])
        taken += check_plan(B, H, Nq, Nk, rng.randint(0, 1), no_skip, sms,
                            4 | (1 if no_skip else 0))
    assert taken > 150


def test_rule_choices_on_the_benchmark_shapes(lib):
    # the fitted rule: stream-K where it measured faster on 152 SMs
    # (causal shapes now balance well enough unit by unit in snake order)
    want = {(1, 16, 4096, 0): 0, (1, 16, 8192, 0): 1, (1, 16, 16384, 0): 1, (8, 32, 8192, 1): 0,
            (1, 16, 8192, 1): 0, (1, 12, 2048, 1): 0, (4, 12, 2048, 0): 0, (2, 16, 4096, 0): 1}
    for (B, H, N, causal), sk in want.items():
        _, info, _ = binding.fa_prefill_plan(B, H, N, N, causal, 0, 152)
        assert info[0] == sk, (B, H, N, causal)


def test_whole_units_first_cut_fewer(lib):
    # N = 8192, 16 heads: 512 units on 152 CTAs -> 3 whole units each, and only
    # the last 56 units are cut between CTAs
    _, info, items = binding.fa_prefill_plan(1, 16, 8192, 8192, 0, 0, 152)
    assert info[0] == 1 and info[6] == 3 and info[7] == 3 * 152 * 64
    assert len(items) <= 56 and all(it[0] >= 3 * 152 for it in items)


def test_units_flag_and_packed_rows_never_cut(lib):
    _, info, items = binding.fa_prefill_plan(1, 16, 8192, 8192, 0, 2, 152)
    assert info[0] == 0 and items == []
    # rows that see no key (Nq > Nk, causal) rule stream-K out
    _, info, _ = binding.fa_prefill_plan(1, 16, 8192, 4096, 1, 4, 152)
    assert info[0] == 0


# ---------------------------------------------------------------------------
# The ordered schedule of packed batches (packed_order_kernel and the ordered
# instantiation's unit mapping in fa_prefill_sm103.cu), restated: the classes
# (sequence b, 256-row block qb) are sorted by their 128 x 128 tile products,
# most first, ties by class index; unit u of the grid's round-robin deal is head
# u % Hq of class order[u // Hq].

def packed_order(lens_q, lens_k, n_qb, causal):
    keys = []
    for b, (nq, nk) in enumerate(zip(lens_q, lens_k)):
        for qb in range(n_qb):
            c = kv_tiles(causal, 0, nq, nk, qb * R) + kv_tiles(causal, 0, nq, nk, qb * R + BM)
            keys.append((0x7fffffff - c, b * n_qb + qb))
    return [cls for _, cls in sorted(keys)], {cls: 0x7fffffff - k for k, cls in keys}


def ordered_units(lens_q, lens_k, Hq, causal, G):
    n_qb = (max(lens_q) + R - 1) // R
    order, cost = packed_order(lens_q, lens_k, n_qb, causal)
    B = len(lens_q)
    n_units = B * Hq * n_qb
    per_cta = [[] for _ in range(G)]
    for u in range(n_units):
        k, r = divmod(u, G)
        c = G - 1 - r if k & 1 else r               # the snake deal of the unit schedule
        cls = order[u // Hq]
        per_cta[c].append((cls // n_qb, u % Hq, cls % n_qb, cost[cls]))
    return per_cta, n_units


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [0, 1])
def test_ordered_packed_schedule_deals_every_unit_once_heaviest_first(seed, causal):
    rng = random.Random(seed)
    B = rng.randint(8, 40)
    Hq = rng.choice([1, 2, 6, 16])
    lens = [rng.randint(0, 4096) for _ in range(B)]
    lens[rng.randrange(B)] = max(max(lens), 1)
    G = 152
    per_cta, n_units = ordered_units(lens, lens, Hq, causal, G)
    n_qb = (max(lens) + R - 1) // R
    dealt = sorted((b, h, qb) for units in per_cta for b, h, qb, _ in units)
    assert dealt == sorted((b, h, qb) for b in range(B) for h in range(Hq) for qb in range(n_qb))
    # the deal's rounds never go from a lighter class to a heavier one
    flat = []
    for u in range(n_units):
        k, r = divmod(u, G)
        flat.append(per_cta[G - 1 - r if k & 1 else r][k][3])
    assert all(a >= b for a, b in zip(flat, flat[1:]))
    # and the busiest CTA is within one heaviest unit of the average
    loads = [sum(x[3] for x in units) for units in per_cta]
    assert max(loads) <= sum(loads) / G + max(flat)
