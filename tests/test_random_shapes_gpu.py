"""Seeded random shapes against the fp64 oracle, element by element.

Each case draws its shape and options from a fixed seed: batch, query and
key/value heads (grouped or not), query and key lengths (square, chunked, or
more queries than keys), head size, causal mask, input and output types and
the schedule flags for prefill; a packed batch of random lengths; decode with
random lengths (zero included) and a random split count, plain and grouped;
the backward with grouped heads, both masks, every gradient type and tiny
lengths.  The sizes stay small enough for the oracle to finish in seconds,
and span several tiles and ragged tails; a larger set (up to 6000 keys and 32
heads) reaches the stream-K cuts and the persistent grids' several units per
CTA, checked on sampled rows or whole key/value groups.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module")
def fa():
    import torch
    from attention_forward_prefill_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3), "libfa_gb300 targets sm_103a"
    build.build()
    binding.load()
    assert binding.fa_device_status(True) == 0
    yield binding
    assert binding.fa_device_status(False) == 0, "a kernel reported a fault"


def draw_prefill(rng):
    B = int(rng.integers(1, 4))
    Hkv = int(rng.integers(1, 5))
    Hq = Hkv * int(rng.choice([1, 2, 3, 4]))
    Nk = int(rng.integers(1, 700))
    Nq = int(rng.choice([Nk, int(rng.integers(1, 700))]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    in_dt = str(rng.choice(["f16", "bf16"]))
    out_dt = str(rng.choice(["f16", "bf16", "f32"]))
    flags = int(rng.choice([0, 0, 2, 4]))  # auto, units, stream-K where it applies
    scale = float(rng.choice([1.0 / np.sqrt(d), 0.3, -0.2]))
    return B, Hq, Hkv, Nq, Nk, d, causal, in_dt, out_dt, flags, scale


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_prefill(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(9000 + case)
    B, Hq, Hkv, Nq, Nk, d, causal, in_dt, out_dt, flags, scale = draw_prefill(rng)
    q = inputs.normal_bits((B, Hq, Nq, d), 9100 + case, in_dt)
    k = inputs.normal_bits((B, Hkv, Nk, d), 9200 + case, in_dt)
    v = inputs.normal_bits((B, Hkv, Nk, d), 9300 + case, in_dt)
    qd, kd, vd = (G.bits_to_device(x, in_dt) for x in (q, k, v))
    out = fa.prefill(qd, kd, vd, causal=causal, scale=scale, out_dtype=G.torch_dtype(out_dt),
                     flags=flags)
    torch.cuda.synchronize()
    want = oracle_mod.attention(*(oracle_mod.bits_to_f64(x, in_dt) for x in (q, k, v)), causal, scale,
                                threads=G.THREADS)
    G.assert_close(G.device_to_f64(out), want, in_dt, out_dt,
                   f"case {case}: B={B} Hq={Hq} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} causal={causal} "
                   f"{in_dt}->{out_dt} flags={flags} scale={scale:.3f}")


@pytest.mark.parametrize("case", range(8))
def test_random_packed_batch(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(9400 + case)
    nseq = int(rng.integers(1, 7))
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.choice([1, 2]))
    d = int(rng.choice([64, 128]))
    dt = "bf16" if d == 128 else "f16"
    causal = bool(rng.integers(0, 2))
    lq = rng.integers(0, 500, size=nseq)
    lk = lq.copy() if rng.integers(0, 2) else rng.integers(0, 500, size=nseq)
    if nseq > 1 and case % 2 == 0:
        lq[int(rng.integers(0, nseq))] = 0          # a sequence with no queries
    if nseq > 1 and case % 4 == 1:
        lk[int(rng.integers(0, nseq))] = 0          # a sequence with no keys
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    tq, tk = int(cq[-1]), int(ck[-1])
    if tq == 0 or tk == 0:
        pytest.skip("no query rows or no keys drawn")
    q = inputs.normal_bits((tq, Hq, d), 9500 + case, dt)
    k = inputs.normal_bits((tk, Hkv, d), 9600 + case, dt)
    v = inputs.normal_bits((tk, Hkv, d), 9700 + case, dt)
    qd, kd, vd = (G.bits_to_device(x, dt) for x in (q, k, v))
    out = fa.prefill_varlen(qd, kd, vd, torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda(),
                            int(lq.max()), int(lk.max()), causal=causal, scale=1.0 / np.sqrt(d),
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = oracle_mod.attention_varlen(*(oracle_mod.bits_to_f64(x, dt) for x in (q, k, v)), cq, ck,
                                       causal, 1.0 / np.sqrt(d))
    G.assert_close(G.device_to_f64(out), want, dt, "f32",
                   f"packed case {case}: lengths q {lq.tolist()} k {lk.tolist()} Hq={Hq} Hkv={Hkv} d={d}")


@pytest.mark.parametrize("case", range(12))
def test_random_decode(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(9800 + case)
    B = int(rng.integers(1, 9))
    Hkv = int(rng.integers(1, 5))
    Hq = Hkv * int(rng.choice([1, 1, 2, 7, 8, 12]))
    L = int(rng.integers(1, 3000))
    d = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    lens = rng.integers(0, L + 1, size=B).astype(np.int32)
    if case % 3 == 0:
        lens[int(rng.integers(0, B))] = 0            # an empty cache row: zero output
    max_splits = (L + 63) // 64
    splits = int(rng.choice([0, 0, int(rng.integers(1, max_splits + 1))]))
    q = inputs.normal_bits((B, Hq, 1, d), 9900 + case, dt)
    kc = inputs.normal_bits((B, Hkv, L, d), 9950 + case, dt)
    vc = inputs.normal_bits((B, Hkv, L, d), 9990 + case, dt)
    out = fa.decode(G.bits_to_device(q, dt), G.bits_to_device(kc, dt), G.bits_to_device(vc, dt),
                    torch.from_numpy(lens).cuda(), scale=1.0 / np.sqrt(d), out_dtype=torch.float32,
                    num_splits=splits)
    torch.cuda.synchronize()
    want = oracle_mod.decode(*(oracle_mod.bits_to_f64(x, dt) for x in (q, kc, vc)), lens, 1.0 / np.sqrt(d))
    G.assert_close(G.device_to_f64(out), want, dt, "f32",
                   f"decode case {case}: B={B} Hq={Hq} Hkv={Hkv} L={L} d={d} splits={splits}")


# The backward: the bound against the exact gradient is the per-tensor one of
# the fixed-shape backward tests (1% / 0.15% of max|G| for bf16 / fp16 inputs),
# or 1.25 times the error that the method's own rounding points (16-bit P and dS
# into the products, D = dO.O over the 16-bit forward output) give on the same
# inputs in fp64, whichever is larger, plus the rounding of the gradient's output
# type.  The second term matters for tiny problems: with two keys per row, dQ is
# small next to the rounding of O inside D.
BWD_TOL = {"bf16": 1e-2, "f16": 1.5e-3}
GRAD_ROUND = {"f32": 0.0, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def rounding_model_backward(f, causal, scale, dt, group):
    from oracle import method_model as mm
    q, k, v, g = f
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            a, bb, c = mm.backward_with_rounding(q[b, h], k[b, h // group], v[b, h // group], g[b, h],
                                                 causal, scale, dt)
            dq[b, h] = a
            dk[b, h // group] += bb
            dv[b, h // group] += c
    return dq, dk, dv


@pytest.mark.parametrize("case", range(12))
def test_random_backward(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(8000 + case)
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 4))
    H = Hkv * int(rng.choice([1, 2, 3]))
    N = int(rng.integers(1, 600))
    if case % 4 == 3:
        N = int(rng.choice([1, 2, 127, 129]))  # a single row, a single tile, one past a tile
    d = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    causal = case % 2 == 1
    grad = str(rng.choice(["f32", "f16", "bf16"]))
    scale = float(rng.choice([1.0 / np.sqrt(d), 0.3, -0.2]))
    q, g = (inputs.normal_bits((B, H, N, d), 8100 + 10 * case + i, dt) for i in (0, 3))
    k, v = (inputs.normal_bits((B, Hkv, N, d), 8100 + 10 * case + i, dt) for i in (1, 2))
    qd, kd, vd, gd = (G.bits_to_device(x, dt) for x in (q, k, v, g))
    out, lse = fa.prefill_with_lse(qd, kd, vd, causal=causal, scale=scale)
    grads = fa.prefill_backward(qd, kd, vd, out, gd, lse, causal=causal, scale=scale,
                                grad_dtype=G.torch_dtype(grad))
    torch.cuda.synchronize()
    f = [oracle_mod.bits_to_f64(x, dt) for x in (q, k, v, g)]
    want = oracle_mod.attention_backward(*f, causal, scale, threads=G.THREADS)
    model = rounding_model_backward(f, causal, scale, dt, H // Hkv)
    for name, got_t, w, m in zip(("dq", "dk", "dv"), grads, want, model):
        got = G.device_to_f64(got_t)
        assert got.shape == w.shape
        # A row that sees a single key has P = 1 and O = V, so dS = P (dP - D) and the
        # exact dQ and dK are zero; only the fp32 rounding of dP - D remains.  Errors
        # are therefore measured against at least 0.01, a hundredth of the gradient
        # scale of these unit-variance inputs.
        top = max(np.abs(w).max(), 1e-2)
        tol = max(BWD_TOL[dt], 1.25 * float(np.abs(m - w).max() / top)) + GRAD_ROUND[grad]
        e = float(np.abs(got - w).max() / top)
        assert e <= tol, (f"{name} case {case}: B={B} H={H} Hkv={Hkv} N={N} d={d} {dt}->{grad} "
                          f"causal={causal} scale={scale:.3f}: {e:.3e} > {tol:.3e}")


# Packed batches over several rounds of units (8 to 40 sequences of 0 to 1500
# tokens, up to 16 query heads), which the kernel deals heaviest (sequence, block)
# class first in an order computed on the device: every sequence's rows must be
# bit-identical to that sequence run alone as a dense batch under the unit
# schedule, and one sequence is checked against the oracle on sampled rows.
@pytest.mark.parametrize("case", range(8))
def test_random_large_packed_batch(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(70000 + case)
    nseq = int(rng.integers(8, 41))
    Hkv = int(rng.integers(1, 5))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    d = int(rng.choice([64, 128]))
    dt = "bf16" if d == 128 else "f16"
    causal = bool(rng.integers(0, 2))
    lens = rng.integers(0, 1501, size=nseq)
    lens[int(rng.integers(0, nseq))] = max(int(lens.max()), 1)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    scale = 1.0 / np.sqrt(d)
    q = inputs.normal_bits((T, Hq, d), 71000 + case, dt)
    k = inputs.normal_bits((T, Hkv, d), 72000 + case, dt)
    v = inputs.normal_bits((T, Hkv, d), 73000 + case, dt)
    cu_d = torch.from_numpy(cu).cuda()
    out = fa.prefill_varlen(*(G.bits_to_device(x, dt) for x in (q, k, v)), cu_d, cu_d, int(lens.max()),
                            int(lens.max()), causal=causal, scale=scale, out_dtype=torch.float32)
    got = G.device_to_f64(out)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = slice(int(cu[b]), int(cu[b + 1]))
        alone = fa.prefill(*(G.bits_to_device(np.ascontiguousarray(x[sl].transpose(1, 0, 2)[None]), dt)
                             for x in (q, k, v)), causal=causal, scale=scale, out_dtype=torch.float32,
                           flags=fa.FA_FLAG_SCHEDULE_UNITS)
        assert np.array_equal(got[sl].transpose(1, 0, 2)[None], G.device_to_f64(alone)), (
            f"packed case {case}: sequence {b} of {nseq} ({n} tokens), Hq={Hq} Hkv={Hkv} d={d} causal={causal}")
    b = int(rng.integers(0, nseq))
    while lens[b] == 0:
        b = (b + 1) % nseq
    sl = slice(int(cu[b]), int(cu[b + 1]))
    rows = G.sample_rows(int(lens[b]), case)
    want = oracle_mod.attention(*(oracle_mod.bits_to_f64(np.ascontiguousarray(x[sl].transpose(1, 0, 2)[None]), dt)
                                  for x in (q, k, v)), causal, scale, rows=rows, threads=G.THREADS)
    G.assert_close(got[sl].transpose(1, 0, 2)[None][:, :, rows], want, dt, "f32",
                   f"packed case {case}: sequence {b} against the oracle")


# Larger shapes: 700 to 6000 keys and up to 32 heads, so that stream-K cuts units
# between CTAs and the persistent grids run several units per CTA; the forward is
# checked on sampled rows (tile edges, the middle, the end and seeded rows), the
# backward on two whole key/value groups.
@pytest.mark.parametrize("case", range(24))
def test_random_large_prefill(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(50000 + case)
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 9))
    Hq = Hkv * int(rng.choice([1, 1, 2, 4]))
    Nk = int(rng.integers(700, 6000))
    Nq = Nk if rng.integers(0, 3) else int(rng.integers(100, Nk + 1))
    d = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    causal = bool(rng.integers(0, 2))
    flags = int(rng.choice([0, 2, 4]))
    out_dt = str(rng.choice(["f32", dt]))
    scale = 1 / np.sqrt(d)
    q = inputs.normal_bits((B, Hq, Nq, d), 51000 + case, dt)
    k = inputs.normal_bits((B, Hkv, Nk, d), 52000 + case, dt)
    v = inputs.normal_bits((B, Hkv, Nk, d), 53000 + case, dt)
    out = fa.prefill(*(G.bits_to_device(x, dt) for x in (q, k, v)), causal=causal, scale=scale,
                     out_dtype=G.torch_dtype(out_dt), flags=flags)
    torch.cuda.synchronize()
    rows = G.sample_rows(Nq, case)
    want = oracle_mod.attention(*(oracle_mod.bits_to_f64(x, dt) for x in (q, k, v)), causal, scale,
                                rows=rows, threads=G.THREADS)
    G.assert_close(G.device_to_f64(out)[:, :, rows], want, dt, out_dt,
                   f"large case {case}: B={B} Hq={Hq} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} causal={causal} "
                   f"flags={flags}")


@pytest.mark.parametrize("case", range(8))
def test_random_large_backward(fa, oracle_mod, case):
    import torch
    rng = np.random.default_rng(60000 + case)
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 9))
    grp = int(rng.choice([1, 2, 4]))
    H = Hkv * grp
    N = int(rng.integers(500, 4000))
    d = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    causal = bool(rng.integers(0, 2))
    scale = 1 / np.sqrt(d)
    q, g = (inputs.normal_bits((B, H, N, d), 61000 + 10 * case + i, dt) for i in (0, 3))
    k, v = (inputs.normal_bits((B, Hkv, N, d), 61000 + 10 * case + i, dt) for i in (1, 2))
    qd, kd, vd, gd = (G.bits_to_device(x, dt) for x in (q, k, v, g))
    out, lse = fa.prefill_with_lse(qd, kd, vd, causal=causal, scale=scale)
    grads = [G.device_to_f64(t) for t in fa.prefill_backward(qd, kd, vd, out, gd, lse, causal=causal,
                                                             scale=scale, grad_dtype=torch.float32)]
    torch.cuda.synchronize()
    for b, kvh in ((0, 0), (B - 1, Hkv - 1)):
        qs, ks = slice(grp * kvh, grp * kvh + grp), slice(kvh, kvh + 1)
        f = [oracle_mod.bits_to_f64(np.ascontiguousarray(x[b:b + 1, sl]), dt)
             for x, sl in ((q, qs), (k, ks), (v, ks), (g, qs))]
        want = oracle_mod.attention_backward(*f, causal, scale, threads=G.THREADS)
        for name, got, sl, w in zip(("dq", "dk", "dv"), grads, (qs, ks, ks), want):
            e = float(np.abs(got[b:b + 1, sl] - w).max() / max(np.abs(w).max(), 1e-2))
            assert e <= BWD_TOL[dt], (f"{name} large case {case}: B={B} H={H} Hkv={Hkv} N={N} d={d} {dt} "
                                      f"causal={causal}, batch {b} kv head {kvh}: {e:.3e}")
