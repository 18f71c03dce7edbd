"""Seeded random shapes against the fp64 oracle, element by element.

Each case draws its shape and options from a fixed seed: batch, query and
key/value heads (grouped or not), query and key lengths (square, chunked, or
more queries than keys), head size, causal mask, input and output types and
the schedule flags for prefill; a packed batch of random lengths; decode with
random lengths (zero included) and a random split count, plain and grouped.
The sizes stay small enough for the oracle to finish in seconds, and span
several tiles and ragged tails.
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
