"""GPU parity of the backward pass (and the forward's log-sum-exp) against
the fp64 oracle, through the C ABI.

The inputs are 16-bit N(0,1) Q, K, V and an N(0,1) upstream gradient dO; the
forward output O comes from the library itself in the input type (as a
training step would have it).  The oracle differentiates the exact forward,
so the bound per gradient tensor is relative to its largest entry (see the
tolerance note below), checked on every element.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

# Rounding points of the kernels: P and dS enter the tensor core as 16-bit
# (relative 2^-9 for bf16, 2^-12 for fp16), O (for D = dO.O) is the 16-bit
# forward output, accumulation is fp32.  The fp64 model of those rounding
# points (oracle/method_model.py, backward_with_rounding) puts the worst
# element error at about 0.2% (bf16) / 0.03% (fp16) of max|G|; the kernels
# measured up to 0.41% / 0.051% on these shapes.  The bounds below are 1% /
# 0.15% of max|G| per tensor.
REL_TOL = {"bf16": 1e-2, "f16": 1.5e-3}
# The log-sum-exp sums the 16-bit weights the forward normalised by, so it
# carries their rounding: at most about 2^-8 (bf16) / 2^-11 (fp16) in log units.
LSE_TOL = {"bf16": 4e-3, "f16": 5e-4}


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
    assert binding.fa_device_status(False) == 0, "a kernel watchdog fired"


def run(fa, shape, dtype, causal, seed, grad="f32", hkv=None, flags=0):
    import torch
    kv_shape = shape if hkv is None else (shape[0], hkv, shape[2], shape[3])
    q, g = (inputs.normal_bits(shape, seed + i, dtype) for i in (0, 3))
    k, v = (inputs.normal_bits(kv_shape, seed + i, dtype) for i in (1, 2))
    qd, kd, vd, gd = (G.bits_to_device(x, dtype) for x in (q, k, v, g))
    scale = 1.0 / np.sqrt(shape[-1])
    out, lse = fa.prefill_with_lse(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.prefill_backward(qd, kd, vd, out, gd, lse, causal=causal, scale=scale,
                                     grad_dtype=G.torch_dtype(grad), flags=flags)
    torch.cuda.synchronize()
    return (q, k, v, g), scale, lse, (dq, dk, dv)


def rel_err(got, want):
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))


@pytest.mark.parametrize("shape,dtype", [((1, 2, 128, 64), "f16"), ((2, 3, 257, 64), "f16"),
                                         ((1, 2, 300, 128), "bf16"), ((1, 4, 1024, 128), "bf16"),
                                         ((1, 2, 1000, 64), "bf16")])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dq_path", ["ds_table", "recompute"])
def test_gradients_match_oracle(fa, oracle_mod, shape, dtype, causal, dq_path):
    flags = fa.FA_BWD_RECOMPUTE_DQ if dq_path == "recompute" else 0
    (q, k, v, g), scale, lse, grads = run(fa, shape, dtype, causal, 3000 + shape[2], flags=flags)
    f = [oracle_mod.bits_to_f64(x, dtype) for x in (q, k, v, g)]
    want = oracle_mod.attention_backward(*f, causal, scale, threads=G.THREADS)
    for name, got_t, w in zip(("dq", "dk", "dv"), grads, want):
        e = rel_err(G.device_to_f64(got_t), w)
        assert e <= REL_TOL[dtype], f"{name} {shape} {dtype} causal={causal} {dq_path}: {e:.3e}"


@pytest.mark.parametrize("shape,dtype,hkv", [((2, 3, 1000, 128), "bf16", None), ((1, 6, 643, 64), "f16", 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_ds_table_and_recompute_paths_agree(fa, shape, dtype, hkv, causal):
    # dK and dV come from the same pass either way: bit-identical.  dQ from the
    # stored 16-bit dS and from the recomputed one differ only by the fp32 order
    # of the score products, far inside the oracle bound.
    a = run(fa, shape, dtype, causal, 3800, hkv=hkv)[3]
    b = run(fa, shape, dtype, causal, 3800, hkv=hkv, flags=fa.FA_BWD_RECOMPUTE_DQ)[3]
    for name, x, y in zip(("dk", "dv"), a[1:], b[1:]):
        assert np.array_equal(G.device_to_f64(x), G.device_to_f64(y)), name
    e = rel_err(G.device_to_f64(a[0]), G.device_to_f64(b[0]))
    assert e <= REL_TOL[dtype] / 4, f"dq {shape} causal={causal}: {e:.3e}"


@pytest.mark.parametrize("shape,dtype,hkv", [((1, 16, 16384, 128), "bf16", None), ((2, 20, 8192, 64), "f16", 5)])
@pytest.mark.parametrize("causal", [False, True])
def test_a_table_over_the_limit_runs_in_chunks(fa, shape, dtype, hkv, causal):
    # A dS table over 4 GiB (8 GiB, and 5 GiB over 10 key/value heads) is taken in
    # two chunks of key/value heads on a table half that size; the second shape's
    # chunk boundary falls between the two sequences.  dK and dV come from the same
    # pass as with the recomputing dQ pass (bit-identical); dQ agrees within a
    # fraction of the oracle bound (that pass is checked against the oracle above).
    import torch
    rc, _ = fa.fa_pool_stats(reset_high=True)
    assert rc == fa.FA_OK
    a = run(fa, shape, dtype, causal, 3900, hkv=hkv)[3]
    rc, stats = fa.fa_pool_stats()
    assert rc == fa.FA_OK
    B, H, N, d = shape
    n_t = (N + 127) // 128
    table = B * H * n_t * n_t * 32768
    assert table > 4 << 30
    assert table // 2 <= stats[3] < table // 2 + (64 << 20), stats  # in-use high-water mark
    b = run(fa, shape, dtype, causal, 3900, hkv=hkv, flags=fa.FA_BWD_RECOMPUTE_DQ)[3]
    for name, x, y in zip(("dk", "dv"), a[1:], b[1:]):
        assert torch.equal(x, y), name
    e = rel_err(G.device_to_f64(a[0]), G.device_to_f64(b[0]))
    assert e <= REL_TOL[dtype] / 4, f"dq {shape} causal={causal}: {e:.3e}"


@pytest.mark.parametrize("N", [4096, 8192])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_at_bench_size_on_sampled_heads(fa, oracle_mod, N, causal):
    # the timed backward shape (1, 16, N, 128) bf16, run whole on the GPU; heads
    # are independent, so two of them (every row and column) are checked in full
    shape, dtype = (1, 16, N, 128), "bf16"
    (q, k, v, g), scale, lse, grads = run(fa, shape, dtype, causal, 3600 + N)
    heads = [0, 15]
    f = [oracle_mod.bits_to_f64(np.ascontiguousarray(x[:, heads]), dtype) for x in (q, k, v, g)]
    want = oracle_mod.attention_backward(*f, causal, scale, threads=len(heads))
    for name, got_t, w in zip(("dq", "dk", "dv"), grads, want):
        e = rel_err(G.device_to_f64(got_t)[:, heads], w)
        assert e <= REL_TOL[dtype], f"{name} N={N} causal={causal}: {e:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_forward_lse_matches_oracle(fa, oracle_mod, causal):
    shape, dtype = (2, 3, 700, 128), "bf16"
    (q, k, v, g), scale, lse, _ = run(fa, shape, dtype, causal, 3100)
    want = oracle_mod.attention_lse(oracle_mod.bits_to_f64(q, dtype), oracle_mod.bits_to_f64(k, dtype),
                                    causal, scale)
    assert np.abs(G.device_to_f64(lse) - want).max() <= LSE_TOL[dtype]


def test_lse_under_the_stream_k_schedule(fa, oracle_mod):
    # the fixup kernel writes the log-sum-exp of rows whose keys were cut
    import torch
    shape = (1, 3, 1000, 64)
    q, k, v = (inputs.normal_bits(shape, 3200 + i, "f16") for i in range(3))
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, k, v))
    _, lse = fa.prefill_with_lse(qd, kd, vd, causal=False, scale=0.125,
                                 flags=fa.FA_FLAG_SCHEDULE_STREAM_K)
    torch.cuda.synchronize()
    want = oracle_mod.attention_lse(oracle_mod.bits_to_f64(q, "f16"), oracle_mod.bits_to_f64(k, "f16"),
                                    False, 0.125)
    assert np.abs(G.device_to_f64(lse) - want).max() <= LSE_TOL["f16"]


@pytest.mark.parametrize("shape,hkv,dtype", [((1, 6, 300, 64), 2, "f16"), ((2, 8, 512, 128), 1, "bf16"),
                                             ((1, 14, 257, 64), 2, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dq_path", ["ds_table", "recompute"])
def test_grouped_head_gradients_match_oracle(fa, oracle_mod, shape, hkv, dtype, causal, dq_path):
    # a shared key/value head collects the gradients of all its query heads
    flags = fa.FA_BWD_RECOMPUTE_DQ if dq_path == "recompute" else 0
    (q, k, v, g), scale, lse, grads = run(fa, shape, dtype, causal, 3500 + shape[1], hkv=hkv, flags=flags)
    f = [oracle_mod.bits_to_f64(x, dtype) for x in (q, k, v, g)]
    want = oracle_mod.attention_backward(*f, causal, scale, threads=G.THREADS)
    for name, got_t, w in zip(("dq", "dk", "dv"), grads, want):
        got = G.device_to_f64(got_t)
        assert got.shape == w.shape
        e = rel_err(got, w)
        assert e <= REL_TOL[dtype], f"{name} {shape}/{hkv} {dtype} causal={causal}: {e:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_gradients_with_several_units_per_cta(fa, oracle_mod, causal):
    # 64 query heads over 16 key/value heads at N = 2048: 256 dK/dV units and 1024 dQ
    # units on the persistent grids, so every CTA runs several units in turn, each
    # dK/dV unit summing over its 4 query heads.  Two whole groups are checked.
    shape, hkv, dtype = (1, 64, 2048, 64), 16, "f16"
    (q, k, v, g), scale, lse, grads = run(fa, shape, dtype, causal, 3700, hkv=hkv)
    got = [G.device_to_f64(t) for t in grads]
    for kvh in (0, hkv - 1):
        qs = slice(4 * kvh, 4 * kvh + 4)
        f = [oracle_mod.bits_to_f64(np.ascontiguousarray(x[:, sl]), dtype)
             for x, sl in ((q, qs), (k, slice(kvh, kvh + 1)), (v, slice(kvh, kvh + 1)), (g, qs))]
        want = oracle_mod.attention_backward(*f, causal, scale, threads=4)
        for name, got_t, sl, w in zip(("dq", "dk", "dv"), got, (qs, slice(kvh, kvh + 1), slice(kvh, kvh + 1)),
                                      want):
            e = rel_err(got_t[:, sl], w)
            assert e <= REL_TOL[dtype], f"{name} kv head {kvh} causal={causal}: {e:.3e}"


@pytest.mark.parametrize("shape,dtype,hkv", [((2, 4, 1000, 128), "bf16", None), ((2, 6, 1000, 64), "f16", 2)])
@pytest.mark.parametrize("flags", [0, 1])
def test_gradients_are_bit_identical_run_to_run(fa, shape, dtype, hkv, flags):
    # d = 64 runs the dK/dV pipeline whose score products overlap the elementwise work;
    # flags 1 is the dQ pass that recomputes S and dP
    import torch
    a = run(fa, shape, dtype, True, 3300, grad=dtype, hkv=hkv, flags=flags)[3]
    b = run(fa, shape, dtype, True, 3300, grad=dtype, hkv=hkv, flags=flags)[3]
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_key_gradients_sum_to_zero(fa):
    # rows of dS sum to zero, so dK summed over the keys vanishes (fp32 grads)
    (q, k, v, g), scale, lse, (dq, dk, dv) = run(fa, (1, 2, 512, 64), "f16", False, 3400)
    s = G.device_to_f64(dk).sum(axis=2)
    assert np.abs(s).max() <= 1e-3 * np.abs(G.device_to_f64(dk)).max() * 512 ** 0.5
