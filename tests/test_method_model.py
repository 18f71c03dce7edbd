"""The tiled online-softmax recurrence, in fp64, reaches the oracle's answer.

``oracle/method_model.py`` restates the method the kernels run (blocks of
keys, running m and l, lazy rescale with threshold tau, cut key ranges merged
exactly); the oracle is the plain definition with explicit score rows.  Their
agreement to 1e-12 shows the recurrence -- including the lazy rescale under
outlier keys and the merge of cut ranges -- is exact in arithmetic, before any
GPU result is compared.  The rounded variant predicts the size of the GPU's
deviation (16-bit weights, output rounding) and checks it sits inside the
tolerance.  All CPU.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from oracle import method_model as mm

EXACT = 1e-12


def normal(shape, seed):
    return np.random.default_rng(seed).normal(size=shape)


@pytest.mark.parametrize("n", [1, 127, 128, 129, 300, 700])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_recurrence_equals_definition(oracle_mod, n, d, causal):
    q, k, v = normal((3, n, d), 10 * n + d)
    scale = 1.0 / np.sqrt(d)
    got = mm.tiled_attention(q, k, v, causal, scale)
    want = oracle_mod.attention(q, k, v, causal, scale)
    assert np.abs(got - want).max() <= EXACT


@pytest.mark.parametrize("tau", [0.0, 1.0, 8.0, 30.0])
def test_lazy_threshold_does_not_change_the_result(oracle_mod, tau):
    # keys whose norm grows block by block make the row maximum move in almost
    # every block, so each tau takes a different set of rescale decisions
    n, d = 640, 64
    q, k, v = normal((3, n, d), 5)
    k *= np.linspace(0.2, 3.0, n)[:, None]
    got = mm.tiled_attention(q, k, v, True, 0.125, tau=tau)
    want = oracle_mod.attention(q, k, v, True, 0.125)
    assert np.abs(got - want).max() <= EXACT


def test_outlier_keys_stress_recipe(oracle_mod):
    # the stress recipe: 1% of the key rows scaled x20 before bf16 rounding
    n, d = 512, 128
    q = oracle_mod.bits_to_f64(inputs.normal_bits((n, d), 41, "bf16"), "bf16")
    kb, _ = inputs.keys_with_outliers((1, 1, n, d), 42, 43, "bf16")
    k = oracle_mod.bits_to_f64(kb[0, 0], "bf16")
    v = oracle_mod.bits_to_f64(inputs.normal_bits((n, d), 44, "bf16"), "bf16")
    scale = float(np.float32(1.0 / np.sqrt(d)))
    for causal in (False, True):
        got = mm.tiled_attention(q, k, v, causal, scale)
        want = oracle_mod.attention(q, k, v, causal, scale)
        assert np.abs(got - want).max() <= EXACT


@pytest.mark.parametrize("cuts", [(128,), (64, 200), (1, 2, 3), (256, 384, 511), (100,)])
@pytest.mark.parametrize("causal", [False, True])
def test_cut_key_ranges_merge_exactly(oracle_mod, cuts, causal):
    # a cut can leave a causal row with nothing visible in one part: that
    # part's (m = -inf, l = 0) must drop out of the merge
    n, d = 512, 64
    q, k, v = normal((3, n, d), 7)
    got = mm.tiled_attention(q, k, v, causal, 0.2, cuts=cuts)
    want = oracle_mod.attention(q, k, v, causal, 0.2)
    assert np.abs(got - want).max() <= EXACT


@pytest.mark.parametrize("chunk", [64, 128, 192, 512, 4096])
def test_split_decode_merges_exactly(oracle_mod, chunk):
    L, d = 1500, 64
    q = normal((4, 1, d), 8)
    kc, vc = normal((2, 4, L, d), 9)
    lens = [1, 64, 700, 1500]
    want = oracle_mod.decode(q[:, None], kc[:, None], vc[:, None], lens, 0.125)
    for b in range(4):
        got = mm.split_decode(q[b], kc[b], vc[b], lens[b], 0.125, chunk)
        assert np.abs(got - want[b, 0, 0]).max() <= EXACT


def test_bf16_rounding_model_fits_the_tolerance(oracle_mod):
    # 16-bit weights and a bf16 output: the predicted deviation from the
    # definition is inside 8e-3 + half an output ulp, with room to spare
    n, d = 512, 128
    q = oracle_mod.bits_to_f64(inputs.normal_bits((n, d), 51, "bf16"), "bf16")
    kb, _ = inputs.keys_with_outliers((1, 1, n, d), 52, 53, "bf16")
    k = oracle_mod.bits_to_f64(kb[0, 0], "bf16")
    v = oracle_mod.bits_to_f64(inputs.normal_bits((n, d), 54, "bf16"), "bf16")
    scale = float(np.float32(1.0 / np.sqrt(d)))
    want = oracle_mod.attention(q, k, v, True, scale)
    got = mm.tiled_attention(q, k, v, True, scale, p_dtype="bf16", out_dtype="bf16")
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -126))) - 8)
    assert (np.abs(got - want) <= 8e-3 + half_ulp).all()
    # without the output rounding the weights alone stay well under the bound
    got32 = mm.tiled_attention(q, k, v, True, scale, p_dtype="bf16")
    assert np.abs(got32 - want).max() < 4e-3


def test_l_over_rounded_weights_is_an_exact_convex_combination():
    # with l summing the rounded weights the tensor core applies, the output is
    # an exact convex combination of value rows: identical rows come back
    # unchanged.  Summing the unrounded weights leaves the 2^-9 relative
    # rounding of the weights in the result.
    n, d = 300, 64
    q, k, _ = normal((3, n, d), 60)
    v = np.broadcast_to(normal((d,), 61), (n, d)).copy()
    got = mm.tiled_attention(q, k, v, True, 0.3, p_dtype="bf16")
    bad = mm.tiled_attention(q, k, v, True, 0.3, p_dtype="bf16", l_from_rounded=False)
    assert np.abs(got - v).max() <= 1e-12
    assert np.abs(bad - v).max() > 1e-5


def test_bf16_rounding_helper_ties_to_even():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5, 0.0])
    assert list(mm.round_to(x, "bf16")) == [1.0, 1.0 + 2.0 ** -6, 1.0, -2.5, 0.0]


@pytest.mark.parametrize("dtype,bound", [("bf16", 1e-2), ("f16", 1.5e-3)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_rounding_model_fits_the_gradient_tolerance(oracle_mod, dtype, bound, causal):
    # the kernels' rounding points predict errors well inside the GPU bound
    # (max |err| / max |grad| per tensor), with at least a 2x margin
    n, d = 300, 128 if dtype == "bf16" else 64
    q, k, v, g = (oracle_mod.bits_to_f64(inputs.normal_bits((n, d), 70 + i, dtype), dtype)
                  for i in range(4))
    scale = 1.0 / np.sqrt(d)
    got = mm.backward_with_rounding(q, k, v, g, causal, scale, dtype)
    want = oracle_mod.attention_backward(q[None, None], k[None, None], v[None, None], g[None, None],
                                         causal, scale)
    for a, b in zip(got, want):
        rel = np.abs(a - b[0, 0]).max() / np.abs(b).max()
        assert rel <= bound / 2, rel


def test_backward_model_without_rounding_is_exact(oracle_mod):
    n, d = 200, 32
    q, k, v, g = normal((4, n, d), 80)
    got = mm.backward_with_rounding(q, k, v, g, True, 0.3, None)
    want = oracle_mod.attention_backward(q[None, None], k[None, None], v[None, None], g[None, None],
                                         True, 0.3)
    for a, b in zip(got, want):
        assert np.abs(a - b[0, 0]).max() <= 1e-11
