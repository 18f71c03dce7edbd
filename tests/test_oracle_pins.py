"""Pins for the fp64 oracle, checked against facts that do not come from it.

Each test fixes a property that the definition of attention (flash-attention-
cuda README, "What is Attention?" / "The Problem" / "Kernel design") forces,
so that a plausible slip in the oracle -- a dropped scale, a wrong mask
direction or off-by-one, a transposed operand, a missing normalisation -- fails
at least one of them.  All run on CPU.
"""
import json
import math
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- decoders
def test_f16_decoder_known_patterns(oracle_mod):
    bits = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF, 0x3555, 0x8000], dtype=np.uint16)
    want = [1.0, -2.0, 2.0 ** -24, 65504.0, 0.333251953125, -0.0]
    got = oracle_mod.f16_bits_to_f64(bits)
    assert list(got) == want


def test_bf16_decoder_known_patterns(oracle_mod):
    bits = np.array([0x3F80, 0xC040, 0x0001, 0x7F7F, 0x3EAB], dtype=np.uint16)
    want = [1.0, -3.0, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, 0.333984375]
    got = oracle_mod.bf16_bits_to_f64(bits)
    assert list(got) == want


# ---------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_that_value(oracle_mod, causal):
    r = rng(1)
    q, k, v = r.normal(size=(3, 1, 7))
    out = oracle_mod.attention(q, k, v, causal, 0.3)
    assert np.array_equal(out, v)


def test_two_keys_logistic_closed_form(oracle_mod):
    # d = 1: softmax over two scores is the logistic function of their gap.
    q = np.array([[0.7], [-1.3]])
    k = np.array([[1.9], [-0.4]])
    v = np.array([[2.5], [-3.0]])
    scale = 0.37
    out = oracle_mod.attention(q, k, v, False, scale)
    for i in range(2):
        s0, s1 = scale * q[i, 0] * k[0, 0], scale * q[i, 0] * k[1, 0]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        want = w0 * v[0, 0] + (1.0 - w0) * v[1, 0]
        assert abs(out[i, 0] - want) < 1e-14
    # causal: row 0 sees only key 0, row 1 sees both
    outc = oracle_mod.attention(q, k, v, True, scale)
    assert outc[0, 0] == v[0, 0]
    assert abs(outc[1, 0] - out[1, 0]) < 1e-15


def test_large_logit_gap_selects_the_max_key(oracle_mod):
    # exp(-1000) underflows to 0: the output is exactly the winning value row
    # and nothing overflows (the max is subtracted first).
    q = np.array([[1.0, 0.0]])
    k = np.array([[1000.0, 0.0], [0.0, 5.0], [-3.0, 1.0]])
    v = np.array([[1.5, -2.0], [9.0, 9.0], [7.0, 7.0]])
    out = oracle_mod.attention(q, k, v, False, 1.0)
    assert np.array_equal(out[0], v[0])


def test_classroom_example_golden(oracle_mod):
    with open(os.path.join(HERE, "golden", "classroom_attention.json")) as f:
        g = json.load(f)
    w = np.array(g["weights"])
    q = np.ones((1, 1, 1, 1))
    kc = np.log(w).reshape(1, 1, 4, 1)
    vc = np.eye(4).reshape(1, 1, 4, 4)
    # d differs between keys (1) and values (4) here; use the head-level
    # routine with the weight rows instead of the value product.
    p = oracle_mod.attention_weights(q[0, 0], kc[0, 0], False, 1.0)
    assert np.max(np.abs(p[0] - np.array(g["expected_output"]))) <= g["tolerance"]
    # and the output through decode with V = I4 embedded in d = 4
    q4 = np.zeros((1, 1, 1, 4)); q4[..., 0] = 1.0
    k4 = np.zeros((1, 1, 4, 4)); k4[0, 0, :, 0] = np.log(w)
    out = oracle_mod.decode(q4, k4, vc, [4], 1.0)
    assert np.max(np.abs(out[0, 0, 0] - np.array(g["expected_output"]))) <= g["tolerance"]


# ---------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_weight_rows_sum_to_one_and_mask_is_lower_triangular(oracle_mod, causal):
    r = rng(2)
    q, k = r.normal(size=(2, 33, 16))
    p = oracle_mod.attention_weights(q, k, causal, 0.25)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
    assert np.all(p >= 0)
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)
        assert np.all(np.diag(p) > 0.0)
    else:
        assert np.all(p > 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(oracle_mod, causal):
    r = rng(3)
    n, d = 19, 8
    q = np.zeros((n, d))
    k, v = r.normal(size=(2, n, d))
    out = oracle_mod.attention(q, k, v, causal, 0.5)
    for i in range(n):
        vis = v[: i + 1] if causal else v
        assert np.max(np.abs(out[i] - vis.mean(axis=0))) < 1e-13
    # scale = 0 is the same special case
    q2 = r.normal(size=(n, d))
    out2 = oracle_mod.attention(q2, k, v, causal, 0.0)
    assert np.max(np.abs(out2 - out)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows_reproduce_that_row(oracle_mod, causal):
    r = rng(4)
    n, d = 25, 12
    q, k = r.normal(size=(2, n, d)) * 3.0
    row = r.normal(size=d)
    v = np.tile(row, (n, 1))
    out = oracle_mod.attention(q, k, v, causal, 0.7)
    assert np.max(np.abs(out - row)) < 1e-13


def test_causal_row_zero_is_first_value(oracle_mod):
    r = rng(5)
    q, k, v = r.normal(size=(3, 40, 9))
    out = oracle_mod.attention(q, k, v, True, 1.1)
    assert np.array_equal(out[0], v[0])


def test_causal_last_row_equals_full_last_row(oracle_mod):
    r = rng(6)
    q, k, v = r.normal(size=(3, 30, 6))
    a = oracle_mod.attention(q, k, v, True, 0.4)
    b = oracle_mod.attention(q, k, v, False, 0.4)
    assert np.max(np.abs(a[-1] - b[-1])) < 1e-15
    assert np.max(np.abs(a[0] - b[0])) > 1e-3  # the mask does something


def test_decode_of_token_t_equals_causal_prefill_row_t(oracle_mod):
    r = rng(7)
    B, H, N, d = 2, 3, 24, 8
    q, k, v = r.normal(size=(3, B, H, N, d))
    pre = oracle_mod.attention(q, k, v, True, 0.125)
    for t in [0, 1, 11, N - 1]:
        dec = oracle_mod.decode(q[:, :, t:t + 1], k, v, [t + 1] * B, 0.125)
        assert np.max(np.abs(dec[:, :, 0] - pre[:, :, t])) < 1e-12


def test_decode_ragged_lengths_use_only_visible_rows(oracle_mod):
    r = rng(8)
    B, H, L, d = 3, 2, 20, 5
    q = r.normal(size=(B, H, 1, d))
    kc, vc = r.normal(size=(2, B, H, L, d))
    lens = [1, 7, 20]
    out = oracle_mod.decode(q, kc, vc, lens, 0.3)
    kc2, vc2 = kc.copy(), vc.copy()
    for b, n in enumerate(lens):   # garbage past the length must not matter
        kc2[b, :, n:] = 1e6
        vc2[b, :, n:] = -1e6
    out2 = oracle_mod.decode(q, kc2, vc2, lens, 0.3)
    assert np.array_equal(out, out2)
    assert np.array_equal(out[0, :, 0], vc[0, :, 0])


def test_decode_zero_length_gives_zero_row(oracle_mod):
    out = oracle_mod.decode(np.ones((1, 1, 1, 4)), np.ones((1, 1, 3, 4)),
                            np.ones((1, 1, 3, 4)), [0], 1.0)
    assert np.array_equal(out, np.zeros((1, 1, 1, 4)))


def test_shift_of_all_keys_leaves_output_unchanged(oracle_mod):
    r = rng(9)
    q, k, v = r.normal(size=(3, 16, 8))
    c = r.normal(size=8)
    for causal in (False, True):
        a = oracle_mod.attention(q, k, v, causal, 0.5)
        b = oracle_mod.attention(q, k + c, v, causal, 0.5)
        assert np.max(np.abs(a - b)) < 1e-12


def test_joint_key_value_permutation_invariance(oracle_mod):
    r = rng(10)
    q, k, v = r.normal(size=(3, 21, 8))
    perm = r.permutation(21)
    a = oracle_mod.attention(q, k, v, False, 0.6)
    b = oracle_mod.attention(q, k[perm], v[perm], False, 0.6)
    assert np.max(np.abs(a - b)) < 1e-13
    # permuting keys alone changes the answer (operands are not symmetric)
    c = oracle_mod.attention(q, k[perm], v, False, 0.6)
    assert np.max(np.abs(a - c)) > 1e-3


def test_affine_in_values(oracle_mod):
    r = rng(11)
    q, k, v = r.normal(size=(3, 18, 8))
    a_, b_ = -1.7, r.normal(size=8)
    for causal in (False, True):
        o1 = oracle_mod.attention(q, k, v, causal, 0.5)
        o2 = oracle_mod.attention(q, k, a_ * v + b_, causal, 0.5)
        assert np.max(np.abs(o2 - (a_ * o1 + b_))) < 1e-12


def test_query_scaling_equals_scale_argument(oracle_mod):
    r = rng(12)
    q, k, v = r.normal(size=(3, 14, 8))
    a = oracle_mod.attention(q, k, v, True, 0.25)
    b = oracle_mod.attention(0.25 * q, k, v, True, 1.0)
    assert np.max(np.abs(a - b)) < 1e-13


def test_row_subset_matches_full_computation(oracle_mod):
    r = rng(13)
    q, k, v = r.normal(size=(3, 2, 2, 50, 8))
    full = oracle_mod.attention(q, k, v, True, 0.3)
    rows = [0, 7, 49, 13]
    sub = oracle_mod.attention(q, k, v, True, 0.3, rows=rows, threads=2)
    assert np.array_equal(sub, full[:, :, rows])


# ------------------------------------------- independent library routine
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_in_float64(oracle_mod, causal):
    torch = pytest.importorskip("torch")
    r = rng(14)
    B, H, N, d = 2, 3, 37, 16
    q, k, v = r.normal(size=(3, B, H, N, d))
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        is_causal=causal, scale=0.125).numpy()
    got = oracle_mod.attention(q, k, v, causal, 0.125)
    assert np.max(np.abs(got - want)) < 1e-12


def test_decode_matches_torch_sdpa_on_truncated_cache(oracle_mod):
    torch = pytest.importorskip("torch")
    r = rng(15)
    B, H, L, d = 3, 2, 40, 16
    q = r.normal(size=(B, H, 1, d))
    kc, vc = r.normal(size=(2, B, H, L, d))
    lens = [5, 40, 17]
    got = oracle_mod.decode(q, kc, vc, lens, 0.125)
    for b, n in enumerate(lens):
        want = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[b:b + 1]), torch.from_numpy(kc[b:b + 1, :, :n]),
            torch.from_numpy(vc[b:b + 1, :, :n]), scale=0.125).numpy()
        assert np.max(np.abs(got[b:b + 1] - want)) < 1e-12


# ------------------------------- chunked prefill, grouped heads, packed batches
def test_chunk_rows_equal_the_tail_of_the_square_causal_problem(oracle_mod):
    # a prompt chunk of the last Nq positions over all Nk keys is the last Nq
    # rows of the square causal problem (same visible sets, row by row)
    r = rng(20)
    Nk, Nq, d = 40, 15, 8
    q, k, v = r.normal(size=(3, Nk, d))
    square = oracle_mod.attention(q, k, v, True, 0.3)
    chunk = oracle_mod.attention(q[Nk - Nq:], k, v, True, 0.3)
    assert np.array_equal(chunk, square[Nk - Nq:])
    # the last query row sees every key, and a one-row chunk is a decode step
    full = oracle_mod.attention(q[Nk - Nq:], k, v, False, 0.3)
    assert np.array_equal(chunk[-1], full[-1])
    dec = oracle_mod.decode(q[None, None, -1:], k[None, None], v[None, None], [Nk], 0.3)
    one = oracle_mod.attention(q[-1:], k, v, True, 0.3)
    assert np.max(np.abs(dec[0, 0, 0] - one[0])) < 1e-15


def test_more_queries_than_keys_leaves_leading_rows_empty(oracle_mod):
    # Nq > Nk: query i sees keys j <= i - (Nq - Nk); the first Nq - Nk rows
    # see nothing (zero rows), the next sees key 0 alone
    r = rng(21)
    q = r.normal(size=(10, 6))
    k, v = r.normal(size=(2, 4, 6))
    out = oracle_mod.attention(q, k, v, True, 0.5)
    assert np.array_equal(out[:6], np.zeros((6, 6)))
    assert np.array_equal(out[6], v[0])
    full = oracle_mod.attention(q, k, v, False, 0.5)
    assert np.max(np.abs(out[-1] - full[-1])) < 1e-15


def test_chunk_matches_an_explicit_library_mask(oracle_mod):
    torch = pytest.importorskip("torch")
    r = rng(22)
    Nq, Nk, d = 23, 57, 16
    q = r.normal(size=(1, 2, Nq, d))
    k, v = r.normal(size=(2, 1, 2, Nk, d))
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    mask = torch.from_numpy(j <= i + (Nk - Nq))
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=mask,
        scale=0.2).numpy()
    got = oracle_mod.attention(q, k, v, True, 0.2)
    assert np.max(np.abs(got - want)) < 1e-12


def test_grouped_heads_equal_repeated_kv_heads(oracle_mod):
    r = rng(23)
    B, Hq, Hkv, N, d = 2, 6, 2, 19, 8
    q = r.normal(size=(B, Hq, N, d))
    k, v = r.normal(size=(2, B, Hkv, N, d))
    got = oracle_mod.attention(q, k, v, True, 0.4)
    rep = oracle_mod.attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), True, 0.4)
    assert np.array_equal(got, rep)
    # consecutive query heads share a kv head (h // 3), not h % 2
    alt = oracle_mod.attention(q, np.tile(k, (1, 3, 1, 1)), np.tile(v, (1, 3, 1, 1)), True, 0.4)
    assert np.max(np.abs(got - alt)) > 1e-3


def test_grouped_heads_match_library_gqa(oracle_mod):
    torch = pytest.importorskip("torch")
    r = rng(24)
    B, Hq, Hkv, N, d = 1, 14, 2, 21, 16
    q = r.normal(size=(B, Hq, N, d))
    k, v = r.normal(size=(2, B, Hkv, N, d))
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True,
        scale=0.25, enable_gqa=True).numpy()
    got = oracle_mod.attention(q, k, v, True, 0.25)
    assert np.max(np.abs(got - want)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_packed_batch_equals_each_sequence_alone(oracle_mod, causal):
    r = rng(25)
    Hq, Hkv, d = 4, 2, 8
    lens_q = [5, 17, 1, 0, 12]
    lens_k = [5, 30, 9, 4, 12]
    cu_q = np.concatenate([[0], np.cumsum(lens_q)])
    cu_k = np.concatenate([[0], np.cumsum(lens_k)])
    q = r.normal(size=(cu_q[-1], Hq, d))
    k, v = r.normal(size=(2, cu_k[-1], Hkv, d))
    got = oracle_mod.attention_varlen(q, k, v, cu_q, cu_k, causal, 0.35)
    for b in range(len(lens_q)):
        if lens_q[b] == 0:
            continue
        qs = q[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2)[None]
        ks = k[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2)[None]
        vs = v[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2)[None]
        want = oracle_mod.attention(qs, ks, vs, causal, 0.35)[0].transpose(1, 0, 2)
        assert np.array_equal(got[cu_q[b]:cu_q[b + 1]], want)
    # keys of other sequences are never seen: changing them changes nothing
    k2 = k.copy()
    k2[cu_k[1]:cu_k[2]] *= 3.0   # (a shift would cancel in the softmax)
    got2 = oracle_mod.attention_varlen(q, k2, v, cu_q, cu_k, causal, 0.35)
    assert np.array_equal(got2[cu_q[0]:cu_q[1]], got[cu_q[0]:cu_q[1]])
    assert np.array_equal(got2[cu_q[2]:], got[cu_q[2]:])
    assert np.max(np.abs(got2[cu_q[1]:cu_q[2]] - got[cu_q[1]:cu_q[2]])) > 1e-3


def test_grouped_decode_equals_repeated_caches_and_a_one_row_chunk(oracle_mod):
    r = rng(26)
    B, Hq, Hkv, L, d = 3, 14, 2, 50, 8
    q = r.normal(size=(B, Hq, 1, d))
    kc, vc = r.normal(size=(2, B, Hkv, L, d))
    lens = [1, 33, 50]
    got = oracle_mod.decode(q, kc, vc, lens, 0.3)
    rep = oracle_mod.decode(q, np.repeat(kc, 7, axis=1), np.repeat(vc, 7, axis=1), lens, 0.3)
    assert np.array_equal(got, rep)
    for b, n in enumerate(lens):   # the same row as a one-query causal chunk over n keys
        one = oracle_mod.attention(q[b:b + 1], kc[b:b + 1, :, :n], vc[b:b + 1, :, :n], True, 0.3)
        assert np.max(np.abs(one[0, :, 0] - got[b, :, 0])) < 1e-15
