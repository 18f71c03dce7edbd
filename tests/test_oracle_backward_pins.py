"""Pins for the oracle's backward pass and log-sum-exp (CPU).

The gradients are the chain rule through the plain definition; they are
pinned to central finite differences of the oracle's forward (the derivative
the backward must be), to torch autograd in float64 (an independent library
routine), and to invariants of the softmax Jacobian.
"""

import numpy as np
import pytest


def rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_equal_finite_differences(oracle_mod, causal):
    r = rng(30)
    B, H, N, d = 1, 1, 5, 3
    q, k, v, g = r.normal(size=(4, B, H, N, d))
    scale = 0.7
    dq, dk, dv = oracle_mod.attention_backward(q, k, v, g, causal, scale)

    def loss(q_, k_, v_):
        return float(np.sum(oracle_mod.attention(q_, k_, v_, causal, scale) * g))

    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if n == name else a for n, a in (("q", q), ("k", k), ("v", v))]
            args_m = [xm if n == name else a for n, a in (("q", q), ("k", k), ("v", v))]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert np.max(np.abs(num - grad)) < 1e-7, name


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd(oracle_mod, causal):
    torch = pytest.importorskip("torch")
    r = rng(31)
    B, H, N, d = 2, 2, 33, 16
    q, k, v, g = r.normal(size=(4, B, H, N, d))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.25)
    out.backward(torch.from_numpy(g))
    dq, dk, dv = oracle_mod.attention_backward(q, k, v, g, causal, 0.25)
    for ours, theirs in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.max(np.abs(ours - theirs.numpy())) < 1e-12


def test_jacobian_invariants(oracle_mod):
    # rows of dS sum to zero, so the key gradients sum to zero over the keys;
    # dV sums (over keys) to the column sums of dO, because rows of P sum to 1
    r = rng(32)
    q, k, v, g = r.normal(size=(4, 1, 2, 40, 8))
    for causal in (False, True):
        dq, dk, dv = oracle_mod.attention_backward(q, k, v, g, causal, 0.3)
        assert np.max(np.abs(dk.sum(axis=2))) < 1e-12
        assert np.max(np.abs(dv.sum(axis=2) - g.sum(axis=2))) < 1e-12
    # a single key: the output is V[0] whatever Q and K are, so dQ = dK = 0
    dq, dk, dv = oracle_mod.attention_backward(q[..., :1, :], k[..., :1, :], v[..., :1, :],
                                               g[..., :1, :], False, 0.3)
    assert np.array_equal(dq, np.zeros_like(dq)) and np.array_equal(dk, np.zeros_like(dk))
    assert np.max(np.abs(dv - g[..., :1, :])) < 1e-15


def test_lse_closed_forms_and_library(oracle_mod):
    r = rng(33)
    q, k = r.normal(size=(2, 1, 1, 6, 4))
    lse = oracle_mod.attention_lse(q, k, True, 0.0)      # scale 0: log of the visible count
    assert np.max(np.abs(lse[0, 0] - np.log(np.arange(1, 7)))) < 1e-15
    s = 0.5 * q[0, 0] @ k[0, 0].T
    want = np.log(np.exp(s).sum(axis=1))
    assert np.max(np.abs(oracle_mod.attention_lse(q, k, False, 0.5)[0, 0] - want)) < 1e-12
    # Nq > Nk, causal: the leading rows see nothing
    lse2 = oracle_mod.attention_lse(q, k[..., :3, :], True, 0.5)
    assert np.all(np.isneginf(lse2[0, 0, :3])) and np.all(np.isfinite(lse2[0, 0, 3:]))
    # the weights the backward recomputes: exp(s - lse) equals the forward's P
    p = oracle_mod.attention_weights(q[0, 0], k[0, 0], False, 0.5)
    assert np.max(np.abs(np.exp(s - want[:, None]) - p)) < 1e-14


def test_grouped_head_gradients_match_library_autograd(oracle_mod):
    # a shared key/value head collects the gradients of every query head that
    # reads it: torch's own grouped SDPA in float64 differentiates the same thing
    torch = pytest.importorskip("torch")
    r = rng(34)
    B, Hq, Hkv, N, d = 1, 6, 2, 21, 8
    q, g = r.normal(size=(2, B, Hq, N, d))
    k, v = r.normal(size=(2, B, Hkv, N, d))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.3,
                                                           enable_gqa=True)
    out.backward(torch.from_numpy(g))
    dq, dk, dv = oracle_mod.attention_backward(q, k, v, g, True, 0.3)
    for ours, theirs in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert ours.shape == tuple(theirs.shape)
        assert np.max(np.abs(ours - theirs.numpy())) < 1e-12
