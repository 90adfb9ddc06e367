"""Pins for the oracle's backward pass (dQ, dK, dV of O for a given dO).

* central finite differences of the (separately pinned) forward oracle:
  L = sum(O * dO), so dL/dX must equal the backward's gradient for X;
* a library routine: torch float64 autograd through softmax and matmul;
* closed forms: sum_j dK_j = 0 (softmax is shift invariant along keys) and
  sum_j dV_j = sum_i dO_i (rows of P sum to 1);
* the bf16 front end is the exact widening.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_82_gb300.inputs import bf16_bits, make_qkv
from test_oracle_pins import torch_reference


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def _loss(q, k, v, g, scale, causal, window, lib):
    o, _ = oracle.attn_fwd(q, k, v, scale, causal, window, lib=lib)
    return float(np.sum(o * g))


@pytest.mark.parametrize("causal,window", [(False, (-1, -1)), (True, (-1, -1)), (True, (1, -1)),
                                           (False, (1, 2))])
def test_backward_matches_finite_differences(causal, window, oracle_lib):
    rng = np.random.default_rng(17)
    B, H, Sq, Sk, D = 1, 2, 4, 4, 3
    q, k, v = _rand((B, H, Sq, D), rng), _rand((B, H, Sk, D), rng), _rand((B, H, Sk, D), rng)
    g = _rand((B, H, Sq, D), rng)
    scale = 0.8
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, scale, causal, window, lib=oracle_lib)
    h = 1e-5
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], g, scale, causal, window,
                              oracle_lib)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], g, scale, causal, window,
                                oracle_lib)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=0, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("shape", [(2, 2, 37, 53, 16), (1, 3, 70, 70, 32)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(shape, causal, oracle_lib):
    B, H, Sq, Sk, D = shape
    if causal and Sq != Sk:
        pytest.skip("causal needs square")
    rng = np.random.default_rng(23)
    q, k, v = _rand((B, H, Sq, D), rng, 2.0), _rand((B, H, Sk, D), rng), _rand((B, H, Sk, D), rng)
    g = _rand((B, H, Sq, D), rng)
    scale = 1 / math.sqrt(D)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, -1) @ tv
    o.backward(torch.tensor(g))
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, scale, causal, lib=oracle_lib)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-11)


def test_backward_closed_form_sums(oracle_lib):
    rng = np.random.default_rng(29)
    B, H, S, D = 2, 2, 50, 8
    q, k, v, g = (_rand((B, H, S, D), rng) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.4, causal, lib=oracle_lib)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(axis=2), g.sum(axis=2), rtol=0, atol=1e-12)


def test_backward_bf16_front_end(oracle_lib):
    q, k, v = make_qkv(1, 2, 40, 40, 16, seed=31)
    g, _, _ = make_qkv(1, 2, 40, 40, 16, seed=32)
    a = oracle.attn_bwd(*(bf16_bits(t) for t in (q, k, v, g)), 0.25, True, lib=oracle_lib)
    b = oracle.attn_bwd(*(t.double().numpy() for t in (q, k, v, g)), 0.25, True, lib=oracle_lib)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_forward_of_backward_oracle_agrees(oracle_lib):
    """The backward recomputes O itself; its Delta uses that O.  Check the forward
    pieces it rebuilds agree with the forward oracle via the dV = P^T dO identity
    with dO = one-hot rows (dV_j then holds column P_ij)."""
    rng = np.random.default_rng(37)
    q, k, v = (_rand((1, 1, 6, 4), rng) for _ in range(3))
    o_ref, _ = oracle.attn_fwd(q, k, v, 0.5, False, lib=oracle_lib)
    ref_p = torch.softmax(0.5 * torch.tensor(q[0, 0]) @ torch.tensor(k[0, 0]).T, -1).numpy()
    for i in range(6):
        g = np.zeros((1, 1, 6, 4))
        g[0, 0, i, 0] = 1.0
        _, _, dv = oracle.attn_bwd(q, k, v, g, 0.5, False, lib=oracle_lib)
        np.testing.assert_allclose(dv[0, 0, :, 0], ref_p[i], rtol=0, atol=1e-14)
