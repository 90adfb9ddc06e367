"""GPU parity of the backward (fa_bwd: dQ, dK, dV) against the fp64 oracle.

The forward runs on the GPU (fa_fwd), its O and LSE feed fa_bwd; the oracle
computes the gradients from the definition on the same bf16 Q, K, V and dO.
Tolerance: gradients have no fixed scale, so errors are taken relative to the
reference: max |g - g_ref| <= 2e-2 * max |g_ref| and mean |g - g_ref| <=
1e-2 * mean |g_ref|.  bf16 rounding of P and dS before the products (2^-9
relative per term), of O (it enters Delta) and of the outputs (2^-9) give
errors of a few 1e-3 relative; fp32 accumulation and ex2.approx add far less.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import bf16_bits, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert fa.fa_device_status() == fa.FA_OK


def _grads_gpu(q, k, v, g, scale, causal):
    dq_, dk_, dv_, dg = (t.cuda() for t in (q, k, v, g))
    o, lse = fa.fa_fwd(dq_, dk_, dv_, scale=scale, causal=causal)
    gq, gk, gv = fa.fa_bwd(dq_, dk_, dv_, o, lse, dg, scale=scale, causal=causal)
    torch.cuda.synchronize()
    return tuple(t.float().cpu().double().numpy() for t in (gq, gk, gv))


def _check(got, ref, what):
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(a)), f"{what} {name}: non-finite"
        err = np.abs(a - b)
        scale_max, scale_mean = np.abs(b).max(), np.abs(b).mean()
        msg = (f"{what} {name}: max err {err.max():.3e} (ref max {scale_max:.3e}), "
               f"mean err {err.mean():.3e} (ref mean {scale_mean:.3e})")
        assert err.max() <= 2e-2 * scale_max + 1e-6, msg
        assert err.mean() <= 1e-2 * scale_mean + 1e-7, msg


def _case(B, H, Sq, Sk, D, causal, seed, q_mult=1.0):
    q, k, v = make_qkv(B, H, Sq, Sk, D, seed, q_mult)
    g, _, _ = make_qkv(B, H, Sq, Sk, D, seed + 7777)
    scale = D ** -0.5
    got = _grads_gpu(q, k, v, g, scale, causal)
    ref = oracle.attn_bwd(*(bf16_bits(t) for t in (q, k, v, g)), scale, causal)
    _check(got, ref, f"B{B} H{H} Sq{Sq} Sk{Sk} D{D} causal{int(causal)}")


SHAPES = [(1, 1, 128, 128, 64), (1, 1, 128, 128, 128), (1, 2, 1, 1, 64), (2, 1, 100, 100, 128),
          (1, 2, 129, 129, 128), (2, 3, 389, 389, 128), (1, 2, 1000, 1000, 64), (2, 2, 256, 256, 64)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_parity(shape, causal):
    _case(*shape, causal, seed=500 + sum(shape))


@pytest.mark.parametrize("Sq,Sk", [(200, 300), (300, 77), (1, 260), (640, 128)])
@pytest.mark.parametrize("D", [64, 128])
def test_bwd_rectangular(Sq, Sk, D):
    _case(2, 2, Sq, Sk, D, False, seed=Sq + Sk + D)


def test_bwd_peaky():
    _case(2, 2, 384, 384, 64, True, seed=12, q_mult=4.0)


def test_bwd_deterministic():
    q, k, v, g = (t.cuda() for t in make_qkv(2, 4, 700, 700, 128, seed=3) + make_qkv(2, 4, 700, 700, 128, seed=4)[:1])
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    a = fa.fa_bwd(q, k, v, o, lse, g, causal=True)
    b = fa.fa_bwd(q, k, v, o, lse, g, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_bwd_closed_form_sums_at_size():
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (per head), up to bf16 rounding."""
    q, k, v = make_qkv(2, 4, 2048, 2048, 128, seed=8)
    g, _, _ = make_qkv(2, 4, 2048, 2048, 128, seed=9)
    gq, gk, gv = _grads_gpu(q, k, v, g, 128 ** -0.5, False)
    gsum = g.double().sum(dim=2).numpy()
    assert np.abs(gv.sum(axis=2) - gsum).max() <= 2e-2 * np.abs(gsum).max() + 0.05
    assert np.abs(gk.sum(axis=2)).max() <= 2e-2 * np.abs(gk).sum(axis=2).max() + 1e-3


@pytest.mark.parametrize("index", [i for i, w in enumerate(__import__(
    "exact_attention_82_gb300.inputs", fromlist=["WORKLOADS"]).WORKLOADS) if w.path == "bwd"])
def test_bwd_workload_sampled_heads(index):
    """The backward workloads at full size, in the bench's launch configuration;
    the oracle checks three whole heads (a head's dK and dV need all its rows)."""
    from exact_attention_82_gb300.inputs import SEED_BASE, WORKLOADS, workload_qkv

    w = WORKLOADS[index]
    q, k, v = workload_qkv(index)
    g = make_qkv(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + 999)[0]
    got = _grads_gpu(q, k, v, g, w.scale, w.causal)
    BH = w.B * w.H
    for bh in (0, BH // 2, BH - 1):
        b, h = divmod(bh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attn_bwd(*(bf16_bits(t[sl].contiguous()) for t in (q, k, v, g)), w.scale,
                              w.causal)
        _check(tuple(x[sl] for x in got), ref, f"{w.name} head {bh}")
