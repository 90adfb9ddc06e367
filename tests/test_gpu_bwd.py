"""GPU parity of the backward (fa_bwd: dQ, dK, dV) against the fp64 oracle.

The forward runs on the GPU (fa_fwd), its O and LSE feed fa_bwd; the oracle
computes the gradients from the definition on the same bf16 Q, K, V and dO.

Tolerance, per element, derived from the arithmetic the kernels do (u = 2^-8,
the unit roundoff of bf16; gamma_n = n 2^-24 for an fp32 sum of n terms; all
magnitudes are the exact values, computed here in fp64):
  * O enters Delta_i = dO_i . O_i as the forward's bf16 output:
      |dO err| <= u (|O| + P |V|)  (P rounded to bf16 before P V, O rounded)
      |Delta err| <= sum_d |dO_id| |O err_id| + gamma_D sum_d |dO_id O_id|
  * P is recomputed from the saved LSE: |P err| <= e_P P, with e_P =
    eps + gamma_Sk + scale gamma_D (|Q| |K|^T): ex2/lg2.approx (eps = 4e-6),
    the fp32 row sum behind LSE, and the fp32 sum behind S = Q K^T;
    dP = dO V^T in fp32: |dP err| <= gamma_D |dO| |V|^T
  * dS = P (dP - Delta), rounded to bf16:
      |dS err| <= u |dS| + P (|Delta err| + |dP err|) + |P err| |dP - Delta|
  * dQ = scale dS K and dK = scale dS^T Q accumulate in fp32 and are rounded
    to bf16:  |dQ err| <= u |dQ| + scale (|dS err| + gamma_Sk |dS|) |K|, and
    the same for dK with Q;  dV = P^T dO with P rounded to bf16:
      |dV err| <= u |dV| + ((u + gamma_Sq) P + |P err|)^T |dO|
  * plus 1e-6 absolute for values that round to zero.
Every element must be within its bound, and the mean error within a quarter
of the mean bound (rounding errors are not all of one sign and size).
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


U = 2.0 ** -8      # bf16 unit roundoff (8 significant bits)
EPS_P = 4e-6       # ex2.approx and lg2.approx behind a recomputed P


def _f64(t):
    from exact_attention_82_gb300.inputs import bf16_bits

    return oracle.bf16_bits_to_f64(bf16_bits(t))


def _bounds(q, k, v, g, scale, causal):
    """Per-element error bounds of dQ, dK, dV (see the module docstring), from
    exact fp64 magnitudes of one head's inputs (q, g: [Sq, D]; k, v: [Sk, D])."""
    Sq, D = q.shape
    Sk = k.shape[0]
    s = scale * q @ k.T
    if causal:
        s = np.where(np.arange(Sk)[None, :] <= np.arange(Sq)[:, None], s, -np.inf)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    P = e / e.sum(axis=1, keepdims=True)
    O = P @ v
    dP = g @ v.T
    Delta = (g * O).sum(axis=1)
    dS = P * (dP - Delta[:, None])
    gam = lambda n: n * 2.0 ** -24
    aq, ak, av, ag = np.abs(q), np.abs(k), np.abs(v), np.abs(g)
    o_err = U * (np.abs(O) + P @ av)
    delta_err = (ag * o_err).sum(axis=1) + gam(D) * np.abs(g * O).sum(axis=1)
    dp_err = gam(D) * (ag @ av.T)
    p_err = P * (EPS_P + gam(Sk) + scale * gam(D) * (aq @ ak.T))
    ds_err = (U * np.abs(dS) + P * (delta_err[:, None] + dp_err)
              + p_err * np.abs(dP - Delta[:, None]))
    bq = U * np.abs(scale * dS @ k) + scale * (ds_err + gam(Sk) * np.abs(dS)) @ ak
    bk = U * np.abs(scale * dS.T @ q) + scale * (ds_err + gam(Sq) * np.abs(dS)).T @ aq
    bv = U * np.abs(P.T @ g) + ((U + gam(Sq)) * P + p_err).T @ ag
    return tuple(b + 1e-6 for b in (bq, bk, bv))


def _check(got, ref, bounds, what):
    """got, ref, bounds: (dQ, dK, dV) arrays of one shape."""
    for name, a, b, bd in zip(("dQ", "dK", "dV"), got, ref, bounds):
        assert np.all(np.isfinite(a)), f"{what} {name}: non-finite"
        err = np.abs(a - b)
        ratio = err / bd
        msg = (f"{what} {name}: max err/bound {ratio.max():.3f} (err {err.max():.3e}), "
               f"mean err {err.mean():.3e} vs mean bound {bd.mean():.3e}")
        assert ratio.max() <= 1.0, msg
        assert err.mean() <= 0.25 * bd.mean(), msg


def _bounds_all(q, k, v, g, scale, causal):
    """Bounds for [B, H, S, D] CPU bf16 tensors, head by head."""
    B, H = q.shape[:2]
    qs, ks, vs, gs = (_f64(t) for t in (q, k, v, g))
    out = [np.zeros(qs.shape), np.zeros(ks.shape), np.zeros(vs.shape)]
    for b in range(B):
        for h in range(H):
            for o, x in zip(out, _bounds(qs[b, h], ks[b, h], vs[b, h], gs[b, h], scale, causal)):
                o[b, h] = x
    return tuple(out)


def _case(B, H, Sq, Sk, D, causal, seed, q_mult=1.0):
    q, k, v = make_qkv(B, H, Sq, Sk, D, seed, q_mult)
    g, _, _ = make_qkv(B, H, Sq, Sk, D, seed + 7777)
    scale = D ** -0.5
    got = _grads_gpu(q, k, v, g, scale, causal)
    ref = oracle.attn_bwd(*(bf16_bits(t) for t in (q, k, v, g)), scale, causal)
    _check(got, ref, _bounds_all(q, k, v, g, scale, causal), f"B{B} H{H} Sq{Sq} Sk{Sk} D{D} causal{int(causal)}")


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


def test_backward_kernels_give_up_cleanly():
    """Both backward kernels' own give-up path: with every wait limited to 0 ns,
    the first wait in progress when the global timer ticks gives up, raises its
    CTA's abort flag and records FA_ERR_TIMEOUT; the other roles stop, copies and
    MMAs in flight are waited for (bounded), TMEM is freed and the kernels
    return.  The key and query sequences are long (8,192), so that a timer tick
    falls inside some wait.  A normal backward after it must pass parity, so the
    context is still usable."""
    assert fa.fa_device_status() == fa.FA_OK
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 8192, 8192, 128, seed=41))
    g = make_qkv(1, 2, 8192, 8192, 128, seed=42)[0].cuda()
    o, lse = fa.fa_fwd(q, k, v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty_like(lse)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert fa.fa_selftest_bwd_timeout(q, k, v, o, lse, g, dq, dk, dv, delta, 128 ** -0.5, False, 0) == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_device_status() == fa.FA_OK  # cleared by the read
    _case(1, 2, 300, 300, 128, True, seed=43)


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
        hs = [t[sl].contiguous() for t in (q, k, v, g)]
        ref = oracle.attn_bwd(*(bf16_bits(t) for t in hs), w.scale, w.causal)
        _check(tuple(x[sl] for x in got), ref, _bounds_all(*hs, w.scale, w.causal), f"{w.name} head {bh}")
