"""Pins for the fp64 oracle: it is checked against things other than itself.

* brute force on tiny inputs, in pure Python, with a different formula (no
  max shift: O = sum e^s v / sum e^s, LSE = ln sum e^s);
* a library routine: torch float64 softmax / logsumexp on CPU;
* closed forms stored as hand-derived golden fixtures (tests/golden);
* invariants: rows of P sum to 1, identical V rows, Sk = 1, first causal row,
  Q = 0 (uniform P), two-key logistic form, shift and permutation
  invariance, and the tiled online-softmax loop agreeing with the
  materialised definition.

Definition followed (source walk-through "FlashAttention-2 相比 FlashAttention-1，
到底改了什么", section "第二处源码差异：kernel 主循环怎么组织"):
O = softmax(scale QK^T [+mask]) V and the row log-sum-exp.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_82_gb300.inputs import bf16_bits, make_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def _allowed(i, j, Sk, causal, wl, wr):
    return (0 <= j < Sk and (not causal or j <= i) and (wl < 0 or j >= i - wl)
            and (wr < 0 or j <= i + wr))


def brute_force(q, k, v, scale, causal, wl=-1, wr=-1):
    """Pure-Python fp64 attention without the max shift (tiny inputs only)."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = np.zeros((B, H, Sq, D))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                js = [j for j in range(Sk) if _allowed(i, j, Sk, causal, wl, wr)]
                s = [scale * math.fsum(float(q[b, h, i, d]) * float(k[b, h, j, d])
                                       for d in range(D)) for j in js]
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                for d in range(D):
                    o[b, h, i, d] = math.fsum(e[t] * float(v[b, h, js[t], d])
                                              for t in range(len(js))) / z
                lse[b, h, i] = math.log(z)
    return o, lse


def torch_reference(q, k, v, scale, causal, wl=-1, wr=-1):
    """torch float64 CPU softmax / logsumexp with an explicit boolean mask."""
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    Sq, Sk = q.shape[2], k.shape[2]
    s = scale * torch.matmul(q, k.transpose(-1, -2))
    i = torch.arange(Sq).view(-1, 1)
    j = torch.arange(Sk).view(1, -1)
    allowed = torch.ones(Sq, Sk, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if wl >= 0:
        allowed &= j >= i - wl
    if wr >= 0:
        allowed &= j <= i + wr
    s = s.masked_fill(~allowed, float("-inf"))
    o = torch.matmul(torch.softmax(s, dim=-1), v)
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------- brute force
TINY = [(1, 1, 1, 1, 1), (1, 2, 3, 4, 2), (2, 1, 4, 3, 4), (1, 1, 4, 4, 3), (2, 2, 2, 4, 1)]


@pytest.mark.parametrize("shape", TINY)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (1, -1), (0, 2), (2, 1)])
def test_brute_force_tiny(shape, causal, window, oracle_lib):
    B, H, Sq, Sk, D = shape
    rng = np.random.default_rng(hash((shape, causal, window)) % 2**32)
    q, k, v = _rand((B, H, Sq, D), rng), _rand((B, H, Sk, D), rng), _rand((B, H, Sk, D), rng)
    scale = 0.7
    # a row with no allowed key is an error in the oracle
    for i in range(Sq):
        if not any(_allowed(i, j, Sk, causal, *window) for j in range(Sk)):
            with pytest.raises(oracle.OracleError):
                oracle.attn_fwd(q, k, v, scale, causal, window, lib=oracle_lib)
            return
    o, lse = oracle.attn_fwd(q, k, v, scale, causal, window, lib=oracle_lib)
    ob, lb = brute_force(q, k, v, scale, causal, *window)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


# ------------------------------------------------------------ library routine
@pytest.mark.parametrize("shape", [(2, 2, 67, 93, 16), (1, 3, 130, 130, 64), (1, 1, 5, 300, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_float64(shape, causal, oracle_lib):
    B, H, Sq, Sk, D = shape
    if causal and Sq > Sk:
        pytest.skip("causal rows beyond Sk have keys; covered by square shapes")
    rng = np.random.default_rng(7)
    q, k, v = _rand((B, H, Sq, D), rng, 2.0), _rand((B, H, Sk, D), rng), _rand((B, H, Sk, D), rng)
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attn_fwd(q, k, v, scale, causal, lib=oracle_lib)
    ot, lt = torch_reference(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ot, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lt, rtol=0, atol=1e-12)


def test_matches_torch_window(oracle_lib):
    rng = np.random.default_rng(11)
    q, k, v = (_rand((1, 2, 150, 32), rng) for _ in range(3))
    for wl, wr in [(17, -1), (0, 0), (40, 9)]:
        for causal in (False, True):
            o, lse = oracle.attn_fwd(q, k, v, 0.3, causal, (wl, wr), lib=oracle_lib)
            ot, lt = torch_reference(q, k, v, 0.3, causal, wl, wr)
            np.testing.assert_allclose(o, ot, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lt, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- golden files
def _read_golden(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = rest
    ints = {key: int(vals[key][0]) for key in ("B", "H", "Sq", "Sk", "D", "causal")}
    B, H, Sq, Sk, D = (ints[x] for x in ("B", "H", "Sq", "Sk", "D"))

    def arr(key, shape):
        return np.array([float(x) for x in vals[key]], np.float64).reshape(shape)

    return dict(
        q=arr("q", (B, H, Sq, D)), k=arr("k", (B, H, Sk, D)), v=arr("v", (B, H, Sk, D)),
        o=arr("o", (B, H, Sq, D)), lse=arr("lse", (B, H, Sq)),
        scale=float(vals["scale"][0]), causal=bool(ints["causal"]),
        window=tuple(int(x) for x in vals["window"]), tol=float(vals["tol"][0]))


GOLDEN_FILES = sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt"))


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_golden_closed_forms(name, oracle_lib):
    g = _read_golden(os.path.join(GOLDEN, name))
    o, lse = oracle.attn_fwd(g["q"], g["k"], g["v"], g["scale"], g["causal"], g["window"],
                             lib=oracle_lib)
    np.testing.assert_allclose(o, g["o"], rtol=0, atol=g["tol"])
    np.testing.assert_allclose(lse, g["lse"], rtol=0, atol=g["tol"])
    ot, lt = oracle.attn_fwd_tiled(g["q"], g["k"], g["v"], g["scale"], g["causal"], g["window"],
                                   block_m=2, block_n=2, lib=oracle_lib)
    np.testing.assert_allclose(ot, g["o"], rtol=0, atol=g["tol"])
    np.testing.assert_allclose(lt, g["lse"], rtol=0, atol=g["tol"])


def test_golden_files_present():
    assert len(GOLDEN_FILES) >= 4


# ------------------------------------------------------- invariants / closed forms
def test_rows_of_p_sum_to_one(oracle_lib):
    """With a V column of ones, O's column is sum_j p_ij, which must be 1."""
    rng = np.random.default_rng(3)
    B, H, S, D = 2, 2, 97, 8
    q, k = _rand((B, H, S, D), rng, 3.0), _rand((B, H, S, D), rng)
    v = _rand((B, H, S, D), rng)
    v[..., 3] = 1.0
    for causal in (False, True):
        o, _ = oracle.attn_fwd(q, k, v, 0.5, causal, lib=oracle_lib)
        np.testing.assert_allclose(o[..., 3], 1.0, rtol=0, atol=1e-14)
        # all p >= 0 and sum 1 => O is a convex combination of V rows
        assert np.all(o <= v.max(axis=2, keepdims=True) + 1e-12)
        assert np.all(o >= v.min(axis=2, keepdims=True) - 1e-12)


def test_identical_v_rows(oracle_lib):
    rng = np.random.default_rng(4)
    q, k = _rand((1, 2, 40, 16), rng, 2.0), _rand((1, 2, 55, 16), rng)
    u = _rand((1, 2, 1, 16), rng)
    v = np.repeat(u, 55, axis=2)
    o, _ = oracle.attn_fwd(q, k, v, 0.25, False, lib=oracle_lib)
    np.testing.assert_allclose(o, np.broadcast_to(u, o.shape), rtol=0, atol=1e-14)


def test_single_key(oracle_lib):
    rng = np.random.default_rng(5)
    q, k, v = _rand((2, 1, 9, 8), rng), _rand((2, 1, 1, 8), rng), _rand((2, 1, 1, 8), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.4, False, lib=oracle_lib)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=0)
    np.testing.assert_allclose(lse, 0.4 * np.einsum("bhid,bhd->bhi", q, k[:, :, 0]), atol=1e-14)


def test_first_causal_row(oracle_lib):
    rng = np.random.default_rng(6)
    q, k, v = (_rand((2, 3, 33, 16), rng) for _ in range(3))
    o, lse = oracle.attn_fwd(q, k, v, 0.25, True, lib=oracle_lib)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=0)
    np.testing.assert_allclose(lse[:, :, 0], 0.25 * np.sum(q[:, :, 0] * k[:, :, 0], -1),
                               rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_when_q_zero(causal, oracle_lib):
    rng = np.random.default_rng(8)
    S, D = 70, 8
    q = np.zeros((1, 1, S, D))
    k, v = _rand((1, 1, S, D), rng), _rand((1, 1, S, D), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.3, causal, lib=oracle_lib)
    for i in range(S):
        n = i + 1 if causal else S
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].mean(0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-14


def test_two_key_logistic(oracle_lib):
    rng = np.random.default_rng(9)
    q, k, v = _rand((1, 1, 6, 4), rng, 3.0), _rand((1, 1, 2, 4), rng), _rand((1, 1, 2, 4), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.9, False, lib=oracle_lib)
    for i in range(6):
        s1 = 0.9 * float(q[0, 0, i] @ k[0, 0, 0])
        s2 = 0.9 * float(q[0, 0, i] @ k[0, 0, 1])
        p1 = 1.0 / (1.0 + math.exp(s2 - s1))
        np.testing.assert_allclose(o[0, 0, i], p1 * v[0, 0, 0] + (1 - p1) * v[0, 0, 1],
                                   rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - (max(s1, s2) + math.log1p(math.exp(-abs(s1 - s2))))) < 1e-13


def test_shift_invariance(oracle_lib):
    """Appending a dimension with q=1, k=c/scale shifts every score by c."""
    rng = np.random.default_rng(10)
    B, H, S, D = 1, 2, 45, 8
    scale, c = 0.5, 3.75
    q, k, v = (_rand((B, H, S, D), rng) for _ in range(3))
    q2 = np.concatenate([q, np.ones((B, H, S, 1))], -1)
    k2 = np.concatenate([k, np.full((B, H, S, 1), c / scale)], -1)
    v2 = np.concatenate([v, np.zeros((B, H, S, 1))], -1)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, scale, causal, lib=oracle_lib)
        o2, lse2 = oracle.attn_fwd(q2, k2, v2, scale, causal, lib=oracle_lib)
        np.testing.assert_allclose(o2[..., :D], o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse2, lse + c, rtol=0, atol=1e-12)


def test_permutation_invariance(oracle_lib):
    rng = np.random.default_rng(12)
    q, k, v = _rand((2, 1, 30, 8), rng), _rand((2, 1, 41, 8), rng), _rand((2, 1, 41, 8), rng)
    perm = rng.permutation(41)
    o, lse = oracle.attn_fwd(q, k, v, 0.6, False, lib=oracle_lib)
    o2, lse2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.6, False, lib=oracle_lib)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


@pytest.mark.parametrize("bm,bn", [(1, 1), (7, 7), (64, 64), (128, 128), (16, 48)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_online_equals_materialised(bm, bn, causal, oracle_lib):
    rng = np.random.default_rng(13)
    B, H, S, D = 1, 2, 150, 16
    q, k, v = _rand((B, H, S, D), rng, 3.0), _rand((B, H, S, D), rng), _rand((B, H, S, D), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.25, causal, lib=oracle_lib)
    ot, lt = oracle.attn_fwd_tiled(q, k, v, 0.25, causal, block_m=bm, block_n=bn,
                                   lib=oracle_lib)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lt, lse, rtol=0, atol=1e-12)


def test_tiled_online_window(oracle_lib):
    """Windows leave whole key blocks empty for some rows; the loop skips them."""
    rng = np.random.default_rng(14)
    q, k, v = (_rand((1, 1, 200, 8), rng) for _ in range(3))
    o, lse = oracle.attn_fwd(q, k, v, 0.5, True, (20, -1), lib=oracle_lib)
    ot, lt = oracle.attn_fwd_tiled(q, k, v, 0.5, True, (20, -1), block_m=32, block_n=16,
                                   lib=oracle_lib)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lt, lse, rtol=0, atol=1e-12)


# ------------------------------------------------------------- bf16 front ends
def test_bf16_front_end_is_exact_widening(oracle_lib):
    q, k, v = make_qkv(2, 2, 37, 53, 16, seed=99)
    qb, kb, vb = (bf16_bits(t) for t in (q, k, v))
    o, lse = oracle.attn_fwd(qb, kb, vb, 0.25, False, lib=oracle_lib)
    qf, kf, vf = (t.to(torch.float64).numpy() for t in (q, k, v))
    o2, lse2 = oracle.attn_fwd(qf, kf, vf, 0.25, False, lib=oracle_lib)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(qb), qf)


def test_rows_api_matches_full(oracle_lib):
    q, k, v = make_qkv(2, 3, 300, 300, 32, seed=5)
    qb, kb, vb = (bf16_bits(t) for t in (q, k, v))
    o, lse = oracle.attn_fwd(qb, kb, vb, 0.2, True, lib=oracle_lib)
    rng = np.random.default_rng(0)
    bh = rng.integers(0, 6, size=50)
    rows = rng.integers(0, 300, size=50)
    os_, ls_ = oracle.attn_fwd_rows(qb, kb, vb, bh, rows, 0.2, True, lib=oracle_lib)
    ref_o = o.reshape(6, 300, 32)[bh, rows]
    ref_l = lse.reshape(6, 300)[bh, rows]
    assert np.array_equal(os_, ref_o) and np.array_equal(ls_, ref_l)


def test_threads_do_not_change_results(oracle_lib):
    q, k, v = make_qkv(2, 2, 600, 600, 16, seed=1)
    qb, kb, vb = (bf16_bits(t) for t in (q, k, v))
    a = oracle.attn_fwd(qb, kb, vb, 0.25, True, nthreads=1, lib=oracle_lib)
    b = oracle.attn_fwd(qb, kb, vb, 0.25, True, nthreads=5, lib=oracle_lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_empty_row_is_an_error(oracle_lib):
    """Row i may only see key i (window 0,0), but Sk = 1: rows 1 and 2 see nothing."""
    q = np.zeros((1, 1, 3, 2))
    kv = np.zeros((1, 1, 1, 2))
    with pytest.raises(oracle.OracleError):
        oracle.attn_fwd(q, kv, kv, 1.0, False, (0, 0), lib=oracle_lib)
    with pytest.raises(oracle.OracleError):
        oracle.attn_fwd_tiled(q, kv, kv, 1.0, False, (0, 0), block_m=2, block_n=2,
                              lib=oracle_lib)
