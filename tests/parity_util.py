"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI on seeded inputs and compare with the fp64 oracle.

Tolerances (stated for this attention forward on bf16 inputs): max |dO| <= 2e-2,
mean |dO| <= 2e-3, max |dLSE| <= 1e-3.  They cover bf16 rounding of P before
P*V (at most 2^-8 relative per term: bf16 keeps 8 significant bits), fp32
accumulation, the bf16 rounding of O (half an ulp is at most 2^-8 relative;
1.6e-2 absolute at |O| in [4, 8)) and
ex2.approx / lg2.approx (relative error ~2^-22).
"""
import numpy as np
import torch

import oracle
import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import bf16_bits, make_qkv

TOL_O_MAX = 2e-2
TOL_O_MEAN = 2e-3
TOL_LSE = 1e-3


def run_gpu(q, k, v, scale, causal, stream=None, window=None, splits=None):
    """q, k, v: CPU bf16 tensors.  Returns (O float64 numpy, LSE float64 numpy).
    With `window` = (wl, wr) the banded entry point is used; with `splits` (an
    int, 0 = automatic) the split-KV decode entry point."""
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    if splits is not None:
        o, lse = fa.fa_fwd_splitkv(dq, dk, dv, scale=scale, num_splits=splits, stream=stream)
    elif window is None:
        o, lse = fa.fa_fwd(dq, dk, dv, scale=scale, causal=causal, stream=stream)
    else:
        o, lse = fa.fa_fwd_window(dq, dk, dv, window[0], window[1], scale=scale, stream=stream)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    d = np.abs(o_gpu - o_ref)
    dl = np.abs(lse_gpu - lse_ref)
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu)), f"{what}: non-finite"
    msg = (f"{what}: max|dO|={d.max():.3e} mean|dO|={d.mean():.3e} max|dLSE|={dl.max():.3e}")
    assert d.max() <= TOL_O_MAX, msg
    assert d.mean() <= TOL_O_MEAN, msg
    assert dl.max() <= TOL_LSE, msg
    return d.max(), d.mean(), dl.max()


def full_parity(B, H, Sq, Sk, D, causal, seed, q_mult=1.0, scale=None):
    q, k, v = make_qkv(B, H, Sq, Sk, D, seed, q_mult)
    scale = D ** -0.5 if scale is None else scale
    og, lg = run_gpu(q, k, v, scale, causal)
    orf, lrf = oracle.attn_fwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), scale, causal)
    return compare(og, lg, orf, lrf, f"B{B} H{H} Sq{Sq} Sk{Sk} D{D} causal{int(causal)}")


def sample_rows(B, H, Sq, n_random, seed, block=128):
    """(bh, row) pairs: tile edges of a few heads plus random rows."""
    rng = np.random.default_rng(seed)
    heads = sorted(set([0, B * H - 1] + list(rng.integers(0, B * H, size=6))))
    edges = sorted(set(r for m in range(0, Sq, block) for r in (m, m + block - 1) if r < Sq)
                   | {Sq - 1})
    bh, rows = [], []
    for h in heads:
        pick = edges if len(edges) <= 40 else list(rng.choice(edges, 40, replace=False))
        bh += [h] * len(pick)
        rows += list(pick)
    bh += list(rng.integers(0, B * H, size=n_random))
    rows += list(rng.integers(0, Sq, size=n_random))
    return np.array(bh, np.int64), np.array(rows, np.int64)
