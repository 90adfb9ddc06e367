"""Pins for the block-mask oracle (``oracle.attn_fwd_blockmask``).

Definition followed ("FlashAttention-2 -- L3 Cross-Paper Synthesis", section 5
item 4, the unified sparse-block-skip mechanism): key j is allowed for query i
iff j < Sk, the window keeps it, and the block mask keeps block
(i // bm, j // bn) of the head; O = softmax over the allowed keys times V, LSE
the log-sum-exp; a row with no allowed key gets O = 0 and LSE = -inf.

It is pinned against things other than itself:
* an all-ones mask reduces it to the C oracle's full, causal and banded
  attention (pinned on its own by brute force, torch and golden values);
* attention over a subset of keys is attention over those keys alone: each
  query block's rows against the gathered keys of its kept blocks, through the
  C oracle with no mask at all;
* brute force in pure Python on tiny inputs, per-head masks, a window and
  empty rows included (no max shift);
* planted mistakes (a transposed block index, swapped block sizes, the first
  head's mask for every head, the window's right bound ignored, the scale
  dropped) each fail one of the above.
"""
import inspect
import math
import textwrap

import numpy as np
import pytest

import oracle

BLOCKS = [(16, 8), (8, 16), (32, 32)]


def _qkv(rng, B, H, Sq, Sk, D):
    return (rng.standard_normal((B, H, Sq, D)), rng.standard_normal((B, H, Sk, D)),
            rng.standard_normal((B, H, Sk, D)))


def _nblk(S, b):
    return -(-S // b)


# -------------------------------------------------- all-ones mask = C oracle
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("window,causal", [((-1, -1), False), ((-1, 0), True), ((7, 3), False), ((0, 0), False)])
def test_all_ones_mask_is_the_plain_oracle(block, window, causal, oracle_lib, fn=None):
    fn = fn or oracle.attn_fwd_blockmask
    rng = np.random.default_rng(11)
    S = 45
    q, k, v = _qkv(rng, 2, 2, S, S, 8)
    mask = np.ones((1, _nblk(S, block[0]), _nblk(S, block[1])), np.uint8)
    o, l = fn(q, k, v, 0.3, mask, window=window, block=block)
    ro, rl = oracle.attn_fwd(q, k, v, 0.3, causal, (-1, -1) if causal else window, lib=oracle_lib)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


# ------------------------------------------- subset of keys = gathered keys
def _gathered_reference(q, k, v, scale, mask, block, lib):
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    bm, bn = block
    o = np.zeros((B, H, Sq, D))
    lse = np.full((B, H, Sq), -np.inf)
    for bh in range(B * H):
        b, h = divmod(bh, H)
        kept = mask[0 if mask.shape[0] == 1 else bh]
        for a in range(_nblk(Sq, bm)):
            keys = [j for c in range(_nblk(Sk, bn)) if kept[a, c] for j in range(c * bn, min(Sk, c * bn + bn))]
            rows = slice(a * bm, min(Sq, a * bm + bm))
            if not keys:
                continue
            qa = np.ascontiguousarray(q[b, h, rows][None, None])
            ka = np.ascontiguousarray(k[b, h, keys][None, None])
            va = np.ascontiguousarray(v[b, h, keys][None, None])
            ro, rl = oracle.attn_fwd(qa, ka, va, scale, lib=lib)
            o[b, h, rows] = ro[0, 0]
            lse[b, h, rows] = rl[0, 0]
    return o, lse


@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("per_head", [False, True])
def test_masked_keys_equal_gathered_keys(block, per_head, oracle_lib, fn=None):
    fn = fn or oracle.attn_fwd_blockmask
    rng = np.random.default_rng(12 + per_head)
    B, H, Sq, Sk = 2, 3, 70, 53
    q, k, v = _qkv(rng, B, H, Sq, Sk, 8)
    nq, nk = _nblk(Sq, block[0]), _nblk(Sk, block[1])
    mask = (rng.random((B * H if per_head else 1, nq, nk)) < 0.5).astype(np.uint8)
    mask[0, 0, :] = 0  # an empty query block: rows get O = 0, LSE = -inf
    o, l = fn(q, k, v, 0.4, mask, block=block)
    ro, rl = _gathered_reference(q, k, v, 0.4, mask, block, oracle_lib)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(l[fin], rl[fin], rtol=0, atol=1e-12)
    assert np.all(o[0, 0, :block[0]] == 0) and np.all(np.isneginf(l[0, 0, :block[0]]))


# ----------------------------------------------- brute force, pure Python
def brute_force_blockmask(q, k, v, scale, mask, wl, wr, bm, bn):
    """Pure-Python fp64 attention over the allowed keys, without the max shift;
    a row with no allowed key: O = 0, LSE = -inf."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = np.zeros((B, H, Sq, D))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            kept = mask[0 if mask.shape[0] == 1 else b * H + h]
            for i in range(Sq):
                js = [j for j in range(Sk) if (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr)
                      and kept[i // bm, j // bn]]
                if not js:
                    lse[b, h, i] = -math.inf
                    continue
                e = [math.exp(scale * math.fsum(float(q[b, h, i, d]) * float(k[b, h, j, d]) for d in range(D)))
                     for j in js]
                z = math.fsum(e)
                for d in range(D):
                    o[b, h, i, d] = math.fsum(e[t] * float(v[b, h, js[t], d]) for t in range(len(js))) / z
                lse[b, h, i] = math.log(z)
    return o, lse


CASES = [  # B, H, Sq, Sk, D, (wl, wr), (bm, bn), per_head
    (1, 1, 7, 9, 3, (-1, -1), (2, 3), False),
    (2, 2, 9, 9, 2, (-1, 0), (3, 2), True),
    (1, 3, 10, 10, 4, (2, 1), (4, 4), True),
    (2, 1, 5, 11, 3, (-1, -1), (5, 1), False),
]


@pytest.mark.parametrize("case", CASES)
def test_brute_force_tiny(case, fn=None):
    fn = fn or oracle.attn_fwd_blockmask
    B, H, Sq, Sk, D, (wl, wr), (bm, bn), per_head = case
    rng = np.random.default_rng(sum(case[:5]))
    q, k, v = _qkv(rng, B, H, Sq, Sk, D)
    mask = (rng.random((B * H if per_head else 1, _nblk(Sq, bm), _nblk(Sk, bn))) < 0.6).astype(np.uint8)
    mask[-1, -1, :] = 0  # the last query block of the last mask head sees nothing
    o, l = fn(q, k, v, 0.7, mask, window=(wl, wr), block=(bm, bn))
    ro, rl = brute_force_blockmask(q, k, v, 0.7, mask, wl, wr, bm, bn)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    np.testing.assert_allclose(l[np.isfinite(rl)], rl[np.isfinite(rl)], rtol=0, atol=1e-12)


def test_bf16_front_end_widens_exactly():
    rng = np.random.default_rng(5)
    bits = [(rng.standard_normal((1, 1, 20, 4)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            for _ in range(3)]
    mask = np.array([[[1, 0], [1, 1]]], np.uint8)
    o, l = oracle.attn_fwd_blockmask(*bits, 0.5, mask, block=(16, 16))
    wide = [oracle.bf16_bits_to_f64(b) for b in bits]
    ro, rl = oracle.attn_fwd_blockmask(*wide, 0.5, mask, block=(16, 16))
    assert np.array_equal(o, ro) and np.array_equal(l, rl)


def test_rejects_a_mask_of_the_wrong_shape():
    rng = np.random.default_rng(6)
    q, k, v = _qkv(rng, 1, 2, 20, 20, 4)
    with pytest.raises(ValueError):
        oracle.attn_fwd_blockmask(q, k, v, 1.0, np.ones((1, 2, 3)), block=(16, 16))
    with pytest.raises(ValueError):
        oracle.attn_fwd_blockmask(q, k, v, 1.0, np.ones((3, 2, 2)), block=(16, 16))


# --------------------------------------------------------- planted mistakes
MUTANTS = {
    "transposed block index": ("kept[np.arange(Sq) // bm][:, np.arange(Sk) // bn]",
                               "kept.T[np.arange(Sq) // bm][:, np.arange(Sk) // bn]"),
    "block sizes swapped": ("kept[np.arange(Sq) // bm][:, np.arange(Sk) // bn]",
                            "kept[np.arange(Sq) // bn % kept.shape[0]][:, np.arange(Sk) // bm % kept.shape[1]]"),
    "first head's mask everywhere": ("mask[0 if mask.shape[0] == 1 else bh]", "mask[0]"),
    "right window bound ignored": ("band &= j <= i + window[1]", "pass"),
    "scale dropped": ("float(scale) * (q[b, h] @ k[b, h].T)", "(q[b, h] @ k[b, h].T)"),
}


def _mutant(before, after):
    src = textwrap.dedent(inspect.getsource(oracle.attn_fwd_blockmask))
    assert src.count(before) == 1, before
    ns = dict(vars(oracle))
    exec(compile(src.replace(before, after), "<mutant>", "exec"), ns)
    return ns["attn_fwd_blockmask"]


def _battery(fn, lib):
    failures = 0
    checks = [lambda: test_all_ones_mask_is_the_plain_oracle((8, 16), (7, 3), False, lib, fn=fn),
              lambda: test_all_ones_mask_is_the_plain_oracle((16, 8), (-1, 0), True, lib, fn=fn)]
    checks += [lambda c=c: test_brute_force_tiny(c, fn=fn) for c in CASES]
    checks += [lambda p=p: test_masked_keys_equal_gathered_keys((16, 8), p, lib, fn=fn) for p in (False, True)]
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    return failures


def test_unmutated_oracle_passes_battery(oracle_lib):
    assert _battery(oracle.attn_fwd_blockmask, oracle_lib) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, oracle_lib):
    assert _battery(_mutant(*MUTANTS[name]), oracle_lib) > 0, name
