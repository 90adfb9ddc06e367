"""GPU parity of the banded entry point fa_fwd_window against the fp64 oracle.

Key j is allowed for query i iff i - wl <= j <= i + wr ("FlashAttention-2 —
L3 Cross-Paper Synthesis", §5 item 4: sliding-window block skipping).  The
windows below put band edges inside tiles, on tile edges (multiples of the
128-key tile) and one key either side of them, so both skipped tiles and
tiles masked at either edge occur; left-only and right-only bands leave
whole first tiles empty for some rows.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import bf16_bits, make_qkv
from parity_util import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert fa.fa_device_status() == fa.FA_OK


WINDOWS = [(0, 0), (1, 0), (17, 0), (127, 0), (128, 0), (129, 0), (300, 0), (1000, 0),
           (0, 5), (64, 64), (130, 200), (200, -1), (-1, 50), (-1, 0), (-1, -1)]


@pytest.mark.parametrize("window", WINDOWS, ids=lambda w: f"wl{w[0]}_wr{w[1]}")
@pytest.mark.parametrize("D", [64, 128])
def test_window_parity(window, D):
    B, H, S = 1, 3, 700
    q, k, v = make_qkv(B, H, S, S, D, seed=300 + window[0] * 7 + window[1] + D)
    og, lg = run_gpu(q, k, v, D ** -0.5, False, window=window)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), D ** -0.5, False, window)
    compare(og, lg, *ref, f"window {window} D{D}")


@pytest.mark.parametrize("S", [1, 2, 129, 257, 1000])
def test_window_ragged_lengths(S):
    q, k, v = make_qkv(2, 2, S, S, 128, seed=S)
    for window in [(50, 0), (130, 10)]:
        og, lg = run_gpu(q, k, v, 128 ** -0.5, False, window=window)
        ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), 128 ** -0.5, False, window)
        compare(og, lg, *ref, f"S{S} window {window}")


def test_window_peaky():
    q, k, v = make_qkv(2, 2, 600, 600, 64, seed=11, q_mult=4.0)
    og, lg = run_gpu(q, k, v, 0.125, False, window=(255, 0))
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), 0.125, False, (255, 0))
    compare(og, lg, *ref, "peaky window")


@pytest.mark.parametrize("causal", [False, True])
def test_unbounded_window_equals_fa_fwd_bitwise(causal):
    q, k, v = (t.cuda() for t in make_qkv(2, 3, 555, 555, 128, seed=2))
    o1, l1 = fa.fa_fwd(q, k, v, causal=causal)
    o2, l2 = fa.fa_fwd_window(q, k, v, -1, 0 if causal else -1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_larger_than_sequence_equals_causal():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 300, 300, 64, seed=4))
    o1, l1 = fa.fa_fwd(q, k, v, causal=True)
    o2, l2 = fa.fa_fwd_window(q, k, v, 5000, 0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o1.float().cpu().numpy(), o2.float().cpu().numpy())
    np.testing.assert_array_equal(l1.cpu().numpy(), l2.cpu().numpy())


def test_window_rejects_rectangular_band():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError):
        fa.fa_fwd_window(q, kv, kv, 16, 0)
