"""GPU parity of the split-KV decode entry point fa_fwd_splitkv against the
fp64 oracle: 1..8 query rows per head, every key visible, the keys of each
head split into ranges whose partial results are merged
("FlashAttention-2 — L3 Cross-Paper Synthesis", §5 item 5)."""
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


@pytest.mark.parametrize("Sq", [1, 2, 3, 8])
@pytest.mark.parametrize("Sk", [1, 63, 64, 65, 1000, 4099])
@pytest.mark.parametrize("D", [64, 128])
def test_splitkv_parity(Sq, Sk, D):
    q, k, v = make_qkv(2, 3, Sq, Sk, D, seed=Sq * 1000 + Sk + D)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), D ** -0.5, False)
    for splits in (0, 1, 3):
        og, lg = run_gpu(q, k, v, D ** -0.5, False, splits=splits)
        compare(og, lg, *ref, f"Sq{Sq} Sk{Sk} D{D} splits{splits}")


@pytest.mark.parametrize("splits", [2, 7, 64, 256])
def test_splitkv_many_splits(splits):
    q, k, v = make_qkv(3, 2, 1, 20000, 128, seed=splits)
    og, lg = run_gpu(q, k, v, 128 ** -0.5, False, splits=splits)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), 128 ** -0.5, False)
    compare(og, lg, *ref, f"splits {splits}")


def test_splitkv_peaky_and_growing_scores():
    """Q x4 (peaky softmax) and a key range far above the others, so splits
    disagree strongly on their maxima before the merge."""
    q, k, v = make_qkv(2, 2, 4, 3000, 64, seed=9, q_mult=4.0)
    k[:, :, 2500:2600] = (k[:, :, 2500:2600].float() * 3).to(torch.bfloat16)
    og, lg = run_gpu(q, k, v, 0.125, False, splits=0)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), 0.125, False)
    compare(og, lg, *ref, "peaky split-KV")


def test_splitkv_matches_fa_fwd():
    """The split path and the query-block path compute the same attention."""
    q, k, v = make_qkv(2, 4, 3, 5000, 128, seed=5)
    o1, l1 = run_gpu(q, k, v, 128 ** -0.5, False)
    o2, l2 = run_gpu(q, k, v, 128 ** -0.5, False, splits=0)
    assert np.max(np.abs(o1 - o2)) <= 2e-2 and np.max(np.abs(l1 - l2)) <= 1e-3


def test_splitkv_deterministic_and_workspace_reuse():
    q, k, v = (t.cuda() for t in make_qkv(4, 8, 1, 7777, 128, seed=3))
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(4, 8, 1, 7777, 128), dtype=torch.uint8,
                     device="cuda")
    o1, l1 = fa.fa_fwd_splitkv(q, k, v, workspace=ws)
    o2, l2 = fa.fa_fwd_splitkv(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_splitkv_rejects_short_workspace_on_device():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 1, 3000, 64, seed=1))
    need = fa.fa_fwd_splitkv_workspace_bytes(1, 2, 1, 3000, 64)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_splitkv(q, k, v, workspace=ws)
    assert e.value.status == fa.FA_ERR_WORKSPACE


def test_splitkv_kernel_gives_up_cleanly():
    """The decode kernels' give-up path: with every wait of the partial kernel
    limited to 0 ns (four splits of 16,384 keys, so that a timer tick falls
    inside some wait), FA_ERR_TIMEOUT is recorded, and every output row is
    either exactly what a normal call gives (all of its splits finished) or NaN
    (a split gave up and marked its partial invalid) -- never a blend of stale
    workspace bytes.  A normal call after it must pass parity."""
    q, k, v = make_qkv(2, 4, 1, 65536, 128, seed=51)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = fa.fa_fwd_splitkv(qd, kd, vd, num_splits=4)
    need = fa.fa_fwd_splitkv_workspace_bytes(2, 4, 1, 65536, 128, 4)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert fa.fa_selftest_splitkv_timeout(qd, kd, vd, o, lse, ws, 128 ** -0.5, 0, num_splits=4) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_device_status() == fa.FA_OK  # cleared by the read
    nan_rows = torch.isnan(lse)
    assert nan_rows.any()
    assert torch.equal(lse[~nan_rows], lse_ref[~nan_rows])
    assert torch.equal(o[~nan_rows], o_ref[~nan_rows])
    assert torch.isnan(o[nan_rows].float()).all()
    qs, ks, vs = make_qkv(1, 2, 3, 3000, 128, seed=52)
    og, lg = run_gpu(qs, ks, vs, 128 ** -0.5, False, splits=0)
    compare(og, lg, *oracle.attn_fwd(*(bf16_bits(t) for t in (qs, ks, vs)), 128 ** -0.5, False), "after timeout")
