"""The head split on one GPU: every rank's share of one workload, run in turn.

Each rank of a split writes only the rows of O and LSE of its own block of
heads (contiguous blocks of the flattened B*H axis).  Here the ranks' calls
run one after another on one GPU into the same output buffers (a rank's call
waits on nothing another rank does, so running them in turn is exactly what N
GPUs would compute): after every call the rows of the ranks still to come must
be untouched, and after the last one O and LSE must equal a single whole-
workload call bit for bit, which the parity tests tie to the oracle.
"""
import numpy as np
import pytest
import torch

import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import make_qkv
from exact_attention_82_gb300.shard import fa_fwd_shard, head_range

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3, 7])
@pytest.mark.parametrize("causal,D,window", [(False, 128, None), (True, 64, None),
                                             (False, 128, (100, 0))])
def test_split_heads_equal_one_call(world, causal, D, window):
    B, H, S = 2, 3, 300   # 6 heads: 7 ranks leave one rank without work
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, D, seed=55))
    if window is None:
        o_ref, lse_ref = fa.fa_fwd(q, k, v, causal=causal)
    else:
        o_ref, lse_ref = fa.fa_fwd_window(q, k, v, *window)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    for rank in range(world):
        start, count = fa_fwd_shard(q, k, v, o, lse, rank, world, causal=causal, window=window)
        assert (start, count) == head_range(B * H, world, rank)
        torch.cuda.synchronize()
        of = o.reshape(B * H, S, D)
        lf = lse.reshape(B * H, S)
        done = start + count
        assert not torch.isnan(of[:done]).any() and not torch.isnan(lf[:done]).any()
        assert torch.isnan(of[done:]).all() and torch.isnan(lf[done:]).all()  # later ranks' rows untouched
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert fa.fa_device_status() == fa.FA_OK


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("per_head,causal,stride", [(True, False, 1), (False, True, 2)])
def test_split_heads_block_mask_equal_one_call(world, per_head, causal, stride):
    from exact_attention_82_gb300.inputs import dilated_block_mask, random_block_mask

    B, H, S, D = 1, 6, 700, 128
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, D, seed=56))
    n = -(-S // 128)
    mask = (random_block_mask(B * H, n, n, 0.5, 57) if per_head else dilated_block_mask(n, n, 2, causal)).cuda()
    o_ref, lse_ref = fa.fa_fwd_blockmask(q, k, v, mask, -1, 0 if causal else -1, pair_stride=stride)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    for rank in range(world):
        start, count = fa_fwd_shard(q, k, v, o, lse, rank, world, causal=causal, block_mask=mask,
                                    pair_stride=stride)
        assert (start, count) == head_range(B * H, world, rank)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
    fin = torch.isfinite(lse_ref)
    assert torch.equal(lse[fin], lse_ref[fin])
    assert fa.fa_device_status() == fa.FA_OK
