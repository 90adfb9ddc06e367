"""Splitting one attention workload across ranks, one process per GPU.

Every (batch, head) pair is an independent problem with its own keys and
values: the launch grid of the source walk-through "FlashAttention-2 相比
FlashAttention-1，到底改了什么" (section "第一处源码差异：launch grid 怎么铺")
spans batch and heads, and "FlashAttention-2 — L3 Cross-Paper Synthesis"
(§2 item 2) makes query blocks and heads the outer, independent loop.  So the
B*H heads are dealt out in contiguous blocks: rank r owns heads
[start, start + count) of the flattened B*H axis and writes only those rows of
O and LSE.  Nothing moves between ranks on the data path; a caller that wants
the whole O on one device gathers the slices itself.

Because [B, H, S, D] is row-major with B*H outermost, a rank's heads are one
contiguous slice of every tensor, and its share of the work is one call of the
library's forward on that slice (B = 1, H = count).
"""
from __future__ import annotations


def head_range(bh: int, world: int, rank: int):
    """(start, count) of the heads rank `rank` of `world` owns out of `bh`:
    contiguous blocks of bh // world heads, the first bh % world ranks taking
    one more.  Blocks are disjoint and cover [0, bh); a rank beyond bh gets
    count 0."""
    if bh < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad partition request: bh={bh} world={world} rank={rank}")
    base, extra = divmod(bh, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def head_slice(t, start: int, count: int):
    """Heads [start, start + count) of a [B, H, ...] tensor as a contiguous
    [1, count, ...] view (no copy)."""
    B, H = t.shape[0], t.shape[1]
    flat = t.reshape(B * H, *t.shape[2:])
    return flat[start:start + count].reshape(1, count, *t.shape[2:])


def fa_fwd_shard(q, k, v, o, lse, rank: int, world: int, scale: float | None = None,
                 causal: bool = False, window=None, stream=None, block_mask=None, pair_stride: int = 1):
    """This rank's share of the forward over whole [B, H, S, D] tensors: the
    heads head_range(B*H, world, rank) of O and LSE are written, no other row
    is touched.  q, k, v, o, lse are CUDA tensors as fa_fwd takes them;
    `window` = (window_left, window_right) selects the banded call, and
    `block_mask` ([1 or B*H, n_qb, n_kb], as fa_fwd_blockmask takes it; a
    per-head mask is cut to the rank's heads) the block-mask call.  Returns
    (start, count)."""
    from . import fa_fwd, fa_fwd_blockmask, fa_fwd_window

    B, H = q.shape[0], q.shape[1]
    start, count = head_range(B * H, world, rank)
    if count == 0:
        return start, 0
    qs, ks, vs, os_, ls = (head_slice(t, start, count) for t in (q, k, v, o, lse))
    if block_mask is not None:
        ms = block_mask if block_mask.shape[0] == 1 else block_mask[start:start + count]
        wl, wr = window if window is not None else (-1, 0 if causal else -1)
        fa_fwd_blockmask(qs, ks, vs, ms, wl, wr, o=os_, lse=ls, scale=scale, pair_stride=pair_stride,
                         stream=stream)
    elif window is None:
        fa_fwd(qs, ks, vs, o=os_, lse=ls, scale=scale, causal=causal, stream=stream)
    else:
        fa_fwd_window(qs, ks, vs, window[0], window[1], o=os_, lse=ls, scale=scale, stream=stream)
    return start, count
