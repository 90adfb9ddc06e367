"""GPU parity of fa_fwd_blockmask (attention over the key blocks a block mask
keeps) against the fp64 block-mask oracle.

"FlashAttention-2 — L3 Cross-Paper Synthesis", §5 item 4: causal block
skipping generalises to sliding windows and dilated patterns as one
sparse-block-skip mechanism.  The masks below are random (per head and shared
by every head), dilated (every 2nd / 3rd key block from the diagonal, with and
without causal), combined with a band, with query blocks that keep nothing
(O = 0, LSE = -inf) and with more work items than SMs; both head dims (16-bit
D = 64 takes the separate-P pipeline, D = 128 the P-over-S one).
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import bf16_bits, dilated_block_mask, make_qkv, random_block_mask
from parity_util import TOL_LSE, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu

BLK = (fa.FA_BLOCK_M, fa.FA_BLOCK_N)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert fa.fa_device_status() == fa.FA_OK


def _nb(S, b):
    return -(-S // b)


def run_mask(q, k, v, mask, window=(-1, -1), scale=None, pair_stride=1):
    D = q.shape[3]
    scale = D ** -0.5 if scale is None else scale
    o, lse = fa.fa_fwd_blockmask(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), window[0], window[1], scale=scale,
                                 pair_stride=pair_stride)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def compare_masked(og, lg, ro, rl, what):
    """Rows with no allowed key must be exactly O = 0, LSE = -inf; the rest within
    the forward's tolerances."""
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lg), empty), f"{what}: rows with LSE = -inf differ"
    assert np.all(og[empty] == 0.0), f"{what}: an empty row has O != 0"
    live = ~empty
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg[live])), f"{what}: non-finite"
    if not live.any():
        return
    d = np.abs(og[live] - ro[live])
    dl = np.abs(lg[live] - rl[live])
    msg = f"{what}: max|dO|={d.max():.3e} mean|dO|={d.mean():.3e} max|dLSE|={dl.max():.3e}"
    assert d.max() <= TOL_O_MAX, msg
    assert d.mean() <= TOL_O_MEAN, msg
    assert dl.max() <= TOL_LSE, msg


def check(q, k, v, mask, window, what, scale=None, pair_stride=1):
    D = q.shape[3]
    scale = D ** -0.5 if scale is None else scale
    og, lg = run_mask(q, k, v, mask, window, scale, pair_stride)
    ro, rl = oracle.attn_fwd_blockmask(*(bf16_bits(t) for t in (q, k, v)), scale, mask.numpy(),
                                       window=window, block=BLK)
    compare_masked(og, lg, ro, rl, what)


def _patterns(H, B, n_qb, n_kb, seed):
    return {
        "random_shared": random_block_mask(1, n_qb, n_kb, 0.5, seed),
        "random_per_head": random_block_mask(B * H, n_qb, n_kb, 0.4, seed + 1),
        "dilated2": dilated_block_mask(n_qb, n_kb, 2),
        "dilated3_causal": dilated_block_mask(n_qb, n_kb, 3, causal=True),
        "sparse_with_empty_blocks": random_block_mask(B * H, n_qb, n_kb, 0.15, seed + 2),
    }


@pytest.mark.parametrize("pattern", ["random_shared", "random_per_head", "dilated2", "dilated3_causal",
                                     "sparse_with_empty_blocks"])
@pytest.mark.parametrize("D", [64, 128])
def test_blockmask_parity(pattern, D):
    B, H, S = 2, 3, 1000
    q, k, v = make_qkv(B, H, S, S, D, seed=500 + D + len(pattern))
    mask = _patterns(H, B, _nb(S, 128), _nb(S, 128), 40 + D)[pattern]
    window = (-1, 0) if "causal" in pattern else (-1, -1)
    check(q, k, v, mask, window, f"{pattern} D{D}")


@pytest.mark.parametrize("window", [(300, 0), (0, 0), (130, 200), (-1, 50)], ids=lambda w: f"wl{w[0]}_wr{w[1]}")
@pytest.mark.parametrize("D", [64, 128])
def test_blockmask_with_band(window, D):
    B, H, S = 1, 4, 777
    q, k, v = make_qkv(B, H, S, S, D, seed=600 + window[0] + D)
    n = _nb(S, 128)
    mask = random_block_mask(B * H, n, n, 0.6, 70 + D)
    check(q, k, v, mask, window, f"band {window} D{D}")


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (129, 300), (300, 129), (256, 256), (1100, 700), (65, 1500)])
def test_blockmask_ragged_lengths(Sq, Sk):
    q, k, v = make_qkv(2, 2, Sq, Sk, 128, seed=Sq * 7 + Sk)
    mask = random_block_mask(4, _nb(Sq, 128), _nb(Sk, 128), 0.5, Sq + Sk)
    check(q, k, v, mask, (-1, -1), f"Sq{Sq} Sk{Sk}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("keep", [0.3, 0.9])
def test_blockmask_long_key_rows(D, keep):
    # 157 key tiles per row: the MMA warp's participation bits cover 128 load-order
    # tiles at a time and are refilled past them, and a mask row is scanned in
    # five 32-tile batches
    B, H, Sq, Sk = 1, 2, 300, 20000
    q, k, v = make_qkv(B, H, Sq, Sk, D, seed=950 + D + int(keep * 10))
    mask = random_block_mask(B * H, _nb(Sq, 128), _nb(Sk, 128), keep, 95 + D)
    mask[0, 0, 130:] = 0   # a row whose kept tiles end before the second window
    mask[1, 1, :140] = 0   # a row whose kept tiles start in the second window
    check(q, k, v, mask, (-1, -1), f"long rows D{D} keep{keep}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("stride,causal", [(2, True), (3, False), (4, True)])
def test_dilated_with_matching_pair_stride(D, stride, causal):
    # query blocks a and a + stride share an item: for a dilated pattern they keep
    # the same key blocks (causal: one more for the second); 11 query blocks leave
    # a tail of blocks paired with their neighbours
    B, H, S = 2, 2, 1400
    q, k, v = make_qkv(B, H, S, S, D, seed=1000 + D + stride)
    n = _nb(S, 128)
    mask = dilated_block_mask(n, n, stride, causal=causal)
    check(q, k, v, mask, (-1, 0) if causal else (-1, -1), f"dilated {stride} D{D}", pair_stride=stride)


@pytest.mark.parametrize("D", [64, 128])
def test_pair_stride_changes_nothing_but_the_schedule(D):
    # every stride (1 .. beyond the block count) gives bitwise the same O and LSE,
    # for a random per-head mask with a band and query blocks that keep nothing
    B, H, S = 1, 3, 1300
    q, k, v = make_qkv(B, H, S, S, D, seed=1100 + D)
    n = _nb(S, 128)
    mask = random_block_mask(B * H, n, n, 0.4, 110 + D)
    mask[1, 2] = 0
    for window in [(-1, -1), (500, 0)]:
        ref = run_mask(q, k, v, mask, window, pair_stride=1)
        for s in (2, 3, 5, 7, 100):
            got = run_mask(q, k, v, mask, window, pair_stride=s)
            assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), (window, s)
    check(q, k, v, mask, (500, 0), f"stride 3 band D{D}", pair_stride=3)


@pytest.mark.parametrize("D", [64, 128])
def test_blockmask_many_items(D):
    # 320 items of 256 query rows on at most one CTA per SM: persistent CTAs take
    # several items whose sub-tiles keep different, gapped sets of key tiles
    B, H, S = 4, 16, 1100
    q, k, v = make_qkv(B, H, S, S, D, seed=700 + D)
    n = _nb(S, 128)
    mask = random_block_mask(B * H, n, n, 0.35, 80 + D)
    check(q, k, v, mask, (-1, -1), f"many items D{D}")


@pytest.mark.parametrize("D", [64, 128])
def test_blockmask_empty_query_blocks(D):
    # query blocks that keep nothing: in one sub-tile of an item, in both, and a
    # band that leaves rows of kept blocks empty
    B, H, S = 1, 2, 900
    q, k, v = make_qkv(B, H, S, S, D, seed=800 + D)
    n = _nb(S, 128)
    mask = torch.ones((B * H, n, n), dtype=torch.uint8)
    mask[0, 0] = 0          # item 0: sub-tile 0 empty, sub-tile 1 not
    mask[0, 3] = 0          # item 1: sub-tile 1 empty
    mask[1, 4:6] = 0        # item 2: both sub-tiles empty
    mask[1, 6, 6] = 0       # with the (0, 0) band below, rows of query block 6 lose their only key
    for window in [(-1, -1), (0, 0)]:
        og, lg = run_mask(q, k, v, mask, window)
        ro, rl = oracle.attn_fwd_blockmask(*(bf16_bits(t) for t in (q, k, v)), D ** -0.5, mask.numpy(),
                                           window=window, block=BLK)
        assert np.isneginf(rl[0, 0, :128]).all() and np.isneginf(rl[0, 1, 512:768]).all()
        compare_masked(og, lg, ro, rl, f"empty blocks D{D} window {window}")
    # every block masked: the whole output is O = 0, LSE = -inf
    og, lg = run_mask(q, k, v, torch.zeros((1, n, n), dtype=torch.uint8))
    assert np.all(og == 0) and np.all(np.isneginf(lg))


@pytest.mark.parametrize("D", [64, 128])
def test_skipped_key_blocks_are_never_read(D):
    # key blocks no query block keeps hold NaN: the result must be bitwise the
    # one with zeros there (a skipped tile that were loaded and multiplied, even
    # by P = 0, would turn O into NaN)
    B, H, S = 2, 2, 1024
    q, k, v = make_qkv(B, H, S, S, D, seed=900 + D)
    n = _nb(S, 128)
    mask = random_block_mask(1, n, n, 0.6, 90 + D)
    mask[0, :, 0] = 1                     # block 0 is kept by every query block
    mask[0, :, 3] = 0
    mask[0, :, 6] = 0
    kz, vz, kn, vn = k.clone(), v.clone(), k.clone(), v.clone()
    for c in (3, 6):
        rows = slice(c * 128, c * 128 + 128)
        kz[:, :, rows] = 0
        vz[:, :, rows] = 0
        kn[:, :, rows] = float("nan")
        vn[:, :, rows] = float("nan")
    o1, l1 = run_mask(q, kz, vz, mask)
    o2, l2 = run_mask(q, kn, vn, mask)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ro, rl = oracle.attn_fwd_blockmask(*(bf16_bits(t) for t in (q, kz, vz)), D ** -0.5, mask.numpy(), block=BLK)
    compare_masked(o1, l1, ro, rl, f"NaN blocks D{D}")


@pytest.mark.parametrize("window", [(200, 0), (0, 7), (129, 128)])
def test_all_ones_mask_equals_window_bitwise(window):
    q, k, v = (t.cuda() for t in make_qkv(2, 3, 555, 555, 128, seed=3))
    n = _nb(555, 128)
    o1, l1 = fa.fa_fwd_window(q, k, v, window[0], window[1])
    o2, l2 = fa.fa_fwd_blockmask(q, k, v, torch.ones((1, n, n), dtype=torch.uint8, device="cuda"),
                                 window[0], window[1])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_matches_oracle(causal):
    q, k, v = make_qkv(2, 2, 700, 700, 64, seed=5)
    n = _nb(700, 128)
    check(q, k, v, torch.ones((1, n, n), dtype=torch.uint8), (-1, 0) if causal else (-1, -1),
          f"all ones causal{int(causal)}")


def test_bool_mask_and_shape_checks():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 300, 300, 64, seed=6))
    m = dilated_block_mask(3, 3, 2).cuda()
    o1, l1 = fa.fa_fwd_blockmask(q, k, v, m)
    o2, l2 = fa.fa_fwd_blockmask(q, k, v, m.bool())
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(ValueError):
        fa.fa_fwd_blockmask(q, k, v, torch.ones((1, 3, 2), dtype=torch.uint8, device="cuda"))
    with pytest.raises(fa.FAError):
        fa.fa_fwd_blockmask(q, k, v, torch.ones((3, 3, 3), dtype=torch.uint8, device="cuda"))
