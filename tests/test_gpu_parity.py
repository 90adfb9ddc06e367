"""GPU parity: the sm_103a kernel, called through the C ABI, against the fp64
oracle on the same seeded bf16 inputs, element by element (small and
mid-size shapes spanning several tiles and a ragged tail) and on sampled rows
at the five full workload sizes, in the launch configuration the benchmark
times."""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import SEED_BASE, WORKLOADS, bf16_bits, make_qkv, workload_qkv
from parity_util import compare, full_parity, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    """Every test must leave the on-device status word at FA_OK."""
    yield
    assert fa.fa_device_status() == fa.FA_OK


# ------------------------------------------------------------ small / ragged
SMALL = [
    # B, H, Sq, Sk, D
    (1, 1, 128, 128, 64),
    (1, 1, 128, 128, 128),
    (1, 1, 1, 1, 64),
    (1, 1, 1, 1, 128),
    (1, 1, 2, 2, 64),
    (3, 1, 63, 63, 128),
    (1, 3, 64, 64, 64),
    (1, 1, 65, 65, 128),
    (3, 3, 127, 127, 64),
    (1, 3, 129, 129, 128),
    (2, 3, 389, 389, 128),
    (1, 2, 1000, 1000, 64),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_parity_small(shape, causal):
    B, H, Sq, Sk, D = shape
    full_parity(B, H, Sq, Sk, D, causal, seed=1000 + sum(shape))


@pytest.mark.parametrize("Sq,Sk", [(1, 300), (200, 70), (128, 1), (300, 511), (77, 1024)])
@pytest.mark.parametrize("D", [64, 128])
def test_parity_rectangular_noncausal(Sq, Sk, D):
    full_parity(2, 2, Sq, Sk, D, False, seed=Sq * 7 + Sk)


def test_parity_peaky_softmax():
    """Q x4 (the peaky workload's recipe) at a small size, both head dims."""
    for D in (64, 128):
        full_parity(2, 2, 300, 300, D, True, seed=77, q_mult=4.0)


def test_parity_other_scale():
    full_parity(1, 2, 257, 257, 128, False, seed=5, scale=0.3)


# ------------------------------------------------ the benchmark's workloads
@pytest.mark.parametrize("index", range(len(WORKLOADS)), ids=[w.name for w in WORKLOADS])
def test_parity_workload(index):
    w = WORKLOADS[index]
    if w.path == "bwd":
        pytest.skip("backward workloads: tests/test_gpu_bwd.py")
    q, k, v = workload_qkv(index)
    if w.path == "blockmask":
        _parity_blockmask_workload(w, index, q, k, v)
        return
    win = w.window if w.window_left >= 0 else None
    og, lg = run_gpu(q, k, v, w.scale, w.causal, window=win,
                     splits=0 if w.path == "splitkv" else None)
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    if w.B * w.H * w.Sq <= 4096:
        orf, lrf = oracle.attn_fwd(qb, kb, vb, w.scale, w.causal, w.window)
        compare(og, lg, orf, lrf, w.name)
        return
    bh, rows = sample_rows(w.B, w.H, w.Sq, n_random=160, seed=index)
    orf, lrf = oracle.attn_fwd_rows(qb, kb, vb, bh, rows, w.scale, w.causal, w.window)
    og2 = og.reshape(w.B * w.H, w.Sq, w.D)[bh, rows]
    lg2 = lg.reshape(w.B * w.H, w.Sq)[bh, rows]
    compare(og2, lg2, orf, lrf, w.name + " (sampled rows)")
    # properties that hold at any size: O is a convex combination of V rows
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    vmax = v.float().amax(dim=2, keepdim=True).double().numpy()
    vmin = v.float().amin(dim=2, keepdim=True).double().numpy()
    assert np.all(og <= vmax + 2e-2) and np.all(og >= vmin - 2e-2)


def _parity_blockmask_workload(w, index, q, k, v):
    """The block-mask workload in the benchmark's launch (its pattern and pairing
    stride): whole query blocks of a few heads (first, second and last blocks
    among them) against the block-mask oracle on those rows with every key, and
    at every element the convex-combination bound."""
    mask = w.block_mask
    o, l = fa.fa_fwd_blockmask(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), w.window[0], w.window[1],
                               scale=w.scale, pair_stride=w.dilation)
    torch.cuda.synchronize()
    BH, Bq = w.B * w.H, 128
    og = o.float().cpu().double().numpy().reshape(BH, w.Sq, w.D)
    lg = l.cpu().double().numpy().reshape(BH, w.Sq)
    qb, kb, vb = (bf16_bits(t).reshape(BH, -1, w.D) for t in (q, k, v))
    rng = np.random.default_rng(index)
    n_qb = -(-w.Sq // Bq)
    for bh in sorted(set([0, BH - 1] + [int(x) for x in rng.integers(0, BH, 2)])):
        for a in sorted(set([0, 1, n_qb - 1] + [int(x) for x in rng.integers(0, n_qb, 2)])):
            rows = slice(a * Bq, min(w.Sq, a * Bq + Bq))
            win = (-1, a * Bq) if w.causal else (-1, -1)
            ro, rl = oracle.attn_fwd_blockmask(qb[bh][rows][None, None], kb[bh][None, None], vb[bh][None, None],
                                               w.scale, mask.numpy()[:, a:a + 1], window=win, block=(Bq, Bq))
            compare(og[bh][rows], lg[bh][rows], ro[0, 0], rl[0, 0], f"{w.name} head {bh} block {a}")
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    vmax = v.float().amax(dim=2).double().numpy().reshape(BH, 1, w.D)
    vmin = v.float().amin(dim=2).double().numpy().reshape(BH, 1, w.D)
    assert np.all(og <= vmax + 2e-2) and np.all(og >= vmin - 2e-2)


# ------------------------------------------------------------- properties
def test_deterministic_bitwise():
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 777, 777, 128, seed=3))
    o1, l1 = fa.fa_fwd(q, k, v, causal=True)
    o2, l2 = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_guard_bands_untouched():
    """Outputs carved out of larger buffers: bytes around O and LSE keep their canary."""
    B, H, S, D = 2, 3, 300, 64
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, D, seed=4))
    pad = 4096
    n_o = B * H * S * D
    obuf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * S + 2 * pad,), -3.0, dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + n_o].view(B, H, S, D)
    lse = lbuf[pad:pad + B * H * S].view(B, H, S)
    fa.fa_fwd(q, k, v, o=o, lse=lse, causal=True)
    torch.cuda.synchronize()
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[pad + n_o:] == 7.0)
    assert torch.all(lbuf[:pad] == -3.0) and torch.all(lbuf[pad + B * H * S:] == -3.0)
    ref_o, ref_l = oracle.attn_fwd(*(bf16_bits(t.cpu()) for t in (q, k, v)), D ** -0.5, True)
    compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_o, ref_l, "guard")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_output_16_byte_aligned_only(D, causal):
    """O at an address that is 16-byte but not 32-byte aligned (the least the
    interface asks for): the bytes equal those written to a 512-byte aligned O,
    and the guard bands stay."""
    B, H, S = 2, 3, 300
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, D, seed=12))
    n_o = B * H * S * D
    obuf = torch.full((n_o + 64,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = obuf[8:8 + n_o].view(B, H, S, D)  # 16 bytes past a 512-byte aligned allocation
    assert o.data_ptr() % 32 == 16
    o_ref, l_ref = fa.fa_fwd(q, k, v, causal=causal)
    _, lse = fa.fa_fwd(q, k, v, o=o, causal=causal)
    torch.cuda.synchronize()
    assert o_ref.data_ptr() % 32 == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert torch.all(obuf[:8] == 7.0) and torch.all(obuf[8 + n_o:] == 7.0)


def test_side_stream():
    s = torch.cuda.Stream()
    q, k, v = make_qkv(1, 2, 200, 200, 128, seed=8)
    with torch.cuda.stream(s):
        og, lg = run_gpu(q, k, v, 128 ** -0.5, False, stream=s)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), 128 ** -0.5, False)
    compare(og, lg, *ref, "side stream")


def test_identical_v_rows_on_gpu():
    q, k, v = make_qkv(1, 2, 256, 256, 128, seed=9)
    v = v[:, :, :1].expand_as(v).contiguous()
    og, _ = run_gpu(q, k, v, 128 ** -0.5, False)
    want = v[:, :, :1].float().double().numpy()
    assert np.max(np.abs(og - want)) <= 2e-2


def test_bounded_wait_gives_up_and_reports():
    """A wait nothing satisfies ends after its limit with FA_ERR_TIMEOUT in the
    status word; the context stays usable."""
    assert fa.fa_device_status() == fa.FA_OK
    assert fa.fa_selftest_bounded_wait(20_000) == fa.FA_OK  # 20 ms limit
    assert fa.fa_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_device_status() == fa.FA_OK  # cleared by the read
    full_parity(1, 1, 128, 128, 64, False, seed=1)  # context still works


@pytest.mark.parametrize("D", [64, 128])
def test_forward_kernel_gives_up_cleanly(D):
    """The attention kernel's own give-up path, on one CTA's worth of work (one
    item of 256 query rows): with every wait limited to 0 ns, the first wait in
    progress when the global timer ticks gives up, raises the CTA's abort flag
    and records FA_ERR_TIMEOUT; the other roles stop, the producer and the MMA
    issuer wait (bounded) for their copies and MMAs in flight, TMEM is freed and
    the kernel returns.  The key sequence is long (65,536 keys, about a
    millisecond of tile waits), so that a timer tick falls inside some wait
    whatever the timer's resolution.  A normal call after it must pass parity,
    so the context is still usable."""
    assert fa.fa_device_status() == fa.FA_OK
    q, k, v = make_qkv(1, 1, 256, 65536, D, seed=31)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 256), dtype=torch.float32, device="cuda")
    assert fa.fa_selftest_fwd_timeout(q, k, v, o, lse, D ** -0.5, False, 0) == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_device_status() == fa.FA_OK  # cleared by the read
    full_parity(1, 2, 300, 300, D, True, seed=32)
    assert fa.fa_device_status() == fa.FA_OK


def _growing_scores(D, lift, causal, keys=(0, 128)):
    """Keys [keys[0], keys[1]) of the first key tile (index 0, processed last)
    score `lift` (in exp2 units) above every other key, so later tiles outgrow
    the max taken from the first tile processed."""
    B, H, S = 1, 2, 384
    q, k, v = make_qkv(B, H, S, S, D, seed=21)
    q = torch.ones_like(q)  # every score is (scale) * sum(k_j)
    target = lift * (D ** 0.5) / 1.4426950408889634 / D  # per-element key value
    k = k * 0.05
    a, b = keys
    k[:, :, a:b] = (k[:, :, a:b].float() + target).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lift", [40.0, 70.0])
@pytest.mark.parametrize("causal", [False, True])
def test_scores_growing_past_first_tile_max(D, lift, causal):
    """Large late scores: P grows to ~2^40 against the first tile's max (kept),
    or past 2^64 (the tile is redone against its true max, O rescaled)."""
    q, k, v = _growing_scores(D, lift, causal)
    og, lg = run_gpu(q, k, v, D ** -0.5, causal)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), D ** -0.5, causal)
    compare(og, lg, *ref, f"lift {lift} D{D}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("keys", [(0, 64), (64, 128), (60, 70)], ids=["first-half", "second-half", "both-halves"])
@pytest.mark.parametrize("causal", [False, True])
def test_scores_growing_in_part_of_a_tile(D, keys, causal):
    """Scores more than 2^64 past the max in use in only part of a key tile.
    The 16-bit D = 128 kernel hands P over in two halves (keys 0-63, 64-127):
    an overflow in the first half redoes the tile before anything is handed
    over; one only in the second half raises the max after the first half's
    product has reached O, rescales O and redoes the second half."""
    q, k, v = _growing_scores(D, 70.0, causal, keys)
    og, lg = run_gpu(q, k, v, D ** -0.5, causal)
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), D ** -0.5, causal)
    compare(og, lg, *ref, f"keys {keys} D{D}")


# ------------------------------------------------- many items per launch
# More (query block, head) items than SMs, so persistent CTAs walk several
# items each and hand Q and O buffers over between them; ragged lengths leave
# the second sub-tile empty in some items.  Every element against the oracle.
MANY = [
    # B, H, S, D, causal
    (2, 80, 300, 128, True),
    (3, 64, 600, 64, True),
    (2, 90, 333, 64, False),
    (1, 160, 257, 128, False),
]


@pytest.mark.parametrize("case", MANY, ids=lambda c: "b{}h{}s{}d{}{}".format(*c[:4], "c" if c[4] else ""))
def test_parity_many_items(case):
    B, H, S, D, causal = case
    full_parity(B, H, S, S, D, causal, seed=4242 + S + H)


def test_window_many_items():
    """D = 64 bounded bands run on persistent CTAs too."""
    q, k, v = make_qkv(2, 80, 500, 500, 64, seed=77)
    og, lg = run_gpu(q, k, v, 0.125, False, window=(100, 0))
    ref = oracle.attn_fwd(*(bf16_bits(t) for t in (q, k, v)), 0.125, False, (100, 0))
    compare(og, lg, *ref, "window (100, 0), 160 heads")
