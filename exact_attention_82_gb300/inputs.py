"""Seeded synthetic inputs for the attention-forward workloads.

This module is shared by the CUDA path (tests, bench, smoke check) and by the
oracle's tests.  It holds none of the attention arithmetic: only the workload
table, seeded normal draws and the rounding of those draws to bf16 or e4m3.

Recipe (the pages fix none of it; every workload draws i.i.d. N(0, 1)):
  * a torch CPU ``Generator`` seeded with ``seed``;
  * Q, then K, then V, each drawn as float32 ``randn`` of its full shape and
    rounded to bf16 (round-to-nearest-even, torch's ``.to(bfloat16)``);
  * for the peaky-softmax workload Q is then multiplied by 4, which is exact
    in bf16 (a power of two, far from overflow).
  * 8-bit (e4m3) inputs: the same float32 draws, each tensor given its own
    scale (descale = amax / 448, 448 being e4m3's largest finite value) and
    rounded to e4m3 codes by torch's ``.to(float8_e4m3fn)``; the codes travel
    as uint8 and the real value is code * descale.
Workload i uses seed ``SEED_BASE + i``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

SEED_BASE = 20260


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    q_mult: float = 1.0
    window_left: int = -1   # keys i - window_left .. i (+ window_right); -1: unbounded
    path: str = "fwd"       # "fwd", "splitkv" (decode, key-split), "bwd" (gradients), "fp8",
                            # "blockmask" (a dilated block pattern)
    dilation: int = 0       # "blockmask": the pattern's stride (also the pairing stride)

    @property
    def window(self):
        """(wl, wr) of the key band: causal is (-1, 0), full attention (-1, -1)."""
        return (self.window_left, 0 if self.causal else -1)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def block_mask(self) -> torch.Tensor:
        """The "blockmask" path's uint8 [1, ceil(Sq/128), ceil(Sk/128)] mask."""
        return dilated_block_mask(-(-self.Sq // BLOCK), -(-self.Sk // BLOCK), self.dilation, self.causal)

    @property
    def flops(self) -> float:
        """Matmul FLOPs 4*B*H*Sq*Sk*D, halved when causal (the metric's rule); with a
        bounded window or a block mask, 4*B*H*D times the exact number of allowed
        (query, key) pairs."""
        if self.path == "blockmask":
            return 4.0 * self.B * self.H * self.D * float(block_mask_pairs(self.block_mask[0].numpy(), self.Sq,
                                                                           self.Sk, self.causal))
        if self.window_left >= 0:
            i = np.arange(self.Sq)
            hi = np.minimum(self.Sk - 1, i if self.causal else self.Sk - 1)
            lo = np.maximum(0, i - self.window_left)
            return 4.0 * self.B * self.H * self.D * float(np.maximum(hi - lo + 1, 0).sum())
        f = 4.0 * self.B * self.H * self.Sq * self.Sk * self.D
        if self.path == "bwd":
            f *= 2.5  # five products (dV, dP, dQ, dK, and S recomputed) against the forward's two
        return f / 2 if self.causal else f

    @property
    def hbm_bytes(self) -> float:
        """Algorithmic HBM bytes: Q, K, V read once, O and LSE written once."""
        eb = 1 if self.path == "fp8" else 2
        mask = -(-self.Sq // BLOCK) * -(-self.Sk // BLOCK) if self.path == "blockmask" else 0
        return float(self.B * self.H * (eb * (self.Sq + 2 * self.Sk) * self.D + 2 * self.Sq * self.D
                                        + 4 * self.Sq) + mask)

    def describe(self) -> str:
        c = "causal" if self.causal else "non-causal"
        if self.window_left >= 0:
            c += f", sliding window of {self.window_left + 1} keys"
        if self.path == "splitkv":
            c += ", split-KV decode"
        if self.path == "bwd":
            c += ", backward (dQ, dK, dV)"
        if self.path == "blockmask":
            c += (f", dilated block mask (128 x 128 blocks; key block c kept for query block a iff "
                  f"a - c is a multiple of {self.dilation}), pair_stride {self.dilation}")
        extra = f", Q x{self.q_mult:g}" if self.q_mult != 1.0 else ""
        dt = "e4m3 (per-tensor scale)" if self.path == "fp8" else "bf16"
        return (f"B={self.B},H={self.H},Sq={self.Sq},Sk={self.Sk},D={self.D}, {dt} N(0,1)"
                f"{extra}, scale=1/sqrt({self.D}), {c}")


# The attention-forward workloads, in order (index = seed offset).
WORKLOADS = [
    Workload("b1h1s128d64", 1, 1, 128, 128, 64, False),
    Workload("b8h16s2048d128", 8, 16, 2048, 2048, 128, False),
    Workload("b4h16s4096d128_causal", 4, 16, 4096, 4096, 128, True),
    Workload("b1h16s16384d128_causal", 1, 16, 16384, 16384, 128, True),
    Workload("b16h32s1000d64_causal_q4", 16, 32, 1000, 1000, 64, True, 4.0),
    # sliding-window causal attention (4096-key window), long sequence
    Workload("b2h32s16384d128_swa4096", 2, 32, 16384, 16384, 128, True, 1.0, 4095),
    # decode: one query row per head against a 16384-key cache (HBM-bound)
    Workload("b8h32q1s16384d128_decode", 8, 32, 1, 16384, 128, False, path="splitkv"),
    # backward of the headline and the causal workloads
    Workload("b8h16s2048d128_bwd", 8, 16, 2048, 2048, 128, False, path="bwd"),
    Workload("b4h16s4096d128_causal_bwd", 4, 16, 4096, 4096, 128, True, path="bwd"),
    # 8-bit (e4m3) Q, K, V with per-tensor scales, the headline shape and causal
    Workload("b8h16s2048d128_fp8", 8, 16, 2048, 2048, 128, False, path="fp8"),
    Workload("b4h16s4096d128_causal_fp8", 4, 16, 4096, 4096, 128, True, path="fp8"),
    # a dilated causal block pattern (every 2nd 128-key block): a quarter of the pairs
    Workload("b2h32s16384d128_dilated2_causal", 2, 32, 16384, 16384, 128, True, path="blockmask", dilation=2),
]
BLOCK = 128  # rows and keys per block of a block mask


def make_qkv(B: int, H: int, Sq: int, Sk: int, D: int, seed: int, q_mult: float = 1.0):
    """bf16 CPU tensors q [B,H,Sq,D], k and v [B,H,Sk,D] from one seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, Sq, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, H, Sk, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, H, Sk, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    if q_mult != 1.0:
        q = (q.to(torch.float32) * q_mult).to(torch.bfloat16)
    return q, k, v


E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor scaling of a float32 CPU tensor to e4m3: returns (uint8 codes,
    descale) with descale = amax / 448 as a float32 value (1.0 for an all-zero
    tensor) and codes = round-to-nearest(x / descale) in e4m3."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    descale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    y = (x.to(torch.float32) / descale).clamp(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), descale


def make_qkv_fp8(B: int, H: int, Sq: int, Sk: int, D: int, seed: int, q_mult: float = 1.0):
    """e4m3 codes (uint8 CPU tensors) q [B,H,Sq,D], k and v [B,H,Sk,D] and their
    descales (dq, dk, dv), from the same draws as make_qkv."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, Sq, D), generator=g, dtype=torch.float32) * q_mult
    k = torch.randn((B, H, Sk, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Sk, D), generator=g, dtype=torch.float32)
    (qc, dq), (kc, dk), (vc, dv) = (quantize_e4m3(t) for t in (q, k, v))
    return (qc, kc, vc), (dq, dk, dv)


def workload_qkv(index: int):
    """bf16 inputs of workload ``index`` with its own seed."""
    w = WORKLOADS[index]
    return make_qkv(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + index, w.q_mult)


def workload_qkv_fp8(index: int):
    """e4m3 inputs (codes, descales) of workload ``index`` with its own seed."""
    w = WORKLOADS[index]
    return make_qkv_fp8(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + index, w.q_mult)


def u8_codes(t: torch.Tensor) -> np.ndarray:
    """uint8 numpy copy of a CPU code tensor, for the oracle."""
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns (uint16 numpy) of a bf16 CPU tensor, for the oracle."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def random_block_mask(heads: int, n_qb: int, n_kb: int, keep: float, seed: int) -> torch.Tensor:
    """uint8 CPU block mask [heads, n_qb, n_kb]: each block kept with probability
    ``keep``, drawn from one seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return (torch.rand((heads, n_qb, n_kb), generator=g) < keep).to(torch.uint8)


def dilated_block_mask(n_qb: int, n_kb: int, stride: int, causal: bool = False) -> torch.Tensor:
    """uint8 CPU block mask [1, n_qb, n_kb] of a dilated block pattern: query block a
    keeps key block c iff (a - c) is a multiple of ``stride`` (and c <= a when
    ``causal``).  The pages name dilated patterns beside sliding windows without
    defining one; this is the plainest block-level reading (every stride-th block
    counted from the diagonal), not a pattern the pages fix."""
    a = torch.arange(n_qb).view(-1, 1)
    c = torch.arange(n_kb).view(1, -1)
    keep = (a - c) % stride == 0
    if causal:
        keep &= c <= a
    return keep.to(torch.uint8).unsqueeze(0).contiguous()


def block_mask_pairs(mask, Sq: int, Sk: int, causal: bool) -> int:
    """Allowed (query, key) pairs of a [n_qb, n_kb] block mask (FLOP accounting):
    a kept block contributes its rows x keys, a causal diagonal block its lower
    triangle (Sq == Sk), a block above the diagonal nothing."""
    n = 0
    for a in range(mask.shape[0]):
        rq = min(BLOCK, Sq - BLOCK * a)
        for c in range(mask.shape[1]):
            if not mask[a, c] or (causal and c > a):
                continue
            rk = min(BLOCK, Sk - BLOCK * c)
            n += rq * (rq + 1) // 2 if (causal and c == a) else rq * rk
    return n
