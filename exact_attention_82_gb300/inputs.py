"""Seeded synthetic inputs for the attention-forward workloads.

This module is shared by the CUDA path (tests, bench, smoke check) and by the
oracle's tests.  It holds none of the attention arithmetic: only the workload
table, seeded normal draws and the rounding of those draws to bf16.

Recipe (the pages fix none of it; all five workloads are i.i.d. N(0, 1)):
  * a torch CPU ``Generator`` seeded with ``seed``;
  * Q, then K, then V, each drawn as float32 ``randn`` of its full shape and
    rounded to bf16 (round-to-nearest-even, torch's ``.to(bfloat16)``);
  * for the peaky-softmax workload Q is then multiplied by 4, which is exact
    in bf16 (a power of two, far from overflow).
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
    path: str = "fwd"       # "fwd", "splitkv" (decode, key-split) or "bwd" (gradients)

    @property
    def window(self):
        """(wl, wr) of the key band: causal is (-1, 0), full attention (-1, -1)."""
        return (self.window_left, 0 if self.causal else -1)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Matmul FLOPs 4*B*H*Sq*Sk*D, halved when causal (the metric's rule); with a
        bounded window, 4*B*H*D times the exact number of allowed (query, key) pairs."""
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
        return float(self.B * self.H * (2 * (self.Sq + 2 * self.Sk) * self.D + 2 * self.Sq * self.D
                                        + 4 * self.Sq))

    def describe(self) -> str:
        c = "causal" if self.causal else "non-causal"
        if self.window_left >= 0:
            c += f", sliding window of {self.window_left + 1} keys"
        if self.path == "splitkv":
            c += ", split-KV decode"
        if self.path == "bwd":
            c += ", backward (dQ, dK, dV)"
        extra = f", Q x{self.q_mult:g}" if self.q_mult != 1.0 else ""
        return (f"B={self.B},H={self.H},Sq={self.Sq},Sk={self.Sk},D={self.D}, bf16 N(0,1)"
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
]


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


def workload_qkv(index: int):
    """Inputs of workload ``index`` (0..4) with its own seed."""
    w = WORKLOADS[index]
    return make_qkv(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + index, w.q_mult)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns (uint16 numpy) of a bf16 CPU tensor, for the oracle."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
