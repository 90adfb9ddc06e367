"""fa_fwd_splitkv_noalloc: split-KV decode with the library's built-in scratch.

Some callers cannot allocate device memory -- for instance a process whose
device memory is all reserved up front by another allocator, or a code path
that must not take the synchronisation cudaMalloc can imply -- so this entry
point takes no workspace.  Its results must match fa_fwd_splitkv (the same
computation with a caller-provided workspace) within the parity tolerance,
on two calls in a row: the second call reuses the scratch the first one
left behind, with different sizes and a different split count.  Small calls
are also checked against the fp64 oracle directly, so a mistake shared by
both CUDA entry points (a wrong offset into the scratch, say) cannot hide.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.  It passes alone in a fresh
process as well as after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import exact_attention_82_gb300 as fa
from exact_attention_82_gb300.inputs import bf16_bits, make_qkv
from parity_util import compare

pytestmark = pytest.mark.gpu


def _noalloc(q, k, v, num_splits):
    """The new entry point through the C ABI; returns (O, LSE) as float64 numpy."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = fa.lib().fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, H, Sq, Sk, D,
                                         ctypes.c_float(D ** -0.5), num_splits, stream)
    assert st == fa.FA_OK, fa.fa_strerror(st)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def _with_workspace(q, k, v, num_splits):
    o, lse = fa.fa_fwd_splitkv(q, k, v, num_splits=num_splits)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def _close(a, b):
    (oa, la), (ob, lb) = a, b
    d = np.abs(oa - ob)
    assert np.all(np.isfinite(oa)) and np.all(np.isfinite(la))
    assert d.max() <= 2e-2 and d.mean() <= 2e-3, (d.max(), d.mean())
    assert np.abs(la - lb).max() <= 1e-3


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    # call 1: larger problem, automatic split count
    q, k, v = (t.cuda() for t in make_qkv(4, 16, 1, 9000, 128, seed=41))
    _close(_noalloc(q, k, v, 0), _with_workspace(q, k, v, 0))
    # call 2: other sizes and split count, so stale partials from call 1 would show
    q2, k2, v2 = (t.cuda() for t in make_qkv(2, 8, 3, 2500, 64, seed=42, q_mult=2.0))
    _close(_noalloc(q2, k2, v2, 5), _with_workspace(q2, k2, v2, 5))
    assert fa.fa_device_status() == fa.FA_OK


def test_noalloc_refuses_beyond_its_scratch():
    q, k, v = (t.cuda() for t in make_qkv(1, 64, 8, 16384, 128, seed=43))
    o = torch.empty_like(q)
    lse = torch.empty((1, 64, 8), dtype=torch.float32, device="cuda")
    need = fa.fa_fwd_splitkv_workspace_bytes(1, 64, 8, 16384, 128, 256)
    assert need > 16 << 20
    st = fa.lib().fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), 1, 64, 8, 16384, 128, ctypes.c_float(0.1),
                                         256, torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_ERR_SCRATCH_LIMIT


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    for (B, H, Sq, Sk, D, splits, seed) in [(1, 2, 3, 700, 64, 0, 44), (2, 1, 1, 1500, 128, 7, 45)]:
        q, k, v = make_qkv(B, H, Sq, Sk, D, seed=seed)
        og, lg = _noalloc(q.cuda(), k.cuda(), v.cuda(), splits)
        ro, rl = oracle.attn_fwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), D ** -0.5, False)
        compare(og, lg, ro, rl, f"noalloc B{B} H{H} Sq{Sq} Sk{Sk} D{D} splits{splits}")
    assert fa.fa_device_status() == fa.FA_OK
