"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before touching the GPU.  No GPU needed."""
import glob
import os
import re

import pytest
import torch

import exact_attention_82_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# harmless fake device addresses: the calls below fail validation first
A = 1 << 20
A2 = 1 << 30
A3 = 1 << 34
A4 = 1 << 38
A5 = 1 << 40


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_strerror", "fa_device_status", "fa_selftest_bounded_wait",
              "fa_version"):
        assert n in names


@pytest.mark.parametrize("name", declared_functions())
def test_library_exports_declared_symbol(name):
    lib = fa.lib()
    assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_library_is_in_tree():
    assert os.path.commonpath([fa.library_path(), ROOT]) == ROOT
    assert os.path.exists(fa.library_path())


def test_version_and_strerror():
    assert fa.fa_version() >= 100
    for code in range(0, -14, -1):
        s = fa.fa_strerror(code)
        assert s and s != "unknown status", code
    assert fa.fa_strerror(12345) == "unknown status"


def call(q=A, k=A2, v=A3, o=A4, lse=A5, B=1, H=1, Sq=128, Sk=128, D=64, scale=0.125, causal=0):
    return fa.fa_fwd_raw(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, 0)


def test_null_pointers():
    assert call(q=0) == fa.FA_ERR_NULLPTR
    assert call(lse=0) == fa.FA_ERR_NULLPTR


def test_misaligned():
    assert call(k=A2 + 8) == fa.FA_ERR_MISALIGNED
    assert call(lse=A5 + 4) == fa.FA_ERR_MISALIGNED


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(Sq=0), dict(Sk=-1)])
def test_bad_shape(kw):
    assert call(**kw) == fa.FA_ERR_BAD_SHAPE


@pytest.mark.parametrize("D", [0, 32, 96, 256])
def test_unsupported_d(D):
    assert call(D=D) == fa.FA_ERR_UNSUPPORTED_D


def test_causal_rules():
    assert call(causal=1, Sq=128, Sk=256) == fa.FA_ERR_UNSUPPORTED_CAUSAL
    assert call(causal=2) == fa.FA_ERR_UNSUPPORTED_CAUSAL


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), 0.0, -0.5])
def test_bad_scale(scale):
    assert call(scale=scale) == fa.FA_ERR_BAD_SCALE


def test_alias():
    # o overlapping q (both 1*1*128*64*2 bytes = 16 KiB)
    assert call(o=A + 4096) == fa.FA_ERR_ALIAS
    assert call(lse=A4 + 16) == fa.FA_ERR_ALIAS


def test_selftest_argument_check():
    st = fa.lib().fa_selftest_fwd_timeout(A, A2, A3, A4, A5, 1, 1, 128, 128, 64, 0.125, 0,
                                          2_000_000_001, 0)
    assert st == fa.FA_ERR_BAD_SHAPE  # wait limit above 2 s
    st = fa.lib().fa_selftest_fwd_timeout(None, A2, A3, A4, A5, 1, 1, 128, 128, 64, 0.125, 0, 0, 0)
    assert st == fa.FA_ERR_NULLPTR
    assert fa.fa_selftest_bounded_wait(0, stream=0) == fa.FA_ERR_BAD_SHAPE
    assert fa.fa_selftest_bounded_wait(2_000_000, stream=0) == fa.FA_ERR_BAD_SHAPE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path only")
def test_valid_call_without_gpu_reports_cuda_error():
    assert call() == fa.FA_ERR_CUDA
    assert "CUDA error" in fa.fa_strerror(fa.FA_ERR_CUDA)


def test_torch_wrapper_rejects_cpu_tensors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, o=q.clone(), lse=torch.zeros(1, 1, 128), stream=0)


def wcall(wl, wr, Sq=128, Sk=128, **kw):
    return fa.fa_fwd_window_raw(A, A2, A3, A4, A5, 1, 1, Sq, Sk, 64, 0.125, wl, wr, 0)


def test_window_argument_checks():
    assert wcall(-2, 0) == fa.FA_ERR_BAD_WINDOW
    assert wcall(5, -3) == fa.FA_ERR_BAD_WINDOW
    assert wcall(16, 0, Sq=128, Sk=256) == fa.FA_ERR_BAD_WINDOW
    assert fa.fa_fwd_window_raw(0, A2, A3, A4, A5, 1, 1, 128, 128, 64, 0.125, 4, 0, 0) == \
        fa.FA_ERR_NULLPTR
    assert fa.fa_fwd_window_raw(A, A2, A3, A4, A5, 1, 1, 128, 128, 96, 0.125, 4, 0, 0) == \
        fa.FA_ERR_UNSUPPORTED_D


def mcall(mask=1 << 42, heads=1, B=1, H=1, Sq=300, Sk=300, wl=-1, wr=-1, o=A4, lse=A5, D=64, stride=1):
    return fa.fa_fwd_blockmask_raw(A, A2, A3, o, lse, B, H, Sq, Sk, D, 0.125, wl, wr, mask, heads, stride, 0)


def test_blockmask_argument_checks():
    assert mcall(mask=0) == fa.FA_ERR_NULLPTR
    assert mcall(heads=2, B=1, H=3) == fa.FA_ERR_BAD_MASK
    assert mcall(heads=0) == fa.FA_ERR_BAD_MASK
    assert mcall(stride=0) == fa.FA_ERR_BAD_MASK
    assert mcall(wl=-2) == fa.FA_ERR_BAD_WINDOW
    assert mcall(wl=16, wr=0, Sq=128, Sk=256) == fa.FA_ERR_BAD_WINDOW
    assert mcall(D=96) == fa.FA_ERR_UNSUPPORTED_D
    # the mask may not overlap O (bytes [A4, A4 + 300*64*2)) or LSE
    assert mcall(mask=A4 + 100) == fa.FA_ERR_ALIAS
    assert mcall(mask=A5 + 4) == fa.FA_ERR_ALIAS
    # one byte before O with a mask of 3 x 3 blocks overlaps it
    assert mcall(mask=A4 - 1) == fa.FA_ERR_ALIAS
    assert "mask" in fa.fa_strerror(fa.FA_ERR_BAD_MASK)


def test_blockmask_wrapper_rejects_bad_masks_before_the_call():
    q = torch.zeros(1, 1, 300, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # CPU tensors
        fa.fa_fwd_blockmask(q, q, q, torch.ones(1, 3, 3, dtype=torch.uint8), o=q.clone(),
                            lse=torch.zeros(1, 1, 300), stream=0)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path only")
def test_blockmask_valid_call_without_gpu_reports_cuda_error():
    assert mcall(heads=3, B=1, H=3) == fa.FA_ERR_CUDA
    assert mcall(stride=1 << 30) == fa.FA_ERR_CUDA
    assert mcall(mask=A4 - 9) == fa.FA_ERR_CUDA  # 9 bytes of mask end right before O


def test_splitkv_sizes_and_checks():
    n = fa.fa_splitkv_num_splits(8, 32, 1, 16384, 128)
    assert 1 <= n <= 256
    need = fa.fa_fwd_splitkv_workspace_bytes(8, 32, 1, 16384, 128, 4)
    assert need >= 8 * 32 * 4 * 1 * (128 + 1) * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 9, 100, 128, 0) == 0   # Sq > 8
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 1, 100, 96, 0) == 0    # D
    W = 1 << 42

    def scall(Sq=1, Sk=4096, D=128, splits=0, ws=W, ws_bytes=1 << 30):
        return fa.fa_fwd_splitkv_raw(A, A2, A3, A4, A5, 1, 1, Sq, Sk, D, 0.1, splits, ws,
                                     ws_bytes, 0)

    assert scall(Sq=9) == fa.FA_ERR_BAD_SHAPE
    assert scall(splits=300) == fa.FA_ERR_BAD_SHAPE
    assert scall(ws=0) == fa.FA_ERR_WORKSPACE
    assert scall(ws=W + 8) == fa.FA_ERR_WORKSPACE
    assert scall(ws_bytes=16) == fa.FA_ERR_WORKSPACE
    assert scall(ws=A + 64) == fa.FA_ERR_ALIAS


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """64 heads x 8 rows x 256 splits of fp32 partials need ~68 MB > 16 MiB; the
    call refuses before touching the GPU (pointers here are never used)."""
    big = [1 << 36, 1 << 38, 1 << 40, 1 << 42, 1 << 44]
    st = fa.lib().fa_fwd_splitkv_noalloc(*big, 1, 64, 8, 16384, 128, 0.1, 256, 0)
    assert st == fa.FA_ERR_SCRATCH_LIMIT
    assert "16 MiB" in fa.fa_strerror(st)
    assert fa.lib().fa_fwd_splitkv_noalloc(0, *big[1:], 1, 1, 1, 64, 128, 0.1, 0, 0) == \
        fa.FA_ERR_NULLPTR


def test_bwd_argument_checks():
    P = [1 << 20, 1 << 30, 1 << 32, 1 << 34, 1 << 36, 1 << 38, 1 << 40, 1 << 42, 1 << 44, 1 << 46]

    def bcall(ptrs=P, Sq=128, Sk=128, D=64, causal=0, scale=0.125):
        return fa.fa_bwd_raw(*ptrs, 1, 1, Sq, Sk, D, scale, causal, 0)

    assert bcall(ptrs=[0] + P[1:]) == fa.FA_ERR_NULLPTR
    assert bcall(ptrs=P[:9] + [P[9] + 4]) == fa.FA_ERR_MISALIGNED
    assert bcall(D=96) == fa.FA_ERR_UNSUPPORTED_D
    assert bcall(causal=1, Sq=128, Sk=256) == fa.FA_ERR_UNSUPPORTED_CAUSAL
    assert bcall(scale=float("nan")) == fa.FA_ERR_BAD_SCALE
    assert bcall(ptrs=P[:6] + [P[0] + 16] + P[7:]) == fa.FA_ERR_ALIAS   # dq over q
    assert bcall(ptrs=P[:7] + [P[6]] + P[8:]) == fa.FA_ERR_ALIAS        # dk == dq

    def kcall(q=A, timeout_ns=0, ws=A2 + (1 << 24), wsb=1 << 20):
        return fa.lib().fa_selftest_splitkv_timeout(q, A2, A3, A4, A5, 1, 1, 1, 128, 64, 0.125, 0, ws, wsb,
                                                    timeout_ns, 0)

    assert kcall(timeout_ns=2_000_000_001) == fa.FA_ERR_BAD_SHAPE   # wait limit above 2 s
    assert kcall(q=0) == fa.FA_ERR_NULLPTR                            # fa_fwd_splitkv's checks apply
    assert kcall(ws=0) == fa.FA_ERR_WORKSPACE

    def tcall(ptrs=P, timeout_ns=0, D=64):
        return fa.lib().fa_selftest_bwd_timeout(*ptrs, 1, 1, 128, 128, D, 0.125, 0, timeout_ns, 0)

    assert tcall(timeout_ns=2_000_000_001) == fa.FA_ERR_BAD_SHAPE   # wait limit above 2 s
    assert tcall(ptrs=[0] + P[1:]) == fa.FA_ERR_NULLPTR             # fa_bwd's checks apply
    assert tcall(D=96) == fa.FA_ERR_UNSUPPORTED_D


def test_fp8_argument_checks():
    def fcall(q=A, D=128, causal=0, Sq=128, Sk=128, scale=0.1, ds=(0.01, 0.01, 0.01), lse=A5,
              o=A4):
        return fa.fa_fwd_fp8_raw(q, A2, A3, o, lse, 1, 1, Sq, Sk, D, scale, causal, *ds, 0)

    assert fcall(q=0) == fa.FA_ERR_NULLPTR
    assert fcall(lse=A5 + 4) == fa.FA_ERR_MISALIGNED
    assert fcall(D=64) == fa.FA_ERR_UNSUPPORTED_D
    assert fcall(causal=1, Sk=256) == fa.FA_ERR_UNSUPPORTED_CAUSAL
    assert fcall(ds=(0.01, 0.0, 0.01)) == fa.FA_ERR_BAD_SCALE
    assert fcall(ds=(0.01, 0.01, float("inf"))) == fa.FA_ERR_BAD_SCALE
    assert fcall(ds=(1e-30, 1e-30, 1.0)) == fa.FA_ERR_BAD_SCALE   # product underflows
    assert fcall(o=A + 8192) == fa.FA_ERR_ALIAS   # O (32 KiB bf16) over 16 KiB of q codes
    assert fcall(Sq=0) == fa.FA_ERR_BAD_SHAPE
