"""GB300-native (sm_103a) FlashAttention-2-style attention forward.

The compute lives in ``_build/libfa_gb300.so`` (hand-written CUDA: TMA,
tcgen05 MMAs into tensor memory, online softmax).  This module is a thin
ctypes binding with the C ABI's names (``include/fa.h``): it only marshals
arguments.  torch is used for device memory and streams.  There is no CPU
or library fallback: if the shared library cannot be built or loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

__all__ = ["fa_fwd", "fa_fwd_raw", "fa_fwd_window", "fa_fwd_window_raw", "fa_strerror", "fa_device_status",
           "fa_selftest_bounded_wait", "fa_selftest_fwd_timeout", "fa_selftest_bwd_timeout", "fa_selftest_splitkv_timeout", "fa_version", "FAError", "lib", "library_path",
           "FA_OK", "FA_ERR_NULLPTR", "FA_ERR_BAD_SHAPE", "FA_ERR_UNSUPPORTED_D",
           "FA_ERR_UNSUPPORTED_CAUSAL", "FA_ERR_MISALIGNED", "FA_ERR_BAD_SCALE", "FA_ERR_CUDA",
           "FA_ERR_TIMEOUT", "FA_ERR_ALIAS", "FA_ERR_BAD_WINDOW", "FA_ERR_WORKSPACE",
           "fa_fwd_splitkv", "fa_fwd_splitkv_raw", "fa_fwd_splitkv_workspace_bytes",
           "fa_splitkv_num_splits", "FA_ERR_SCRATCH_LIMIT",
           "fa_bwd", "fa_bwd_raw", "fa_fwd_fp8", "fa_fwd_fp8_raw",
           "fa_fwd_blockmask", "fa_fwd_blockmask_raw", "FA_ERR_BAD_MASK", "FA_BLOCK_M", "FA_BLOCK_N"]

FA_OK = 0
FA_ERR_NULLPTR = -1
FA_ERR_BAD_SHAPE = -2
FA_ERR_UNSUPPORTED_D = -3
FA_ERR_UNSUPPORTED_CAUSAL = -4
FA_ERR_MISALIGNED = -5
FA_ERR_BAD_SCALE = -6
FA_ERR_CUDA = -7
FA_ERR_TIMEOUT = -8
FA_ERR_ALIAS = -9
FA_ERR_BAD_WINDOW = -10
FA_ERR_WORKSPACE = -11
FA_ERR_SCRATCH_LIMIT = -12
FA_ERR_BAD_MASK = -13
FA_BLOCK_M = 128  # query rows per block-mask row
FA_BLOCK_N = 128  # keys per block-mask column

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int

# name -> (restype, argtypes), mirroring include/fa.h
_SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _vp]),
    "fa_fwd_window": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i,
                           _vp]),
    "fa_fwd_blockmask": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i,
                              _vp, _i, _i, _vp]),
    "fa_fwd_splitkv": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _vp,
                            ctypes.c_size_t, _vp]),
    "fa_fwd_splitkv_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i]),
    "fa_fwd_splitkv_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float,
                                    _i, _vp]),
    "fa_splitkv_num_splits": (_i, [_i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp] * 10 + [_i, _i, _i, _i, _i, ctypes.c_float, _i, _vp]),
    "fa_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i,
                        ctypes.c_float, ctypes.c_float, ctypes.c_float, _vp]),
    "fa_strerror": (ctypes.c_char_p, [_i]),
    "fa_device_status": (_i, [_vp]),
    "fa_selftest_bounded_wait": (_i, [_i, _vp]),
    "fa_selftest_fwd_timeout": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float,
                                     _i, ctypes.c_ulonglong, _vp]),
    "fa_selftest_bwd_timeout": (_i, [_vp] * 10 + [_i, _i, _i, _i, _i, ctypes.c_float, _i, ctypes.c_ulonglong,
                                                  _vp]),
    "fa_selftest_splitkv_timeout": (_i, [_vp] * 5 + [_i] * 5 + [ctypes.c_float, _i, _vp, ctypes.c_size_t,
                                                               ctypes.c_ulonglong, _vp]),
    "fa_version": (_i, []),
}


class FAError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = fa_strerror(status)
        super().__init__(f"{where}: {msg} (status {status})" if where else msg)


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded shared library (built in-tree with nvcc on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            handle = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def fa_strerror(status: int) -> str:
    return lib().fa_strerror(int(status)).decode()


def fa_version() -> int:
    return lib().fa_version()


def _stream_ptr(stream) -> int:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
               Sq: int, Sk: int, D: int, scale: float, causal: int, stream_ptr: int) -> int:
    """The C call with raw device pointers; returns the status code."""
    return lib().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, D, float(scale),
                        int(causal), stream_ptr)


def fa_fwd_window_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                      H: int, Sq: int, Sk: int, D: int, scale: float, window_left: int,
                      window_right: int, stream_ptr: int) -> int:
    """The windowed C call with raw device pointers; returns the status code."""
    return lib().fa_fwd_window(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, D, float(scale),
                               int(window_left), int(window_right), stream_ptr)


def fa_fwd_blockmask_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                         H: int, Sq: int, Sk: int, D: int, scale: float, window_left: int,
                         window_right: int, mask_ptr: int, mask_heads: int, pair_stride: int,
                         stream_ptr: int) -> int:
    """The block-mask C call with raw device pointers; returns the status code."""
    return lib().fa_fwd_blockmask(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, D, float(scale),
                                  int(window_left), int(window_right), mask_ptr, int(mask_heads),
                                  int(pair_stride), stream_ptr)


def _prepare(q, k, v, o, lse):
    import torch

    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if o is None:
        o = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D):
        raise ValueError("k and v must be [B, H, Sk, D] matching q")
    if tuple(o.shape) != (B, H, Sq, D) or tuple(lse.shape) != (B, H, Sq):
        raise ValueError("o must be [B, H, Sq, D] and lse [B, H, Sq]")
    return o, lse, B, H, Sq, Sk, D


def fa_fwd(q, k, v, o=None, lse=None, scale: float | None = None, causal: bool = False,
           stream=None):
    """Attention forward on torch CUDA tensors.

    q: bf16 [B,H,Sq,D]; k, v: bf16 [B,H,Sk,D] (contiguous, same device).
    o (bf16 [B,H,Sq,D]) and lse (fp32 [B,H,Sq]) are allocated if not given.
    scale defaults to 1/sqrt(D).  Launches on ``stream`` (default: torch's
    current stream) and returns (o, lse) without synchronising.
    """
    o, lse, B, H, Sq, Sk, D = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = D ** -0.5
    st = fa_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    B, H, Sq, Sk, D, scale, int(bool(causal)), _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd")
    return o, lse


def fa_fwd_window(q, k, v, window_left: int, window_right: int, o=None, lse=None,
                  scale: float | None = None, stream=None):
    """Banded attention: key j allowed for query i iff i-window_left <= j <= i+window_right
    (-1 = unbounded on that side).  Same tensors and return value as fa_fwd."""
    o, lse, B, H, Sq, Sk, D = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = D ** -0.5
    st = fa_fwd_window_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, Sq, Sk, D, scale, window_left, window_right,
                           _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_window")
    return o, lse


def fa_fwd_blockmask(q, k, v, block_mask, window_left: int = -1, window_right: int = -1, o=None,
                     lse=None, scale: float | None = None, pair_stride: int = 1, stream=None):
    """Attention over the key blocks ``block_mask`` keeps (uint8 or bool CUDA tensor
    ``[mask_heads, ceil(Sq/128), ceil(Sk/128)]``, ``mask_heads`` 1 or B*H; nonzero
    keeps a 128-row x 128-key block), within the band of fa_fwd_window.  Rows with
    no allowed key get O = 0, LSE = -inf.  ``pair_stride``: query blocks a and
    a + pair_stride are computed together (a hint; the stride of a dilated
    pattern suits it).  Same tensors and return value as fa_fwd."""
    import torch

    o, lse, B, H, Sq, Sk, D = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = D ** -0.5
    n_qb, n_kb = -(-Sq // FA_BLOCK_M), -(-Sk // FA_BLOCK_N)
    if (block_mask.dtype not in (torch.uint8, torch.bool) or not block_mask.is_cuda
            or not block_mask.is_contiguous() or block_mask.dim() != 3
            or tuple(block_mask.shape[1:]) != (n_qb, n_kb)):
        raise ValueError(f"block_mask must be a contiguous CUDA uint8/bool tensor [mask_heads, {n_qb}, {n_kb}]")
    st = fa_fwd_blockmask_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              B, H, Sq, Sk, D, scale, window_left, window_right,
                              block_mask.data_ptr(), block_mask.shape[0], pair_stride, _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_blockmask")
    return o, lse


def fa_fwd_splitkv_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                       H: int, Sq: int, Sk: int, D: int, scale: float, num_splits: int,
                       ws_ptr: int, ws_bytes: int, stream_ptr: int) -> int:
    """The split-KV C call with raw device pointers; returns the status code."""
    return lib().fa_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, D, float(scale),
                                int(num_splits), ws_ptr, int(ws_bytes), stream_ptr)


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, Sq: int, Sk: int, D: int,
                                   num_splits: int = 0) -> int:
    return lib().fa_fwd_splitkv_workspace_bytes(B, H, Sq, Sk, D, num_splits)


def fa_splitkv_num_splits(B: int, H: int, Sq: int, Sk: int, D: int) -> int:
    return lib().fa_splitkv_num_splits(B, H, Sq, Sk, D)


def fa_fwd_splitkv(q, k, v, o=None, lse=None, scale: float | None = None, num_splits: int = 0,
                   workspace=None, stream=None):
    """Decode attention (1..8 query rows per head, every key visible) with the keys
    of each head split across CTAs.  ``workspace`` is a CUDA uint8 tensor of at
    least fa_fwd_splitkv_workspace_bytes(...) bytes (allocated here if None)."""
    import torch

    o, lse, B, H, Sq, Sk, D = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = D ** -0.5
    need = fa_fwd_splitkv_workspace_bytes(B, H, Sq, Sk, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = fa_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, Sq, Sk, D, scale, num_splits,
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv")
    return o, lse


def fa_fwd_fp8_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
                   Sq: int, Sk: int, D: int, scale: float, causal: int, descale_q: float,
                   descale_k: float, descale_v: float, stream_ptr: int) -> int:
    """The 8-bit C call with raw device pointers; returns the status code."""
    return lib().fa_fwd_fp8(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, D, float(scale),
                            int(causal), float(descale_q), float(descale_k), float(descale_v),
                            stream_ptr)


def fa_fwd_fp8(q, k, v, descale_q: float, descale_k: float, descale_v: float, o=None, lse=None,
               scale: float | None = None, causal: bool = False, stream=None):
    """Attention forward on e4m3 inputs with per-tensor scales (real value = code * descale).

    q: [B,H,Sq,128], k, v: [B,H,Sk,128], each a contiguous CUDA tensor of dtype uint8
    (the codes) or torch.float8_e4m3fn.  o (bf16 [B,H,Sq,128]) and lse (fp32 [B,H,Sq])
    are allocated if not given.  Returns (o, lse) without synchronising."""
    import torch

    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_cuda or \
                not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA uint8 / float8_e4m3fn tensor")
    if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D):
        raise ValueError("k and v must be [B, H, Sk, D] matching q")
    if o is None:
        o = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if o.dtype != torch.bfloat16 or tuple(o.shape) != (B, H, Sq, D) or not o.is_contiguous() \
            or lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq) or \
            not lse.is_contiguous() or not o.is_cuda or not lse.is_cuda:
        raise ValueError("o must be contiguous CUDA bf16 [B,H,Sq,D] and lse fp32 [B,H,Sq]")
    if scale is None:
        scale = D ** -0.5
    st = fa_fwd_fp8_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, H, Sq, Sk, D, scale, int(bool(causal)), descale_q, descale_k,
                        descale_v, _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return o, lse


def fa_bwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, do_ptr, dq_ptr, dk_ptr, dv_ptr, delta_ptr,
               B, H, Sq, Sk, D, scale, causal, stream_ptr) -> int:
    """The backward C call with raw device pointers; returns the status code."""
    return lib().fa_bwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, do_ptr, dq_ptr, dk_ptr, dv_ptr,
                        delta_ptr, B, H, Sq, Sk, D, float(scale), int(causal), stream_ptr)


def fa_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, delta=None,
           scale: float | None = None, causal: bool = False, stream=None):
    """Gradients (dq, dk, dv) of fa_fwd for output gradient ``dout`` (torch CUDA tensors;
    o and lse are fa_fwd's outputs).  Outputs and the fp32 ``delta`` scratch [B,H,Sq] are
    allocated if not given.  Returns (dq, dk, dv) without synchronising."""
    import torch

    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if delta is None:
        delta = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    for name, t in (("lse", lse), ("delta", delta)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor")
    if scale is None:
        scale = D ** -0.5
    st = fa_bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                    delta.data_ptr(), B, H, Sq, Sk, D, scale, int(bool(causal)),
                    _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv


def fa_device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the kernels' status word."""
    return lib().fa_device_status(_stream_ptr(stream))


def fa_selftest_bounded_wait(timeout_us: int, stream=None) -> int:
    return lib().fa_selftest_bounded_wait(int(timeout_us), _stream_ptr(stream))


def fa_selftest_fwd_timeout(q, k, v, o, lse, scale, causal, timeout_ns: int, stream=None) -> int:
    """fa_fwd with every on-chip wait bounded by `timeout_ns` (tests of the give-up
    path); returns the launch status.  q, k, v, o, lse: contiguous CUDA tensors."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    return lib().fa_selftest_fwd_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, H, Sq, Sk, D, float(scale),
                                         int(bool(causal)), int(timeout_ns), _stream_ptr(stream))


def fa_selftest_bwd_timeout(q, k, v, o, lse, dout, dq, dk, dv, delta, scale, causal, timeout_ns: int,
                            stream=None) -> int:
    """fa_bwd with every on-chip wait of both kernels bounded by `timeout_ns`
    (tests of the give-up path); returns the launch status.  All arguments are
    contiguous CUDA tensors as for fa_bwd."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    return lib().fa_selftest_bwd_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                         dv.data_ptr(), delta.data_ptr(), B, H, Sq, Sk, D, float(scale),
                                         int(bool(causal)), int(timeout_ns), _stream_ptr(stream))


def fa_selftest_splitkv_timeout(q, k, v, o, lse, workspace, scale, timeout_ns: int, num_splits: int = 0,
                                stream=None) -> int:
    """fa_fwd_splitkv with every on-chip wait of the partial kernel bounded by
    `timeout_ns` (tests of the give-up path); returns the launch status.  All
    arguments are contiguous CUDA tensors as for fa_fwd_splitkv; ``workspace`` is a
    byte tensor of at least fa_fwd_splitkv_workspace_bytes."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    return lib().fa_selftest_splitkv_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                             lse.data_ptr(), B, H, Sq, Sk, D, float(scale), int(num_splits),
                                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                             int(timeout_ns), _stream_ptr(stream))
