"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product library never
imports, links or calls it, and this package imports nothing from the
product: the two share only the seeded input generator, which holds none of
the method's arithmetic.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64).  This module
compiles it with gcc on first use (or from ``build()``) and marshals numpy
arrays through ctypes.

Inputs are either float64 arrays (any values) or uint16 arrays holding raw
bf16 bit patterns, which the C code widens exactly to fp64.  Layout
``[B, H, S, D]`` contiguous; outputs are float64 ``O [B, H, Sq, D]`` and
``LSE [B, H, Sq]``.  ``window=(wl, wr)`` keeps keys ``i-wl <= j <= i+wr``;
a negative bound means unbounded on that side.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_attn.so")

_lock = threading.Lock()
_lib = None

ORC_OK = 0
ORC_ERR_ARG = -1
ORC_ERR_NOMEM = -2
ORC_ERR_EMPTY_ROW = -3


class OracleError(RuntimeError):
    pass


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, portable flags)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.c_void_p
    L = ctypes.c_long
    common = [L, L, L, L, L, ctypes.c_double, ctypes.c_int, L, L]
    lib.oracle_attn_fwd_f64.argtypes = [dp] * 5 + common + [ctypes.c_int]
    lib.oracle_attn_fwd_bf16.argtypes = [dp] * 5 + common + [ctypes.c_int]
    lib.oracle_attn_fwd_rows_bf16.argtypes = [dp] * 5 + [L, dp, dp] + common + [ctypes.c_int]
    lib.oracle_attn_fwd_tiled_f64.argtypes = [dp] * 5 + common + [L, L]
    lib.oracle_attn_bwd_f64.argtypes = [dp] * 7 + common + [ctypes.c_int]
    lib.oracle_attn_bwd_bf16.argtypes = [dp] * 7 + common + [ctypes.c_int]
    for f in (lib.oracle_attn_fwd_f64, lib.oracle_attn_fwd_bf16,
              lib.oracle_attn_fwd_rows_bf16, lib.oracle_attn_fwd_tiled_f64,
              lib.oracle_attn_bwd_f64, lib.oracle_attn_bwd_bf16):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Return the bound library, building it first if needed."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _prep(q, k, v):
    q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (np.float64, np.uint16):
        raise TypeError("q, k, v must all be float64, or all uint16 bf16 bit patterns")
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("expected [B, H, S, D] arrays")
    B, H, Sq, D = q.shape
    if k.shape[:2] != (B, H) or v.shape != k.shape or k.shape[3] != D:
        raise ValueError(f"shape mismatch: q{q.shape} k{k.shape} v{v.shape}")
    return q, k, v, B, H, Sq, k.shape[2], D


def _check(st: int):
    if st != ORC_OK:
        raise OracleError({ORC_ERR_ARG: "bad argument", ORC_ERR_NOMEM: "out of memory",
                           ORC_ERR_EMPTY_ROW: "a query row has no allowed key"}.get(st, str(st)))


def attn_fwd(q, k, v, scale: float, causal: bool = False, window=(-1, -1),
             nthreads: int | None = None, lib=None):
    """Materialised fp64 attention.  Returns (O float64 [B,H,Sq,D], LSE float64 [B,H,Sq])."""
    lib = lib or load()
    q, k, v, B, H, Sq, Sk, D = _prep(q, k, v)
    o = np.empty((B, H, Sq, D), np.float64)
    lse = np.empty((B, H, Sq), np.float64)
    fn = lib.oracle_attn_fwd_bf16 if q.dtype == np.uint16 else lib.oracle_attn_fwd_f64
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, D, float(scale),
            int(bool(causal)), int(window[0]), int(window[1]), nthreads or default_threads())
    _check(st)
    return o, lse


def attn_fwd_rows(q, k, v, bh, rows, scale: float, causal: bool = False, window=(-1, -1),
                  nthreads: int | None = None, lib=None):
    """Oracle outputs for selected (head, row) pairs only.

    ``q, k, v`` are uint16 bf16 bit arrays ``[B,H,S,D]``; ``bh`` (= b*H+h) and
    ``rows`` are int arrays of equal length.  Returns (O [n, D], LSE [n]) in
    the order given.
    """
    lib = lib or load()
    q, k, v, B, H, Sq, Sk, D = _prep(q, k, v)
    if q.dtype != np.uint16:
        raise TypeError("attn_fwd_rows takes bf16 bit patterns (uint16)")
    bh = np.asarray(bh, np.int64)
    rows = np.asarray(rows, np.int64)
    order = np.argsort(bh, kind="stable")
    sbh = np.ascontiguousarray(bh[order]).astype(np.int64)
    srow = np.ascontiguousarray(rows[order]).astype(np.int64)
    n = len(sbh)
    o = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    st = lib.oracle_attn_fwd_rows_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(sbh), _ptr(srow), n,
                                       _ptr(o), _ptr(lse), B, H, Sq, Sk, D, float(scale),
                                       int(bool(causal)), int(window[0]), int(window[1]),
                                       nthreads or default_threads())
    _check(st)
    out_o = np.empty_like(o)
    out_l = np.empty_like(lse)
    out_o[order] = o
    out_l[order] = lse
    return out_o, out_l


def attn_fwd_tiled(q, k, v, scale: float, causal: bool = False, window=(-1, -1),
                   block_m: int = 128, block_n: int = 128, lib=None):
    """The tiled online-softmax loop in fp64 (float64 inputs only)."""
    lib = lib or load()
    q, k, v, B, H, Sq, Sk, D = _prep(q, k, v)
    if q.dtype != np.float64:
        raise TypeError("attn_fwd_tiled takes float64 arrays")
    o = np.empty((B, H, Sq, D), np.float64)
    lse = np.empty((B, H, Sq), np.float64)
    st = lib.oracle_attn_fwd_tiled_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                       B, H, Sq, Sk, D, float(scale), int(bool(causal)),
                                       int(window[0]), int(window[1]), int(block_m),
                                       int(block_n))
    _check(st)
    return o, lse


def attn_fwd_blockmask(q, k, v, scale: float, block_mask, window=(-1, -1), block=(128, 128)):
    """Attention over the keys that a block mask keeps, in fp64 (numpy).

    "FlashAttention-2 -- L3 Cross-Paper Synthesis", section 5 item 4: the causal
    block skip generalises to sliding windows and dilated patterns, one
    sparse-block-skip mechanism.  The pages define no pattern beyond the window,
    so the mechanism is taken as given by the caller: ``block_mask[h, a, c]``
    nonzero keeps key block ``c`` (keys ``c*bn .. c*bn+bn-1``) for query block
    ``a`` (rows ``a*bm .. a*bm+bm-1``) of head ``h``.  Key ``j`` is allowed for
    query ``i`` iff ``j < Sk``, the window keeps it (``i-wl <= j <= i+wr``, a
    negative bound unbounded; causal is ``(-1, 0)``) and its block is kept.

    ``q, k, v``: ``[B,H,S,D]`` float64, or uint16 bf16 bit patterns (widened
    exactly).  ``block_mask``: ``[Hm, ceil(Sq/bm), ceil(Sk/bn)]`` with ``Hm``
    1 (one pattern for every head) or ``B*H`` (head ``b*H+h``).

    The definition written out: S = scale Q K^T, S = -inf where not allowed,
    P = softmax over the row, O = P V, LSE = ln sum exp S.  A row with no
    allowed key gets O = 0 and LSE = -inf (a reading: with every key masked the
    row takes no value from V, and its log-sum-exp is that of an empty sum).
    Returns (O float64 [B,H,Sq,D], LSE float64 [B,H,Sq]).
    """
    q, k, v, B, H, Sq, Sk, D = _prep(q, k, v)
    if q.dtype == np.uint16:
        q, k, v = (bf16_bits_to_f64(x) for x in (q, k, v))
    bm, bn = int(block[0]), int(block[1])
    mask = np.asarray(block_mask)
    n_qb, n_kb = -(-Sq // bm), -(-Sk // bn)
    if mask.ndim != 3 or mask.shape[1:] != (n_qb, n_kb) or mask.shape[0] not in (1, B * H):
        raise ValueError(f"block_mask must be [1 or B*H, {n_qb}, {n_kb}], got {mask.shape}")
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    band = np.ones((Sq, Sk), bool)
    if window[0] >= 0:
        band &= j >= i - window[0]
    if window[1] >= 0:
        band &= j <= i + window[1]
    o = np.zeros((B, H, Sq, D), np.float64)
    lse = np.full((B, H, Sq), -np.inf)
    for bh in range(B * H):
        b, h = divmod(bh, H)
        kept = mask[0 if mask.shape[0] == 1 else bh] != 0
        allowed = band & kept[np.arange(Sq) // bm][:, np.arange(Sk) // bn]
        s = np.where(allowed, float(scale) * (q[b, h] @ k[b, h].T), -np.inf)
        m = s.max(axis=1)
        live = m > -np.inf
        p = np.exp(s[live] - m[live, None])
        l = p.sum(axis=1)
        o[b, h, live] = (p @ v[b, h]) / l[:, None]
        lse[b, h, live] = m[live] + np.log(l)
    return o, lse


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of uint16 bf16 bit patterns to float64 (for tests)."""
    u32 = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of each e4m3 code (uint8), written from the format's definition
    in the OCP 8-bit floating point specification: bit 7 sign, bits 6..3 a biased
    exponent E (bias 7), bits 2..0 a mantissa M.  E = 0 is subnormal,
    M/8 * 2^-6; otherwise (1 + M/8) * 2^(E-7).  There are no infinities; the two
    codes with E = 15 and M = 7 (0x7F, 0xFF) are NaN, so 448 is the largest
    finite magnitude."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    val = np.where((c & 0x80) != 0, -mag, mag)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def attn_fwd_fp8(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float,
                 scale: float, causal: bool = False, nthreads: int | None = None, lib=None):
    """fp64 attention of the dequantised 8-bit inputs: Q = e4m3(q8) * descale_q and
    likewise K and V (per-tensor scaling), then the materialised forward.  The
    descales are taken as float32 values, as the kernel receives them.  Returns
    (O float64 [B,H,Sq,D], LSE float64 [B,H,Sq])."""
    deq = [e4m3_to_f64(x) * float(np.float32(d))
           for x, d in ((q8, descale_q), (k8, descale_k), (v8, descale_v))]
    return attn_fwd(*deq, scale, causal, nthreads=nthreads, lib=lib)


def attn_bwd(q, k, v, dout, scale: float, causal: bool = False, window=(-1, -1),
             nthreads: int | None = None, lib=None):
    """Gradients (dQ, dK, dV) of the attention forward for output gradient ``dout``
    ([B,H,Sq,D], same dtype as q: float64 or uint16 bf16 bits), in float64."""
    lib = lib or load()
    q, k, v, B, H, Sq, Sk, D = _prep(q, k, v)
    dout = np.ascontiguousarray(dout)
    if dout.dtype != q.dtype or dout.shape != q.shape:
        raise ValueError("dout must match q in dtype and shape")
    dq = np.empty((B, H, Sq, D), np.float64)
    dk = np.empty((B, H, Sk, D), np.float64)
    dv = np.empty((B, H, Sk, D), np.float64)
    fn = lib.oracle_attn_bwd_bf16 if q.dtype == np.uint16 else lib.oracle_attn_bwd_f64
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Sq, Sk, D,
            float(scale), int(bool(causal)), int(window[0]), int(window[1]),
            nthreads or default_threads())
    _check(st)
    return dq, dk, dv
