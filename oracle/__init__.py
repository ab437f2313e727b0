"""ORACLE for the sparse MoE layer forward -- test infrastructure only.

Thin ctypes binding of ``moe_oracle.c`` (plain single-threaded C, fp64
accumulation, its own e4m3 table).  Only the tests, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` may import this package; the CUDA
library never does.  Each C function names the passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile liboracle.so: IEEE fp32/fp64, no fused multiply-add, no fast-math."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                               "-o", _LIB, _SRC, "-lm"])
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i32, vp, f32, f64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_double
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = f64
        L.oracle_e4m3_encode.argtypes = [f32]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode_scan.argtypes = [f32]
        L.oracle_e4m3_encode_scan.restype = ctypes.c_uint8
        L.oracle_bf16_from_f32.argtypes = [f32]
        L.oracle_bf16_from_f32.restype = ctypes.c_uint16
        L.oracle_bf16_from_f64.argtypes = [f64]
        L.oracle_bf16_from_f64.restype = ctypes.c_uint16
        L.oracle_quant_rows_bf16.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_quant_rows_f32.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_pack_w13.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_pack_w2.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_router.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.oracle_forward.argtypes = [vp] * 9 + [i32] * 5 + [vp, i32, vp, vp, vp, vp, vp]
        L.oracle_mx_quant_rows_f32.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_mx_quant_rows_bf16.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_mx_pack_w13.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_mx_pack_w2.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_mx_forward.argtypes = [vp] * 9 + [i32] * 5 + [vp, i32, vp, vp, vp, vp, vp]
        L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_decode.restype = f64
        L.oracle_e2m1_encode.argtypes = [f32]
        L.oracle_e2m1_encode.restype = ctypes.c_uint8
        L.oracle_mx4_quant_rows_f32.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_mx4_pack_w13.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_mx4_pack_w2.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_mx4_forward.argtypes = [vp] * 9 + [i32] * 5 + [vp, i32, vp, vp, vp, vp, vp]
        for f in ("oracle_quant_rows_bf16", "oracle_quant_rows_f32", "oracle_pack_w13", "oracle_pack_w2",
                  "oracle_router", "oracle_permute", "oracle_forward", "oracle_mx_quant_rows_f32",
                  "oracle_mx_quant_rows_bf16", "oracle_mx_pack_w13", "oracle_mx_pack_w2", "oracle_mx_forward",
                  "oracle_mx4_quant_rows_f32", "oracle_mx4_pack_w13", "oracle_mx4_pack_w2", "oracle_mx4_forward"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous, "oracle arrays must be C-contiguous numpy"
    return a.ctypes.data


def _pad128(n: int) -> int:
    return (n + 127) // 128 * 128


# ---- e4m3 / bf16 scalars (vectorised loops for tests) ----
def e4m3_decode_table() -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: np.ndarray, scan: bool = False) -> np.ndarray:
    L = lib()
    f = L.oracle_e4m3_encode_scan if scan else L.oracle_e4m3_encode
    flat = np.asarray(v, dtype=np.float32).ravel()
    return np.array([f(float(x)) for x in flat], dtype=np.uint8).reshape(np.shape(v))


def bf16_from_f64(v: np.ndarray) -> np.ndarray:
    L = lib()
    flat = np.asarray(v, dtype=np.float64).ravel()
    return np.array([L.oracle_bf16_from_f64(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(v))


# ---- quantisers ----
def quant_rows_bf16(x: np.ndarray):
    """x [rows, cols] bf16 bits -> (codes [rows, cols_p] u8, scales [rows, cols_p/128] f32)."""
    rows, cols = x.shape
    cp = _pad128(cols)
    q = np.empty((rows, cp), np.uint8)
    s = np.empty((rows, cp // 128), np.float32)
    lib().oracle_quant_rows_bf16(_p(np.ascontiguousarray(x, np.uint16)), rows, cols, _p(q), _p(s))
    return q, s


def quant_rows_f32(x: np.ndarray):
    rows, cols = x.shape
    cp = _pad128(cols)
    q = np.empty((rows, cp), np.uint8)
    s = np.empty((rows, cp // 128), np.float32)
    lib().oracle_quant_rows_f32(_p(np.ascontiguousarray(x, np.float32)), rows, cols, _p(q), _p(s))
    return q, s


def pack_w13(w13: np.ndarray, q: np.ndarray | None = None, s: np.ndarray | None = None):
    """fp32 [n, 2I, H] -> codes [n, 2Ip, Hp], scales [n, 2Ip/128, Hp/128]."""
    n, twoI, H = w13.shape
    I = twoI // 2
    Hp, Ip = _pad128(H), _pad128(I)
    q = np.empty((n, 2 * Ip, Hp), np.uint8) if q is None else q
    s = np.empty((n, 2 * Ip // 128, Hp // 128), np.float32) if s is None else s
    lib().oracle_pack_w13(_p(np.ascontiguousarray(w13, np.float32)), H, I, n, _p(q), _p(s))
    return q, s


def pack_w2(w2: np.ndarray, q: np.ndarray | None = None, s: np.ndarray | None = None):
    """fp32 [n, H, I] -> codes [n, Hp, Ip], scales [n, Hp/128, Ip/128]."""
    n, H, I = w2.shape
    Hp, Ip = _pad128(H), _pad128(I)
    q = np.empty((n, Hp, Ip), np.uint8) if q is None else q
    s = np.empty((n, Hp // 128, Ip // 128), np.float32) if s is None else s
    lib().oracle_pack_w2(_p(np.ascontiguousarray(w2, np.float32)), H, I, n, _p(q), _p(s))
    return q, s


# ---- router / permutation ----
def router(x, rw, rb, k: int, want_logits: bool = False):
    """-> dict(idx [T,k] i32, w_f32 [T,k], w_bf16 [T,k] u16, margin [T] f64, logits [T,E] f64 optional)."""
    T, H = x.shape
    E = rw.shape[0]
    idx = np.empty((T, k), np.int32)
    wf = np.empty((T, k), np.float32)
    wb = np.empty((T, k), np.uint16)
    margin = np.empty(T, np.float64)
    logits = np.empty((T, E), np.float64) if want_logits else None
    lib().oracle_router(_p(np.ascontiguousarray(x, np.uint16)), _p(np.ascontiguousarray(rw, np.uint16)),
                        _p(np.ascontiguousarray(rb, np.uint16)), T, H, E, k, _p(idx), _p(wf), _p(wb), _p(logits),
                        _p(margin))
    out = dict(idx=idx, w_f32=wf, w_bf16=wb, margin=margin)
    if want_logits:
        out["logits"] = logits
    return out


def permute(idx: np.ndarray, E: int):
    """-> dict(count [E], offset [E+1], perm [T*k], inv [T*k]) (int32)."""
    T, k = idx.shape
    count = np.empty(E, np.int32)
    offset = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    lib().oracle_permute(_p(np.ascontiguousarray(idx, np.int32)), T, E, k, _p(count), _p(offset), _p(perm), _p(inv))
    return dict(count=count, offset=offset, perm=perm, inv=inv)


# ---- full layer ----
def forward(x, rw, rb, w13, s13, b13, w2, s2, b2, k: int, tokens=None, want_intermediates: bool = False):
    """Layer output rows (bf16 bits) for `tokens` (all when None).

    Weights are the packed FP8 codes/scales (full [E, ...] arrays; only the
    experts the listed tokens select are read)."""
    T, H = x.shape
    E = rw.shape[0]
    I = b13.shape[1] // 2
    Ip = _pad128(I)
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tok is None else len(tok)
    out = np.empty((n, H), np.uint16)
    hq = np.empty((n * k, Ip), np.uint8) if want_intermediates else None
    sh = np.empty((n * k, Ip // 128), np.float32) if want_intermediates else None
    y = np.empty((n * k, H), np.float64) if want_intermediates else None
    ids = np.empty(n * k, np.int32) if want_intermediates else None
    lib().oracle_forward(_p(np.ascontiguousarray(x, np.uint16)), _p(np.ascontiguousarray(rw, np.uint16)),
                         _p(np.ascontiguousarray(rb, np.uint16)), _p(w13), _p(s13),
                         _p(np.ascontiguousarray(b13, np.uint16)), _p(w2), _p(s2),
                         _p(np.ascontiguousarray(b2, np.uint16)), T, H, I, E, k, _p(tok), n, _p(out), _p(hq), _p(sh),
                         _p(y), _p(ids))
    if want_intermediates:
        return out, dict(hq=hq, sh=sh, y=y, idx=ids)
    return out


# ---- MXFP8 variant (1x32 UE8M0 scales) ----
def mx_quant_rows_f32(x: np.ndarray):
    """fp32 [rows, cols] -> codes [rows, Cp], scale bytes [rows, Cp/32] (Cp = cols padded to 128)."""
    rows, cols = x.shape
    cp = _pad128(cols)
    q = np.empty((rows, cp), np.uint8)
    s = np.empty((rows, cp // 32), np.uint8)
    lib().oracle_mx_quant_rows_f32(_p(np.ascontiguousarray(x, np.float32)), rows, cols, _p(q), _p(s))
    return q, s


def mx_quant_rows_bf16(x: np.ndarray):
    rows, cols = x.shape
    cp = _pad128(cols)
    q = np.empty((rows, cp), np.uint8)
    s = np.empty((rows, cp // 32), np.uint8)
    lib().oracle_mx_quant_rows_bf16(_p(np.ascontiguousarray(x, np.uint16)), rows, cols, _p(q), _p(s))
    return q, s


def mx_pack_w13(w13: np.ndarray, q: np.ndarray | None = None, s: np.ndarray | None = None):
    """fp32 [n, 2I, H] -> codes [n, 2Ip, Hp], scale bytes [n, 2Ip, Hp/32]."""
    n, twoI, H = w13.shape
    I = twoI // 2
    Hp, Ip = _pad128(H), _pad128(I)
    q = np.empty((n, 2 * Ip, Hp), np.uint8) if q is None else q
    s = np.empty((n, 2 * Ip, Hp // 32), np.uint8) if s is None else s
    lib().oracle_mx_pack_w13(_p(np.ascontiguousarray(w13, np.float32)), H, I, n, _p(q), _p(s))
    return q, s


def mx_pack_w2(w2: np.ndarray, q: np.ndarray | None = None, s: np.ndarray | None = None):
    """fp32 [n, H, I] -> codes [n, Hp, Ip], scale bytes [n, Hp, Ip/32]."""
    n, H, I = w2.shape
    Hp, Ip = _pad128(H), _pad128(I)
    q = np.empty((n, Hp, Ip), np.uint8) if q is None else q
    s = np.empty((n, Hp, Ip // 32), np.uint8) if s is None else s
    lib().oracle_mx_pack_w2(_p(np.ascontiguousarray(w2, np.float32)), H, I, n, _p(q), _p(s))
    return q, s


def mx_forward(x, rw, rb, w13, s13, b13, w2, s2, b2, k: int, tokens=None, want_intermediates: bool = False,
               weights: str = "mxfp8"):
    """Layer output rows (bf16 bits) of the MXFP8 variant; arguments as forward()
    with MX codes and scale bytes (s13 [E, 2Ip, Hp/32], s2 [E, Hp, Ip/32]).
    weights="mxfp4": the weight codes are E2M1 (one per byte, from mx4_pack_*)."""
    T, H = x.shape
    E = rw.shape[0]
    I = b13.shape[1] // 2
    Ip = _pad128(I)
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tok is None else len(tok)
    out = np.empty((n, H), np.uint16)
    hq = np.empty((n * k, Ip), np.uint8) if want_intermediates else None
    sh = np.empty((n * k, Ip // 32), np.uint8) if want_intermediates else None
    y = np.empty((n * k, H), np.float64) if want_intermediates else None
    ids = np.empty(n * k, np.int32) if want_intermediates else None
    fwd = lib().oracle_mx4_forward if weights == "mxfp4" else lib().oracle_mx_forward
    fwd(_p(np.ascontiguousarray(x, np.uint16)), _p(np.ascontiguousarray(rw, np.uint16)),
                            _p(np.ascontiguousarray(rb, np.uint16)), _p(w13), _p(s13),
                            _p(np.ascontiguousarray(b13, np.uint16)), _p(w2), _p(s2),
                            _p(np.ascontiguousarray(b2, np.uint16)), T, H, I, E, k, _p(tok), n, _p(out), _p(hq),
                            _p(sh), _p(y), _p(ids))
    if want_intermediates:
        return out, dict(hq=hq, sh=sh, y=y, idx=ids)
    return out


# ---- MXFP4 weights (E2M1 codes, one per byte) ----
def e2m1_decode(c: int) -> float:
    return float(lib().oracle_e2m1_decode(int(c)))


def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_encode(float(v)))


def mx4_quant_rows_f32(x: np.ndarray):
    """fp32 [rows, cols] -> E2M1 codes [rows, Cp] (one per byte), scale bytes [rows, Cp/32]."""
    rows, cols = x.shape
    cp = _pad128(cols)
    q = np.empty((rows, cp), np.uint8)
    s = np.empty((rows, cp // 32), np.uint8)
    lib().oracle_mx4_quant_rows_f32(_p(np.ascontiguousarray(x, np.float32)), rows, cols, _p(q), _p(s))
    return q, s


def mx4_pack_w13(w13: np.ndarray, q: np.ndarray | None = None, s: np.ndarray | None = None):
    """fp32 [n, 2I, H] -> E2M1 codes [n, 2Ip, Hp], scale bytes [n, 2Ip, Hp/32]."""
    n, twoI, H = w13.shape
    I = twoI // 2
    Hp, Ip = _pad128(H), _pad128(I)
    q = np.empty((n, 2 * Ip, Hp), np.uint8) if q is None else q
    s = np.empty((n, 2 * Ip, Hp // 32), np.uint8) if s is None else s
    lib().oracle_mx4_pack_w13(_p(np.ascontiguousarray(w13, np.float32)), H, I, n, _p(q), _p(s))
    return q, s


def mx4_pack_w2(w2: np.ndarray, q: np.ndarray | None = None, s: np.ndarray | None = None):
    """fp32 [n, H, I] -> E2M1 codes [n, Hp, Ip], scale bytes [n, Hp, Ip/32]."""
    n, H, I = w2.shape
    Hp, Ip = _pad128(H), _pad128(I)
    q = np.empty((n, Hp, Ip), np.uint8) if q is None else q
    s = np.empty((n, Hp, Ip // 32), np.uint8) if s is None else s
    lib().oracle_mx4_pack_w2(_p(np.ascontiguousarray(w2, np.float32)), H, I, n, _p(q), _p(s))
    return q, s


def mx4_forward(x, rw, rb, w13, s13, b13, w2, s2, b2, k: int, tokens=None, want_intermediates: bool = False):
    """The layer with MXFP4 weights and MXFP8 activations (see mx_forward)."""
    return mx_forward(x, rw, rb, w13, s13, b13, w2, s2, b2, k, tokens=tokens, want_intermediates=want_intermediates,
                      weights="mxfp4")
