"""Sparse Mixture-of-Experts MLP layer forward (gpt-oss style) on GB300.

Thin Python binding of the C ABI in ``include/moe_gb300.h`` (library
``libmoe_gb300.so``, built in-tree for sm_103a).  Every step of the layer runs
in the library's CUDA kernels; this module only checks tensors and passes
pointers, sizes and the current CUDA stream.  There is no CPU fallback: if the
library is missing, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB, build

__all__ = ["MoeError", "build", "lib", "workspace_size", "workspace_layout", "workspace_views", "forward",
           "pack_weights", "pack_weights_into", "w13_shape", "w2_shape", "unblock", "quantize_rows",
           "read_device_status", "test_bounded_wait", "MoeLayer", "pad128", "pack_weights_mx",
           "pack_weights_into_mx", "s13_mx_shape", "s2_mx_shape", "unblock_scales_mx", "quantize_rows_mx",
           "pack_weights_mxfp4", "pack_weights_into_mxfp4", "w13_shape_fp4", "w2_shape_fp4", "unblock_fp4",
           "weight_format", "route_debug", "block_weights", "read_static_scratch_status"]

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small", 4: "CUDA error",
          5: "device wait timed out"}


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: moe_status {code} ({STATUS.get(code, '?')})")
        self.code = code


_LAYOUT_FIELDS = ["total_bytes", "status", "hist", "count", "offset", "chunk_base", "tiles1", "tiles2", "topk_idx",
                  "topk_w", "topk_wb", "perm", "inv", "xq", "sx", "hq", "sh", "part"]


class _Layout(ctypes.Structure):
    _fields_ = [(f, ctypes.c_size_t) for f in _LAYOUT_FIELDS]


_lib = None


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB)
        vp, i32, sz, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
        L.moe_workspace_size.argtypes = [i32] * 5
        L.moe_workspace_size.restype = sz
        L.moe_get_workspace_layout.argtypes = [i32] * 5 + [ctypes.POINTER(_Layout)]
        L.moe_get_workspace_layout.restype = i32
        L.moe_forward.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp, sz, vp]
        L.moe_forward.restype = i32
        L.moe_forward_profiled.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp, sz, vp, vp]
        L.moe_forward_profiled.restype = i32
        L.moe_forward_static_scratch.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp]
        L.moe_forward_static_scratch.restype = i32
        L.moe_read_static_scratch_status.argtypes = [vp]
        L.moe_read_static_scratch_status.restype = i32
        L.moe_route_workspace_size.argtypes = [i32] * 4
        L.moe_route_workspace_size.restype = sz
        L.moe_route_debug.argtypes = [vp] * 3 + [i32] * 4 + [vp] * 7 + [sz, vp]
        L.moe_route_debug.restype = i32
        L.moe_block_weights.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
        L.moe_block_weights.restype = i32
        L.moe_pack_weights.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
        L.moe_pack_weights.restype = i32
        L.moe_quantize_rows.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_quantize_rows.restype = i32
        L.moe_workspace_size_mx.argtypes = [i32] * 5
        L.moe_workspace_size_mx.restype = sz
        L.moe_get_workspace_layout_mx.argtypes = [i32] * 5 + [ctypes.POINTER(_Layout)]
        L.moe_get_workspace_layout_mx.restype = i32
        L.moe_forward_mx.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp, sz, vp]
        L.moe_forward_mx.restype = i32
        L.moe_forward_mx_profiled.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp, sz, vp, vp]
        L.moe_forward_mx_profiled.restype = i32
        L.moe_pack_weights_mx.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
        L.moe_pack_weights_mx.restype = i32
        L.moe_quantize_rows_mx.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_quantize_rows_mx.restype = i32
        L.moe_forward_mxfp4.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp, sz, vp]
        L.moe_forward_mxfp4.restype = i32
        L.moe_forward_mxfp4_profiled.argtypes = [vp] * 9 + [i32] * 5 + [vp, vp, sz, vp, vp]
        L.moe_forward_mxfp4_profiled.restype = i32
        L.moe_pack_weights_mxfp4.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
        L.moe_pack_weights_mxfp4.restype = i32
        L.moe_read_device_status.argtypes = [vp, vp]
        L.moe_read_device_status.restype = i32
        L.moe_test_bounded_wait.argtypes = [u64, i32, vp, vp]
        L.moe_test_bounded_wait.restype = i32
        L.moe_status_str.argtypes = [i32]
        L.moe_status_str.restype = ctypes.c_char_p
        _lib = L
    return _lib


def pad128(n: int) -> int:
    return (n + 127) // 128 * 128


def _check(code: int, what: str):
    if code != 0:
        raise MoeError(code, what)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def workspace_size(T: int, H: int, I: int, E: int, top_k: int, mx: bool = False) -> int:
    """Workspace bytes of moe_forward (mx=True: moe_forward_mx)."""
    f = lib().moe_workspace_size_mx if mx else lib().moe_workspace_size
    return int(f(T, H, I, E, top_k))


def workspace_layout(T: int, H: int, I: int, E: int, top_k: int, mx: bool = False) -> dict:
    L = _Layout()
    f = lib().moe_get_workspace_layout_mx if mx else lib().moe_get_workspace_layout
    _check(f(T, H, I, E, top_k, ctypes.byref(L)), "moe_get_workspace_layout")
    return {f: getattr(L, f) for f in _LAYOUT_FIELDS}


def new_workspace(T: int, H: int, I: int, E: int, top_k: int, device=None, mx: bool = False) -> torch.Tensor:
    n = workspace_size(T, H, I, E, top_k, mx)
    if n == 0:
        raise MoeError(1, "workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def m_tile_rows(T: int, E: int, top_k: int) -> int:
    """Rows per GEMM m-tile: 32 for decode-sized batches (T*top_k <= 64*E), else 128."""
    return 32 if T * top_k <= 64 * E else 128


def workspace_views(ws: torch.Tensor, T: int, H: int, I: int, E: int, top_k: int, mx: bool = False) -> dict:
    """Typed views of the intermediates a forward call left in `ws` (mx: of moe_forward_mx,
    whose sx / sh are scale atoms [m-tiles bound, K blocks, 512] of uint8)."""
    L = workspace_layout(T, H, I, E, top_k, mx)
    R, Hp, Ip = T * top_k, pad128(H), pad128(I)
    nch = (T + 255) // 256
    mtb = E + (R + m_tile_rows(T, E, top_k) - 1) // m_tile_rows(T, E, top_k)

    def v(name, n, dtype, shape):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[L[name]:L[name] + nbytes].view(dtype).view(shape)

    return dict(
        status=v("status", 64, torch.int32, (64,)),
        hist=v("hist", nch * E, torch.int32, (nch, E)),
        count=v("count", E, torch.int32, (E,)),
        offset=v("offset", E + 1, torch.int32, (E + 1,)),
        chunk_base=v("chunk_base", nch * E, torch.int32, (nch, E)),
        tiles1=v("tiles1", E + 1, torch.int32, (E + 1,)),
        tiles2=v("tiles2", E + 1, torch.int32, (E + 1,)),
        topk_idx=v("topk_idx", R, torch.int32, (T, top_k)),
        topk_w=v("topk_w", R, torch.float32, (T, top_k)),
        topk_wb=v("topk_wb", R, torch.bfloat16, (T, top_k)),
        perm=v("perm", R, torch.int32, (R,)),
        inv=v("inv", R, torch.int32, (R,)),
        xq=v("xq", R * Hp, torch.uint8, (R, Hp)),
        sx=(v("sx", mtb * Hp // 128 * 512, torch.uint8, (mtb, Hp // 128, 512)) if mx else
            v("sx", R * Hp // 128, torch.float32, (Hp // 128, R)).t()),  # stored K-block-major
        hq=v("hq", R * Ip, torch.uint8, (R, Ip)),
        sh=(v("sh", mtb * Ip // 128 * 512, torch.uint8, (mtb, Ip // 128, 512)) if mx else
            v("sh", R * Ip // 128, torch.float32, (Ip // 128, R)).t()),
        part=v("part", R * Hp, torch.float32, (R, Hp)),
    )


STAGES = ("router", "permute_quant", "gemm_gateup", "gemm_down", "combine")


def weight_format(w13: torch.Tensor, s13: torch.Tensor) -> str:
    """"block128" (fp32 block scales), "mxfp8" (uint8 scale atoms, e4m3 codes) or
    "mxfp4" (uint8 scale atoms, E2M1 codes two per byte: 64-byte block rows)."""
    if s13.dtype != torch.uint8:
        return "block128"
    return "mxfp4" if w13.shape[-1] == 64 else "mxfp8"


def forward(x, router_w, router_b, w13, s13, b13, w2, s2, b2, top_k: int, out=None, workspace=None, stream=None,
            events=None):
    """out [T, H] bf16 = the MoE layer applied to x [T, H] bf16.

    Weights from pack_weights (fp32 128x128 block scales: moe_forward), from
    pack_weights_mx (uint8 MX scale atoms: moe_forward_mx) or from
    pack_weights_mxfp4 (packed E2M1 codes: moe_forward_mxfp4); weight_format()
    tells them apart.  events: optional list of 6
    torch.cuda.Event(enable_timing=True); event i is recorded before stage i
    (STAGES) and event 5 after the last stage."""
    T, H = x.shape
    E = router_w.shape[0]
    I = b13.shape[1] // 2
    Hp, Ip = pad128(H), pad128(I)
    fmt = weight_format(w13, s13)
    mx = fmt != "block128"
    shapes = (w13_shape_fp4(E, H, I), w2_shape_fp4(E, H, I)) if fmt == "mxfp4" else (w13_shape(E, H, I),
                                                                                     w2_shape(E, H, I))
    if (tuple(w13.shape), tuple(w2.shape)) != shapes:
        raise ValueError(f"packed weight shapes {tuple(w13.shape)}, {tuple(w2.shape)} do not match H={H} I={I} E={E}")
    if mx:
        if tuple(s13.shape) != s13_mx_shape(E, H, I) or tuple(s2.shape) != s2_mx_shape(E, H, I):
            raise ValueError("MX scale atom shapes do not match")
    elif tuple(s13.shape) != (E, 2 * Ip // 128, Hp // 128) or tuple(s2.shape) != (E, Hp // 128, Ip // 128):
        raise ValueError("block scale shapes do not match")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_workspace(T, H, I, E, top_k, x.device, mx)
    sdt = torch.uint8 if mx else torch.float32
    ptrs = [_dev(x, torch.bfloat16, "x"), _dev(router_w, torch.bfloat16, "router_w"),
            _dev(router_b, torch.bfloat16, "router_b"), _dev(w13, torch.uint8, "w13"), _dev(s13, sdt, "s13"),
            _dev(b13, torch.bfloat16, "b13"), _dev(w2, torch.uint8, "w2"), _dev(s2, sdt, "s2"),
            _dev(b2, torch.bfloat16, "b2")]
    tail = (_dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
            _stream(stream))
    L = lib()
    name = {"block128": "moe_forward", "mxfp8": "moe_forward_mx", "mxfp4": "moe_forward_mxfp4"}[fmt]
    if events is None:
        code = getattr(L, name)(*ptrs, T, H, I, E, top_k, *tail)
    else:
        if len(events) != 6:
            raise ValueError("events must hold 6 CUDA events")
        arr = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
        code = getattr(L, name + "_profiled")(*ptrs, T, H, I, E, top_k, *tail, arr)
    _check(code, name)
    return out


def w13_shape(E: int, H: int, I: int) -> tuple:
    """Packed gate/up codes: blocked [E, 2*Ip/128, Hp/128, 128, 128] (each 128x128 block contiguous)."""
    return (E, 2 * pad128(I) // 128, pad128(H) // 128, 128, 128)


def w2_shape(E: int, H: int, I: int) -> tuple:
    """Packed down codes: blocked [E, Hp/128, Ip/128, 128, 128]."""
    return (E, pad128(H) // 128, pad128(I) // 128, 128, 128)


def unblock(q: torch.Tensor) -> torch.Tensor:
    """Blocked codes [E, RB, KB, 128, 128] -> row-major [E, RB*128, KB*128] (for inspection)."""
    E, RB, KB = q.shape[:3]
    return q.permute(0, 1, 3, 2, 4).reshape(E, RB * 128, KB * 128)


def pack_weights(w13_f32: torch.Tensor, w2_f32: torch.Tensor, stream=None, out=None):
    """fp32 masters w13 [E, 2I, H], w2 [E, H, I] -> (w13 e4m3 codes, s13, w2 codes, s2) in the layer's layout."""
    E, twoI, H = w13_f32.shape
    I = twoI // 2
    Hp, Ip = pad128(H), pad128(I)
    dev = w13_f32.device
    if out is None:
        out = (torch.empty(w13_shape(E, H, I), dtype=torch.uint8, device=dev),
               torch.empty((E, 2 * Ip // 128, Hp // 128), dtype=torch.float32, device=dev),
               torch.empty(w2_shape(E, H, I), dtype=torch.uint8, device=dev),
               torch.empty((E, Hp // 128, Ip // 128), dtype=torch.float32, device=dev))
    q13, s13, q2, s2 = out
    if tuple(w2_f32.shape) != (E, H, I):
        raise ValueError("w2 shape does not match w13")
    code = lib().moe_pack_weights(_dev(w13_f32, torch.float32, "w13_f32"), _dev(w2_f32, torch.float32, "w2_f32"), H,
                                  I, E, _dev(q13, torch.uint8, "w13"), _dev(s13, torch.float32, "s13"),
                                  _dev(q2, torch.uint8, "w2"), _dev(s2, torch.float32, "s2"), _stream(stream))
    _check(code, "moe_pack_weights")
    return q13, s13, q2, s2


def pack_weights_into(w13_f32, w2_f32, H: int, I: int, E: int, q13, s13, q2, s2, stream=None):
    """Pack a slice of experts (either master may be None) into preallocated outputs."""
    code = lib().moe_pack_weights(None if w13_f32 is None else _dev(w13_f32, torch.float32, "w13_f32"),
                                  None if w2_f32 is None else _dev(w2_f32, torch.float32, "w2_f32"), H, I, E,
                                  None if q13 is None else q13.data_ptr(), None if s13 is None else s13.data_ptr(),
                                  None if q2 is None else q2.data_ptr(), None if s2 is None else s2.data_ptr(),
                                  _stream(stream))
    _check(code, "moe_pack_weights")


def s13_mx_shape(E: int, H: int, I: int) -> tuple:
    """MX gate/up scale atoms: [E, 2*Ip/128, Hp/128, 512] uint8 (one atom per code block)."""
    return (E, 2 * pad128(I) // 128, pad128(H) // 128, 512)


def s2_mx_shape(E: int, H: int, I: int) -> tuple:
    """MX down scale atoms: [E, Hp/128, Ip/128, 512] uint8."""
    return (E, pad128(H) // 128, pad128(I) // 128, 512)


def unblock_scales_mx(s: torch.Tensor) -> torch.Tensor:
    """Scale atoms [E, RB, KB, 512] -> row-major UE8M0 bytes [E, RB*128, KB*4] (for inspection).
    Atom byte (r % 32) * 16 + (r // 32) * 4 + g holds row r, group g."""
    E, RB, KB = s.shape[:3]
    rows = s.reshape(E, RB, KB, 32, 4, 4).permute(0, 1, 2, 4, 3, 5).reshape(E, RB, KB, 128, 4)
    return rows.permute(0, 1, 3, 2, 4).reshape(E, RB * 128, KB * 4)


def pack_weights_mx(w13_f32: torch.Tensor, w2_f32: torch.Tensor, stream=None):
    """fp32 masters w13 [E, 2I, H], w2 [E, H, I] -> (w13 codes, s13 atoms, w2 codes, s2 atoms), MXFP8."""
    E, twoI, H = w13_f32.shape
    I = twoI // 2
    dev = w13_f32.device
    if tuple(w2_f32.shape) != (E, H, I):
        raise ValueError("w2 shape does not match w13")
    out = (torch.empty(w13_shape(E, H, I), dtype=torch.uint8, device=dev),
           torch.empty(s13_mx_shape(E, H, I), dtype=torch.uint8, device=dev),
           torch.empty(w2_shape(E, H, I), dtype=torch.uint8, device=dev),
           torch.empty(s2_mx_shape(E, H, I), dtype=torch.uint8, device=dev))
    pack_weights_into_mx(w13_f32, w2_f32, H, I, E, *out, stream=stream)
    return out


def pack_weights_into_mx(w13_f32, w2_f32, H: int, I: int, E: int, q13, s13, q2, s2, stream=None):
    """MXFP8-pack a slice of experts (either master may be None) into preallocated outputs."""
    code = lib().moe_pack_weights_mx(None if w13_f32 is None else _dev(w13_f32, torch.float32, "w13_f32"),
                                     None if w2_f32 is None else _dev(w2_f32, torch.float32, "w2_f32"), H, I, E,
                                     None if q13 is None else _dev(q13, torch.uint8, "w13"),
                                     None if s13 is None else _dev(s13, torch.uint8, "s13"),
                                     None if q2 is None else _dev(q2, torch.uint8, "w2"),
                                     None if s2 is None else _dev(s2, torch.uint8, "s2"), _stream(stream))
    _check(code, "moe_pack_weights_mx")


def w13_shape_fp4(E: int, H: int, I: int) -> tuple:
    """Packed MXFP4 gate/up codes: blocked [E, 2*Ip/128, Hp/128, 128, 64], two E2M1 codes per byte."""
    return (E, 2 * pad128(I) // 128, pad128(H) // 128, 128, 64)


def w2_shape_fp4(E: int, H: int, I: int) -> tuple:
    """Packed MXFP4 down codes: blocked [E, Hp/128, Ip/128, 128, 64]."""
    return (E, pad128(H) // 128, pad128(I) // 128, 128, 64)


def unblock_fp4(q: torch.Tensor) -> torch.Tensor:
    """Blocked packed E2M1 codes [E, RB, KB, 128, 64] -> one code per byte, row-major
    [E, RB*128, KB*128] (value 2j of a row is the low nibble of byte j; for inspection)."""
    codes = torch.stack((q & 15, q >> 4), dim=-1).reshape(*q.shape[:4], 128)
    return unblock(codes)


def pack_weights_mxfp4(w13_f32: torch.Tensor, w2_f32: torch.Tensor, stream=None):
    """fp32 masters w13 [E, 2I, H], w2 [E, H, I] -> (w13 packed E2M1 codes, s13 atoms, w2 codes, s2 atoms)."""
    E, twoI, H = w13_f32.shape
    I = twoI // 2
    dev = w13_f32.device
    if tuple(w2_f32.shape) != (E, H, I):
        raise ValueError("w2 shape does not match w13")
    out = (torch.empty(w13_shape_fp4(E, H, I), dtype=torch.uint8, device=dev),
           torch.empty(s13_mx_shape(E, H, I), dtype=torch.uint8, device=dev),
           torch.empty(w2_shape_fp4(E, H, I), dtype=torch.uint8, device=dev),
           torch.empty(s2_mx_shape(E, H, I), dtype=torch.uint8, device=dev))
    pack_weights_into_mxfp4(w13_f32, w2_f32, H, I, E, *out, stream=stream)
    return out


def pack_weights_into_mxfp4(w13_f32, w2_f32, H: int, I: int, E: int, q13, s13, q2, s2, stream=None):
    """MXFP4-pack a slice of experts (either master may be None) into preallocated outputs."""
    code = lib().moe_pack_weights_mxfp4(None if w13_f32 is None else _dev(w13_f32, torch.float32, "w13_f32"),
                                        None if w2_f32 is None else _dev(w2_f32, torch.float32, "w2_f32"), H, I, E,
                                        None if q13 is None else _dev(q13, torch.uint8, "w13"),
                                        None if s13 is None else _dev(s13, torch.uint8, "s13"),
                                        None if q2 is None else _dev(q2, torch.uint8, "w2"),
                                        None if s2 is None else _dev(s2, torch.uint8, "s2"), _stream(stream))
    _check(code, "moe_pack_weights_mxfp4")


def quantize_rows_mx(v: torch.Tensor, stream=None):
    """1x32 MX quantisation of fp32 rows [rows, cols] -> (codes [rows, cols_p] u8, UE8M0 bytes [rows, cols_p/32])."""
    rows, cols = v.shape
    cp = pad128(cols)
    q = torch.empty((rows, cp), dtype=torch.uint8, device=v.device)
    s = torch.empty((rows, cp // 32), dtype=torch.uint8, device=v.device)
    _check(lib().moe_quantize_rows_mx(_dev(v, torch.float32, "v"), rows, cols, cols, q.data_ptr(), s.data_ptr(),
                                      _stream(stream)), "moe_quantize_rows_mx")
    return q, s


def quantize_rows(v: torch.Tensor, stream=None):
    """1x128 group quantisation of fp32 rows [rows, cols] -> (codes [rows, cols_p] u8, scales [rows, cols_p/128])."""
    rows, cols = v.shape
    cp = pad128(cols)
    q = torch.empty((rows, cp), dtype=torch.uint8, device=v.device)
    s = torch.empty((rows, cp // 128), dtype=torch.float32, device=v.device)
    _check(lib().moe_quantize_rows(_dev(v, torch.float32, "v"), rows, cols, cols, q.data_ptr(), s.data_ptr(),
                                   _stream(stream)), "moe_quantize_rows")
    return q, s


def route_debug(x, router_w, router_b, top_k: int, stream=None) -> dict:
    """The routing steps alone (moe_route_debug): topk_idx [T, k] int32, topk_w [T, k]
    fp32, offset [E+1], perm [R], xq [R, Hp] e4m3 codes and sx [R, Hp/128] (stored
    K-block-major, returned transposed as a view) in new device tensors."""
    T, H = x.shape
    E = router_w.shape[0]
    R, Hp = T * top_k, pad128(H)
    dev = x.device
    need = int(lib().moe_route_workspace_size(T, H, E, top_k))
    if need == 0:
        raise MoeError(1, "moe_route_workspace_size")
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    o = dict(topk_idx=torch.empty((T, top_k), dtype=torch.int32, device=dev),
             topk_w=torch.empty((T, top_k), dtype=torch.float32, device=dev),
             offset=torch.empty(E + 1, dtype=torch.int32, device=dev),
             perm=torch.empty(R, dtype=torch.int32, device=dev),
             xq=torch.empty((R, Hp), dtype=torch.uint8, device=dev),
             sx_kmajor=torch.empty((Hp // 128, R), dtype=torch.float32, device=dev))
    code = lib().moe_route_debug(_dev(x, torch.bfloat16, "x"), _dev(router_w, torch.bfloat16, "router_w"),
                                 _dev(router_b, torch.bfloat16, "router_b"), T, H, E, top_k, o["topk_idx"].data_ptr(),
                                 o["topk_w"].data_ptr(), o["offset"].data_ptr(), o["perm"].data_ptr(),
                                 o["xq"].data_ptr(), o["sx_kmajor"].data_ptr(), ws.data_ptr(), ws.numel(),
                                 _stream(stream))
    _check(code, "moe_route_debug")
    o["sx"] = o["sx_kmajor"].t()
    return o


def block_weights(w13_rm: torch.Tensor, w2_rm: torch.Tensor, H: int, I: int, stream=None):
    """Row-major e4m3 codes w13 [E, 2*Ip, Hp], w2 [E, Hp, Ip] (uint8) -> the blocked
    layout of w13_shape / w2_shape (moe_block_weights)."""
    E = w13_rm.shape[0]
    Hp, Ip = pad128(H), pad128(I)
    if tuple(w13_rm.shape) != (E, 2 * Ip, Hp) or tuple(w2_rm.shape) != (E, Hp, Ip):
        raise ValueError("row-major code shapes do not match H, I")
    q13 = torch.empty(w13_shape(E, H, I), dtype=torch.uint8, device=w13_rm.device)
    q2 = torch.empty(w2_shape(E, H, I), dtype=torch.uint8, device=w13_rm.device)
    _check(lib().moe_block_weights(_dev(w13_rm, torch.uint8, "w13_rm"), _dev(w2_rm, torch.uint8, "w2_rm"), H, I, E,
                                   q13.data_ptr(), q2.data_ptr(), _stream(stream)), "moe_block_weights")
    return q13, q2


def read_static_scratch_status(stream=None) -> int:
    """Synchronise and return the device status code moe_forward_static_scratch
    left in its array on the current device (0 = ok, 5 = a wait timed out)."""
    return int(lib().moe_read_static_scratch_status(_stream(stream)))


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the device status code of the last forward (0 = ok, 5 = a wait timed out)."""
    return int(lib().moe_read_device_status(_dev(workspace, torch.uint8, "workspace"), _stream(stream)))


def test_bounded_wait(timeout_ns: int, arrivals: int, stream=None) -> int:
    """1 if a barrier wait completed, 2 if it gave up after timeout_ns (see moe_test_bounded_wait)."""
    r = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(lib().moe_test_bounded_wait(int(timeout_ns), int(arrivals), r.data_ptr(), _stream(stream)),
           "moe_test_bounded_wait")
    torch.cuda.synchronize()
    return int(r.item())


class MoeLayer:
    """A layer with packed weights resident on the GPU and a reusable workspace."""

    def __init__(self, router_w, router_b, w13, s13, b13, w2, s2, b2, top_k: int):
        self.router_w, self.router_b = router_w, router_b
        self.w13, self.s13, self.b13, self.w2, self.s2, self.b2 = w13, s13, b13, w2, s2, b2
        self.top_k = top_k
        self.E, self.H = router_w.shape
        self.I = b13.shape[1] // 2
        self.mx = s13.dtype == torch.uint8  # MX scale atoms (pack_weights_mx / pack_weights_mxfp4)
        self._ws = None

    def workspace(self, T: int) -> torch.Tensor:
        need = workspace_size(T, self.H, self.I, self.E, self.top_k, self.mx)
        if self._ws is None or self._ws.numel() < need:
            self._ws = new_workspace(T, self.H, self.I, self.E, self.top_k, self.router_w.device, self.mx)
        return self._ws

    def __call__(self, x: torch.Tensor, out=None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        return forward(x, self.router_w, self.router_b, self.w13, self.s13, self.b13, self.w2, self.s2, self.b2,
                       self.top_k, out=out, workspace=self.workspace(T), stream=stream)

    def graphed(self, T: int) -> "GraphedMoeLayer":
        """The layer for batches of exactly T tokens captured once as a CUDA graph
        (see GraphedMoeLayer)."""
        return GraphedMoeLayer(self, T)


class GraphedMoeLayer:
    """One batch size of a MoeLayer captured as a CUDA graph: the workspace memset
    and the five kernels of a forward, with their programmatic dependencies.
    `x` and `out` are the graph's static device buffers ([T, H] bf16): write the
    batch into `x`, call, read `out`.  A call replays the graph on the current
    stream, one launch instead of six."""

    def __init__(self, layer: MoeLayer, T: int):
        dev = layer.router_w.device
        self.layer, self.T = layer, T
        self.x = torch.zeros((T, layer.H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=dev)
        ws = layer.workspace(T)
        # one eager call first: kernel attributes and tensor-map encoders are set up outside the capture
        layer(self.x, out=self.out)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            forward(self.x, layer.router_w, layer.router_b, layer.w13, layer.s13, layer.b13, layer.w2, layer.s2,
                    layer.b2, layer.top_k, out=self.out, workspace=ws)

    def __call__(self) -> torch.Tensor:
        self.graph.replay()
        return self.out
