"""Thin ctypes binding of libqk (include/qk.h): argument marshalling only.

Each function has the C entry point's name and argument order. Tensor
arguments are torch CUDA tensors (or None); they are passed as raw device
pointers. The stream defaults to torch's current CUDA stream. Every step of
the computation runs in the library's kernels; nothing here computes.
A non-QK_OK status raises QkError with the library's one-line reason. If the
shared library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(HERE), "include", "qk.h")

QK_OK = 0
STATUS = {0: "QK_OK", 1: "QK_ERR_ARG", 2: "QK_ERR_SHAPE", 3: "QK_ERR_ALIAS", 4: "QK_ERR_WORKSPACE",
          5: "QK_ERR_UNSUPPORTED", 6: "QK_ERR_CUDA"}
NORM = {"plain": 0, "mul": 1, "mul_add": 2, "scale": 3}
GLU = {"swiglu": 0, "geglu_tanh": 1, "reglu": 2, "geglu_erf": 3, "geglu_quick": 4, "swiglu_oai": 5,
       "swiglu_clamp": 6}
LAYOUT = {"separate": 0, "packed": 1, "packed_swapped": 2}
WTYPE = {"q4_0": 0, "q8_0": 1}
Q8_1_BLOCK_BYTES = 36


class QkError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{func}: {self.name}: {detail}")


class qk_proj(C.Structure):
    _fields_ = [("wtype", C.c_int32), ("reserved", C.c_int32), ("w", C.c_void_p), ("N", C.c_int64),
                ("K", C.c_int64), ("y", C.c_void_p), ("y_stride", C.c_int64)]


class qk_proj_id(C.Structure):
    _fields_ = [("wtype", C.c_int32), ("n_experts", C.c_int32), ("w", C.c_void_p), ("N", C.c_int64),
                ("K", C.c_int64), ("y", C.c_void_p)]


class qk_image_memo(C.Structure):
    """The consecutive-window memo (see qk.h): all zeros is empty."""
    _fields_ = [("format", C.c_int32), ("reserved", C.c_int32), ("x", C.c_void_p), ("T", C.c_int64),
                ("K", C.c_int64), ("x_stride", C.c_int64), ("row_blocks", C.c_int64), ("dst0", C.c_void_p),
                ("dst1", C.c_void_p), ("stream", C.c_void_p)]


MEMO_Q8_0, MEMO_Q8_1 = 1, 2

_lock = threading.Lock()
_lib = None

P, I32, I64, F32, SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t
_SIGS = {
    "qk_status_string": ([C.c_int], C.c_char_p),
    "qk_last_error": ([], C.c_char_p),
    "qk_last_error_string": ([], C.c_char_p),
    "qk_launch_count": ([], C.c_uint64),
    "qk_quantize_q8_1": ([P, I64, I64, I64, P, I64, P, P], C.c_int),
    "qk_quantize_q8_0": ([P, I64, I64, I64, P, P, I64, P, P], C.c_int),
    "qk_rmsnorm_q8_1": ([P, I64, I64, I64, C.c_int, P, P, F32, F32, P, I64, P, I64, P, P], C.c_int),
    "qk_rmsnorm_q8_0": ([P, I64, I64, I64, C.c_int, P, P, F32, F32, P, I64, P, P, I64, P, P], C.c_int),
    "qk_glu_q8_1": ([C.c_int, C.c_int, P, I64, P, I64, I64, I64, P, I64, P, I64, P, P], C.c_int),
    "qk_glu_q8_1_ex": ([C.c_int, C.c_int, P, I64, P, I64, I64, I64, P, I64, P, I64, C.c_float, C.c_float, P, P],
                       C.c_int),
    "qk_weight_packed_bytes": ([C.c_int, I64, I64], SZ),
    "qk_weight_pack": ([C.c_int, P, I64, I64, P, SZ, P], C.c_int),
    "qk_device_faults": ([C.POINTER(C.c_uint32)], C.c_int),
    "qk_selftest_wait_timeout": ([C.c_void_p], C.c_int),
    "qk_mmvq_workspace_bytes": ([I32, C.POINTER(qk_proj)], SZ),
    "qk_mmvq": ([P, I64, I64, I32, C.POINTER(qk_proj), P, P, SZ, P], C.c_int),
    "qk_mmvq_static_ws": ([P, I64, I64, I32, C.POINTER(qk_proj), P, P], C.c_int),
    "qk_topk_route": ([P, I64, I32, I32, P, P, P, P], C.c_int),
    "qk_moe_plan": ([P, I64, I32, I32, P, P, P, P, P], C.c_int),
    "qk_route_plan": ([P, I64, I32, I32, P, P, P, P, P, P, P], C.c_int),
    "qk_mmvq_id": ([P, I64, I64, I32, I32, C.POINTER(qk_proj_id), P, P, P, P], C.c_int),
    "qk_mmvq_id_slots": ([P, I64, I64, I32, I32, C.POINTER(qk_proj_id), P, P, P, P], C.c_int),
    "qk_moe_combine": ([P, I64, P, I64, I32, I64, P, I64, P, P], C.c_int),
    "qk_mmq_workspace_bytes": ([I64, I32, C.POINTER(qk_proj)], C.c_size_t),
    "qk_image_memo_clear": ([C.POINTER(qk_image_memo)], None),
    "qk_image_memo_match": ([C.POINTER(qk_image_memo), I32, P, I64, I64, I64, P, P, I64, P], I32),
    "qk_image_memo_quantize_q8_0": ([C.POINTER(qk_image_memo), P, I64, I64, I64, P, P, I64, C.POINTER(I32), P],
                                    C.c_int),
    "qk_image_memo_quantize_q8_1": ([C.POINTER(qk_image_memo), P, I64, I64, I64, P, I64, C.POINTER(I32), P],
                                    C.c_int),
    "qk_mmq": ([P, P, I64, I64, I32, C.POINTER(qk_proj), P, C.c_size_t, P], C.c_int),
}


def library_path() -> str:
    from . import build as _build
    return _build.LIB


def load(build_if_missing: bool = True):
    """Loads libqk.so (building it with nvcc first if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libqk.so is not built ({path}); run quantized_activation_q4_gb300.build.build()")
                from . import build as _build
                path = _build.build()
            lib = C.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def declared_symbols() -> list[str]:
    """Every qk_* function declared in include/qk.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(qk_\w+)\s*\(", text, flags=re.M)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return C.c_void_p(t)
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _check(func: str, st: int):
    if st != QK_OK:
        raise QkError(st, func, load().qk_last_error().decode())


def launch_count() -> int:
    return int(load().qk_launch_count())


# ------------------------------------------------------------------ image
def qk_quantize_q8_1(x, T, K, x_stride, img, img_row_blocks, d_live_rows=None, stream=None):
    _check("qk_quantize_q8_1", load().qk_quantize_q8_1(_ptr(x), T, K, x_stride, _ptr(img), img_row_blocks,
                                                       _ptr(d_live_rows), _stream(stream)))


def qk_quantize_q8_0(x, T, K, x_stride, qs, d, row_blocks, d_live_rows=None, stream=None):
    _check("qk_quantize_q8_0", load().qk_quantize_q8_0(_ptr(x), T, K, x_stride, _ptr(qs), _ptr(d), row_blocks,
                                                       _ptr(d_live_rows), _stream(stream)))


def qk_rmsnorm_q8_1(x, T, K, x_stride, kind, w, b, scale, eps, y, y_stride, img, img_row_blocks,
                    d_live_rows=None, stream=None):
    kind = NORM[kind] if isinstance(kind, str) else int(kind)
    _check("qk_rmsnorm_q8_1", load().qk_rmsnorm_q8_1(_ptr(x), T, K, x_stride, kind, _ptr(w), _ptr(b),
                                                     float(scale), float(eps), _ptr(y), y_stride, _ptr(img),
                                                     img_row_blocks, _ptr(d_live_rows), _stream(stream)))


def qk_rmsnorm_q8_0(x, T, K, x_stride, kind, w, b, scale, eps, y, y_stride, qs, d, row_blocks,
                    d_live_rows=None, stream=None):
    kind = NORM[kind] if isinstance(kind, str) else int(kind)
    _check("qk_rmsnorm_q8_0", load().qk_rmsnorm_q8_0(_ptr(x), T, K, x_stride, kind, _ptr(w), _ptr(b),
                                                     float(scale), float(eps), _ptr(y), y_stride, _ptr(qs), _ptr(d),
                                                     row_blocks, _ptr(d_live_rows), _stream(stream)))


def qk_glu_q8_1(kind, layout, a, a_stride, b, b_stride, T, N, out, out_stride, img, img_row_blocks,
                d_live_rows=None, stream=None):
    kind = GLU[kind] if isinstance(kind, str) else int(kind)
    layout = LAYOUT[layout] if isinstance(layout, str) else int(layout)
    _check("qk_glu_q8_1", load().qk_glu_q8_1(kind, layout, _ptr(a), a_stride, _ptr(b), b_stride, T, N, _ptr(out),
                                             out_stride, _ptr(img), img_row_blocks, _ptr(d_live_rows),
                                             _stream(stream)))


def qk_glu_q8_1_ex(kind, layout, a, a_stride, b, b_stride, T, N, out, out_stride, img, img_row_blocks,
                   alpha=1.702, limit=7.0, d_live_rows=None, stream=None):
    kind = GLU[kind] if isinstance(kind, str) else int(kind)
    layout = LAYOUT[layout] if isinstance(layout, str) else int(layout)
    _check("qk_glu_q8_1_ex", load().qk_glu_q8_1_ex(kind, layout, _ptr(a), a_stride, _ptr(b), b_stride, T, N,
                                                   _ptr(out), out_stride, _ptr(img), img_row_blocks,
                                                   float(alpha), float(limit), _ptr(d_live_rows),
                                                   _stream(stream)))


# ------------------------------------------------------------------ weights
def qk_weight_packed_bytes(wtype, N, K) -> int:
    wtype = WTYPE[wtype] if isinstance(wtype, str) else int(wtype)
    return int(load().qk_weight_packed_bytes(wtype, N, K))


def qk_weight_pack(wtype, blocks, N, K, packed, packed_bytes, stream=None):
    wtype = WTYPE[wtype] if isinstance(wtype, str) else int(wtype)
    _check("qk_weight_pack", load().qk_weight_pack(wtype, _ptr(blocks), N, K, _ptr(packed), packed_bytes,
                                                   _stream(stream)))


# ------------------------------------------------------------------ projections
def make_proj(wtype, w, N, K, y, y_stride) -> qk_proj:
    wtype = WTYPE[wtype] if isinstance(wtype, str) else int(wtype)
    return qk_proj(wtype, 0, _ptr(w), N, K, _ptr(y), y_stride)


def make_proj_id(wtype, n_experts, w, N, K, y) -> qk_proj_id:
    wtype = WTYPE[wtype] if isinstance(wtype, str) else int(wtype)
    return qk_proj_id(wtype, n_experts, _ptr(w), N, K, _ptr(y))


def qk_mmvq_workspace_bytes(projs) -> int:
    arr = (qk_proj * len(projs))(*projs)
    return int(load().qk_mmvq_workspace_bytes(len(projs), arr))


def qk_mmvq(img, img_row_blocks, T, projs, ws, ws_bytes, d_live_rows=None, stream=None):
    arr = (qk_proj * len(projs))(*projs)
    _check("qk_mmvq", load().qk_mmvq(_ptr(img), img_row_blocks, T, len(projs), arr, _ptr(d_live_rows),
                                     _ptr(ws), ws_bytes, _stream(stream)))


def qk_mmvq_static_ws(img, img_row_blocks, T, projs, d_live_rows=None, stream=None):
    """qk_mmvq with the library's own static scratch array (no workspace argument)."""
    arr = (qk_proj * len(projs))(*projs)
    _check("qk_mmvq_static_ws", load().qk_mmvq_static_ws(_ptr(img), img_row_blocks, T, len(projs), arr,
                                                         _ptr(d_live_rows), _stream(stream)))


def qk_selftest_wait_timeout(stream=None):
    _check("qk_selftest_wait_timeout", load().qk_selftest_wait_timeout(_stream(stream)))


def qk_device_faults() -> int:
    v = C.c_uint32(0)
    _check("qk_device_faults", load().qk_device_faults(C.byref(v)))
    return int(v.value)


def qk_mmvq_id(img, img_row_blocks, rows, k, projs, counts, offsets, items, stream=None):
    arr = (qk_proj_id * len(projs))(*projs)
    _check("qk_mmvq_id", load().qk_mmvq_id(_ptr(img), img_row_blocks, rows, k, len(projs), arr, _ptr(counts),
                                           _ptr(offsets), _ptr(items), _stream(stream)))


def qk_mmvq_id_slots(img, img_row_blocks, rows, k, projs, counts, offsets, items, stream=None):
    arr = (qk_proj_id * len(projs))(*projs)
    _check("qk_mmvq_id_slots", load().qk_mmvq_id_slots(_ptr(img), img_row_blocks, rows, k, len(projs), arr,
                                                       _ptr(counts), _ptr(offsets), _ptr(items), _stream(stream)))


def qk_moe_combine(expert_out, out_stride, wts, rows, k, N, y, y_stride, d_live_rows=None, stream=None):
    _check("qk_moe_combine", load().qk_moe_combine(_ptr(expert_out), out_stride, _ptr(wts), rows, k, N, _ptr(y),
                                                   y_stride, _ptr(d_live_rows), _stream(stream)))


def qk_mmq_workspace_bytes(T, projs) -> int:
    arr = (qk_proj * len(projs))(*projs)
    return int(load().qk_mmq_workspace_bytes(T, len(projs), arr))


def qk_image_memo_clear(memo):
    load().qk_image_memo_clear(C.byref(memo))


def qk_image_memo_quantize_q8_0(memo, x, T, K, x_stride, qs, d, row_blocks, stream=None) -> bool:
    """Quantises x into (qs, d) unless memo says they already hold it; returns whether it was a hit."""
    hit = I32(0)
    _check("qk_image_memo_quantize_q8_0",
           load().qk_image_memo_quantize_q8_0(C.byref(memo), _ptr(x), T, K, x_stride, _ptr(qs), _ptr(d), row_blocks,
                                              C.byref(hit), _stream(stream)))
    return bool(hit.value)


def qk_image_memo_quantize_q8_1(memo, x, T, K, x_stride, img, img_row_blocks, stream=None) -> bool:
    hit = I32(0)
    _check("qk_image_memo_quantize_q8_1",
           load().qk_image_memo_quantize_q8_1(C.byref(memo), _ptr(x), T, K, x_stride, _ptr(img), img_row_blocks,
                                              C.byref(hit), _stream(stream)))
    return bool(hit.value)


def qk_mmq(qs, d, row_blocks, T, projs, ws, ws_bytes, stream=None):
    arr = (qk_proj * len(projs))(*projs)
    _check("qk_mmq", load().qk_mmq(_ptr(qs), _ptr(d), row_blocks, T, len(projs), arr, _ptr(ws), ws_bytes,
                                   _stream(stream)))


# ------------------------------------------------------------------ routing
def qk_topk_route(logits, rows, E, k, ids, wts, d_live_rows=None, stream=None):
    _check("qk_topk_route", load().qk_topk_route(_ptr(logits), rows, E, k, _ptr(ids), _ptr(wts),
                                                 _ptr(d_live_rows), _stream(stream)))


def qk_moe_plan(ids, rows, k, E, counts, offsets, items, d_live_rows=None, stream=None):
    _check("qk_moe_plan", load().qk_moe_plan(_ptr(ids), rows, k, E, _ptr(counts), _ptr(offsets), _ptr(items),
                                             _ptr(d_live_rows), _stream(stream)))


def qk_route_plan(logits, rows, E, k, ids, wts, counts, offsets, items, d_live_rows=None, stream=None):
    _check("qk_route_plan", load().qk_route_plan(_ptr(logits), rows, E, k, _ptr(ids), _ptr(wts), _ptr(counts),
                                                 _ptr(offsets), _ptr(items), _ptr(d_live_rows), _stream(stream)))
