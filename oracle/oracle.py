"""Python face of the CPU oracle (TEST INFRASTRUCTURE ONLY).

Only tests/, the smoke check and the benchmark's CPU-baseline leg may import
this module. It compiles qk_oracle.c with gcc (no CUDA, no shared code with the
product library) and wraps each entry point for numpy arrays. The one step
done here rather than in C is the plain definition of a projection,
y = x @ W.T in float64, where numpy's matmul serves as the library primitive.

Page citations are on the C functions in qk_oracle.c.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qk_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

Q8_1_BYTES = 36
WTYPE = {"q4_0": 0, "q8_0": 1}
NORM_KIND = {"plain": 0, "mul": 1, "mul_add": 2, "scale": 3}
GLU_KIND = {"swiglu": 0, "geglu_tanh": 1, "reglu": 2, "geglu_erf": 3, "geglu_quick": 4, "swiglu_oai": 5,
            "swiglu_clamp": 6}
GLU_LAYOUT = {"separate": 0, "packed": 1, "packed_swapped": 2}


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, host arch)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P = C.c_void_p
            I64 = C.c_int64
            lib.or_f32_to_f16.argtypes = [C.c_float]
            lib.or_f32_to_f16.restype = C.c_uint16
            lib.or_f16_to_f32.argtypes = [C.c_uint16]
            lib.or_f16_to_f32.restype = C.c_float
            lib.or_f32_to_f16_array.argtypes = [P, I64, P]
            lib.or_f32_to_f16_array.restype = None
            lib.or_quantize_q8_1.argtypes = [P, I64, I64, I64, P, I64, P]
            lib.or_quantize_q8_0.argtypes = [P, I64, I64, I64, P, P, I64, P]
            lib.or_rmsnorm.argtypes = [P, I64, I64, I64, C.c_int, P, P, C.c_double, C.c_double, P, P]
            lib.or_glu.argtypes = [C.c_int, C.c_int, P, I64, P, I64, I64, I64, C.c_double, C.c_double, P, P]
            lib.or_dequant.argtypes = [C.c_int, P, I64, I64, P]
            lib.or_proj_q8_1.argtypes = [C.c_int, P, I64, I64, P, I64, I64, P]
            lib.or_proj_q8_0_sampled.argtypes = [C.c_int, P, I64, I64, P, P, I64, P, I64, P, I64, P]
            lib.or_topk_route.argtypes = [P, I64, C.c_int, C.c_int, P, P, P]
            lib.or_moe_plan.argtypes = [P, I64, C.c_int, C.c_int, P, P, P, P]
            lib.or_proj_id_q8_1.argtypes = [C.c_int, P, C.c_int, I64, I64, P, I64, P, C.c_int, P, I64, P]
            for name in ("or_quantize_q8_1", "or_quantize_q8_0", "or_rmsnorm", "or_glu", "or_dequant",
                         "or_proj_q8_1", "or_proj_q8_0_sampled", "or_topk_route", "or_moe_plan",
                         "or_proj_id_q8_1"):
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _live(live):
    if live is None:
        return None, None
    arr = np.array([int(live)], dtype=np.int32)
    return arr, _p(arr)


# ---------------------------------------------------------------- conversions
def f32_to_f16_bits(x) -> np.ndarray:
    """Oracle binary32 -> binary16 (RNE); returns uint16 bits, same shape as x."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().or_f32_to_f16_array(_p(x), x.size, _p(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    return np.fromiter((lib.or_f16_to_f32(int(v)) for v in h), dtype=np.float32, count=h.size)


# ---------------------------------------------------------------- quantizers
def quantize_q8_1(x: np.ndarray, K: int | None = None, row_blocks: int | None = None,
                  live: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Q8_1 image bytes [T, row_blocks*36] of F32 rows x[T, stride] (first K columns)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, stride = x.shape
    K = stride if K is None else K
    kb = (K + 31) // 32
    row_blocks = kb if row_blocks is None else row_blocks
    if out is None:
        out = np.zeros((T, row_blocks * Q8_1_BYTES), dtype=np.uint8)
    la, lp = _live(live)
    _load().or_quantize_q8_1(_p(x), T, K, stride, _p(out), row_blocks, lp)
    return out


def quantize_q8_0(x: np.ndarray, K: int | None = None, row_blocks: int | None = None,
                  live: int | None = None):
    """Q8_0 planes (qs int8 [T, row_blocks*32], d half-bits uint16 [T, row_blocks])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, stride = x.shape
    K = stride if K is None else K
    kb = (K + 31) // 32
    row_blocks = kb if row_blocks is None else row_blocks
    qs = np.zeros((T, row_blocks * 32), dtype=np.int8)
    dh = np.zeros((T, row_blocks), dtype=np.uint16)
    la, lp = _live(live)
    _load().or_quantize_q8_0(_p(x), T, K, stride, _p(qs), _p(dh), row_blocks, lp)
    return qs, dh


# ---------------------------------------------------------------- producers
def rmsnorm(x: np.ndarray, kind: str = "plain", w=None, b=None, scale: float = 1.0,
            eps: float = 1e-6, K: int | None = None, live: int | None = None) -> np.ndarray:
    """RMSNorm producer output in float64, shape [T, K]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, stride = x.shape
    K = stride if K is None else K
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    y = np.zeros((T, K), dtype=np.float64)
    la, lp = _live(live)
    _load().or_rmsnorm(_p(x), T, K, stride, NORM_KIND[kind], _p(w), _p(b), float(scale), float(eps), _p(y), lp)
    return y


def glu(kind: str, layout: str, a: np.ndarray, b: np.ndarray | None, N: int,
        live: int | None = None, alpha: float = 1.702, limit: float = 7.0) -> np.ndarray:
    """GLU producer output in float64, shape [T, N].

    layout "separate": a holds g rows, b holds u rows. "packed": a rows are
    [g | u]. "packed_swapped": a rows are [u | g]. alpha and limit are the
    SwiGLU-OAI parameters (taken as binary32 values, as the device receives them).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    T = a.shape[0]
    bb = a if b is None else np.ascontiguousarray(b, dtype=np.float32)
    out = np.zeros((T, N), dtype=np.float64)
    la, lp = _live(live)
    _load().or_glu(GLU_KIND[kind], GLU_LAYOUT[layout], _p(a), a.shape[1], _p(bb), bb.shape[1], T, N,
                   float(np.float32(alpha)), float(np.float32(limit)), _p(out), lp)
    return out


# ---------------------------------------------------------------- projections
def dequant(wtype: str, W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    out = np.zeros((N, K), dtype=np.float64)
    _load().or_dequant(WTYPE[wtype], _p(W), N, K, _p(out))
    return out


def proj_q8_1(wtype: str, W: np.ndarray, N: int, K: int, img: np.ndarray, row_blocks: int) -> np.ndarray:
    """Quantised-path projection of every image row: float64 [T, N]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    img = np.ascontiguousarray(img, dtype=np.uint8)
    T = img.shape[0]
    y = np.zeros((T, N), dtype=np.float64)
    _load().or_proj_q8_1(WTYPE[wtype], _p(W), N, K, _p(img), row_blocks, T, _p(y))
    return y


def proj_plain(wtype: str, W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    """Plain definition y = x @ W_deq.T in float64, from the F32 activation."""
    Wd = dequant(wtype, W, N, K)
    return np.asarray(x, dtype=np.float64)[:, :K] @ Wd.T


def proj_q8_0_sampled(wtype: str, W: np.ndarray, N: int, K: int, qs: np.ndarray, dh: np.ndarray,
                      row_blocks: int, rows, cols) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    qs = np.ascontiguousarray(qs, dtype=np.int8)
    dh = np.ascontiguousarray(dh, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.zeros((rows.size, cols.size), dtype=np.float64)
    _load().or_proj_q8_0_sampled(WTYPE[wtype], _p(W), N, K, _p(qs), _p(dh), row_blocks,
                                 _p(rows), rows.size, _p(cols), cols.size, _p(out))
    return out


# ---------------------------------------------------------------- routing
def topk_route(logits: np.ndarray, k: int, live: int | None = None, ids=None, wts=None):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    rows, E = logits.shape
    ids = np.full((rows, k), -1, dtype=np.int32) if ids is None else np.array(ids, dtype=np.int32)
    wts = np.full((rows, k), np.nan, dtype=np.float64) if wts is None else np.array(wts, dtype=np.float64)
    la, lp = _live(live)
    _load().or_topk_route(_p(logits), rows, E, k, _p(ids), _p(wts), lp)
    return ids, wts


def moe_plan(ids: np.ndarray, E: int, live: int | None = None):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rows, k = ids.shape
    counts = np.zeros(E, dtype=np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    items = np.full(rows * k, -1, dtype=np.int32)
    la, lp = _live(live)
    _load().or_moe_plan(_p(ids), rows, k, E, _p(counts), _p(offsets), _p(items), lp)
    n = int(offsets[E])
    return counts, offsets, items[:n].copy()


def proj_id_q8_1(wtype: str, W: np.ndarray, E: int, N: int, K: int, img: np.ndarray, row_blocks: int,
                 ids: np.ndarray, items: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Routed projection: float64 y[rows*k, N]; rows of unplanned pairs stay as given (NaN by default)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    img = np.ascontiguousarray(img, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    items = np.ascontiguousarray(items, dtype=np.int32)
    rows, k = ids.shape
    y = np.full((rows * k, N), np.nan, dtype=np.float64) if out is None else out
    _load().or_proj_id_q8_1(WTYPE[wtype], _p(W), E, N, K, _p(img), row_blocks, _p(ids), k,
                            _p(items), items.size, _p(y))
    return y


def proj_id_slots_q8_1(wtype: str, W: np.ndarray, E: int, N: int, K: int, img: np.ndarray, row_blocks: int,
                       ids: np.ndarray, items: np.ndarray) -> np.ndarray:
    """Per-slot routed projection (the down projection of a routed FFN; llama.cpp
    PR #117, "GLU producer evidence" table, the per-slot routed components):
    pair p = row*k + slot reads image row p, its own GLU output, instead of the
    token's row. This is the routed projection of the flattened pairs, one slot
    per row, so it reuses proj_id_q8_1 with ids viewed as [rows*k][1]."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    return proj_id_q8_1(wtype, W, E, N, K, img, row_blocks, ids.reshape(-1, 1), items)


def moe_combine(expert_out: np.ndarray, wts: np.ndarray, live: int | None = None) -> np.ndarray:
    """Weighted combine closing the routed FFN (tf_moe_combine; TensorFold PR #1047,
    "What this changes": padding rows get no combine), in float64:
    y[r] = sum over slots s of wts[r, s] * expert_out[r*k + s], for the first
    `live` rows; the remaining rows are NaN (the caller's buffer is not written)."""
    wts = np.asarray(wts, dtype=np.float64)
    rows, k = wts.shape
    eo = np.asarray(expert_out, dtype=np.float64).reshape(rows, k, -1)
    live = rows if live is None else live
    y = np.full((rows, eo.shape[2]), np.nan, dtype=np.float64)
    y[:live] = np.einsum("rs,rsn->rn", wts[:live], eo[:live])
    return y


# ---------------------------------------------------------------- metrics
def nmse(a, ref) -> float:
    """Normalised mean squared error sum((a-ref)^2) / sum(ref^2)."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.sum(ref * ref))
    return float(np.sum((a - ref) ** 2)) / den if den > 0 else float(np.sum((a - ref) ** 2))
