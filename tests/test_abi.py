"""The C ABI library loads, exports every declared entry point, and rejects bad
calls on the host before anything is launched (no GPU needed: the pointers
below are never dereferenced)."""
import ctypes as C

import pytest

from quantized_activation_q4_gb300 import binding as qk


@pytest.fixture(scope="module")
def lib():
    return qk.load()


def test_exports_every_declared_symbol(lib):
    names = qk.declared_symbols()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []


def test_status_strings(lib):
    assert lib.qk_status_string(0) == b"QK_OK"
    assert lib.qk_status_string(3) == b"QK_ERR_ALIAS"


X = 0x10000000       # fake, never-dereferenced device addresses
IMG = 0x20000000
Y = 0x30000000
W = 0x40000000
S0 = 0               # null stream: never used by a call that fails validation


def _st(fn, *args):
    return fn(*args)


def test_quantize_rejects_bad_shapes(lib):
    P = C.c_void_p
    assert lib.qk_quantize_q8_1(P(X), 2, 33, 32, P(IMG), 2, None, None) == 2       # x_stride < K
    assert lib.qk_quantize_q8_1(P(X), 2, 33, 40, P(IMG), 1, None, None) == 2       # too few image blocks
    assert lib.qk_quantize_q8_1(None, 2, 32, 32, P(IMG), 1, None, None) == 1       # null x
    assert lib.qk_quantize_q8_1(P(X), 2, 0, 32, P(IMG), 1, None, None) == 1        # K < 1
    assert lib.qk_quantize_q8_1(P(X + 2), 2, 32, 32, P(IMG), 1, None, None) == 1   # misaligned x
    # image overlapping the input rows
    assert lib.qk_quantize_q8_1(P(X), 4, 64, 64, P(X + 512), 2, None, None) == 3
    assert b"overlaps" in lib.qk_last_error()


def test_producers_reject_partial_blocks_and_aliases(lib):
    P = C.c_void_p
    # K not a whole number of 32-blocks
    assert lib.qk_rmsnorm_q8_1(P(X), 1, 48, 48, 0, None, None, 1.0, 1e-6, P(Y), 48, P(IMG), 2, None, None) == 2
    # MUL without w
    assert lib.qk_rmsnorm_q8_1(P(X), 1, 64, 64, 1, None, None, 1.0, 1e-6, P(Y), 64, P(IMG), 2, None, None) == 1
    # y written over x
    assert lib.qk_rmsnorm_q8_1(P(X), 1, 64, 64, 0, None, None, 1.0, 1e-6, P(X), 64, P(IMG), 2, None, None) == 3
    # GLU: N not whole blocks; bad layout; out over the packed input
    assert lib.qk_glu_q8_1(0, 0, P(X), 40, P(W), 40, 1, 40, P(Y), 40, P(IMG), 2, None, None) == 2
    assert lib.qk_glu_q8_1(0, 7, P(X), 64, P(W), 64, 1, 32, P(Y), 32, P(IMG), 1, None, None) == 1
    assert lib.qk_glu_q8_1(0, 1, P(X), 128, None, 0, 1, 64, P(X + 64), 64, P(IMG), 2, None, None) == 3


def test_projection_checks(lib):
    P = C.c_void_p
    WS = 0x50000000
    good = qk.qk_proj(0, 0, W, 64, 256, Y, 64)
    arr = (qk.qk_proj * 1)(good)
    assert lib.qk_mmvq(P(IMG), 8, 9, 1, arr, None, P(WS), 1 << 20, None) == 5       # T > 8
    arr = (qk.qk_proj * 1)(qk.qk_proj(0, 0, W, 64, 288, Y, 64))
    assert lib.qk_mmvq(P(IMG), 8, 8, 1, arr, None, P(WS), 1 << 20, None) == 2       # K past the image row
    arr = (qk.qk_proj * 1)(qk.qk_proj(0, 0, W + 8, 64, 256, Y, 64))
    assert lib.qk_mmvq(P(IMG), 8, 8, 1, arr, None, P(WS), 1 << 20, None) == 1       # misaligned weights
    arr = (qk.qk_proj * 2)(good, qk.qk_proj(0, 0, W, 64, 256, Y + 128, 64))
    assert lib.qk_mmvq(P(IMG), 8, 8, 2, arr, None, P(WS), 1 << 20, None) == 3       # overlapping outputs
    # column windows of one fused [T][64 + 32] output buffer: accepted (then the tiny workspace is refused)
    fused = (qk.qk_proj * 2)(qk.qk_proj(0, 0, W, 64, 256, Y, 96), qk.qk_proj(0, 0, W, 32, 256, Y + 256, 96))
    assert lib.qk_mmvq(P(IMG), 8, 8, 2, fused, None, P(WS), 16, None) == 4
    # windows that share a column, or rows that wrap into the next row's window: refused
    clash = (qk.qk_proj * 2)(qk.qk_proj(0, 0, W, 64, 256, Y, 96), qk.qk_proj(0, 0, W, 32, 256, Y + 252, 96))
    assert lib.qk_mmvq(P(IMG), 8, 8, 2, clash, None, P(WS), 16, None) == 3
    wrap = (qk.qk_proj * 2)(qk.qk_proj(0, 0, W, 64, 256, Y, 96), qk.qk_proj(0, 0, W, 64, 256, Y + 256, 96))
    assert lib.qk_mmvq(P(IMG), 8, 8, 2, wrap, None, P(WS), 16, None) == 3
    arr = (qk.qk_proj * 1)(qk.qk_proj(0, 0, W, 64, 256, IMG + 4, 64))
    assert lib.qk_mmvq(P(IMG), 8, 8, 1, arr, None, P(WS), 1 << 20, None) == 3       # output over the image
    arr = (qk.qk_proj * 1)(good)
    assert lib.qk_mmvq(P(IMG), 8, 8, 1, arr, None, None, 0, None) == 4              # no workspace
    assert lib.qk_mmvq(P(IMG), 8, 8, 1, arr, None, P(WS), 16, None) == 4            # workspace too small
    assert lib.qk_mmvq(P(IMG), 8, 8, 1, arr, None, P(Y), 1 << 20, None) == 3        # workspace over y


def test_static_workspace_checks_everything_before_touching_the_device(lib):
    """qk_mmvq_static_ws runs every argument check of qk_mmvq before it looks up its
    scratch array or enqueues its counter clear. On a machine without a GPU any CUDA
    call would report QK_ERR_CUDA (6), so the codes below come from the checks alone."""
    P = C.c_void_p
    good = qk.qk_proj(0, 0, W, 64, 256, Y, 64)
    arr = (qk.qk_proj * 1)(good)
    assert lib.qk_mmvq_static_ws(P(IMG), 8, 9, 1, arr, None, None) == 5           # T > 8
    arr = (qk.qk_proj * 1)(qk.qk_proj(0, 0, W, -5, 256, Y, 64))
    assert lib.qk_mmvq_static_ws(P(IMG), 8, 8, 1, arr, None, None) == 1           # N < 0
    arr = (qk.qk_proj * 1)(qk.qk_proj(7, 0, W, 64, 256, Y, 64))
    assert lib.qk_mmvq_static_ws(P(IMG), 8, 8, 1, arr, None, None) == 1           # bad weight type
    arr = (qk.qk_proj * 2)(good, qk.qk_proj(0, 0, W, 64, 256, Y + 128, 64))
    assert lib.qk_mmvq_static_ws(P(IMG), 8, 8, 2, arr, None, None) == 3           # overlapping outputs
    arr = (qk.qk_proj * 1)(qk.qk_proj(0, 0, W, 64, 288, Y, 64))
    assert lib.qk_mmvq_static_ws(P(IMG), 8, 8, 1, arr, None, None) == 2           # K past the image row


def test_routing_checks(lib):
    P = C.c_void_p
    assert lib.qk_topk_route(P(X), 16, 512, 8, P(Y), P(W), None, None) == 5    # E > 256
    assert lib.qk_topk_route(P(X), 16, 128, 8, P(X), P(W), None, None) == 3    # ids over logits
    assert lib.qk_moe_plan(P(X), 16, 8, 2048, P(Y), P(W), P(IMG), None, None) == 5
    assert lib.qk_moe_plan(P(X), 16, 8, 128, P(Y), P(Y + 16), P(IMG), None, None) == 3


def test_weight_pack_checks(lib):
    P = C.c_void_p
    need = lib.qk_weight_packed_bytes(0, 100, 256)
    assert need == 1 * 2 * 9216                                                  # 128-row x 128-col units
    assert lib.qk_weight_packed_bytes(1, 300, 300) == 3 * 3 * 17408
    assert lib.qk_weight_pack(0, P(X), 100, 256, P(W), need - 1, None) == 4
    assert lib.qk_weight_pack(0, P(X), 100, 250, P(W), need, None) == 2
    assert lib.qk_weight_pack(0, P(X), 100, 256, P(X + 64), need, None) == 3


def test_routed_ffn_checks(lib):
    """Argument refusals of the per-slot projection and the combine (host checks only: no launch)."""
    P = C.c_void_p
    # combine: N not a multiple of 4, stride < N, misaligned y, y over expert_out, N too large, k out of range
    assert lib.qk_moe_combine(P(X), 64, P(W), 4, 2, 62, P(Y), 64, None, None) == 1
    assert lib.qk_moe_combine(P(X), 60, P(W), 4, 2, 64, P(Y), 64, None, None) == 2
    assert lib.qk_moe_combine(P(X), 64, P(W), 4, 2, 64, P(Y + 4), 64, None, None) == 1
    assert lib.qk_moe_combine(P(X), 64, P(W), 4, 2, 64, P(X + 256), 64, None, None) == 3
    assert lib.qk_moe_combine(P(X), 1 << 26, P(W), 1, 1, 1 << 26, P(Y), 1 << 26, None, None) == 1
    assert lib.qk_moe_combine(P(X), 64, P(W), 4, 0, 64, P(Y), 64, None, None) == 1
    # per-slot projection: the image has rows * k rows, so an output placed after rows image rows
    # overlaps it (the per-token call would not see an overlap there)
    rows, k, rb = 2, 4, 8
    y_in_img = IMG + rows * rb * 36
    arr = (qk.qk_proj_id * 1)(qk.qk_proj_id(0, 4, W, 128, 256, y_in_img))
    assert lib.qk_mmvq_id_slots(P(IMG), rb, rows, k, 1, arr, P(X), P(X + 64), P(X + 128), None) == 3
    arr9 = (qk.qk_proj_id * 9)(*[qk.qk_proj_id(0, 4, W, 128, 256, Y + i * (1 << 20)) for i in range(9)])
    assert lib.qk_mmvq_id_slots(P(IMG), rb, rows, k, 9, arr9, P(X), P(X + 64), P(X + 128), None) == 5
    assert lib.qk_mmvq_id_slots(P(IMG), rb, rows, 65, 1, arr, P(X), P(X + 64), P(X + 128), None) == 1
    # an output may not overlap the plan it is read from (counts, offsets or items)
    ok = (qk.qk_proj_id * 1)(qk.qk_proj_id(0, 4, W, 128, 256, Y))
    for counts, offsets, items in ((Y + 64, X, X + 64), (X, Y + 4000, X + 64), (X, X + 64, Y + 8)):
        for fn in (lib.qk_mmvq_id, lib.qk_mmvq_id_slots):
            assert fn(P(IMG), rb, rows, k, 1, ok, P(counts), P(offsets), P(items), None) == 3


def test_grid_limits_are_refused(lib):
    """Row-block and width limits that keep every grid dimension in range."""
    P = C.c_void_p
    assert lib.qk_quantize_q8_1(P(X), 1, 32, 32, P(IMG), (1 << 20) + 1, None, None) == 1
    assert lib.qk_quantize_q8_1(P(X), 1, (1 << 25) + 32, (1 << 25) + 32, P(IMG), 1 << 20, None, None) == 1
    assert lib.qk_glu_q8_1(0, 0, P(X), 1 << 26, P(W), 1 << 26, 1, 1 << 26, P(Y), 1 << 26, P(IMG), 1 << 21,
                           None, None) == 1


def test_glu_parameter_checks(lib):
    """qk_glu_q8_1_ex refuses a non-finite alpha and a limit that is not positive and finite,
    and unknown kinds (host checks only: no launch)."""
    P = C.c_void_p
    inf, nan = float("inf"), float("nan")
    args = (P(X), 64, P(W), 64, 2, 64, P(Y), 64, P(IMG), 2)
    assert lib.qk_glu_q8_1_ex(5, 0, *args, 1.702, 0.0, None, None) == 1
    assert lib.qk_glu_q8_1_ex(5, 0, *args, 1.702, -1.0, None, None) == 1
    assert lib.qk_glu_q8_1_ex(5, 0, *args, 1.702, inf, None, None) == 1
    assert lib.qk_glu_q8_1_ex(5, 0, *args, nan, 7.0, None, None) == 1
    assert lib.qk_glu_q8_1_ex(7, 0, *args, 1.702, 7.0, None, None) == 1
    assert lib.qk_glu_q8_1(7, 0, *args, None, None) == 1
    assert lib.qk_glu_q8_1_ex(6, 0, *args, 1.702, -1.0, None, None) == 1    # SwiGLU-clamp reads limit too


def _memo_match(lib, m, fmt=1, x=X, T=8, K=256, xs=256, d0=IMG, d1=Y, rb=8, s=None):
    P = C.c_void_p
    return lib.qk_image_memo_match(C.byref(m), fmt, P(x), T, K, xs, P(d0), P(d1) if d1 else None, rb,
                                   P(s) if s else None)


def _memo_fill(m):
    """The key a successful Q8_0 quantise of X into (IMG, Y) on the null stream records."""
    m.format, m.x, m.T, m.K, m.x_stride, m.row_blocks, m.dst0, m.dst1, m.stream = 1, X, 8, 256, 256, 8, IMG, Y, None


def test_image_memo_hits_only_on_the_whole_key(lib):
    """minfer doc 52 r49, section 3.1: the key is (source pointer, shape) plus the destination
    pointers (the physical-pointer check) and the image form; any differing field is a miss."""
    m = qk.qk_image_memo()
    assert _memo_match(lib, m) == 0                      # empty
    _memo_fill(m)
    assert _memo_match(lib, m) == 1
    for field, other in [("fmt", 2), ("x", X + 4096), ("T", 7), ("K", 224), ("xs", 320), ("d0", IMG + 4096),
                         ("d1", Y + 4096), ("rb", 9), ("s", 0x1234)]:
        assert _memo_match(lib, m, **{field: other}) == 0, field
    lib.qk_image_memo_clear(C.byref(m))
    assert m.format == 0 and _memo_match(lib, m) == 0


def test_image_memo_hit_enqueues_nothing_and_errors_clear_it(lib):
    P = C.c_void_p
    m = qk.qk_image_memo()
    _memo_fill(m)
    hit = C.c_int32(-1)
    n0 = lib.qk_launch_count()
    # a hit returns at once (no device is touched, nothing is launched)
    assert lib.qk_image_memo_quantize_q8_0(C.byref(m), P(X), 8, 256, 256, P(IMG), P(Y), 8, C.byref(hit), None) == 0
    assert hit.value == 1 and lib.qk_launch_count() == n0 and m.format == 1
    # a Q8_1 request never takes a Q8_0 record
    assert lib.qk_image_memo_match(C.byref(m), 2, P(X), 8, 256, 256, P(IMG), None, 8, None) == 0
    # a null hit pointer is refused and clears the memo
    assert lib.qk_image_memo_quantize_q8_0(C.byref(m), P(X), 8, 256, 256, P(IMG), P(Y), 8, None, None) == 1
    assert m.format == 0
    # a miss that fails the quantiser's checks (x_stride < K) reports its error, hit = 0, memo cleared
    _memo_fill(m)
    assert lib.qk_image_memo_quantize_q8_0(C.byref(m), P(X), 8, 256, 128, P(IMG), P(Y), 8, C.byref(hit), None) == 2
    assert hit.value == 0 and m.format == 0
    # a null memo
    assert lib.qk_image_memo_quantize_q8_1(None, P(X), 8, 256, 256, P(IMG), 8, C.byref(hit), None) == 1
