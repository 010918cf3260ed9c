"""GPU parity: quantisers and producers against the oracle (via the C ABI).

Images are compared bit for bit. The producers' F32 outputs are compared with
the oracle's binary64 values within a tolerance derived from binary32
rounding; their images must equal, byte for byte, the oracle's quantisation
of the very F32 values the GPU stored, and the standalone GPU quantiser run on
those values (fused == unfused).
"""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.golden.golden import q8_hand_blocks
from tests.gpu_helpers import dev, empty_u8, host, live_ptr

pytestmark = pytest.mark.gpu


def gpu_quantize_q8_1(x: np.ndarray, K: int, row_blocks: int, live=None, fill=0xA5):
    T, stride = x.shape
    img = empty_u8(max(1, T * row_blocks * 36), fill)
    qk.qk_quantize_q8_1(dev(x), T, K, stride, img, row_blocks, live_ptr(live) if live is not None else None)
    return host(img)[:T * row_blocks * 36].reshape(T, row_blocks * 36)


@pytest.mark.parametrize("case", list(q8_hand_blocks()), ids=lambda c: c["name"])
def test_quantize_q8_1_hand_blocks(case):
    got = gpu_quantize_q8_1(case["x"], case["K"], case["row_blocks"])
    assert np.array_equal(got, O.quantize_q8_1(case["x"], K=case["K"], row_blocks=case["row_blocks"]))


@pytest.mark.parametrize("T,K,stride,rb", [(1, 256, 256, 8), (8, 3584, 3584, 112), (8, 3584, 3584, 128),
                                           (3, 200, 203, 10), (5, 33, 33, 2), (16, 2560, 2560, 80),
                                           (8, 18944, 18944, 592), (2, 1, 1, 1)])
def test_quantize_q8_1_matches_oracle(T, K, stride, rb):
    x = synth.activations(1000 + K, T, K, stride) * np.float32(2.5)
    if T > 2:
        x[1, : min(K, 64)] *= np.float32(1e-6)        # tiny blocks
        x[2, : min(K, 32)] = 0.0                      # zero block
    got = gpu_quantize_q8_1(x, K, rb)
    assert np.array_equal(got, O.quantize_q8_1(x, K=K, row_blocks=rb))


def test_quantize_and_glu_more_rows_than_a_grid_y_dimension():
    """70,000 rows (over the 65,535 limit of a grid's y dimension): rows run on grid x."""
    import torch
    T, K = 70000, 64
    x = synth.activations(1200, T, K)
    assert np.array_equal(gpu_quantize_q8_1(x, K, 2), O.quantize_q8_1(x))
    u = synth.activations(1201, T, K)
    out = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    img = empty_u8(T * 2 * 36)
    qk.qk_glu_q8_1("reglu", "separate", dev(x), K, dev(u), K, T, K, out, K, img, 2)
    og = host(out)
    assert np.array_equal(og, (np.maximum(x, 0.0) * u).astype(np.float32))   # one binary32 product each
    assert np.array_equal(host(img).reshape(T, -1), O.quantize_q8_1(og))


def test_quantize_q8_1_live_rows_untouched():
    T, K = 16, 256
    x = synth.poison_rows(synth.activations(1100, T, K), live=9)
    got = gpu_quantize_q8_1(x, K, 8, live=9)
    assert np.all(got[9:] == 0xA5)
    assert np.array_equal(got[:9], O.quantize_q8_1(x[:9]))
    got0 = gpu_quantize_q8_1(x, K, 8, live=0)
    assert np.all(got0 == 0xA5)


def test_quantize_q8_0_matches_oracle_prefill_size():
    """c4 size: [3325, 3584] ~N(0,1) -> split planes, all elements bit-exact."""
    import torch
    T, K = 3325, 3584
    x = synth.activations(4000, T, K)
    qs = torch.full((T * 112 * 32,), 0x5A, dtype=torch.uint8, device="cuda")
    d = torch.full((T * 112,), 0x5A5A, dtype=torch.int16, device="cuda")
    qk.qk_quantize_q8_0(dev(x), T, K, K, qs, d, 112)
    rq, rd = O.quantize_q8_0(x)
    assert np.array_equal(host(qs).view(np.int8).reshape(T, -1), rq)
    assert np.array_equal(host(d).view(np.uint16).reshape(T, -1), rd)


def test_quantize_q8_0_ragged_and_padding():
    import torch
    T, K, rb = 7, 100, 6
    x = synth.activations(4100, T, K, 101)
    qs = torch.full((T * rb * 32,), 0x5A, dtype=torch.uint8, device="cuda")
    d = torch.full((T * rb,), 0x5A5A, dtype=torch.int16, device="cuda")
    qk.qk_quantize_q8_0(dev(x), T, K, 101, qs, d, rb, live_ptr(5))
    rq, rd = O.quantize_q8_0(x, K=K, row_blocks=rb)
    gq = host(qs).view(np.int8).reshape(T, -1)
    gd = host(d).view(np.uint16).reshape(T, -1)
    assert np.array_equal(gq[:5], rq[:5]) and np.array_equal(gd[:5], rd[:5])
    assert np.all(gq[5:].view(np.uint8) == 0x5A) and np.all(gd[5:] == 0x5A5A)


# ------------------------------------------------------------------ producers
def _y_tolerance(y_ref: np.ndarray, b: np.ndarray | None) -> np.ndarray:
    # binary32 sum of squares (per-thread runs of K/1024 terms then a tree),
    # the sqrt and divide, and up to three rounded products and one add: about
    # 30 ulp of the larger of |y| and the product term before the bias add
    mag = np.abs(y_ref) + (np.abs(b) if b is not None else 0.0)
    return mag * 2e-6 + 1e-30


@pytest.mark.parametrize("kind", ["plain", "mul", "mul_add", "scale"])
@pytest.mark.parametrize("T,K,live", [(1, 256, None), (8, 3584, None), (16, 2560, 9), (128, 2560, 113)])
def test_rmsnorm_q8_1(kind, T, K, live):
    import torch
    x = synth.activations(2000 + K + T, T, K)
    if live is not None:
        x = synth.poison_rows(x, live)
    w = synth.norm_weight(2001, K)
    b = synth.activations(2002, 1, K)[0] * np.float32(0.1)
    rb = K // 32 + 3                                     # with row padding
    y = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    img = empty_u8(T * rb * 36)
    qk.qk_rmsnorm_q8_1(dev(x), T, K, K, kind, dev(w), dev(b), -0.75, 1e-6, y, K, img, rb,
                       live_ptr(live) if live is not None else None)
    n = T if live is None else live
    yg = host(y)
    ig = host(img).reshape(T, rb * 36)
    yref = O.rmsnorm(x[:n], kind, w=w, b=b, scale=-0.75, eps=1e-6)
    assert np.all(np.abs(yg[:n] - yref) <= _y_tolerance(yref, b if kind == 'mul_add' else None))
    # image of exactly the stored y: oracle quantiser and the GPU's own standalone quantiser
    assert np.array_equal(ig[:n], O.quantize_q8_1(yg[:n], row_blocks=rb))
    assert np.array_equal(ig[:n], gpu_quantize_q8_1(yg[:n], K, rb))
    # rows past live untouched
    assert np.all(np.isnan(yg[n:])) and np.all(ig[n:] == 0xA5)
    # the oracle's own image of its own y differs only in blocks whose y differ
    io = O.quantize_q8_1(yref.astype(np.float32), row_blocks=rb).reshape(n, rb, 36)
    same_y = (yref.astype(np.float32).reshape(n, -1, 32) == yg[:n].reshape(n, -1, 32)).all(axis=2)
    blocks_equal = (io[:, :K // 32] == ig[:n].reshape(n, rb, 36)[:, :K // 32]).all(axis=2)
    assert np.all(blocks_equal[same_y])


@pytest.mark.parametrize("kind", ["swiglu", "geglu_tanh", "reglu", "geglu_erf", "geglu_quick", "swiglu_oai",
                                  "swiglu_clamp"])
@pytest.mark.parametrize("layout", ["separate", "packed", "packed_swapped"])
@pytest.mark.parametrize("T,N", [(8, 18944), (3, 96)])
def test_glu_q8_1(kind, layout, T, N):
    import torch
    g = synth.activations(3000 + N, T, N) * np.float32(2.0)
    u = synth.activations(3001 + N, T, N)
    if layout == "separate":
        a = np.zeros((T, N + 32), dtype=np.float32)      # independent row strides
        b = np.zeros((T, N + 64), dtype=np.float32)
        a[:, :N], b[:, :N] = g, u
        a_d, b_d, a_stride, b_stride = dev(a), dev(b), N + 32, N + 64
        ref = O.glu(kind, layout, a, b, N)
    else:
        a = np.concatenate([g, u] if layout == "packed" else [u, g], axis=1)
        a_d, b_d, a_stride, b_stride = dev(a), None, 2 * N, 0
        ref = O.glu(kind, layout, a, None, N)
    rb = N // 32
    out = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    img = empty_u8(T * rb * 36)
    qk.qk_glu_q8_1(kind, layout, a_d, a_stride, b_d, b_stride, T, N, out, N, img, rb)
    og = host(out)
    ig = host(img).reshape(T, rb * 36)
    # a few ulp of binary32 expf/tanhf and products; 1 + tanh(z) cancels for
    # very negative z, so allow a few ulp of |g u| as an absolute term too
    # (SwiGLU-OAI: the rounding of v + 1 gives an absolute term in |g| (|u| + 1))
    uterm = np.abs(u) + 1.0 if kind == "swiglu_oai" else np.abs(u)
    tol = np.abs(ref) * 2e-6 + 3e-7 * np.abs(g.astype(np.float64)) * uterm + 1e-30
    assert np.all(np.abs(og - ref) <= tol)
    assert np.array_equal(ig, O.quantize_q8_1(og, row_blocks=rb))
    assert np.array_equal(ig, gpu_quantize_q8_1(og, N, rb))


@pytest.mark.parametrize("alpha,limit", [(1.0, 1.5), (2.5, 0.75), (1.702, 7.0)])
def test_glu_swiglu_oai_parameters(alpha, limit):
    """qk_glu_q8_1_ex passes alpha and limit through; both clamps are hit at these limits."""
    import torch
    T, N = 5, 320
    g = synth.activations(3200, T, N) * np.float32(3.0)
    u = synth.activations(3201, T, N) * np.float32(3.0)
    ref = O.glu("swiglu_oai", "separate", g, u, N, alpha=alpha, limit=limit)
    out = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    img = empty_u8(T * (N // 32) * 36)
    qk.qk_glu_q8_1_ex("swiglu_oai", "separate", dev(g), N, dev(u), N, T, N, out, N, img, N // 32,
                      alpha=alpha, limit=limit)
    og, ig = host(out), host(img).reshape(T, -1)
    tol = np.abs(ref) * 2e-6 + 3e-7 * np.abs(g.astype(np.float64)) * (np.abs(u) + 1.0) + 1e-30
    assert np.all(np.abs(og - ref) <= tol)
    assert np.array_equal(ig, O.quantize_q8_1(og, row_blocks=N // 32))
    assert np.sum(g > limit) > 0 and np.sum(np.abs(u) > limit) > 0


def test_glu_live_rows():
    import torch
    T, N, live = 16, 256, 9
    g = synth.poison_rows(synth.activations(3100, T, N), live)
    u = synth.activations(3101, T, N)
    out = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    img = empty_u8(T * 8 * 36)
    qk.qk_glu_q8_1("swiglu", "separate", dev(g), N, dev(u), N, T, N, out, N, img, 8, live_ptr(live))
    og, ig = host(out), host(img).reshape(T, -1)
    assert np.all(np.isnan(og[live:])) and np.all(ig[live:] == 0xA5)
    assert np.array_equal(ig[:live], O.quantize_q8_1(og[:live]))


@pytest.mark.parametrize("kind", ["mul", "plain", "mul_add", "scale"])
@pytest.mark.parametrize("T,K,live", [(5, 3584, None), (3325, 3584, None), (9, 256, 6), (2, 12288, None)])
def test_rmsnorm_q8_0_planes(kind, T, K, live):
    """The fused RMS -> Q8_0 producer (prefill): the planes are bit-exact to the oracle's Q8_0
    quantiser applied to the GPU's own stored y, and y matches the oracle RMS within tolerance."""
    import torch
    if T > 64 and kind != "mul":
        pytest.skip("the full prefill size runs once, with the config's MUL kind")
    x = synth.activations(2100 + K + T, T, K)
    if live is not None:
        x = synth.poison_rows(x, live)
    w = synth.norm_weight(2101, K)
    b = synth.activations(2102, 1, K)[0] * np.float32(0.1)
    rb = K // 32 + 2                                     # with row padding
    y = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    qs = torch.full((T * rb * 32,), 0x5A, dtype=torch.int8, device="cuda")
    d = torch.full((T * rb,), 0x5A5A, dtype=torch.int16, device="cuda")
    qk.qk_rmsnorm_q8_0(dev(x), T, K, K, kind, dev(w), dev(b), 0.5, 1e-6, y, K, qs, d, rb,
                       live_ptr(live) if live is not None else None)
    n = T if live is None else live
    yg = host(y)
    qg = host(qs).reshape(T, rb * 32)
    dg = host(d).view(np.uint16).reshape(T, rb)
    rows = np.arange(n) if n <= 64 else np.random.default_rng(5).choice(n, 64, replace=False)
    yref = O.rmsnorm(x[rows], kind, w=w, b=b, scale=0.5, eps=1e-6)
    assert np.all(np.abs(yg[rows] - yref) <= _y_tolerance(yref, b if kind == 'mul_add' else None))
    q_o, d_o = O.quantize_q8_0(yg[:n], row_blocks=rb)
    assert np.array_equal(qg[:n], q_o) and np.array_equal(dg[:n], d_o)
    assert np.all(np.isnan(yg[n:])) and np.all(qg[n:] == 0x5A) and np.all(dg[n:] == 0x5A5A)


@pytest.mark.parametrize("K", [3584, 8192, 256])
@pytest.mark.parametrize("q81", [True, False])
def test_rmsnorm_bits_do_not_depend_on_the_row_count(K, q81):
    """Many rows run in 256-thread CTAs that reduce in the 1024-thread order: the first rows of a
    300-row call equal an 8-row call byte for byte (F32 output and image)."""
    import torch
    T_big, T_small, rb = 300, 8, K // 32
    x = synth.activations(5100 + K, T_big, K)
    w = dev(synth.norm_weight(5101, K))

    def run(T):
        y = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
        xd = dev(x[:T])
        if q81:
            img = empty_u8(T * rb * 36)
            qk.qk_rmsnorm_q8_1(xd, T, K, K, "mul", w, None, 1.0, 1e-6, y, K, img, rb)
            return host(y), host(img).reshape(T, -1)
        qs = torch.zeros((T * rb * 32,), dtype=torch.int8, device="cuda")
        d = torch.zeros((T * rb,), dtype=torch.int16, device="cuda")
        qk.qk_rmsnorm_q8_0(xd, T, K, K, "mul", w, None, 1.0, 1e-6, y, K, qs, d, rb)
        return host(y), np.concatenate([host(qs).reshape(T, -1).view(np.uint8), host(d).reshape(T, -1).view(np.uint8)], 1)

    yb, ib = run(T_big)
    ys, is_ = run(T_small)
    assert np.array_equal(yb[:T_small].view(np.uint32), ys.view(np.uint32))
    assert np.array_equal(ib[:T_small], is_)
    ref = O.rmsnorm(x, "mul", w=synth.norm_weight(5101, K), eps=1e-6)
    assert np.all(np.abs(yb - ref) <= _y_tolerance(ref, None))
