"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute: hand-worked
blocks, an independent library routine (numpy / Python struct binary16
conversion, numpy matmul, numpy argsort, scipy softmax/erf), closed forms,
invariants or brute force. Each is chosen so that a plausible slip in the
oracle (a dropped term, wrong sign, swapped field, wrong rounding, transposed
operand, wrong nibble order) fails at least one of them.
"""
import struct

import numpy as np
import pytest
import scipy.special as sp

from oracle import oracle as O
from quantized_activation_q4_gb300 import synth
from tests.golden.golden import block_bytes, q8_hand_blocks


# ----------------------------------------------------------------- binary16
def _all_f32_chunk(i, n):
    return np.arange(i, i + n, dtype=np.uint64).astype(np.uint32).view(np.float32)


def test_f16_conversion_exhaustive_vs_torch():
    """Every binary32 pattern converts like torch's CPU binary16 cast (RNE, subnormals, overflow)."""
    import torch
    step = 1 << 26
    bad = 0
    for i in range(0, 1 << 32, step):
        x = _all_f32_chunk(i, step)
        ours = O.f32_to_f16_bits(x)
        ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(x)
        bad += int(np.count_nonzero((ours != ref) & ~nan))
        # NaN stays NaN with its sign
        on = ours[nan]
        assert np.all((on & 0x7C00) == 0x7C00) and np.all((on & 0x3FF) != 0)
        assert np.array_equal(on >> 15, (x[nan].view(np.uint32) >> 31).astype(np.uint16))
    assert bad == 0


def test_f16_conversion_rounding_points_vs_numpy():
    """Every sign, exponent and top-10 significand pattern, with the low 13 bits at and around
    each rounding point, against numpy's binary16 cast (a second independent routine)."""
    low = {0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x0800, 0x17FF, 0x1800}
    base = (np.arange(1 << 19, dtype=np.uint64) << np.uint64(13)).astype(np.uint32)  # sign|exp|top10
    x = np.concatenate([(base | np.uint32(v)) for v in sorted(low)]).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    ours = O.f32_to_f16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("v", [0.0, -0.0, 1.0, 1.0 / 3.0, 65504.0, 65519.99, 65520.0, 6.1e-5,
                               5.96e-8, 2.98e-8, 2.99e-8, 1e-10, -2.5e-6, 1234.5678, 0.1])
def test_f16_conversion_vs_python_struct(v):
    """Spot values against Python's own binary16 packer (a second independent routine)."""
    x = np.float32(v)
    try:
        ref = struct.unpack("<H", struct.pack("<e", float(x)))[0]
    except OverflowError:
        ref = 0x7C00 if x > 0 else 0xFC00
    assert int(O.f32_to_f16_bits(np.array([x]))[0]) == ref


def test_f16_to_f32_roundtrip_all_halves():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    finite = ~np.isnan(ref)
    assert np.array_equal(f[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.all(np.isnan(f[~finite]))


# ----------------------------------------------------------------- Q8 blocks
@pytest.mark.parametrize("case", list(q8_hand_blocks()), ids=lambda c: c["name"])
def test_q8_1_hand_blocks(case):
    img = O.quantize_q8_1(case["x"], K=case["K"], row_blocks=case["row_blocks"])
    for b, (d, s, q) in case["blocks"].items():
        got = bytes(img[0, b * 36:(b + 1) * 36])
        assert got == block_bytes(d, s, q), f"block {b}"


@pytest.mark.parametrize("case", list(q8_hand_blocks()), ids=lambda c: c["name"])
def test_q8_0_hand_blocks(case):
    qs, dh = O.quantize_q8_0(case["x"], K=case["K"], row_blocks=case["row_blocks"])
    for b, (d, s, q) in case["blocks"].items():
        assert int(dh[0, b]) == d
        assert np.array_equal(qs[0, b * 32:(b + 1) * 32], q)


def _decode_q8_1(img, T, rb):
    blk = img.reshape(T, rb, 36)
    d = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    s = blk[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    q = blk[:, :, 4:].view(np.int8).astype(np.int64)
    return d, s, q


def test_q8_1_roundtrip_and_amax_invariants():
    """|x - d_h q| <= d (1/2 + 2^-17) + 127 |d - d_h|; the amax element has |q| = 127 and x's sign."""
    T, K = 16, 1024
    x = synth.activations(11, T, K) * np.float32(3.0)
    x[3, 64:96] *= np.float32(1e-3)          # small-magnitude blocks
    x[4, 96:128] = 0.0                        # an all-zero block
    img = O.quantize_q8_1(x)
    d_h, s_h, q = _decode_q8_1(img, T, K // 32)
    xb = x.reshape(T, K // 32, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    d = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    err = np.abs(xb - d_h[..., None] * q)
    bound = d * (0.5 + 2.0 ** -17) + 127 * np.abs(d - d_h)
    assert np.all(err <= bound[..., None] * (1 + 1e-12) + 1e-300)
    arg = np.abs(xb).argmax(axis=2)
    qa = np.take_along_axis(q, arg[..., None], 2)[..., 0]
    xa = np.take_along_axis(xb, arg[..., None], 2)[..., 0]
    nz = amax > 0
    assert np.all(np.abs(qa[nz]) == 127) and np.all(np.sign(qa[nz]) == np.sign(xa[nz]))
    assert np.all(q[~nz] == 0) and np.all(d_h[~nz] == 0) and np.all(s_h[~nz] == 0)
    # s holds d * sum(q) to half precision
    S = q.sum(axis=2)
    assert np.all(np.abs(s_h - d * S) <= np.abs(d * S) * 2.0 ** -11 + 2.0 ** -25)


def test_q8_0_matches_q8_1_codes_and_scales():
    """The Q8_0 planes carry the same d and codes as the Q8_1 image (only s is absent)."""
    x = synth.activations(12, 5, 200)
    img = O.quantize_q8_1(x, row_blocks=8)
    qs, dh = O.quantize_q8_0(x, row_blocks=8)
    blk = img.reshape(5, 8, 36)
    assert np.array_equal(blk[:, :, 0:2].copy().view(np.uint16)[..., 0], dh)
    assert np.array_equal(blk[:, :, 4:].reshape(5, 256).view(np.int8), qs)


def test_quantize_leaves_rows_past_live_untouched():
    x = synth.poison_rows(synth.activations(13, 8, 64), live=3)
    sentinel = np.full((8, 2 * 36), 0xA5, dtype=np.uint8)
    img = O.quantize_q8_1(x, live=3, out=sentinel.copy())
    assert np.all(img[3:] == 0xA5)
    assert np.array_equal(img[:3], O.quantize_q8_1(x[:3]))


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_forms():
    K = 256
    c = np.float32(0.75)
    x = np.full((1, K), c, dtype=np.float32)
    y = O.rmsnorm(x, eps=1e-6)
    assert np.allclose(y, 0.75 / np.sqrt(0.75 ** 2 + 1e-6), rtol=1e-15, atol=0)
    onehot = np.zeros((1, K), dtype=np.float32)
    onehot[0, 7] = 2.0
    y = O.rmsnorm(onehot, eps=1e-6)
    assert y[0, 7] == pytest.approx(2.0 / np.sqrt(4.0 / K + 1e-6), rel=1e-15)
    assert np.count_nonzero(y) == 1


def test_rmsnorm_invariants_and_variants():
    T, K = 4, 384
    x = synth.activations(21, T, K)
    w = synth.norm_weight(22, K)
    b = synth.activations(23, 1, K)[0]
    y0 = O.rmsnorm(x, eps=0.0)
    assert np.allclose((y0 ** 2).mean(axis=1), 1.0, rtol=1e-13)
    assert np.array_equal(O.rmsnorm(x * np.float32(4.0), eps=0.0), y0)     # scale invariance (power of two)
    ones = np.ones(K, dtype=np.float32)
    zeros = np.zeros(K, dtype=np.float32)
    yp = O.rmsnorm(x, "plain")
    assert np.array_equal(O.rmsnorm(x, "mul", w=ones), yp)
    assert np.array_equal(O.rmsnorm(x, "mul_add", w=w, b=zeros), O.rmsnorm(x, "mul", w=w))
    assert np.array_equal(O.rmsnorm(x, "mul_add", w=zeros, b=b), np.broadcast_to(b.astype(np.float64), (T, K)))
    assert np.array_equal(O.rmsnorm(x, "scale", scale=1.0), yp)
    assert np.allclose(O.rmsnorm(x, "scale", scale=-0.5), -0.5 * yp, rtol=1e-15)


# ----------------------------------------------------------------- GLU
def test_glu_against_library_functions():
    T, N = 3, 512
    g = synth.activations(31, T, N) * np.float32(3.0)
    u = synth.activations(32, T, N)
    g64, u64 = g.astype(np.float64), u.astype(np.float64)
    assert np.allclose(O.glu("swiglu", "separate", g, u, N), g64 * sp.expit(g64) * u64, rtol=1e-13, atol=1e-300)
    assert np.array_equal(O.glu("reglu", "separate", g, u, N), np.maximum(g64, 0.0) * u64)
    gelu_erf = 0.5 * g64 * (1.0 + sp.erf(g64 / np.sqrt(2.0)))
    gt = O.glu("geglu_tanh", "separate", g, np.ones_like(u), N)
    # the tanh form tracks the erf GELU to better than 1e-3 absolute everywhere
    # (dropping the cubic term or the sqrt(2/pi) factor breaks this by > 1e-2)
    assert np.max(np.abs(gt - gelu_erf)) < 1e-3
    # odd-part identity of the tanh form: gelu(g) - gelu(-g) = g
    gm = O.glu("geglu_tanh", "separate", -g, np.ones_like(u), N)
    assert np.allclose(gt - gm, g64, rtol=1e-13, atol=1e-13)


def test_geglu_tanh_against_torch_tanh_gelu():
    """GeGLU-tanh against torch's tanh-approximated GELU in float64 (a library routine
    with the published constants sqrt(2/pi) and 0.044715): a truncated constant
    (0.0447, 0.7978) moves the result by more than 1e-6 at |g| ~ 2..3, far past 1e-13."""
    import torch
    T, N = 4, 1024
    g = synth.activations(33, T, N) * np.float32(3.0)
    u = synth.activations(34, T, N)
    g64 = torch.from_numpy(g.astype(np.float64))
    ref = (torch.nn.functional.gelu(g64, approximate="tanh") * torch.from_numpy(u.astype(np.float64))).numpy()
    got = O.glu("geglu_tanh", "separate", g, u, N)
    assert np.max(np.abs(got - ref)) <= 1e-13 * max(1.0, float(np.max(np.abs(ref))))
    # the same through the packed layouts (the half order of the two layouts)
    gu = np.concatenate([g, u], axis=1)
    ug = np.concatenate([u, g], axis=1)
    assert np.array_equal(O.glu("geglu_tanh", "packed", gu, None, N), got)
    assert np.array_equal(O.glu("geglu_tanh", "packed_swapped", ug, None, N), got)


def test_glu_gelu_variants_against_library_and_identities():
    """GeGLU-erf against torch's exact GELU; GeGLU-quick within the sigmoid approximation's
    known distance of it (a wrong constant, e.g. SiLU's 1.0, misses by > 0.1); both odd parts
    equal g."""
    import torch
    T, N = 3, 512
    g = synth.activations(33, T, N) * np.float32(3.0)
    g64 = g.astype(np.float64)
    ones = np.ones_like(g)
    ge = O.glu("geglu_erf", "separate", g, ones, N)
    ref = torch.nn.functional.gelu(torch.from_numpy(g64), approximate="none").numpy()
    assert np.allclose(ge, ref, rtol=1e-13, atol=1e-15)
    gq = O.glu("geglu_quick", "separate", g, ones, N)
    assert np.max(np.abs(gq - ref)) < 0.021
    for kind in ("geglu_erf", "geglu_quick"):
        pos = O.glu(kind, "separate", g, ones, N)
        neg = O.glu(kind, "separate", -g, ones, N)
        assert np.allclose(pos - neg, g64, rtol=1e-13, atol=1e-13)
    u = synth.activations(34, T, N)
    assert np.allclose(O.glu("geglu_erf", "separate", g, u, N), ge * u.astype(np.float64), rtol=1e-15, atol=0)


def test_glu_swiglu_oai_reductions_and_clamps():
    """SwiGLU-OAI inside its clamp range equals SwiGLU (alpha = 1) or GeGLU-quick (alpha = 1.702)
    times (u + 1); past the limits it is constant in g (from above) and in u (both ways);
    u = -1 gives 0."""
    T, N = 2, 256
    g = np.clip(synth.activations(35, T, N) * np.float32(2.0), -6.5, 6.5).astype(np.float32)
    u = np.clip(synth.activations(36, T, N), -6.5, 6.5).astype(np.float32)
    up1 = u.astype(np.float64) + 1.0
    ones = np.ones_like(u)
    oai1 = O.glu("swiglu_oai", "separate", g, u, N, alpha=1.0, limit=7.0)
    assert np.allclose(oai1, O.glu("swiglu", "separate", g, ones, N) * up1, rtol=1e-13, atol=1e-300)
    oai = O.glu("swiglu_oai", "separate", g, u, N)
    # alpha arrives as the binary32 1.702 (1.702 + 2.2e-8) and GeGLU-quick uses 1.702 itself: for
    # negative g the relative difference is about |g| * 2.2e-8 <= 1.5e-7 at |g| <= 6.5
    assert np.allclose(oai, O.glu("geglu_quick", "separate", g, ones, N) * up1, rtol=1.5e-7, atol=1e-300)
    big_g = np.full_like(g, 7.0) + np.abs(g)                          # g >= limit
    at_lim = O.glu("swiglu_oai", "separate", np.full_like(g, 7.0), u, N)
    assert np.array_equal(O.glu("swiglu_oai", "separate", big_g, u, N), at_lim)
    for sgn in (1.0, -1.0):
        far = np.float32(sgn) * (np.float32(7.0) + np.abs(u))        # |u| >= limit
        lim = np.full_like(u, np.float32(sgn * 7.0))
        assert np.array_equal(O.glu("swiglu_oai", "separate", g, far, N), O.glu("swiglu_oai", "separate", g, lim, N))
    assert np.all(O.glu("swiglu_oai", "separate", g, -np.ones_like(u), N) == 0.0)
    # g below -limit is not clamped (the clamp on g is one-sided)
    low = np.full_like(g, -9.0)
    assert not np.array_equal(O.glu("swiglu_oai", "separate", low, u, N),
                              O.glu("swiglu_oai", "separate", np.full_like(g, -7.0), u, N))


def test_glu_swiglu_clamp_reductions_and_clamps():
    """SwiGLU-clamp (a reading: SwiGLU with SwiGLU-OAI's clamps): inside the limits it is SwiGLU;
    past them it is constant in g (from above) and in u (both ways); below -limit g is not clamped."""
    T, N = 2, 256
    g = np.clip(synth.activations(37, T, N) * np.float32(2.0), -6.5, 6.5).astype(np.float32)
    u = np.clip(synth.activations(38, T, N) * np.float32(2.0), -6.5, 6.5).astype(np.float32)
    assert np.array_equal(O.glu("swiglu_clamp", "separate", g, u, N), O.glu("swiglu", "separate", g, u, N))
    lim = np.full_like(g, 7.0)
    assert np.array_equal(O.glu("swiglu_clamp", "separate", lim + np.abs(g), u, N),
                          O.glu("swiglu_clamp", "separate", lim, u, N))
    for sgn in (1.0, -1.0):
        far = np.float32(sgn) * (np.float32(7.0) + np.abs(u))
        assert np.array_equal(O.glu("swiglu_clamp", "separate", g, far, N),
                              O.glu("swiglu_clamp", "separate", g, np.float32(sgn) * lim, N))
    low = np.full_like(g, -9.0)
    assert np.array_equal(O.glu("swiglu_clamp", "separate", low, u, N), O.glu("swiglu", "separate", low, u, N))


@pytest.mark.parametrize("kind", ["swiglu", "geglu_tanh", "reglu", "geglu_erf", "geglu_quick", "swiglu_oai",
                                  "swiglu_clamp"])
def test_glu_layouts(kind):
    T, N = 4, 96
    g = synth.activations(41, T, N)
    u = synth.activations(42, T, N)
    sep = O.glu(kind, "separate", g, u, N)
    packed = np.concatenate([g, u], axis=1)
    swapped = np.concatenate([u, g], axis=1)
    assert np.array_equal(O.glu(kind, "packed", packed, None, N), sep)
    assert np.array_equal(O.glu(kind, "packed_swapped", swapped, None, N), sep)
    # independent row strides: separate inputs taken from wider rows
    gw = np.zeros((T, N + 32), dtype=np.float32)
    uw = np.zeros((T, N + 64), dtype=np.float32)
    gw[:, :N], uw[:, :N] = g, u
    assert np.array_equal(O.glu(kind, "separate", gw, uw, N), sep)


# ----------------------------------------------------------------- weights / projections
def _decode_q4_0(W, N, K):
    """Independent decode: float64 W[n, k] from canonical blocks (low nibbles first, then high)."""
    blk = W.reshape(N, K // 32, 18)
    d = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    lo = (blk[:, :, 2:] & 0x0F).astype(np.int64)
    hi = (blk[:, :, 2:] >> 4).astype(np.int64)
    nib = np.concatenate([lo, hi], axis=2)
    return ((nib - 8) * d[..., None]).reshape(N, K), nib


def test_dequant_q4_0_matches_independent_decode():
    N, K = 8, 128
    W = synth.q4_0_weight(51, N, K)
    ref, _ = _decode_q4_0(W, N, K)
    assert np.array_equal(O.dequant("q4_0", W, N, K), ref)


def test_identity_weight_closed_form():
    """W = identity in Q4_0 (d=1, nibble 9 on the diagonal, 8 elsewhere): W x = x."""
    T, K = 3, 256
    N = K
    W = synth.q4_0_identity(N, K)
    x = synth.activations(52, T, K)
    assert np.array_equal(O.proj_plain("q4_0", W, N, K, x), x.astype(np.float64))
    img = O.quantize_q8_1(x)
    d, s, q = _decode_q8_1(img, T, K // 32)
    y = O.proj_q8_1("q4_0", W, N, K, img, K // 32)
    # quantised path: every block b of row n contributes d_a (D - 8 S) + 8 (d_a S - s_a) with
    # D = sum nib*q = 8 S (+ q_n in the diagonal's block), so y = d_a q_n + 8 sum_b (d_a S - s_a)
    S = q.sum(axis=2)
    corr = 8.0 * (d * S - s).sum(axis=1, keepdims=True)
    expect = (d[..., None] * q).reshape(T, K) + corr
    assert np.allclose(y, expect, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
@pytest.mark.parametrize("T,N,K", [(1, 5, 32), (3, 16, 96), (8, 33, 256)])
def test_quantized_projection_equals_matmul_of_decoded_operands(wtype, T, N, K):
    """Brute force on tiny shapes: the block-scaled integer dot equals a float64 matmul of the
    decoded operands, up to the half rounding of s (Q4_0 only), bounded exactly."""
    W = synth.q4_0_weight(60 + N, N, K) if wtype == "q4_0" else synth.q8_0_weight(60 + N, N, K)
    x = synth.activations(61 + K, T, K)
    img = O.quantize_q8_1(x)
    d, s, q = _decode_q8_1(img, T, K // 32)
    xq = (d[..., None] * q).reshape(T, K)
    if wtype == "q4_0":
        Wd, _ = _decode_q4_0(W, N, K)
        dw = W.reshape(N, K // 32, 18)[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
        # sum_b d_w (d_a sum(nib q) - 8 s_a) = xq @ Wd.T - 8 sum_b d_w (s_a - d_a S)
        S = q.sum(axis=2)
        expect = xq @ Wd.T - 8.0 * (s - d * S) @ dw.T
    else:
        blk = W.reshape(N, K // 32, 34)
        dw = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
        Wd = (blk[:, :, 2:].view(np.int8).astype(np.float64) * dw[..., None]).reshape(N, K)
        expect = xq @ Wd.T
    y = O.proj_q8_1(wtype, W, N, K, img, K // 32)
    assert np.allclose(y, expect, rtol=1e-12, atol=1e-12)
    # and the quantised path approximates the plain definition within the pages' bound
    assert O.nmse(y, O.proj_plain(wtype, W, N, K, x)) < 5e-4


def test_projection_uniform_weight_closed_form():
    """All nibbles 9 with one scale d: every output is d * sum(x) (plain definition)."""
    N, K = 4, 64
    W = np.zeros((N, K // 32, 18), dtype=np.uint8)
    W[:, :, 0:2] = np.array([0.125], dtype=np.float16).view(np.uint8)
    W[:, :, 2:] = 0x99
    x = synth.activations(70, 2, K)
    y = O.proj_plain("q4_0", W, N, K, x)
    assert np.allclose(y, 0.125 * x.astype(np.float64).sum(axis=1, keepdims=True), rtol=1e-14)


def test_q8_0_activation_projection_matches_decoded_matmul():
    T, N, K = 7, 9, 160
    W = synth.q4_0_weight(80, N, K)
    x = synth.activations(81, T, K)
    qs, dh = O.quantize_q8_0(x)
    da = dh.view(np.float16).astype(np.float64)
    xq = (qs.reshape(T, K // 32, 32).astype(np.float64) * da[..., None]).reshape(T, K)
    Wd, _ = _decode_q4_0(W, N, K)
    rows = np.arange(T)
    cols = np.array([0, 3, 8])
    got = O.proj_q8_0_sampled("q4_0", W, N, K, qs, dh, K // 32, rows, cols)
    assert np.allclose(got, (xq @ Wd.T)[:, cols], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- routing
def test_topk_matches_stable_argsort_and_softmax():
    rows, E, k = 20, 128, 8
    logits = synth.router_logits(90, rows, E)
    logits[5] = np.round(logits[5])           # many exact ties
    logits[6] = 0.0                           # all tied: experts 0..7
    ids, wts = O.topk_route(logits, k)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref)
    p = sp.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(wts, np.take_along_axis(p, ref, 1), rtol=1e-12, atol=0)
    assert np.array_equal(ids[6], np.arange(8))


def test_topk_skips_rows_past_live():
    rows, E, k = 16, 128, 8
    logits = synth.poison_rows(synth.router_logits(91, rows, E), live=9)
    stale = synth.stale_ids(92, rows, k, E)
    ids, wts = O.topk_route(logits, k, live=9, ids=stale.copy())
    assert np.array_equal(ids[9:], stale[9:])
    assert np.all(np.isnan(wts[9:]))
    ids9, _ = O.topk_route(logits[:9], k)
    assert np.array_equal(ids[:9], ids9)


@pytest.mark.parametrize("rows,live,k", [(16, 1, 8), (16, 9, 8), (32, 17, 8), (128, 113, 8),
                                         (128, 128, 8), (128, 113, 9), (128, 114, 9), (1, 1, 8)])
def test_plan_matches_stable_sort(rows, live, k):
    E = 128
    g = synth.rng(100 + rows * 7 + live)
    ids = g.integers(0, E, size=(rows, k), dtype=np.int32)
    counts, offsets, items = O.moe_plan(ids, E, live=live)
    npairs = live * k
    flat = ids.ravel()[:npairs]
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[E] == npairs and np.all(np.diff(offsets) == counts)
    assert np.array_equal(items, np.array(sorted(range(npairs), key=lambda p: flat[p]), dtype=np.int32))
    assert items.size == 0 or items.max() < npairs


@pytest.mark.parametrize("rows,live,k", [(16, 9, 8), (128, 113, 9), (4, 4, 2)])
def test_plan_leaves_out_pairs_with_invalid_ids(rows, live, k):
    """A pair whose id lies outside [0, E) names no expert: it gets no count and
    no item, and the plan of the rest equals the stable sort of the valid pairs."""
    E = 128
    g = synth.rng(140 + rows + live)
    ids = g.integers(0, E, size=(rows, k), dtype=np.int32)
    bad = g.random(size=ids.shape) < 0.2
    ids[bad] = g.choice(np.array([-1, -7, E, E + 5, 2**31 - 1], dtype=np.int64), size=int(bad.sum())).astype(np.int32)
    counts, offsets, items = O.moe_plan(ids, E, live=live)
    flat = ids.ravel()[:live * k]
    valid = [p for p in range(live * k) if 0 <= flat[p] < E]
    assert len(valid) < live * k   # the case really has invalid ids in the live range
    assert np.array_equal(counts, np.bincount(flat[valid], minlength=E))
    assert offsets[0] == 0 and offsets[E] == len(valid) and np.all(np.diff(offsets) == counts)
    assert np.array_equal(items, np.array(sorted(valid, key=lambda p: flat[p]), dtype=np.int32))


def test_routed_projection_rows():
    E, N, K, rows, k, live = 6, 8, 64, 4, 2, 3
    W = np.concatenate([synth.q4_0_weight(110 + e, N, K) for e in range(E)], axis=0)
    x = synth.activations(120, rows, K)
    img = O.quantize_q8_1(x)
    ids = synth.rng(121).integers(0, E, size=(rows, k), dtype=np.int32)
    _, _, items = O.moe_plan(ids, E, live=live)
    y = O.proj_id_q8_1("q4_0", W, E, N, K, img, K // 32, ids, items)
    for p in range(rows * k):
        if p < live * k:
            e = ids.ravel()[p]
            We = W[e * N:(e + 1) * N]
            assert np.array_equal(y[p], O.proj_q8_1("q4_0", We, N, K, img[p // k:p // k + 1], K // 32)[0])
        else:
            assert np.all(np.isnan(y[p]))


def test_per_slot_projection_reads_each_pairs_own_row():
    """Per-slot pairs: pair p's output is its expert's projection of image row p
    (not row p // k); checked against the single-matrix projection of that row."""
    E, N, K, rows, k, live = 5, 8, 64, 3, 4, 2
    W = np.concatenate([synth.q4_0_weight(130 + e, N, K) for e in range(E)], axis=0)
    xs = synth.activations(131, rows * k, K)
    img = O.quantize_q8_1(xs)
    ids = synth.rng(132).integers(0, E, size=(rows, k), dtype=np.int32)
    _, _, items = O.moe_plan(ids, E, live=live)
    y = O.proj_id_slots_q8_1("q4_0", W, E, N, K, img, K // 32, ids, items)
    for p in range(rows * k):
        if p < live * k:
            e = ids.ravel()[p]
            ref = O.proj_q8_1("q4_0", W[e * N:(e + 1) * N], N, K, img[p:p + 1], K // 32)[0]
            assert np.array_equal(y[p], ref)
        else:
            assert np.all(np.isnan(y[p]))


def test_combine_one_hot_selects_the_slot():
    """One-hot weights pick exactly one slot's output (catches a slot/row index mix-up),
    zero weights give zero, and weights summing to one over equal outputs give that output."""
    rows, k, N = 5, 3, 7
    eo = synth.rng(140).standard_normal((rows * k, N))
    pick = np.array([2, 0, 1, 1, 2])
    w = np.zeros((rows, k))
    w[np.arange(rows), pick] = 1.0
    y = O.moe_combine(eo, w)
    for r in range(rows):
        assert np.array_equal(y[r], eo[r * k + pick[r]])
    assert np.array_equal(O.moe_combine(eo, np.zeros((rows, k))), np.zeros((rows, N)))
    same = np.repeat(eo[:rows], k, axis=0)          # every slot of row r holds eo[r]
    wn = synth.rng(141).random((rows, k))
    wn /= wn.sum(axis=1, keepdims=True)
    assert np.allclose(O.moe_combine(same, wn), eo[:rows], rtol=1e-14, atol=1e-14)


def test_combine_skips_rows_past_live():
    rows, k, N, live = 6, 2, 4, 3
    eo = synth.rng(142).standard_normal((rows * k, N))
    w = synth.rng(143).random((rows, k))
    y = O.moe_combine(eo, w, live=live)
    assert np.all(np.isnan(y[live:])) and np.all(np.isfinite(y[:live]))
    assert np.array_equal(y[:live], O.moe_combine(eo[:live * k], w[:live]))
