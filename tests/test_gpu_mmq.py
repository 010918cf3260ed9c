"""GPU parity: prefill contraction qk_mmq on a Q8_0 image, against the oracle.

Gate: NMSE <= 5e-4 against the plain definition (the pages' bound).
Diagnostic against the oracle's exact quantised path: the GEMM runs on the
tensor cores with binary16 operands (nibble - 8) * d_w and q * d_a, each
rounded once (unit roundoff u = 2^-11), accumulated in binary32. Each product
then carries a relative error of at most about 2u with random sign, so the
NMSE against the exact block form is about 2u^2/3 = 1.6e-7; the test allows
2e-6. A wrong block, scale or index gives an NMSE above 1e-3.
At the prefill size (3325 tokens, d = 3584) the oracle computes every row of
64 seeded random columns plus 16 full rows of each projection.
"""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import assert_exact_path, dev, host, pack_weight

pytestmark = pytest.mark.gpu

NMSE_GATE = 5e-4
NMSE_EXACT = 2e-6   # binary16 operand rounding, see the module docstring
# element by element: each product carries about 2^-11 relative error, so an element's error is
# about 4e-4 of the output's rms (5 rms ~ the largest output); a dropped block moves an element by
# about rms / sqrt(112) at K = 3584, far past 2e-3 of the largest output
REL_EXACT = 2e-3


def quantize_q8_0(x, K, rb):
    import torch
    T = x.shape[0]
    qs = torch.zeros((T * rb * 32,), dtype=torch.int8, device="cuda")
    d = torch.zeros((T * rb,), dtype=torch.int16, device="cuda")
    qk.qk_quantize_q8_0(dev(x), T, K, x.shape[1], qs, d, rb)
    return qs, d


def run_mmq(qs, d, rb, T, specs):
    import torch
    outs, projs, keep = [], [], []
    for (W, N, K) in specs:
        y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
        pw = pack_weight(W, "q4_0", N, K)
        keep.append(pw)                   # the descriptors hold raw pointers only
        outs.append(y)
        projs.append(qk.make_proj("q4_0", pw, N, K, y, N))
    n = qk.qk_mmq_workspace_bytes(T, projs)
    ws = torch.empty((n,), dtype=torch.uint8, device="cuda")
    keep.append(ws)
    qk.qk_mmq(qs, d, rb, T, projs, ws, n)
    outs = [host(y) for y in outs]
    assert qk.qk_device_faults() == 0
    return outs, keep


@pytest.mark.parametrize("T,N,K,rb", [(100, 200, 384, 12), (65, 130, 160, 6), (1, 128, 128, 4), (64, 256, 256, 8),
                                      (130, 64, 1056, 33),
                                      (1, 1, 32, 1),       # one token, one weight row, one block
                                      (257, 129, 96, 3),   # a 1-token and a 1-row tail tile, K of 3 blocks
                                      (3, 300, 32, 2)])    # K of one block inside a wider image row
def test_mmq_small_full(T, N, K, rb):
    x = synth.activations(7000 + T + N, T, K)
    W = synth.q4_0_weight(7001 + N, N, K)
    qs, d = quantize_q8_0(x, K, rb)
    (yg,), _ = run_mmq(qs, d, rb, T, [(W, N, K)])
    qsh = host(qs).view(np.int8).reshape(T, -1)
    dh = host(d).view(np.uint16).reshape(T, -1)
    exact = O.proj_q8_0_sampled("q4_0", W, N, K, qsh, dh, rb, np.arange(T), np.arange(N))
    assert_exact_path(yg, exact, NMSE_EXACT, REL_EXACT, what="mmq")
    assert O.nmse(yg, O.proj_plain("q4_0", W, N, K, x)) <= NMSE_GATE


def test_mmq_b_operand_is_each_code_times_its_scale_rounded_once():
    """The dequantised B operand the call leaves in its workspace: every code times its block's
    scale, the exact product rounded once to binary16, in the K order of the tensor-memory A
    stages (halves 4w .. 4w+3 of a 16-element half-block hold elements 4w, 4w+2, 4w+1, 4w+3),
    against numpy's float64 product rounded to float16; bit for bit, including subnormal
    products of tiny blocks."""
    T, K, rb, N = 70, 384, 13, 64
    x = synth.activations(7400, T, K) * np.float32(3.0)
    x[5, :64] *= np.float32(1e-5)            # tiny scales: subnormal binary16 products
    x[6, 32:64] = 0.0                        # a zero block: d = 0
    W = synth.q4_0_weight(7401, N, K)
    qs, d = quantize_q8_0(x, K, rb)
    _, keep = run_mmq(qs, d, rb, T, [(W, N, K)])
    kb = K // 32
    B = host(keep[-1])[:T * kb * 32 * 2].view(np.uint16).reshape(T, kb, 32)
    q = host(qs).view(np.int8).reshape(T, rb, 32)[:, :kb].astype(np.float64)
    dd = host(d).view(np.float16).reshape(T, rb)[:, :kb].astype(np.float64)
    order = [16 * (p // 16) + 4 * (p % 16 // 4) + (0, 2, 1, 3)[p % 4] for p in range(32)]
    want = (q[:, :, order] * dd[:, :, None]).astype(np.float16).view(np.uint16)
    assert np.array_equal(B, want)


def test_mmq_projections_of_different_k_in_one_launch():
    """Several projections of one image with different K in one launch: B is dequantised for the
    largest K and each projection reads only its own 128-K stages (a partial last stage meets the
    weights' zero padding). Every output against the oracle's exact path."""
    T, rb = 70, 12
    x = synth.activations(7200, T, rb * 32)
    qs, d = quantize_q8_0(x, rb * 32, rb)
    specs = [(synth.q4_0_weight(7201, 200, 384), 200, 384), (synth.q4_0_weight(7202, 96, 160), 96, 160),
             (synth.q4_0_weight(7203, 130, 256), 130, 256)]
    outs, _ = run_mmq(qs, d, rb, T, specs)
    qsh = host(qs).view(np.int8).reshape(T, -1)
    dh = host(d).view(np.uint16).reshape(T, -1)
    for (W, N, K), yg in zip(specs, outs):
        assert not np.isnan(yg).any()
        exact = O.proj_q8_0_sampled("q4_0", W, N, K, qsh, dh, rb, np.arange(T), np.arange(N))
        assert_exact_path(yg, exact, NMSE_EXACT, REL_EXACT, what=f"mmq K={K}")
        assert O.nmse(yg, O.proj_plain("q4_0", W, N, K, x[:, :K])) <= NMSE_GATE


def _sampled_check(yg, W, N, K, qsh, dh, rb, x, seed, ncols=64, nrows=16):
    T = yg.shape[0]
    g = synth.rng(seed)
    cols = np.sort(g.choice(N, size=min(ncols, N), replace=False))
    rows = np.sort(g.choice(T, size=nrows, replace=False))
    exact_cols = O.proj_q8_0_sampled("q4_0", W, N, K, qsh, dh, rb, np.arange(T), cols)
    assert_exact_path(yg[:, cols], exact_cols, NMSE_EXACT, REL_EXACT, what="mmq columns")
    exact_rows = O.proj_q8_0_sampled("q4_0", W, N, K, qsh, dh, rb, rows, np.arange(N))
    assert_exact_path(yg[rows], exact_rows, NMSE_EXACT, REL_EXACT, what="mmq rows")
    Wd = O.dequant("q4_0", W[cols], len(cols), K)
    assert O.nmse(yg[:, cols], x.astype(np.float64) @ Wd.T) <= NMSE_GATE


def test_prefill_qkv_one_image_three_readers():
    """3325 tokens x d=3584: one Q8_0 image read by q [3584->3584], k, v [3584->512] in one launch."""
    T, K = 3325, 3584
    x = synth.activations(4000, T, K)
    qs, d = quantize_q8_0(x, K, 112)
    shapes = [3584, 512, 512]
    Ws = [synth.q4_0_weight(4010 + i, N, K) for i, N in enumerate(shapes)]
    n0 = qk.launch_count()
    outs, _ = run_mmq(qs, d, 112, T, [(W, N, K) for W, N in zip(Ws, shapes)])
    # weight packing launched one kernel per projection; the contraction is two launches
    # (the dequantised image, then one GEMM for the three readers)
    assert qk.launch_count() - n0 == len(shapes) + 2
    qsh = host(qs).view(np.int8).reshape(T, -1)
    dh = host(d).view(np.uint16).reshape(T, -1)
    for i, (W, N, yg) in enumerate(zip(Ws, shapes, outs)):
        _sampled_check(yg, W, N, K, qsh, dh, 112, x, 4020 + i)


def test_prefill_gate_projection():
    """The gate shape 3584 -> 18944 at 3325 tokens (sampled outputs)."""
    T, K, N = 3325, 3584, 18944
    x = synth.activations(4100, T, K)
    qs, d = quantize_q8_0(x, K, 112)
    W = synth.q4_0_weight(4101, N, K)
    (yg,), _ = run_mmq(qs, d, 112, T, [(W, N, K)])
    _sampled_check(yg, W, N, K, host(qs).view(np.int8).reshape(T, -1), host(d).view(np.uint16).reshape(T, -1),
                   112, x, 4102)


def test_dedup_one_quantize_per_distinct_activation():
    """Shared-A dedup (minfer doc 52): the image made once and read by q, k and v equals
    three independent quantisations byte for byte (a pure function of the input), and a
    layer needs 2 quantize launches (normed, normed2), not one per GEMM."""
    T, K = 257, 512
    x = synth.activations(4200, T, K)
    x2 = synth.activations(4201, T, K)
    n0 = qk.launch_count()
    qs, d = quantize_q8_0(x, K, 16)
    qs2, d2 = quantize_q8_0(x2, K, 16)
    assert qk.launch_count() - n0 == 2
    for _ in range(3):
        qa, da = quantize_q8_0(x, K, 16)
        assert np.array_equal(host(qa), host(qs)) and np.array_equal(host(da), host(d))
    Wq = [synth.q4_0_weight(4210 + i, N, K) for i, N in enumerate((512, 128, 128))]
    Wg = [synth.q4_0_weight(4220 + i, 1024, K) for i in range(2)]
    outs_qkv, _ = run_mmq(qs, d, 16, T, [(W, W.shape[0], K) for W in Wq])
    outs_gu, _ = run_mmq(qs2, d2, 16, T, [(W, W.shape[0], K) for W in Wg])
    for W, yg in zip(Wq, outs_qkv):
        assert O.nmse(yg, O.proj_plain("q4_0", W, W.shape[0], K, x)) <= NMSE_GATE
    for W, yg in zip(Wg, outs_gu):
        assert O.nmse(yg, O.proj_plain("q4_0", W, W.shape[0], K, x2)) <= NMSE_GATE


def test_prefill_layers_with_fresh_seeds():
    """Several prefill layers in a row (3325 tokens, d = 3584), each with its own seeded weights
    and activations (seed 4000 + layer): per layer one Q8_0 image of the attention input read by
    q/k/v in one launch and one image of the FFN input read by gate/up in one launch. The image
    planes and the workspace are reused from layer to layer, as in a whole prefill; every layer's
    outputs are checked on sampled columns and rows against the oracle."""
    import torch
    T, K, rb, NFF = 3325, 3584, 112, 18944
    qs = torch.zeros((T * rb * 32,), dtype=torch.int8, device="cuda")
    d = torch.zeros((T * rb,), dtype=torch.int16, device="cuda")
    # one workspace for both launches: the larger of the two sizes (it depends on the projections)
    n = max(qk.qk_mmq_workspace_bytes(T, [qk.make_proj("q4_0", 16, N, K, 16, N) for N in shapes])
            for shapes in ((3584, 512, 512), (NFF, NFF)))
    ws = torch.empty((n,), dtype=torch.uint8, device="cuda")
    for layer in range(3):
        seed = 4000 + layer
        for part, shapes in (("attn", (3584, 512, 512)), ("ffn", (NFF, NFF))):
            x = synth.activations(seed * 10 + (0 if part == "attn" else 1), T, K)
            qk.qk_quantize_q8_0(dev(x), T, K, K, qs, d, rb)
            Ws = [synth.q4_0_weight(seed * 100 + (0 if part == "attn" else 10) + i, N, K) for i, N in enumerate(shapes)]
            keep, projs, outs = [], [], []
            for W, N in zip(Ws, shapes):
                pw = pack_weight(W, "q4_0", N, K)
                y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
                keep += [pw, y]
                outs.append(y)
                projs.append(qk.make_proj("q4_0", pw, N, K, y, N))
            qk.qk_mmq(qs, d, rb, T, projs, ws, n)
            qsh = host(qs).view(np.int8).reshape(T, -1)
            dh = host(d).view(np.uint16).reshape(T, -1)
            for i, (W, N, y) in enumerate(zip(Ws, shapes, outs)):
                yg = host(y)
                assert not np.isnan(yg).any()
                _sampled_check(yg, W, N, K, qsh, dh, rb, x, seed * 7 + i, ncols=24, nrows=6)
    assert qk.qk_device_faults() == 0
