"""GPU parity: the closing steps of the routed FFN and the whole chain, live-row aware.

The per-slot down projection (qk_mmvq_id_slots) reads one image row per
(row, slot) pair, its own GLU output; the combine (qk_moe_combine) sums the
pairs' outputs with the router weights. Both follow TensorFold PR #1047:
padding rows get no plan items, no expert work and no combine, and the
captured chain replayed at changing live counts gives live rows equal byte for
byte to an uncaptured run at the exact row count.

Tolerances:
- projections against the oracle's exact block arithmetic: NMSE <= 1e-10 (the
  block dot is exact; only the binary32 sums over blocks differ);
- combine against float64: each of the k fused multiply-adds rounds once, so
  |y - ref| <= k * 2^-24 * sum_s |w_s * e_s| elementwise (plus a 1e-30 floor);
- chain end to end against the plain float64 definition: NMSE <= 5e-4, the
  pages' bound, over two Q8_1 quantisations (RMS output and GLU output).
"""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import assert_exact_path, dev, empty_u8, host, live_ptr, pack_experts

pytestmark = pytest.mark.gpu

SENTINEL = np.float32(-12345.5)
E, TOPK, HID, NF = 128, 8, 2560, 768


def _plan(ids_h, n_exp, live):
    import torch
    rows, k = ids_h.shape
    counts = torch.zeros((n_exp,), dtype=torch.int32, device="cuda")
    offsets = torch.zeros((n_exp + 1,), dtype=torch.int32, device="cuda")
    items = torch.full((rows * k,), -3, dtype=torch.int32, device="cuda")
    qk.qk_moe_plan(dev(ids_h), rows, k, n_exp, counts, offsets, items, live_ptr(live))
    return counts, offsets, items


# ------------------------------------------------------------------ per-slot projection
@pytest.mark.parametrize("rows,k,n_exp,N,K,live", [
    (8, 4, 32, 512, 8192, 8),        # 8 tokens x 4 slots = 32 slots, K = 8192
    (8, 16, 128, 768, 2560, 8),      # 8 tokens x 16 slots = 128 slots, K = 2560
    (16, 8, 128, 2560, 768, 9),      # the down projection of the 128-expert FFN, bucket 16, 9 live rows
    (5, 3, 7, 200, 384, 4),          # ragged row tile, 3 column chunks
])
def test_per_slot_matches_oracle(rows, k, n_exp, N, K, live):
    import torch
    rb = K // 32
    seed = 9700 + rows * k + K
    xs = synth.poison_rows(synth.activations(seed, rows * k, K), live * k)
    img = empty_u8(rows * k * rb * 36)
    qk.qk_quantize_q8_1(dev(xs), rows * k, K, K, img, rb)
    ids_h = synth.rng(seed + 1).integers(0, n_exp, size=(rows, k), dtype=np.int32)
    counts, offsets, items = _plan(ids_h, n_exp, live)
    Ws = [synth.q4_0_weight(seed + 10 + e, N, K) for e in range(n_exp)]
    pw = pack_experts(Ws, "q4_0", N, K)
    y = torch.full((rows * k, N), float(SENTINEL), dtype=torch.float32, device="cuda")
    qk.qk_mmvq_id_slots(img, rb, rows, k, [qk.make_proj_id("q4_0", n_exp, pw, N, K, y)], counts, offsets, items)
    assert qk.qk_device_faults() == 0
    img_h = host(img).reshape(rows * k, -1)
    assert np.array_equal(img_h[:live * k], O.quantize_q8_1(xs[:live * k], row_blocks=rb))
    _, _, rit = O.moe_plan(ids_h, n_exp, live=live)
    assert np.array_equal(host(items)[:live * k], rit)
    got = host(y)
    ref = O.proj_id_slots_q8_1("q4_0", np.concatenate(Ws, axis=0), n_exp, N, K, img_h, rb, ids_h, rit)
    npl = live * k
    assert_exact_path(got[:npl], ref[:npl], what="per-slot")
    assert np.all(got[npl:] == SENTINEL)                   # padding pairs: no expert work
    flat = ids_h.ravel()
    for p in range(0, npl, max(1, npl // 6)):              # plain definition, each pair's own row
        e = flat[p]
        plain = O.proj_plain("q4_0", Ws[e], N, K, xs[p:p + 1])
        assert O.nmse(got[p:p + 1], plain) <= 5e-4


def test_per_slot_two_projections_one_launch():
    """Two per-slot projections of different widths and weight types read one image: one launch
    per weight type."""
    import torch
    rows, k, n_exp, K, live = 12, 4, 9, 256, 11
    rb = K // 32
    xs = synth.activations(9800, rows * k, K)
    img_h = O.quantize_q8_1(xs, row_blocks=rb)
    ids_h = synth.rng(9801).integers(0, n_exp, size=(rows, k), dtype=np.int32)
    counts, offsets, items = _plan(ids_h, n_exp, live)
    specs = [("q4_0", 136, synth.q4_0_weight), ("q8_0", 64, synth.q8_0_weight)]
    keep, ys, projs = [], [], []
    for j, (wt, N, gen) in enumerate(specs):
        Ws = [gen(9810 + 100 * j + e, N, K) for e in range(n_exp)]
        pw = pack_experts(Ws, wt, N, K)
        y = torch.full((rows * k, N), float(SENTINEL), dtype=torch.float32, device="cuda")
        keep.append((Ws, pw))
        ys.append(y)
        projs.append(qk.make_proj_id(wt, n_exp, pw, N, K, y))
    n0 = qk.launch_count()
    qk.qk_mmvq_id_slots(dev(img_h.reshape(-1)), rb, rows, k, projs, counts, offsets, items)
    assert qk.launch_count() - n0 == 2
    _, _, rit = O.moe_plan(ids_h, n_exp, live=live)
    for (wt, N, _), (Ws, _), y in zip(specs, keep, ys):
        got = host(y)
        ref = O.proj_id_slots_q8_1(wt, np.concatenate(Ws, axis=0), n_exp, N, K, img_h, rb, ids_h, rit)
        assert_exact_path(got[:live * k], ref[:live * k], what="per-slot")
        assert np.all(got[live * k:] == SENTINEL)


# ------------------------------------------------------------------ combine
def _combine_case(rows, k, N, live, seed, one_hot=False):
    import torch
    g = synth.rng(seed)
    eo_stride, y_stride = N + 8, N + 4
    eo_h = g.standard_normal((rows * k, eo_stride)).astype(np.float32) * 3
    eo_h[live * k:] = np.nan                                # padding pairs: never read
    if one_hot:
        w_h = np.zeros((rows, k), dtype=np.float32)
        w_h[np.arange(rows), g.integers(0, k, size=rows)] = 1.0
    else:
        w_h = g.random((rows, k)).astype(np.float32)
        w_h /= w_h.sum(axis=1, keepdims=True)
    w_h[live:] = np.nan
    y = torch.full((rows, y_stride), float(SENTINEL), dtype=torch.float32, device="cuda")
    qk.qk_moe_combine(dev(eo_h), eo_stride, dev(w_h), rows, k, N, y, y_stride, live_ptr(live))
    return eo_h, w_h, host(y)


@pytest.mark.parametrize("rows,live", [(1, 1), (15, 9), (16, 15), (17, 16), (64, 63), (128, 113), (128, 128),
                                       (16, 0)])
def test_combine_matches_float64(rows, live):
    k, N = TOPK, HID
    eo_h, w_h, got = _combine_case(rows, k, N, live, 9900 + rows + live)
    ref = O.moe_combine(eo_h[:, :N], w_h, live=live)
    terms = np.abs(w_h[:live, :, None].astype(np.float64) * eo_h[:live * k, :N].reshape(live, k, N))
    bound = k * 2.0 ** -24 * terms.sum(axis=1) + 1e-30
    assert np.all(np.abs(got[:live, :N] - ref[:live]) <= bound)
    assert np.all(got[live:] == SENTINEL)                    # padding rows: no combine
    assert np.all(got[:, N:] == SENTINEL)                    # columns past N untouched


@pytest.mark.parametrize("rows,k,N", [(16, 8, 2560), (3, 9, 4), (7, 1, 96)])
def test_combine_one_hot_is_exact(rows, k, N):
    eo_h, w_h, got = _combine_case(rows, k, N, rows, 9950 + rows, one_hot=True)
    pick = np.argmax(w_h, axis=1)
    for r in range(rows):
        assert np.array_equal(got[r, :N], eo_h[r * k + pick[r], :N])


def test_combine_without_live_count_keeps_every_row():
    import torch
    rows, k, N = 6, 2, 64
    g = synth.rng(9990)
    eo_h = g.standard_normal((rows * k, N)).astype(np.float32)
    w_h = g.random((rows, k)).astype(np.float32)
    y = torch.full((rows, N), float(SENTINEL), dtype=torch.float32, device="cuda")
    qk.qk_moe_combine(dev(eo_h), N, dev(w_h), rows, k, N, y, N, None)
    got = host(y)
    assert np.allclose(got, O.moe_combine(eo_h, w_h), rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------------ the whole routed FFN
@pytest.fixture(scope="module")
def ffn():
    """128 experts: gate and up Q4_0 [2560 -> 768], down Q4_0 [768 -> 2560]."""
    Wg = [synth.q4_0_weight(20000 + e, NF, HID) for e in range(E)]
    Wu = [synth.q4_0_weight(21000 + e, NF, HID) for e in range(E)]
    Wd = [synth.q4_0_weight(22000 + e, HID, NF) for e in range(E)]
    return (Wg, Wu, Wd, pack_experts(Wg, "q4_0", NF, HID), pack_experts(Wu, "q4_0", NF, HID),
            pack_experts(Wd, "q4_0", HID, NF))


def _bufs(rows):
    import torch

    def f(*shape):
        return torch.full(shape, float(SENTINEL), dtype=torch.float32, device="cuda")
    return {
        "w": dev(synth.norm_weight(9001, HID)),
        "xn": f(rows, HID), "img": empty_u8(rows * (HID // 32) * 36),
        "ids": torch.zeros((rows, TOPK), dtype=torch.int32, device="cuda"), "wts": f(rows, TOPK),
        "counts": torch.zeros((E,), dtype=torch.int32, device="cuda"),
        "offsets": torch.zeros((E + 1,), dtype=torch.int32, device="cuda"),
        "items": torch.full((rows * TOPK,), -3, dtype=torch.int32, device="cuda"),
        "yg": f(rows * TOPK, NF), "yu": f(rows * TOPK, NF),
        "h": f(rows * TOPK, NF), "himg": empty_u8(rows * TOPK * (NF // 32) * 36),
        "yd": f(rows * TOPK, HID), "y": f(rows, HID),
    }


def _ffn_chain(ffn, x_d, logits_d, rows, live_d, b):
    """RMSNorm+image -> route+plan -> gate/up (token rows) -> SwiGLU+image (pair rows) ->
    down (pair rows) -> weighted combine, all on the current stream. The GLU's live count is
    the plan's total offsets[E] = live * k planned pairs, so padding pairs get no GLU work."""
    _, _, _, pg, pu, pd = ffn
    qk.qk_rmsnorm_q8_1(x_d, rows, HID, HID, "mul", b["w"], None, 1.0, 1e-6, b["xn"], HID, b["img"], HID // 32, live_d)
    qk.qk_route_plan(logits_d, rows, E, TOPK, b["ids"], b["wts"], b["counts"], b["offsets"], b["items"], live_d)
    qk.qk_mmvq_id(b["img"], HID // 32, rows, TOPK,
                  [qk.make_proj_id("q4_0", E, pg, NF, HID, b["yg"]), qk.make_proj_id("q4_0", E, pu, NF, HID, b["yu"])],
                  b["counts"], b["offsets"], b["items"])
    qk.qk_glu_q8_1("swiglu", "separate", b["yg"], NF, b["yu"], NF, rows * TOPK, NF, b["h"], NF, b["himg"], NF // 32,
                   b["offsets"][E:])
    qk.qk_mmvq_id_slots(b["himg"], NF // 32, rows, TOPK, [qk.make_proj_id("q4_0", E, pd, HID, NF, b["yd"])],
                        b["counts"], b["offsets"], b["items"])
    qk.qk_moe_combine(b["yd"], HID, b["wts"], rows, TOPK, HID, b["y"], HID, live_d)


def _poison(b, x_d, l_d, rows, live, seed):
    import torch
    x_h = synth.poison_rows(synth.activations(seed, rows, HID), live)
    l_h = synth.router_logits(seed + 1, rows, E)
    l_h[live:] = np.nan
    x_d.copy_(torch.from_numpy(x_h))
    l_d.copy_(torch.from_numpy(l_h))
    b["ids"].copy_(torch.from_numpy(synth.stale_ids(seed + 2, rows, TOPK, E)))
    for name in ("wts", "xn", "yg", "yu", "h", "yd", "y"):
        b[name].fill_(float(SENTINEL))
    b["items"].fill_(-3)
    b["img"].fill_(0xA5)
    b["himg"].fill_(0xA5)
    return x_h, l_h


def test_routed_ffn_chain_matches_oracle(ffn):
    """Bucket 16 with 9 live rows, uncaptured: every step against the oracle on its own device
    inputs, then the whole FFN against the plain float64 definition."""
    import torch
    Wg, Wu, Wd = ffn[:3]
    rows, live = 16, 9
    npl = live * TOPK
    b = _bufs(rows)
    x_d = torch.empty((rows, HID), dtype=torch.float32, device="cuda")
    l_d = torch.empty((rows, E), dtype=torch.float32, device="cuda")
    x_h, l_h = _poison(b, x_d, l_d, rows, live, 30000)
    _ffn_chain(ffn, x_d, l_d, rows, live_ptr(live), b)
    assert qk.qk_device_faults() == 0
    H = {k: host(v) for k, v in b.items()}
    ids = H["ids"]
    ri, rw = O.topk_route(l_h[:live], TOPK)
    assert np.array_equal(ids[:live], ri)
    _, ro, rit = O.moe_plan(ids, E, live=live)
    assert np.array_equal(H["offsets"], ro) and np.array_equal(H["items"][:npl], rit)
    img = H["img"].reshape(rows, -1)
    ref_g = O.proj_id_q8_1("q4_0", np.concatenate(Wg, axis=0), E, NF, HID, img, HID // 32, ids, rit)
    ref_u = O.proj_id_q8_1("q4_0", np.concatenate(Wu, axis=0), E, NF, HID, img, HID // 32, ids, rit)
    assert_exact_path(H["yg"][:npl], ref_g[:npl], what="gate")
    assert_exact_path(H["yu"][:npl], ref_u[:npl], what="up")
    # GLU over the planned pairs only; its image is the quantisation of the stored output
    ref_h = O.glu("swiglu", "separate", H["yg"][:npl], H["yu"][:npl], NF)
    gu = np.abs(H["yg"][:npl].astype(np.float64) * H["yu"][:npl])
    assert np.all(np.abs(H["h"][:npl] - ref_h) <= np.abs(ref_h) * 2e-6 + 3e-7 * gu + 1e-30)
    assert np.all(H["h"][npl:] == SENTINEL)
    himg = H["himg"].reshape(rows * TOPK, -1)
    assert np.array_equal(himg[:npl], O.quantize_q8_1(H["h"][:npl], row_blocks=NF // 32))
    assert np.all(himg[npl:] == 0xA5)
    # per-slot down projection and combine
    ref_d = O.proj_id_slots_q8_1("q4_0", np.concatenate(Wd, axis=0), E, HID, NF, himg, NF // 32, ids, rit)
    assert_exact_path(H["yd"][:npl], ref_d[:npl], what="down")
    assert np.all(H["yd"][npl:] == SENTINEL)
    ref_y = O.moe_combine(H["yd"][:npl], H["wts"][:live])
    terms = np.abs(H["wts"][:live, :, None].astype(np.float64) * H["yd"][:npl].reshape(live, TOPK, HID))
    assert np.all(np.abs(H["y"][:live] - ref_y) <= TOPK * 2.0 ** -24 * terms.sum(axis=1) + 1e-30)
    assert np.all(H["y"][live:] == SENTINEL)
    # the whole FFN in float64 from the input rows and the decoded weights
    xn = O.rmsnorm(x_h[:live], "mul", w=synth.norm_weight(9001, HID), eps=1e-6)
    full = np.zeros((live, HID))
    for r in range(live):
        for s in range(TOPK):
            e = ri[r, s]
            g = O.dequant("q4_0", Wg[e], NF, HID) @ xn[r]
            u = O.dequant("q4_0", Wu[e], NF, HID) @ xn[r]
            h = g / (1.0 + np.exp(-g)) * u
            full[r] += rw[r, s] * (O.dequant("q4_0", Wd[e], HID, NF) @ h)
    assert O.nmse(H["y"][:live], full) <= 5e-4


@pytest.mark.parametrize("bucket,lives", [(16, [1, 9, 16, 3]), (32, [17, 32, 2])])
def test_captured_ffn_replay_with_poisoned_padding(ffn, bucket, lives):
    """The chain captured once per bucket and replayed at changing live counts: padding pairs and
    rows keep their poison, live rows equal an uncaptured run at the exact row count byte for byte."""
    import torch
    b = _bufs(bucket)
    x_d = torch.empty((bucket, HID), dtype=torch.float32, device="cuda")
    l_d = torch.empty((bucket, E), dtype=torch.float32, device="cuda")
    live_d = torch.zeros((1,), dtype=torch.int32, device="cuda")
    live_d.fill_(bucket)
    _poison(b, x_d, l_d, bucket, bucket, 1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _ffn_chain(ffn, x_d, l_d, bucket, live_d, b)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _ffn_chain(ffn, x_d, l_d, bucket, live_d, b)
    for i, live in enumerate(lives):
        npl = live * TOPK
        live_d.fill_(live)
        x_h, l_h = _poison(b, x_d, l_d, bucket, live, 31000 + 10 * i)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert qk.qk_device_faults() == 0
        H = {k: host(b[k]) for k in ("items", "h", "yd", "y")}
        assert np.all(H["items"][npl:] == -3)
        assert np.all(H["h"][npl:] == SENTINEL) and np.all(H["yd"][npl:] == SENTINEL)
        assert np.all(H["y"][live:] == SENTINEL)
        ref = _bufs(live)
        xr = torch.from_numpy(x_h[:live].copy()).cuda()
        lr = torch.from_numpy(l_h[:live].copy()).cuda()
        _ffn_chain(ffn, xr, lr, live, None, ref)
        torch.cuda.synchronize()
        assert np.array_equal(H["yd"][:npl].view(np.uint32), host(ref["yd"]).view(np.uint32))
        assert np.array_equal(H["y"][:live].view(np.uint32), host(ref["y"]).view(np.uint32))


def test_combine_more_rows_than_a_grid_y_dimension():
    """70,000 rows (over the 65,535 limit of a grid's y dimension): rows run on grid x."""
    import torch
    rows, k, N, live = 70000, 2, 8, 69999
    g = synth.rng(9995)
    eo_h = g.standard_normal((rows * k, N)).astype(np.float32)
    w_h = g.random((rows, k)).astype(np.float32)
    y = torch.full((rows, N), float(SENTINEL), dtype=torch.float32, device="cuda")
    qk.qk_moe_combine(dev(eo_h), N, dev(w_h), rows, k, N, y, N, live_ptr(live))
    got = host(y)
    ref = O.moe_combine(eo_h, w_h, live=live)
    terms = np.abs(w_h[:live, :, None].astype(np.float64) * eo_h[:live * k].reshape(live, k, N))
    assert np.all(np.abs(got[:live] - ref[:live]) <= k * 2.0 ** -24 * terms.sum(axis=1) + 1e-30)
    assert np.all(got[live:] == SENTINEL)


def test_per_slot_at_the_expert_and_slot_limits():
    """1024 experts (the most a routed call takes) and 64 slots per row (the most a plan takes):
    every planned pair within the exact-path NMSE, padding pairs untouched."""
    import torch
    rows, k, n_exp, N, K, live = 3, 64, 1024, 64, 128, 2
    rb = K // 32
    xs = synth.activations(9960, rows * k, K)
    img_h = O.quantize_q8_1(xs, row_blocks=rb)
    ids_h = synth.rng(9961).integers(0, n_exp, size=(rows, k), dtype=np.int32)
    counts, offsets, items = _plan(ids_h, n_exp, live)
    Ws = [synth.q4_0_weight(10000 + e, N, K) for e in range(n_exp)]
    pw = pack_experts(Ws, "q4_0", N, K)
    y = torch.full((rows * k, N), float(SENTINEL), dtype=torch.float32, device="cuda")
    qk.qk_mmvq_id_slots(dev(img_h.reshape(-1)), rb, rows, k, [qk.make_proj_id("q4_0", n_exp, pw, N, K, y)],
                        counts, offsets, items)
    assert qk.qk_device_faults() == 0
    _, _, rit = O.moe_plan(ids_h, n_exp, live=live)
    got = host(y)
    ref = O.proj_id_slots_q8_1("q4_0", np.concatenate(Ws, axis=0), n_exp, N, K, img_h, rb, ids_h, rit)
    assert_exact_path(got[:live * k], ref[:live * k], what="per-slot")
    assert np.all(got[live * k:] == SENTINEL)


def test_combine_at_the_slot_limit():
    eo_h, w_h, got = _combine_case(5, 64, 96, 4, 9970)
    ref = O.moe_combine(eo_h[:, :96], w_h, live=4)
    terms = np.abs(w_h[:4, :, None].astype(np.float64) * eo_h[:4 * 64, :96].reshape(4, 64, 96))
    assert np.all(np.abs(got[:4, :96] - ref[:4]) <= 64 * 2.0 ** -24 * terms.sum(axis=1) + 1e-30)
    assert np.all(got[4:] == SENTINEL)
