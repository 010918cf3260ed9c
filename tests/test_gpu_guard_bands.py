"""Guard bands around every output of every entry point: out-of-bounds writes are
caught from the outside, without a device-side memory checker.

Each output buffer sits inside a larger allocation whose bytes before and after
it are a canary pattern, and, where an output has a row stride wider than its
rows, the bytes between rows are canaries too. After each call the test checks
that every canary byte is unchanged, so a write past the end of a buffer, past
the end of a row, into a row at or past the live count, or before the start of
a buffer is caught. Shapes are ragged (partial blocks, partial tiles, live
counts below the row count) so that the tail paths of the kernels run.
"""
import numpy as np
import pytest

from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import dev, live_ptr, pack_experts, pack_weight

pytestmark = pytest.mark.gpu

CANARY = 0xC3
PAD = 4096   # canary bytes before and after each output


class Guarded:
    """An output of `nbytes` bytes (a view into a canary-filled allocation). For row-strided
    outputs, rows=(n_rows, row_bytes, pitch_bytes) marks the bytes [row_bytes, pitch_bytes) of each
    row as canaries as well; `written` may narrow the rows that a call may write."""

    def __init__(self, nbytes, dtype="uint8", rows=None):
        import torch
        self.nbytes = nbytes
        self.buf = torch.full((PAD + nbytes + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        self.rows = rows
        self.t = self.buf[PAD:PAD + nbytes].view(getattr(torch, dtype))

    def check(self, what, writable_rows=None):
        import torch
        torch.cuda.synchronize()
        b = self.buf.cpu().numpy()
        assert (b[:PAD] == CANARY).all(), f"{what}: write before the buffer"
        assert (b[PAD + self.nbytes:] == CANARY).all(), f"{what}: write past the buffer"
        inner = b[PAD:PAD + self.nbytes]
        if self.rows is not None:
            n_rows, row_bytes, pitch = self.rows
            for r in range(n_rows):
                seg = inner[r * pitch:(r + 1) * pitch]
                if writable_rows is not None and r >= writable_rows:
                    assert (seg == CANARY).all(), f"{what}: row {r} at or past the live count written"
                else:
                    assert (seg[row_bytes:] == CANARY).all(), f"{what}: row {r} written past its width"


def test_quantizers_and_producers():
    import torch
    T, K, live = 7, 200, 5                    # K: six whole blocks and a partial one
    rb = 9                                    # two zero-padding blocks past ceil(K / 32)
    x = dev(synth.activations(9600, T, K))
    img = Guarded(T * rb * 36, rows=(T, rb * 36, rb * 36))
    qk.qk_quantize_q8_1(x, T, K, K, img.t, rb, d_live_rows=live_ptr(live))
    img.check("quantize_q8_1", writable_rows=live)

    qs = Guarded(T * rb * 32, "int8", rows=(T, rb * 32, rb * 32))
    dh = Guarded(T * rb * 2, "int16", rows=(T, rb * 2, rb * 2))
    qk.qk_quantize_q8_0(x, T, K, K, qs.t, dh.t, rb, d_live_rows=live_ptr(live))
    qs.check("quantize_q8_0 codes", writable_rows=live)
    dh.check("quantize_q8_0 scales", writable_rows=live)

    Kp = 224                                  # the producers' widths are whole blocks
    xp = dev(synth.activations(9604, T, Kp))
    w = dev(synth.norm_weight(9601, Kp))
    ys = Kp + 24                              # output pitch wider than the row
    y = Guarded(T * ys * 4, "float32", rows=(T, Kp * 4, ys * 4))
    img2 = Guarded(T * rb * 36, rows=(T, rb * 36, rb * 36))
    qk.qk_rmsnorm_q8_1(xp, T, Kp, Kp, "mul", w, None, 1.0, 1e-6, y.t, ys, img2.t, rb, d_live_rows=live_ptr(live))
    y.check("rmsnorm_q8_1 y", writable_rows=live)
    img2.check("rmsnorm_q8_1 image", writable_rows=live)

    y3 = Guarded(T * ys * 4, "float32", rows=(T, Kp * 4, ys * 4))
    qs3 = Guarded(T * rb * 32, "int8", rows=(T, rb * 32, rb * 32))
    dh3 = Guarded(T * rb * 2, "int16", rows=(T, rb * 2, rb * 2))
    qk.qk_rmsnorm_q8_0(xp, T, Kp, Kp, "mul", w, None, 1.0, 1e-6, y3.t, ys, qs3.t, dh3.t, rb,
                       d_live_rows=live_ptr(live))
    y3.check("rmsnorm_q8_0 y", writable_rows=live)
    qs3.check("rmsnorm_q8_0 codes", writable_rows=live)
    dh3.check("rmsnorm_q8_0 scales", writable_rows=live)

    N = 160
    a = dev(np.concatenate([synth.activations(9602, T, N), synth.activations(9603, T, N)], axis=1))
    os_ = N + 8
    out = Guarded(T * os_ * 4, "float32", rows=(T, N * 4, os_ * 4))
    gimg = Guarded(T * 6 * 36, rows=(T, 6 * 36, 6 * 36))
    qk.qk_glu_q8_1("swiglu", "packed", a, 2 * N, None, 0, T, N, out.t, os_, gimg.t, 6, d_live_rows=live_ptr(live))
    out.check("glu_q8_1 out", writable_rows=live)
    gimg.check("glu_q8_1 image", writable_rows=live)


def test_weight_pack_and_ordinary_projections():
    import torch
    T, K, live = 6, 640, 4
    rb = K // 32
    img = torch.empty((T * rb * 36,), dtype=torch.uint8, device="cuda")
    qk.qk_quantize_q8_1(dev(synth.activations(9610, T, K)), T, K, K, img, rb)
    shapes = (200, 72)                        # partial 128-row tiles
    packs = []
    for i, N in enumerate(shapes):
        nb = qk.qk_weight_packed_bytes("q4_0", N, K)
        p = Guarded(nb)
        qk.qk_weight_pack("q4_0", dev(synth.q4_0_weight(9611 + i, N, K).reshape(-1)), N, K, p.t, nb)
        p.check("weight_pack")
        packs.append(p)
    # both projections write column windows of one fused output with a gap between them and after them
    pitch = 200 + 8 + 72 + 16
    y = Guarded(T * pitch * 4, "float32")
    projs = [qk.make_proj("q4_0", packs[0].t, 200, K, y.t[0:], pitch),
             qk.make_proj("q4_0", packs[1].t, 72, K, y.t[208:], pitch)]
    ws_n = qk.qk_mmvq_workspace_bytes(projs)
    ws = torch.zeros((ws_n,), dtype=torch.uint8, device="cuda")
    for call in ("qk_mmvq", "qk_mmvq_static_ws"):
        y.buf.fill_(CANARY)
        if call == "qk_mmvq":
            qk.qk_mmvq(img, rb, T, projs, ws, ws_n, d_live_rows=live_ptr(live))
        else:
            qk.qk_mmvq_static_ws(img, rb, T, projs, d_live_rows=live_ptr(live))
        y.check(call)
        b = y.buf.cpu().numpy()[PAD:PAD + T * pitch * 4].reshape(T, pitch * 4)
        assert (b[:, 200 * 4:208 * 4] == CANARY).all(), f"{call}: gap between the windows written"
        assert (b[:, 280 * 4:] == CANARY).all(), f"{call}: columns after the second window written"
        assert (b[live:] == CANARY).all(), f"{call}: rows past the live count written"
        assert not (b[:live, :200 * 4] == CANARY).all(), f"{call}: first window not written"
    assert qk.qk_device_faults() == 0


def test_routing_plan_routed_projections_and_combine():
    import torch
    E, k, rows, live, K, N = 32, 4, 12, 9, 256, 192
    logits = dev(synth.router_logits(9620, rows, E))
    ids = Guarded(rows * k * 4, "int32", rows=(rows, k * 4, k * 4))
    wts = Guarded(rows * k * 4, "float32", rows=(rows, k * 4, k * 4))
    qk.qk_topk_route(logits, rows, E, k, ids.t, wts.t, d_live_rows=live_ptr(live))
    ids.check("topk_route ids", writable_rows=live)
    wts.check("topk_route wts", writable_rows=live)

    counts = Guarded(E * 4, "int32")
    offsets = Guarded((E + 1) * 4, "int32")
    items = Guarded(rows * k * 4, "int32")
    qk.qk_moe_plan(ids.t, rows, k, E, counts.t, offsets.t, items.t, d_live_rows=live_ptr(live))
    counts.check("moe_plan counts")
    offsets.check("moe_plan offsets")
    items.check("moe_plan items")
    assert (items.buf.cpu().numpy()[PAD + live * k * 4:PAD + rows * k * 4] == CANARY).all(), \
        "moe_plan: items past the planned pairs written"

    ids2 = Guarded(rows * k * 4, "int32", rows=(rows, k * 4, k * 4))
    wts2 = Guarded(rows * k * 4, "float32", rows=(rows, k * 4, k * 4))
    counts2, offsets2, items2 = Guarded(E * 4, "int32"), Guarded((E + 1) * 4, "int32"), Guarded(rows * k * 4, "int32")
    qk.qk_route_plan(logits, rows, E, k, ids2.t, wts2.t, counts2.t, offsets2.t, items2.t, d_live_rows=live_ptr(live))
    for g, name in ((ids2, "ids"), (wts2, "wts")):
        g.check(f"route_plan {name}", writable_rows=live)
    for g, name in ((counts2, "counts"), (offsets2, "offsets"), (items2, "items")):
        g.check(f"route_plan {name}")

    x = dev(synth.activations(9621, rows, K))
    img = torch.empty((rows * (K // 32) * 36,), dtype=torch.uint8, device="cuda")
    qk.qk_quantize_q8_1(x, rows, K, K, img, K // 32)
    Ws = pack_experts([synth.q4_0_weight(9630 + e, N, K) for e in range(E)], "q4_0", N, K)
    y = Guarded(rows * k * N * 4, "float32", rows=(rows * k, N * 4, N * 4))
    qk.qk_mmvq_id(img, K // 32, rows, k, [qk.make_proj_id("q4_0", E, Ws, N, K, y.t)], counts.t, offsets.t, items.t)
    y.check("mmvq_id", writable_rows=live * k)

    h = torch.empty((rows * k * N,), dtype=torch.float32, device="cuda")
    himg = torch.empty((rows * k * (N // 32) * 36,), dtype=torch.uint8, device="cuda")
    qk.qk_quantize_q8_1(dev(synth.activations(9622, rows * k, N)), rows * k, N, N, himg, N // 32)
    Wd = pack_experts([synth.q4_0_weight(9680 + e, K, N) for e in range(E)], "q4_0", K, N)
    yd = Guarded(rows * k * K * 4, "float32", rows=(rows * k, K * 4, K * 4))
    qk.qk_mmvq_id_slots(himg, N // 32, rows, k, [qk.make_proj_id("q4_0", E, Wd, K, N, yd.t)],
                        counts.t, offsets.t, items.t)
    yd.check("mmvq_id_slots", writable_rows=live * k)

    ysd = K + 40
    yo = Guarded(rows * ysd * 4, "float32", rows=(rows, K * 4, ysd * 4))
    expert_out = torch.randn((rows * k, K), dtype=torch.float32, device="cuda")
    qk.qk_moe_combine(expert_out, K, wts.t, rows, k, K, yo.t, ysd, d_live_rows=live_ptr(live))
    yo.check("moe_combine", writable_rows=live)
    del h
    assert qk.qk_device_faults() == 0


def test_prefill_contraction():
    import torch
    T, K, N = 333, 352, 200                   # a partial 256-token tile, 11 blocks, a partial row tile
    rb = K // 32
    qs = torch.empty((T * rb * 32,), dtype=torch.int8, device="cuda")
    d = torch.empty((T * rb,), dtype=torch.int16, device="cuda")
    qk.qk_quantize_q8_0(dev(synth.activations(9640, T, K)), T, K, K, qs, d, rb)
    pw = pack_weight(synth.q4_0_weight(9641, N, K), "q4_0", N, K)
    ys = N + 24
    y = Guarded(T * ys * 4, "float32", rows=(T, N * 4, ys * 4))
    projs = [qk.make_proj("q4_0", pw, N, K, y.t, ys)]
    n = qk.qk_mmq_workspace_bytes(T, projs)
    ws = Guarded(n)
    qk.qk_mmq(qs, d, rb, T, projs, ws.t, n)
    y.check("mmq")
    ws.check("mmq workspace")
    assert qk.qk_device_faults() == 0
