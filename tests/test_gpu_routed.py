"""GPU parity: router top-k, stable plan and routed MMVQ_ID, live-row aware.

Follows the routed live-row recipe on TensorFold PR #1047 ("Receipt"): the
routed chain is captured once per bucket as a CUDA graph and replayed at
changing live counts; before every replay the padding is poisoned (input rows
NaN / +1e30 / -1e30, stale picks naming real experts, NaN logits, sentinel
expert outputs). Every replay must plan exactly live*k pairs, leave padding
pairs' outputs and padding rows untouched, and give live rows equal byte for
byte to an uncaptured run at the exact row count.
"""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import assert_exact_path, dev, empty_u8, host, live_ptr, pack_experts

pytestmark = pytest.mark.gpu

E, TOPK, K, NF = 128, 8, 2560, 768


@pytest.mark.parametrize("rows,live", [(16, 1), (16, 9), (32, 17), (128, 113), (128, 128)])
def test_topk_matches_oracle(rows, live):
    import torch
    logits = synth.router_logits(6000 + rows + live, rows, E)
    logits[min(live, rows) - 1] = np.round(logits[min(live, rows) - 1] * 2)   # ties in one live row
    logits = synth.poison_rows(logits, live)
    stale = synth.stale_ids(6001, rows, TOPK, E)
    ids = dev(stale.copy())
    wts = torch.full((rows, TOPK), float("nan"), dtype=torch.float32, device="cuda")
    qk.qk_topk_route(dev(logits), rows, E, TOPK, ids, wts, live_ptr(live))
    gi, gw = host(ids), host(wts)
    ri, rw = O.topk_route(logits[:live], TOPK)
    assert np.array_equal(gi[:live], ri)
    assert np.allclose(gw[:live], rw, rtol=2e-6, atol=0)
    assert np.array_equal(gi[live:], stale[live:]) and np.all(np.isnan(gw[live:]))


@pytest.mark.parametrize("rows,live,k", [(16, 1, 8), (16, 9, 8), (32, 17, 8), (128, 113, 8), (128, 128, 8),
                                         (128, 113, 9), (128, 114, 9), (16, 0, 8), (600, 597, 8)])
def test_plan_matches_oracle(rows, live, k):
    import torch
    ids_h = synth.rng(6100 + rows + live + k).integers(0, E, size=(rows, k), dtype=np.int32)
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    items = torch.full((rows * k,), -7, dtype=torch.int32, device="cuda")
    qk.qk_moe_plan(dev(ids_h), rows, k, E, counts, offsets, items, live_ptr(live))
    rc, ro, ri = O.moe_plan(ids_h, E, live=live)
    gc, go, gi = host(counts), host(offsets), host(items)
    assert np.array_equal(gc, rc) and np.array_equal(go, ro)
    assert np.array_equal(gi[:live * k], ri)
    assert np.all(gi[live * k:] == -7)                     # positions past live*k untouched
    assert gc.sum() == live * k and (ri.size == 0 or ri.max() < live * k)


@pytest.mark.parametrize("rows,live,k", [(16, 9, 8), (128, 113, 9), (128, 128, 8)])
def test_plan_leaves_out_invalid_ids_like_the_oracle(rows, live, k):
    """Pairs whose id is outside [0, E) (-1, E, E + 5, INT32_MAX) get no count and no
    item on the GPU, exactly as in the oracle; the valid pairs keep their stable order."""
    import torch
    g = synth.rng(6200 + rows + live + k)
    ids_h = g.integers(0, E, size=(rows, k), dtype=np.int32)
    bad = g.random(size=ids_h.shape) < 0.25
    ids_h[bad] = g.choice(np.array([-1, E, E + 5, 2**31 - 1], dtype=np.int64), size=int(bad.sum())).astype(np.int32)
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    items = torch.full((rows * k,), -7, dtype=torch.int32, device="cuda")
    qk.qk_moe_plan(dev(ids_h), rows, k, E, counts, offsets, items, live_ptr(live))
    rc, ro, ri = O.moe_plan(ids_h, E, live=live)
    n_valid = int(((ids_h.ravel()[:live * k] >= 0) & (ids_h.ravel()[:live * k] < E)).sum())
    assert ro[E] == n_valid < live * k
    gc, go, gi = host(counts), host(offsets), host(items)
    assert np.array_equal(gc, rc) and np.array_equal(go, ro)
    assert np.array_equal(gi[:n_valid], ri)
    assert np.all(gi[n_valid:] == -7)                      # positions past the planned pairs untouched


def _experts(seed, n, N, K):
    return [synth.q4_0_weight(seed + e, N, K) for e in range(n)]


@pytest.fixture(scope="module")
def moe():
    """128 experts x (gate, up) Q4_0 [2560 -> 768], packed once."""
    Wg = _experts(7000, E, NF, K)
    Wu = _experts(8000, E, NF, K)
    return Wg, Wu, pack_experts(Wg, "q4_0", NF, K), pack_experts(Wu, "q4_0", NF, K)


def _routed_chain(moe, x_d, logits_d, rows, live_d, bufs):
    """RMSNorm(+image) -> top-k -> plan -> gate/up MMVQ_ID, all on the current stream."""
    Wg, Wu, pg, pu = moe
    qk.qk_rmsnorm_q8_1(x_d, rows, K, K, "mul", bufs["w"], None, 1.0, 1e-6, bufs["y"], K, bufs["img"], 80, live_d)
    qk.qk_topk_route(logits_d, rows, E, TOPK, bufs["ids"], bufs["wts"], live_d)
    qk.qk_moe_plan(bufs["ids"], rows, TOPK, E, bufs["counts"], bufs["offsets"], bufs["items"], live_d)
    projs = [qk.make_proj_id("q4_0", E, pg, NF, K, bufs["yg"]), qk.make_proj_id("q4_0", E, pu, NF, K, bufs["yu"])]
    qk.qk_mmvq_id(bufs["img"], 80, rows, TOPK, projs, bufs["counts"], bufs["offsets"], bufs["items"])


def _bufs(rows):
    import torch
    return {
        "w": dev(synth.norm_weight(9001, K)),
        "y": torch.full((rows, K), float("nan"), dtype=torch.float32, device="cuda"),
        "img": empty_u8(rows * 80 * 36),
        "ids": torch.zeros((rows, TOPK), dtype=torch.int32, device="cuda"),
        "wts": torch.zeros((rows, TOPK), dtype=torch.float32, device="cuda"),
        "counts": torch.zeros((E,), dtype=torch.int32, device="cuda"),
        "offsets": torch.zeros((E + 1,), dtype=torch.int32, device="cuda"),
        "items": torch.zeros((rows * TOPK,), dtype=torch.int32, device="cuda"),
        "yg": torch.zeros((rows * TOPK, NF), dtype=torch.float32, device="cuda"),
        "yu": torch.zeros((rows * TOPK, NF), dtype=torch.float32, device="cuda"),
    }


SENTINEL = np.float32(-12345.5)


def _poison(bufs, x_d, logits_d, rows, live, seed):
    """Poisons every padding input and output before a replay."""
    import torch
    x_h = synth.poison_rows(synth.activations(seed, rows, K), live)
    l_h = synth.router_logits(seed + 1, rows, E)
    l_h[live:] = np.nan
    x_d.copy_(torch.from_numpy(x_h))
    logits_d.copy_(torch.from_numpy(l_h))
    bufs["ids"].copy_(torch.from_numpy(synth.stale_ids(seed + 2, rows, TOPK, E)))
    bufs["wts"].fill_(float("nan"))
    bufs["yg"].fill_(float(SENTINEL))
    bufs["yu"].fill_(float(SENTINEL))
    bufs["items"].fill_(-3)
    bufs["y"].fill_(float("nan"))
    bufs["img"].fill_(0xA5)
    return x_h, l_h


def test_routed_projection_matches_oracle(moe):
    """Uncaptured chain at bucket 16, live 9: plan bit-exact, gate/up within the exact-path NMSE."""
    import torch
    Wg, Wu, _, _ = moe
    rows, live = 16, 9
    bufs = _bufs(rows)
    x_d = torch.empty((rows, K), dtype=torch.float32, device="cuda")
    l_d = torch.empty((rows, E), dtype=torch.float32, device="cuda")
    x_h, l_h = _poison(bufs, x_d, l_d, rows, live, 9100)
    _routed_chain(moe, x_d, l_d, rows, live_ptr(live), bufs)
    y = host(bufs["y"])
    img = host(bufs["img"]).reshape(rows, -1)
    ids = host(bufs["ids"])
    ri, _ = O.topk_route(l_h[:live], TOPK)
    assert np.array_equal(ids[:live], ri)
    rc, ro, rit = O.moe_plan(ids, E, live=live)
    assert np.array_equal(host(bufs["items"])[:live * TOPK], rit)
    assert np.array_equal(img[:live], O.quantize_q8_1(y[:live], row_blocks=80))
    Wall_g = np.concatenate(Wg, axis=0)
    Wall_u = np.concatenate(Wu, axis=0)
    for name, Wall in (("yg", Wall_g), ("yu", Wall_u)):
        yg = host(bufs[name])
        ref = O.proj_id_q8_1("q4_0", Wall, E, NF, K, img, 80, ids, rit)
        live_pairs = np.arange(live * TOPK)
        assert_exact_path(yg[live_pairs], ref[live_pairs], what="routed")
        assert np.all(yg[live * TOPK:] == SENTINEL)             # padding pairs: no expert work
        # plain definition gate on each pair's expert
        for p in live_pairs[::13]:
            e = ids.ravel()[p]
            plain = O.proj_plain("q4_0", Wall[e * NF:(e + 1) * NF], NF, K, y[p // TOPK:p // TOPK + 1])
            assert O.nmse(yg[p:p + 1], plain) <= 5e-4


@pytest.mark.parametrize("bucket,lives", [(16, [1, 2, 9, 16, 3]), (32, [17, 32, 5]),
                                          (128, [1, 9, 113, 114, 128, 2])])
def test_captured_bucket_replay_with_poisoned_padding(moe, bucket, lives):
    import torch
    bufs = _bufs(bucket)
    x_d = torch.empty((bucket, K), dtype=torch.float32, device="cuda")
    l_d = torch.empty((bucket, E), dtype=torch.float32, device="cuda")
    live_d = torch.zeros((1,), dtype=torch.int32, device="cuda")
    # warm up once uncaptured, then capture the whole chain once for this bucket
    live_d.fill_(bucket)
    _poison(bufs, x_d, l_d, bucket, bucket, 1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _routed_chain(moe, x_d, l_d, bucket, live_d, bufs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _routed_chain(moe, x_d, l_d, bucket, live_d, bufs)
    for i, live in enumerate(lives):
        live_d.fill_(live)
        x_h, l_h = _poison(bufs, x_d, l_d, bucket, live, 9200 + 10 * i)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        counts, items = host(bufs["counts"]), host(bufs["items"])
        assert counts.sum() == live * TOPK
        assert items[:live * TOPK].max() < live * TOPK and np.all(items[live * TOPK:] == -3)
        yg, yu, y = host(bufs["yg"]), host(bufs["yu"]), host(bufs["y"])
        assert np.all(yg[live * TOPK:] == SENTINEL) and np.all(yu[live * TOPK:] == SENTINEL)
        assert np.all(np.isnan(y[live:]))
        # live rows equal an uncaptured run at the exact row count, byte for byte
        ref = _bufs(live)
        xr = torch.from_numpy(x_h[:live].copy()).cuda()
        lr = torch.from_numpy(l_h[:live].copy()).cuda()
        _routed_chain(moe, xr, lr, live, None, ref)
        torch.cuda.synchronize()
        ids_b, ids_r = host(bufs["ids"])[:live], host(ref["ids"])
        assert np.array_equal(ids_b, ids_r)
        assert np.array_equal(y[:live].view(np.uint32), host(ref["y"]).view(np.uint32))
        assert np.array_equal(yg[:live * TOPK].view(np.uint32), host(ref["yg"]).view(np.uint32))
        assert np.array_equal(yu[:live * TOPK].view(np.uint32), host(ref["yu"]).view(np.uint32))


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
@pytest.mark.parametrize("n_exp,k", [(1, 1), (37, 4), (300, 4)])
def test_routed_widths_passes_and_ragged_tiles(wtype, n_exp, k):
    """Expert counts that are not a multiple of 32 and above one 32-expert run per warp, experts with
    more than 8 pairs (several passes), an odd number of 128-column chunks, ragged row tiles and two
    projections of different widths: outputs within the exact-path NMSE of the oracle, every planned
    pair written, every unplanned pair left as it was."""
    import torch
    rows, live, Kp = 48, 45, 384                      # 3 column chunks
    Ns = (200, 64)                                    # 2 row tiles (ragged) and 1
    g = synth.rng(9400 + n_exp + k)
    hot = max(1, min(5, n_exp))                       # half the pairs go to a few experts (> 8 pairs each)
    ids_h = np.where(g.random((rows, k)) < 0.5, g.integers(0, hot, size=(rows, k)),
                     g.integers(0, n_exp, size=(rows, k))).astype(np.int32)
    x = synth.activations(9401 + n_exp, rows, Kp)
    img_h = O.quantize_q8_1(x, row_blocks=Kp // 32)
    counts = torch.zeros((n_exp,), dtype=torch.int32, device="cuda")
    offsets = torch.zeros((n_exp + 1,), dtype=torch.int32, device="cuda")
    items = torch.zeros((rows * k,), dtype=torch.int32, device="cuda")
    qk.qk_moe_plan(dev(ids_h), rows, k, n_exp, counts, offsets, items, live_ptr(live))
    rc, ro, rit = O.moe_plan(ids_h, n_exp, live=live)
    assert np.array_equal(host(counts), rc) and rc.max() > 8
    gen = synth.q4_0_weight if wtype == "q4_0" else synth.q8_0_weight
    Ws = [[gen(9500 + 1000 * j + e, N, Kp) for e in range(n_exp)] for j, N in enumerate(Ns)]
    bufs = [pack_experts(Ws[j], wtype, N, Kp) for j, N in enumerate(Ns)]
    ys = [torch.full((rows * k, N), float(SENTINEL), dtype=torch.float32, device="cuda") for N in Ns]
    projs = [qk.make_proj_id(wtype, n_exp, bufs[j], N, Kp, ys[j]) for j, N in enumerate(Ns)]
    qk.qk_mmvq_id(dev(img_h.reshape(-1)), Kp // 32, rows, k, projs, counts, offsets, items)
    assert qk.qk_device_faults() == 0
    planned = np.zeros(rows * k, dtype=bool)
    planned[rit] = True
    for j, N in enumerate(Ns):
        got = host(ys[j])
        ref = O.proj_id_q8_1(wtype, np.concatenate(Ws[j], axis=0), n_exp, N, Kp, img_h, Kp // 32, ids_h, rit)
        assert_exact_path(got[planned], ref[planned], what="routed")
        assert np.all(got[~planned] == SENTINEL)


@pytest.mark.parametrize("rows,live,E_,k", [(16, 1, 128, 8), (16, 9, 128, 8), (32, 17, 128, 8), (32, 32, 256, 8),
                                            (16, 0, 128, 8), (8, 5, 37, 4), (128, 113, 128, 8)])
def test_route_plan_one_launch_equals_the_two_calls(rows, live, E_, k):
    """qk_route_plan (one CTA up to 32 rows, else the two launches) writes the same bytes as
    qk_topk_route followed by qk_moe_plan, and both match the oracle."""
    import torch
    logits = synth.poison_rows(synth.router_logits(9600 + rows + live, rows, E_), live)
    stale = synth.stale_ids(9601, rows, k, E_)
    l_d = dev(logits)

    def fresh():
        return (dev(stale.copy()), torch.full((rows, k), float("nan"), dtype=torch.float32, device="cuda"),
                torch.full((E_,), -7, dtype=torch.int32, device="cuda"),
                torch.full((E_ + 1,), -7, dtype=torch.int32, device="cuda"),
                torch.full((rows * k,), -7, dtype=torch.int32, device="cuda"))

    a = fresh()
    qk.qk_topk_route(l_d, rows, E_, k, a[0], a[1], live_ptr(live))
    qk.qk_moe_plan(a[0], rows, k, E_, a[2], a[3], a[4], live_ptr(live))
    b = fresh()
    qk.qk_route_plan(l_d, rows, E_, k, b[0], b[1], b[2], b[3], b[4], live_ptr(live))
    ha, hb = [host(t) for t in a], [host(t) for t in b]
    for x, y in zip(ha, hb):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    ri, rw = O.topk_route(logits[:live], k)
    assert np.array_equal(hb[0][:live], ri)
    rc, ro, rit = O.moe_plan(hb[0], E_, live=live)
    assert np.array_equal(hb[2], rc) and np.array_equal(hb[3], ro) and np.array_equal(hb[4][:live * k], rit)
