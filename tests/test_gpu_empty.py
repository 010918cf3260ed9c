"""GPU: empty inputs. A row count of 0 where a call accepts it (the producers' T, the routing
calls' rows) launches nothing and writes nothing; the plans write the zero counts and offsets of
an empty plan (the oracle's plan of no pairs); the projections refuse T = 0 before launching; a
device live count of 0 leaves every output of a projection as it was."""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import dev, empty_u8, host, live_ptr, mmvq, pack_weight

pytestmark = pytest.mark.gpu

K, N = 256, 128


def f32(n, fill=np.nan):
    import torch
    return torch.full((n,), float(fill), dtype=torch.float32, device="cuda")


def test_producers_with_no_rows_launch_and_write_nothing():
    import torch
    x = dev(synth.activations(7000, 2, K))
    w = dev(synth.norm_weight(7001, K))
    img = empty_u8(2 * (K // 32) * 36)
    qs = torch.full((2 * K,), 0x5A, dtype=torch.int8, device="cuda")
    d = torch.full((2 * (K // 32),), 0x1234, dtype=torch.int16, device="cuda")
    y = f32(2 * K)
    g = dev(synth.activations(7002, 2, 2 * K))
    out = f32(2 * K)
    before = [host(t).copy() for t in (img, qs, d, y, out)]
    n0 = qk.launch_count()
    qk.qk_quantize_q8_1(x, 0, K, K, img, K // 32)
    qk.qk_quantize_q8_0(x, 0, K, K, qs, d, K // 32)
    qk.qk_rmsnorm_q8_1(x, 0, K, K, "mul", w, None, 1.0, 1e-6, y, K, img, K // 32)
    qk.qk_rmsnorm_q8_0(x, 0, K, K, "mul", w, None, 1.0, 1e-6, y, K, qs, d, K // 32)
    qk.qk_glu_q8_1("swiglu", "packed", g, 2 * K, None, 0, 0, K, out, K, img, K // 32)
    assert qk.launch_count() == n0
    after = [host(t) for t in (img, qs, d, y, out)]
    for a, b in zip(before, after):
        assert np.array_equal(a, b, equal_nan=True)
    assert qk.qk_device_faults() == 0


@pytest.mark.parametrize("E,k", [(128, 8), (8, 2)])
def test_plans_of_no_rows_are_the_empty_plan(E, k):
    import torch
    logits = dev(synth.router_logits(7010, 1, E))
    ids = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    wts = f32(k, 3.0)
    n0 = qk.launch_count()
    qk.qk_topk_route(logits, 0, E, k, ids, wts)            # nothing to route: no launch
    assert qk.launch_count() == n0
    assert np.all(host(ids) == -7) and np.all(host(wts) == 3.0)
    oc, oo, oi = O.moe_plan(np.zeros((0, k), dtype=np.int32), E)
    assert oi.size == 0 and not oc.any() and not oo.any()
    for call in ("plan", "route_plan"):
        counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
        items = torch.full((k,), -3, dtype=torch.int32, device="cuda")
        if call == "plan":
            qk.qk_moe_plan(ids, 0, k, E, counts, offsets, items)
        else:
            qk.qk_route_plan(logits, 0, E, k, ids, wts, counts, offsets, items)
        assert np.array_equal(host(counts), oc) and np.array_equal(host(offsets), oo), call
        assert np.all(host(items) == -3), call
        assert np.all(host(ids) == -7), call
    assert qk.qk_device_faults() == 0


def test_combine_of_no_rows_launches_nothing():
    import torch
    k = 4
    eo = dev(synth.activations(7020, k, N))
    wts = dev(np.full((1, k), 0.25, dtype=np.float32))
    y = f32(N)
    n0 = qk.launch_count()
    qk.qk_moe_combine(eo, N, wts, 0, k, N, y, N)
    assert qk.launch_count() == n0
    assert np.all(np.isnan(host(y)))


def test_projections_refuse_no_rows_before_launching():
    import torch
    W = synth.q4_0_weight(7030, N, K)
    pw = pack_weight(W, "q4_0", N, K)
    img = empty_u8(8 * (K // 32) * 36)
    y = torch.full((8, N), float("nan"), dtype=torch.float32, device="cuda")
    projs = [qk.make_proj("q4_0", pw, N, K, y, N)]
    ws = torch.zeros((max(16, qk.qk_mmvq_workspace_bytes(projs)),), dtype=torch.uint8, device="cuda")
    n0 = qk.launch_count()
    with pytest.raises(qk.QkError) as e:
        qk.qk_mmvq(img, K // 32, 0, projs, ws, ws.numel())
    assert e.value.name == "QK_ERR_ARG"
    qs = torch.zeros((8 * K,), dtype=torch.int8, device="cuda")
    d = torch.zeros((8 * (K // 32),), dtype=torch.int16, device="cuda")
    wsq = torch.zeros((1 << 20,), dtype=torch.uint8, device="cuda")
    with pytest.raises(qk.QkError) as e:
        qk.qk_mmq(qs, d, K // 32, 0, projs, wsq, wsq.numel())
    assert e.value.name == "QK_ERR_ARG"
    assert qk.launch_count() == n0
    assert np.all(np.isnan(host(y)))


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
def test_projection_with_a_live_count_of_zero_writes_nothing(wtype):
    import torch
    T = 8
    x = synth.activations(7040, T, K)
    img = empty_u8(T * (K // 32) * 36)
    qk.qk_quantize_q8_1(dev(x), T, K, K, img, K // 32)
    W = synth.q4_0_weight(7041, N, K) if wtype == "q4_0" else synth.q8_0_weight(7041, N, K)
    y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    mmvq(img, K // 32, T, [qk.make_proj(wtype, pack_weight(W, wtype, N, K), N, K, y, N)], live=live_ptr(0))
    assert np.all(np.isnan(host(y)))
    assert qk.qk_device_faults() == 0
