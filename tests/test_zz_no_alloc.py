"""qk_mmvq_static_ws: the projection entry point for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc where they project: a
plugin that is handed only its input and output tensors (it owns no allocator
and may not keep memory between calls), or a latency-critical path that must
not touch the allocator (cudaMalloc can synchronise the device). For them qk_mmvq_static_ws runs the same kernels as
qk_mmvq, with the library's own fixed scratch array in place of a
caller-supplied workspace (the scratch holds the partial sums of row tiles
that several CTAs share, and their completion counters). This test calls it
through the C ABI twice in a row and checks both results against qk_mmvq with
an ordinary workspace, within the exact-path tolerance the other projection
tests use, on q/k/v and on an 8192 x 8192 projection whose launch shares row
tiles between CTAs through the scratch. It lives in its own
file, collected last, and passes both alone and after the other tests.
"""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import assert_exact_path

pytestmark = pytest.mark.gpu

NMSE_EXACT = 1e-10


@pytest.mark.parametrize("K,shapes", [(3584, [3584, 512, 512]),   # q, k, v reading one image
                                      (8192, [8192])])             # a launch that keeps partial sums in the scratch
def test_static_workspace_matches_workspace_entry_point_twice(K, shapes):
    import torch

    T = 8
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    x = synth.activations(9500 + K, T, K)
    img = torch.empty((T * (K // 32) * 36,), dtype=torch.uint8, device="cuda")
    qk.qk_quantize_q8_1(dev(x), T, K, K, img, K // 32)
    packed, ref_out, new_out = [], [], []
    for i, N in enumerate(shapes):
        nb = qk.qk_weight_packed_bytes("q4_0", N, K)
        w = torch.empty((nb,), dtype=torch.uint8, device="cuda")
        qk.qk_weight_pack("q4_0", dev(synth.q4_0_weight(9510 + i, N, K).reshape(-1)), N, K, w, nb)
        packed.append(w)
        ref_out.append(torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda"))
        new_out.append(torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda"))

    ref_projs = [qk.make_proj("q4_0", w, N, K, y, N) for w, N, y in zip(packed, shapes, ref_out)]
    ws_n = qk.qk_mmvq_workspace_bytes(ref_projs)
    ws = torch.zeros((ws_n,), dtype=torch.uint8, device="cuda")
    qk.qk_mmvq(img, K // 32, T, ref_projs, ws, ws_n)
    torch.cuda.synchronize()
    refs = [y.cpu().numpy() for y in ref_out]

    new_projs = [qk.make_proj("q4_0", w, N, K, y, N) for w, N, y in zip(packed, shapes, new_out)]
    for call in range(2):
        for y in new_out:
            y.fill_(float("nan"))
        qk.qk_mmvq_static_ws(img, K // 32, T, new_projs)
        torch.cuda.synchronize()
        for ref, y in zip(refs, new_out):
            got = y.cpu().numpy()
            assert not np.isnan(got).any(), f"call {call}: output not fully written"
            assert_exact_path(got, ref, NMSE_EXACT, what=f"call {call}")
    assert qk.qk_device_faults() == 0


def test_static_workspace_honours_a_device_live_row_count():
    """With a device live count below T, rows at or past it are left as they were and
    the live rows equal those of qk_mmvq with an ordinary workspace."""
    import torch

    T, K, N, live = 8, 2048, 1024, 5
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    img = torch.empty((T * (K // 32) * 36,), dtype=torch.uint8, device="cuda")
    qk.qk_quantize_q8_1(dev(synth.activations(9520, T, K)), T, K, K, img, K // 32)
    nb = qk.qk_weight_packed_bytes("q4_0", N, K)
    w = torch.empty((nb,), dtype=torch.uint8, device="cuda")
    qk.qk_weight_pack("q4_0", dev(synth.q4_0_weight(9521, N, K).reshape(-1)), N, K, w, nb)
    live_d = torch.tensor([live], dtype=torch.int32, device="cuda")
    ref = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    got = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    ref_p = [qk.make_proj("q4_0", w, N, K, ref, N)]
    ws_n = qk.qk_mmvq_workspace_bytes(ref_p)
    ws = torch.zeros((ws_n,), dtype=torch.uint8, device="cuda")
    qk.qk_mmvq(img, K // 32, T, ref_p, ws, ws_n, d_live_rows=live_d)
    qk.qk_mmvq_static_ws(img, K // 32, T, [qk.make_proj("q4_0", w, N, K, got, N)], d_live_rows=live_d)
    torch.cuda.synchronize()
    r, g = ref.cpu().numpy(), got.cpu().numpy()
    assert np.isnan(g[live:]).all()
    assert not np.isnan(g[:live]).any()
    assert_exact_path(g[:live], r[:live], NMSE_EXACT, what="live rows")
    assert qk.qk_device_faults() == 0


def test_static_workspace_refuses_oversized_problems():
    """A problem whose scratch need exceeds the static array is refused before any launch."""
    import torch

    big_N = 1 << 27                       # row tiles alone need more counters than the array holds
    # fake, never-dereferenced pointers far enough apart that the arguments pass every other check
    w, y, img = 1 << 36, 1 << 38, 1 << 12
    projs = [qk.make_proj("q4_0", w, big_N, 128, y, big_N)]
    with pytest.raises(qk.QkError) as e:
        qk.qk_mmvq_static_ws(img, 4, 8, projs, stream=torch.cuda.current_stream())
    assert e.value.name == "QK_ERR_UNSUPPORTED"
