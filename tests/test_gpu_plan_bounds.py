"""GPU: the routed projection reads its plan without trusting it. Counts, offsets and items that
did not come from qk_moe_plan give unspecified outputs, but every read stays inside counts,
offsets, items, the image and the weights: counts are clamped to [0, rows * k], item positions
outside items and pairs outside the bucket are skipped, and a total of passes that no plan of the
bucket can have stops the launch before any work (bit 1 of the fault word). Every index below was
checked against those rules by reading the kernel; nothing here can address memory outside the
buffers."""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import assert_exact_path, dev, empty_u8, host, pack_experts

pytestmark = pytest.mark.gpu

E, N, K, ROWS, TOPK = 4, 128, 256, 8, 8
RB = K // 32
SENT = np.float32(-777.25)


def _setup():
    import torch
    Ws = [synth.q4_0_weight(9100 + e, N, K) for e in range(E)]
    pw = pack_experts(Ws, "q4_0", N, K)
    x = synth.activations(9110, ROWS, K)
    img = empty_u8(ROWS * RB * 36)
    qk.qk_quantize_q8_1(dev(x), ROWS, K, K, img, RB)
    y = torch.full((ROWS * TOPK, N), float(SENT), dtype=torch.float32, device="cuda")
    return Ws, pw, img, y


def _run(pw, img, y, counts, offsets, items, per_pair=False):
    fn = qk.qk_mmvq_id_slots if per_pair else qk.qk_mmvq_id
    rows_img = ROWS * TOPK if per_pair else ROWS
    assert img.numel() >= rows_img * RB * 36
    fn(img, RB, ROWS, TOPK, [qk.make_proj_id("q4_0", E, pw, N, K, y)], dev(np.asarray(counts, np.int32)),
       dev(np.asarray(offsets, np.int32)), dev(np.asarray(items, np.int32)))
    return host(y)


def test_counts_no_plan_can_have_stop_the_launch():
    Ws, pw, img, y = _setup()
    qk.qk_device_faults()                                  # start from a clear word
    # every count far above rows * k: clamped to 64 each, 8 passes each, 32 in all, more than
    # ceil(64 / 8) + 4 = 12 that any plan of this bucket has
    got = _run(pw, img, y, [1000, 2**30, 70, 65], [0, 0, 0, 0, 0], np.arange(ROWS * TOPK))
    assert np.all(got == SENT)
    assert qk.qk_device_faults() == 2


def test_out_of_range_positions_and_pairs_are_skipped():
    Ws, pw, img, y = _setup()
    qk.qk_device_faults()
    items = np.full(ROWS * TOPK, 5, np.int32)
    items[60:64] = [3, 70, -2, 10]          # 70 is past the bucket's 64 pairs, -2 is no pair
    # expert 0: positions 60..67, of which 64..67 lie past items; expert 1: positions -5..-3;
    # expert 2: no pairs; expert 3: positions 1000.. (all past items)
    got = _run(pw, img, y, [8, 3, 0, 5], [60, -5, 0, 1000, 0], items)
    assert qk.qk_device_faults() == 0
    img_h = host(img).reshape(ROWS, -1)
    ref = O.proj_q8_1("q4_0", Ws[0], N, K, img_h[[3 // TOPK, 10 // TOPK]], RB)
    assert_exact_path(got[[3, 10]], ref, what="pairs 3 and 10 of expert 0")
    untouched = np.ones(ROWS * TOPK, bool)
    untouched[[3, 10]] = False
    assert np.all(got[untouched] == SENT)


def test_per_pair_mode_skips_the_same_way():
    import torch
    Ws, pw, _, y = _setup()
    xp = synth.activations(9120, ROWS * TOPK, K)
    imgp = empty_u8(ROWS * TOPK * RB * 36)
    qk.qk_quantize_q8_1(dev(xp), ROWS * TOPK, K, K, imgp, RB)
    qk.qk_device_faults()
    items = np.full(ROWS * TOPK, 5, np.int32)
    items[0:4] = [63, 64, -1, 0]
    got = _run(pw, imgp, y, [4, 0, 2**31 - 1, -9], [0, 0, 2**31 - 1, -(2**31), 0], items, per_pair=True)
    assert qk.qk_device_faults() == 0
    imgp_h = host(imgp).reshape(ROWS * TOPK, -1)
    ref = O.proj_q8_1("q4_0", Ws[0], N, K, imgp_h[[63, 0]], RB)
    assert_exact_path(got[[63, 0]], ref, what="pairs 63 and 0 of expert 0, own image rows")
    untouched = np.ones(ROWS * TOPK, bool)
    untouched[[63, 0]] = False
    assert np.all(got[untouched] == SENT)
    del torch
