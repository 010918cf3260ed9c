"""GPU: the consecutive-window image memo (minfer doc 52, "r49 A-quantize prepass shared-A
dedup", sections 2-3). Within a window of GEMMs that read one activation, the memo quantises it
once; a hit enqueues nothing and the planes it keeps are byte-identical to a fresh quantisation
(the quantiser is a pure function of its key). The memo cannot see writes to the source: the
caller's two clearing rules (any other node, every synchronisation) are what make a hit safe,
and the last case shows the stale hit they exist to prevent."""
import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

T, K, RB = 300, 512, 16


def planes():
    import torch
    return (torch.zeros((T * RB * 32,), dtype=torch.int8, device="cuda"),
            torch.zeros((T * RB,), dtype=torch.int16, device="cuda"))


def fresh_q8_0(x):
    qs, d = planes()
    qk.qk_quantize_q8_0(x, T, K, K, qs, d, RB)
    return host(qs), host(d)


def test_memo_quantises_once_per_window_and_hits_are_byte_identical():
    x = dev(synth.activations(5100, T, K))
    qs, d = planes()
    m = qk.qk_image_memo()
    n0 = qk.launch_count()
    hits = [qk.qk_image_memo_quantize_q8_0(m, x, T, K, K, qs, d, RB) for _ in range(3)]   # q, k, v
    assert hits == [False, True, True]
    assert qk.launch_count() - n0 == 1
    rq, rd = fresh_q8_0(x)
    assert np.array_equal(host(qs), rq) and np.array_equal(host(d), rd)
    oq, od = O.quantize_q8_0(host(x), row_blocks=RB)
    assert np.array_equal(host(qs).view(np.int8).reshape(T, -1), oq)
    assert np.array_equal(host(d).view(np.uint16).reshape(T, -1), od)


def test_memo_misses_on_any_other_key_and_after_a_clear():
    import torch
    x = dev(synth.activations(5200, T, K))
    x2 = dev(synth.activations(5201, T, K))
    qs, d = planes()
    qs2, d2 = planes()
    m = qk.qk_image_memo()
    assert not qk.qk_image_memo_quantize_q8_0(m, x, T, K, K, qs, d, RB)
    assert not qk.qk_image_memo_quantize_q8_0(m, x2, T, K, K, qs, d, RB)       # other source pointer
    assert np.array_equal(host(qs), fresh_q8_0(x2)[0])
    assert not qk.qk_image_memo_quantize_q8_0(m, x2, T, K, K, qs2, d2, RB)     # other planes
    assert not qk.qk_image_memo_quantize_q8_0(m, x2, T - 1, K, K, qs2, d2, RB)  # other T
    assert not qk.qk_image_memo_quantize_q8_0(m, x2, T - 1, K - 32, K, qs2, d2, RB)   # other K
    s = torch.cuda.Stream()
    assert not qk.qk_image_memo_quantize_q8_0(m, x2, T - 1, K - 32, K, qs2, d2, RB, stream=s)   # other stream
    torch.cuda.synchronize()
    # rule 1: a node that is not one of the window's GEMMs (here: it rewrites x) clears first
    qk.qk_image_memo_clear(m)
    assert not qk.qk_image_memo_quantize_q8_0(m, x, T, K, K, qs, d, RB)
    x.copy_(x2)
    qk.qk_image_memo_clear(m)
    assert not qk.qk_image_memo_quantize_q8_0(m, x, T, K, K, qs, d, RB)
    assert np.array_equal(host(qs), fresh_q8_0(x2)[0])


def test_memo_q8_1_image_and_forms_do_not_mix():
    import torch
    x = dev(synth.activations(5300, 8, K))
    img = torch.zeros((8 * RB * 36,), dtype=torch.uint8, device="cuda")
    m = qk.qk_image_memo()
    n0 = qk.launch_count()
    assert [qk.qk_image_memo_quantize_q8_1(m, x, 8, K, K, img, RB) for _ in range(3)] == [False, True, True]
    assert qk.launch_count() - n0 == 1
    assert np.array_equal(host(img).reshape(8, -1), O.quantize_q8_1(host(x)))
    qs = torch.zeros((8 * RB * 32,), dtype=torch.int8, device="cuda")
    d = torch.zeros((8 * RB,), dtype=torch.int16, device="cuda")
    assert not qk.qk_image_memo_quantize_q8_0(m, x, 8, K, K, qs, d, RB)   # a Q8_1 record never serves Q8_0


def test_memo_cannot_see_writes_which_is_why_the_caller_clears():
    """The failure the clearing rules prevent: x rewritten with no clear in between, and the
    memo still hits, so the planes keep the old activation's image."""
    x = dev(synth.activations(5400, T, K))
    x_new = dev(synth.activations(5401, T, K))
    qs, d = planes()
    m = qk.qk_image_memo()
    assert not qk.qk_image_memo_quantize_q8_0(m, x, T, K, K, qs, d, RB)
    old = host(qs).copy()
    x.copy_(x_new)                                                   # no clear: a broken caller
    assert qk.qk_image_memo_quantize_q8_0(m, x, T, K, K, qs, d, RB)   # stale hit
    assert np.array_equal(host(qs), old) and not np.array_equal(host(qs), fresh_q8_0(x_new)[0])
