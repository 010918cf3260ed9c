"""The failure path on the GPU without faulting it: every wait in the kernels is bounded, and a
wait that runs out sets bit 0 of the device fault word and lets its kernel return. A one-CTA
self-test waits on a shared-memory barrier that nothing completes; the host must see the bit,
and the same context must then run a projection correctly with a clean fault word."""
import time

import numpy as np
import pytest

from oracle import oracle as O
from quantized_activation_q4_gb300 import binding as qk
from quantized_activation_q4_gb300 import synth
from tests.gpu_helpers import dev, empty_u8, host, mmvq, pack_weight

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    import torch
    assert qk.qk_device_faults() == 0            # clean before
    t0 = time.perf_counter()
    qk.qk_selftest_wait_timeout()
    faults = qk.qk_device_faults()               # synchronises
    dt = time.perf_counter() - t0
    assert faults & 1
    assert dt < 10.0
    assert qk.qk_device_faults() == 0            # reading cleared it

    T, N, K = 4, 256, 512
    x = synth.activations(8100, T, K)
    W = synth.q4_0_weight(8101, N, K)
    img = empty_u8(T * (K // 32) * 36, 0)
    qk.qk_quantize_q8_1(dev(x), T, K, K, img, K // 32)
    y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    packed = pack_weight(W, "q4_0", N, K)        # kept alive: the descriptor holds a raw pointer
    mmvq(img, K // 32, T, [qk.make_proj("q4_0", packed, N, K, y, N)], None)
    got = host(y)
    assert qk.qk_device_faults() == 0
    exact = O.proj_q8_1("q4_0", W, N, K, host(img).reshape(T, -1), K // 32)
    assert O.nmse(got, exact) <= 1e-10
