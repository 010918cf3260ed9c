"""Named single-kernel cases for profiling the library under ncu.

    python -m quantized_activation_q4_gb300.profile_cases <case> [--reps N]

Each case builds its seeded inputs, runs the case's kernel `reps` times
through the C ABI (the first launches warm up) and synchronises, so that an
ncu capture of the last launch (`-k regex:<kernel> -s <reps-1> -c 1`) sees
one steady-state launch. Cases:

  mmvq_8192     qk_mmvq, Q4_0 8192x8192, T=8        (kernel mmvq_sk)
  mmvq_qkv      qk_mmvq, q/k/v 3584->3584/512/512   (kernel mmvq_sk)
  mmvq_down     qk_mmvq, Q4_0 18944->3584, T=8      (kernel mmvq_sk)
  rmsnorm       qk_rmsnorm_q8_1, [8, 3584] x w      (kernel rmsnorm_q8_1)
  quantize      qk_quantize_q8_1, [8, 8192]         (kernel quantize)
  glu           qk_glu_q8_1 SwiGLU packed [8, 18944] (kernel glu_q8_1)
  mmvq_id       qk_mmvq_id, 128 experts, top-8, live 128 rows (kernel mmvq_id)
  mmq_qkv       qk_mmq, 3325 tokens, q/k/v          (kernel mmq)
  quantize_q8_0 qk_quantize_q8_0, [3325, 3584]      (kernel quantize)
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from quantized_activation_q4_gb300 import binding as qk  # noqa: E402
from quantized_activation_q4_gb300 import synth  # noqa: E402


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _packed(seed, N, K):
    import torch
    nb = qk.qk_weight_packed_bytes("q4_0", N, K)
    w = torch.empty((nb,), dtype=torch.uint8, device="cuda")
    qk.qk_weight_pack("q4_0", _dev(synth.q4_0_weight(seed, N, K).reshape(-1)), N, K, w, nb)
    return w


def _image(T, K, seed=2):
    import torch
    img = torch.empty((T * (K // 32) * 36,), dtype=torch.uint8, device="cuda")
    qk.qk_quantize_q8_1(_dev(synth.activations(seed, T, K)), T, K, K, img, K // 32)
    return img


def _mmvq_case(shapes, K, T=8):
    import torch
    keep, projs = [], []
    for i, N in enumerate(shapes):
        w = _packed(10 + i, N, K)
        y = torch.empty((T, N), dtype=torch.float32, device="cuda")
        keep += [w, y]
        projs.append(qk.make_proj("q4_0", w, N, K, y, N))
    img = _image(T, K)
    n = qk.qk_mmvq_workspace_bytes(projs)
    ws = torch.zeros((n,), dtype=torch.uint8, device="cuda")
    keep += [img, ws]
    return lambda: qk.qk_mmvq(img, K // 32, T, projs, ws, n), keep


def build_case(name):
    import torch
    if name == "mmvq_8192":
        return _mmvq_case([8192], 8192)
    if name == "mmvq_qkv":
        return _mmvq_case([3584, 512, 512], 3584)
    if name == "mmvq_down":
        return _mmvq_case([3584], 18944)
    if name == "rmsnorm":
        T, K = 8, 3584
        x, w = _dev(synth.activations(1, T, K)), _dev(synth.norm_weight(2, K))
        y = torch.empty((T, K), dtype=torch.float32, device="cuda")
        img = torch.empty((T * K // 32 * 36,), dtype=torch.uint8, device="cuda")
        return lambda: qk.qk_rmsnorm_q8_1(x, T, K, K, "mul", w, None, 1.0, 1e-6, y, K, img, K // 32), [x, w, y, img]
    if name == "quantize":
        T, K = 8, 8192
        x = _dev(synth.activations(1, T, K))
        img = torch.empty((T * K // 32 * 36,), dtype=torch.uint8, device="cuda")
        return lambda: qk.qk_quantize_q8_1(x, T, K, K, img, K // 32), [x, img]
    if name == "glu":
        T, N = 8, 18944
        a = _dev(np.concatenate([synth.activations(1, T, N), synth.activations(2, T, N)], axis=1))
        out = torch.empty((T, N), dtype=torch.float32, device="cuda")
        img = torch.empty((T * N // 32 * 36,), dtype=torch.uint8, device="cuda")
        return lambda: qk.qk_glu_q8_1("swiglu", "packed", a, 2 * N, None, 0, T, N, out, N, img, N // 32), [a, out, img]
    if name == "mmvq_id":
        E, k, K, NF, rows = 128, 8, 2560, 768, 128
        per = qk.qk_weight_packed_bytes("q4_0", NF, K)
        ws = []
        for p in range(2):
            buf = torch.empty((E * per,), dtype=torch.uint8, device="cuda")
            for e in range(E):
                qk.qk_weight_pack("q4_0", _dev(synth.q4_0_weight(1000 * p + e, NF, K).reshape(-1)), NF, K,
                                  buf[e * per:(e + 1) * per], per)
            ws.append(buf)
        img = _image(rows, K)
        ids = torch.empty((rows, k), dtype=torch.int32, device="cuda")
        wts = torch.empty((rows, k), dtype=torch.float32, device="cuda")
        qk.qk_topk_route(_dev(synth.router_logits(3, rows, E)), rows, E, k, ids, wts)
        counts = torch.empty((E,), dtype=torch.int32, device="cuda")
        offsets = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
        items = torch.empty((rows * k,), dtype=torch.int32, device="cuda")
        qk.qk_moe_plan(ids, rows, k, E, counts, offsets, items)
        ys = [torch.empty((rows * k, NF), dtype=torch.float32, device="cuda") for _ in range(2)]
        projs = [qk.make_proj_id("q4_0", E, ws[p], NF, K, ys[p]) for p in range(2)]
        keep = ws + ys + [img, ids, wts, counts, offsets, items]
        return lambda: qk.qk_mmvq_id(img, K // 32, rows, k, projs, counts, offsets, items), keep
    if name in ("mmq_qkv", "quantize_q8_0"):
        T, K = 3325, 3584
        x = _dev(synth.activations(4, T, K))
        qs = torch.empty((T * 112 * 32,), dtype=torch.int8, device="cuda")
        d = torch.empty((T * 112,), dtype=torch.int16, device="cuda")
        quant = lambda: qk.qk_quantize_q8_0(x, T, K, K, qs, d, 112)
        if name == "quantize_q8_0":
            return quant, [x, qs, d]
        quant()
        keep, projs = [x, qs, d], []
        for i, N in enumerate((3584, 512, 512)):
            w = _packed(20 + i, N, K)
            y = torch.empty((T, N), dtype=torch.float32, device="cuda")
            keep += [w, y]
            projs.append(qk.make_proj("q4_0", w, N, K, y, N))
        return lambda: qk.qk_mmq(qs, d, 112, T, projs), keep
    raise SystemExit(f"unknown case {name!r}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=4)
    args = ap.parse_args()
    import torch
    qk.load(build_if_missing=True)
    run, keep = build_case(args.case)
    torch.cuda.synchronize()
    for _ in range(args.reps):
        run()
    torch.cuda.synchronize()
    faults = qk.qk_device_faults()
    if faults:
        raise SystemExit(f"device fault word {faults:#x}")
    print(f"{args.case}: {args.reps} launches ok")


if __name__ == "__main__":
    main()
