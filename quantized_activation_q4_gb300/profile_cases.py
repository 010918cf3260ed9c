"""Named single-kernel cases for profiling the library under ncu.

    python -m quantized_activation_q4_gb300.profile_cases <case> [--reps N]

Each case builds its seeded inputs, runs the case's kernel `reps` times
through the C ABI (the first launches warm up) and synchronises, so that an
ncu capture of the last launch (`-k regex:<kernel> -s <reps-1> -c 1`) sees
one steady-state launch. With `--time N` it then times N more launches, one
by one with CUDA events on the current stream, each after a 512 MB write that
flushes the 129 MB L2 (so weights come from HBM), and prints the median
duration with the case's algorithmic bytes (or flops) per launch. Cases:

  mmvq_8192     qk_mmvq, Q4_0 8192x8192, T=8        (kernel mmvq_sk)
  mmvq_qkv      qk_mmvq, q/k/v 3584->3584/512/512   (kernel mmvq_sk)
  mmvq_down     qk_mmvq, Q4_0 18944->3584, T=8      (kernel mmvq_sk)
  rmsnorm       qk_rmsnorm_q8_1, [8, 3584] x w      (kernel rmsnorm_q8_1)
  quantize      qk_quantize_q8_1, [8, 8192]         (kernel quantize)
  glu           qk_glu_q8_1 SwiGLU packed [8, 18944] (kernel glu_q8_1)
  mmvq_id_<R>   qk_mmvq_id, gate+up 2560->768 over 128 experts, top-8 of R rows (kernel mmvq_id)
  mmvq_id_slots_<R>  qk_mmvq_id_slots, per-slot down 768->2560 over 128 experts, top-8 of R rows
                (one image row per pair; kernel mmvq_id)
  routed_<R>    the routed chain for R live rows of a 16/128 bucket: RMSNorm*w -> image, top-8 of
                128, plan, mmvq_id gate+up (kernels rmsnorm_q8_1, topk, plan, mmvq_id)
  mmq_qkv       qk_mmq, 3325 tokens, q/k/v          (kernels dequant_b, mmq_tc)
  quantize_q8_0 qk_quantize_q8_0, [3325, 3584]      (kernel quantize)
  rmsnorm_q8_0  qk_rmsnorm_q8_0, [3325, 3584] x w -> F32 + Q8_0 planes (kernel rmsnorm_q8_1)
"""
from __future__ import annotations

import argparse
import json
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


Q4_ROW_BYTES = 18          # one Q4_0 block of 32 weights
Q8_1_BLOCK = 36


def _mmvq_case(shapes, K, T=8):
    import torch
    keep, projs = [], []
    nbytes = sum(N * (K // 32) * Q4_ROW_BYTES + T * N * 4 for N in shapes) + T * (K // 32) * Q8_1_BLOCK
    for i, N in enumerate(shapes):
        w = _packed(10 + i, N, K)
        y = torch.empty((T, N), dtype=torch.float32, device="cuda")
        keep += [w, y]
        projs.append(qk.make_proj("q4_0", w, N, K, y, N))
    img = _image(T, K)
    n = qk.qk_mmvq_workspace_bytes(projs)
    ws = torch.zeros((n,), dtype=torch.uint8, device="cuda")
    keep += [img, ws]
    return lambda: qk.qk_mmvq(img, K // 32, T, projs, ws, n), keep, {"bytes": nbytes}


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
        nbytes = 2 * T * K * 4 + K * 4 + T * (K // 32) * Q8_1_BLOCK
        return (lambda: qk.qk_rmsnorm_q8_1(x, T, K, K, "mul", w, None, 1.0, 1e-6, y, K, img, K // 32),
                [x, w, y, img], {"bytes": nbytes})
    if name == "quantize":
        T, K = 8, 8192
        x = _dev(synth.activations(1, T, K))
        img = torch.empty((T * K // 32 * 36,), dtype=torch.uint8, device="cuda")
        return (lambda: qk.qk_quantize_q8_1(x, T, K, K, img, K // 32), [x, img],
                {"bytes": T * K * 4 + T * (K // 32) * Q8_1_BLOCK})
    if name == "glu":
        T, N = 8, 18944
        a = _dev(np.concatenate([synth.activations(1, T, N), synth.activations(2, T, N)], axis=1))
        out = torch.empty((T, N), dtype=torch.float32, device="cuda")
        img = torch.empty((T * N // 32 * 36,), dtype=torch.uint8, device="cuda")
        nbytes = 3 * T * N * 4 + T * (N // 32) * Q8_1_BLOCK
        return (lambda: qk.qk_glu_q8_1("swiglu", "packed", a, 2 * N, None, 0, T, N, out, N, img, N // 32),
                [a, out, img], {"bytes": nbytes})
    if name.startswith("mmvq_id_slots_"):
        # per-slot down projection of the 128-expert FFN: pair p reads image row p (768 columns)
        E, k, K, N, rows = 128, 8, 768, 2560, int(name.rsplit("_", 1)[1])
        per = qk.qk_weight_packed_bytes("q4_0", N, K)
        wd = torch.empty((E * per,), dtype=torch.uint8, device="cuda")
        for e in range(E):
            qk.qk_weight_pack("q4_0", _dev(synth.q4_0_weight(3000 + e, N, K).reshape(-1)), N, K,
                              wd[e * per:(e + 1) * per], per)
        img = _image(rows * k, K)
        ids = torch.empty((rows, k), dtype=torch.int32, device="cuda")
        wts = torch.empty((rows, k), dtype=torch.float32, device="cuda")
        qk.qk_topk_route(_dev(synth.router_logits(3, rows, E)), rows, E, k, ids, wts)
        counts = torch.empty((E,), dtype=torch.int32, device="cuda")
        offsets = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
        items = torch.empty((rows * k,), dtype=torch.int32, device="cuda")
        qk.qk_moe_plan(ids, rows, k, E, counts, offsets, items)
        y = torch.empty((rows * k, N), dtype=torch.float32, device="cuda")
        projs = [qk.make_proj_id("q4_0", E, wd, N, K, y)]
        live = int((counts > 0).sum().item())
        nbytes = live * per + rows * k * N * 4 + rows * k * (K // 32) * Q8_1_BLOCK
        return (lambda: qk.qk_mmvq_id_slots(img, K // 32, rows, k, projs, counts, offsets, items),
                [wd, img, ids, wts, counts, offsets, items, y], {"bytes": nbytes, "live_experts": live})
    if name.startswith("mmvq_id_"):
        E, k, K, NF, rows = 128, 8, 2560, 768, int(name.rsplit("_", 1)[1])
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
        live = int((counts > 0).sum().item())
        nbytes = 2 * live * NF * (K // 32) * Q4_ROW_BYTES + 2 * rows * k * NF * 4 + rows * (K // 32) * Q8_1_BLOCK
        return (lambda: qk.qk_mmvq_id(img, K // 32, rows, k, projs, counts, offsets, items), keep,
                {"bytes": nbytes, "live_experts": live})
    if name.startswith("routed_"):
        E, k, K, NF, live = 128, 8, 2560, 768, int(name.rsplit("_", 1)[1])
        bucket = 16 if live <= 16 else 128
        per = qk.qk_weight_packed_bytes("q4_0", NF, K)
        ws = []
        for p in range(2):
            buf = torch.empty((E * per,), dtype=torch.uint8, device="cuda")
            for e in range(E):
                qk.qk_weight_pack("q4_0", _dev(synth.q4_0_weight(1000 * p + e, NF, K).reshape(-1)), NF, K,
                                  buf[e * per:(e + 1) * per], per)
            ws.append(buf)
        x, w = _dev(synth.activations(5, bucket, K)), _dev(synth.norm_weight(6, K))
        y = torch.empty((bucket, K), dtype=torch.float32, device="cuda")
        img = torch.empty((bucket * (K // 32) * 36,), dtype=torch.uint8, device="cuda")
        logits = _dev(synth.router_logits(3, bucket, E))
        ids = torch.empty((bucket, k), dtype=torch.int32, device="cuda")
        wts = torch.empty((bucket, k), dtype=torch.float32, device="cuda")
        counts = torch.empty((E,), dtype=torch.int32, device="cuda")
        offsets = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
        items = torch.empty((bucket * k,), dtype=torch.int32, device="cuda")
        lv = torch.tensor([live], dtype=torch.int32, device="cuda")
        ys = [torch.empty((bucket * k, NF), dtype=torch.float32, device="cuda") for _ in range(2)]
        projs = [qk.make_proj_id("q4_0", E, ws[p], NF, K, ys[p]) for p in range(2)]

        def chain():
            qk.qk_rmsnorm_q8_1(x, bucket, K, K, "mul", w, None, 1.0, 1e-6, y, K, img, K // 32, d_live_rows=lv)
            qk.qk_topk_route(logits, bucket, E, k, ids, wts, d_live_rows=lv)
            qk.qk_moe_plan(ids, bucket, k, E, counts, offsets, items, d_live_rows=lv)
            qk.qk_mmvq_id(img, K // 32, bucket, k, projs, counts, offsets, items)

        chain()
        torch.cuda.synchronize()
        live_e = int((counts > 0).sum().item())
        keep = ws + ys + [x, w, y, img, logits, ids, wts, counts, offsets, items, lv]
        nbytes = 2 * live_e * per + 2 * bucket * k * NF * 4 + bucket * (K // 32) * Q8_1_BLOCK
        return chain, keep, {"bytes": nbytes, "live_experts": live_e}
    if name == "rmsnorm_q8_0":
        T, K, rb = 3325, 3584, 112
        x, w = _dev(synth.activations(4, T, K)), _dev(synth.norm_weight(2, K))
        y = torch.empty((T, K), dtype=torch.float32, device="cuda")
        qs = torch.empty((T * rb * 32,), dtype=torch.int8, device="cuda")
        d = torch.empty((T * rb,), dtype=torch.int16, device="cuda")
        nbytes = 2 * T * K * 4 + K * 4 + T * K + T * rb * 2
        return (lambda: qk.qk_rmsnorm_q8_0(x, T, K, K, "mul", w, None, 1.0, 1e-6, y, K, qs, d, rb),
                [x, w, y, qs, d], {"bytes": nbytes})
    if name in ("mmq_qkv", "quantize_q8_0"):
        T, K = 3325, 3584
        x = _dev(synth.activations(4, T, K))
        qs = torch.empty((T * 112 * 32,), dtype=torch.int8, device="cuda")
        d = torch.empty((T * 112,), dtype=torch.int16, device="cuda")
        quant = lambda: qk.qk_quantize_q8_0(x, T, K, K, qs, d, 112)
        if name == "quantize_q8_0":
            return quant, [x, qs, d], {"bytes": T * K * 4 + T * K + T * (K // 32) * 2}
        quant()
        keep, projs = [x, qs, d], []
        for i, N in enumerate((3584, 512, 512)):
            w = _packed(20 + i, N, K)
            y = torch.empty((T, N), dtype=torch.float32, device="cuda")
            keep += [w, y]
            projs.append(qk.make_proj("q4_0", w, N, K, y, N))
        n = qk.qk_mmq_workspace_bytes(T, projs)
        ws = torch.empty((n,), dtype=torch.uint8, device="cuda")
        keep.append(ws)
        return lambda: qk.qk_mmq(qs, d, 112, T, projs, ws, n), keep, {"flops": 2 * T * K * (3584 + 512 + 512)}
    raise SystemExit(f"unknown case {name!r}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--time", type=int, default=0, metavar="N")
    args = ap.parse_args()
    import torch
    qk.load(build_if_missing=True)
    run, keep, info = build_case(args.case)
    torch.cuda.synchronize()
    for _ in range(args.reps):
        run()
    torch.cuda.synchronize()
    faults = qk.qk_device_faults()
    if faults:
        raise SystemExit(f"device fault word {faults:#x}")
    print(f"{args.case}: {args.reps} launches ok")
    if args.time:
        flush = torch.empty((512 << 20,), dtype=torch.uint8, device="cuda")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.time)]
        for e0, e1 in ev:
            flush.fill_(1)
            e0.record()
            run()
            e1.record()
        torch.cuda.synchronize()
        us = float(np.median([e0.elapsed_time(e1) * 1e3 for e0, e1 in ev]))
        line = {"case": args.case, "median_us": round(us, 3), "launches": args.time, **info}
        if "bytes" in info:
            line["GB_per_s"] = round(info["bytes"] / us / 1e3, 1)
        if "flops" in info:
            line["TFLOP_per_s"] = round(info["flops"] / us / 1e6, 2)
        print(json.dumps(line))


if __name__ == "__main__":
    main()
