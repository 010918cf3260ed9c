"""Device-side helpers for the GPU parity tests (allocation and copies only)."""
from __future__ import annotations

import numpy as np

from quantized_activation_q4_gb300 import binding as qk


def dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def empty_u8(n: int, fill: int = 0xA5):
    import torch
    return torch.full((n,), fill, dtype=torch.uint8, device="cuda")


def live_ptr(n: int):
    import torch
    return torch.tensor([n], dtype=torch.int32, device="cuda")


def pack_weight(W: np.ndarray, wtype: str, N: int, K: int):
    """Canonical blocks (host) -> packed device weights via qk_weight_pack."""
    import torch
    nbytes = qk.qk_weight_packed_bytes(wtype, N, K)
    src = dev(W.reshape(-1))
    packed = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
    qk.qk_weight_pack(wtype, src, N, K, packed, nbytes)
    return packed


def pack_experts(Ws: list[np.ndarray], wtype: str, N: int, K: int):
    """E experts' canonical blocks -> one buffer, expert e at e * packed_bytes."""
    import torch
    per = qk.qk_weight_packed_bytes(wtype, N, K)
    out = torch.empty((len(Ws) * per,), dtype=torch.uint8, device="cuda")
    for e, W in enumerate(Ws):
        qk.qk_weight_pack(wtype, dev(W.reshape(-1)), N, K, out[e * per:(e + 1) * per], per)
    return out


_WS = {}


def workspace(projs):
    """A qk_mmvq workspace, zeroed once when first made and then reused by every
    later call of the same size (the library keeps its counters at zero)."""
    import torch
    n = max(16, qk.qk_mmvq_workspace_bytes(projs))
    if n not in _WS:
        _WS[n] = torch.zeros((n,), dtype=torch.uint8, device="cuda")
    return _WS[n], n


def mmvq(img, rb, T, projs, live=None):
    ws, n = workspace(projs)
    qk.qk_mmvq(img, rb, T, projs, ws, n, live)
    return ws


def assert_exact_path(got, exact, nmse_max=1e-10, rel_max=1e-5, what=""):
    """A GPU projection against the oracle's exact quantised path, as a whole and element by element.

    Whole output: NMSE <= nmse_max. Every element: |got - exact| <= rel_max * max|exact|. Only
    binary32 summation order separates the exact block paths from the oracle (about 2^-24 times
    the square root of the block count, relative), so 1e-5 of the largest output leaves a margin
    of more than 20x at K = 18944; a dropped, doubled or misplaced block moves an element by about
    max|exact| / (4 sqrt(blocks)), hundreds of times the bound."""
    from oracle import oracle as O
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    assert got.shape == exact.shape, what
    assert O.nmse(got, exact) <= nmse_max, f"{what}: NMSE {O.nmse(got, exact):.3e}"
    if exact.size:
        bound = rel_max * float(np.max(np.abs(exact)))
        worst = float(np.max(np.abs(got - exact)))
        assert worst <= bound, f"{what}: element off by {worst:.3e} > {bound:.3e}"
