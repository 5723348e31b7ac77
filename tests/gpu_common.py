"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs the oracle)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import fp4_compressed_sparse_03_b300 as csa2
import oracle

DEV = "cuda"
SOFTMAX_SCALE = float(np.float32(1.0 / np.sqrt(512.0)))
ATTN_REL_TOL = 2e-3      # max |out_gpu - out_oracle| <= 2e-3 * RMS(out_oracle), per query
TIE_REL_TOL = 1e-5       # top-K sets equal except ties within 1e-5 * max(1, |s_K|)

_pool = ThreadPoolExecutor(max_workers=os.cpu_count() or 4)


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    if a.dtype == np.uint64:
        a = a.view(np.int64)
    return torch.from_numpy(a).to(DEV)


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def oracle_quantize_parallel(x: np.ndarray):
    """The oracle's block quantiser over row chunks on all host cores (ctypes releases
    the GIL); identical results to one call."""
    T = x.shape[0]
    parts = np.array_split(np.arange(T), min(T, 4 * (os.cpu_count() or 4)))
    res = list(_pool.map(lambda r: oracle.quantize(x[r[0]:r[-1] + 1]) if len(r) else None, parts))
    res = [r for r in res if r is not None]
    return np.concatenate([c for c, _ in res]), np.concatenate([s for _, s in res])


def gpu_quantize(x: torch.Tensor):
    T, D = x.shape
    slots = torch.arange(T, dtype=torch.int32, device=x.device)
    codes = torch.zeros((T, D // 2), dtype=torch.uint8, device=x.device)
    scales = torch.zeros((T, D // 16), dtype=torch.uint8, device=x.device)
    csa2.check(csa2.csa2_quantize(x, slots, codes, scales, T, D, T), "csa2_quantize")
    return codes, scales


def assert_topk_close(got: np.ndarray, want: np.ndarray, score_of, what: str = ""):
    """Index sets must be equal except for candidates whose oracle score ties the
    boundary score (the smallest selected oracle score) within the tolerance."""
    g = set(int(v) for v in got if v >= 0)
    w = set(int(v) for v in want if v >= 0)
    assert len(g) == len(w), f"{what}: {len(g)} selected vs {len(w)}"
    assert np.all(np.diff(got[got >= 0]) > 0), f"{what}: output not strictly ascending"
    assert np.all(got[len(g):] == -1), f"{what}: padding is not -1"
    if g == w:
        return 0
    kth = min(score_of(t) for t in w)
    tol = TIE_REL_TOL * max(1.0, abs(kth))
    for t in g ^ w:
        assert abs(score_of(t) - kth) <= tol, \
            f"{what}: token {t} score {score_of(t)!r} vs boundary {kth!r}"
    return len(g ^ w)


def assert_attn_close(out_g: np.ndarray, out_o: np.ndarray, lse_g=None, lse_o=None, what=""):
    rms = float(np.sqrt(np.mean(out_o.astype(np.float64) ** 2)))
    err = float(np.max(np.abs(out_g.astype(np.float64) - out_o)))
    assert err <= ATTN_REL_TOL * max(rms, 1e-30), f"{what}: max err {err} vs rms {rms}"
    if lse_g is not None:
        fin = np.isfinite(lse_o)
        assert np.array_equal(np.isfinite(lse_g), fin), f"{what}: lse finiteness differs"
        assert np.max(np.abs(lse_g[fin] - lse_o[fin]), initial=0.0) <= 1e-4 * max(
            1.0, float(np.max(np.abs(lse_o[fin]), initial=1.0))), f"{what}: lse differs"
