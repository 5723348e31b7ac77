"""CPU oracle for the CSA2 FP4 compressed global KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``fp4_compressed_sparse_03_b300`` / ``libcsa2``) never imports it, and the two
share no code: the arithmetic lives in plain C (``csa2_oracle.c``); this module
only marshals numpy arrays and composes the per-mode steps in the order the pages
give them (tech-report digest, "Compressed Sparse Attention 2 (CSA2)": Full, Reindex and Reuse
modes and the Hierarchical Sparse Indexer).

Every function is plain and slow; floating-point sums are in double.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_quantize_rows.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _u8p, _u8p]
        L.orc_dequantize_rows.argtypes = [_u8p, _u8p, ctypes.c_int64, ctypes.c_int32, _f64p]
        L.orc_project_rows.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _f32p]
        L.orc_index_scores.argtypes = [_u16p, _u16p, ctypes.c_int64, _f64p]
        L.orc_select_topk.argtypes = [_f64p, _i32p, ctypes.c_int64, ctypes.c_int32, _i32p]
        L.orc_sparse_attention.argtypes = [_u16p, _f64p, ctypes.c_int64, ctypes.c_float, _f32p, _f32p]
        L.orc_e2m1_encode_array.argtypes = [_f32p, ctypes.c_int64, _u8p]
        L.orc_e8m0_scale_for.restype = ctypes.c_uint8
        L.orc_e8m0_scale_for.argtypes = [ctypes.c_float]
        L.orc_e8m0_decode.restype = ctypes.c_double
        L.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.orc_mx_quantize_rows.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _u8p, _u8p]
        L.orc_mx_dequantize_rows.argtypes = [_u8p, _u8p, ctypes.c_int64, ctypes.c_int32, _f64p]
        L.orc_e4m3_encode_array.argtypes = [_f32p, ctypes.c_int64, _u8p]
        _lib = L
    return _lib


def _p(a: np.ndarray, ptype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ptype)


# ------------------------------------------------------------------- codec -------

def e2m1_encode(y) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32).ravel()
    out = np.empty(y.size, np.uint8)
    lib().orc_e2m1_encode_array(_p(y, _f32p), y.size, _p(out, _u8p))
    return out


def e2m1_decode(codes) -> np.ndarray:
    return np.array([lib().orc_e2m1_decode(int(c)) for c in np.ravel(codes)], dtype=np.float64)


def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e4m3_encode_array(_p(v, _f32p), v.size, _p(out, _u8p))
    return out


def e4m3_decode(b) -> np.ndarray:
    return np.array([lib().orc_e4m3_decode(int(c)) for c in np.ravel(b)], dtype=np.float64)


def quantize(x: np.ndarray):
    """fp32 [T, D] -> (codes u8 [T, D/2], scales u8 [T, D/16])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, D = x.shape
    assert D % 16 == 0
    codes = np.zeros((T, D // 2), np.uint8)
    scales = np.zeros((T, D // 16), np.uint8)
    lib().orc_quantize_rows(_p(x, _f32p), T, D, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    T, half = codes.shape
    out = np.empty((T, half * 2), np.float64)
    lib().orc_dequantize_rows(_p(codes, _u8p), _p(scales, _u8p), T, half * 2, _p(out, _f64p))
    return out


# -------------------------------------------------------------- MXFP4 variant --
# Tech-report digest, "FP4 メイン KV Cache と SWA Bounded Replay" (OCP-standard MXFP4,
# E2M1 elements), read as OCP MX: E8M0 scale per 32 channels (see csa2_oracle.c).

def e8m0_scale_for(amax: float) -> int:
    return int(lib().orc_e8m0_scale_for(float(amax)))


def e8m0_decode(b) -> np.ndarray:
    return np.array([lib().orc_e8m0_decode(int(c)) for c in np.ravel(b)], dtype=np.float64)


def mx_quantize(x: np.ndarray):
    """fp32 [T, D] -> (codes u8 [T, D/2], E8M0 scales u8 [T, D/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, D = x.shape
    assert D % 32 == 0
    codes = np.zeros((T, D // 2), np.uint8)
    scales = np.zeros((T, D // 32), np.uint8)
    lib().orc_mx_quantize_rows(_p(x, _f32p), T, D, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def mx_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    T, half = codes.shape
    out = np.empty((T, half * 2), np.float64)
    lib().orc_mx_dequantize_rows(_p(codes, _u8p), _p(scales, _u8p), T, half * 2, _p(out, _f64p))
    return out


# ------------------------------------------------------------------- write path --

def project(H: np.ndarray, Wt: np.ndarray) -> np.ndarray:
    """fp32 C = H . W with double accumulation; H bf16 bits [R, d], Wt bf16 bits [n, d]."""
    H = np.ascontiguousarray(H, dtype=np.uint16)
    Wt = np.ascontiguousarray(Wt, dtype=np.uint16)
    R, d = H.shape
    n = Wt.shape[0]
    C = np.empty((R, n), np.float32)
    lib().orc_project_rows(_p(H, _u16p), _p(Wt, _u16p), R, d, n, _p(C, _f32p))
    return C


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bits (the indexer-key store)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def kv_write_rows(H: np.ndarray, Wt: np.ndarray, n_kv_proj: int, n_idx_proj: int):
    """Write path for some token rows (tech-report digest CED equation, ezic blog FP4 format).

    Returns (codes [n_kv_proj, R, 256], scales [n_kv_proj, R, 32], keys [n_idx_proj, R, 128]).
    The pre-quantisation value is the float32 of the double-accumulated product.
    """
    C = project(H, Wt)
    R = C.shape[0]
    codes = np.empty((n_kv_proj, R, 256), np.uint8)
    scales = np.empty((n_kv_proj, R, 32), np.uint8)
    for p in range(n_kv_proj):
        codes[p], scales[p] = quantize(C[:, p * 512:(p + 1) * 512])
    keys = np.empty((n_idx_proj, R, 128), np.uint16)
    base = n_kv_proj * 512
    for p in range(n_idx_proj):
        keys[p] = f32_to_bf16_bits(C[:, base + p * 128: base + (p + 1) * 128])
    return codes, scales, keys, C


# ------------------------------------------------------------------- indexer -----

def index_scores(q_idx: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Double scores of one query (bf16 bits [4, 128]) against keys (bf16 bits [n, 128])."""
    q_idx = np.ascontiguousarray(q_idx, dtype=np.uint16)
    keys = np.ascontiguousarray(keys, dtype=np.uint16)
    n = keys.shape[0]
    out = np.empty(n, np.float64)
    lib().orc_index_scores(_p(q_idx, _u16p), _p(keys, _u16p), n, _p(out, _f64p))
    return out


def select_topk(scores: np.ndarray, tokens: np.ndarray, k: int) -> np.ndarray:
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.empty(k, np.int32)
    lib().orc_select_topk(_p(scores, _f64p), _p(tokens, _i32p), scores.size, k, _p(out, _i32p))
    return out


def index_full(q_idx: np.ndarray, keys: np.ndarray, topk: int, pool_size: int):
    """Full mode (tech-report digest "Full Mode"; pool: "Hierarchical Sparse Indexer").

    Scores every context token; the pool is the top-min(P, N) and the selection the
    top-min(K, N) by (score desc, token asc), both ascending and -1 padded.
    Returns (idx [K], pool [P] or None, scores [N]).
    """
    s = index_scores(q_idx, keys)
    tok = np.arange(keys.shape[0], dtype=np.int32)
    idx = select_topk(s, tok, topk)
    pool = select_topk(s, tok, pool_size) if pool_size > 0 else None
    return idx, pool, s


def index_reindex(q_idx: np.ndarray, keys: np.ndarray, pool: np.ndarray, topk: int):
    """Reindex mode (tech-report digest "Reindex Mode" + "Hierarchical Sparse Indexer"): re-score
    only the valid entries of the pool with this layer's query and the keys of the
    Full layer; keep the top-min(K, |pool|).  Returns (idx [K], scores of the pool)."""
    valid = pool[pool >= 0].astype(np.int32)
    s = index_scores(q_idx, keys[valid])
    return select_topk(s, valid, topk), s


def index_reuse(inherit_idx: np.ndarray) -> np.ndarray:
    """Reuse mode (tech-report digest "Reuse Mode"): the indices of the earlier layer, unchanged."""
    return np.array(inherit_idx, dtype=np.int32, copy=True)


# ------------------------------------------------------------------- attention ---

def sparse_attention(q: np.ndarray, chat: np.ndarray, softmax_scale: float):
    """q bf16 bits [16, 512]; chat float64 [n, 512] (already dequantised rows).
    Returns (out float32 [16, 512], lse float32 [16])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    chat = np.ascontiguousarray(chat, dtype=np.float64)
    n = chat.shape[0]
    out = np.empty((16, 512), np.float32)
    lse = np.empty(16, np.float32)
    lib().orc_sparse_attention(_p(q, _u16p), _p(chat, _f64p), n, ctypes.c_float(softmax_scale),
                               _p(out, _f32p), _p(lse, _f32p))
    return out, lse


def attention_over_cache(q: np.ndarray, codes_rows: np.ndarray, scales_rows: np.ndarray,
                         idx: np.ndarray, softmax_scale: float, mx: bool = False):
    """Gather the selected rows (codes/scales given per logical token of the sequence),
    dequantise them (E4M3 / 16, or the MXFP4 variant with `mx`), attend.  -1 entries of
    idx are skipped."""
    sel = idx[idx >= 0]
    deq = mx_dequantize if mx else dequantize
    chat = deq(codes_rows[sel], scales_rows[sel]) if sel.size else np.zeros((0, 512))
    return sparse_attention(q, chat, softmax_scale)


# ------------------------------------------------------------- persistent tier ---
# zaikei article, opening section: the persistent KV cache that resumes sessions lives on
# SSD or in host memory; tech-report digest, "FP4 メイン KV Cache と SWA Bounded Replay":
# the sliding-window KV is left out of it, so the persisted state is the global cache.
# One record per page: the codes of its 64 slots, then their scales, then their keys
# (bf16, little-endian bytes).

def pack_pages(codes: np.ndarray, scales: np.ndarray, keys: np.ndarray, page_ids) -> np.ndarray:
    """codes u8 [slots, 256], scales u8 [slots, S], keys u16 [slots, 128] -> the records of
    `page_ids`, back to back (a page id outside the pool gives a zero record)."""
    S = scales.shape[1]
    rec = 64 * (256 + S + 256)
    n_pages = codes.shape[0] // 64
    out = []
    for pg in np.asarray(page_ids).ravel():
        pg = int(pg)
        if pg < 0 or pg >= n_pages:
            out.append(np.zeros(rec, np.uint8))
            continue
        rows = slice(64 * pg, 64 * pg + 64)
        out.append(np.concatenate([codes[rows].ravel(), scales[rows].ravel(),
                                   np.ascontiguousarray(keys[rows], dtype="<u2").view(np.uint8).ravel()]))
    return np.concatenate(out) if out else np.zeros(0, np.uint8)


# ------------------------------------------------------------------- footprint ---

PAGES_FOOTPRINT = {
    # zaikei article "CSA2とFP4でキャッシュを圧縮": HBM-resident global KV bytes per token
    "v4.1-flash": 890,
    "v4-flash": 3514,
    "v3.2": 48068,
    "v1": 389120,
}


def layout_bytes_per_token(n_full_groups: int = 1, d_kv: int = 512, group: int = 16,
                           d_idx: int = 128, key_bytes: int = 2) -> int:
    """Bytes per token that this layout keeps in HBM: per Full group, FP4 codes
    (d_kv / 2), E4M3 scales (d_kv / group) and bf16 indexer keys (d_idx * 2)."""
    return n_full_groups * (d_kv // 2 + d_kv // group + d_idx * key_bytes)


def session_bytes(bytes_per_token: int, tokens: int = 1_000_000) -> int:
    """Cache bytes of one session (ezic blog: 890 B x 1M tokens ~ 890 MB)."""
    return bytes_per_token * tokens
