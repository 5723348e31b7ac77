"""ctypes wrapper of libcsa2_inputs: the generator of gen.py in C (host threads) and
CUDA (device).  Bit-identical to the numpy definition; faster for large inputs."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import gen

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "gen.cu")
LIB = os.path.join(HERE, "libcsa2_inputs.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        subprocess.check_call([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                               "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fopenmp",
                               "-o", LIB, SRC, "-lgomp"])
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        L.csa2g_fill_bf16_host.argtypes = [u64, u64, i64, ctypes.c_int, vp]
        L.csa2g_fill_latent_host.argtypes = [u64, i64, i64, vp, vp]
        L.csa2g_fill_normal_host.argtypes = [u64, u64, i64, vp]
        L.csa2g_fill_bf16_dev.argtypes = [u64, u64, i64, ctypes.c_int, vp, vp]
        L.csa2g_fill_latent_dev.argtypes = [u64, i64, i64, vp, vp, vp]
        L.csa2g_fill_keys_paged_dev.argtypes = [vp, vp, vp, ctypes.c_int32, ctypes.c_int32, vp, vp]
        for f in ("csa2g_fill_bf16_dev", "csa2g_fill_latent_dev", "csa2g_fill_keys_paged_dev"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


# ------------------------------------------------------------------ host ----------

def normal_bf16_host(key: int, i0: int, n: int, pow2: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint16)
    lib().csa2g_fill_bf16_host(key, i0, n, pow2, out.ctypes.data)
    return out


def normal_host(key: int, i0: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().csa2g_fill_normal_host(key, i0, n, out.ctypes.data)
    return out


def key_rows_host(seed: int, group: int, seq: int, t0: int, n: int) -> np.ndarray:
    """Same values as gen.key_rows(seed, group, seq, arange(t0, t0 + n))."""
    key = gen.stream_key(seed, gen.TAG_KEY, (group << 24) | seq)
    return normal_bf16_host(key, t0 * gen.D_IDX, n * gen.D_IDX).reshape(n, gen.D_IDX)


def latent_rows_host(seed: int, group: int, seq: int, t0: int, n: int, gains: np.ndarray) -> np.ndarray:
    """Same values as gen.latent_rows(seed, group, seq, arange(t0, t0 + n), gains)."""
    key = gen.stream_key(seed, gen.TAG_LATENT, (group << 24) | seq)
    g = np.ascontiguousarray(gains, np.float32)
    out = np.empty((n, gen.D_KV), np.float32)
    lib().csa2g_fill_latent_host(key, t0, n, g.ctypes.data, out.ctypes.data)
    return out


# ------------------------------------------------------------------ device --------

def _stream(stream):
    import torch
    return (stream or torch.cuda.current_stream()).cuda_stream


def _ok(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed with CUDA error {rc}")


def fill_bf16_dev(out, key: int, i0: int, pow2: int = 0, stream=None):
    """out (int16/bf16 tensor, contiguous) <- bf16(normal(key, i0 + i) * 2**pow2)."""
    _ok(lib().csa2g_fill_bf16_dev(key, i0, out.numel(), pow2, out.data_ptr(), _stream(stream)),
        "fill_bf16_dev")


def fill_latent_dev(out, key: int, t0: int, gains_dev, stream=None):
    """out float32 [T, 512] <- latent rows t0 .. t0 + T of the stream."""
    _ok(lib().csa2g_fill_latent_dev(key, t0, out.shape[0], gains_dev.data_ptr(), out.data_ptr(),
                                    _stream(stream)), "fill_latent_dev")


def fill_keys_paged_dev(pool, seq_keys_dev, seq_lens_dev, page_table_dev, stream=None):
    """pool int16 [num_pages*64, 128] <- every sequence's indexer keys at their slots."""
    _ok(lib().csa2g_fill_keys_paged_dev(seq_keys_dev.data_ptr(), seq_lens_dev.data_ptr(),
                                        page_table_dev.data_ptr(), page_table_dev.shape[1],
                                        page_table_dev.shape[0], pool.data_ptr(), _stream(stream)),
        "fill_keys_paged_dev")


def seq_keys(seed: int, tag: int, group: int, num_seqs: int) -> np.ndarray:
    """Stream keys of every sequence (uint64), for the paged device fill."""
    return np.array([gen.stream_key(seed, tag, (group << 24) | b) for b in range(num_seqs)],
                    dtype=np.uint64)


# ------------------------------------------------------------------ queries -------

def layer_queries_host(wl: "gen.DecodeWorkload", layer: int):
    """(q_idx bf16 bits [num_q, 4, 128], q bf16 bits [num_q, 16, 512]) of one layer."""
    nq = wl.num_q
    q_idx = np.empty((nq, gen.H_IDX, gen.D_IDX), np.uint16)
    q = np.empty((nq, gen.H_Q, gen.D_KV), np.uint16)
    for i in range(nq):
        kq = gen.stream_key(wl.seed, gen.TAG_QIDX, (layer << 24) | i)
        q_idx[i] = normal_bf16_host(kq, 0, gen.H_IDX * gen.D_IDX).reshape(gen.H_IDX, gen.D_IDX)
        ka = gen.stream_key(wl.seed, gen.TAG_Q, (layer << 24) | i)
        q[i] = normal_bf16_host(ka, 0, gen.H_Q * gen.D_KV).reshape(gen.H_Q, gen.D_KV)
    return q_idx, q


def all_queries_host(wl: "gen.DecodeWorkload"):
    """Stacked per-layer queries: q_idx [L, num_q, 4, 128], q [L, num_q, 16, 512] (bf16 bits)."""
    qs = [layer_queries_host(wl, l) for l in range(len(wl.schedule))]
    return np.stack([a for a, _ in qs]), np.stack([b for _, b in qs])
