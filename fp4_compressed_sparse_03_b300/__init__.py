"""Python binding of libcsa2, the B300 (sm_103a) CSA2 FP4 compressed global KV cache.

Argument marshalling only: every step runs in the library's CUDA kernels.  The
functions keep the C ABI's names and argument order (see include/csa2.h); tensors
are torch CUDA tensors (their data pointers are passed), sizes are Python ints.
If libcsa2.so is missing the import fails: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

CSA2_OK, CSA2_ERR_INVALID_ARGUMENT, CSA2_ERR_UNSUPPORTED = 0, 1, 2
CSA2_ERR_CUDA, CSA2_ERR_DEVICE_FAULT, CSA2_ERR_TIMEOUT = 3, 4, 5
CSA2_FULL, CSA2_REINDEX, CSA2_REUSE = 0, 1, 2
CSA2_DEV_BAD_INDEX, CSA2_DEV_BAD_PAGE, CSA2_DEV_BAD_SLOT = 0x1, 0x2, 0x4
CSA2_DEV_TIMEOUT, CSA2_DEV_BAD_QSEQ = 0x8, 0x10

PAGE = 64
D_KV = 512
D_IDX = 128
H_IDX = 4
H_Q = 16

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libcsa2.so not found at {LIB_PATH}; build it with "
        "`python fp4_compressed_sparse_03_b300/build.py` (nvcc, sm_103a). "
        "There is no CPU fallback.")

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class Csa2Pages(ctypes.Structure):
    _fields_ = [("num_seqs", _i32), ("seq_lens", _vp), ("page_table", _vp),
                ("max_pages_per_seq", _i32), ("num_pages", _i32), ("page_size", _i32)]


class Csa2IndexArgs(ctypes.Structure):
    _fields_ = [("num_q", _i32), ("q_seq", _vp), ("max_q_per_seq", _i32), ("pool_size", _i32),
                ("inherit_idx", _vp), ("workspace", _vp), ("workspace_bytes", _sz),
                ("dev_status", _vp)]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_kv_write = _sig("csa2_kv_write", ctypes.c_int,
                 [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i64, _vp, _vp])
_index = _sig("csa2_index", ctypes.c_int,
              [ctypes.c_int, _vp, _vp, _vp, _i32, _vp, ctypes.POINTER(Csa2Pages),
               ctypes.POINTER(Csa2IndexArgs), _vp])
_index_ws = _sig("csa2_index_workspace_size", _sz, [ctypes.c_int, _i32, _i32, _i32])
_attn = _sig("csa2_sparse_attn", ctypes.c_int,
             [_vp, _vp, _vp, _vp, ctypes.POINTER(Csa2Pages), _vp, _vp, _i32, _vp, _i32,
              ctypes.c_float, _vp, _sz, _vp, _vp])
_attn_mx = _sig("csa2_sparse_attn_mx", ctypes.c_int,
                [_vp, _vp, _vp, _vp, ctypes.POINTER(Csa2Pages), _vp, _vp, _i32, _vp, _i32,
                 ctypes.c_float, _vp, _sz, _vp, _vp])
_attn_ws = _sig("csa2_attn_workspace_size", _sz, [_i32, _i32])
_attn_static = _sig("csa2_sparse_attn_static", ctypes.c_int,
                    [_vp, _vp, _vp, _vp, ctypes.POINTER(Csa2Pages), _vp, _vp, _i32, _vp, _i32,
                     ctypes.c_float, _vp, _vp])
ATTN_STATIC_SCRATCH_BYTES = 16 << 20  # CSA2_ATTN_STATIC_SCRATCH_BYTES
ATTN_MAX_TOPK = 65536  # CSA2_ATTN_MAX_TOPK
_attn_chunked = _sig("csa2_sparse_attn_chunked", ctypes.c_int,
                     [_vp, _vp, _vp, _vp, ctypes.POINTER(Csa2Pages), _vp, _vp, _i32, _vp, _i32,
                      _i32, ctypes.c_float, _vp, _sz, _vp, _vp])
_chunk_ws = _sig("csa2_chunk_attn_workspace_size", _sz, [_i32, _i32, _i32])
CHUNK_ATTN_MAX_UNION = 8192  # CSA2_CHUNK_ATTN_MAX_UNION
_quantize = _sig("csa2_quantize", ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp])
_dequantize = _sig("csa2_dequantize", ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp])
_quantize_mx = _sig("csa2_quantize_mx", ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp])
_dequantize_mx = _sig("csa2_dequantize_mx", ctypes.c_int,
                      [_vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp])
_page_bytes = _sig("csa2_page_export_bytes", _sz, [_i32])
_export_pages = _sig("csa2_export_pages", ctypes.c_int,
                     [_vp, _vp, _vp, _i32, _i64, _vp, _i32, _vp, _vp, _vp])
_import_pages = _sig("csa2_import_pages", ctypes.c_int,
                     [_vp, _i32, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp])
_read_status = _sig("csa2_read_status", ctypes.c_int, [_vp, ctypes.POINTER(_i32), _vp])
_check_wait = _sig("csa2_check_bounded_wait", ctypes.c_int, [_i32, ctypes.c_uint32, _vp, _vp])
_status_string = _sig("csa2_status_string", ctypes.c_char_p, [ctypes.c_int])
_version = _sig("csa2_version", _i32, [])


class Csa2Error(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def status_string(status: int) -> str:
    return _status_string(status).decode()


def version() -> int:
    return int(_version())


def _ptr(t):
    """Data pointer of a tensor (or an int address), None for None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int, where: str = "csa2") -> None:
    if status != CSA2_OK:
        raise Csa2Error(status, where)


def make_pages(seq_lens, page_table, num_pages: int, page_size: int = PAGE) -> Csa2Pages:
    """Pages descriptor over device tensors seq_lens [B] and page_table [B, max_pages]."""
    return Csa2Pages(int(seq_lens.shape[0]), _ptr(seq_lens), _ptr(page_table),
                     int(page_table.shape[1]), int(num_pages), int(page_size))


def make_index_args(num_q: int, q_seq, max_q_per_seq: int = 1, pool_size: int = 0,
                    inherit_idx=None, workspace=None, workspace_bytes: int | None = None,
                    dev_status=None) -> Csa2IndexArgs:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return Csa2IndexArgs(int(num_q), _ptr(q_seq), int(max_q_per_seq), int(pool_size),
                         _ptr(inherit_idx), _ptr(workspace), int(workspace_bytes), _ptr(dev_status))


# ---------------------------------------------------------------- C ABI calls -----

def csa2_kv_write(H, Wt, codes, scales, k_idx, T, d_model, n_kv_proj, n_idx_proj, slot_of_token,
                  num_slots, dev_status=None, stream=None) -> int:
    return _kv_write(_ptr(H), _ptr(Wt), _ptr(codes), _ptr(scales), _ptr(k_idx), T, d_model,
                     n_kv_proj, n_idx_proj, _ptr(slot_of_token), num_slots, _ptr(dev_status),
                     _stream(stream))


def csa2_index(mode, q_idx, k_idx, pool, topk, out_idx, pages: Csa2Pages, args: Csa2IndexArgs,
               stream=None) -> int:
    return _index(mode, _ptr(q_idx), _ptr(k_idx), _ptr(pool), topk, _ptr(out_idx),
                  ctypes.byref(pages), ctypes.byref(args), _stream(stream))


def csa2_index_workspace_size(mode, num_q, max_pages_per_seq, pool_size) -> int:
    return int(_index_ws(mode, num_q, max_pages_per_seq, pool_size))


def csa2_sparse_attn(q, codes, scales, idx, pages: Csa2Pages, out, lse, num_q, q_seq, topk,
                     softmax_scale, workspace=None, workspace_bytes=None, dev_status=None,
                     stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _attn(_ptr(q), _ptr(codes), _ptr(scales), _ptr(idx), ctypes.byref(pages), _ptr(out),
                 _ptr(lse), num_q, _ptr(q_seq), topk, ctypes.c_float(softmax_scale),
                 _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream(stream))


def csa2_attn_workspace_size(num_q, topk) -> int:
    return int(_attn_ws(num_q, topk))


def csa2_sparse_attn_chunked(q, codes, scales, idx, pages: Csa2Pages, out, lse, num_q, q_seq,
                             chunk, topk, softmax_scale, workspace=None, workspace_bytes=None,
                             dev_status=None, stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _attn_chunked(_ptr(q), _ptr(codes), _ptr(scales), _ptr(idx), ctypes.byref(pages),
                         _ptr(out), _ptr(lse), num_q, _ptr(q_seq), chunk, topk,
                         ctypes.c_float(softmax_scale), _ptr(workspace), workspace_bytes,
                         _ptr(dev_status), _stream(stream))


def csa2_chunk_attn_workspace_size(num_q, chunk, topk) -> int:
    return int(_chunk_ws(num_q, chunk, topk))


def csa2_sparse_attn_static(q, codes, scales, idx, pages: Csa2Pages, out, lse, num_q, q_seq, topk,
                            softmax_scale, dev_status=None, stream=None) -> int:
    return _attn_static(_ptr(q), _ptr(codes), _ptr(scales), _ptr(idx), ctypes.byref(pages),
                        _ptr(out), _ptr(lse), num_q, _ptr(q_seq), topk,
                        ctypes.c_float(softmax_scale), _ptr(dev_status), _stream(stream))


def csa2_sparse_attn_mx(q, codes, scales, idx, pages: Csa2Pages, out, lse, num_q, q_seq, topk,
                        softmax_scale, workspace=None, workspace_bytes=None, dev_status=None,
                        stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _attn_mx(_ptr(q), _ptr(codes), _ptr(scales), _ptr(idx), ctypes.byref(pages), _ptr(out),
                    _ptr(lse), num_q, _ptr(q_seq), topk, ctypes.c_float(softmax_scale),
                    _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream(stream))


def csa2_quantize(x, slot_of_token, codes, scales, T, D, num_slots, dev_status=None,
                  stream=None) -> int:
    return _quantize(_ptr(x), _ptr(slot_of_token), _ptr(codes), _ptr(scales), T, D, num_slots,
                     _ptr(dev_status), _stream(stream))


def csa2_dequantize(codes, scales, slot_of_token, x, T, D, num_slots, dev_status=None,
                    stream=None) -> int:
    return _dequantize(_ptr(codes), _ptr(scales), _ptr(slot_of_token), _ptr(x), T, D, num_slots,
                       _ptr(dev_status), _stream(stream))


def csa2_quantize_mx(x, slot_of_token, codes, scales, T, D, num_slots, dev_status=None,
                     stream=None) -> int:
    return _quantize_mx(_ptr(x), _ptr(slot_of_token), _ptr(codes), _ptr(scales), T, D, num_slots,
                        _ptr(dev_status), _stream(stream))


def csa2_dequantize_mx(codes, scales, slot_of_token, x, T, D, num_slots, dev_status=None,
                       stream=None) -> int:
    return _dequantize_mx(_ptr(codes), _ptr(scales), _ptr(slot_of_token), _ptr(x), T, D,
                          num_slots, _ptr(dev_status), _stream(stream))


def csa2_page_export_bytes(scale_row_bytes: int) -> int:
    return int(_page_bytes(scale_row_bytes))


def csa2_export_pages(codes, scales, keys, scale_row_bytes, num_pages, page_ids, n_pages, packed,
                      dev_status=None, stream=None) -> int:
    return _export_pages(_ptr(codes), _ptr(scales), _ptr(keys), scale_row_bytes, num_pages,
                         _ptr(page_ids), n_pages, _ptr(packed), _ptr(dev_status), _stream(stream))


def csa2_import_pages(packed, scale_row_bytes, page_ids, n_pages, num_pages, codes, scales, keys,
                      dev_status=None, stream=None) -> int:
    return _import_pages(_ptr(packed), scale_row_bytes, _ptr(page_ids), n_pages, num_pages,
                         _ptr(codes), _ptr(scales), _ptr(keys), _ptr(dev_status), _stream(stream))


def csa2_read_status(dev_status, stream=None):
    """Returns (status, bits)."""
    bits = _i32(0)
    st = _read_status(_ptr(dev_status), ctypes.byref(bits), _stream(stream))
    return int(st), int(bits.value)


def csa2_check_bounded_wait(arrive, limit, dev_status, stream=None) -> int:
    return _check_wait(1 if arrive else 0, limit, _ptr(dev_status), _stream(stream))


from .decode import DecodeCache, DecodeStep  # noqa: E402,F401
