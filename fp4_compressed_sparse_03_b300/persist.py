"""Persistent KV tier: a sequence's cache pages to a file (SSD or host memory) and back.

zaikei.co.jp article, opening section: the persistent KV cache that resumes sessions lives
on SSD or in host memory.  Tech-report digest (jiwasawa.github.io), "FP4 メイン KV Cache と
SWA Bounded Replay": the sliding-window KV is left out of it, so what persists is the
global cache: per Full group, the FP4 latent pages (codes and scales) and the indexer-key
pages.  The page records are packed and unpacked on the GPU by csa2_export_pages /
csa2_import_pages; this module only moves them between the device and a file.

File layout: a 64-byte header, then the records of the sequence's pages in logical order.
  header: magic b"CSA2PAGE", u32 version (1), u32 scale_row_bytes (32: E4M3 per 16
  channels, 16: MXFP4), u32 n_pages, i32 seq_len, u64 record_bytes, zero padding.
A sequence resumes into any free physical pages: load_sequence takes the page ids to fill.
"""
from __future__ import annotations

import struct

import numpy as np
import torch

from . import (PAGE, check, csa2_export_pages, csa2_import_pages, csa2_page_export_bytes,
               csa2_read_status)

MAGIC = b"CSA2PAGE"
VERSION = 1
HEADER_BYTES = 64
_HEADER = struct.Struct("<8sIIIiQ")


def pack_header(scale_row: int, n_pages: int, seq_len: int, record_bytes: int) -> bytes:
    h = _HEADER.pack(MAGIC, VERSION, scale_row, n_pages, seq_len, record_bytes)
    return h + bytes(HEADER_BYTES - len(h))


def unpack_header(buf: bytes):
    """(scale_row, n_pages, seq_len, record_bytes); raises ValueError on a foreign file."""
    magic, version, scale_row, n_pages, seq_len, record_bytes = _HEADER.unpack_from(buf, 0)
    if magic != MAGIC or version != VERSION:
        raise ValueError("not a CSA2 page file (magic or version mismatch)")
    if record_bytes != 64 * (256 + scale_row + 256):
        raise ValueError("page record size does not match the scale format")
    return scale_row, n_pages, seq_len, record_bytes


def persisted_bytes_per_token(n_full_groups: int = 1, mx: bool = False) -> int:
    """Bytes a token occupies in the persistent tier: per Full group, 256 B of codes, 32 B
    of E4M3 scales (16 B of E8M0 scales for MXFP4) and 256 B of bf16 indexer key."""
    return n_full_groups * (256 + (16 if mx else 32) + 256)


def footprint_report(tokens: int, n_full_groups: int = 1, mx: bool = False) -> dict:
    """Persistent-tier size of a session of `tokens` tokens (whole pages)."""
    pages = -(-tokens // PAGE)
    rec = csa2_page_export_bytes(16 if mx else 32)
    return {"tokens": tokens, "pages": pages, "bytes_per_token": persisted_bytes_per_token(n_full_groups, mx),
            "bytes": n_full_groups * pages * rec, "format": "mxfp4" if mx else "e4m3/16"}


def _scale_row(cache) -> int:
    return int(cache.scales.shape[-1])


def export_pages(cache, group: int, page_ids, stream=None) -> np.ndarray:
    """The packed records of `page_ids` (physical pages of Full group `group`), on the host."""
    ids = torch.as_tensor(np.asarray(page_ids, np.int32), device=cache.device)
    S = _scale_row(cache)
    rec = csa2_page_export_bytes(S)
    packed = torch.empty(max(1, ids.numel()) * rec, dtype=torch.uint8, device=cache.device)
    st = torch.zeros(1, dtype=torch.int32, device=cache.device)
    check(csa2_export_pages(cache.codes[group], cache.scales[group], cache.keys[group], S,
                            cache.num_pages, ids, ids.numel(), packed, st, stream), "export_pages")
    status, bits = csa2_read_status(st, stream)
    check(status, f"export_pages (device status {bits:#x})")
    return packed[: ids.numel() * rec].cpu().numpy()


def import_pages(cache, group: int, packed: np.ndarray, page_ids, stream=None) -> None:
    """Write packed records into the physical pages `page_ids` of Full group `group`."""
    ids = torch.as_tensor(np.asarray(page_ids, np.int32), device=cache.device)
    S = _scale_row(cache)
    if packed.size != ids.numel() * csa2_page_export_bytes(S):
        raise ValueError("packed size does not match the number of pages")
    host_packed = np.require(packed, np.uint8, ["C_CONTIGUOUS", "WRITEABLE"])
    dev_packed = torch.as_tensor(host_packed, device=cache.device)
    st = torch.zeros(1, dtype=torch.int32, device=cache.device)
    check(csa2_import_pages(dev_packed, S, ids, ids.numel(), cache.num_pages, cache.codes[group],
                            cache.scales[group], cache.keys[group], st, stream), "import_pages")
    status, bits = csa2_read_status(st, stream)
    check(status, f"import_pages (device status {bits:#x})")


def save_sequence(cache, group: int, seq: int, path: str) -> int:
    """Write sequence `seq`'s pages of Full group `group` to `path`; returns the bytes written."""
    seq_len = int(cache.seq_lens[seq].item())
    n_pages = -(-seq_len // PAGE)
    ids = cache.page_table[seq, :n_pages].cpu().numpy()
    data = export_pages(cache, group, ids)
    S = _scale_row(cache)
    with open(path, "wb") as f:
        f.write(pack_header(S, n_pages, seq_len, csa2_page_export_bytes(S)))
        f.write(data.tobytes())
    return HEADER_BYTES + data.size


def load_sequence(path: str, cache, group: int, page_ids) -> int:
    """Read a page file into the physical pages `page_ids` (one per saved page, in logical
    order) of Full group `group`; returns the saved sequence length."""
    with open(path, "rb") as f:
        head = f.read(HEADER_BYTES)
        scale_row, n_pages, seq_len, rec = unpack_header(head)
        if scale_row != _scale_row(cache):
            raise ValueError("the file's scale format differs from the cache's")
        if len(page_ids) != n_pages:
            raise ValueError(f"the file holds {n_pages} pages, {len(page_ids)} page ids given")
        data = np.frombuffer(f.read(n_pages * rec), dtype=np.uint8)
    if data.size != n_pages * rec:
        raise ValueError("truncated page file")
    import_pages(cache, group, data, page_ids)
    return seq_len
