"""Host logic of the persistent KV tier (no GPU): the page file header, the footprint
arithmetic and the C-ABI's argument checks."""
import ctypes

import pytest

import fp4_compressed_sparse_03_b300 as csa2
from fp4_compressed_sparse_03_b300 import persist


def test_header_round_trip_and_rejection():
    h = persist.pack_header(16, 5, 300, 64 * (256 + 16 + 256))
    assert len(h) == persist.HEADER_BYTES
    assert persist.unpack_header(h) == (16, 5, 300, 33792)
    with pytest.raises(ValueError):
        persist.unpack_header(b"NOTAFILE" + h[8:])
    with pytest.raises(ValueError):  # record size inconsistent with the scale format
        persist.unpack_header(persist.pack_header(32, 5, 300, 33792))


def test_footprint_arithmetic():
    # per Full group and token: 256 B codes + 32 B E4M3 scales (16 B E8M0) + 256 B key
    assert persist.persisted_bytes_per_token() == 544
    assert persist.persisted_bytes_per_token(mx=True) == 528
    assert persist.persisted_bytes_per_token(n_full_groups=5) == 5 * 544
    rep = persist.footprint_report(1_000_001)
    assert rep["pages"] == 15626 and rep["bytes"] == 15626 * 34816
    assert csa2.csa2_page_export_bytes(32) == 34816 and csa2.csa2_page_export_bytes(16) == 33792
    assert csa2.csa2_page_export_bytes(8) == 0


def test_page_copy_argument_checks():
    L = csa2._lib
    fake = 1 << 12
    assert L.csa2_export_pages(fake, fake, fake, 8, 4, fake, 1, fake, None, None) == \
        csa2.CSA2_ERR_UNSUPPORTED
    assert L.csa2_import_pages(fake, 32, fake, -1, 4, fake, fake, fake, None, None) == \
        csa2.CSA2_ERR_INVALID_ARGUMENT
    assert L.csa2_export_pages(None, None, None, 32, 4, None, 0, None, None, None) == csa2.CSA2_OK
    assert L.csa2_export_pages(fake + 8, fake, fake, 32, 4, fake, 1, fake, None, None) == \
        csa2.CSA2_ERR_INVALID_ARGUMENT  # misaligned pool
