"""Persistent KV tier on the GPU: page export / import through the C ABI, bit-exact against
the oracle's record layout (zaikei article: the persistent cache lives on SSD or in host
memory; digest "FP4 メイン KV Cache と SWA Bounded Replay": it holds the global cache)."""
import os

import numpy as np
import pytest
import torch

import csa2_inputs as gen
import fp4_compressed_sparse_03_b300 as csa2
import oracle
from fp4_compressed_sparse_03_b300 import persist
from fp4_compressed_sparse_03_b300.decode import DecodeCache
from fp4_compressed_sparse_03_b300.workload import fill_decode_cache
from gpu_common import SOFTMAX_SCALE, dev, host

pytestmark = pytest.mark.gpu


def _cache(mx=False):
    lens = np.array([1000, 150, 4096], np.int32)
    wl = gen.DecodeWorkload("pages", 43, lens, np.ones(3, np.int32), [gen.FULL], 0, 16)
    return wl, fill_decode_cache(wl, mx=mx)


@pytest.mark.parametrize("mx", [False, True])
def test_export_matches_oracle_layout_and_import_restores_pages(mx):
    wl, cache = _cache(mx)
    S = int(cache.scales.shape[-1])
    ids = np.array([5, 0, cache.num_pages - 1, 17, cache.num_pages + 3, 2], np.int32)  # one bad id
    n = len(ids)
    rec = csa2.csa2_page_export_bytes(S)
    packed = torch.full((n * rec,), 0xAB, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_export_pages(cache.codes[0], cache.scales[0], cache.keys[0], S,
                                      cache.num_pages, dev(ids), n, packed, st), "export")
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_ERR_DEVICE_FAULT and bits & csa2.CSA2_DEV_BAD_PAGE
    codes, scales = host(cache.codes[0]), host(cache.scales[0])
    keys = host(cache.keys[0]).view(np.uint16)
    expect = oracle.pack_pages(codes, scales, keys, ids)
    assert np.array_equal(host(packed), expect)
    # import into a fresh pool at other pages: each destination page equals its source
    dst = DecodeCache(host(cache.seq_lens), host(cache.page_table), cache.num_pages, 1, mx=mx)
    to = np.array([9, 3, 1, 40, 0, cache.num_pages + 1], np.int32)  # the bad record goes nowhere
    csa2.check(csa2.csa2_import_pages(packed, S, dev(to), n, dst.num_pages, dst.codes[0],
                                      dst.scales[0], dst.keys[0], st), "import")
    status, bits = csa2.csa2_read_status(st)
    assert bits & csa2.CSA2_DEV_BAD_PAGE
    dc, ds, dk = host(dst.codes[0]), host(dst.scales[0]), host(dst.keys[0]).view(np.uint16)
    for src_pg, dst_pg in zip(ids[:4], to[:4]):
        a, b = slice(64 * src_pg, 64 * src_pg + 64), slice(64 * dst_pg, 64 * dst_pg + 64)
        assert np.array_equal(dc[b], codes[a]) and np.array_equal(ds[b], scales[a])
        assert np.array_equal(dk[b], keys[a])
    # the zero record of the bad id was imported as page 0
    assert not dc[:64].any() and not ds[:64].any() and not dk[:64].any()


def test_saved_sequence_resumes_in_other_pages(tmp_path):
    """A sequence saved to a file and loaded into a cache with a different page table gives
    the same attention output, bit for bit."""
    wl, cache = _cache()
    seq = 2
    path = os.path.join(tmp_path, "seq.csa2pages")
    nbytes = persist.save_sequence(cache, 0, seq, path)
    n_pages = 4096 // 64
    assert nbytes == persist.HEADER_BYTES + n_pages * csa2.csa2_page_export_bytes(32)
    pool = n_pages + 7
    pt = np.random.default_rng(3).permutation(pool)[:n_pages].astype(np.int32).reshape(1, -1)
    dst = DecodeCache(np.array([4096], np.int32), pt, pool, 1)
    assert persist.load_sequence(path, dst, 0, pt[0]) == 4096
    idx = gen.random_index_set(43, 7, 4096, 1024).reshape(1, -1)
    q = gen.q_rows(43, 1, np.array([0]))
    outs = []
    for c, qs in ((cache, seq), (dst, 0)):
        out = torch.zeros((1, 16, 512), dtype=torch.float32, device="cuda")
        lse = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(csa2.csa2_attn_workspace_size(1, 1024), 16), dtype=torch.uint8,
                         device="cuda")
        csa2.check(csa2.csa2_sparse_attn(dev(q), c.codes[0], c.scales[0], dev(idx), c.pages, out,
                                         lse, 1, dev(np.array([qs], np.int32)), 1024,
                                         SOFTMAX_SCALE, ws), "attn")
        outs.append((host(out), host(lse)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_mx_pages_round_trip_through_a_file(tmp_path):
    """MXFP4 pools (16-byte scale rows) save and load like E4M3 ones: the resumed pages are
    byte-identical to the saved ones."""
    wl, cache = _cache(mx=True)
    path = os.path.join(tmp_path, "seq_mx.csa2pages")
    persist.save_sequence(cache, 0, 0, path)
    n_pages = -(-1000 // 64)
    pt = np.arange(5, 5 + n_pages, dtype=np.int32).reshape(1, -1)
    dst = DecodeCache(np.array([1000], np.int32), pt, 5 + n_pages, 1, mx=True)
    assert persist.load_sequence(path, dst, 0, pt[0]) == 1000
    src_ids = host(cache.page_table)[0, :n_pages]
    for a, b in zip(src_ids, pt[0]):
        ra, rb = slice(64 * a, 64 * a + 64), slice(64 * b, 64 * b + 64)
        assert torch.equal(cache.codes[0][ra], dst.codes[0][rb])
        assert torch.equal(cache.scales[0][ra], dst.scales[0][rb])
        assert torch.equal(cache.keys[0][ra], dst.keys[0][rb])
    with pytest.raises(ValueError):  # an E4M3 cache refuses an MXFP4 file
        persist.load_sequence(path, DecodeCache(np.array([1000], np.int32), pt, 5 + n_pages, 1),
                              0, pt[0])
