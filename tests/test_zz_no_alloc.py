"""csa2_sparse_attn_static (split partials in the library's fixed device array) against
csa2_sparse_attn (caller workspace): identical outputs on consecutive calls, and the
size limit is refused on the host.  Kept in its own file, collected last, so that it
runs both alone in a fresh process and after every other test."""
import numpy as np
import pytest
import torch

import csa2_inputs as gen
import fp4_compressed_sparse_03_b300 as csa2
from fp4_compressed_sparse_03_b300.workload import fill_decode_cache

pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1.0 / np.sqrt(512.0)))


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


def test_static_scratch_matches_workspace_on_consecutive_calls():
    lens = np.array([3000, 100, 5000], np.int32)
    wl = gen.DecodeWorkload("noalloc", 41, lens, np.ones(3, np.int32), [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl)
    q_seq = _dev(np.array([0, 1, 2], np.int32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, topk in enumerate([2048, 2048, 256]):   # two multi-split calls in a row, then one more
        assert csa2.csa2_attn_workspace_size(3, topk) <= csa2.ATTN_STATIC_SCRATCH_BYTES
        idx = np.stack([gen.random_index_set(41, 1000 * call + i, int(lens[i]), topk,
                                             n_invalid=3 * i) for i in range(3)])
        q = np.stack([gen.q_rows(41, call, np.array([i]))[0] for i in range(3)])
        qd, idxd = _dev(q), _dev(idx)
        out_ws = torch.full((3, 16, 512), np.nan, dtype=torch.float32, device="cuda")
        lse_ws = torch.full((3, 16), np.nan, dtype=torch.float32, device="cuda")
        out_st = torch.full_like(out_ws, np.nan)
        lse_st = torch.full_like(lse_ws, np.nan)
        ws = torch.empty(max(csa2.csa2_attn_workspace_size(3, topk), 16), dtype=torch.uint8,
                         device="cuda")
        csa2.check(csa2.csa2_sparse_attn(qd, cache.codes[0], cache.scales[0], idxd, cache.pages,
                                         out_ws, lse_ws, 3, q_seq, topk, SCALE, ws, None, st), "ws")
        csa2.check(csa2.csa2_sparse_attn_static(qd, cache.codes[0], cache.scales[0], idxd,
                                                cache.pages, out_st, lse_st, 3, q_seq, topk,
                                                SCALE, st), "static")
        torch.cuda.synchronize()
        assert torch.equal(out_ws, out_st), f"call {call}"
        assert torch.equal(lse_ws, lse_st), f"call {call}"
        assert not torch.isnan(out_st).any()
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)


def test_static_scratch_rejects_oversized_requests():
    # 8 queries over 65536 selected entries need at least 128 splits (512 entries each) of
    # 16 x 512 fp32 partials: 32.1 MiB, over the 16 MiB array.  Refused before any device
    # work.
    assert csa2.csa2_attn_workspace_size(8, 65536) > csa2.ATTN_STATIC_SCRATCH_BYTES
    pages = csa2.Csa2Pages(1, None, None, 1, 1, 64)
    assert csa2.csa2_sparse_attn_static(None, None, None, None, pages, None, None, 8, None, 65536,
                                        SCALE) == csa2.CSA2_ERR_UNSUPPORTED
