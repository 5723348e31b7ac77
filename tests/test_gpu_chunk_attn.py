"""Multi-query sparse attention in dense-contraction form (csa2_sparse_attn_chunked): each
query of a chunk against the oracle over its own selection, and against the per-query CUDA
path on the same arguments.

A chunk is up to four queries of one sequence with their own top-K entries: the draft
tokens of a decode step (tech-report digest, jiwasawa.github.io, DSpark item under
"さらなるアーキテクチャ拡張技術"; per-query selection: "Hierarchical Sparse Indexer") or
consecutive positions of a prefill chunk; attention over each query's selected FP4 rows
(digest "Reuse Mode"; zaikei.co.jp article, "CSA2とFP4でキャッシュを圧縮").  Outputs within
2e-3 x RMS per query, lse within 1e-4."""
import numpy as np
import pytest
import torch

import csa2_inputs as gen
import fp4_compressed_sparse_03_b300 as csa2
import oracle
from fp4_compressed_sparse_03_b300.workload import fill_decode_cache
from gpu_common import SOFTMAX_SCALE, assert_attn_close, dev, host

pytestmark = pytest.mark.gpu


def _cache(seed, lens):
    lens = np.asarray(lens, np.int32)
    wl = gen.DecodeWorkload("chunk", seed, lens, np.ones(len(lens), np.int32), [gen.FULL], 0, 16)
    return fill_decode_cache(wl)


def _chunked(cache, q, idx, q_seq, chunk, topk, st=None):
    nq = len(q_seq)
    out = torch.full((nq, 16, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((nq, 16), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(csa2.csa2_chunk_attn_workspace_size(nq, chunk, topk), dtype=torch.uint8,
                     device="cuda")
    if st is None:
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_sparse_attn_chunked(dev(q), cache.codes[0], cache.scales[0], dev(idx),
                                             cache.pages, out, lse, nq, dev(q_seq), chunk, topk,
                                             SOFTMAX_SCALE, ws, None, st), "chunked attention")
    return host(out), host(lse), st


def _per_query(cache, q, idx, q_seq, topk):
    nq = len(q_seq)
    out = torch.zeros((nq, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((nq, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(nq, topk), 16), dtype=torch.uint8, device="cuda")
    csa2.check(csa2.csa2_sparse_attn(dev(q), cache.codes[0], cache.scales[0], dev(idx), cache.pages,
                                     out, lse, nq, dev(q_seq), topk, SOFTMAX_SCALE, ws), "attention")
    return host(out), host(lse)


def _oracle(seed, b, sel, q):
    sel = sel[sel >= 0]
    if sel.size == 0:
        return oracle.sparse_attention(q, np.zeros((0, 512)), SOFTMAX_SCALE)
    x = gen.latent_rows(seed, 0, b, sel, gen.latent_gains(seed))
    c, s = oracle.quantize(x)
    return oracle.sparse_attention(q, oracle.dequantize(c, s), SOFTMAX_SCALE)


@pytest.mark.parametrize("chunk", [1, 2, 3, 4])
def test_chunk_matches_oracle_and_per_query_path(chunk):
    """Three sequences (one shorter than top-K, so its selections are -1 padded), half of
    each selection shared by the chunk's queries; unions of several spans with a ragged
    tail."""
    seed, topk = 61, 1024
    lens = [5000, 700, 3100]
    cache = _cache(seed, lens)
    idx = np.concatenate([gen.overlapping_index_sets(seed, b, lens[b], topk, chunk, 0.5)
                          for b in range(len(lens))])
    q_seq = np.repeat(np.arange(len(lens), dtype=np.int32), chunk)
    q = gen.q_rows(seed, chunk, np.arange(len(q_seq)))
    out, lse, st = _chunked(cache, q, idx, q_seq, chunk, topk)
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)
    ref_out, ref_lse = _per_query(cache, q, idx, q_seq, topk)
    for i in range(len(q_seq)):
        o, l = _oracle(seed, int(q_seq[i]), idx[i], q[i])
        assert_attn_close(out[i], o, lse[i], l, f"chunk {chunk} query {i}")
        assert_attn_close(out[i], ref_out[i], lse[i], ref_lse[i], f"chunk {chunk} query {i} vs per-query")


def test_chunk_disjoint_identical_and_empty_selections():
    """Chunk 0: four disjoint selections (the union is four times one selection); chunk 1:
    four identical selections; chunk 2: one query with no valid entry next to three with
    a few entries each."""
    seed, topk = 67, 512
    lens = [4096, 4096, 900]
    cache = _cache(seed, lens)
    perm = np.argsort(gen.draws(gen.stream_key(seed, gen.TAG_IDX, 99), np.arange(4096)), kind="stable")
    disjoint = np.stack([np.sort(perm[g * topk:(g + 1) * topk]) for g in range(4)]).astype(np.int32)
    same = np.tile(np.sort(perm[:topk]).astype(np.int32), (4, 1))
    sparse = np.full((4, topk), -1, np.int32)
    sparse[1, :3] = [5, 77, 899]
    sparse[2, :1] = [0]
    sparse[3, :2] = [77, 400]
    idx = np.concatenate([disjoint, same, sparse])
    q_seq = np.repeat(np.arange(3, dtype=np.int32), 4)
    q = gen.q_rows(seed, 0, np.arange(12))
    out, lse, st = _chunked(cache, q, idx, q_seq, 4, topk)
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)
    assert np.all(out[8] == 0) and np.all(np.isneginf(lse[8]))
    for i in range(12):
        if i == 8:
            continue
        o, l = _oracle(seed, int(q_seq[i]), idx[i], q[i])
        assert_attn_close(out[i], o, lse[i], l, f"query {i}")


def test_chunk_bad_entries_reported_and_skipped():
    """An index past the context and a chunk whose queries name two sequences: both are
    reported; the bad index is skipped, the mixed chunk's queries get zeros and -inf."""
    seed, topk = 71, 256
    lens = [2000, 2000]
    cache = _cache(seed, lens)
    idx = np.concatenate([gen.overlapping_index_sets(seed, b, 2000, topk, 2, 0.25) for b in range(2)])
    idx[1, 7] = 2500  # past the context of sequence 0
    q_seq = np.array([0, 0, 1, 0], np.int32)  # the second chunk mixes sequences
    q = gen.q_rows(seed, 0, np.arange(4))
    out, lse, st = _chunked(cache, q, idx, q_seq, 2, topk)
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_ERR_DEVICE_FAULT
    assert bits & csa2.CSA2_DEV_BAD_INDEX and bits & csa2.CSA2_DEV_BAD_QSEQ
    for i in (0, 1):
        sel = idx[i][(idx[i] >= 0) & (idx[i] < 2000)]
        o, l = _oracle(seed, 0, sel, q[i])
        assert_attn_close(out[i], o, lse[i], l, f"query {i}")
    assert np.all(out[2:] == 0) and np.all(np.isneginf(lse[2:]))


def test_chunk_union_at_the_size_limit():
    """chunk x topk = 8192, the largest union, with every selection drawn independently
    (no shared part): two chunks of one 16384-token sequence."""
    seed, topk = 73, 2048
    lens = [16384]
    cache = _cache(seed, lens)
    idx = np.concatenate([gen.overlapping_index_sets(seed, s, 16384, topk, 4, 0.0) for s in (1, 2)])
    q_seq = np.zeros(8, np.int32)
    q = gen.q_rows(seed, 0, np.arange(8))
    out, lse, st = _chunked(cache, q, idx, q_seq, 4, topk)
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)
    for i in (0, 3, 5):
        o, l = _oracle(seed, 0, idx[i], q[i])
        assert_attn_close(out[i], o, lse[i], l, f"query {i}")
