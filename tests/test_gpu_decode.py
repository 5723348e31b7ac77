"""Decode path parity: CSA2 indexer (Full / Reindex / Reuse, hierarchical pool) and
FP4 gather-dequantise sparse attention, CUDA path through the C ABI vs the oracle.

Modes: tech-report digest (jiwasawa.github.io), "Compressed Sparse Attention 2 (CSA2)";
format and dequantisation before attention: zaikei.co.jp article, "CSA2とFP4でキャッシュを
圧縮".  Index sets must match except for ties within 1e-5 relative; attention outputs
within 2e-3 x RMS per query."""
import numpy as np
import pytest
import torch

import csa2_inputs as gen
import fp4_compressed_sparse_03_b300 as csa2
import oracle
from csa2_inputs import native
from fp4_compressed_sparse_03_b300.decode import DecodeCache, DecodeStep
from fp4_compressed_sparse_03_b300.workload import all_queries_host, fill_decode_cache
from gpu_common import (SOFTMAX_SCALE, TIE_REL_TOL, assert_attn_close, assert_topk_close, dev,
                        host)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ oracle side ----

class OracleQuery:
    """The oracle's view of one query token: its sequence's keys per group (regenerated
    on the host), the per-layer indices and the per-layer attention outputs."""

    def __init__(self, wl: gen.DecodeWorkload, qi: int, q_idx, q):
        self.wl, self.qi = wl, qi
        self.b = int(wl.q_seq[qi])
        self.n = int(wl.seq_lens[self.b])
        self.groups = wl.groups()
        self.keys = {}
        self.idx, self.pool, self.scores, self.full_scores = {}, {}, {}, {}
        self.q_idx, self.q = q_idx, q

    def keys_of(self, g):
        if g not in self.keys:
            self.keys[g] = native.key_rows_host(self.wl.seed, g, self.b, 0, self.n)
        return self.keys[g]

    def run_index(self):
        wl = self.wl
        src = wl.index_source()
        for l, m in enumerate(wl.schedule):
            g = self.groups[l]
            if m == gen.FULL:
                s = oracle.index_scores(self.q_idx[l][self.qi], self.keys_of(g))
                tok = np.arange(self.n, dtype=np.int32)
                self.idx[l] = oracle.select_topk(s, tok, wl.topk)
                self.pool[g] = oracle.select_topk(s, tok, wl.pool_size) if wl.pool_size else None
                self.scores[l] = s
            elif m == gen.REINDEX:
                self.idx[l], _ = oracle.index_reindex(self.q_idx[l][self.qi], self.keys_of(g),
                                                      self.pool[g], wl.topk)
                self.scores[l] = oracle.index_scores(self.q_idx[l][self.qi], self.keys_of(g))
            else:
                self.idx[l] = oracle.index_reuse(self.idx[src[l]])

    def attention(self, l):
        g = self.groups[l]
        sel = self.idx[self.wl.index_source()[l]]
        sel = sel[sel >= 0]
        gains = gen.latent_gains(self.wl.seed, g)
        x = gen.latent_rows(self.wl.seed, g, self.b, sel, gains)
        codes, scales = oracle.quantize(x)
        chat = oracle.dequantize(codes, scales)
        return oracle.sparse_attention(self.q[l][self.qi], chat, SOFTMAX_SCALE)


def _near(v, ref):
    return abs(v - ref) <= TIE_REL_TOL * max(1.0, abs(ref))


def check_query(wl, step: DecodeStep, oq: OracleQuery, attn_budget=None):
    """Compare one query's indices (every layer) and attention outputs."""
    qi = oq.qi
    src = wl.index_source()
    same_src = {}
    for l, m in enumerate(wl.schedule):
        g = oq.groups[l]
        got = host(step.indices(l)[qi])
        if m == gen.FULL:
            s = oq.scores[l]
            assert_topk_close(got, oq.idx[l], lambda t: s[t], f"q{qi} L{l} full idx")
            if step.use_pool:
                gp = host(step.pool[g][qi])
                assert_topk_close(gp, oq.pool[g], lambda t: s[t], f"q{qi} L{l} pool")
                oq.gpu_pool = gp
            same_src[l] = set(got[got >= 0]) == set(oq.idx[l][oq.idx[l] >= 0])
        elif m == gen.REINDEX:
            s1 = oq.scores[l]
            s0 = oq.scores[max(k for k in range(l) if wl.schedule[k] == gen.FULL)]
            gp = oq.gpu_pool
            gpool, opool = set(gp[gp >= 0]), set(oq.pool[g][oq.pool[g] >= 0])
            gset, oset = set(got[got >= 0]), set(oq.idx[l][oq.idx[l] >= 0])
            assert gset <= gpool, f"q{qi} L{l}: reindex output outside the pool"
            if gpool == opool:
                assert_topk_close(got, oq.idx[l], lambda t: s1[t], f"q{qi} L{l} reindex")
            else:
                kth = min(s1[t] for t in oset) if oset else 0.0
                p_kth = min(s0[t] for t in opool) if opool else 0.0
                for t in gset ^ oset:
                    assert _near(s1[t], kth) or (
                        (t not in opool or t not in gpool) and _near(s0[t], p_kth)), \
                        f"q{qi} L{l}: reindex token {t}"
            same_src[l] = gset == oset
        else:
            assert np.array_equal(got, host(step.indices(src[l])[qi]))
    compared = 0
    for l in range(len(wl.schedule)):
        if attn_budget is not None and compared >= attn_budget:
            break
        if not same_src[src[l]]:
            continue
        out_o, lse_o = oq.attention(l)
        assert_attn_close(host(step.out[l][qi]), out_o, host(step.lse[l][qi]), lse_o,
                          f"q{qi} L{l} attention")
        compared += 1
    return compared


def run_workload(wl, max_q_per_seq=None, n_groups=None):
    cache = fill_decode_cache(wl, n_groups)
    q_idx, q = all_queries_host(wl)
    mq = int(wl.q_per_seq.max()) if max_q_per_seq is None else max_q_per_seq
    step = DecodeStep(cache, wl.q_seq, wl.schedule, wl.pool_size, wl.topk, mq)
    step.run(dev(q_idx), dev(q))
    torch.cuda.synchronize()
    status, bits = csa2.csa2_read_status(step.dev_status)
    assert status == csa2.CSA2_OK, bits
    return cache, step, q_idx, q


def check_sampled(wl, queries, step, q_idx, q, attn_budget=None, min_attn=1):
    total = 0
    for qi in queries:
        oq = OracleQuery(wl, int(qi), q_idx, q)
        oq.run_index()
        total += check_query(wl, step, oq, attn_budget)
    assert total >= min_attn


# ------------------------------------------------------------------ generator ------

def test_device_generator_matches_host_definition():
    key = gen.stream_key(5, gen.TAG_KEY, 3)
    a = torch.empty(10000, dtype=torch.int16, device="cuda")
    native.fill_bf16_dev(a, key, 777, -6)
    torch.cuda.synchronize()
    want = gen.normal_bf16(key, np.arange(777, 10777), pow2=-6)
    assert np.array_equal(host(a).view(np.uint16), want)
    gains = gen.latent_gains(5)
    x = torch.empty((300, 512), dtype=torch.float32, device="cuda")
    native.fill_latent_dev(x, gen.stream_key(5, gen.TAG_LATENT, 9), 40, dev(gains))
    torch.cuda.synchronize()
    assert np.array_equal(host(x), gen.latent_rows(5, 0, 9, np.arange(40, 340), gains))
    wl = gen.DecodeWorkload("t", 5, np.array([200, 64, 1], np.int32), np.ones(3, np.int32),
                            [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl)
    keys = host(cache.keys[0]).view(np.uint16)
    for b in range(3):
        n = int(wl.seq_lens[b])
        slots = wl.layout.slots(b, np.arange(n))
        assert np.array_equal(keys[slots], gen.key_rows(5, 0, b, np.arange(n)))


# ------------------------------------------------------------------ small cases ----

def test_tiny_full_layer():
    """1 sequence x 4096 tokens, identity pages, one Full layer, top-K 256."""
    wl = gen.config_tiny(0)
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, [0], step, q_idx, q)


@pytest.mark.parametrize("drafts", [False, True])
def test_small_ragged_all_modes(drafts):
    """Ragged lengths (N < K, N = 1, partial pages), shuffled pages, F->Ri->Ru->Ru with
    a pool; with drafts, several queries per sequence go through the batched scorer."""
    lens = np.array([5000, 64, 1, 300, 2113, 130], np.int32)
    qps = np.array([3, 1, 2, 4, 1, 2], np.int32) if drafts else np.ones(6, np.int32)
    wl = gen.DecodeWorkload("small", 11 + drafts, lens, qps,
                            [gen.FULL, gen.REINDEX, gen.REUSE, gen.REUSE], pool_size=512, topk=128)
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, range(wl.num_q), step, q_idx, q, min_attn=wl.num_q)


@pytest.mark.parametrize("parallel,schedule,mx", [
    (False, [gen.FULL, gen.REINDEX, gen.REUSE, gen.REUSE], False),
    (True, [gen.FULL, gen.REINDEX, gen.REUSE, gen.REUSE], False),
    (True, [gen.FULL, gen.REINDEX, gen.REUSE, gen.REUSE, gen.FULL, gen.REINDEX, gen.REUSE], False),
    (True, [gen.FULL, gen.REINDEX, gen.REUSE, gen.REUSE], True)])
def test_graph_replay_matches_eager_step(parallel, schedule, mx):
    """The CUDA-graph step (what the benchmark times) replays the same launches: its
    indices, pools, outputs and lse are bit-identical to the eager step's, and a replay
    after new queries are copied into the captured buffers matches an eager run on them.
    With `parallel` the graph is of the parallel schedule (index calls in order, attention
    calls on side branches after their source layer's index call), two Full groups wrap
    the branches around; `mx` takes the MXFP4 cache (the other attention kernel)."""
    lens = np.array([5000, 64, 300, 2113], np.int32)
    wl = gen.DecodeWorkload("graph", 31, lens, np.array([2, 1, 1, 3], np.int32),
                            schedule, pool_size=512, topk=128)
    if mx:
        cache = fill_decode_cache(wl, mx=True)
        q_idx_h, q_h = all_queries_host(wl)
        step = DecodeStep(cache, wl.q_seq, wl.schedule, wl.pool_size, wl.topk,
                          int(wl.q_per_seq.max()))
    else:
        cache, step, q_idx_h, q_h = run_workload(wl)
    q_idx, q = dev(q_idx_h), dev(q_h)
    written = sorted(set(step.src))  # layers whose index output the step writes

    def outputs():
        return [step.idx[l].clone() for l in written] + [step.pool.clone(), step.out.clone(),
                                                          step.lse.clone()]

    def clobber():
        for l in written:
            step.idx[l].fill_(7)
        for t in (step.pool, step.out, step.lse):
            t.fill_(7)

    step.run(q_idx, q)
    torch.cuda.synchronize()
    ref = outputs()
    g = step.capture(q_idx, q, parallel=parallel)
    clobber()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, outputs()):
        assert torch.equal(a, b)
    # new queries through the captured buffers
    q_idx.copy_(torch.flip(q_idx, dims=[1]))
    q.copy_(torch.flip(q, dims=[1]))
    clobber()
    g.replay()
    torch.cuda.synchronize()
    got = outputs()
    clobber()
    step.run(q_idx, q)
    torch.cuda.synchronize()
    for a, b in zip(got, outputs()):
        assert torch.equal(a, b)
    status, bits = csa2.csa2_read_status(step.dev_status)
    assert status == csa2.CSA2_OK, bits


def test_wide_selection_beyond_2_18_tokens():
    """Contexts beyond 2^18 tokens take the multi-CTA filter + finishing selection; a
    shorter sequence in the same batch leaves some filter CTAs without positions."""
    lens = np.array([300000, 70000], np.int32)
    wl = gen.DecodeWorkload("wide", 37, lens, np.array([2, 1], np.int32),
                            [gen.FULL, gen.REINDEX, gen.REUSE], pool_size=4096, topk=1024)
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, range(wl.num_q), step, q_idx, q, min_attn=wl.num_q)


def test_two_groups_pool_larger_than_context():
    lens = np.array([700, 3000], np.int32)
    wl = gen.DecodeWorkload("groups", 17, lens, np.ones(2, np.int32),
                            [gen.FULL, gen.REINDEX, gen.FULL, gen.REINDEX, gen.REUSE],
                            pool_size=1024, topk=256)
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, range(2), step, q_idx, q)


@pytest.mark.parametrize("pool,topk", [(999, 300), (2049, 2048), (12000, 700)])
def test_reindex_pool_sizes(pool, topk):
    """Reindex over pools of sizes that are not multiples of 4 or of the selection's
    per-thread key count, one of them larger than 8192 entries; the 700-token sequence
    has fewer valid pool entries than some of the top-K sizes."""
    lens = np.array([20000, 700, 5000], np.int32)
    wl = gen.DecodeWorkload("pools", 41, lens, np.array([1, 2, 1], np.int32),
                            [gen.FULL, gen.REINDEX, gen.REUSE], pool_size=pool, topk=topk)
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, range(wl.num_q), step, q_idx, q)


@pytest.mark.parametrize("tiles", [4, 5])
def test_context_length_edges(tiles):
    """Empty contexts, one token, page and selection boundaries (63/64/65, 255/256/257 =
    top-K, 511/512/513 = pool), with 1-4 draft queries per sequence: 140 queries (one
    selection CTA per target) and 175 (more queries than SMs: the two-per-SM form, taken
    in order of context length)."""
    base = np.array([0, 1, 63, 64, 65, 255, 256, 257, 511, 512, 513, 2049, 0, 5000], np.int32)
    lens = np.tile(base, tiles)
    qps = (np.arange(len(lens)) % 4 + 1).astype(np.int32)
    wl = gen.DecodeWorkload("edges", 53 + tiles, lens, qps,
                            [gen.FULL, gen.REINDEX, gen.REUSE], pool_size=512, topk=256)
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, range(wl.num_q), step, q_idx, q)


def _bf16_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("num_seqs,n,topk,pool", [
    (4, 3000, 300, 1000),       # one CTA per target (few queries), pool of 1000
    (150, 1500, 200, 700),      # more queries than SMs: the 512-thread form
    (1, 300000, 2048, 8192),    # beyond 2^18 tokens: filter, resolve and emit kernels
])
def test_selection_ties_break_by_lower_position(num_seqs, n, topk, pool):
    """Exact ties: every key row is one of 8 rows whose scores (one-hot queries, values
    exact in bf16 and fp32) are 4 v_r for Full and 4 w_r for Reindex, so the top-K, the
    pool and the Reindex top-K cut through groups of equal scores.  The lower position
    must win every tie (tech-report digest, "Hierarchical Sparse Indexer": the top-K of
    each search; the tie rule is this build's reading), and the outputs must equal the
    oracle's selections exactly."""
    P = 64
    max_pages = (n + P - 1) // P
    lens = np.full(num_seqs, n, np.int32)
    table = np.arange(num_seqs * max_pages, dtype=np.int32).reshape(num_seqs, max_pages)
    cache = DecodeCache(lens, table, num_seqs * max_pages, 1)
    v = np.array([0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5, 4.0], np.float32)
    w = v[::-1].copy()
    pos = np.arange(n, dtype=np.int64)
    keys_host = []
    keys = torch.zeros((num_seqs * max_pages * P, gen.D_IDX), dtype=torch.int16)
    for b in range(num_seqs):
        r = (pos * 7 + b) % 8
        k = np.zeros((n, gen.D_IDX), np.uint16)
        k[:, 0] = _bf16_bits(v[r])
        k[:, 1] = _bf16_bits(w[r])
        keys_host.append(k)
        slots = table[b][pos // P].astype(np.int64) * P + pos % P
        keys[torch.from_numpy(slots)] = torch.from_numpy(k.view(np.int16))
    cache.keys[0].copy_(keys.to(cache.keys.device))
    schedule = [gen.FULL, gen.REINDEX, gen.REUSE]
    q_idx = np.zeros((3, num_seqs, gen.H_IDX, gen.D_IDX), np.uint16)
    q_idx[0, :, :, 0] = _bf16_bits(1.0)
    q_idx[1, :, :, 1] = _bf16_bits(1.0)
    q = np.zeros((3, num_seqs, gen.H_Q, gen.D_KV), np.uint16)
    step = DecodeStep(cache, np.arange(num_seqs, dtype=np.int32), schedule, pool, topk, 1)
    step.run(dev(q_idx), dev(q))
    torch.cuda.synchronize()
    status, bits = csa2.csa2_read_status(step.dev_status)
    assert status == csa2.CSA2_OK, bits
    got_k, got_p, got_r = host(step.indices(0)), host(step.pool[0]), host(step.indices(1))
    tok = np.arange(n, dtype=np.int32)
    for b in range(num_seqs):
        s = oracle.index_scores(q_idx[0][b], keys_host[b])
        want_p = oracle.select_topk(s, tok, pool)
        assert np.array_equal(got_p[b], want_p), f"seq {b}: pool"
        assert np.array_equal(got_k[b], oracle.select_topk(s, tok, topk)), f"seq {b}: top-K"
        want_r, _ = oracle.index_reindex(q_idx[1][b], keys_host[b], want_p, topk)
        assert np.array_equal(got_r[b], want_r), f"seq {b}: reindex"


def test_attention_random_index_sets():
    """Attention alone on seeded random selections (with -1 padding and an empty set),
    single- and multi-split launches (up to 36 splits of 128 entries, most of them empty
    for the 100-token sequence)."""
    lens = np.array([3000, 100, 5000], np.int32)
    wl = gen.DecodeWorkload("attn", 23, lens, np.ones(3, np.int32), [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl)
    for topk, nq in [(256, 3), (2048, 3), (64, 3), (4608, 3)]:
        q_seq = np.array([0, 1, 2][:nq], np.int32)
        idx = np.stack([gen.random_index_set(23, 100 * topk + i, int(lens[b]), topk,
                                             n_invalid=(7 if i == 0 else 0))
                        for i, b in enumerate(q_seq)])
        if topk == 64:
            idx[1] = -1
        q = np.stack([gen.q_rows(23, topk, np.array([i]))[0] for i in range(nq)])
        out = torch.zeros((nq, 16, 512), dtype=torch.float32, device="cuda")
        lse = torch.zeros((nq, 16), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(csa2.csa2_attn_workspace_size(nq, topk), 16), dtype=torch.uint8,
                         device="cuda")
        csa2.check(csa2.csa2_sparse_attn(dev(q), cache.codes[0], cache.scales[0], dev(idx),
                                         cache.pages, out, lse, nq, dev(q_seq), topk,
                                         SOFTMAX_SCALE, ws), "attn")
        for i, b in enumerate(q_seq):
            sel = idx[i][idx[i] >= 0]
            x = gen.latent_rows(23, 0, int(b), sel, gen.latent_gains(23))
            c, s = oracle.quantize(x)
            o, l = oracle.sparse_attention(q[i], oracle.dequantize(c, s), SOFTMAX_SCALE)
            if sel.size == 0:
                assert np.all(host(out[i]) == 0) and np.all(np.isneginf(host(lse[i])))
            else:
                assert_attn_close(host(out[i]), o, host(lse[i]), l, f"topk {topk} q{i}")


def _trend_cache(n_tok: int, slope: float, seed: int):
    """A one-sequence cache (identity page table) whose latent rows drift along a fixed
    direction d: x_t = base_t + slope * t * d, quantised by libcsa2's codec (bit-exact with
    the oracle's).  Returns (cache, d, dequantised rows [n_tok, 512] from the oracle)."""
    from fp4_compressed_sparse_03_b300.decode import DecodeCache
    rng = np.random.default_rng(seed)
    d = rng.standard_normal(512).astype(np.float32)
    base = (rng.standard_normal((n_tok, 512)) * np.exp(0.5 * rng.standard_normal(512))).astype(np.float32)
    x = (base + slope * np.arange(n_tok, dtype=np.float32)[:, None] * d).astype(np.float32)
    pages = n_tok // 64
    cache = DecodeCache(np.array([n_tok], np.int32), np.arange(pages, dtype=np.int32)[None, :], pages)
    slots = torch.arange(n_tok, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_quantize(dev(x), slots, cache.codes[0], cache.scales[0], n_tok, 512,
                                  cache.num_slots), "quantize")
    c, s = oracle.quantize(x)
    return cache, d, oracle.dequantize(c, s)


@pytest.mark.parametrize("direction", ["rising", "falling"])
def test_attention_logits_far_apart_across_tiles_and_splits(direction):
    """Logits that move by ~12 log2 units per 128-token tile (q_h = beta_h * d on rows drifting
    along d), over 2048 selected entries: rising, the lazily moved reference max moves on
    nearly every tile and the four 512-entry splits' maxima lie 2^40 and more apart, so
    the split combine merges partials whose weights differ by many orders of magnitude;
    falling, the first tile holds the maximum and no later tile rescales.  The earliest
    entries' weights underflow to zero in both the kernel and the oracle."""
    n_tok, topk = 4096, 2048
    cache, d, chat = _trend_cache(n_tok, 2e-3 if direction == "rising" else -2e-3, 61)
    beta = np.linspace(0.7, 2.2, 16, dtype=np.float32)
    rng = np.random.default_rng(62)
    q32 = beta[:, None] * d[None, :] + 0.05 * rng.standard_normal((16, 512)).astype(np.float32)
    q = gen.f32_to_bf16_bits(q32)[None]
    idx = np.arange(0, n_tok, 2, dtype=np.int32)[None, :]
    assert idx.shape[1] == topk
    out = torch.zeros((1, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(1, topk), 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_seq = dev(np.zeros(1, np.int32))
    csa2.check(csa2.csa2_sparse_attn(dev(q), cache.codes[0], cache.scales[0], dev(idx), cache.pages,
                                     out, lse, 1, q_seq, topk, SOFTMAX_SCALE, ws, dev_status=st), "attn")
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)
    o, l = oracle.sparse_attention(q[0], chat[idx[0]], SOFTMAX_SCALE)
    # the logits really span far more than the lazy gap and the split combine's range
    z = (gen.bf16_bits_to_f32(q[0]).astype(np.float64) @ chat[idx[0]].T) * SOFTMAX_SCALE / np.log(2)
    span = z.max(axis=1) - z.min(axis=1)
    assert span.min() > 100, span.min()
    split_max = z.reshape(16, 4, 512).max(axis=2)
    assert np.abs(split_max[:, 3] - split_max[:, 0]).min() > 40
    assert_attn_close(host(out[0]), o, host(lse[0]), l, f"{direction} logits")


def test_mx_attention_random_index_sets():
    """The MXFP4 read path (csa2_sparse_attn_mx over a cache written by csa2_quantize_mx)
    against the oracle's attention over its own MXFP4 dequantisation: single- and
    multi-split launches, -1 padding and an empty set."""
    lens = np.array([3000, 100, 5000], np.int32)
    wl = gen.DecodeWorkload("attn_mx", 23, lens, np.ones(3, np.int32), [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl, mx=True)
    for topk, nq in [(256, 3), (2048, 3), (64, 3)]:
        q_seq = np.array([0, 1, 2][:nq], np.int32)
        idx = np.stack([gen.random_index_set(23, 100 * topk + i, int(lens[b]), topk,
                                             n_invalid=(7 if i == 0 else 0))
                        for i, b in enumerate(q_seq)])
        if topk == 64:
            idx[1] = -1
        q = np.stack([gen.q_rows(23, topk, np.array([i]))[0] for i in range(nq)])
        out = torch.zeros((nq, 16, 512), dtype=torch.float32, device="cuda")
        lse = torch.zeros((nq, 16), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(csa2.csa2_attn_workspace_size(nq, topk), 16), dtype=torch.uint8,
                         device="cuda")
        csa2.check(csa2.csa2_sparse_attn_mx(dev(q), cache.codes[0], cache.scales[0], dev(idx),
                                            cache.pages, out, lse, nq, dev(q_seq), topk,
                                            SOFTMAX_SCALE, ws), "attn_mx")
        for i, b in enumerate(q_seq):
            sel = idx[i][idx[i] >= 0]
            x = gen.latent_rows(23, 0, int(b), sel, gen.latent_gains(23))
            c, s = oracle.mx_quantize(x)
            o, l = oracle.sparse_attention(q[i], oracle.mx_dequantize(c, s), SOFTMAX_SCALE)
            if sel.size == 0:
                assert np.all(host(out[i]) == 0) and np.all(np.isneginf(host(lse[i])))
            else:
                assert_attn_close(host(out[i]), o, host(lse[i]), l, f"mx topk {topk} q{i}")


def test_mx_attention_scale_spread():
    """Rows scaled by 2^k, k in [-10, 10] per token, so the E8M0 bytes of one split span
    more than 20 values: the kernel's rebasing on the split's largest scale keeps the
    result within tolerance of the oracle."""
    T = 512
    cache = DecodeCache(np.array([T], np.int32), np.arange(T // 64, dtype=np.int32).reshape(1, -1),
                        T // 64, mx=True)
    k = np.random.default_rng(11).integers(-10, 11, T)
    x = (gen.latent_rows(31, 0, 0, np.arange(T), gen.latent_gains(31)) *
         np.exp2(k)[:, None]).astype(np.float32)
    csa2.check(csa2.csa2_quantize_mx(dev(x), dev(np.arange(T, dtype=np.int32)), cache.codes[0],
                                     cache.scales[0], T, 512, cache.num_slots), "quantize_mx")
    c, s = oracle.mx_quantize(x)
    assert np.array_equal(host(cache.codes[0]), c) and np.array_equal(host(cache.scales[0]), s)
    assert int(s.max()) - int(s.min()) > 20
    q = gen.q_rows(31, 0, np.array([0]))
    idx = np.arange(T, dtype=np.int32).reshape(1, T)
    out = torch.zeros((1, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(1, T), 16), dtype=torch.uint8, device="cuda")
    csa2.check(csa2.csa2_sparse_attn_mx(dev(q), cache.codes[0], cache.scales[0], dev(idx),
                                        cache.pages, out, lse, 1, dev(np.zeros(1, np.int32)), T,
                                        SOFTMAX_SCALE, ws), "attn_mx")
    o, l = oracle.sparse_attention(q[0], oracle.mx_dequantize(c, s), SOFTMAX_SCALE)
    assert_attn_close(host(out[0]), o, host(lse[0]), l, "mx scale spread")


def test_prefill_chunk_queries_against_their_own_topk():
    """A prefill chunk: the 32 query positions 8160 .. 8191 of one 8192-token sequence, each
    attending to its own top-512 among the tokens it may see (causal).  Each query is an
    entry of the pages descriptor with its own length, all sharing the sequence's
    page-table row; the read path treats them as independent queries."""
    n, C, K = 8192, 32, 512
    wl = gen.DecodeWorkload("chunk", 47, np.array([n], np.int32), np.ones(1, np.int32),
                            [gen.FULL], 0, 16)
    src = fill_decode_cache(wl)
    pos = np.arange(n - C, n, dtype=np.int32)
    row = host(src.page_table)[0]
    cache = DecodeCache(pos + 1, np.tile(row, (C, 1)), src.num_pages, 1)
    cache.codes.copy_(src.codes)
    cache.scales.copy_(src.scales)
    idx = np.stack([gen.random_index_set(47, i, int(p) + 1, K) for i, p in enumerate(pos)])
    q = np.stack([gen.q_rows(47, 3, np.array([i]))[0] for i in range(C)])
    out = torch.zeros((C, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((C, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(C, K), 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.check(csa2.csa2_sparse_attn(dev(q), cache.codes[0], cache.scales[0], dev(idx), cache.pages,
                                     out, lse, C, dev(np.arange(C, dtype=np.int32)), K,
                                     SOFTMAX_SCALE, ws, None, st), "attn")
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_OK, hex(bits)
    gains = gen.latent_gains(47)
    for i in range(C):
        x = gen.latent_rows(47, 0, 0, idx[i], gains)
        c, s = oracle.quantize(x)
        o, l = oracle.sparse_attention(q[i], oracle.dequantize(c, s), SOFTMAX_SCALE)
        assert_attn_close(host(out[i]), o, host(lse[i]), l, f"chunk query {i}")


def test_mx_attention_split_with_no_valid_entry():
    """MXFP4 read path: a query whose selection is all -1 over several splits gets zero output
    and -inf lse; the other query is unaffected."""
    lens = np.array([3000, 900], np.int32)
    wl = gen.DecodeWorkload("mx_empty", 53, lens, np.ones(2, np.int32), [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl, mx=True)
    topk = 1536
    idx = np.stack([gen.random_index_set(53, 1, 3000, topk), np.full(topk, -1, np.int32)])
    q = np.stack([gen.q_rows(53, 0, np.array([i]))[0] for i in range(2)])
    out = torch.full((2, 16, 512), np.nan, dtype=torch.float32, device="cuda")
    lse = torch.full((2, 16), np.nan, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(2, topk), 16), dtype=torch.uint8, device="cuda")
    csa2.check(csa2.csa2_sparse_attn_mx(dev(q), cache.codes[0], cache.scales[0], dev(idx),
                                        cache.pages, out, lse, 2, dev(np.array([0, 1], np.int32)),
                                        topk, SOFTMAX_SCALE, ws), "attn_mx")
    assert np.all(host(out[1]) == 0) and np.all(np.isneginf(host(lse[1])))
    x = gen.latent_rows(53, 0, 0, idx[0], gen.latent_gains(53))
    c, s = oracle.mx_quantize(x)
    o, l = oracle.sparse_attention(q[0], oracle.mx_dequantize(c, s), SOFTMAX_SCALE)
    assert_attn_close(host(out[0]), o, host(lse[0]), l, "mx query 0")


def test_attention_dense_equals_all_tokens():
    """K = N: the sparse path over every token equals the oracle's dense attention."""
    wl = gen.DecodeWorkload("dense", 29, np.array([512], np.int32), np.ones(1, np.int32),
                            [gen.FULL], 0, 512)
    cache = fill_decode_cache(wl)
    idx = np.arange(512, dtype=np.int32).reshape(1, 512)
    q = gen.q_rows(29, 0, np.array([0]))
    out = torch.zeros((1, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(1, 512), 16), dtype=torch.uint8, device="cuda")
    csa2.check(csa2.csa2_sparse_attn(dev(q), cache.codes[0], cache.scales[0], dev(idx), cache.pages,
                                     out, lse, 1, dev(np.zeros(1, np.int32)), 512, SOFTMAX_SCALE, ws),
               "attn")
    x = gen.latent_rows(29, 0, 0, np.arange(512), gen.latent_gains(29))
    c, s = oracle.quantize(x)
    o, l = oracle.sparse_attention(q[0], oracle.dequantize(c, s), SOFTMAX_SCALE)
    assert_attn_close(host(out[0]), o, host(lse[0]), l, "dense")


def test_page_shuffle_invariance():
    """The same logical cache under two physical page permutations gives bitwise equal
    indices and outputs."""
    lens = np.array([4000, 2500], np.int32)
    res = []
    for shuffle_seed in (101, 202):
        wl = gen.DecodeWorkload("perm", 31, lens, np.ones(2, np.int32),
                                [gen.FULL, gen.REINDEX, gen.REUSE], 512, 128)
        wl.layout = gen.make_layout(shuffle_seed, lens, True)
        _, step, _, _ = run_workload(wl)
        res.append((host(step.idx), host(step.out), host(step.lse)))
    assert np.array_equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1], res[1][1]) and np.array_equal(res[0][2], res[1][2])


def test_bad_indices_are_reported_and_skipped():
    lens = np.array([1000], np.int32)
    wl = gen.DecodeWorkload("bad", 37, lens, np.ones(1, np.int32), [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl)
    idx = np.array([[3, 17, 999, 1000, 5000, -5, -1, 40]], np.int32)
    q = gen.q_rows(37, 0, np.array([0]))
    out = torch.zeros((1, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(csa2.csa2_attn_workspace_size(1, 8), 16), dtype=torch.uint8, device="cuda")
    csa2.check(csa2.csa2_sparse_attn(dev(q), cache.codes[0], cache.scales[0], dev(idx), cache.pages,
                                     out, lse, 1, dev(np.zeros(1, np.int32)), 8, SOFTMAX_SCALE, ws,
                                     None, st), "attn")
    status, bits = csa2.csa2_read_status(st)
    assert status == csa2.CSA2_ERR_DEVICE_FAULT and bits & csa2.CSA2_DEV_BAD_INDEX
    sel = np.array([3, 17, 999, 40])
    x = gen.latent_rows(37, 0, 0, sel, gen.latent_gains(37))
    c, s = oracle.quantize(x)
    o, l = oracle.sparse_attention(q[0], oracle.dequantize(c, s), SOFTMAX_SCALE)
    assert_attn_close(host(out[0]), o, host(lse[0]), l, "bad idx skipped")


def test_index_host_argument_errors():
    lens = np.array([100], np.int32)
    wl = gen.DecodeWorkload("err", 41, lens, np.ones(1, np.int32), [gen.FULL], 0, 16)
    cache = fill_decode_cache(wl)
    qs = dev(np.zeros(1, np.int32))
    out = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    q_idx = dev(gen.q_idx_rows(41, 0, np.array([0])))
    ws = torch.empty(csa2.csa2_index_workspace_size(csa2.CSA2_FULL, 1, cache.max_pages, 0),
                     dtype=torch.uint8, device="cuda")
    small = csa2.make_index_args(1, qs, 1, 0, None, ws, 16)
    assert csa2.csa2_index(csa2.CSA2_FULL, q_idx, cache.keys[0], None, 16, out, cache.pages,
                           small) == csa2.CSA2_ERR_INVALID_ARGUMENT
    args = csa2.make_index_args(1, qs, 5, 0, None, ws)
    assert csa2.csa2_index(csa2.CSA2_FULL, q_idx, cache.keys[0], None, 16, out, cache.pages,
                           args) == csa2.CSA2_ERR_UNSUPPORTED
    bad_pages = csa2.make_pages(cache.seq_lens, cache.page_table, cache.num_pages, 32)
    args = csa2.make_index_args(1, qs, 1, 0, None, ws)
    assert csa2.csa2_index(csa2.CSA2_FULL, q_idx, cache.keys[0], None, 16, out, bad_pages,
                           args) == csa2.CSA2_ERR_UNSUPPORTED
    assert csa2.csa2_index(csa2.CSA2_REINDEX, q_idx, cache.keys[0], None, 16, out, cache.pages,
                           args) == csa2.CSA2_ERR_INVALID_ARGUMENT
    # REUSE copies the inherited indices
    inherit = dev(np.arange(16, dtype=np.int32).reshape(1, 16))
    args = csa2.make_index_args(1, qs, 1, 0, inherit, None)
    assert csa2.csa2_index(csa2.CSA2_REUSE, None, None, None, 16, out, cache.pages, args) == 0
    torch.cuda.synchronize()
    assert np.array_equal(host(out), np.arange(16).reshape(1, 16))


# ------------------------------------------------------------------ full-size ------

def test_decode_batch_64x131072_sampled():
    """64 sequences x 131072 tokens, F->Ri->Ru->Ru, pool 8192, K 2048 (the benchmark's
    launch configuration); 8 sampled queries compared in full."""
    wl = gen.config_decode_batch()
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, [0, 9, 18, 27, 36, 45, 54, 63], step, q_idx, q, min_attn=16)


def test_long_context_4x1m():
    wl = gen.config_long_context()
    _, step, q_idx, q = run_workload(wl)
    check_sampled(wl, range(4), step, q_idx, q, min_attn=6)


def test_ragged_serving_sampled():
    """256 sequences (lognormal lengths 1K..256K), 1-4 draft queries each (batched
    tensor-core scoring), 20 layers in 5 Full groups; 16 sampled queries."""
    wl = gen.config_ragged()
    _, step, q_idx, q = run_workload(wl)
    rng = np.random.default_rng(4)
    picks = np.sort(rng.choice(wl.num_q, 16, replace=False))
    check_sampled(wl, picks, step, q_idx, q, attn_budget=6, min_attn=30)
