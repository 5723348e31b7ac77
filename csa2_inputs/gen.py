"""Seeded, counter-based synthetic inputs shared by the CUDA path and the CPU oracle.

This module holds no arithmetic of the method itself (no quantisation, scoring,
selection or attention).  It only draws numbers.  Every value is a pure function
of (seed, tag, sub, counter), so any single element can be regenerated on its own:
the oracle regenerates exactly the tokens it needs, and the CUDA generator in
``csa2_inputs/csrc/gen.cu`` fills HBM with the same bits.

Generator definition (implemented identically, bit for bit, on both sides):

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014; constants as in
  Vigna's public-domain reference ``splitmix64.c``).
* A stream key is ``mix64(mix64(seed) ^ (tag << 40) ^ sub)``.
* The j-th 64-bit draw of a stream is ``mix64(key + (j + 1) * 0x9E3779B97F4A7C15)``
  (the j-th output of a SplitMix64 generator whose state starts at ``key``).
* ``normal(key, i)`` is the classical sum-of-twelve-uniforms approximation of a
  standard normal variate: draws ``3i, 3i+1, 3i+2`` give twelve 16-bit integers
  u_0..u_11; with S = sum(u), the value is ``(2 S - 786420) * 2**-17``.  Its mean is
  exactly 0, its variance 1 - 2**-32, its support [-6, 6].  The result is an exact
  float32 (an integer below 2**20 times a power of two), so no rounding and no
  transcendental function is involved and the CPU and GPU agree on every bit.
* bfloat16 values are the round-to-nearest-even of that float32.

Only host-side quantities (per-channel gains, sequence lengths, page
permutations) use floating-point functions (``exp``); they are computed once here
in float64 and handed to both sides as inputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX_C1 = 0xBF58476D1CE4E5B9
MIX_C2 = 0x94D049BB133111EB

# Stream tags.  One tag per kind of input; ``sub`` separates sequences, layers, groups.
TAG_LATENT = 1   # latent KV values, before quantisation
TAG_GAIN = 2     # per-channel log-gain z_c of the latent
TAG_KEY = 3      # indexer keys (bf16)
TAG_QIDX = 4     # indexer queries (bf16)
TAG_Q = 5        # attention queries (bf16)
TAG_H = 6        # encoder final hidden state H (bf16)
TAG_WKV = 7      # KV projection weights (bf16)
TAG_WIDX = 8     # indexer-key projection weights (bf16)
TAG_PERM = 9     # physical page permutation
TAG_LENS = 10    # ragged context lengths
TAG_DRAFT = 11   # speculative draft-token counts
TAG_IDX = 12     # random selected-index sets (attention-only tests)
TAG_CHUNK = 13   # per-query parts of overlapping selections (multi-query chunks)

_U64 = np.uint64


def _u64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.uint64)


def mix64(z):
    """SplitMix64 output function on uint64 arrays (wrapping arithmetic)."""
    z = _u64(z)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> _U64(30))) * _U64(MIX_C1)
        z = (z ^ (z >> _U64(27))) * _U64(MIX_C2)
    return z ^ (z >> _U64(31))


def stream_key(seed: int, tag: int, sub: int = 0) -> int:
    """Key of the stream (seed, tag, sub); sub < 2**40."""
    assert 0 <= sub < (1 << 40) and 0 <= tag < (1 << 24)
    k = int(mix64(_u64(seed & (2**64 - 1))))
    return int(mix64(_u64(k ^ (tag << 40) ^ sub)))


def draws(key: int, j) -> np.ndarray:
    """64-bit draws number j (array) of the stream with the given key."""
    j = _u64(j)
    with np.errstate(over="ignore"):
        return mix64(_u64(key) + (j + _U64(1)) * _U64(GAMMA))


def normal(key: int, i) -> np.ndarray:
    """Approximately N(0, 1) float32 values number i (array) of a stream."""
    i = _u64(i)
    s = np.zeros(i.shape, dtype=np.int64)
    for r in range(3):
        d = draws(key, i * _U64(3) + _U64(r))
        for sh in (0, 16, 32, 48):
            s += ((d >> _U64(sh)) & _U64(0xFFFF)).astype(np.int64)
    return ((2 * s - 786420).astype(np.float32) * np.float32(2.0**-17)).astype(np.float32)


def uniform_u32(key: int, i) -> np.ndarray:
    """Upper 32 bits of draw i: uniform integers in [0, 2**32)."""
    return (draws(key, i) >> _U64(32)).astype(np.uint64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(key: int, i, pow2: int = 0) -> np.ndarray:
    """bf16 bits of normal(key, i) * 2**pow2 (power-of-two scaling is exact)."""
    x = normal(key, i)
    if pow2:
        x = (x * np.float32(2.0**pow2)).astype(np.float32)
    return f32_to_bf16_bits(x)


# ----------------------------------------------------------------------------------
# Workload recipes.  Sizes and distributions follow the workloads the decode and
# write paths are measured on; every random quantity comes from the streams above.
# ----------------------------------------------------------------------------------

PAGE = 64        # tokens per page
D_KV = 512       # latent channels (head dim of the MQA attention)
GROUP = 16       # channels per E4M3 scale
D_IDX = 128      # indexer head dim
H_IDX = 4        # indexer heads
H_Q = 16         # attention query heads

FULL, REINDEX, REUSE = 0, 1, 2


def latent_gains(seed: int, group: int = 0) -> np.ndarray:
    """Per-channel gains g_c = exp(0.5 z_c), z_c ~ N(0,1), rounded to float32."""
    z = normal(stream_key(seed, TAG_GAIN, group), np.arange(D_KV)).astype(np.float64)
    return np.exp(0.5 * z).astype(np.float32)


def latent_rows(seed: int, group: int, seq: int, tokens: np.ndarray, gains: np.ndarray) -> np.ndarray:
    """float32 latent [len(tokens), 512] = normal * gain (one IEEE float32 product)."""
    key = stream_key(seed, TAG_LATENT, (group << 24) | seq)
    t = _u64(tokens).reshape(-1, 1)
    i = t * _U64(D_KV) + np.arange(D_KV, dtype=np.uint64).reshape(1, -1)
    return (normal(key, i) * gains.reshape(1, -1)).astype(np.float32)


def key_rows(seed: int, group: int, seq: int, tokens: np.ndarray) -> np.ndarray:
    """bf16 bits of indexer keys [len(tokens), 128], ~N(0,1)."""
    key = stream_key(seed, TAG_KEY, (group << 24) | seq)
    t = _u64(tokens).reshape(-1, 1)
    i = t * _U64(D_IDX) + np.arange(D_IDX, dtype=np.uint64).reshape(1, -1)
    return normal_bf16(key, i)


def q_idx_rows(seed: int, layer: int, queries: np.ndarray) -> np.ndarray:
    """bf16 bits of indexer queries [len(queries), 4, 128], ~N(0,1) (head weights 1)."""
    out = np.empty((len(queries), H_IDX, D_IDX), dtype=np.uint16)
    for n, qi in enumerate(queries):
        key = stream_key(seed, TAG_QIDX, (layer << 24) | int(qi))
        out[n] = normal_bf16(key, np.arange(H_IDX * D_IDX)).reshape(H_IDX, D_IDX)
    return out


def q_rows(seed: int, layer: int, queries: np.ndarray) -> np.ndarray:
    """bf16 bits of attention queries [len(queries), 16, 512], ~N(0,1)."""
    out = np.empty((len(queries), H_Q, D_KV), dtype=np.uint16)
    for n, qi in enumerate(queries):
        key = stream_key(seed, TAG_Q, (layer << 24) | int(qi))
        out[n] = normal_bf16(key, np.arange(H_Q * D_KV)).reshape(H_Q, D_KV)
    return out


def page_permutation(seed: int, num_pages: int, shuffle: bool = True, group: int = 0) -> np.ndarray:
    """Physical page id of each logical page (identity, or a seeded permutation)."""
    if not shuffle:
        return np.arange(num_pages, dtype=np.int32)
    r = draws(stream_key(seed, TAG_PERM, group), np.arange(num_pages))
    return np.argsort(r, kind="stable").astype(np.int32)


def ragged_lengths(seed: int, num_seqs: int, median: int = 16384, sigma: float = 1.0,
                   lo: int = 1024, hi: int = 262144) -> np.ndarray:
    """N_i = clip(round(median * exp(sigma z_i)), lo, hi), z_i ~ N(0,1)."""
    z = normal(stream_key(seed, TAG_LENS), np.arange(num_seqs)).astype(np.float64)
    n = np.rint(median * np.exp(sigma * z))
    return np.clip(n, lo, hi).astype(np.int32)


def draft_counts(seed: int, num_seqs: int, max_draft: int = 4) -> np.ndarray:
    """Speculative query tokens per sequence, uniform on 1..max_draft."""
    u = uniform_u32(stream_key(seed, TAG_DRAFT), np.arange(num_seqs))
    return (1 + (u % _U64(max_draft))).astype(np.int32)


def random_index_set(seed: int, sub: int, n_ctx: int, k: int, n_invalid: int = 0) -> np.ndarray:
    """A sorted random subset of min(k, n_ctx) - n_invalid tokens of [0, n_ctx), -1 padded to k."""
    m = max(0, min(k, n_ctx) - n_invalid)
    r = draws(stream_key(seed, TAG_IDX, sub), np.arange(n_ctx))
    pick = np.sort(np.argsort(r, kind="stable")[:m]).astype(np.int32)
    out = np.full(k, -1, dtype=np.int32)
    out[:m] = pick
    return out


def overlapping_index_sets(seed: int, sub: int, n_ctx: int, k: int, count: int,
                           shared: float) -> np.ndarray:
    """`count` sorted selections of min(k, n_ctx) tokens of [0, n_ctx), each -1 padded to
    k: round(shared * m) tokens common to all (a random subset), the rest of each drawn
    independently from the other tokens.  int32 [count, k]; sub < 2**35."""
    m = min(k, n_ctx)
    s = int(round(shared * m))
    base = np.argsort(draws(stream_key(seed, TAG_IDX, sub), np.arange(n_ctx)), kind="stable")
    common, rest = base[:s], base[s:]
    out = np.full((count, k), -1, dtype=np.int32)
    for g in range(count):
        r = draws(stream_key(seed, TAG_CHUNK, (sub << 5) | g), np.arange(rest.size))
        own = rest[np.argsort(r, kind="stable")[:m - s]]
        out[g, :m] = np.sort(np.concatenate([common, own])).astype(np.int32)
    return out


@dataclass
class PagedLayout:
    """Logical -> physical page mapping for a batch of sequences."""
    seq_lens: np.ndarray            # int32 [B]
    page_table: np.ndarray          # int32 [B, max_pages]; unused entries -1
    num_pages: int                  # physical pages in the pool

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    def slots(self, seq: int, tokens: np.ndarray) -> np.ndarray:
        """Physical row (slot) of logical tokens of one sequence."""
        tokens = np.asarray(tokens, dtype=np.int64)
        return self.page_table[seq, tokens // PAGE].astype(np.int64) * PAGE + tokens % PAGE


def make_layout(seed: int, seq_lens, shuffle: bool = True, group: int = 0) -> PagedLayout:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    pages_per = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    total = int(pages_per.sum())
    perm = page_permutation(seed, total, shuffle, group)
    max_pages = int(pages_per.max()) if len(pages_per) else 0
    table = np.full((len(seq_lens), max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for b, p in enumerate(pages_per):
        table[b, :p] = perm[off:off + p]
        off += p
    return PagedLayout(seq_lens, table, total)


@dataclass
class DecodeWorkload:
    """A decode step: sequences, their queries, a per-layer mode schedule."""
    name: str
    seed: int
    seq_lens: np.ndarray                  # int32 [B]
    q_per_seq: np.ndarray                 # int32 [B] query tokens per sequence
    schedule: list                        # modes per layer
    pool_size: int
    topk: int
    shuffle: bool = True
    layout: PagedLayout = field(default=None)

    def __post_init__(self):
        if self.layout is None:
            self.layout = make_layout(self.seed, self.seq_lens, self.shuffle)

    @property
    def num_q(self) -> int:
        return int(self.q_per_seq.sum())

    @property
    def q_seq(self) -> np.ndarray:
        return np.repeat(np.arange(len(self.seq_lens), dtype=np.int32), self.q_per_seq)

    def groups(self):
        """Full-layer group id of every layer (the most recent Full layer at or before it)."""
        g, out = -1, []
        for m in self.schedule:
            if m == FULL:
                g += 1
            out.append(g)
        return out

    def index_source(self):
        """For each layer, the most recent layer (itself included) that produced indices."""
        src, out = -1, []
        for l, m in enumerate(self.schedule):
            if m in (FULL, REINDEX):
                src = l
            out.append(src)
        return out


def config_tiny(seed: int = 0) -> DecodeWorkload:
    """1 sequence x 4096 tokens, identity page table, one Full layer, top-K 256, no pool."""
    return DecodeWorkload("tiny", seed, np.array([4096], np.int32), np.array([1], np.int32),
                          [FULL], pool_size=0, topk=256, shuffle=False)


def config_decode_batch(seed: int = 1) -> DecodeWorkload:
    """64 sequences x 131072 tokens, shuffled pages, Full->Reindex->Reuse->Reuse, P 8192, K 2048."""
    return DecodeWorkload("decode_batch_64x131072", seed, np.full(64, 131072, np.int32),
                          np.ones(64, np.int32), [FULL, REINDEX, REUSE, REUSE],
                          pool_size=8192, topk=2048)


def config_long_context(seed: int = 3) -> DecodeWorkload:
    """4 sequences x 2**20 tokens, shuffled pages, Full->Reindex->Reuse, P 16384, K 2048."""
    return DecodeWorkload("long_context_4x1048576", seed, np.full(4, 1 << 20, np.int32),
                          np.ones(4, np.int32), [FULL, REINDEX, REUSE],
                          pool_size=16384, topk=2048)


def config_ragged(seed: int = 4, num_seqs: int = 256, layers: int = 20) -> DecodeWorkload:
    """256 sequences, lognormal lengths (median 16K, 1K..256K), 1-4 draft tokens each,
    20 layers: Full at 4g, Reindex at 4g+1, Reuse at 4g+2 and 4g+3; P 8192, K 2048."""
    sched = [(FULL, REINDEX, REUSE, REUSE)[l % 4] for l in range(layers)]
    return DecodeWorkload("ragged_256seq_20layer", seed, ragged_lengths(seed, num_seqs),
                          draft_counts(seed, num_seqs), sched, pool_size=8192, topk=2048)


@dataclass
class WriteWorkload:
    """CED write path: H [T, d] times per-layer projections, quantised on write."""
    name: str
    seed: int
    T: int
    d_model: int
    n_kv_proj: int
    n_idx_proj: int
    shuffle: bool = True
    append_pos: int = -1  # >= 0: token t is the new token of sequence t, at this position

    @property
    def n_out(self) -> int:
        return self.n_kv_proj * D_KV + self.n_idx_proj * D_IDX

    @property
    def num_pages(self) -> int:
        if self.append_pos >= 0:
            return self.T  # one (current) page per sequence
        return (self.T + PAGE - 1) // PAGE

    def slot_of_token(self) -> np.ndarray:
        perm = page_permutation(self.seed, self.num_pages, self.shuffle)
        t = np.arange(self.T, dtype=np.int64)
        if self.append_pos >= 0:  # sequence t's current page, at the new position's offset
            return (perm[t].astype(np.int64) * PAGE + self.append_pos % PAGE).astype(np.int32)
        return (perm[t // PAGE].astype(np.int64) * PAGE + t % PAGE).astype(np.int32)

    def h_rows(self, rows) -> np.ndarray:
        key = stream_key(self.seed, TAG_H)
        r = _u64(rows).reshape(-1, 1)
        return normal_bf16(key, r * _U64(self.d_model) + np.arange(self.d_model, dtype=np.uint64))

    def w_rows(self, out_cols) -> np.ndarray:
        """Rows of the stored projection matrix Wt [n_out, d_model] (output-major), ~N(0, 1/4096)."""
        out_cols = np.asarray(out_cols, dtype=np.int64)
        res = np.empty((len(out_cols), self.d_model), dtype=np.uint16)
        kv_cols = self.n_kv_proj * D_KV
        kkv, kidx = stream_key(self.seed, TAG_WKV), stream_key(self.seed, TAG_WIDX)
        ar = np.arange(self.d_model, dtype=np.uint64)
        p2 = d_model_pow2_scale(self.d_model)
        for n, c in enumerate(out_cols):
            if c < kv_cols:
                res[n] = normal_bf16(kkv, _U64(c) * _U64(self.d_model) + ar, pow2=p2)
            else:
                res[n] = normal_bf16(kidx, _U64(c - kv_cols) * _U64(self.d_model) + ar, pow2=p2)
        return res


def config_write(seed: int = 2) -> WriteWorkload:
    """H [32768, 4096] ~N(0,1); 20 KV projections [4096, 512] and 20 indexer-key
    projections [4096, 128] ~N(0, 1/4096); 512 shuffled pages of 64 tokens."""
    return WriteWorkload("ced_write_32768x4096_20x512_20x128", seed, 32768, 4096, 20, 20)


def config_append(seed: int = 5) -> WriteWorkload:
    """Decode-time append: the new token of each of the decode batch's 64 sequences (at
    position 131072, the first slot of a fresh page), projected by the same 20 latent and
    20 indexer-key projections of d_model 4096."""
    return WriteWorkload("decode_append_64x4096_20x512_20x128", seed, 64, 4096, 20, 20,
                         append_pos=131072)


def d_model_pow2_scale(d_model: int) -> int:
    """Weights are N(0, 1/d_model) scaled by a power of two: the exponent of the power of
    two nearest at or above 1/sqrt(d_model) (exactly 1/sqrt(d) = 2**-6 for d = 4096)."""
    return -(int(math.log2(d_model)) // 2)
