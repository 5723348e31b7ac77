// CSA2 indexer kernels (tech-report digest, jiwasawa.github.io, section "Compressed
// Sparse Attention 2 (CSA2)": Full / Reindex / Reuse modes and the Hierarchical
// Sparse Indexer; zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮").
//
// Scoring (score_s = sum_h ReLU(q_h . k_s), 4 heads x 128 dims, fp32 accumulation)
// writes one 32-bit ranking key per candidate into the workspace:
//     key = (bits(score) & 0x7fffffff) + 1   for a valid candidate (score >= 0),
//     key = 0                                for an invalid one (pool padding, bad page).
// Keys order like the scores, every valid key is above every invalid one, and bit 31
// of a valid key is always clear.  Selection then takes the top-min(K, #valid) keys
// (and the top-min(P, #valid) pool), the lower candidate position winning ties, and
// writes their tokens in ascending order.
//
// Kernels:
//   group_prefix_kernel  FULL: compact work list (runs of queries, units of rows); its
//                        extra CTAs clear the selection histograms
//   score_pages_kernel   FULL: 64-token pages streamed by TMA into a shared ring, scored
//                        by tensor-core MMAs (1-4 draft queries of a sequence at once);
//                        also builds each query's selection histogram
//   score_gather_kernel  REINDEX: pool rows gathered by per-lane cp.async rings, scored
//                        by the same MMAs (an arithmetic work list: P rows per query)
//   select_cta_kernel    one 1024-thread CTA per query up to 2^18 keys: exact histogram,
//                        boundary bins, ordered filter, radix passes over the boundary
//                        bin, ordered emit
//   select_pool_kernel   REINDEX pools up to 16384 entries: one 512-thread CTA per query,
//                        keys in registers, three radix steps, one scan for the emit
//   select_filter_kernel / select_resolve_kernel / select_emit_kernel
//                        FULL beyond 2^18 tokens: several filter CTAs per query, one
//                        resolving CTA, one emitting warp per candidate list
//   select_kernel        1-8-CTA cluster per query for more than 8192 outputs: four
//                        8-bit radix passes with per-warp histograms merged through
//                        distributed shared memory, then an ordered compaction
#include <cooperative_groups.h>
#include <cstddef>

#include "async.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

// ------------------------------------------------------------------ scoring -------

// Selection histograms: the top 11 bits of a ranking key (8 exponent + 3 mantissa bits).
constexpr int kHistBins = 2048;
__device__ __forceinline__ uint32_t hist_bin(uint32_t key) {
  return min(key >> 20, (uint32_t)kHistBins - 1);  // finite scores give bins < 2041
}

constexpr int kScoreThreads = 128;     // Reindex scorer: 4 warps per CTA
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kGatherCtasPerSm = 5;    // five such CTAs per SM

struct ScoreGeom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t max_pages;
  int32_t num_pages;
  int32_t num_seqs;
};

__device__ __forceinline__ uint32_t rank_key(float score) {
  return (__float_as_uint(score) & 0x7FFFFFFFu) + 1u;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

// The warp's contiguous share [g0, g1) of `total` groups.
__device__ __forceinline__ void warp_share(int64_t total, int64_t& g0, int64_t& g1) {
  const int64_t nw = (int64_t)gridDim.x * kScoreWarps;
  const int64_t w = (int64_t)blockIdx.x * kScoreWarps + (threadIdx.x >> 5);
  const int64_t per = (total + nw - 1) / nw;
  g0 = min(total, w * per);
  g1 = min(total, g0 + per);
}

// Compact work list of a scoring launch.  A run is one query (single-query scorer) or
// the queries of one sequence (batched scorer); run r covers used(r) = ceil(rows / u)
// work units of u rows (u = 8: a group of 8 key rows; u = 64: a whole page).  group_prefix_kernel (one CTA) writes
//   meta[0] = R (runs), meta[1] = total groups,
//   run_q0[r] = first query of run r (r <= R, run_q0[R] = num_q),
//   prefix[r] = groups before run r (r <= R).
struct RunList {
  const int64_t* meta;
  const int64_t* prefix;
  const int32_t* run_q0;
};

// CTA order of the Full selection: bucket 0 holds the longest contexts (2^18 rows)
constexpr int kOrderBuckets = 65;
__device__ __forceinline__ int order_bucket(int rows) { return 64 - min(rows >> 12, 64); }

__device__ __forceinline__ int run_rows(bool reindex, const int32_t* __restrict__ q_seq, int q,
                                        const ScoreGeom& g, int32_t pool_size) {
  if (reindex) return pool_size;
  const int b = __ldg(q_seq + q);
  if (b < 0 || b >= g.num_seqs) return 0;
  return min(max(0, __ldg(g.seq_lens + b)), g.max_pages * kPage);
}

// CTA 0 builds the run list; CTAs 1.. clear `zero_buf` (zero_vecs 16-byte vectors: the
// Full scorer's selection histograms), which saves a separate memset in the stream.  With
// `order`, the last CTA writes the Full selection's CTA order: the queries by descending
// context length (buckets of 4096 rows), so that the longest selections start first and
// the short ones fill in behind them.
__global__ void __launch_bounds__(1024) group_prefix_kernel(bool batched, bool reindex,
                                                            const int32_t* __restrict__ q_seq,
                                                            int32_t num_q, ScoreGeom g,
                                                            int32_t pool_size, int32_t unit_rows,
                                                            int64_t* meta, int64_t* prefix,
                                                            int32_t* run_q0, uint4* zero_buf,
                                                            int64_t zero_vecs, int32_t* order) {
  grid_dep_wait();
  if (order != nullptr && blockIdx.x == gridDim.x - 1) {
    __shared__ uint32_t cb[kOrderBuckets];
    for (int i = threadIdx.x; i < kOrderBuckets; i += blockDim.x) cb[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < num_q; i += blockDim.x)
      atomicAdd(&cb[order_bucket(run_rows(false, q_seq, i, g, 0))], 1u);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t run = 0;
      for (int b = 0; b < kOrderBuckets; ++b) {
        const uint32_t c = cb[b];
        cb[b] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < num_q; i += blockDim.x)
      order[atomicAdd(&cb[order_bucket(run_rows(false, q_seq, i, g, 0))], 1u)] = i;
    return;
  }
  if (blockIdx.x > 0) {
    const int64_t stride = (int64_t)(gridDim.x - 1 - (order != nullptr)) * blockDim.x;
    for (int64_t i = (int64_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < zero_vecs; i += stride)
      zero_buf[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  __shared__ int64_t wsum[32];
  __shared__ int64_t carry_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto block_incl_scan = [&](int64_t v) -> int64_t {  // inclusive scan, returns the value
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int64_t add = 0;
    for (int w = 0; w < warp; ++w) add += wsum[w];
    __syncthreads();
    return x + add;
  };
  // pass 1: run starts (one query per run unless batched)
  if (tid == 0) carry_s = batched ? 0 : num_q;
  __syncthreads();
  if (!batched)
    for (int i = tid; i < num_q; i += 1024) run_q0[i] = i;
  for (int base = 0; batched && base < num_q; base += 1024) {
    const int i = base + tid;
    int start = 0;
    if (i < num_q) {
      const int b = __ldg(q_seq + i);
      start = (!batched || i == 0 || b != __ldg(q_seq + i - 1)) ? 1 : 0;
    }
    const int64_t incl = block_incl_scan(start);
    const int64_t carry = carry_s;
    if (start) run_q0[carry + incl - 1] = i;
    __syncthreads();
    if (tid == 1023) carry_s = carry + incl;
    __syncthreads();
  }
  const int R = (int)carry_s;
  if (tid == 0) run_q0[R] = num_q;
  __threadfence_block();
  __syncthreads();
  // pass 2: groups per run, exclusive prefix
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < R; base += 1024) {
    const int r = base + tid;
    int64_t used = 0;
    if (r < R) used = (run_rows(reindex, q_seq, run_q0[r], g, pool_size) + unit_rows - 1) / unit_rows;
    const int64_t incl = block_incl_scan(used);
    const int64_t carry = carry_s;
    if (r < R) prefix[r + 1] = carry + incl;
    __syncthreads();
    if (tid == 1023) carry_s = carry + incl;
    __syncthreads();
  }
  if (tid == 0) {
    prefix[0] = 0;
    meta[0] = R;
    meta[1] = carry_s;
  }
}

// Cursor over the compact list: run index and its [start, end) group range.
struct RunCursor {
  int r;
  int64_t start, end;
};
__device__ __forceinline__ void cursor_seek(RunCursor& cu, const RunList& rl, int R, int64_t gg) {
  int lo = 0, hi = R - 1;  // last run with prefix[r] <= gg
  while (lo < hi) {
    const int m = (lo + hi + 1) >> 1;
    if (__ldg(rl.prefix + m) <= gg) lo = m; else hi = m - 1;
  }
  cu.r = lo;
  cu.start = __ldg(rl.prefix + lo);
  cu.end = __ldg(rl.prefix + lo + 1);
}
__device__ __forceinline__ void cursor_advance(RunCursor& cu, const RunList& rl, int64_t gg) {
  while (gg >= cu.end) {
    ++cu.r;
    cu.start = cu.end;
    cu.end = __ldg(rl.prefix + cu.r + 1);
  }
}

// REINDEX: query q's P pool positions are groups [q u, (q + 1) u) of 16 rows, u =
// ceil(P / 16), so the work list is plain arithmetic; the rows are
// gathered (pool entry -> page table -> slot) through the per-lane cp.async ring and
// scored on the tensor cores exactly like the page scorer (M = 16 gathered keys,
// N = 8 columns holding the query's 4 heads, K = 128 dims in the shared permuted order).
// More warps with one group in flight each measured faster than fewer warps with three
// (decode batch Reindex call 41.5 -> 39.8 us at 5 CTAs per SM and 2-group rings).
constexpr int kGatherRing = 2;                       // 16-row groups staged per warp
constexpr int kGatherGroup = 16 * kKeyRow;           // 4 KB
constexpr int kGatherSmem = kScoreWarps * kGatherRing * kGatherGroup;  // 32 KB

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kScoreThreads, kGatherCtasPerSm)
    score_gather_kernel(const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ keys,
                        const int32_t* __restrict__ q_seq, int32_t num_q, ScoreGeom g,
                        const int32_t* __restrict__ pool, int32_t pool_size,
                        uint32_t* __restrict__ ws, int32_t* st) {
  grid_dep_wait();
  extern __shared__ __align__(128) unsigned char gather_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, c = lane & 3;
  // chunk XOR of this lane's rows: the two rows read in one quarter-warp phase
  // (gq = 2p, 2p + 1) get masks p and p + 4, so their 16-byte chunks fill all 32 banks
  const int sw = (gq >> 1) | ((gq & 1) << 2);
  const uint32_t ring = smem_addr(gather_smem) + warp * kGatherRing * kGatherGroup;
  const int64_t used = (pool_size + 15) / 16;  // groups per query
  int64_t g0, g1;
  warp_share((int64_t)num_q * used, g0, g1);
  if (g0 >= g1) return;

  struct QInfo {
    int q = -1, b = -1, n_ctx = 0;
  };
  auto info = [&](int q) {
    QInfo f;
    f.q = q;
    const int b = __ldg(q_seq + q);
    if (b >= 0 && b < g.num_seqs) {
      f.b = b;
      f.n_ctx = min(max(0, __ldg(g.seq_lens + b)), g.max_pages * kPage);
    }
    return f;
  };
  // Rows of a group as loaded pool entries: the pool loads of group gg + kGatherRing are
  // issued one iteration before the group's page-table lookups and copies, so their
  // latency overlaps the scoring of the current group.
  struct PoolRows {
    int b = -1, n_ctx = 0;
    int ta = -1, tb = -1;  // tokens of rows gq and gq + 8 (-1: none)
  };
  // cursor over the queries: query r owns groups [start, start + used)
  auto advance = [&](RunCursor& cu, int64_t gg) {
    while (gg >= cu.end) {
      ++cu.r;
      cu.start = cu.end;
      cu.end = cu.start + used;
    }
  };
  RunCursor lc, cc;
  lc.r = (int)(g0 / used);
  lc.start = (int64_t)lc.r * used;
  lc.end = lc.start + used;
  cc = lc;
  QInfo li = info(lc.r), ci;
  auto load_pool = [&](int64_t gg) -> PoolRows {
    PoolRows r;
    if (gg >= g1) return r;
    advance(lc, gg);
    if (lc.r != li.q) li = info(lc.r);
    if (li.b < 0) return r;
    r.b = li.b;
    r.n_ctx = li.n_ctx;
    const int pos = (int)(gg - lc.start) * 16 + gq;
    const int32_t* pq = pool + (int64_t)li.q * pool_size;
    if (pos < pool_size) r.ta = __ldg(pq + pos);
    if (pos + 8 < pool_size) r.tb = __ldg(pq + pos + 8);
    return r;
  };
  // token -> key row (nullptr: skip), with fault reporting
  auto row_of = [&](int b, int n_ctx, int t) -> const uint16_t* {
    if (t < 0 || t >= n_ctx) {
      if (t != -1 && c == 0) report(st, CSA2_DEV_BAD_INDEX);
      return nullptr;
    }
    const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (t >> 6));
    if (pg < 0 || pg >= g.num_pages) {
      if (c == 0) report(st, CSA2_DEV_BAD_PAGE);
      return nullptr;
    }
    return keys + ((int64_t)pg * kPage + (t & (kPage - 1))) * kDidx;
  };
  uint32_t okmask = 0;  // 2 bits per ring slot: rows gq and gq + 8 of the group loaded
  auto issue = [&](const PoolRows& pr, int sl) {
    okmask &= ~(3u << (2 * sl));
    if (pr.b >= 0) {
      const uint32_t slot = ring + sl * kGatherGroup;
      const uint16_t* ra = row_of(pr.b, pr.n_ctx, pr.ta);
      const uint16_t* rb = row_of(pr.b, pr.n_ctx, pr.tb);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = 4 * j + c;
        if (ra) cp_async16(slot + gq * kKeyRow + ((k ^ sw) << 4), reinterpret_cast<const char*>(ra) + 16 * k);
        if (rb) cp_async16(slot + (gq + 8) * kKeyRow + ((k ^ sw) << 4), reinterpret_cast<const char*>(rb) + 16 * k);
      }
      okmask |= ((ra ? 1u : 0u) | (rb ? 2u : 0u)) << (2 * sl);
    }
    cp_async_commit();
  };
  uint32_t bq[4][4];
  int slot = 0;
#pragma unroll
  for (int i = 0; i < kGatherRing - 1; ++i) issue(load_pool(g0 + i), i);
  PoolRows next = load_pool(g0 + kGatherRing - 1);
  for (int64_t gg = g0; gg < g1; ++gg) {
    const PoolRows cur = next;
    next = load_pool(gg + kGatherRing);
    issue(cur, (slot + kGatherRing - 1) & (kGatherRing - 1));
    cp_async_wait<kGatherRing - 1>();
    advance(cc, gg);
    if (cc.r != ci.q) {
      ci = info(cc.r);
      if (ci.b < 0 && lane == 0) report(st, CSA2_DEV_BAD_QSEQ);
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // B fragments: column gq < 4 holds head gq
        uint4 v = make_uint4(0, 0, 0, 0);
        if (gq < kHidx)
          v = __ldg(reinterpret_cast<const uint4*>(q_idx + ((int64_t)ci.q * kHidx + gq) * kDidx +
                                                   32 * j + 8 * c));
        bq[j][0] = v.x; bq[j][1] = v.y; bq[j][2] = v.z; bq[j][3] = v.w;
      }
    }
    const uint32_t sbase = ring + slot * kGatherGroup;
    uint4 k0[4], k1[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = 4 * j + c;
      k0[j] = lds128(sbase + gq * kKeyRow + ((k ^ sw) << 4));
      k1[j] = lds128(sbase + (gq + 8) * kKeyRow + ((k ^ sw) << 4));
    }
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mma_bf16_16816(d, k0[j].x, k1[j].x, k0[j].y, k1[j].y, bq[j][0], bq[j][1]);
      mma_bf16_16816(d, k0[j].z, k1[j].z, k0[j].w, k1[j].w, bq[j][2], bq[j][3]);
    }
    float s0 = fmaxf(d[0], 0.f) + fmaxf(d[1], 0.f);
    float s1 = fmaxf(d[2], 0.f) + fmaxf(d[3], 0.f);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    if (c == 0 && ci.b >= 0) {
      const uint32_t ok = okmask >> (2 * slot);
      const int pos = (int)(gg - cc.start) * 16 + gq;
      uint32_t* out = ws + (int64_t)ci.q * pool_size;
      if (pos < pool_size) out[pos] = (ok & 1u) ? rank_key(s0) : 0u;
      if (pos + 8 < pool_size) out[pos + 8] = (ok & 2u) ? rank_key(s1) : 0u;
    }
    slot = (slot + 1) & (kGatherRing - 1);
  }
}

// ------------------------------------------------------------------ TMA page scorer --
// Full mode, contiguous context: the unit of work is a whole 64-token page (16 KB of
// keys).  One producer thread streams pages through a 2D tensor map (two 64 x 64 bf16
// boxes per page, 128-byte swizzle) into a 4-slot shared-memory ring; two such CTAs run
// on each SM.  The 4 consumer warps take every page: warp w scores rows 16w .. 16w+15
// as the 16 rows of one tensor-core tile:
//   D[16 keys][8 cols] = K[16 keys][16 dims] x Q^T[16 dims][8 cols]   (m16n8k16, bf16)
// where the 8 columns of an n-tile are (query, head) pairs 4t + h of two queries, so
// one n-tile serves 1-2 queries and two serve 3-4 draft queries of a sequence.  Dims
// are visited in the same permuted order on both sides: lane c's 16-byte chunk of dims
// 32j + 8c .. +7 supplies its A and B fragments for k-steps 2j and 2j + 1.  A consumer
// releases a page as soon as it holds its rows in registers.
// Measured on B300: the CUDA-core form of this dot product (packed FFMA2, one key per 4
// lanes) ran at 124 us of pure arithmetic for 2.1M keys against 85 us to stream them,
// so the contraction runs on the tensor cores even for a single query; and one 9-warp
// CTA per SM with an 8-page ring streamed 2.1M keys in 115 us where two 5-warp CTAs
// per SM with 4-page rings take 96 us (ring depth alone made no difference).

constexpr int kPageStages = 4;  // ring depth per CTA
constexpr int kPageBytes = kPage * kKeyRow;            // 16 KB
constexpr int kConsumerWarps = 4;
constexpr int kTmaThreads = (kConsumerWarps + 1) * 32;  // + 1 producer warp
constexpr int kScoreCtasPerSm = 2;

struct PageRing {
  uint64_t full[kPageStages];
  uint64_t empty[kPageStages];
  int32_t run[kPageStages];   // run of the staged page
  int32_t page[kPageStages];  // page index within the run
  int32_t valid[kPageStages]; // 1 if its keys were loaded
  volatile int abort;
};
constexpr int kMaxDraft = 4;  // query tokens of one sequence scored together
constexpr size_t kRingOff = (sizeof(PageRing) + 15) / 16 * 16;
// page ring | ring state | per-query selection histograms of the current run
constexpr size_t kTmaSmem = (size_t)kPageStages * kPageBytes + kRingOff +
                            (size_t)kMaxDraft * kHistBins * 4 + 1024;

// Row `row` (0..63), 16-byte chunk `k` (0..15) of a staged page: two 8 KB halves
// (dims 0-63, 64-127), each 64 rows of 128 bytes with the chunk index XOR-ed by row % 8.
__device__ __forceinline__ uint32_t page_chunk(uint32_t base, int row, int k) {
  return base + (uint32_t)((k >> 3) * 8192 + row * 128 + (((k & 7) ^ (row & 7)) << 4));
}
__device__ __forceinline__ void read_page_row(uint4 (&kv)[4], uint32_t base, int row, int c) {
#pragma unroll
  for (int j = 0; j < 4; ++j) kv[j] = lds128(page_chunk(base, row, 4 * j + c));
}

__global__ void __launch_bounds__(kTmaThreads, kScoreCtasPerSm)
    score_pages_kernel(const __grid_constant__ CUtensorMap keymap, const uint16_t* __restrict__ q_idx,
                       const int32_t* __restrict__ q_seq, int32_t num_q, ScoreGeom g,
                       uint32_t* __restrict__ ws, int64_t ws_stride, RunList rl,
                       uint32_t* __restrict__ ghist, int32_t* st) {
  grid_dep_wait();
  extern __shared__ __align__(1024) unsigned char page_smem_raw[];
  unsigned char* data = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(page_smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int S = kPageStages;
  PageRing* ring = reinterpret_cast<PageRing*>(data + S * kPageBytes);
  uint32_t* shist = reinterpret_cast<uint32_t*>(data + S * kPageBytes + kRingOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ring->full[s], 1);
      mbar_init(&ring->empty[s], kConsumerWarps);
    }
    ring->abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const int R = (int)__ldg(rl.meta);
  const int64_t total = __ldg(rl.meta + 1);
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const int64_t p0 = min(total, (int64_t)blockIdx.x * per), p1 = min(total, p0 + per);
  const uint32_t data_s = saddr(data);

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0 && p0 < p1) {
      RunCursor cu;
      cursor_seek(cu, rl, R, p0);
      uint32_t issued = 0, last_par = 0;
      int s = 0;
      uint32_t ph = 0;
      for (int64_t i = p0; i < p1; ++i) {
        if (!mbar_wait(&ring->abort, &ring->empty[s], ph ^ 1u, st)) break;
        cursor_advance(cu, rl, i);
        const int page = (int)(i - cu.start);
        const int b = __ldg(q_seq + __ldg(rl.run_q0 + cu.r));
        int32_t pg = -1;
        if (b >= 0 && b < g.num_seqs) pg = __ldg(g.page_table + (int64_t)b * g.max_pages + page);
        ring->run[s] = cu.r;
        ring->page[s] = page;
        if (pg >= 0 && pg < g.num_pages) {
          ring->valid[s] = 1;
          unsigned char* dst = data + s * kPageBytes;
          mbar_expect_tx(&ring->full[s], kPageBytes);
          tma_load_2d(dst, &keymap, &ring->full[s], 0, pg * kPage);
          tma_load_2d(dst + 8192, &keymap, &ring->full[s], 64, pg * kPage);
          issued |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
        } else {
          ring->valid[s] = 0;
          report(st, CSA2_DEV_BAD_PAGE);
          mbar_arrive(&ring->full[s]);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ring->abort)  // our copies must land before the CTA's shared memory is released
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) (void)mbar_wait(&ring->abort, &ring->full[s], (last_par >> s) & 1u, st, 1u << 20);
    }
  } else {
    // ---------------- consumers: every warp takes every page ----
    // this lane's rows rr and rr + 8 of each page: the lane groups gq = 2p, 2p + 1 of a
    // quarter-warp phase read rows whose 128-byte swizzle masks (row % 8) are p and p + 4,
    // so their 16-byte chunks land in disjoint bank halves (no bank conflict)
    const int rr = 16 * warp + ((gq >> 1) | ((gq & 1) << 2));
    int cur_run = -1, rows = 0, q0 = 0, T = 0, NT = 0;
    uint32_t bq[2][4][4];  // [n-tile][j][word]: B fragments of Q^T
    // Selection histograms (ghist != nullptr): per query of the current run, counts of
    // the stored ranking keys by top 11 bits, added to the global per-query histograms
    // when the run ends.  Every consumer warp sees every page, so all of them reach each
    // flush together (named barrier 1 over the consumer warps).
    auto consumers_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); };
    auto flush = [&]() {
      consumers_sync();
      for (int i = threadIdx.x; i < T * kHistBins; i += kConsumerWarps * 32) {
        const uint32_t v = shist[i];
        if (v != 0) {
          atomicAdd(ghist + (int64_t)(q0 + i / kHistBins) * kHistBins + (i % kHistBins), v);
          shist[i] = 0;
        }
      }
      consumers_sync();
    };
    if (ghist != nullptr) {
      for (int i = threadIdx.x; i < kMaxDraft * kHistBins; i += kConsumerWarps * 32) shist[i] = 0;
      consumers_sync();
    }
    auto enter = [&](int r) {
      if (r == cur_run) return;
      if (cur_run >= 0 && ghist != nullptr) flush();
      cur_run = r;
      q0 = __ldg(rl.run_q0 + r);
      T = __ldg(rl.run_q0 + r + 1) - q0;
      if (T > 4) {
        if (lane == 0) report(st, CSA2_DEV_BAD_QSEQ);
        T = 4;
      }
      NT = (T + 1) >> 1;
      const int b = __ldg(q_seq + q0);
      rows = (b >= 0 && b < g.num_seqs) ? min(max(0, __ldg(g.seq_lens + b)), g.max_pages * kPage) : 0;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int t = 2 * nt + (gq >> 2), h = gq & 3;  // column gq of n-tile nt
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (t < T)
            v = __ldg(reinterpret_cast<const uint4*>(
                q_idx + ((int64_t)(q0 + t) * kHidx + h) * kDidx + 32 * j + 8 * c));
          bq[nt][j][0] = v.x; bq[nt][j][1] = v.y; bq[nt][j][2] = v.z; bq[nt][j][3] = v.w;
        }
      }
    };
    // MMA over rows ra and rb of one page with the current run's Q
    auto tile = [&](const uint4 (&ka)[4], const uint4 (&kb)[4], int page, int ra, int rb,
                    bool valid) {
      float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // k-step 2j: words x, y; k-step 2j + 1: words z, w
        mma_bf16_16816(d[0], ka[j].x, kb[j].x, ka[j].y, kb[j].y, bq[0][j][0], bq[0][j][1]);
        mma_bf16_16816(d[0], ka[j].z, kb[j].z, ka[j].w, kb[j].w, bq[0][j][2], bq[0][j][3]);
        if (NT > 1) {
          mma_bf16_16816(d[1], ka[j].x, kb[j].x, ka[j].y, kb[j].y, bq[1][j][0], bq[1][j][1]);
          mma_bf16_16816(d[1], ka[j].z, kb[j].z, ka[j].w, kb[j].w, bq[1][j][2], bq[1][j][3]);
        }
      }
      // d[nt][0..1]: row a, columns 2c, 2c+1; d[nt][2..3]: row b.  Columns 4t'+h of
      // query t' = 2nt + c/2: ReLU, then sum the query's 4 heads over lanes c, c^1.
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        if (nt >= NT) break;
        float s0 = fmaxf(d[nt][0], 0.f) + fmaxf(d[nt][1], 0.f);
        float s1 = fmaxf(d[nt][2], 0.f) + fmaxf(d[nt][3], 0.f);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        const int t = 2 * nt + (c >> 1);
        if ((c & 1) == 0 && t < T) {
          uint32_t* out = ws + (int64_t)(q0 + t) * ws_stride;
          const int ta = page * kPage + ra, tb = page * kPage + rb;
          const uint32_t k0 = valid ? rank_key(s0) : 0u, k1 = valid ? rank_key(s1) : 0u;
          if (ta < rows) out[ta] = k0;
          if (tb < rows) out[tb] = k1;
          if (ghist != nullptr && valid) {
            if (ta < rows) atomicAdd(&shist[t * kHistBins + hist_bin(k0)], 1u);
            if (tb < rows) atomicAdd(&shist[t * kHistBins + hist_bin(k1)], 1u);
          }
        }
      }
    };
    int s = 0;
    uint32_t ph = 0;
    for (int64_t i = p0; i < p1; ++i) {
      if (!mbar_wait(&ring->abort, &ring->full[s], ph, st)) break;
      const int run = ring->run[s], page = ring->page[s];
      const bool valid = ring->valid[s] != 0;
      uint4 k0[4], k1[4];
      read_page_row(k0, data_s + s * kPageBytes, rr, c);
      read_page_row(k1, data_s + s * kPageBytes, rr + 8, c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ring->empty[s]);  // the keys are in registers now
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
      enter(run);
      tile(k0, k1, page, rr, rr + 8, valid);
    }
    if (cur_run >= 0 && ghist != nullptr) flush();
  }
  __syncthreads();
}

// ------------------------------------------------------------------ selection -----

constexpr int kSelMaxCluster = 8;  // CTAs per query: 1, 2, 4 or 8, chosen per launch
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCacheKeys = 16384;  // per-CTA keys kept in shared memory (64 KB)
constexpr int kDigit = 256;
constexpr int kSamplesPerCta = 256;
constexpr int kMaxSamples = kSelMaxCluster * kSamplesPerCta;  // up to 2048 samples per query
constexpr int kCandCap = 256;                           // kept positions per warp per target

struct SelShared {
  union {
    uint32_t whist[kSelWarps][2][kDigit];  // per-warp histograms (full-sweep path)
    struct {
      uint32_t samp[kMaxSamples];           // the cluster's samples
      uint32_t mysamp[kSamplesPerCta];      // this CTA's samples (read by the cluster)
      uint32_t samp2[2048];                 // histogram of the samples' top 11 bits
      uint16_t cand[2][kSelWarps][kCandCap];  // kept positions per target, per warp
    } f;
  } u;
  uint32_t lhist[2][kDigit];                // CTA histograms (samples, kept keys)
  uint32_t chist[2][2][kDigit];             // [buffer][target][bin]: read by the cluster
  uint32_t wcnt[kSelWarps][4];              // per-warp (gt, eq) counts of both targets
  uint32_t ccnt[4];                         // this CTA's (gt, eq) counts
  uint32_t wvalid[kSelWarps];
  uint32_t cvalid;
  uint32_t wcand[kSelWarps][2];             // kept keys per warp and target
  uint32_t ccand[2];
  uint32_t cover;                           // a warp of this CTA overflowed its buffer
  uint32_t nzs;                             // non-zero samples of the cluster
  uint32_t scan[2][kDigit / 32];
  uint32_t res_prefix[2], res_above[2];
};

// The key cache follows SelShared at a 128-byte boundary (it is read as uint4).
constexpr size_t kSelCacheOff = (sizeof(SelShared) + 127) / 128 * 128;
static_assert(kSelCacheOff % 16 == 0, "key cache must be 16-byte aligned");

// Warp-wide exclusive prefix sum of v and the warp total.
__device__ __forceinline__ uint32_t warp_excl(uint32_t v, uint32_t& total) {
  const int lane = threadIdx.x & 31;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// One radix step for up to two targets.  Thread tid holds v = keys in bin tid % 256 of
// target tid / 256 (keys whose higher digits equal pre_t).  For each target with
// want_t > 0, find the bin in which the count of keys in strictly higher bins plus
// abv_t first reaches want_t, and extend pre_t by it (abv_t += keys above that bin).
__device__ __forceinline__ void find_bins(SelShared& sh, uint32_t v, int width, uint32_t want0,
                                          uint32_t want1, uint32_t& pre0, uint32_t& pre1,
                                          uint32_t& abv0, uint32_t& abv1) {
  const int tid = threadIdx.x, lane = tid & 31, t = tid / kDigit, bin = tid % kDigit;
  const int tw = bin >> 5;
  uint32_t x = v;  // inclusive suffix sum within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) sh.scan[t][tw] = x;
  __syncthreads();
  const uint32_t want_t = t == 0 ? want0 : want1;
  if (want_t > 0) {
    uint32_t later = 0;
    for (int w = tw + 1; w < kDigit / 32; ++w) later += sh.scan[t][w];
    const uint32_t above_bin = (t == 0 ? abv0 : abv1) + later + x - v;
    if (above_bin < want_t && above_bin + v >= want_t) {
      sh.res_prefix[t] = ((t == 0 ? pre0 : pre1) << width) | (uint32_t)bin;
      sh.res_above[t] = above_bin;
    }
  }
  __syncthreads();
  if (want0 > 0) {
    pre0 = sh.res_prefix[0];
    abv0 = sh.res_above[0];
  }
  if (want1 > 0) {
    pre1 = sh.res_prefix[1];
    abv1 = sh.res_above[1];
  }
  __syncthreads();
}

__device__ __forceinline__ int digit_shift(int pass) {
  return pass == 0 ? 23 : pass == 1 ? 15 : pass == 2 ? 7 : 0;
}
__device__ __forceinline__ int digit_width(int pass) { return pass == 3 ? 7 : 8; }

// Top-k selection for one query per C-CTA cluster (gridDim.y = num_q).  Target t = 0 is
// the top-K output, t = 1 the candidate pool (FULL with a pool output only).
//
// Fast path: every CTA takes 256 evenly spaced samples of its range; from the
// cluster's 256 C samples each target gets a threshold tau_t: the lower edge of the
// 1/8-octave bin holding the r-th largest sample, r = 1.25 e + 4 sqrt(e) + 8, where
// e = want * 256 C / n samples are expected above the answer.  One ordered sweep keeps the positions of keys >= tau_t; if the kept
// keys number at least want_t (and no warp overflowed its buffer) they contain every
// key of the answer, ties included, so the exact radix select and the ordered output
// run over the kept keys only.  Otherwise the cluster falls back to radix passes over
// the whole range.  Either way the result is exact.
template <bool kReindex, int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(kSelThreads, 2)
    select_kernel(const uint32_t* __restrict__ ws, int64_t ws_stride,
                  const int32_t* __restrict__ q_seq, const int32_t* __restrict__ seq_lens,
                  int32_t num_seqs, const int32_t* __restrict__ pool_in, int32_t pool_size,
                  int32_t topk, int32_t* __restrict__ out_idx, int32_t* __restrict__ pool_out,
                  int32_t max_ctx, int32_t* st) {
  grid_dep_wait();
  constexpr int kS = C * kSamplesPerCta;  // samples per query
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem_raw + kSelCacheOff);  // 16-B vector reads
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int q = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int n;
  if (kReindex) {
    n = pool_size;
  } else {
    const int b = __ldg(q_seq + q);
    n = (b >= 0 && b < num_seqs) ? min(max(0, __ldg(seq_lens + b)), max_ctx) : 0;
  }
  const bool two = (!kReindex && pool_out != nullptr && pool_size > 0);
  const uint32_t want_max0 = (uint32_t)topk, want_max1 = two ? (uint32_t)pool_size : 0u;

  // This CTA's range of candidate positions, cut into 16 contiguous warp segments
  // (multiples of 128) so that outputs keep index order with warp scans.
  int L = (n + C - 1) / C;
  L = (L + 127) & ~127;
  const int lo = min(n, rank * L), hi = min(n, lo + L);
  const int len = hi - lo;
  int S = (len + kSelWarps - 1) / kSelWarps;
  S = (S + 127) & ~127;
  const int seg_lo = min(len, warp * S), seg_hi = min(len, seg_lo + S);
  const uint32_t* src = ws + (int64_t)q * ws_stride + lo;
  const bool cached = len <= kSelCacheKeys;
  if (cached) {
    for (int i = tid; i < len; i += kSelThreads) cache[i] = __ldcg(src + i);
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : __ldcg(src + i); };
  // keys i .. i+3 of this CTA's range (i a multiple of 4); positions past seg_hi read 0
  auto load4 = [&](int i, uint32_t (&k)[4]) {
    if (cached && i + 4 <= seg_hi) {
      const uint4 v = *reinterpret_cast<const uint4*>(cache + i);
      k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) k[e] = (i + e < seg_hi) ? key_at(i + e) : 0u;
    }
  };

  uint32_t want0 = 0, want1 = 0, pre0 = 0, pre1 = 0, abv0 = 0, abv1 = 0;
  int32_t* out0 = out_idx + (int64_t)q * topk;
  int32_t* out1 = two ? pool_out + (int64_t)q * pool_size : nullptr;
  const int32_t* pin = kReindex ? pool_in + (int64_t)q * pool_size + lo : nullptr;

  // ======== fast path, part 1: samples -> thresholds -> one filtering sweep ========
  const bool fast_ok = L <= 65535;  // kept positions are stored as 16 bits
  bool fast = false;
  if (fast_ok) {
    for (int i = tid; i < kSamplesPerCta; i += kSelThreads) {
      uint32_t v = 0;
      if (len >= kSamplesPerCta) v = key_at((int)(((int64_t)i * len) / kSamplesPerCta));
      else if (i < len) v = key_at(i);
      sh.u.f.mysamp[i] = v;
    }
    cluster.sync();
    uint32_t nz = 0;
    for (int i = tid; i < kS; i += kSelThreads) {
      const uint32_t v = *cluster.map_shared_rank(&sh.u.f.mysamp[i % kSamplesPerCta], i / kSamplesPerCta);
      sh.u.f.samp[i] = v;
      nz += v != 0;
    }
    nz = __reduce_add_sync(0xffffffffu, nz);
    if (tid == 0) sh.nzs = 0;
    __syncthreads();
    if (lane == 0) atomicAdd(&sh.nzs, nz);
    __syncthreads();
    const uint32_t n_s = sh.nzs;
    // rank of the threshold among the non-zero samples, per target
    uint32_t r0 = 0, r1 = 0;
    {
      const double e0 = (double)want_max0 * kS / (double)max(n, 1);
      const double e1 = (double)want_max1 * kS / (double)max(n, 1);
      r0 = (uint32_t)ceil(1.25 * e0 + 4.0 * sqrt(e0) + 8.0);
      r1 = two ? (uint32_t)ceil(1.25 * e1 + 4.0 * sqrt(e1) + 8.0) : 0u;
      r0 = min(r0, n_s);
      r1 = min(r1, n_s);
    }
    // tau_t = lower edge of the bin (top 11 key bits: exponent + 3 mantissa bits) in
    // which the count of samples from the top reaches r_t; at least r_t samples are >= it
    for (int i = tid; i < 2048; i += kSelThreads) sh.u.f.samp2[i] = 0;
    __syncthreads();
    for (int i = tid; i < kS; i += kSelThreads) {
      const uint32_t k = sh.u.f.samp[i];
      if (k != 0) atomicAdd(&sh.u.f.samp2[k >> 20], 1u);
    }
    __syncthreads();
    uint32_t tau0 = 1u, tau1 = 1u;
    {
      // thread tid owns bins 4 tid .. 4 tid + 3; suffix counts over the block
      uint32_t v4[4], mine = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v4[e] = sh.u.f.samp2[4 * tid + e];
        mine += v4[e];
      }
      uint32_t x = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      if (lane == 0) sh.wvalid[warp] = x;  // warp totals (reused scratch)
      __syncthreads();
      uint32_t later = 0;
      for (int w = warp + 1; w < kSelWarps; ++w) later += sh.wvalid[w];
      uint32_t acc = later + x - mine;  // samples in bins above this thread's bins
      if (tid == 0) {
        sh.res_prefix[0] = 1u;
        sh.res_prefix[1] = 1u;
      }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t r_t = t == 0 ? r0 : r1;
        if (r_t == 0) continue;
        uint32_t a = acc;
        for (int e = 3; e >= 0; --e) {
          if (a < r_t && a + v4[e] >= r_t) sh.res_prefix[t] = (uint32_t)(4 * tid + e) << 20;
          a += v4[e];
        }
      }
      __syncthreads();
      tau0 = max(1u, sh.res_prefix[0]);
      tau1 = max(1u, sh.res_prefix[1]);
      __syncthreads();
    }
    // ordered filtering sweep, 4 consecutive keys per lane per step
    uint32_t cnt0 = 0, cnt1 = 0, nval = 0;
    for (int i0 = seg_lo; i0 < seg_hi; i0 += 128) {
      const int i = i0 + 4 * lane;
      uint32_t k[4];
      load4(i, k);
      uint32_t m0 = 0, m1 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        nval += k[e] != 0;
        if (k[e] != 0 && k[e] >= tau0) m0 |= 1u << e;
        if (two && k[e] != 0 && k[e] >= tau1) m1 |= 1u << e;
      }
      uint32_t tot;
      uint32_t p = cnt0 + warp_excl(__popc(m0), tot);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m0 & (1u << e)) {
          if (p < kCandCap) sh.u.f.cand[0][warp][p] = (uint16_t)(i + e);
          ++p;
        }
      cnt0 += tot;
      if (two) {
        p = cnt1 + warp_excl(__popc(m1), tot);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (m1 & (1u << e)) {
            if (p < kCandCap) sh.u.f.cand[1][warp][p] = (uint16_t)(i + e);
            ++p;
          }
        cnt1 += tot;
      }
    }
    nval = __reduce_add_sync(0xffffffffu, nval);
    if (lane == 0) {
      sh.wcand[warp][0] = cnt0;
      sh.wcand[warp][1] = cnt1;
      sh.wvalid[warp] = nval;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t a = 0, b = 0, v = 0, ov = 0;
      for (int w = 0; w < kSelWarps; ++w) {
        a += sh.wcand[w][0];
        b += sh.wcand[w][1];
        v += sh.wvalid[w];
        ov |= (sh.wcand[w][0] > kCandCap || sh.wcand[w][1] > kCandCap) ? 1u : 0u;
      }
      sh.ccand[0] = a;
      sh.ccand[1] = b;
      sh.cvalid = v;
      sh.cover = ov;
    }
    cluster.sync();
    uint32_t nvalid = 0, ct0 = 0, ct1 = 0, ovf = 0;
#pragma unroll
    for (int r = 0; r < C; ++r) {
      nvalid += *cluster.map_shared_rank(&sh.cvalid, r);
      ct0 += *cluster.map_shared_rank(&sh.ccand[0], r);
      ct1 += *cluster.map_shared_rank(&sh.ccand[1], r);
      ovf |= *cluster.map_shared_rank(&sh.cover, r);
    }
    want0 = min(want_max0, nvalid);
    want1 = min(want_max1, nvalid);
    fast = ovf == 0 && ct0 >= want0 && (!two || ct1 >= want1);
  }

  if (fast) {
    // ======== fast path, part 2: exact radix select over the kept keys ========
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int buf = pass & 1, shift = digit_shift(pass), width = digit_width(pass);
      const uint32_t dmask = (1u << width) - 1u;
      sh.lhist[tid / kDigit][tid % kDigit] = 0;
      __syncthreads();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t want_t = t == 0 ? want0 : want1, pre_t = t == 0 ? pre0 : pre1;
        if (want_t == 0) continue;
        const uint32_t cnt = sh.wcand[warp][t];
        for (uint32_t j = lane; j < cnt; j += 32) {
          const uint32_t k = key_at(sh.u.f.cand[t][warp][j]);
          if (pass == 0 || (k >> (shift + width)) == pre_t)
            atomicAdd(&sh.lhist[t][(k >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      sh.chist[buf][tid / kDigit][tid % kDigit] = sh.lhist[tid / kDigit][tid % kDigit];
      cluster.sync();
      uint32_t v = 0;
      {
        uint32_t part[C];
#pragma unroll
        for (int r = 0; r < C; ++r)
          part[r] = *cluster.map_shared_rank(&sh.chist[buf][tid / kDigit][tid % kDigit], r);
#pragma unroll
        for (int r = 0; r < C; ++r) v += part[r];
      }
      find_bins(sh, v, width, want0, want1, pre0, pre1, abv0, abv1);
    }
    // counts per warp over its kept keys
    uint32_t gt[2] = {0, 0}, eq[2] = {0, 0};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t want_t = t == 0 ? want0 : want1, T = t == 0 ? pre0 : pre1;
      if (want_t == 0) continue;
      const uint32_t cnt = sh.wcand[warp][t];
      for (uint32_t j = lane; j < cnt; j += 32) {
        const uint32_t k = key_at(sh.u.f.cand[t][warp][j]);
        gt[t] += k > T;
        eq[t] += k == T;
      }
      gt[t] = __reduce_add_sync(0xffffffffu, gt[t]);
      eq[t] = __reduce_add_sync(0xffffffffu, eq[t]);
    }
    if (lane == 0) {
      sh.wcnt[warp][0] = gt[0];
      sh.wcnt[warp][1] = eq[0];
      sh.wcnt[warp][2] = gt[1];
      sh.wcnt[warp][3] = eq[1];
    }
  } else {
    // ======== full-sweep path: four radix passes over the whole range ========
    want0 = want1 = pre0 = pre1 = abv0 = abv1 = 0;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int buf = pass & 1, shift = digit_shift(pass), width = digit_width(pass);
      const uint32_t dmask = (1u << width) - 1u;
      const bool h1 = pass > 0 && two && want1 > 0;  // second histogram needed
      for (int i = lane; i < kDigit; i += 32) {
        sh.u.whist[warp][0][i] = 0;
        sh.u.whist[warp][1][i] = 0;
      }
      __syncwarp();
      uint32_t nval = 0;
      for (int i = seg_lo + 4 * lane; i < seg_hi; i += 128) {
        uint32_t k[4];
        load4(i, k);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t kk = k[e];
          if (kk == 0) continue;
          ++nval;
          const uint32_t top = kk >> (shift + width), d = (kk >> shift) & dmask;
          if (pass == 0 || (want0 > 0 && top == pre0)) atomicAdd(&sh.u.whist[warp][0][d], 1u);
          if (h1 && top == pre1) atomicAdd(&sh.u.whist[warp][1][d], 1u);
        }
      }
      if (pass == 0) {
        nval = __reduce_add_sync(0xffffffffu, nval);
        if (lane == 0) sh.wvalid[warp] = nval;
      }
      __syncthreads();
      {
        const int t = tid / kDigit, bin = tid % kDigit;
        uint32_t sum = 0;
#pragma unroll 4
        for (int w = 0; w < kSelWarps; ++w) sum += sh.u.whist[w][t][bin];
        sh.chist[buf][t][bin] = sum;
        if (pass == 0 && tid == 0) {
          uint32_t v = 0;
          for (int w = 0; w < kSelWarps; ++w) v += sh.wvalid[w];
          sh.cvalid = v;
        }
      }
      cluster.sync();
      if (pass == 0) {
        uint32_t nvalid = 0;
#pragma unroll
        for (int r = 0; r < C; ++r) nvalid += *cluster.map_shared_rank(&sh.cvalid, r);
        want0 = min(want_max0, nvalid);
        want1 = min(want_max1, nvalid);
      }
      const int t = tid / kDigit, bin = tid % kDigit;
      const int tsrc = pass == 0 ? 0 : t;
      uint32_t v = 0;
      if (bin <= (int)dmask) {
        uint32_t part[C];
#pragma unroll
        for (int r = 0; r < C; ++r) part[r] = *cluster.map_shared_rank(&sh.chist[buf][tsrc][bin], r);
#pragma unroll
        for (int r = 0; r < C; ++r) v += part[r];
      }
      find_bins(sh, v, width, want0, want1, pre0, pre1, abv0, abv1);
    }
    uint32_t gt0 = 0, eq0 = 0, gt1 = 0, eq1 = 0;
    for (int i = seg_lo + 4 * lane; i < seg_hi; i += 128) {
      uint32_t k[4];
      load4(i, k);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gt0 += want0 > 0 && k[e] > pre0;
        eq0 += want0 > 0 && k[e] == pre0;
        gt1 += want1 > 0 && k[e] > pre1;
        eq1 += want1 > 0 && k[e] == pre1;
      }
    }
    gt0 = __reduce_add_sync(0xffffffffu, gt0);
    eq0 = __reduce_add_sync(0xffffffffu, eq0);
    gt1 = __reduce_add_sync(0xffffffffu, gt1);
    eq1 = __reduce_add_sync(0xffffffffu, eq1);
    if (lane == 0) {
      sh.wcnt[warp][0] = gt0;
      sh.wcnt[warp][1] = eq0;
      sh.wcnt[warp][2] = gt1;
      sh.wcnt[warp][3] = eq1;
    }
  }
  // preT is the exact key of the want-th largest valid key, abvT the number of keys
  // strictly greater; wcnt holds every warp's (gt, eq) counts over what it will emit.
  __syncthreads();
  if (tid < 4) {
    uint32_t s2 = 0;
    for (int w = 0; w < kSelWarps; ++w) s2 += sh.wcnt[w][tid];
    sh.ccnt[tid] = s2;
  }
  cluster.sync();
  // output base and tie quota of this warp for target t
  auto place = [&](int t, uint32_t want_t, uint32_t abv_t, uint32_t& wbase, uint32_t& wtake) {
    const uint32_t quota = want_t - abv_t;  // ties of the boundary key, lowest positions first
    uint32_t ties_before = 0, base = 0;
    for (int r = 0; r < rank; ++r) {
      const uint32_t g_r = *cluster.map_shared_rank(&sh.ccnt[2 * t], r);
      const uint32_t e_r = *cluster.map_shared_rank(&sh.ccnt[2 * t + 1], r);
      base += g_r + (quota > ties_before ? min(quota - ties_before, e_r) : 0u);
      ties_before += e_r;
    }
    for (int w = 0; w < warp; ++w) {
      const uint32_t g_w = sh.wcnt[w][2 * t], e_w = sh.wcnt[w][2 * t + 1];
      base += g_w + (quota > ties_before ? min(quota - ties_before, e_w) : 0u);
      ties_before += e_w;
    }
    wbase = base;
    wtake = quota > ties_before ? min(quota - ties_before, sh.wcnt[warp][2 * t + 1]) : 0u;
  };
  uint32_t wbase0 = 0, wtake0 = 0, wbase1 = 0, wtake1 = 0;
  if (want0 > 0) place(0, want0, abv0, wbase0, wtake0);
  if (want1 > 0) place(1, want1, abv1, wbase1, wtake1);
  // emit the selected keys of a batch of (up to) 32 x NK keys held by the lanes, in
  // index order lane-major: lane l holds batch items [NK l, NK l + NK)
  auto emit = [&](const uint32_t* k, const int* pos, int nk, uint32_t T, uint32_t take,
                  uint32_t wbase, uint32_t want_t, uint32_t& tie_run, uint32_t& sel_run,
                  int32_t* outp) {
    uint32_t nt = 0;
    for (int e = 0; e < nk; ++e) nt += k[e] == T;
    uint32_t ttot;
    uint32_t tr = tie_run + warp_excl(nt, ttot);
    uint32_t selm = 0, ns = 0;
    for (int e = 0; e < nk; ++e) {
      const bool tie = k[e] == T;
      const bool sel = k[e] > T || (tie && tr < take);
      tr += tie;
      if (sel) {
        selm |= 1u << e;
        ++ns;
      }
    }
    uint32_t stot;
    uint32_t p = wbase + sel_run + warp_excl(ns, stot);
    for (int e = 0; e < nk; ++e)
      if (selm & (1u << e)) {
        const int i = pos[e];
        const int token = kReindex ? __ldg(pin + i) : lo + i;
        if (p < want_t) outp[p] = token;
        ++p;
      }
    tie_run += ttot;
    sel_run += stot;
  };
  if (fast) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t want_t = t == 0 ? want0 : want1;
      if (want_t == 0) continue;
      const uint32_t T = t == 0 ? pre0 : pre1;
      const uint32_t take = t == 0 ? wtake0 : wtake1, wbase = t == 0 ? wbase0 : wbase1;
      int32_t* outp = t == 0 ? out0 : out1;
      const uint32_t cnt = sh.wcand[warp][t];
      uint32_t tie_run = 0, sel_run = 0;
      for (uint32_t j0 = 0; j0 < cnt; j0 += 32) {
        const uint32_t j = j0 + lane;
        uint32_t k[1] = {0u};
        int pos[1] = {0};
        if (j < cnt) {
          pos[0] = sh.u.f.cand[t][warp][j];
          k[0] = key_at(pos[0]);
        }
        emit(k, pos, 1, T, take, wbase, want_t, tie_run, sel_run, outp);
      }
    }
  } else {
    uint32_t tie_run0 = 0, sel_run0 = 0, tie_run1 = 0, sel_run1 = 0;
    for (int i0 = seg_lo; i0 < seg_hi; i0 += 128) {
      const int i = i0 + 4 * lane;
      uint32_t k[4];
      load4(i, k);
      const int pos[4] = {i, i + 1, i + 2, i + 3};
      if (want0 > 0) emit(k, pos, 4, pre0, wtake0, wbase0, want0, tie_run0, sel_run0, out0);
      if (want1 > 0) emit(k, pos, 4, pre1, wtake1, wbase1, want1, tie_run1, sel_run1, out1);
    }
  }
  // -1 padding after the selected entries
  if (rank == 0) {
    for (int i = (int)want0 + tid; i < topk; i += kSelThreads) out0[i] = -1;
    if (two)
      for (int i = (int)want1 + tid; i < pool_size; i += kSelThreads) out1[i] = -1;
  }
  cluster.sync();  // no CTA leaves while others may still read its shared memory
}

// ------------------------------------------------------------ single-CTA selection --
// FULL selection with one 1024-thread CTA per query (no cluster synchronisation):
//   1. exact histogram of the top 11 key bits (8 exponent + 3 mantissa bits) over the
//      query's keys, straight from L2;
//   2. per target t (top-K, pool), the boundary bin B_t in which the count from the
//      top first reaches want_t; every key of the answer has bin >= B_t;
//   3. one ordered sweep keeps (position, key) of the keys with bin >= min B_t in
//      per-warp lists (the warps own consecutive position segments);
//   4. three radix passes over the kept keys of bin B_t fix the exact boundary key T_t;
//   5. ordered emit: keys > T_t, then ties of T_t by lowest position up to the quota.
// If a warp's list overflows (many keys in the boundary bins), the CTA falls back to
// radix passes over the whole range; the result is the same.  The two sweeps over L2
// keep eight 16-byte loads per lane in flight.
constexpr int kBigThreads = 1024;
constexpr int kBigWarps = kBigThreads / 32;
constexpr int kBigCap = 512;    // kept keys per warp
constexpr int kBigBatch = 8;    // 16-byte loads in flight per lane in the histogram sweep
constexpr int kFiltBatch = 8;   // 128-key groups in flight per warp in the wide filter's sweep
constexpr int kCtaFiltBatch = 4;  // the same in the single-CTA selection's sweep

// Ordered filter of one warp's position segment [seg_lo, seg_hi) (seg_lo a multiple of
// 128): every valid key whose histogram bin is >= bmin is passed to keep(p, position, key)
// with p its rank among the kept keys, so the kept keys come out in position order.  Lane
// l reads keys 4 l .. 4 l + 3 of each 128-key group with one 16-byte load (kFiltBatch
// groups in flight); ranks come from a warp scan of the per-lane counts.  Returns the
// number kept.
template <typename Keep>
__device__ __forceinline__ uint32_t filter_segment(const uint32_t* __restrict__ src, int seg_lo,
                                                   int seg_hi, uint32_t bmin, Keep keep) {
  const int lane = threadIdx.x & 31;
  uint32_t cnt = 0;
  for (int i0 = seg_lo; i0 < seg_hi; i0 += 128 * kFiltBatch) {
    uint4 k[kFiltBatch];
#pragma unroll
    for (int bb = 0; bb < kFiltBatch; ++bb) {
      const int i = i0 + 128 * bb + 4 * lane;
      if (i + 4 <= seg_hi) {
        k[bb] = __ldcg(reinterpret_cast<const uint4*>(src + i));
      } else {
        k[bb].x = i < seg_hi ? __ldcg(src + i) : 0u;
        k[bb].y = i + 1 < seg_hi ? __ldcg(src + i + 1) : 0u;
        k[bb].z = i + 2 < seg_hi ? __ldcg(src + i + 2) : 0u;
        k[bb].w = 0u;
      }
    }
#pragma unroll
    for (int bb = 0; bb < kFiltBatch; ++bb) {
      const int i = i0 + 128 * bb + 4 * lane;
      const uint32_t kk[4] = {k[bb].x, k[bb].y, k[bb].z, k[bb].w};
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kk[e] != 0 && (kk[e] >> 20) >= bmin) m |= 1u << e;
      const uint32_t c = __popc(m);
      uint32_t x = c;  // inclusive scan of the per-lane counts
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      uint32_t p = cnt + x - c;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m & (1u << e)) keep(p++, (uint32_t)(i + e), kk[e]);
      cnt += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  return cnt;
}

// Shared layout of the single-CTA selection with NT threads and a kept list of CAP keys
// per warp (positions stored as 16-bit offsets into the warp's segment, which is at most
// 2^18 / (NT / 32) <= 16384 positions).  BigShared (1024 threads) also serves the wide
// path's filter and resolve kernels.
template <int NT, int CAP>
struct BigSharedT {
  static constexpr int NW = NT / 32;
  uint32_t hist[kHistBins];
  uint32_t wsel[2][NW];  // per-warp keys > T_t
  uint32_t wtie[2][NW];  // per-warp keys == T_t
  uint32_t wcnt[NW];     // per-warp kept keys
  uint32_t rh[2][256];
  uint32_t scan[2][32];
  uint32_t res[2][2];    // per target: (bin, keys above it)
  uint32_t nvalid;
  uint32_t overflow;
  union {
    struct {
      uint32_t key[NW][CAP];
      uint16_t pos[NW][CAP];
    } c;
    uint32_t raw[1];
  } u;
};
using BigShared = BigSharedT<kBigThreads, kBigCap>;
constexpr int kSmallThreads = 512;  // the selection's 2-CTAs-per-SM form (many queries)
constexpr int kSmallCap = 1024;
using SmallShared = BigSharedT<kSmallThreads, kSmallCap>;
static_assert(sizeof(SmallShared) <= 113 * 1024 && sizeof(BigShared) <= 113 * 1024,
              "two selection CTAs per SM");

// Block-wide: thread tid holds v = count of bin (tid % nb) for target tid / nb (two
// targets, nb bins each, 2 nb <= 1024 threads).  For each target with want_t > 0, find
// the bin where (abv_t + keys in strictly higher bins) < want_t <= ... + v, and return
// it in res[t][0] (res[t][1] = keys above it, abv_t included).
template <class SH>
__device__ __forceinline__ void big_find(SH& sh, uint32_t v, int nb, uint32_t want0,
                                         uint32_t want1, uint32_t abv0, uint32_t abv1) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int t = tid / nb, bin = tid % nb, tw = bin >> 5;
  uint32_t x = (t < 2) ? v : 0u;  // inclusive suffix sum within the warp (bins descending)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (t < 2 && lane == 0) sh.scan[t][tw] = x;
  __syncthreads();
  if (t < 2) {
    const uint32_t want_t = t == 0 ? want0 : want1;
    if (want_t > 0) {
      uint32_t later = 0;
      for (int w = tw + 1; w < nb / 32; ++w) later += sh.scan[t][w];
      const uint32_t above_bin = (t == 0 ? abv0 : abv1) + later + x - v;
      if (above_bin < want_t && above_bin + v >= want_t) {
        sh.res[t][0] = (uint32_t)bin;
        sh.res[t][1] = above_bin;
      }
    }
  }
  __syncthreads();
}

// kReindex: the query's keys are its P pool entries (n = pool_size), the output is the
// pool entry's token, and no pool is emitted.
template <bool kReindex, int NT, int CAP>
__global__ void __launch_bounds__(NT, 1024 / NT)
    select_cta_kernel(const uint32_t* __restrict__ ws, int64_t ws_stride,
                      const int32_t* __restrict__ q_seq, const int32_t* __restrict__ seq_lens,
                      int32_t num_seqs, const int32_t* __restrict__ pool_in, int32_t pool_size,
                      int32_t topk, int32_t* __restrict__ out_idx, int32_t* __restrict__ pool_out,
                      int32_t max_ctx, const uint32_t* __restrict__ ghist,
                      const int32_t* __restrict__ order, int32_t split_targets) {
  grid_dep_wait();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  using SH = BigSharedT<NT, CAP>;
  constexpr int NW = SH::NW;
  SH& sh = *reinterpret_cast<SH*>(smem_raw);
  const int q = order != nullptr ? __ldg(order + blockIdx.x) : (int)blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int n;
  if (kReindex) {
    n = pool_size;
  } else {
    const int b = __ldg(q_seq + q);
    n = (b >= 0 && b < num_seqs) ? min(max(0, __ldg(seq_lens + b)), max_ctx) : 0;
  }
  const bool two = !kReindex && pool_out != nullptr && pool_size > 0;
  // split_targets: two CTAs per query (grid.y = 2), the first emitting the top-K, the second
  // the pool; each runs the whole search for its own target only
  const bool h0 = !split_targets || blockIdx.y == 0;
  const bool h1 = two && (!split_targets || blockIdx.y == 1);
  const uint32_t* src = ws + (int64_t)q * ws_stride;
  const int32_t* pin = kReindex ? pool_in + (int64_t)q * pool_size : nullptr;
  int32_t* out0 = out_idx + (int64_t)q * topk;
  int32_t* out1 = two ? pool_out + (int64_t)q * pool_size : nullptr;

  // position segment of this warp: multiples of 128, in position order across warps
  int S = (n + NW - 1) / NW;
  S = (S + 127) & ~127;
  const int seg_lo = min(n, warp * S), seg_hi = min(n, seg_lo + S);
  auto load4 = [&](int i, uint32_t (&k)[4]) {
    if (i + 4 <= seg_hi) {
      const uint4 v = __ldcg(reinterpret_cast<const uint4*>(src + i));
      k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) k[e] = (i + e < seg_hi) ? __ldcg(src + i + e) : 0u;
    }
  };

  // ---- 1. histogram of the top 11 bits, valid-key count (or the scorer's histogram) ----
  if (tid == 0) {
    sh.nvalid = 0;
    sh.overflow = 0;
  }
  uint32_t nv = 0;
  if (ghist != nullptr) {
    for (int i = tid; i < kHistBins; i += NT) {
      const uint32_t v = __ldcg(ghist + (int64_t)q * kHistBins + i);
      sh.hist[i] = v;
      nv += v;
    }
  } else {
    for (int i = tid; i < kHistBins; i += NT) sh.hist[i] = 0;
  }
  __syncthreads();
  for (int i0 = seg_lo; ghist == nullptr && i0 < seg_hi; i0 += 128 * kBigBatch) {
    uint32_t k[kBigBatch][4];
#pragma unroll
    for (int bb = 0; bb < kBigBatch; ++bb) load4(i0 + 128 * bb + 4 * lane, k[bb]);
#pragma unroll
    for (int bb = 0; bb < kBigBatch; ++bb)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (k[bb][e] != 0) {
          ++nv;
          atomicAdd(&sh.hist[hist_bin(k[bb][e])], 1u);
        }
  }
  nv = __reduce_add_sync(0xffffffffu, nv);
  if (lane == 0) atomicAdd(&sh.nvalid, nv);
  __syncthreads();
  const uint32_t nvalid = sh.nvalid;
  const uint32_t want0 = h0 ? min((uint32_t)topk, nvalid) : 0u;
  const uint32_t want1 = h1 ? min((uint32_t)pool_size, nvalid) : 0u;

  // ---- 2. boundary bins (thread tid holds bins BPT tid .. BPT tid + BPT - 1) ----
  constexpr int BPT = kHistBins / NT;
  uint32_t B0 = 0, B1 = 0, A0 = 0, A1 = 0;  // boundary bins and keys in higher bins
  {
    uint32_t c[BPT], tot = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      c[j] = sh.hist[BPT * tid + j];
      tot += c[j];
    }
    uint32_t x = tot;  // inclusive suffix sum of the threads' counts within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x += y;
    }
    if (lane == 0) sh.scan[0][warp] = x;
    if (tid < 4) sh.res[tid >> 1][tid & 1] = 0;
    __syncthreads();
    uint32_t later = 0;
    for (int w = warp + 1; w < NW; ++w) later += sh.scan[0][w];
    uint32_t above = later + x - tot;  // keys in bins above this thread's
#pragma unroll
    for (int j = BPT - 1; j >= 0; --j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t want_t = t == 0 ? want0 : want1;
        if (want_t > 0 && above < want_t && above + c[j] >= want_t) {
          sh.res[t][0] = BPT * tid + j;
          sh.res[t][1] = above;
        }
      }
      above += c[j];
    }
    __syncthreads();
    B0 = sh.res[0][0];
    A0 = sh.res[0][1];
    B1 = sh.res[1][0];
    A1 = sh.res[1][1];
    __syncthreads();
  }
  uint32_t bmin = want0 > 0 ? B0 : 0xFFFFFFFFu;
  if (want1 > 0) bmin = min(bmin, B1);

  // ---- 3. ordered sweep: keep keys with bin >= bmin ----
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t cnt = 0;
  if (want0 > 0 || want1 > 0) {
    // slot-major groups (lane l holds keys l, 32 + l, 64 + l, 96 + l): each slot compacts
    // with one ballot.  (The 16-byte-load form of filter_segment measured slower here, where
    // the sweep is bound by instruction issue, not by the loads.)
    for (int i0 = seg_lo; i0 < seg_hi; i0 += 128 * kCtaFiltBatch) {
      uint32_t k[kCtaFiltBatch][4];
#pragma unroll
      for (int bb = 0; bb < kCtaFiltBatch; ++bb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = i0 + 128 * bb + 32 * e + lane;
          k[bb][e] = i < seg_hi ? __ldcg(src + i) : 0u;
        }
#pragma unroll
      for (int bb = 0; bb < kCtaFiltBatch; ++bb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool m = k[bb][e] != 0 && (k[bb][e] >> 20) >= bmin;
          const uint32_t bal = __ballot_sync(0xffffffffu, m);
          const uint32_t p = cnt + __popc(bal & lt);
          if (m && p < (uint32_t)CAP) {
            sh.u.c.pos[warp][p] = (uint16_t)(i0 + 128 * bb + 32 * e + lane - seg_lo);
            sh.u.c.key[warp][p] = k[bb][e];
          }
          cnt += __popc(bal);
        }
    }
    if (lane == 0) {
      sh.wcnt[warp] = cnt;
      if (cnt > (uint32_t)CAP) atomicOr(&sh.overflow, 1u);
    }
  }
  __syncthreads();
  const bool kept = sh.overflow == 0;

  // ---- 4. exact boundary keys T_t ----
  uint32_t T0 = 0, T1 = 0, Q0 = 0, Q1 = 0;  // boundary key and ties to take
  if (want0 > 0 || want1 > 0) {
    uint32_t pre[2] = {B0, B1}, abv[2] = {A0, A1};
    // a target that takes every valid key needs no search (T = 1, the smallest valid key,
    // with every tie taken)
    const uint32_t want[2] = {want0 < nvalid ? want0 : 0u, want1 < nvalid ? want1 : 0u};
    // kept: digits of bits 19..12, 11..4, 3..0 within the boundary bin;
    // full range: digits of bits 30..23, 22..15, 14..7, 6..0
    const int passes = (want[0] == 0 && want[1] == 0) ? 0 : kept ? 3 : 4;
    for (int pass = 0; pass < passes; ++pass) {
      const int shift = kept ? (pass == 0 ? 12 : pass == 1 ? 4 : 0) : (pass == 0 ? 23 : pass == 1 ? 15 : pass == 2 ? 7 : 0);
      const int width = kept ? (pass == 2 ? 4 : 8) : (pass == 3 ? 7 : 8);
      const uint32_t dmask = (1u << width) - 1u;
      if (!kept && pass == 0) {
        pre[0] = pre[1] = 0;
        abv[0] = abv[1] = 0;
      }
      for (int i = tid; i < 2 * 256; i += NT) sh.rh[i >> 8][i & 255] = 0;
      __syncthreads();
      if (kept) {
#pragma unroll 4
        for (uint32_t j = lane; j < cnt; j += 32) {
          const uint32_t k = sh.u.c.key[warp][j];
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (want[t] > 0 && (k >> (shift + width)) == pre[t])
              atomicAdd(&sh.rh[t][(k >> shift) & dmask], 1u);
        }
      } else {
        for (int i = seg_lo + 4 * lane; i < seg_hi; i += 128) {
          uint32_t k[4];
          load4(i, k);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (k[e] == 0) continue;
#pragma unroll
            for (int t = 0; t < 2; ++t)
              if (want[t] > 0 && (pass == 0 || (k[e] >> (shift + width)) == pre[t]))
                atomicAdd(&sh.rh[t][(k[e] >> shift) & dmask], 1u);
          }
        }
      }
      __syncthreads();
      const uint32_t v = tid < 512 ? sh.rh[tid >> 8][tid & 255] : 0u;
      big_find(sh, v, 256, want[0], want[1], abv[0], abv[1]);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (want[t] > 0) {
          pre[t] = (pre[t] << width) | sh.res[t][0];
          abv[t] = sh.res[t][1];
        }
      __syncthreads();
    }
    T0 = want[0] > 0 ? pre[0] : 1u;
    Q0 = want[0] > 0 ? want0 - abv[0] : want0;
    T1 = want[1] > 0 ? pre[1] : 1u;
    Q1 = want[1] > 0 ? want1 - abv[1] : want1;
  }

  // ---- 5. ordered emit ----
  if (kept) {
    // both targets in one traversal of the kept lists: per-warp counts of keys > T_t and
    // == T_t, the warp's output base and tie quota, then ballot ranks per 32-key chunk
    const uint32_t Tt[2] = {T0, T1}, Qt[2] = {Q0, Q1}, wt[2] = {want0, want1};
    int32_t* const ot[2] = {out0, out1};
    uint32_t gt[2] = {0u, 0u}, eq[2] = {0u, 0u};
#pragma unroll 4
    for (uint32_t j = lane; j < cnt; j += 32) {
      const uint32_t k = sh.u.c.key[warp][j];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        gt[t] += k > Tt[t];
        eq[t] += k == Tt[t];
      }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      gt[t] = __reduce_add_sync(0xffffffffu, gt[t]);
      eq[t] = __reduce_add_sync(0xffffffffu, eq[t]);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        sh.wsel[t][warp] = gt[t];
        sh.wtie[t][warp] = eq[t];
      }
    }
    __syncthreads();
    // the warp's output base and tie quota per target: lane w takes warp w's counts; the
    // ties before each warp are an exclusive scan over the warps, a warp's contribution is
    // its keys > T plus the ties it takes, and the base sums the contributions before it
    uint32_t base[2], take[2], tie_run[2] = {0u, 0u}, sel_run[2] = {0u, 0u};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t e_l = lane < NW ? sh.wtie[t][lane] : 0u;
      const uint32_t s_l = lane < NW ? sh.wsel[t][lane] : 0u;
      uint32_t e_tot;
      const uint32_t e_before = warp_excl(e_l, e_tot);
      const uint32_t take_l = Qt[t] > e_before ? min(Qt[t] - e_before, e_l) : 0u;
      uint32_t c_tot;
      const uint32_t c_before = warp_excl(s_l + take_l, c_tot);
      base[t] = __shfl_sync(0xffffffffu, c_before, warp);
      take[t] = __shfl_sync(0xffffffffu, take_l, warp);
    }
    // four 32-key chunks per step: their keys and positions are read before any output
    // store (a store through a generic pointer would order the later shared reads)
    for (uint32_t j0 = 0; j0 < cnt; j0 += 128) {
      uint32_t kc[4], pc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t j = j0 + 32 * u + lane;
        kc[u] = j < cnt ? sh.u.c.key[warp][j] : 0u;
        pc[u] = j < cnt ? (uint32_t)seg_lo + sh.u.c.pos[warp][j] : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t j = j0 + 32 * u + lane;
        const uint32_t k = kc[u], pos = pc[u];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (wt[t] == 0) continue;
          const bool tie = j < cnt && k == Tt[t];
          const uint32_t tb = __ballot_sync(0xffffffffu, tie);
          const bool sel = j < cnt && (k > Tt[t] || (tie && tie_run[t] + __popc(tb & lt) < take[t]));
          const uint32_t sb = __ballot_sync(0xffffffffu, sel);
          const uint32_t p = base[t] + sel_run[t] + __popc(sb & lt);
          if (sel && p < wt[t]) ot[t][p] = kReindex ? __ldg(pin + pos) : (int32_t)pos;
          tie_run[t] += __popc(tb);
          sel_run[t] += __popc(sb);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  // the full-range path (a warp's kept list overflowed): each target in turn, keys read
  // from the workspace again
#pragma unroll
  for (int t = 0; t < 2 && !kept; ++t) {
    const uint32_t want_t = t == 0 ? want0 : want1;
    if (want_t == 0) continue;
    const uint32_t T = t == 0 ? T0 : T1, quota = t == 0 ? Q0 : Q1;
    int32_t* outp = t == 0 ? out0 : out1;
    // per-warp counts of keys > T and == T
    uint32_t gt = 0, eq = 0;
    for (int i = seg_lo + 4 * lane; i < seg_hi; i += 128) {
      uint32_t k[4];
      load4(i, k);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gt += k[e] > T;
        eq += k[e] == T;
      }
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0) {
      sh.wsel[t][warp] = gt;
      sh.wtie[t][warp] = eq;
    }
    __syncthreads();
    uint32_t base = 0, ties_before = 0;
    for (int w = 0; w < warp; ++w) {
      const uint32_t e_w = sh.wtie[t][w];
      base += sh.wsel[t][w] + (quota > ties_before ? min(quota - ties_before, e_w) : 0u);
      ties_before += e_w;
    }
    const uint32_t take = quota > ties_before ? min(quota - ties_before, sh.wtie[t][warp]) : 0u;
    uint32_t tie_run = 0, sel_run = 0;
    for (int i0 = seg_lo; i0 < seg_hi; i0 += 128) {
      const int i = i0 + 4 * lane;
      uint32_t k[4];
      load4(i, k);
      uint32_t nt = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) nt += k[e] == T;
      uint32_t ttot;
      uint32_t tr = tie_run + warp_excl(nt, ttot);
      uint32_t selm = 0, ns = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool tie = k[e] == T;
        if (k[e] > T || (tie && tr < take)) {
          selm |= 1u << e;
          ++ns;
        }
        tr += tie;
      }
      uint32_t stot;
      uint32_t p = base + sel_run + warp_excl(ns, stot);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (selm & (1u << e)) {
          if (p < want_t) outp[p] = kReindex ? __ldg(pin + i + e) : (int32_t)(i + e);
          ++p;
        }
      tie_run += ttot;
      sel_run += stot;
    }
    __syncthreads();
  }
  // -1 padding after the selected entries
  if (h0)
    for (int i = (int)want0 + tid; i < topk; i += NT) out0[i] = -1;
  if (h1)
    for (int i = (int)want1 + tid; i < pool_size; i += NT) out1[i] = -1;
}

// ------------------------------------------------------------ wide selection (Full) --
// Contexts beyond kWideThreshold tokens: the Full scorer's exact histograms give every
// CTA the boundary bins, so a query's keys are filtered by several CTAs at once.
//   select_filter_kernel (C CTAs per query): one ordered sweep of the CTA's position
//     range keeps (position, key) of the keys with bin >= min B_t into per-warp global
//     lists sized for the whole warp segment (no overflow is possible);
//   select_resolve_kernel (one CTA per query): three radix passes over the boundary-bin
//     keys of all lists fix T_t; per-list output bases and tie quotas follow in list
//     order, which is position order (CTA-major, then warp-major);
//   select_emit_kernel (the filter's grid, one warp per list): each list writes its
//     selected positions at its base.
constexpr int kWideThreshold = 1 << 18;  // Full contexts longer than this use the wide path
constexpr int kWideMinKeys = 1 << 15;  // positions per filter CTA at least
constexpr int kWideMaxCtas = 32;       // filter CTAs per query at most (the sweep is issue-bound)
constexpr int kMaxWideLists = kWideMaxCtas * kBigWarps;

// Per-CTA position range of the wide filter: a multiple of 4096 (so each warp segment is
// a multiple of 128) with at most kWideMaxCtas CTAs per query.
inline int wide_range(int32_t n) {
  const int64_t per = std::max<int64_t>(kWideMinKeys, ((int64_t)n + kWideMaxCtas - 1) / kWideMaxCtas);
  return (int)((per + 4095) / 4096 * 4096);
}

// Boundary bins (B_t) and keys in higher bins (A_t) of both targets from a histogram in
// shared memory; every thread gets the same values.  Thread t handles bins 2t, 2t + 1.
__device__ __forceinline__ void boundary_bins(BigShared& sh, uint32_t want0, uint32_t want1,
                                              uint32_t& B0, uint32_t& A0, uint32_t& B1,
                                              uint32_t& A1) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t hi = sh.hist[2 * tid + 1], lo = sh.hist[2 * tid];
  uint32_t x = hi + lo;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) sh.scan[0][warp] = x;
  if (tid < 4) sh.res[tid >> 1][tid & 1] = 0;
  __syncthreads();
  uint32_t later = 0;
  for (int w = warp + 1; w < kBigWarps; ++w) later += sh.scan[0][w];
  const uint32_t above_hi = later + x - (hi + lo), above_lo = above_hi + hi;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const uint32_t want_t = t == 0 ? want0 : want1;
    if (want_t == 0) continue;
    if (above_hi < want_t && above_hi + hi >= want_t) {
      sh.res[t][0] = 2 * tid + 1;
      sh.res[t][1] = above_hi;
    } else if (above_lo < want_t && above_lo + lo >= want_t) {
      sh.res[t][0] = 2 * tid;
      sh.res[t][1] = above_lo;
    }
  }
  __syncthreads();
  B0 = sh.res[0][0];
  A0 = sh.res[0][1];
  B1 = sh.res[1][0];
  A1 = sh.res[1][1];
  __syncthreads();
}

// Histogram of query q from the scorer into shared memory; returns the valid-key count.
__device__ __forceinline__ uint32_t load_hist(BigShared& sh, const uint32_t* __restrict__ ghist,
                                              int q) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) sh.nvalid = 0;
  uint32_t nv = 0;
  for (int i = tid; i < kHistBins; i += kBigThreads) {
    const uint32_t v = __ldcg(ghist + (int64_t)q * kHistBins + i);
    sh.hist[i] = v;
    nv += v;
  }
  __syncthreads();
  nv = __reduce_add_sync(0xffffffffu, nv);
  if (lane == 0) atomicAdd(&sh.nvalid, nv);
  __syncthreads();
  return sh.nvalid;
}

struct WideLists {
  uint32_t* pos;   // [num_q][C][32][seg]
  uint32_t* key;   // [num_q][C][32][seg]
  uint32_t* cnt;   // [num_q][C][32]
  uint32_t* meta;  // [num_q][kWideMeta]: per target T, want, then per-list base and take
  int C, seg;
};
// meta layout per query: [0..1] T_t, [2..3] want_t, then base[2][kMaxWideLists],
// take[2][kMaxWideLists]
constexpr int kWideMeta = 4 + 4 * kMaxWideLists;

__global__ void __launch_bounds__(kBigThreads, 1)
    select_filter_kernel(const uint32_t* __restrict__ ws, int64_t ws_stride,
                         const int32_t* __restrict__ q_seq, const int32_t* __restrict__ seq_lens,
                         int32_t num_seqs, int32_t pool_size, int32_t topk, int32_t max_ctx,
                         const uint32_t* __restrict__ ghist, WideLists wl) {
  grid_dep_wait();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BigShared& sh = *reinterpret_cast<BigShared*>(smem_raw);
  const int c = blockIdx.x, q = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = __ldg(q_seq + q);
  const int n = (b >= 0 && b < num_seqs) ? min(max(0, __ldg(seq_lens + b)), max_ctx) : 0;
  const uint32_t nvalid = load_hist(sh, ghist, q);
  const uint32_t want0 = min((uint32_t)topk, nvalid);
  const uint32_t want1 = pool_size > 0 ? min((uint32_t)pool_size, nvalid) : 0u;
  uint32_t B0, A0, B1, A1;
  boundary_bins(sh, want0, want1, B0, A0, B1, A1);
  uint32_t bmin = want0 > 0 ? B0 : 0xFFFFFFFFu;
  if (want1 > 0) bmin = min(bmin, B1);
  const int L = wl.seg * kBigWarps;
  const int lo = min(n, c * L), hi = min(n, lo + L);
  const int seg_lo = min(hi, lo + warp * wl.seg), seg_hi = min(hi, seg_lo + wl.seg);
  const uint32_t* src = ws + (int64_t)q * ws_stride;
  const int64_t list = ((int64_t)q * wl.C + c) * kBigWarps + warp;
  uint32_t* lpos = wl.pos + list * wl.seg;
  uint32_t* lkey = wl.key + list * wl.seg;
  uint32_t cnt = 0;
  if (want0 > 0)  // at most seg keys in the warp's segment, so p < seg
    cnt = filter_segment(src, seg_lo, seg_hi, bmin, [&](uint32_t p, uint32_t pos, uint32_t key) {
      lpos[p] = pos;
      lkey[p] = key;
    });
  if (lane == 0) wl.cnt[list] = cnt;
}

// Block-wide exclusive scan of one value per thread (1024 threads); returns the
// exclusive prefix and sets total.  Uses sh.scan[0].
__device__ __forceinline__ uint32_t block_excl(BigShared& sh, uint32_t v, uint32_t& total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.scan[0][warp] = x;
  __syncthreads();
  uint32_t before = 0, all = 0;
  for (int w = 0; w < kBigWarps; ++w) {
    const uint32_t s = sh.scan[0][w];
    before += w < warp ? s : 0u;
    all += s;
  }
  __syncthreads();
  total = all;
  return before + x - v;
}

// Resolve (one CTA per query): the candidate lists of the query, concatenated in
// position order (list-major), are staged in shared memory when they fit (a warp per run
// of lists; the kernel takes all the shared memory a CTA may have, about 53k keys), else
// walked from L2 in contiguous per-thread chunks, for three radix passes over the
// boundary-bin keys; the exact boundary keys, the per-list output bases and tie quotas
// (two block-wide scans over the lists) go to the query's meta.
constexpr int kResolveSmem = 232448;  // 227 KB, the per-CTA maximum on sm_103a
constexpr size_t kResolveKeyOff = offsetof(BigShared, u) + (kMaxWideLists + 32) * sizeof(uint32_t);
static_assert(kResolveKeyOff % 4 == 0 && kResolveKeyOff < (size_t)kResolveSmem, "resolve key staging");
static_assert(kMaxWideLists <= kBigThreads, "one thread per list in the base scans");
__global__ void __launch_bounds__(kBigThreads, 1)
    select_resolve_kernel(int32_t pool_size, int32_t topk, const uint32_t* __restrict__ ghist,
                          WideLists wl) {
  grid_dep_wait();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BigShared& sh = *reinterpret_cast<BigShared*>(smem_raw);
  uint32_t* loff = sh.u.raw;                      // [nlists + 1] list offsets
  uint32_t* skey = loff + kMaxWideLists + 32;     // staged keys
  const int q = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nlists = wl.C * kBigWarps;
  const bool two = pool_size > 0;
  const uint32_t nvalid = load_hist(sh, ghist, q);
  const uint32_t want0 = min((uint32_t)topk, nvalid);
  const uint32_t want1 = two ? min((uint32_t)pool_size, nvalid) : 0u;
  uint32_t B0, A0, B1, A1;
  boundary_bins(sh, want0, want1, B0, A0, B1, A1);
  const int64_t list0 = (int64_t)q * nlists;
  uint32_t* meta = wl.meta + (int64_t)q * kWideMeta;

  uint32_t total;
  const uint32_t mine = tid < nlists ? __ldcg(wl.cnt + list0 + tid) : 0u;
  const uint32_t off = block_excl(sh, mine, total);
  if (tid < nlists) loff[tid] = off;
  if (tid == 0) loff[nlists] = total;
  __syncthreads();
  const uint32_t skey_cap = (uint32_t)((kResolveSmem - kResolveKeyOff) / sizeof(uint32_t));
  const bool in_smem = total <= skey_cap;
  if (in_smem) {
    // warp w copies the keys of a contiguous run of lists (contiguous in skey too), lane-
    // strided with 8 loads in flight per lane; each lane follows its list boundary forward
    const int lpw = (nlists + kBigWarps - 1) / kBigWarps;
    const int la = min(nlists, warp * lpw), lb = min(nlists, la + lpw);
    const uint32_t ea = loff[la], eb = loff[lb];
    int l = la;
    for (uint32_t e0 = ea; e0 < eb; e0 += 8 * 32) {
      uint32_t v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t e = e0 + 32 * u + lane;
        if (e < eb) {
          while (loff[l + 1] <= e) ++l;
          v[u] = __ldcg(wl.key + (list0 + l) * wl.seg + (e - loff[l]));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t e = e0 + 32 * u + lane;
        if (e < eb) skey[e] = v[u];
      }
    }
    __syncthreads();
  }
  // every candidate key once (order is irrelevant to the radix histograms): strided over
  // the staged keys, else each thread walks a contiguous chunk of the lists in L2
  const uint32_t per = (total + kBigThreads - 1) / kBigThreads;
  const uint32_t e_lo = min(total, per * tid), e_hi = min(total, e_lo + per);
  int l_first = 0;
  if (!in_smem) {  // the last list with loff[l] <= e_lo
    int hi = nlists - 1;
    while (l_first < hi) {
      const int m = (l_first + hi + 1) >> 1;
      if (loff[m] <= e_lo) l_first = m; else hi = m - 1;
    }
  }
  auto walk = [&](auto f) {
    if (in_smem) {
      for (uint32_t e = tid; e < total; e += kBigThreads) f(skey[e]);
      return;
    }
    int l = l_first;
    for (uint32_t e0 = e_lo; e0 < e_hi; e0 += 8) {  // 8 keys fetched before any is used
      uint32_t v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t e = e0 + u;
        if (e < e_hi) {
          while (loff[l + 1] <= e) ++l;
          v[u] = __ldcg(wl.key + (list0 + l) * wl.seg + (e - loff[l]));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u < e_hi) f(v[u]);
    }
  };

  uint32_t pre[2] = {B0, B1}, abv[2] = {A0, A1};
  const uint32_t want[2] = {want0, want1};
  if (want0 > 0) {
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 12 : pass == 1 ? 4 : 0, width = pass == 2 ? 4 : 8;
      const uint32_t dmask = (1u << width) - 1u;
      for (int i = tid; i < 2 * 256; i += kBigThreads) sh.rh[i >> 8][i & 255] = 0;
      __syncthreads();
      walk([&](uint32_t k) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (want[t] > 0 && (k >> (shift + width)) == pre[t])
            atomicAdd(&sh.rh[t][(k >> shift) & dmask], 1u);
      });
      __syncthreads();
      const uint32_t v = tid < 512 ? sh.rh[tid >> 8][tid & 255] : 0u;
      big_find(sh, v, 256, want[0], want[1], abv[0], abv[1]);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (want[t] > 0) {
          pre[t] = (pre[t] << width) | sh.res[t][0];
          abv[t] = sh.res[t][1];
        }
      __syncthreads();
    }
  }
  if (tid < 2) {
    meta[tid] = pre[tid];
    meta[2 + tid] = want[tid];
  }
  // per-list counts of the keys above and equal to each boundary key (one thread per
  // list, both targets in one pass), then bases and tie quotas in list (= position) order
  uint32_t cgt[2] = {0u, 0u}, ceq[2] = {0u, 0u};
  if (tid < nlists) {
    const uint32_t a = loff[tid], b = loff[tid + 1];
    const uint32_t* lk = wl.key + (list0 + tid) * wl.seg;
#pragma unroll 4
    for (uint32_t e = a; e < b; ++e) {
      const uint32_t k = in_smem ? skey[e] : __ldcg(lk + (e - a));
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        cgt[t] += k > pre[t];
        ceq[t] += k == pre[t];
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (want[t] == 0) continue;
    // list l takes min(its ties, the quota left after the ties of the lists before it),
    // and its base is the count of keys the lists before it take: two block-wide scans
    const uint32_t quota = want[t] - abv[t];
    uint32_t tot;
    const uint32_t ties_before = block_excl(sh, ceq[t], tot);
    const uint32_t take = quota > ties_before ? min(quota - ties_before, ceq[t]) : 0u;
    const uint32_t base = block_excl(sh, cgt[t] + take, tot);
    if (tid < nlists) {
      meta[4 + t * kMaxWideLists + tid] = base;
      meta[4 + (2 + t) * kMaxWideLists + tid] = take;
    }
  }
}

// Emit (the filter's grid, one warp per list): keys > T_t, then ties of T_t up to the
// list's quota, written at the list's base; CTA 0 of a query writes the -1 padding.
__global__ void __launch_bounds__(kBigThreads, 1)
    select_emit_kernel(int32_t pool_size, int32_t topk, int32_t* __restrict__ out_idx,
                       int32_t* __restrict__ pool_out, WideLists wl) {
  grid_dep_wait();
  const int c = blockIdx.x, q = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t list = ((int64_t)q * wl.C + c) * kBigWarps + warp;
  const int l = c * kBigWarps + warp;
  const uint32_t* meta = wl.meta + (int64_t)q * kWideMeta;
  const uint32_t cn = __ldcg(wl.cnt + list);
  const uint32_t* lk = wl.key + list * wl.seg;
  const uint32_t* lp = wl.pos + list * wl.seg;
  const uint32_t lt = (1u << lane) - 1u;
  const bool two = pool_out != nullptr && pool_size > 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const uint32_t want_t = __ldcg(meta + 2 + t);
    if (want_t == 0) continue;
    const uint32_t T = __ldcg(meta + t);
    const uint32_t base = __ldcg(meta + 4 + t * kMaxWideLists + l);
    const uint32_t take = __ldcg(meta + 4 + (2 + t) * kMaxWideLists + l);
    int32_t* outp = t == 0 ? out_idx + (int64_t)q * topk : pool_out + (int64_t)q * pool_size;
    uint32_t tie_run = 0, sel_run = 0;
    for (uint32_t j0 = 0; j0 < cn; j0 += 32) {
      const uint32_t j = j0 + lane;
      const uint32_t k = j < cn ? __ldcg(lk + j) : 0u;
      const bool tie = j < cn && k == T;
      const uint32_t tb = __ballot_sync(0xffffffffu, tie);
      const bool sel = j < cn && (k > T || (tie && tie_run + __popc(tb & lt) < take));
      const uint32_t sb = __ballot_sync(0xffffffffu, sel);
      const uint32_t p = base + sel_run + __popc(sb & lt);
      if (sel && p < want_t) outp[p] = (int32_t)__ldcg(lp + j);
      tie_run += __popc(tb);
      sel_run += __popc(sb);
    }
  }
  if (c == 0) {
    const uint32_t want0 = __ldcg(meta + 2), want1 = __ldcg(meta + 3);
    for (int i = (int)want0 + tid; i < topk; i += kBigThreads) out_idx[(int64_t)q * topk + i] = -1;
    if (two)
      for (int i = (int)want1 + tid; i < pool_size; i += kBigThreads)
        pool_out[(int64_t)q * pool_size + i] = -1;
  }
}

// ------------------------------------------------------------------ pool selection --
// REINDEX over a pool of at most kPoolSelMax entries: one 512-thread CTA per query holds
// the query's P keys in registers, read once with coalesced loads (key j of thread t is
// position 512 j + t).  Three radix steps find the exact boundary key T: the 11-bit
// histogram bin (key >> 20), then bits 19..9 and 8..0 of the keys in the boundary bin.
// The emit takes keys > T and the first Q keys == T in position order: per (j, warp)
// counts of both from two ballots, one scan by a single warp over those 16 KPT counts
// (which are in position order), then each warp writes its selected pool tokens of slot j
// to consecutive outputs.  The pool's tokens are copied to shared memory meanwhile.
constexpr int kPoolThreads = 512;                 // many queries: two CTAs per SM
constexpr int kPoolThreadsWide = 1024;            // queries fit one per SM
constexpr int kPoolSelMax = 32 * kPoolThreads;  // 16384 pool entries, at most 32 per thread

struct PoolShared {
  uint32_t h[2][kHistBins];      // two histograms used in turn (pass 0, 1, 2 on h0, h1, h0)
  uint32_t wsum[32];             // one word per warp
  uint32_t res[2];               // boundary digit, keys above it
};

// Suffix sums over the NW warps: returns the sum of wsum[w] for w > warp (wsum complete
// and visible; warp + 1 < NW, or warp = -1 for all of them).  Lane l reads warp l's total.
template <int NW>
__device__ __forceinline__ uint32_t pool_later_warps(const PoolShared& sh, int warp, int lane) {
  uint32_t x = lane < NW ? sh.wsum[lane] : 0u;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  return __shfl_sync(0xffffffffu, x, warp + 1);
}

// Boundary digit of `want` keys among the NB digits of h (descending), `above` keys lying
// above the histogram's range: returns the digit d with above + (keys in digits > d) <
// want <= ... + h[d], and sets `above` to above + (keys in digits > d).  Thread tid owns
// the BPT consecutive digits from BPT tid (none past NB).
template <int NT, int NB>
__device__ __forceinline__ uint32_t pool_find(PoolShared& sh, const uint32_t* h, uint32_t want,
                                              uint32_t& above) {
  constexpr int NW = NT / 32, BPT = NB >= NT ? NB / NT : 1;
  static_assert(NB % NT == 0 || NT % NB == 0, "digits per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t c[BPT], tot = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    c[j] = BPT * tid + j < NB ? h[BPT * tid + j] : 0u;
    tot += c[j];
  }
  uint32_t x = tot;  // inclusive suffix sum over the warp's threads
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) sh.wsum[warp] = x;
  __syncthreads();
  uint32_t a = above + x - tot + (warp + 1 < NW ? pool_later_warps<NW>(sh, warp, lane) : 0u);
#pragma unroll
  for (int j = BPT - 1; j >= 0; --j) {
    if (a < want && a + c[j] >= want) {
      sh.res[0] = BPT * tid + j;
      sh.res[1] = a;
    }
    a += c[j];
  }
  __syncthreads();
  above = sh.res[1];
  return sh.res[0];
}

template <int NT, int KPT>
__global__ void __launch_bounds__(NT, (NT == kPoolThreads && KPT <= 16) ? 2 : 1)
    select_pool_kernel(const uint32_t* __restrict__ ws, const int32_t* __restrict__ pool_in,
                       int32_t pool_size, int32_t topk, int32_t* __restrict__ out_idx) {
  grid_dep_wait();
  __shared__ PoolShared sh;
  constexpr int NW = NT / 32;
  __shared__ uint32_t cnt[KPT * NW];   // per (slot j, warp): keys > T | (keys == T) << 16
  extern __shared__ __align__(16) int32_t spool[];  // the query's pool tokens (P entries)
  const int q = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = pool_size;
  const uint32_t* src = ws + (int64_t)q * P;
  const int32_t* pin = pool_in + (int64_t)q * P;
  int32_t* out = out_idx + (int64_t)q * topk;

  uint32_t k[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int pos = NT * j + tid;
    k[j] = pos < P ? __ldcg(src + pos) : 0u;
  }
  const uint32_t spool_s = smem_addr(spool);
  if ((P & 3) == 0 && (reinterpret_cast<uintptr_t>(pool_in) & 15) == 0) {
    for (int i = 4 * tid; i < P; i += 4 * NT) cp_async16(spool_s + 4 * i, pin + i);
  } else {
    for (int i = tid; i < P; i += NT)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(spool_s + 4 * i), "l"(pin + i)
                   : "memory");
  }
  cp_async_commit();
  for (int i = tid; i < 2 * kHistBins; i += NT) (&sh.h[0][0])[i] = 0;
  __syncthreads();
  // a NaN score's key can reach 2^31, whose bin (key >> 20) would leave the histogram;
  // clamped, every key's bin is key >> 20 exactly
#pragma unroll
  for (int j = 0; j < KPT; ++j) k[j] = min(k[j], 0x7FFFFFFFu);

  // ---- pass 0: 11-bit bins, valid-key count ----
  uint32_t nv = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j)
    if (k[j] != 0) {
      ++nv;
      atomicAdd(&sh.h[0][k[j] >> 20], 1u);
    }
  nv = __reduce_add_sync(0xffffffffu, nv);
  if (lane == 0) sh.wsum[warp] = nv;
  __syncthreads();
  const uint32_t nvalid = pool_later_warps<NW>(sh, -1, lane);  // the warps after "-1": all of them
  const uint32_t want = min((uint32_t)topk, nvalid);
  __syncthreads();  // wsum is reused by the scans

  // ---- boundary key T and the ties Q to take (T = 0, Q = 0 takes every valid key) ----
  uint32_t T = 0, Q = 0;
  if (want > 0 && want < nvalid) {
    uint32_t above = 0;
    const uint32_t b0 = pool_find<NT, kHistBins>(sh, sh.h[0], want, above);
    for (int i = tid; i < 512; i += NT) sh.h[0][i] = 0;  // pass 2's histogram
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (k[j] != 0 && (k[j] >> 20) == b0) atomicAdd(&sh.h[1][(k[j] >> 9) & 0x7FFu], 1u);
    __syncthreads();
    const uint32_t d1 = pool_find<NT, kHistBins>(sh, sh.h[1], want, above);
    const uint32_t pre = (b0 << 11) | d1;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (k[j] != 0 && (k[j] >> 9) == pre) atomicAdd(&sh.h[0][k[j] & 0x1FFu], 1u);
    __syncthreads();
    const uint32_t d2 = pool_find<NT, 512>(sh, sh.h[0], want, above);
    T = (pre << 9) | d2;
    Q = want - above;
  }

  // ---- ordered emit ----
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t gm = __ballot_sync(0xffffffffu, k[j] > T);
    const uint32_t em = __ballot_sync(0xffffffffu, k[j] == T);
    if (lane == 0) cnt[j * NW + warp] = __popc(gm) | ((uint32_t)__popc(em) << 16);
  }
  cp_async_wait<0>();
  __syncthreads();  // counts complete; every thread's pool tokens have landed
  // exclusive scan of the KPT x 16 packed counts (each half at most P < 2^16), in place,
  // by warp 0: lane l takes the NC / 32 consecutive entries from NC l / 32
  constexpr int NC = KPT * NW, CPL = NC / 32;
  static_assert(NC % 32 == 0, "whole counts per lane");
  if (warp == 0) {
    uint32_t c[CPL], tot = 0;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      c[i] = cnt[CPL * lane + i];
      tot += c[i];
    }
    uint32_t x = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    uint32_t run = x - tot;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      cnt[CPL * lane + i] = run;
      run += c[i];
    }
  }
  __syncthreads();
  // four slots at a time: their shared-memory reads are issued before their global
  // stores (a store through a generic pointer would otherwise order every later read)
#pragma unroll
  for (int j0 = 0; j0 < KPT; j0 += 4) {
    uint32_t cb[4];
    int32_t tok[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int pos = NT * (j0 + u) + tid;
      cb[u] = cnt[(j0 + u) * NW + warp];
      tok[u] = pos < P ? spool[pos] : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t kk = k[j0 + u];
      const uint32_t gm = __ballot_sync(0xffffffffu, kk > T);
      const uint32_t em = __ballot_sync(0xffffffffu, kk == T);
      const uint32_t ties = (cb[u] >> 16) + __popc(em & lt);  // ties of T before this key
      const uint32_t p = (cb[u] & 0xFFFFu) + __popc(gm & lt) + min(Q, ties);
      const bool sel = kk > T || (kk == T && ties < Q);
      if (sel && p < want) out[p] = tok[u];
    }
  }
  for (int i = (int)want + tid; i < topk; i += NT) out[i] = -1;
}

// ------------------------------------------------------------------ launchers -----

size_t select_smem_bytes() { return kSelCacheOff + (size_t)kSelCacheKeys * 4; }

// Bytes of the run list that follows the scores in the workspace (meta, prefix, run
// starts, then the Full selection's CTA order).
size_t runlist_bytes(int32_t num_q) {
  return (size_t)2 * 8 + (size_t)(num_q + 1) * 8 + (size_t)(num_q + 1) * 4 + (size_t)num_q * 4;
}

int32_t* runlist_order(void* base, int32_t num_q) {
  return reinterpret_cast<int32_t*>(static_cast<char*>(base) + 2 * 8 + (size_t)(num_q + 1) * 8 +
                                    (size_t)(num_q + 1) * 4);
}

static RunList make_runlist(void* base, int32_t num_q) {
  int64_t* meta = reinterpret_cast<int64_t*>(base);
  int64_t* prefix = meta + 2;
  int32_t* run_q0 = reinterpret_cast<int32_t*>(prefix + num_q + 1);
  return RunList{meta, prefix, run_q0};
}

cudaError_t launch_score_full(const uint16_t* q_idx, const uint16_t* keys, const int32_t* q_seq,
                              int32_t num_q, int32_t max_q_per_seq, const csa2_pages& pg,
                              uint32_t* ws, int64_t ws_stride, void* runlist, uint32_t* ghist,
                              int32_t* st, cudaStream_t s, int num_sms) {
  ScoreGeom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  RunList rl = make_runlist(runlist, num_q);
  const bool batched = max_q_per_seq > 1;
  // the selection histograms (num_q x kHistBins words, a multiple of 4) are cleared by
  // extra CTAs of the run-list launch, 8 vectors per thread
  const int64_t zero_vecs = ghist != nullptr ? (int64_t)num_q * kHistBins / 4 : 0;
  const int zero_ctas = (int)std::min<int64_t>(64, (zero_vecs + 8 * 1024 - 1) / (8 * 1024));
  cudaError_t e = launch_pdl(group_prefix_kernel, dim3(2 + zero_ctas), dim3(1024), 0, s, batched,
                             false, q_seq, num_q, g, 0, kPage, const_cast<int64_t*>(rl.meta),
                             const_cast<int64_t*>(rl.prefix), const_cast<int32_t*>(rl.run_q0),
                             reinterpret_cast<uint4*>(ghist), zero_vecs,
                             runlist_order(runlist, num_q));
  if (e != cudaSuccess) return e;
  CUtensorMap keymap;
  if (!make_bf16_map(&keymap, keys, (int64_t)pg.num_pages * kPage, kDidx, 64, kPage))
    return cudaErrorInvalidValue;
  const int grid = std::max(1, kScoreCtasPerSm * num_sms);
  e = cudaFuncSetAttribute(score_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kTmaSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(score_pages_kernel, dim3(grid), dim3(kTmaThreads), kTmaSmem, s, keymap, q_idx,
                    q_seq, num_q, g, ws, ws_stride, rl, ghist, st);
}

cudaError_t launch_score_reindex(const uint16_t* q_idx, const uint16_t* keys, const int32_t* q_seq,
                                 int32_t num_q, const csa2_pages& pg, const int32_t* pool,
                                 int32_t pool_size, uint32_t* ws, int32_t* st, cudaStream_t s,
                                 int num_sms) {
  ScoreGeom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  cudaError_t e = cudaFuncSetAttribute(score_gather_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGatherSmem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, kGatherCtasPerSm * num_sms);
  return launch_pdl(score_gather_kernel, dim3(grid), dim3(kScoreThreads), kGatherSmem, s, q_idx,
                    keys, q_seq, num_q, g, pool, pool_size, ws, st);
}

// CTAs per query: enough kept-key capacity (4096 per CTA and target) for twice the
// larger output, and enough CTAs that each one's keys fit its shared-memory cache.
// Measured on the 64 x 131072 decode batch: 8 cached CTAs per query in two waves beat 4
// uncached ones in one wave (Full), and one CTA per query is fastest for the 8192-entry
// Reindex pools.
int select_cluster(int32_t n, int32_t want_max) {
  int c = 1;  // kept positions are 16-bit: at most 65535 keys per CTA on the fast path
  while (c < kSelMaxCluster && ((int64_t)c * kSelWarps * kCandCap < 2LL * want_max ||
                                (int64_t)c * kSelCacheKeys < n))
    c *= 2;
  return c;
}

template <bool R, int C>
cudaError_t launch_select_c(const uint32_t* ws, int64_t ws_stride, const int32_t* q_seq,
                            const csa2_pages& pg, int32_t num_q, const int32_t* pool_in,
                            int32_t pool_size, int32_t topk, int32_t* out_idx, int32_t* pool_out,
                            int32_t* st, cudaStream_t s) {
  const size_t smem = select_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(select_kernel<R, C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel<R, C>, dim3(C, num_q), dim3(kSelThreads), smem, s, ws,
                    ws_stride, q_seq, pg.seq_lens, pg.num_seqs, pool_in, pool_size, topk, out_idx,
                    pool_out, pg.max_pages_per_seq * kPage, st);
}

template <bool R>
cudaError_t launch_select_r(int c, const uint32_t* ws, int64_t ws_stride, const int32_t* q_seq,
                            const csa2_pages& pg, int32_t num_q, const int32_t* pool_in,
                            int32_t pool_size, int32_t topk, int32_t* out_idx, int32_t* pool_out,
                            int32_t* st, cudaStream_t s) {
  switch (c) {
    case 1: return launch_select_c<R, 1>(ws, ws_stride, q_seq, pg, num_q, pool_in, pool_size, topk, out_idx, pool_out, st, s);
    case 2: return launch_select_c<R, 2>(ws, ws_stride, q_seq, pg, num_q, pool_in, pool_size, topk, out_idx, pool_out, st, s);
    case 4: return launch_select_c<R, 4>(ws, ws_stride, q_seq, pg, num_q, pool_in, pool_size, topk, out_idx, pool_out, st, s);
    default: return launch_select_c<R, 8>(ws, ws_stride, q_seq, pg, num_q, pool_in, pool_size, topk, out_idx, pool_out, st, s);
  }
}

// Bytes of the wide selection's candidate lists for FULL over contexts of n > kWideThreshold.
size_t wide_select_bytes(int32_t num_q, int32_t n) {
  if (n <= kWideThreshold) return 0;
  const int L = wide_range(n);
  const int64_t C = ((int64_t)n + L - 1) / L;
  return (size_t)num_q * (C * ((size_t)L * 8 + kBigWarps * 4) + (size_t)kWideMeta * 4);
}

cudaError_t launch_select(bool reindex, const uint32_t* ws, int64_t ws_stride, const int32_t* q_seq,
                          const csa2_pages& pg, int32_t num_q, const int32_t* pool_in,
                          int32_t pool_size, int32_t topk, int32_t* out_idx, int32_t* pool_out,
                          const uint32_t* ghist, void* wide_ws, const int32_t* order,
                          int32_t* st, cudaStream_t s, int num_sms) {
  const int32_t n = reindex ? pool_size : pg.max_pages_per_seq * kPage;
  const int32_t want_max = std::max(topk, (!reindex && pool_out) ? pool_size : 0);
  // FULL beyond 2^18 tokens with the scorer's histograms: C filter CTAs per query, then
  // one finishing CTA per query (the cluster kernel took ~265 us for 4 x 2^20 keys)
  if (!reindex && n > kWideThreshold && ghist != nullptr && wide_ws != nullptr) {
    const int L = wide_range(n);
    const int C = (int)(((int64_t)n + L - 1) / L);
    WideLists wl;
    wl.C = C;
    wl.seg = L / kBigWarps;
    const size_t lists = (size_t)num_q * C * L;
    wl.pos = static_cast<uint32_t*>(wide_ws);
    wl.key = wl.pos + lists;
    wl.cnt = wl.key + lists;
    wl.meta = wl.cnt + (size_t)num_q * C * kBigWarps;
    const size_t fsmem = offsetof(BigShared, u), bsmem = kResolveSmem;
    cudaError_t e = cudaFuncSetAttribute(select_resolve_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsmem);
    if (e != cudaSuccess) return e;
    const int32_t P = pool_out ? pool_size : 0;
    e = launch_pdl(select_filter_kernel, dim3(C, num_q), dim3(kBigThreads), fsmem, s, ws, ws_stride,
                   q_seq, pg.seq_lens, pg.num_seqs, P, topk, n, ghist, wl);
    if (e != cudaSuccess) return e;
    e = launch_pdl(select_resolve_kernel, dim3(num_q), dim3(kBigThreads), bsmem, s, P, topk, ghist, wl);
    if (e != cudaSuccess) return e;
    return launch_pdl(select_emit_kernel, dim3(C, num_q), dim3(kBigThreads), 0, s, P, topk, out_idx,
                      pool_out, wl);
  }
  // Reindex pools of up to 16384 entries: one CTA per query with the keys in registers,
  // 1024 threads while the queries fit one per SM, else 512
  if (reindex && n <= kPoolSelMax && ws_stride == n) {
    const bool wide = num_q <= num_sms;
    const int nt = wide ? kPoolThreadsWide : kPoolThreads;
    const int kpt = n <= 4 * nt ? 4 : n <= 8 * nt ? 8 : n <= 16 * nt ? 16 : 32;
    void (*kern)(const uint32_t*, const int32_t*, int32_t, int32_t, int32_t*) =
        wide ? (kpt == 4 ? select_pool_kernel<kPoolThreadsWide, 4>
                : kpt == 8 ? select_pool_kernel<kPoolThreadsWide, 8> : select_pool_kernel<kPoolThreadsWide, 16>)
             : (kpt == 4 ? select_pool_kernel<kPoolThreads, 4> : kpt == 8 ? select_pool_kernel<kPoolThreads, 8>
                : kpt == 16 ? select_pool_kernel<kPoolThreads, 16> : select_pool_kernel<kPoolThreads, 32>);
    const size_t smem = (size_t)n * sizeof(int32_t);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(num_q), dim3(nt), smem, s, ws, pool_in, pool_size, topk, out_idx);
  }
  // Up to 2^18 keys per query: one CTA per query, no cluster synchronisation (measured on
  // B300: 64 Full queries x 131072 keys took ~90 us in two waves of 8-CTA clusters, 46 us
  // this way; 64 Reindex queries x 8192 pool entries 27 us with single-CTA clusters)
  if (n <= (1 << 18) && want_max <= 8192) {
    // one CTA per query: 1024 threads while the queries fit one per SM; beyond that the
    // 512-thread form runs two CTAs per SM (each warp keeps up to 1024 keys of a segment
    // twice as long).  Reindex pools of up to 16384 entries always take the 512-thread
    // form: its warps' segments then hold at most 1024 keys, so nothing can overflow, and
    // on 8192-entry pools it measured 17 % faster than 1024 threads even at one CTA per SM.
    const bool small = num_q > num_sms || (reindex && n <= kSmallThreads / 32 * kSmallCap);
    const size_t smem = small ? sizeof(SmallShared) : sizeof(BigShared);
    auto kern = small ? (reindex ? select_cta_kernel<true, kSmallThreads, kSmallCap>
                                 : select_cta_kernel<false, kSmallThreads, kSmallCap>)
                      : (reindex ? select_cta_kernel<true, kBigThreads, kBigCap>
                                 : select_cta_kernel<false, kBigThreads, kBigCap>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    // Full with a pool, while two CTAs per query fit one per SM: one CTA per target
    const int split = (!reindex && pool_out != nullptr && pool_size > 0 && !small &&
                       2 * num_q <= num_sms) ? 1 : 0;
    return launch_pdl(kern, dim3(num_q, 1 + split), dim3(small ? kSmallThreads : kBigThreads), smem, s,
                      ws, ws_stride, q_seq, pg.seq_lens, pg.num_seqs, pool_in,
                      reindex ? pool_size : (pool_out ? pool_size : 0), topk, out_idx,
                      reindex ? nullptr : pool_out, pg.max_pages_per_seq * kPage,
                      reindex ? nullptr : ghist, reindex ? nullptr : order, split);
  }
  const int c = select_cluster(n, want_max);
  if (reindex)
    return launch_select_r<true>(c, ws, ws_stride, q_seq, pg, num_q, pool_in, pool_size, topk,
                                 out_idx, nullptr, st, s);
  return launch_select_r<false>(c, ws, ws_stride, q_seq, pg, num_q, nullptr, pool_size, topk,
                                out_idx, pool_out, st, s);
}

}  // namespace csa2
