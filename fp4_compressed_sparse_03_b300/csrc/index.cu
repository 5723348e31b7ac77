// CSA2 indexer kernels (tech-report digest, jiwasawa.github.io, section "Compressed
// Sparse Attention 2 (CSA2)": Full / Reindex / Reuse modes and the Hierarchical
// Sparse Indexer; zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮").
//
// Scoring (score_s = sum_h ReLU(q_h . k_s), 4 heads x 128 dims, fp32 accumulation)
// writes one 32-bit ranking key per candidate into the workspace:
//     key = (bits(score) & 0x7fffffff) + 1   for a valid candidate (score >= 0),
//     key = 0                                for an invalid one (pool padding, bad page).
// Keys order like the scores, and every valid key is above every invalid one.
// Selection (cluster radix select) then takes the top-min(K, #valid) keys with the
// lower candidate position winning ties, and writes their tokens in ascending order.
//
// Kernels:
//   score_q1_kernel      one query per sequence (Full) or per pool (Reindex): a
//                        bandwidth-bound warp dot product on CUDA cores (packed FFMA2)
//   score_batched_kernel up to 4 draft queries per sequence (Full): 16 query-head rows
//                        x 8 keys x 16 dims per tensor-core MMA, keys read once
//   select_kernel        8-CTA cluster per query: 3 histogram passes (11/11/10 bits)
//                        merged through distributed shared memory, then an ordered
//                        compaction
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

// ------------------------------------------------------------------ scoring -------

constexpr int kScoreThreads = 256;   // 8 warps
constexpr int kUnitPages = 16;       // pages per Full work unit (1024 keys)
constexpr int kUnitPool = 1024;      // pool positions per Reindex work unit
constexpr int kDepth = 4;            // key groups in flight per warp

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

// Lane layout of a warp over 8 keys: quad = lane/4 picks the key, c = lane%4 the
// 64-byte quarter of its 256-byte row: bytes [64j + 16c, 64j + 16c + 16), j = 0..3,
// i.e. dims 32j + 8c .. 32j + 8c + 7.  Each lane therefore holds the same 32 dims of
// every key and keeps the matching 4 x 32 query values in registers.
struct QRegs {
  unsigned long long p[kHidx][4][4];  // [head][j][pair] = (q[32j+8c+2e], q[32j+8c+2e+1])
};

__device__ __forceinline__ void load_q1(QRegs& qr, const uint16_t* __restrict__ q, int c) {
#pragma unroll
  for (int h = 0; h < kHidx; ++h)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + h * kDidx + 32 * j + 8 * c));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) qr.p[h][j][e] = pack2(bf16lo(w[e]), bf16hi(w[e]));
    }
}

// Full score of the quad's key, returned on all 4 lanes of the quad.
__device__ __forceinline__ float score_q1(const QRegs& qr, const uint4 (&kv)[4], int c) {
  unsigned long long acc[kHidx] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w[4] = {kv[j].x, kv[j].y, kv[j].z, kv[j].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const unsigned long long k2 = pack2(bf16lo(w[e]), bf16hi(w[e]));
#pragma unroll
      for (int h = 0; h < kHidx; ++h) ffma2(acc[h], k2, qr.p[h][j][e]);
    }
  }
  float d[kHidx];
#pragma unroll
  for (int h = 0; h < kHidx; ++h) d[h] = lo2(acc[h]) + hi2(acc[h]);
  // reduce-scatter over the quad: lane c ends with head c's full dot product
  const bool up = (c & 2) != 0;
  float a0 = up ? d[2] : d[0], a1 = up ? d[3] : d[1];
  const float b0 = up ? d[0] : d[2], b1 = up ? d[1] : d[3];
  a0 += __shfl_xor_sync(0xffffffffu, b0, 2);
  a1 += __shfl_xor_sync(0xffffffffu, b1, 2);
  const bool odd = (c & 1) != 0;
  float mine = odd ? a1 : a0;
  const float other = odd ? a0 : a1;
  mine += __shfl_xor_sync(0xffffffffu, other, 1);
  float r = mine > 0.0f ? mine : 0.0f;  // ReLU per head
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  r += __shfl_xor_sync(0xffffffffu, r, 2);
  return r;
}

__device__ __forceinline__ void load_row(uint4 (&kv)[4], const uint16_t* row, int c) {
  const char* p = reinterpret_cast<const char*>(row) + 16 * c;
#pragma unroll
  for (int j = 0; j < 4; ++j) kv[j] = ldg_stream(p + 64 * j);
}

// One query per unit.  FULL: unit = (query, 16 consecutive pages of its sequence).
// REINDEX: unit = (query, 1024 consecutive pool positions).
template <bool kReindex>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_q1_kernel(const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ keys,
                    const int32_t* __restrict__ q_seq, int32_t num_q, ScoreGeom g,
                    const int32_t* __restrict__ pool, int32_t pool_size,
                    uint32_t* __restrict__ ws, int64_t ws_stride, int32_t units_per_q, int32_t* st) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int quad = lane >> 2, c = lane & 3;
  const int64_t total_units = (int64_t)num_q * units_per_q;
  QRegs qr;
  int cur_q = -1;
  for (int64_t u = blockIdx.x; u < total_units; u += gridDim.x) {
    const int q = (int)(u / units_per_q);
    const int chunk = (int)(u - (int64_t)q * units_per_q);
    const int b = __ldg(q_seq + q);
    if (b < 0 || b >= g.num_seqs) {
      if (threadIdx.x == 0 && chunk == 0) report(st, CSA2_DEV_BAD_QSEQ);
      continue;
    }
    const int n_ctx = __ldg(g.seq_lens + b);
    int begin, count;  // candidate positions [begin, begin + count)
    if (kReindex) {
      begin = chunk * kUnitPool;
      count = min(kUnitPool, pool_size - begin);
    } else {
      begin = chunk * kUnitPages * kPage;
      count = min(kUnitPages * kPage, n_ctx - begin);
    }
    if (count <= 0) continue;
    if (q != cur_q) {
      load_q1(qr, q_idx + (int64_t)q * kHidx * kDidx, c);
      cur_q = q;
    }
    uint32_t* out = ws + (int64_t)q * ws_stride;
    const int groups = (count + 7) >> 3;
    const int mine = groups > warp ? (groups - warp + 7) >> 3 : 0;

    // Resolve the row of the quad's key in group k of this warp; false if invalid.
    auto locate = [&](int k, const uint16_t*& row) -> bool {
      const int pos = begin + 8 * (warp + 8 * k) + quad;
      row = keys;
      if (pos >= begin + count) return false;
      int t;
      if (kReindex) {
        t = __ldg(pool + (int64_t)q * pool_size + pos);
        if (t < 0) {
          if (t != -1 && c == 0) report(st, CSA2_DEV_BAD_INDEX);
          return false;
        }
        if (t >= n_ctx) {
          if (c == 0) report(st, CSA2_DEV_BAD_INDEX);
          return false;
        }
      } else {
        t = pos;
      }
      const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (t >> 6));
      if (pg < 0 || pg >= g.num_pages) {
        if (c == 0) report(st, CSA2_DEV_BAD_PAGE);
        return false;
      }
      row = keys + ((int64_t)pg * kPage + (t & (kPage - 1))) * kDidx;
      return true;
    };

    uint4 buf[kDepth][4];
    bool ok[kDepth];
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
      ok[i] = false;
      if (i < mine) {
        const uint16_t* row;
        ok[i] = locate(i, row);
        load_row(buf[i], row, c);
      }
    }
    for (int k0 = 0; k0 < mine; k0 += kDepth) {
#pragma unroll
      for (int i = 0; i < kDepth; ++i) {
        const int k = k0 + i;
        if (k < mine) {
          const float s = score_q1(qr, buf[i], c);
          const int pos = begin + 8 * (warp + 8 * k) + quad;
          if (c == 0 && pos < begin + count) out[pos] = ok[i] ? rank_key(s) : 0u;
          if (k + kDepth < mine) {
            const uint16_t* row;
            ok[i] = locate(k + kDepth, row);
            load_row(buf[i], row, c);
          }
        }
      }
    }
  }
}

// Batched draft queries (Full): for one sequence with T <= 4 queries, the 4T
// query-head rows form the A operand (16 rows, zero padded) of m16n8k16 bf16 MMAs and
// 8 keys form B, so every key row is read once for all of the sequence's queries.
// The 128 dims are visited in a permuted order shared by A and B: lane c's 16-byte
// load of dims 32j+8c..+7 supplies its B fragments for k-steps 2j and 2j+1.
__global__ void __launch_bounds__(kScoreThreads, 2)
    score_batched_kernel(const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ keys,
                         const int32_t* __restrict__ q_seq, int32_t num_q, ScoreGeom g,
                         uint32_t* __restrict__ ws, int64_t ws_stride, int32_t units_per_seq,
                         int32_t* st) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, c = lane & 3;
  const int64_t total_units = (int64_t)g.num_seqs * units_per_seq;
  uint32_t a[8][4];
  int cur_b = -1, q0 = 0, T = 0;
  for (int64_t u = blockIdx.x; u < total_units; u += gridDim.x) {
    const int b = (int)(u / units_per_seq);
    const int chunk = (int)(u - (int64_t)b * units_per_seq);
    const int n_ctx = __ldg(g.seq_lens + b);
    const int begin = chunk * kUnitPages * kPage;
    const int count = min(kUnitPages * kPage, n_ctx - begin);
    if (count <= 0) continue;
    if (b != cur_b) {
      // queries of sequence b: [lower_bound(b), upper_bound(b)) in the sorted q_seq
      int lo = 0, hi = num_q;
      while (lo < hi) {
        const int m = (lo + hi) >> 1;
        if (__ldg(q_seq + m) < b) lo = m + 1; else hi = m;
      }
      int lo2 = lo, hi2 = num_q;
      while (lo2 < hi2) {
        const int m = (lo2 + hi2) >> 1;
        if (__ldg(q_seq + m) <= b) lo2 = m + 1; else hi2 = m;
      }
      q0 = lo;
      T = lo2 - lo;
      if (T > 4) {
        if (threadIdx.x == 0 && chunk == 0) report(st, CSA2_DEV_BAD_QSEQ);
        T = 4;
      }
      cur_b = b;
      // A fragments: rows r = 4t + h; lane holds rows gq and gq + 8.
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t u0[4] = {0, 0, 0, 0}, u1[4] = {0, 0, 0, 0};
        const int t0 = gq >> 2, t1 = t0 + 2, h = gq & 3;
        if (t0 < T) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(
              q_idx + ((int64_t)(q0 + t0) * kHidx + h) * kDidx + 32 * j + 8 * c));
          u0[0] = v.x; u0[1] = v.y; u0[2] = v.z; u0[3] = v.w;
        }
        if (t1 < T) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(
              q_idx + ((int64_t)(q0 + t1) * kHidx + h) * kDidx + 32 * j + 8 * c));
          u1[0] = v.x; u1[1] = v.y; u1[2] = v.z; u1[3] = v.w;
        }
        a[2 * j][0] = u0[0]; a[2 * j][1] = u1[0]; a[2 * j][2] = u0[1]; a[2 * j][3] = u1[1];
        a[2 * j + 1][0] = u0[2]; a[2 * j + 1][1] = u1[2]; a[2 * j + 1][2] = u0[3]; a[2 * j + 1][3] = u1[3];
      }
    }
    if (T == 0) continue;
    const int groups = (count + 7) >> 3;
    const int mine = groups > warp ? (groups - warp + 7) >> 3 : 0;
    auto locate = [&](int k, const uint16_t*& row) -> bool {
      const int t = begin + 8 * (warp + 8 * k) + gq;
      row = keys;
      if (t >= begin + count) return false;
      const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (t >> 6));
      if (pg < 0 || pg >= g.num_pages) {
        if (c == 0) report(st, CSA2_DEV_BAD_PAGE);
        return false;
      }
      row = keys + ((int64_t)pg * kPage + (t & (kPage - 1))) * kDidx;
      return true;
    };
    uint4 buf[kDepth][4];
    bool ok[kDepth];
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
      ok[i] = false;
      if (i < mine) {
        const uint16_t* row;
        ok[i] = locate(i, row);
        load_row(buf[i], row, c);
      }
    }
    for (int k0 = 0; k0 < mine; k0 += kDepth) {
#pragma unroll
      for (int i = 0; i < kDepth; ++i) {
        const int k = k0 + i;
        if (k < mine) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t bw[4] = {buf[i][j].x, buf[i][j].y, buf[i][j].z, buf[i][j].w};
#pragma unroll
            for (int hs = 0; hs < 2; ++hs) {
              const uint32_t* aa = a[2 * j + hs];
              asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
                  "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                  : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                  : "r"(aa[0]), "r"(aa[1]), "r"(aa[2]), "r"(aa[3]), "r"(bw[2 * hs]),
                    "r"(bw[2 * hs + 1]));
            }
          }
          // d0,d1: row gq (t = gq/4, head gq%4), keys 2c, 2c+1; d2,d3: row gq + 8 (t + 2)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float r = d[e] > 0.0f ? d[e] : 0.0f;
            r += __shfl_xor_sync(0xffffffffu, r, 4);
            r += __shfl_xor_sync(0xffffffffu, r, 8);
            d[e] = r;
          }
          // validity of keys 2c and 2c+1 of this group: held by quads 2c and 2c+1
          const int okb = ok[i] ? 1 : 0;
          const int ok0 = __shfl_sync(0xffffffffu, okb, (2 * c) * 4);
          const int ok1 = __shfl_sync(0xffffffffu, okb, (2 * c + 1) * 4);
          if ((gq & 3) == 0) {
            const int t0 = gq >> 2;
            const int base = begin + 8 * (warp + 8 * k);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int t = t0 + ((e >> 1) << 1);
              const int pos = base + 2 * c + (e & 1);
              const int okk = (e & 1) ? ok1 : ok0;
              if (t < T && pos < begin + count)
                ws[(int64_t)(q0 + t) * ws_stride + pos] = okk ? rank_key(d[e]) : 0u;
            }
          }
          if (k + kDepth < mine) {
            const uint16_t* row;
            ok[i] = locate(k + kDepth, row);
            load_row(buf[i], row, c);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ selection -----

constexpr int kSelCluster = 8;
constexpr int kSelThreads = 512;
constexpr int kSelCacheKeys = 16384;  // per-CTA keys kept in shared memory (64 KB)
constexpr int kBins = 2048;

struct SelShared {
  uint32_t hist[2][2][kBins];        // [buffer][target][bin]
  uint32_t counts[4];                // gtK, eqK, gtP, eqP of this CTA
  uint32_t nvalid;                   // valid keys of this CTA
  uint32_t warp_tmp[kSelThreads / 32][2];
  uint32_t res_prefix[2], res_above[2];
  uint32_t scan_carry[2][2];
};

// Exclusive suffix sums of (v0, v1) over the threads of the block:
// out = sum over threads with a larger index.  Also returns block totals.
__device__ __forceinline__ void block_suffix2(SelShared& sh, uint32_t v0, uint32_t v1,
                                              uint32_t& s0, uint32_t& s1, uint32_t& t0,
                                              uint32_t& t1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x0 = v0, x1 = v1;  // inclusive suffix within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y0 = __shfl_down_sync(0xffffffffu, x0, o);
    const uint32_t y1 = __shfl_down_sync(0xffffffffu, x1, o);
    if (lane + o < 32) {
      x0 += y0;
      x1 += y1;
    }
  }
  __syncthreads();
  if (lane == 0) {
    sh.warp_tmp[warp][0] = x0;
    sh.warp_tmp[warp][1] = x1;
  }
  __syncthreads();
  uint32_t w0 = 0, w1 = 0, a0 = 0, a1 = 0;
  for (int w = 0; w < kSelThreads / 32; ++w) {
    if (w > warp) {
      w0 += sh.warp_tmp[w][0];
      w1 += sh.warp_tmp[w][1];
    }
    a0 += sh.warp_tmp[w][0];
    a1 += sh.warp_tmp[w][1];
  }
  s0 = w0 + x0 - v0;
  s1 = w1 + x1 - v1;
  t0 = a0;
  t1 = a1;
}

// Exclusive prefix sums (lower thread index) of (v0, v1), plus block totals.
__device__ __forceinline__ void block_prefix2(SelShared& sh, uint32_t v0, uint32_t v1,
                                              uint32_t& p0, uint32_t& p1, uint32_t& t0,
                                              uint32_t& t1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x0 = v0, x1 = v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y0 = __shfl_up_sync(0xffffffffu, x0, o);
    const uint32_t y1 = __shfl_up_sync(0xffffffffu, x1, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
    }
  }
  __syncthreads();
  if (lane == 31) {
    sh.warp_tmp[warp][0] = x0;
    sh.warp_tmp[warp][1] = x1;
  }
  __syncthreads();
  uint32_t w0 = 0, w1 = 0, a0 = 0, a1 = 0;
  for (int w = 0; w < kSelThreads / 32; ++w) {
    if (w < warp) {
      w0 += sh.warp_tmp[w][0];
      w1 += sh.warp_tmp[w][1];
    }
    a0 += sh.warp_tmp[w][0];
    a1 += sh.warp_tmp[w][1];
  }
  p0 = w0 + x0 - v0;
  p1 = w1 + x1 - v1;
  t0 = a0;
  t1 = a1;
}

// Top-k selection for one query per cluster (gridDim.y = num_q).  Targets: t = 0 is
// the top-K output, t = 1 the candidate pool (FULL with a pool output only).
template <bool kReindex>
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads, 1)
    select_kernel(const uint32_t* __restrict__ ws, int64_t ws_stride,
                  const int32_t* __restrict__ q_seq, const int32_t* __restrict__ seq_lens,
                  int32_t num_seqs, const int32_t* __restrict__ pool_in, int32_t pool_size,
                  int32_t topk, int32_t* __restrict__ out_idx, int32_t* __restrict__ pool_out,
                  int32_t* st) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem_raw + sizeof(SelShared));
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int q = blockIdx.y;
  const int tid = threadIdx.x;

  int n;
  if (kReindex) {
    n = pool_size;
  } else {
    const int b = __ldg(q_seq + q);
    n = (b >= 0 && b < num_seqs) ? __ldg(seq_lens + b) : 0;
  }
  const int ntargets = (!kReindex && pool_out != nullptr && pool_size > 0) ? 2 : 1;
  const uint32_t want_max[2] = {(uint32_t)topk, (uint32_t)(kReindex ? 0 : pool_size)};

  // this CTA's range of candidate positions
  int L = (n + kSelCluster - 1) / kSelCluster;
  L = (L + 3) & ~3;
  const int lo = min(n, rank * L), hi = min(n, lo + L);
  const int len = hi - lo;
  const uint32_t* src = ws + (int64_t)q * ws_stride + lo;
  const bool cached = len <= kSelCacheKeys;
  if (cached) {
    for (int i = tid; i < len; i += kSelThreads) cache[i] = __ldcg(src + i);
  }
  auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : __ldcg(src + i); };

  // ---- pass 0: histogram of bits 31..21 of the valid keys; count valid keys ----
  for (int i = tid; i < kBins; i += kSelThreads) sh.hist[0][0][i] = 0;
  __syncthreads();
  uint32_t my_valid = 0;
  for (int i = tid; i < len; i += kSelThreads) {
    const uint32_t k = key_at(i);
    if (k != 0) {
      atomicAdd(&sh.hist[0][0][k >> 21], 1u);
      ++my_valid;
    }
  }
  my_valid = __reduce_add_sync(0xffffffffu, my_valid);
  if (tid == 0) sh.nvalid = 0;
  __syncthreads();
  if ((tid & 31) == 0) atomicAdd(&sh.nvalid, my_valid);
  cluster.sync();

  uint32_t nvalid = 0;
  for (int r = 0; r < kSelCluster; ++r) nvalid += *cluster.map_shared_rank(&sh.nvalid, r);
  uint32_t want[2], prefix[2] = {0, 0}, above[2] = {0, 0};
  for (int t = 0; t < 2; ++t) want[t] = min(want_max[t], nvalid);

  // ---- radix passes: (shift of the examined digit, digit width, prefix shift) ----
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int buf = pass & 1;
    const int shift = shifts[pass], width = widths[pass];
    const uint32_t dmask = (1u << width) - 1u;
    if (pass > 0) {
      for (int t = 0; t < ntargets; ++t)
        for (int i = tid; i < kBins; i += kSelThreads) sh.hist[buf][t][i] = 0;
      __syncthreads();
      for (int i = tid; i < len; i += kSelThreads) {
        const uint32_t k = key_at(i);
        if (k == 0) continue;
        const uint32_t hiBits = k >> (shift + width);
        for (int t = 0; t < ntargets; ++t)
          if (want[t] > 0 && hiBits == prefix[t]) atomicAdd(&sh.hist[buf][t][(k >> shift) & dmask], 1u);
      }
      cluster.sync();
    }
    // sum the cluster's histograms: thread handles bins 4*tid .. 4*tid+3
    for (int t = 0; t < ntargets; ++t) {
      const int tsrc = pass == 0 ? 0 : t;
      uint32_t v[4] = {0, 0, 0, 0};
      if (4 * tid < (1 << width)) {
        for (int r = 0; r < kSelCluster; ++r) {
          const uint4 x = *reinterpret_cast<const uint4*>(
              cluster.map_shared_rank(&sh.hist[buf][tsrc][4 * tid], r));
          v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
        }
      }
      const uint32_t mysum = v[0] + v[1] + v[2] + v[3];
      uint32_t suf, dummy, tot, dummy2;
      block_suffix2(sh, mysum, 0u, suf, dummy, tot, dummy2);
      if (want[t] > 0) {
        // bins above this thread's 4 bins hold `above + suf` keys
        uint32_t acc = above[t] + suf;
        if (acc < want[t] && acc + mysum >= want[t]) {
          for (int e = 3; e >= 0; --e) {
            if (acc + v[e] >= want[t]) {
              sh.res_prefix[t] = (prefix[t] << width) | (uint32_t)(4 * tid + e);
              sh.res_above[t] = acc;
              break;
            }
            acc += v[e];
          }
        }
      }
      __syncthreads();
      if (want[t] > 0) {
        prefix[t] = sh.res_prefix[t];
        above[t] = sh.res_above[t];
      }
      __syncthreads();
    }
  }
  // prefix[t] is now the exact key T_t of the want[t]-th largest; above[t] counts keys > T_t.

  // ---- ordered compaction ----
  uint32_t gt[2] = {0, 0}, eq[2] = {0, 0};
  for (int i = tid; i < len; i += kSelThreads) {
    const uint32_t k = key_at(i);
    for (int t = 0; t < ntargets; ++t) {
      if (want[t] == 0) continue;
      gt[t] += k > prefix[t];
      eq[t] += k == prefix[t];
    }
  }
  for (int t = 0; t < 2; ++t) {
    gt[t] = __reduce_add_sync(0xffffffffu, gt[t]);
    eq[t] = __reduce_add_sync(0xffffffffu, eq[t]);
  }
  if (tid < 4) sh.counts[tid] = 0;
  __syncthreads();
  if ((tid & 31) == 0) {
    atomicAdd(&sh.counts[0], gt[0]);
    atomicAdd(&sh.counts[1], eq[0]);
    atomicAdd(&sh.counts[2], gt[1]);
    atomicAdd(&sh.counts[3], eq[1]);
  }
  cluster.sync();
  uint32_t base[2] = {0, 0}, take[2] = {0, 0};
  for (int t = 0; t < ntargets; ++t) {
    if (want[t] == 0) continue;
    const uint32_t quota = want[t] - above[t];
    uint32_t ties_before = 0;
    for (int r = 0; r < kSelCluster; ++r) {
      const uint32_t g_r = *cluster.map_shared_rank(&sh.counts[2 * t], r);
      const uint32_t e_r = *cluster.map_shared_rank(&sh.counts[2 * t + 1], r);
      const uint32_t tk = quota > ties_before ? min(quota - ties_before, e_r) : 0u;
      if (r < rank) base[t] += g_r + tk;
      if (r == rank) take[t] = tk;
      ties_before += e_r;
    }
  }
  // walk the range in tiles of 4 consecutive keys per thread
  int32_t* outp[2] = {out_idx + (int64_t)q * topk,
                      pool_out ? pool_out + (int64_t)q * pool_size : nullptr};
  uint32_t tie_run[2] = {0, 0}, sel_run[2] = {0, 0};
  const int32_t* pin = kReindex ? pool_in + (int64_t)q * pool_size + lo : nullptr;
  for (int t0 = 0; t0 < len; t0 += 4 * kSelThreads) {
    const int i0 = t0 + 4 * tid;
    uint32_t k4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) k4[e] = (i0 + e < len) ? key_at(i0 + e) : 0u;
    for (int t = 0; t < ntargets; ++t) {
      if (want[t] == 0) continue;
      uint32_t nt = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) nt += (k4[e] == prefix[t]);
      uint32_t tie_pre, d0, tie_tot, d1;
      block_prefix2(sh, nt, 0u, tie_pre, d0, tie_tot, d1);
      uint32_t tr = tie_run[t] + tie_pre;
      uint32_t selmask = 0, ns = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool is_tie = k4[e] == prefix[t];
        const bool s = (k4[e] > prefix[t]) || (is_tie && tr < take[t]);
        tr += is_tie;
        if (s) {
          selmask |= 1u << e;
          ++ns;
        }
      }
      uint32_t sel_pre, d2, sel_tot, d3;
      block_prefix2(sh, ns, 0u, sel_pre, d2, sel_tot, d3);
      uint32_t pos = base[t] + sel_run[t] + sel_pre;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (selmask & (1u << e)) {
          const int token = kReindex ? __ldg(pin + i0 + e) : lo + i0 + e;
          if (pos < want[t]) outp[t][pos] = token;
          ++pos;
        }
      }
      tie_run[t] += tie_tot;
      sel_run[t] += sel_tot;
    }
  }
  // -1 padding after the selected entries
  if (rank == 0) {
    for (int i = (int)want[0] + tid; i < topk; i += kSelThreads) outp[0][i] = -1;
    if (ntargets == 2)
      for (int i = (int)want[1] + tid; i < pool_size; i += kSelThreads) outp[1][i] = -1;
  }
  cluster.sync();  // no CTA leaves while others may still read its shared memory
}

// ------------------------------------------------------------------ launchers -----

size_t select_smem_bytes() { return sizeof(SelShared) + (size_t)kSelCacheKeys * 4; }

cudaError_t launch_score_full(const uint16_t* q_idx, const uint16_t* keys, const int32_t* q_seq,
                              int32_t num_q, int32_t max_q_per_seq, const csa2_pages& pg,
                              uint32_t* ws, int64_t ws_stride, int32_t* st, cudaStream_t s,
                              int num_sms) {
  ScoreGeom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  const int units = (pg.max_pages_per_seq + kUnitPages - 1) / kUnitPages;
  if (max_q_per_seq <= 1) {
    int64_t total = (int64_t)num_q * units;
    int grid = (int)std::min<int64_t>(total, (int64_t)num_sms);
    if (grid < 1) grid = 1;
    score_q1_kernel<false><<<grid, kScoreThreads, 0, s>>>(q_idx, keys, q_seq, num_q, g, nullptr, 0,
                                                          ws, ws_stride, units, st);
  } else {
    int64_t total = (int64_t)pg.num_seqs * units;
    int grid = (int)std::min<int64_t>(total, (int64_t)num_sms * 2);
    if (grid < 1) grid = 1;
    score_batched_kernel<<<grid, kScoreThreads, 0, s>>>(q_idx, keys, q_seq, num_q, g, ws,
                                                        ws_stride, units, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_score_reindex(const uint16_t* q_idx, const uint16_t* keys, const int32_t* q_seq,
                                 int32_t num_q, const csa2_pages& pg, const int32_t* pool,
                                 int32_t pool_size, uint32_t* ws, int32_t* st, cudaStream_t s,
                                 int num_sms) {
  ScoreGeom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  const int units = (pool_size + kUnitPool - 1) / kUnitPool;
  int64_t total = (int64_t)num_q * units;
  int grid = (int)std::min<int64_t>(total, (int64_t)num_sms);
  if (grid < 1) grid = 1;
  score_q1_kernel<true><<<grid, kScoreThreads, 0, s>>>(q_idx, keys, q_seq, num_q, g, pool,
                                                       pool_size, ws, pool_size, units, st);
  return cudaGetLastError();
}

cudaError_t launch_select(bool reindex, const uint32_t* ws, int64_t ws_stride, const int32_t* q_seq,
                          const csa2_pages& pg, int32_t num_q, const int32_t* pool_in,
                          int32_t pool_size, int32_t topk, int32_t* out_idx, int32_t* pool_out,
                          int32_t* st, cudaStream_t s) {
  const size_t smem = select_smem_bytes();
  dim3 grid(kSelCluster, num_q);
  if (reindex) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<true><<<grid, kSelThreads, smem, s>>>(ws, ws_stride, q_seq, pg.seq_lens,
                                                        pg.num_seqs, pool_in, pool_size, topk,
                                                        out_idx, nullptr, st);
  } else {
    cudaError_t e = cudaFuncSetAttribute(select_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<false><<<grid, kSelThreads, smem, s>>>(ws, ws_stride, q_seq, pg.seq_lens,
                                                         pg.num_seqs, nullptr, pool_size, topk,
                                                         out_idx, pool_out, st);
  }
  return cudaGetLastError();
}

}  // namespace csa2
