// Multi-query sparse attention in dense-contraction form: a chunk of up to four queries of
// one sequence (the draft tokens of a decode step, or consecutive positions of a prefill
// chunk), each with its own top-K selection.  Draft tokens: tech-report digest, DSpark
// item under "さらなるアーキテクチャ拡張技術" (speculative decoding, semi-autoregressive
// drafts); per-query selection: the digest's "Hierarchical Sparse Indexer".
//
// tech-report digest (jiwasawa.github.io), "Reuse Mode": sparse attention runs over the
// selected top-K entries; zaikei.co.jp article, "CSA2とFP4でキャッシュを圧縮": the main KV
// is FP4 E2M1 and is dequantised before attention.  The result is that of the per-query
// path (`csa2_sparse_attn`) for each query; only the order of work differs:
//   1. chunk_union_kernel (one CTA per chunk): the chunk's G x K entries are sorted as
//      (token << 2 | query) keys in shared memory (bitonic), equal tokens merged into one
//      union entry with a G-bit membership mask, and the entries resolved through the
//      page table and compacted in token order;
//   2. chunk_attn_kernel (one CTA per (chunk, span of the union)): every union
//      row is gathered and dequantised ONCE into an f16 tile in shared memory, and the
//      chunk's G x 16 heads are contracted against it on the tensor cores (mma.sync
//      m16n8k16, f16 operands from ldmatrix, fp32 accumulation): S = Q C^T over the 512
//      channels, the entries a query did not select masked to -inf, an fp32 online
//      softmax per head row, O += P C;
//   3. the split combine of the per-query path, reading only the spans that the chunk's
//      union reaches.
// E2M1 x E4M3 products are exact in f16 (at most 6 significant bits, 2^-10 .. 2688), and
// Q is prescaled per query by a power of two into f16 range, as in the per-query kernel.
// A token selected twice by one query counts once here (the indexer never emits a token
// twice).
#include <algorithm>
#include <cstddef>

#include "common.cuh"

namespace csa2 {

cudaError_t launch_attn_combine(const float* part_o, const float* part_ml, int nsplit,
                                int32_t num_q, float* out, float* lse, const int32_t* span_count,
                                int32_t span_len, int32_t chunk, cudaStream_t s);

namespace {

constexpr int kMaxChunk = 4;           // queries per chunk
constexpr int kUnionMax = 8192;        // chunk x topk at most (the in-shared-memory sort)
constexpr int kUnionThreads = 1024;
constexpr int kCT = 64;                // union entries per tile
constexpr int kSpanMin = 512;          // union entries per CTA at least
constexpr int kChunkThreads = 512;     // 16 warps
constexpr int kRows = kMaxChunk * kHq;  // 64 head rows
constexpr int kQStride = kDkv + 8;     // f16 per row of Q and of the dequantised tile
constexpr int kSStride = kCT + 4;      // fp32 per row of S
constexpr int kPStride = kCT + 8;      // f16 per row of P
constexpr uint32_t kSentinel = 0xFFFFFFFFu;

struct ChunkSmem {
  uint16_t qs[kRows][kQStride];  // Q, f16 after the per-query prescale
  uint16_t cs[kCT][kQStride];    // dequantised tile, f16
  float s[kRows][kSStride];      // logits of the tile
  uint16_t p[kRows][kPStride];   // weights of the tile, f16
  float alpha[kRows];
  float m_fin[kRows], l_fin[kRows];
  float kq[kMaxChunk];
  uint32_t qmax[kMaxChunk];
  int32_t tslot[kCT];
  uint32_t tmask[kCT];
};
static_assert(offsetof(ChunkSmem, cs) % 16 == 0 && offsetof(ChunkSmem, s) % 16 == 0 &&
                  offsetof(ChunkSmem, p) % 16 == 0 && (kQStride * 2) % 16 == 0 &&
                  (kPStride * 2) % 16 == 0 && sizeof(ChunkSmem) <= 232448,
              "16-byte rows for ldmatrix and vector stores; fits one CTA per SM");

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// D += A . B, m16n8k16, f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Four code bytes -> four f16x2 (byte k -> word k, low nibble -> low half), exact.
__device__ __forceinline__ void codes4_to_f16(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t byte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)((byte & 0xFFu) | ((byte & 0xFFu) << 8))));
  return h2;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---- 1. union of a chunk's selections ----
__global__ void __launch_bounds__(kUnionThreads, 1)
    chunk_union_kernel(const int32_t* __restrict__ idx, int32_t topk, int32_t chunk,
                       const int32_t* __restrict__ q_seq, const int32_t* __restrict__ seq_lens,
                       const int32_t* __restrict__ page_table, int32_t max_pages, int32_t num_pages,
                       int32_t num_seqs, int32_t* __restrict__ ucount, int32_t* __restrict__ uslot,
                       uint8_t* __restrict__ umask, int32_t* st) {
  grid_dep_wait();
  __shared__ uint32_t keys[kUnionMax];
  __shared__ uint32_t wsum[kUnionThreads / 32];
  __shared__ int ok_chunk;
  const int c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_tot = chunk * topk;
  int n2 = 2;
  while (n2 < n_tot) n2 <<= 1;
  const int64_t ubase = (int64_t)c * n_tot;

  const int b = __ldg(q_seq + (int64_t)c * chunk);
  if (tid == 0) {
    int ok = b >= 0 && b < num_seqs;
    for (int g = 1; g < chunk; ++g) ok &= __ldg(q_seq + (int64_t)c * chunk + g) == b;
    if (!ok) report(st, CSA2_DEV_BAD_QSEQ);
    ok_chunk = ok;
  }
  __syncthreads();
  if (!ok_chunk) {  // no entry is read: the chunk's queries get zero output, -inf lse
    if (tid == 0) ucount[c] = 0;
    return;
  }
  const int n_ctx = min(max(0, __ldg(seq_lens + b)), max_pages * kPage);

  // keys: (token << 2 | query), invalid entries as the sentinel (sorted last)
  const int32_t* ic = idx + (int64_t)c * n_tot;
  for (int i = tid; i < n2; i += kUnionThreads) {
    uint32_t k = kSentinel;
    if (i < n_tot) {
      const int32_t s = __ldg(ic + i);
      if (s >= 0 && s < n_ctx) k = ((uint32_t)s << 2) | (uint32_t)(i / topk);
      else if (s != -1) report(st, CSA2_DEV_BAD_INDEX);
    }
    keys[i] = k;
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n2; i += kUnionThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint32_t a = keys[i], v = keys[ixj];
          if ((a > v) == ((i & k) == 0)) {
            keys[i] = v;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }

  // union heads (first key of each token), their masks and slots; compaction in order
  const int per = (n2 + kUnionThreads - 1) / kUnionThreads;  // <= 8 consecutive keys
  const int i0 = tid * per;
  uint32_t flags = 0, masks = 0;  // bit e: key i0 + e heads a kept union entry; its mask
  int32_t slots[kUnionMax / kUnionThreads];
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < kUnionMax / kUnionThreads; ++e) {
    slots[e] = -1;
    const int i = i0 + e;
    if (e >= per || i >= n2) continue;
    const uint32_t k = keys[i];
    if (k == kSentinel) continue;
    const uint32_t tok = k >> 2;
    if (i > 0 && (keys[i - 1] >> 2) == tok) continue;
    uint32_t m = 0;
    for (int j = i; j < n2 && keys[j] != kSentinel && (keys[j] >> 2) == tok; ++j) m |= 1u << (keys[j] & 3u);
    const int32_t pg = __ldg(page_table + (int64_t)b * max_pages + (tok >> 6));
    if (pg < 0 || pg >= num_pages) {
      report(st, CSA2_DEV_BAD_PAGE);
      continue;
    }
    slots[e] = pg * kPage + (int32_t)(tok & (kPage - 1));
    flags |= 1u << e;
    masks |= m << (4 * e);
    ++cnt;
  }
  // block exclusive scan of cnt
  uint32_t x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t before = 0, total = 0;
  for (int w = 0; w < kUnionThreads / 32; ++w) {
    if (w < warp) before += wsum[w];
    total += wsum[w];
  }
  uint32_t pos = before + x - cnt;
#pragma unroll
  for (int e = 0; e < kUnionMax / kUnionThreads; ++e)
    if (flags & (1u << e)) {
      uslot[ubase + pos] = slots[e];
      umask[ubase + pos] = (uint8_t)((masks >> (4 * e)) & 0xFu);
      ++pos;
    }
  if (tid == 0) ucount[c] = (int32_t)total;
}

// ---- 2. contraction over the union ----
__global__ void __launch_bounds__(kChunkThreads, 1)
    chunk_attn_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ codes,
                      const uint8_t* __restrict__ scales, int32_t chunk, int32_t n_tot,
                      const int32_t* __restrict__ ucount, const int32_t* __restrict__ uslot,
                      const uint8_t* __restrict__ umask, float softmax_scale, int32_t span_len,
                      int32_t nspan, float* __restrict__ part_o, float* __restrict__ part_ml) {
  grid_dep_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChunkSmem& sm = *reinterpret_cast<ChunkSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, iq = lane & 3;
  const int c = blockIdx.y, span = blockIdx.x;
  const int U = __ldg(ucount + c);
  const int jbeg = span * span_len;
  if (jbeg >= U) return;  // the combine reads only the spans that the union reaches
  const int ecount = min(U - jbeg, span_len);
  const int ntiles = (ecount + kCT - 1) / kCT;
  const int64_t ubase = (int64_t)c * n_tot + jbeg;

  // ---- Q: per-query max |q| -> power-of-two prescale -> f16 rows ----
  if (tid < kMaxChunk) sm.qmax[tid] = 0;
  __syncthreads();
  const uint4* qc = reinterpret_cast<const uint4*>(q + (int64_t)c * chunk * kHq * kDkv);
  constexpr int kVecPerQuery = kHq * kDkv / 8;  // 16-byte vectors of one query
  for (int g = 0; g < chunk; ++g) {
    uint32_t mx = 0;
    for (int v = tid; v < kVecPerQuery; v += kChunkThreads) {
      const uint4 w = __ldg(qc + g * kVecPerQuery + v);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) mx = max(mx, max(ws[e] & 0x7FFFu, (ws[e] >> 16) & 0x7FFFu));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) atomicMax(&sm.qmax[g], mx);
  }
  __syncthreads();
  if (tid < kMaxChunk) {
    int sh = 0;
    const uint32_t m = tid < chunk ? sm.qmax[tid] : 0u;
    if (m != 0) sh = max(-126, min(126, 14 - ((int)((m >> 7) & 0xFF) - 127)));
    sm.qmax[tid] = (uint32_t)(sh + 127);  // biased exponent of 2^sh
    sm.kq[tid] = softmax_scale * 1.4426950408889634f * __uint_as_float((uint32_t)(127 - sh) << 23);
  }
  __syncthreads();
  for (int v = tid; v < kMaxChunk * kVecPerQuery; v += kChunkThreads) {
    const int g = v / kVecPerQuery, r = v % kVecPerQuery;  // row h = r / 64, channels 8 (r % 64)
    uint4 o = make_uint4(0, 0, 0, 0);
    if (g < chunk) {
      const uint4 w = __ldg(qc + g * kVecPerQuery + r);
      const float pre = __uint_as_float(sm.qmax[g] << 23);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t hs[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 h = __floats2half2_rn(bf16lo(ws[e]) * pre, bf16hi(ws[e]) * pre);
        hs[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      o = make_uint4(hs[0], hs[1], hs[2], hs[3]);
    }
    *reinterpret_cast<uint4*>(&sm.qs[g * kHq + r / (kDkv / 8)][8 * (r % (kDkv / 8))]) = o;
  }

  // warp roles: m-block (query) mb; S: tokens 16 nb .. + 15; O: channels 128 nb .. + 127
  const int mb = warp & 3, nb = warp >> 2;
  const bool active = mb < chunk;
  const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lhi = lane >> 4;  // ldmatrix A rows
  float oacc[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.0f;
  // softmax ownership: row sr = tid / 8 (query sr / 16), tokens 8 (tid % 8) .. + 7
  const int sr = tid >> 3, sp = tid & 7, sg = sr >> 4;
  float m_run = -INFINITY, l_run = 0.0f;

  for (int t = 0; t < ntiles; ++t) {
    __syncthreads();  // the previous tile's products are done with cs, p and the metadata
    if (tid < kCT) {
      const int e = t * kCT + tid;
      const bool in = e < ecount;
      sm.tslot[tid] = in ? __ldg(uslot + ubase + e) : -1;
      sm.tmask[tid] = in ? (uint32_t)__ldg(umask + ubase + e) : 0u;
    }
    __syncthreads();
    // ---- gather + dequantise: row tid / 8, channels 64 (tid % 8) .. + 63 ----
    {
      const int row = tid >> 3, part = tid & 7;
      const int32_t slot = sm.tslot[row];
      uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
      uint32_t sc = 0;
      if (slot >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(codes + (int64_t)slot * kCodeRow + 32 * part);
        c0 = __ldg(src);
        c1 = __ldg(src + 1);
        sc = __ldg(reinterpret_cast<const uint32_t*>(scales + (int64_t)slot * kScaleRow + 4 * part));
      }
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint4* dst = reinterpret_cast<uint4*>(&sm.cs[row][64 * part]);
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {  // 16-channel group gi: code words 2 gi, 2 gi + 1
        const uint32_t s2 = scale_f16x2(sc >> (8 * gi));
        uint32_t h0[4], h1[4];
        codes4_to_f16(cw[2 * gi], h0);
        codes4_to_f16(cw[2 * gi + 1], h1);
        dst[2 * gi] = make_uint4(hmul2_u(h0[0], s2), hmul2_u(h0[1], s2), hmul2_u(h0[2], s2),
                                 hmul2_u(h0[3], s2));
        dst[2 * gi + 1] = make_uint4(hmul2_u(h1[0], s2), hmul2_u(h1[1], s2), hmul2_u(h1[2], s2),
                                     hmul2_u(h1[3], s2));
      }
    }
    __syncthreads();

    // ---- S = Q . C^T for query mb, tokens 16 nb .. + 15 ----
    if (active) {
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t a_base = sa(&sm.qs[16 * mb + lrow][8 * lhi]);
      const int mi = lane >> 3;
      const uint32_t b_base = sa(&sm.cs[16 * nb + 8 * (mi >> 1) + (lane & 7)][8 * (mi & 1)]);
#pragma unroll 8
      for (int k = 0; k < kDkv / 16; ++k) {
        uint32_t a[4], bb[4];
        ldsm_x4(a, a_base + 32 * k);
        ldsm_x4(bb, b_base + 32 * k);
        mma_f16(c0, a, bb[0], bb[1]);
        mma_f16(c1, a, bb[2], bb[3]);
      }
      const int col = 16 * nb + 2 * iq;
      *reinterpret_cast<float2*>(&sm.s[16 * mb + gq][col]) = make_float2(c0[0], c0[1]);
      *reinterpret_cast<float2*>(&sm.s[16 * mb + gq + 8][col]) = make_float2(c0[2], c0[3]);
      *reinterpret_cast<float2*>(&sm.s[16 * mb + gq][col + 8]) = make_float2(c1[0], c1[1]);
      *reinterpret_cast<float2*>(&sm.s[16 * mb + gq + 8][col + 8]) = make_float2(c1[2], c1[3]);
    }
    __syncthreads();

    // ---- online softmax (exp2 domain), entries not selected by the row's query masked ----
    if (sg < chunk) {
      const float kq = sm.kq[sg];
      float s[8];
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = 8 * sp + j;
        const bool sel = (sm.tmask[e] >> sg) & 1u;
        s[j] = sel ? sm.s[sr][e] * kq : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float mn = fmaxf(m_run, mt);
      const float alpha = (mn == -INFINITY || mn == m_run) ? 1.0f : exp2_fast(m_run - mn);
      const float mh = mn == -INFINITY ? 0.0f : mn;
      uint32_t pw[4];
      float psum = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 ph = __floats2half2_rn(exp2_fast(s[2 * j] - mh), exp2_fast(s[2 * j + 1] - mh));
        pw[j] = *reinterpret_cast<const uint32_t*>(&ph);
        psum += __low2float(ph) + __high2float(ph);
      }
      *reinterpret_cast<uint4*>(&sm.p[sr][8 * sp]) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l_run = l_run * alpha + psum;
      m_run = mn;
      if (sp == 0) sm.alpha[sr] = alpha;
    }
    __syncthreads();

    // ---- O += P . C for query mb, channels 128 nb .. + 127 ----
    if (active) {
      const float a_lo = sm.alpha[16 * mb + gq], a_hi = sm.alpha[16 * mb + gq + 8];
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        oacc[n][0] *= a_lo;
        oacc[n][1] *= a_lo;
        oacc[n][2] *= a_hi;
        oacc[n][3] *= a_hi;
      }
      const uint32_t pa = sa(&sm.p[16 * mb + lrow][8 * lhi]);
      const int mi = lane >> 3;
      const uint32_t vb = sa(&sm.cs[8 * (mi & 1) + (lane & 7)][128 * nb + 8 * (mi >> 1)]);
#pragma unroll
      for (int ks = 0; ks < kCT / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, pa + 32 * ks);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          uint32_t bb[4];
          ldsm_x4_t(bb, vb + ks * 16 * (kQStride * 2) + jj * 32);
          mma_f16(oacc[2 * jj], a, bb[0], bb[1]);
          mma_f16(oacc[2 * jj + 1], a, bb[2], bb[3]);
        }
      }
    }
  }

  // ---- split partials: unnormalised O, running max (exp2 domain) and sum per head row ----
  if (sg < chunk && sp == 0) {
    sm.m_fin[sr] = m_run;
    sm.l_fin[sr] = l_run;
  }
  __syncthreads();
  if (active) {
    const int qi = c * chunk + mb;
    float* po = part_o + ((int64_t)qi * nspan + span) * kHq * kDkv;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int ch = 128 * nb + 8 * n + 2 * iq;
      *reinterpret_cast<float2*>(po + gq * kDkv + ch) = make_float2(oacc[n][0], oacc[n][1]);
      *reinterpret_cast<float2*>(po + (gq + 8) * kDkv + ch) = make_float2(oacc[n][2], oacc[n][3]);
    }
  }
  if (tid < kRows && (tid >> 4) < chunk) {
    const int qi = c * chunk + (tid >> 4), h = tid & 15;
    float* ml = part_ml + ((int64_t)qi * nspan + span) * 2 * kHq;
    ml[h] = sm.m_fin[tid];
    ml[kHq + h] = sm.l_fin[tid];
  }
}

struct ChunkLayout {
  size_t count_off, slot_off, mask_off, o_off, ml_off, total;
  int span_len, nspan;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Span length: a multiple of the tile, at least kSpanMin entries, sized so that the
// chunks' selections (their upper bound, chunk x topk each) make about two CTAs per SM;
// longer spans write fewer split partials (32 KB per query and span).
ChunkLayout chunk_layout(int32_t num_q, int32_t chunk, int32_t topk, int num_sms) {
  ChunkLayout L{};
  const int64_t num_chunks = num_q / chunk, n_tot = (int64_t)chunk * topk;
  const int64_t slots = 2 * (int64_t)std::max(1, num_sms);
  const int64_t target = (num_chunks * n_tot + slots - 1) / slots;
  const int64_t cap = (n_tot + kCT - 1) / kCT * kCT;
  L.span_len = (int)std::min(cap, std::max<int64_t>(kSpanMin, (target + kCT - 1) / kCT * kCT));
  L.nspan = (int)((n_tot + L.span_len - 1) / L.span_len);
  L.count_off = 0;
  L.slot_off = round256(num_chunks * sizeof(int32_t));
  L.mask_off = L.slot_off + round256(num_chunks * n_tot * sizeof(int32_t));
  L.o_off = L.mask_off + round256(num_chunks * n_tot);
  L.ml_off = L.o_off + round256((size_t)num_q * L.nspan * kHq * kDkv * sizeof(float));
  L.total = L.ml_off + round256((size_t)num_q * L.nspan * 2 * kHq * sizeof(float));
  return L;
}

}  // namespace

int chunk_attn_max_union() { return kUnionMax; }
int chunk_attn_max_chunk() { return kMaxChunk; }

size_t chunk_attn_workspace_bytes(int32_t num_q, int32_t chunk, int32_t topk, int num_sms) {
  return chunk_layout(num_q, chunk, topk, num_sms).total;
}

cudaError_t launch_chunk_attn(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                              const int32_t* idx, const csa2_pages& pg, float* out, float* lse,
                              int32_t num_q, const int32_t* q_seq, int32_t chunk, int32_t topk,
                              float softmax_scale, void* ws, int32_t* st, cudaStream_t s,
                              int num_sms) {
  const ChunkLayout L = chunk_layout(num_q, chunk, topk, num_sms);
  unsigned char* w = reinterpret_cast<unsigned char*>(ws);
  int32_t* ucount = reinterpret_cast<int32_t*>(w + L.count_off);
  int32_t* uslot = reinterpret_cast<int32_t*>(w + L.slot_off);
  uint8_t* umask = w + L.mask_off;
  float* part_o = reinterpret_cast<float*>(w + L.o_off);
  float* part_ml = reinterpret_cast<float*>(w + L.ml_off);
  const int num_chunks = num_q / chunk;
  cudaError_t e = launch_pdl(chunk_union_kernel, dim3(num_chunks), dim3(kUnionThreads), 0, s, idx,
                             topk, chunk, q_seq, pg.seq_lens, pg.page_table, pg.max_pages_per_seq,
                             pg.num_pages, pg.num_seqs, ucount, uslot, umask, st);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(ChunkSmem);
  e = cudaFuncSetAttribute(chunk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(chunk_attn_kernel, dim3(L.nspan, num_chunks), dim3(kChunkThreads), smem, s, q, codes,
                 scales, chunk, chunk * topk, (const int32_t*)ucount, (const int32_t*)uslot,
                 (const uint8_t*)umask, softmax_scale, L.span_len, L.nspan, part_o, part_ml);
  if (e != cudaSuccess) return e;
  return launch_attn_combine(part_o, part_ml, L.nspan, num_q, out, lse, ucount, L.span_len, chunk, s);
}

}  // namespace csa2
