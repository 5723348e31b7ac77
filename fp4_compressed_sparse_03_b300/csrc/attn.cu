// Gather-dequantise sparse attention over the selected FP4 latent rows.
//
// zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮": the main KV is stored as
// FP4 E2M1 and dequantised before attention; tech-report digest (jiwasawa.github.io),
// "Reuse Mode": sparse attention runs directly over the inherited top-K entries.
// MQA over the shared latent: K = V = c_hat (512 channels), 16 query heads.
//
// One CTA (8 warps, two CTAs per SM) handles one (query, split) pair: up to
// `split_len` selected entries in tiles of 128 tokens.  Every code is dequantised once
// per product, from the staged bytes straight into tensor-core operand registers
// (E2M1 x E4M3 is exact in f16: at most 6 significant bits, magnitudes 2^-10 .. 2688):
//   1. cp.async gathers the tile's 128 x (256 B codes + 32 B scales) into a 2-stage
//      ring, 16 lanes per row; codes are laid out [64-channel slice][row][32 B], and
//      rows that are not selected (skipped entries, the ragged end of the split) are
//      zero-filled;
//   2. S^T partial = Q_c . C_c^T: warp w takes channels 128 (w % 4) .. + 127 of tokens
//      64 (w / 4) .. + 63 (mma.sync m16n8k16, f16 operands, fp32 accumulation; M = 16
//      heads, N = 8 tokens per instruction); the four channel partials are summed
//      through shared memory;
//   3. fp32 softmax in the exp2 domain, 16 threads per head, with a lazily moved
//      reference max per head: it only moves (and the output accumulators are
//      rescaled) when a tile's max exceeds it by more than 2^8, so every weight is at
//      most 2^8; P is rounded to f16 and the normaliser sums the rounded weights;
//   4. O_w += P . C_w: warp w owns channels 64 w .. 64 w + 63 of the output (M = 16
//      heads, N = 8 channels, K = 16 tokens per instruction), with the two-token operand
//      pairs assembled from the same staged bytes.
// Q is converted to f16 after a per-query power-of-two prescale (exact for every value
// within 2^28 of the largest |q|); the scale is undone in the logit factor.  Several
// splits per query are merged by a log-sum-exp combine kernel.
//
// MXFP4 variant (tech-report digest, "FP4 メイン KV Cache と SWA Bounded Replay": OCP MXFP4,
// read as one E8M0 scale per 32 channels): E8M0 scales span 2^-127 .. 2^127, beyond f16.
// The kernel gathers the scale bytes of the whole split up front, takes their maximum
// `ref`, and builds the same f16 operands as code x 2^(e - ref), which is exact for
// e >= ref - 23 (smaller contributions, 2^23 below the split's largest scale, lose
// precision or vanish); 2^(ref - 127) is folded into the logit factor and the output.
//
// A 128-token tile holds only 2 M multiply-adds per product, so the kernel is bound by
// the dequantisation arithmetic and per-tile latency, not by tensor throughput; operands
// built in registers avoid writing a dequantised f16 tile to shared memory and reading
// it back for each product.
#include <algorithm>
#include <cstddef>

#include "common.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnCtasPerSm = 2;
constexpr int kTile = 128;         // tokens per tile
constexpr int kStages = 2;         // cp.async ring: one tile in flight ahead of the current one
constexpr int kMaxSplit = 512;     // selected entries per CTA at most
constexpr int kMaxSplits = CSA2_ATTN_MAX_TOPK / kMaxSplit;  // splits per query at most
static_assert(kMaxSplits >= 64, "the split search goes up to 64 splits");
constexpr int kSliceCh = kDkv / kAttnWarps;           // 64 output channels per warp
constexpr int kSliceBytes = kSliceCh / 2;             // 32 code bytes per row and slice
constexpr int kKSplit = 4;                            // S partials: 128-channel quarters
constexpr int kSliceStride = kTile * kSliceBytes;     // 4 KB per channel slice of a stage
constexpr int kStageCodes = kTile * kCodeRow;         // 32 KB: [slice][row][32 B]
constexpr int kScaleHalf = kTile * 16;                // scales: [half][row][16 B]
constexpr int kStageBytes = kStageCodes + 2 * kScaleHalf;  // 36 KB
constexpr int kRedStride = kTile + 8;   // floats per (quarter, head) row of S partials
constexpr int kOStride = kDkv + 4;      // floats per head row of the output staging
constexpr float kRescaleGap = 8.0f;     // log2 units

static_assert(kSliceCh == 64 && kAttnThreads == 2 * kTile, "layout assumes 8 warps, 128-token tiles");

template <bool kMx>
struct AttnSmemT {
  // E4M3: codes + scales of each tile; MXFP4: codes only (the split's scales below)
  unsigned char stage[kStages][kMx ? kStageCodes : kStageBytes];
  float red[kKSplit][kHq][kRedStride];     // S^T partials; reused to stage the output
  uint16_t p[kHq][kTile];                  // P (f16): 16-byte units XOR-swizzled by head
  float alpha[kHq];
  float m_fin[kHq], l_fin[kHq];
  uint32_t qmax[kAttnWarps];
  uint32_t smax[kAttnWarps];
  int32_t slot[kMaxSplit];  // physical row of each selected entry, -1 if skipped
  unsigned char mxs[kMx ? kMaxSplit : 1][16];  // MXFP4: E8M0 bytes of every selected entry
};
template <bool kMx>
constexpr bool attn_layout_ok() {
  return offsetof(AttnSmemT<kMx>, red) % 16 == 0 && offsetof(AttnSmemT<kMx>, p) % 16 == 0 &&
         offsetof(AttnSmemT<kMx>, mxs) % 16 == 0 &&
         kAttnCtasPerSm * (sizeof(AttnSmemT<kMx>) + 1024) <= 233472;
}
static_assert(attn_layout_ok<false>() && attn_layout_ok<true>(),
              "16-byte alignment of vector accesses; two CTAs per SM");
static_assert(kHq * kOStride <= kKSplit * kHq * kRedStride, "output staging fits the partials");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte cp.async; `valid` false writes 16 zero bytes without reading global memory.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 2^x by the MUFU ex2 instruction (flushes subnormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two E4M3 bytes (low byte -> low half) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(two & 0xFFFFu)));
  return h2;
}
// The four bytes of `w` (two E2M1 codes each) -> four f16x2: byte k -> h_k, low nibble
// -> low half; exact.  Unpacking the word in one step feeds the conversions directly.
__device__ __forceinline__ void e2m1x4_unpack(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                              uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// D += A . B, m16n8k16, f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// f16 bits of 2^(e - ref), e <= ref: normal down to 2^-14, subnormal to 2^-24, else 0.
__device__ __forceinline__ uint32_t mx_factor_f16(uint32_t e, int ref) {
  const int d = (int)e - ref;
  if (d >= -14) return (uint32_t)(d + 15) << 10;
  if (d >= -24) return 1u << (d + 24);
  return 0u;
}
// 2^k as a float, k in [-127, 127] (2^-127 is subnormal, exact).
__device__ __forceinline__ float pow2f_attn(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << 22);
}

// Position of tile row r in code slice s: rows 4..7 of every group of 8 are stored in
// reverse order, so that both the S-phase reads (8 consecutive rows, 8 bytes each) and
// the O-phase reads (rows 2i or 2i + 1, i = 0..3, of a group) hit distinct banks; the
// slice index rotates rows within aligned groups of 4, so that the 16 pieces of one row
// written by a gather instruction spread over the banks.
__device__ __forceinline__ int stage_row(int r) { return r ^ (((r >> 2) & 1) * 3); }
__device__ __forceinline__ int slice_row(int r, int s) { return stage_row(r) ^ (s & 3); }

struct AttnGeom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t max_pages;
  int32_t num_pages;
  int32_t num_seqs;
};

// Gather the tile starting at local entry `e0`.  Codes: 16 lanes per row, lane -> one
// 16-byte piece, so each warp instruction reads two whole 256-byte rows.  Scales: two
// lanes per row.
template <bool kMx>
__device__ __forceinline__ void issue_tile(unsigned char* stage, int e0, int ecount,
                                           const int32_t* slot, const uint8_t* __restrict__ codes,
                                           const uint8_t* __restrict__ scales) {
  const int piece = threadIdx.x & 15, sl_i = piece >> 1;
#pragma unroll
  for (int k = 0; k < kTile / 16; ++k) {
    const int r = 16 * k + (threadIdx.x >> 4);
    const int e = e0 + r;
    const int32_t sl = e < ecount ? slot[e] : -1;
    const bool ok = sl >= 0;
    cp_async16(stage + sl_i * kSliceStride + slice_row(r, sl_i) * kSliceBytes + 16 * (piece & 1),
               codes + (ok ? (int64_t)sl * kCodeRow : 0) + 16 * piece, ok);
  }
  if (kMx) return;  // the split's scales were gathered up front
  const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
  const int e = e0 + r;
  const int32_t sl = e < ecount ? slot[e] : -1;
  const bool ok = sl >= 0;
  cp_async16(stage + kStageCodes + h * kScaleHalf + stage_row(r) * 16,
             scales + (ok ? (int64_t)sl * kScaleRow : 0) + 16 * h, ok);
}

template <bool kMx>
__global__ void __launch_bounds__(kAttnThreads, kAttnCtasPerSm)
    sparse_attn_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ codes,
                       const uint8_t* __restrict__ scales, const int32_t* __restrict__ idx,
                       AttnGeom g, const int32_t* __restrict__ q_seq, int32_t topk, int32_t split_len,
                       float softmax_scale, float* __restrict__ out, float* __restrict__ lse,
                       float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st) {
  grid_dep_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmemT<kMx>& sm = *reinterpret_cast<AttnSmemT<kMx>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, iq = lane & 3;  // mma fragment: row group, column pair
  const int qi = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
  const int jbeg = split * split_len;
  const int ecount = max(0, min(topk, jbeg + split_len) - jbeg);
  const int ntiles = (ecount + kTile - 1) / kTile;
  int b = __ldg(q_seq + qi);
  int n_ctx = 0;
  if (b < 0 || b >= g.num_seqs) {
    if (tid == 0) report(st, CSA2_DEV_BAD_QSEQ);
    b = 0;
  } else {
    n_ctx = min(max(0, __ldg(g.seq_lens + b)), g.max_pages * kPage);
  }
  const int32_t* idx_q = idx + (int64_t)qi * topk + jbeg;

  // Q first (its latency overlaps the index and page-table loads): heads gq and gq + 8,
  // channels 64 s + 16 iq .. + 15 of code slices s = 2 (warp % 4) + j, j = 0, 1 -- the
  // S-operand channels of this thread.  qr[4 hh + 2 j + v]: head gq + 8 hh, slice j, half v.
  const int quarter = warp & 3, thalf = warp >> 2;
  const uint4* qg = reinterpret_cast<const uint4*>(q + (int64_t)qi * kHq * kDkv + gq * kDkv +
                                                   2 * quarter * kSliceCh + 16 * iq);
  uint4 qr[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    qr[k] = __ldg(qg + (k >> 2) * (8 * kDkv * 2 / 16) + ((k >> 1) & 1) * (kSliceCh * 2 / 16) + (k & 1));

  // ---- resolve the selected entries to physical rows: the first tiles first ----
  // the index load of an entry is issued separately from its page-table lookup, so that
  // a thread's loads of several entries are in flight together
  auto resolve = [&](int e, int s) {
    int32_t slot = -1;
    if (s >= 0 && s < n_ctx) {
      const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (s >> 6));
      if (pg >= 0 && pg < g.num_pages) slot = pg * kPage + (s & (kPage - 1));
      else report(st, CSA2_DEV_BAD_PAGE);
    } else if (s != -1) {
      report(st, CSA2_DEV_BAD_INDEX);
    }
    sm.slot[e] = slot;
  };
  const int e_first = min(ecount, (kStages - 1) * kTile);
  static_assert((kStages - 1) * kTile <= kAttnThreads, "one first-tile entry per thread");
  if (tid < e_first) resolve(tid, __ldg(idx_q + tid));
  constexpr int kRest = (kMaxSplit - (kStages - 1) * kTile + kAttnThreads - 1) / kAttnThreads;
  int rest_s[kRest];
#pragma unroll
  for (int i = 0; i < kRest; ++i) {
    const int e = e_first + tid + i * kAttnThreads;
    rest_s[i] = e < ecount ? __ldg(idx_q + e) : -1;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < ntiles) issue_tile<kMx>(sm.stage[i], i * kTile, ecount, sm.slot, codes, scales);
    cp_async_commit();
  }
#pragma unroll
  for (int i = 0; i < kRest; ++i) {
    const int e = e_first + tid + i * kAttnThreads;
    if (e < ecount) resolve(e, rest_s[i]);
  }

  // ---- Q: max |q| -> power-of-two prescale -> f16 operand fragments (the barrier
  // below also publishes the remaining slots) ----
  uint32_t mx = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t w[4] = {qr[k].x, qr[k].y, qr[k].z, qr[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) sm.qmax[warp] = mx;
  __syncthreads();
  uint32_t mxa = 0;
#pragma unroll
  for (int w = 0; w < kAttnWarps; ++w) mxa = max(mxa, sm.qmax[w]);
  int sh = 0;
  if (mxa != 0) {
    const int e = (int)((mxa >> 7) & 0xFF) - 127;  // bf16 exponent of max |q|
    sh = max(-126, min(126, 14 - e));
  }
  const float pre = __uint_as_float((uint32_t)(127 + sh) << 23);   // 2^sh
  const float post = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
  float kq = softmax_scale * 1.4426950408889634f * post;  // logits in the exp2 domain
  int mx_ref = 0;  // MXFP4: largest E8M0 byte of the split
  if constexpr (kMx) {
    // gather every selected entry's 16 scale bytes (the slots are published above)
    for (int e = tid; e < kMaxSplit; e += kAttnThreads) {
      const bool ok = e < ecount && sm.slot[e] >= 0;
      cp_async16(&sm.mxs[e][0], scales + (ok ? (int64_t)sm.slot[e] * 16 : 0), ok);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    uint32_t m4 = 0;
    for (int e = tid; e < kMaxSplit; e += kAttnThreads) {
      const uint4 v = *reinterpret_cast<const uint4*>(&sm.mxs[e][0]);
      m4 = __vmaxu4(m4, __vmaxu4(__vmaxu4(v.x, v.y), __vmaxu4(v.z, v.w)));
    }
    uint32_t m = max(max(m4 & 0xFFu, (m4 >> 8) & 0xFFu), max((m4 >> 16) & 0xFFu, m4 >> 24));
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) sm.smax[warp] = m;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) mx_ref = max(mx_ref, (int)sm.smax[w]);
    kq *= pow2f_attn(mx_ref - 127);
  }
  // k-step 4 j + kk covers channels 16 iq + 4 kk .. + 3 of slice j: a0/a1 the first pair
  // (heads gq / gq + 8), a2/a3 the second -- the byte order of the staged codes
  uint32_t qa[8][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) {  // f16x2 word j of the thread's 32 channels
    const uint32_t wl = (&qr[j >> 2].x)[j & 3], wh = (&qr[4 + (j >> 2)].x)[j & 3];
    const __half2 hl = __floats2half2_rn(bf16lo(wl) * pre, bf16hi(wl) * pre);
    const __half2 hh = __floats2half2_rn(bf16lo(wh) * pre, bf16hi(wh) * pre);
    qa[j >> 1][2 * (j & 1)] = *reinterpret_cast<const uint32_t*>(&hl);
    qa[j >> 1][2 * (j & 1) + 1] = *reinterpret_cast<const uint32_t*>(&hh);
  }

  // softmax ownership: thread -> head sh_h, tokens 4 sk .. + 3 and 64 + 4 sk .. + 3
  const int sh_h = tid >> 4, sk = tid & 15;
  float m_ref = -INFINITY, l_run = 0.0f;
  float oacc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.0f;
  const uint32_t p_base = smem_u32(&sm.p[0][0]);
  const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lhi = lane >> 4;  // ldmatrix source rows

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<kStages - 2>();  // this thread's copies of tile t have landed
    __syncthreads();               // everyone's; and every warp is done with tile t - 1
    {
      const int tn = t + kStages - 1;
      if (tn < ntiles)
        issue_tile<kMx>(sm.stage[tn % kStages], tn * kTile, ecount, sm.slot, codes, scales);
      cp_async_commit();
    }
    const unsigned char* stg = sm.stage[t % kStages];

    // ---- S^T partial over channel quarter `quarter`, tokens 64 thalf .. + 63 ----
#pragma unroll 2
    for (int n = 0; n < kTile / 16; ++n) {
      const int tok = 64 * thalf + 8 * n + gq;
      float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int sl_i = 2 * quarter + j;
        const uint2 cw = *reinterpret_cast<const uint2*>(stg + sl_i * kSliceStride +
                                                         slice_row(tok, sl_i) * kSliceBytes + 8 * iq);
        // one scale: these 16 channels are one group
        uint32_t s2;
        if constexpr (kMx) {
          const uint32_t f = mx_factor_f16(sm.mxs[t * kTile + tok][2 * sl_i + (iq >> 1)], mx_ref);
          s2 = f | (f << 16);
        } else {
          const uint32_t sb = stg[kStageCodes + (sl_i >> 2) * kScaleHalf + stage_row(tok) * 16 +
                                  4 * (sl_i & 3) + iq];
          s2 = e4m3x2_to_f16x2(sb | (sb << 8));
        }
        uint32_t bf[8];
        e2m1x4_unpack(cw.x, bf[0], bf[1], bf[2], bf[3]);
        e2m1x4_unpack(cw.y, bf[4], bf[5], bf[6], bf[7]);
#pragma unroll
        for (int k = 0; k < 8; ++k) bf[k] = hmul2(bf[k], s2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma16816(c, qa[4 * j + kk], bf[2 * kk], bf[2 * kk + 1]);
      }
      const int col = 64 * thalf + 8 * n + 2 * iq;
      *reinterpret_cast<float2*>(&sm.red[quarter][gq][col]) = make_float2(c[0], c[1]);
      *reinterpret_cast<float2*>(&sm.red[quarter][gq + 8][col]) = make_float2(c[2], c[3]);
    }
    __syncthreads();

    // ---- softmax ----
    {
      float s[8];
      {
        const float4 a = *reinterpret_cast<const float4*>(&sm.red[0][sh_h][4 * sk]);
        const float4 c = *reinterpret_cast<const float4*>(&sm.red[0][sh_h][64 + 4 * sk]);
        s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
        s[4] = c.x; s[5] = c.y; s[6] = c.z; s[7] = c.w;
      }
#pragma unroll
      for (int w = 1; w < kKSplit; ++w) {
        const float4 a = *reinterpret_cast<const float4*>(&sm.red[w][sh_h][4 * sk]);
        const float4 c = *reinterpret_cast<const float4*>(&sm.red[w][sh_h][64 + 4 * sk]);
        s[0] += a.x; s[1] += a.y; s[2] += a.z; s[3] += a.w;
        s[4] += c.x; s[5] += c.y; s[6] += c.z; s[7] += c.w;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = t * kTile + (j < 4 ? 4 * sk + j : 64 + 4 * sk + j - 4);
        const bool valid = e < ecount && sm.slot[e] >= 0;
        s[j] = valid ? s[j] * kq : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      float mn = m_ref;
      if (m_ref == -INFINITY || mt > m_ref + kRescaleGap) mn = fmaxf(m_ref, mt);
      const float alpha = (mn != m_ref) ? ex2(m_ref - mn) : 1.0f;
      m_ref = mn;
      const float mh = (m_ref == -INFINITY) ? 0.0f : m_ref;  // no valid entry yet: all s are -inf
      uint32_t pw[4];
      float psum = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 ph = __floats2half2_rn(ex2(s[2 * j] - mh), ex2(s[2 * j + 1] - mh));
        pw[j] = *reinterpret_cast<const uint32_t*>(&ph);
        psum += __low2float(ph) + __high2float(ph);
      }
      unsigned char* prow = reinterpret_cast<unsigned char*>(&sm.p[sh_h][0]);
      const int x7 = sh_h & 7;
      *reinterpret_cast<uint2*>(prow + (((sk >> 1) ^ x7) << 4) + 8 * (sk & 1)) = make_uint2(pw[0], pw[1]);
      *reinterpret_cast<uint2*>(prow + (((8 + (sk >> 1)) ^ x7) << 4) + 8 * (sk & 1)) =
          make_uint2(pw[2], pw[3]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l_run = l_run * alpha + psum;
      if (sk == 0) sm.alpha[sh_h] = alpha;
    }
    __syncthreads();

    // ---- O += P . C over this warp's channels ----
    {
      const float a_lo = sm.alpha[gq], a_hi = sm.alpha[gq + 8];
      if (a_lo != 1.0f || a_hi != 1.0f) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          oacc[n][0] *= a_lo;
          oacc[n][1] *= a_lo;
          oacc[n][2] *= a_hi;
          oacc[n][3] *= a_hi;
        }
      }
    }
    const unsigned char* cs = stg + warp * kSliceStride;
    const unsigned char* ss = stg + kStageCodes + (warp >> 2) * kScaleHalf + 4 * (warp & 3);
#pragma unroll 2
    for (int ks = 0; ks < kTile / 16; ++ks) {
      uint32_t a[4];
      const int unit = 2 * ks + lhi;
      ldmatrix_x4(a, p_base + lrow * (kTile * 2) + ((unit ^ (lrow & 7)) << 4));
      const int t0 = 16 * ks + 2 * iq;
      const int r0 = stage_row(t0), r1 = stage_row(t0 + 1), r8 = stage_row(t0 + 8),
                r9 = stage_row(t0 + 9);
      const int xs = warp & 3;  // the slice's row rotation
      const uint32_t x0 = *reinterpret_cast<const uint32_t*>(cs + (r0 ^ xs) * kSliceBytes + 4 * gq);
      const uint32_t x1 = *reinterpret_cast<const uint32_t*>(cs + (r1 ^ xs) * kSliceBytes + 4 * gq);
      const uint32_t x8 = *reinterpret_cast<const uint32_t*>(cs + (r8 ^ xs) * kSliceBytes + 4 * gq);
      const uint32_t x9 = *reinterpret_cast<const uint32_t*>(cs + (r9 ^ xs) * kSliceBytes + 4 * gq);
      uint32_t s01, s89;
      if constexpr (kMx) {  // E8M0 group of channels 8 gq .. 8 gq + 7 of slice `warp`
        const int gi = 2 * warp + (gq >> 2);
        const int eb = t * kTile + t0;
        s01 = mx_factor_f16(sm.mxs[eb][gi], mx_ref) |
              (mx_factor_f16(sm.mxs[eb + 1][gi], mx_ref) << 16);
        s89 = mx_factor_f16(sm.mxs[eb + 8][gi], mx_ref) |
              (mx_factor_f16(sm.mxs[eb + 9][gi], mx_ref) << 16);
      } else {
        const int sg = gq >> 1;  // scale group of this thread's channels 8 gq .. 8 gq + 7
        s01 = e4m3x2_to_f16x2(ss[r0 * 16 + sg] | ((uint32_t)ss[r1 * 16 + sg] << 8));
        s89 = e4m3x2_to_f16x2(ss[r8 * 16 + sg] | ((uint32_t)ss[r9 * 16 + sg] << 8));
      }
      // byte p of lo: the even channel of code byte 4 gq + p for the two tokens (first
      // token in the low nibble); hi: the odd channel
      const uint32_t lo01 = (x0 & 0x0F0F0F0Fu) | ((x1 << 4) & 0xF0F0F0F0u);
      const uint32_t hi01 = ((x0 >> 4) & 0x0F0F0F0Fu) | (x1 & 0xF0F0F0F0u);
      const uint32_t lo89 = (x8 & 0x0F0F0F0Fu) | ((x9 << 4) & 0xF0F0F0F0u);
      const uint32_t hi89 = ((x8 >> 4) & 0x0F0F0F0Fu) | (x9 & 0xF0F0F0F0u);
      uint32_t L01[4], H01[4], L89[4], H89[4];
      e2m1x4_unpack(lo01, L01[0], L01[1], L01[2], L01[3]);
      e2m1x4_unpack(hi01, H01[0], H01[1], H01[2], H01[3]);
      e2m1x4_unpack(lo89, L89[0], L89[1], L89[2], L89[3]);
      e2m1x4_unpack(hi89, H89[0], H89[1], H89[2], H89[3]);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        mma16816(oacc[2 * p], a, hmul2(L01[p], s01), hmul2(L89[p], s89));
        mma16816(oacc[2 * p + 1], a, hmul2(H01[p], s01), hmul2(H89[p], s89));
      }
    }
  }
  cp_async_wait<0>();  // only empty groups remain; drained before the stages are reused
  __syncthreads();     // every warp is done with the partials and P

  // ---- epilogue: stage the 16 x 512 output through shared memory ----
  // n-tile 2 p + hb, column c <-> channel 64 warp + 8 c + 2 p + hb
  float* ob = &sm.red[0][0][0];
  if constexpr (kMx) {  // back to absolute scale: x 2^(ref - 127), exact
    const float fo = pow2f_attn(mx_ref - 127);
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) oacc[n][c] *= fo;
  }
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int ch = warp * kSliceCh + 16 * iq + 2 * (n >> 1) + (n & 1);
    ob[gq * kOStride + ch] = oacc[n][0];
    ob[gq * kOStride + ch + 8] = oacc[n][1];
    ob[(gq + 8) * kOStride + ch] = oacc[n][2];
    ob[(gq + 8) * kOStride + ch + 8] = oacc[n][3];
  }
  if (sk == 0) {
    sm.m_fin[sh_h] = m_ref;
    sm.l_fin[sh_h] = l_run;
  }
  __syncthreads();
  if (nsplit == 1) {
    float* obase = out + (int64_t)qi * kHq * kDkv;
    for (int f = tid; f < kHq * kDkv / 4; f += kAttnThreads) {
      const int h = f / (kDkv / 4), c4 = f % (kDkv / 4);
      const float l = sm.l_fin[h];
      float4 v = *reinterpret_cast<const float4*>(ob + h * kOStride + 4 * c4);
      if (l > 0.0f) {
        v.x /= l; v.y /= l; v.z /= l; v.w /= l;
      } else {
        v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      reinterpret_cast<float4*>(obase + h * kDkv)[c4] = v;
    }
    if (lse != nullptr && tid < kHq) {
      const float l = sm.l_fin[tid];
      lse[(int64_t)qi * kHq + tid] = l > 0.0f ? sm.m_fin[tid] * 0.6931471805599453f + logf(l) : -INFINITY;
    }
  } else {
    float* obase = part_o + ((int64_t)qi * nsplit + split) * kHq * kDkv;
    for (int f = tid; f < kHq * kDkv / 4; f += kAttnThreads) {
      const int h = f / (kDkv / 4), c4 = f % (kDkv / 4);
      reinterpret_cast<float4*>(obase + h * kDkv)[c4] =
          *reinterpret_cast<const float4*>(ob + h * kOStride + 4 * c4);
    }
    if (tid < kHq) {
      float* ml = part_ml + ((int64_t)qi * nsplit + split) * 2 * kHq;
      ml[tid] = sm.m_fin[tid];
      ml[kHq + tid] = sm.l_fin[tid];
    }
  }
}

// Merge the splits of each (query, head): out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// The partials are laid out with `stride` splits per query.  With `span_count` (the
// multi-query form), only the first ceil(span_count[query / chunk] / span_len) splits hold
// partials; none gives zero output and -inf lse.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           int stride, float* __restrict__ out,
                                                           float* __restrict__ lse,
                                                           const int32_t* __restrict__ span_count,
                                                           int span_len, int chunk) {
  grid_dep_wait();
  const int qi = blockIdx.x, h = blockIdx.y;
  const int nsplit = span_count == nullptr
                         ? stride
                         : min(stride, (__ldg(span_count + qi / chunk) + span_len - 1) / span_len);
  __shared__ float wgt[kMaxSplits];
  __shared__ float inv;
  const float* ml = part_ml + (int64_t)qi * stride * 2 * kHq;
  // 128 threads x 4 channels; the first four splits' rows are loaded before the weights
  // are known, so their latency overlaps the weights' reductions
  const float4* po = reinterpret_cast<const float4*>(part_o + ((int64_t)qi * stride * kHq + h) * kDkv);
  float4 v0[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (u < nsplit) v0[u] = __ldcs(po + (int64_t)u * kHq * kDkv / 4 + threadIdx.x);
  if (nsplit <= 4) {
    // every thread takes the (at most four) weights itself: no barrier, no shared memory;
    // the normaliser is summed in the order of the warp reduction below, (0 + 2) + (1 + 3)
    float m[4], l[4], w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m[u] = u < nsplit ? __ldg(ml + u * 2 * kHq + h) : -INFINITY;
      l[u] = u < nsplit ? __ldg(ml + u * 2 * kHq + kHq + h) : 0.f;
    }
    const float M = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = (m[u] == -INFINITY) ? 0.f : exp2f(m[u] - M);
    const float L = (w[0] * l[0] + w[2] * l[2]) + (w[1] * l[1] + w[3] * l[3]);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u < nsplit) {
        a.x += w[u] * v0[u].x;
        a.y += w[u] * v0[u].y;
        a.z += w[u] * v0[u].z;
        a.w += w[u] * v0[u].w;
      }
    }
    const float iv = L > 0.f ? 1.0f / L : 0.f;
    if (threadIdx.x == 0 && lse) lse[(int64_t)qi * kHq + h] = L > 0.f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
    reinterpret_cast<float4*>(out + ((int64_t)qi * kHq + h) * kDkv)[threadIdx.x] =
        make_float4(a.x * iv, a.y * iv, a.z * iv, a.w * iv);
    return;
  }
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int s = threadIdx.x; s < nsplit; s += 32) M = fmaxf(M, ml[s * 2 * kHq + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int s = threadIdx.x; s < nsplit; s += 32) {
      const float m = ml[s * 2 * kHq + h], l = ml[s * 2 * kHq + kHq + h];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      wgt[s] = w;
      L += w * l;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (threadIdx.x == 0) {
      inv = L > 0.f ? 1.0f / L : 0.f;
      if (lse) lse[(int64_t)qi * kHq + h] = L > 0.f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
    }
  }
  __syncthreads();
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (u < nsplit) {
      const float w = wgt[u];
      a.x += w * v0[u].x;
      a.y += w * v0[u].y;
      a.z += w * v0[u].z;
      a.w += w * v0[u].w;
    }
  }
  int s = min(nsplit, 4);
  for (; s + 4 <= nsplit; s += 4) {  // four independent loads in flight
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcs(po + (int64_t)(s + u) * kHq * kDkv / 4 + threadIdx.x);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = wgt[s + u];
      a.x += w * v[u].x;
      a.y += w * v[u].y;
      a.z += w * v[u].z;
      a.w += w * v[u].w;
    }
  }
  for (; s < nsplit; ++s) {
    const float w = wgt[s];
    const float4 v = __ldcs(po + (int64_t)s * kHq * kDkv / 4 + threadIdx.x);
    a.x += w * v.x;
    a.y += w * v.y;
    a.z += w * v.z;
    a.w += w * v.w;
  }
  const float iv = inv;
  reinterpret_cast<float4*>(out + ((int64_t)qi * kHq + h) * kDkv)[threadIdx.x] =
      make_float4(a.x * iv, a.y * iv, a.z * iv, a.w * iv);
}

// Splits per query: the count that minimises (waves of kAttnCtasPerSm CTAs per SM) x
// (tiles per CTA + a fixed start-up cost of ~2 tiles), with at most kMaxSplit entries
// per CTA.
int attn_splits(int32_t num_q, int32_t topk, int num_sms) {
  const int tiles = std::max(1, (topk + kTile - 1) / kTile);
  const int min_splits = (tiles * kTile + kMaxSplit - 1) / kMaxSplit;
  const int max_splits = std::max(min_splits, std::min(64, tiles));
  int best = std::max(1, min_splits);
  double best_cost = 1e300;
  for (int sp = std::max(1, min_splits); sp <= max_splits; ++sp) {
    const int per = (tiles + sp - 1) / sp;     // tiles per split
    const int real = (tiles + per - 1) / per;  // splits actually used
    const int64_t ctas = (int64_t)num_q * real;
    const int64_t slots = (int64_t)num_sms * kAttnCtasPerSm;
    const int64_t waves = (ctas + slots - 1) / slots;
    const double cost = (double)waves * (per + 2);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = real;
    }
  }
  return best;
}

int attn_split_len(int32_t topk, int splits) {
  const int tiles = std::max(1, (topk + kTile - 1) / kTile);
  const int per = (tiles + splits - 1) / splits;
  return per * kTile;
}

size_t attn_smem_bytes(bool mx) { return mx ? sizeof(AttnSmemT<true>) : sizeof(AttnSmemT<false>); }

cudaError_t launch_attn_nvf4(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                             const int32_t* idx, const csa2_pages& pg, float* out, float* lse,
                             int32_t num_q, const int32_t* q_seq, int32_t topk, float softmax_scale,
                             void* ws, int32_t* st, cudaStream_t s, int num_sms);
size_t attn_nvf4_workspace_bytes(int32_t num_q, int32_t topk, int num_sms);

// The E4M3 / 16 cache takes the block-scaled FP4 tensor-core path (attn_nvf4.cu); the
// MXFP4 variant runs sparse_attn_kernel<true> above.
cudaError_t launch_attn(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                        const int32_t* idx, const csa2_pages& pg, float* out, float* lse,
                        int32_t num_q, const int32_t* q_seq, int32_t topk, float softmax_scale,
                        void* ws, int32_t* st, cudaStream_t s, int num_sms, bool mx) {
  if (!mx)
    return launch_attn_nvf4(q, codes, scales, idx, pg, out, lse, num_q, q_seq, topk, softmax_scale, ws,
                            st, s, num_sms);
  AttnGeom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  int splits = attn_splits(num_q, topk, num_sms);
  const int split_len = attn_split_len(topk, splits);
  splits = (topk + split_len - 1) / split_len;
  if (splits < 1) splits = 1;
  const size_t smem = attn_smem_bytes(true);
  auto kern = sparse_attn_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  float* part_o = reinterpret_cast<float*>(ws);
  float* part_ml = part_o + (int64_t)num_q * splits * kHq * kDkv;
  dim3 grid(splits, num_q);
  e = launch_pdl(kern, grid, dim3(kAttnThreads), smem, s, q, codes, scales, idx, g, q_seq, topk,
                 split_len, softmax_scale, out, lse, part_o, part_ml, st);
  if (e != cudaSuccess) return e;
  if (splits > 1)
    e = launch_pdl(attn_combine_kernel, dim3(num_q, kHq), dim3(128), 0, s, (const float*)part_o,
                   (const float*)part_ml, splits, out, lse, (const int32_t*)nullptr, 1, 1);
  return e;
}

cudaError_t launch_attn_combine(const float* part_o, const float* part_ml, int nsplit,
                                int32_t num_q, float* out, float* lse, const int32_t* span_count,
                                int32_t span_len, int32_t chunk, cudaStream_t s) {
  if (nsplit > kMaxSplits) return cudaErrorInvalidValue;
  return launch_pdl(attn_combine_kernel, dim3(num_q, kHq), dim3(128), 0, s, part_o, part_ml, nsplit,
                    out, lse, span_count, (int)span_len, (int)chunk);
}

// Workspace of either scale format (the larger of the two paths' needs).
size_t attn_workspace_bytes(int32_t num_q, int32_t topk, int num_sms) {
  int splits = attn_splits(num_q, topk, num_sms);
  const int split_len = attn_split_len(topk, splits);
  splits = (topk + split_len - 1) / split_len;
  const size_t mx = splits <= 1 ? 0 : (size_t)num_q * splits * (kHq * kDkv + 2 * kHq) * sizeof(float);
  return std::max(mx, attn_nvf4_workspace_bytes(num_q, topk, num_sms));
}

}  // namespace csa2
