// Gather-dequantise sparse attention over the E4M3 / 16 cache, with the logits on the
// block-scaled FP4 tensor cores.
//
// zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮": the main KV is FP4 E2M1
// with one E4M3 scale per 16 channels, dequantised before attention; tech-report digest
// (jiwasawa.github.io), "Reuse Mode": sparse attention over the top-K entries.  MQA over
// the shared latent: K = V = c_hat (512 channels), 16 query heads.
//
// The cache's own encoding -- E2M1 codes with an unsigned E4M3 scale per 16 channels -- is
// the operand format of tcgen05.mma kind::mxf4nvf4 (scale_vec::4X), so the logits
// S[t][h] = sum_c c_hat[t][c] q[h][c] are taken straight from the gathered code rows
// without dequantising them:
//   - q (bf16) is written as a sum of kTerms NVFP4 terms, q ~= sum_k 2^-p_k T_k with T_k
//     = E2M1 codes x UE4M3 scale per 16 channels, each term encoding the residual of the
//     previous ones (scale rounded up, so no code saturates; p_k = p_0 + 2 k keeps every
//     scale in range).  Each term shrinks the residual by at least 16/3, so six terms
//     leave |q - sum| <= (3/16)^6 (about 4e-5) of the block maximum; the terms are made
//     once per query by q_terms_kernel;
//   - one MMA per 64 channels, M = 128 tokens x N = 96 (term, head) rows, A = the gathered
//     codes (128-byte swizzled, K-major), B = the terms, scale factors in TMEM, fp32
//     accumulators in TMEM; the softmax weights the six term columns by 2^-p_k.
// The weighted sum O = P . c_hat contracts over tokens, across the scale groups, so it
// runs on mma.sync with each code dequantised once into operand registers (E2M1 x E4M3 is
// exact in f16): 16 heads x 8 channels x 16 tokens per instruction, once with the hi part
// of P and once with the lo part on the same operand registers.  One f16 part per weight
// (11 significant bits) leaves output errors of the order of the 2e-3 x RMS accuracy bound
// on a fraction of queries; hi + lo carry 22 bits.
//
// Work division: one CTA per (query, split of its selected entries, at most 512), two CTAs
// per SM; splits are merged by attn_combine_kernel (log-sum-exp).
#include <algorithm>
#include <cstddef>

#include "async.cuh"

namespace csa2 {
namespace nvf4 {

constexpr int kTerms = 6;
constexpr int kRows = kTerms * kHq;          // 96 B-operand rows: (term, head)
constexpr int kTile = 128;                   // tokens per tile = MMA M
constexpr int kThreads = 256;                // 8 warps; two CTAs per SM
constexpr int kMaxSplit = 512;               // selected entries per CTA at most (4 tiles)
constexpr int kChunk = kTile * 128;          // one 128-byte-swizzled K-chunk of a tile's codes
constexpr int kStageCodes = 2 * kChunk;      // 32 KB
constexpr int kStageBytes = kStageCodes + kTile * kScaleRow;  // + token-major scale rows: 36 KB
constexpr int kQbChunk = kRows * 128;        // 12 KB
constexpr int kQbBytes = 2 * kQbChunk;       // 24 KB
constexpr int kSfbBytes = 4096;              // B scale-factor image
constexpr int kTermsP0 = kQbBytes + kSfbBytes;  // offset of p_0 in a query's term image
constexpr size_t kTermsBytes = 28928;        // per query: codes image, SFB image, p_0 (256-B multiple)
static_assert(kTermsP0 + 16 <= (int)kTermsBytes && kTermsBytes % 256 == 0, "term image layout");
constexpr uint32_t kColS = 0;                // S^T: columns 0 .. 95
constexpr uint32_t kColSfa = 128;            // A scale factors: 32 columns
constexpr uint32_t kColSfb = 160;            // B scale factors: 32 columns
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleGap = 8.0f;          // log2 units
constexpr int kPRow = 2 * kTile + 16;        // bytes per head row of P: padded so that ldmatrix is conflict-free

struct Smem {
  unsigned char stage[2][kStageBytes];       // codes (2 swizzled chunks) + scale rows [128][32]
  unsigned char qb[kQbBytes];                // B operand: the query's terms
  unsigned char sfb[kSfbBytes];              // their scale-factor image
  int32_t p0[4];
  unsigned char p[2][kHq * kPRow];           // P as f16 hi + lo parts, [head][token] with padded rows
  int32_t slot[kMaxSplit];                   // physical row of each selected entry, -1 if skipped
  float alpha[kHq];
  float m_fin[kHq], l_fin[kHq];
  float red[8][8];
  uint64_t s_full, t_full, fin;
  uint32_t tmem;
  volatile int abort;
};
static_assert(offsetof(Smem, qb) % 1024 == 0 && kStageBytes % 1024 == 0 && kQbChunk % 1024 == 0,
              "swizzled operands need 1024-byte alignment");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");

struct Geom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t max_pages;
  int32_t num_pages;
  int32_t num_seqs;
};

// ---------------------------------------------------------------- PTX helpers ------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;               // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;     // stride byte offset: next group of 8 rows
  d |= (uint64_t)1 << 46;               // descriptor version
  d |= (uint64_t)2 << 61;               // 128-byte swizzle
  return d;
}
// kind::mxf4nvf4: A and B E2M1 (format 1), UE4M3 scale factors (format bit 0), K-major,
// M = 128, N = 96, dense K = 64.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kRows >> 3) << 17) | ((uint32_t)(kTile >> 4) << 24);

__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t ta, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by MUFU ex2 (flushes subnormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(two & 0xFFFFu)));
  return h2;
}
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
__device__ __forceinline__ float pow2i(int k) {  // 2^k, k in [-126, 127]
  return __uint_as_float((uint32_t)(k + 127) << 23);
}
// Bounded wait that ignores the abort flag (used to drain before TMEM is freed).
__device__ __forceinline__ bool mbar_drain(uint64_t* b, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 22); ++i)
    if (mbar_try(b, parity)) return true;
  return false;
}

// ------------------------------------------------------------ query terms ----------
// One CTA (512 threads) per query: thread (h, g) encodes the 16 channels 16 g .. 16 g + 15
// of head h as kTerms NVFP4 terms into the query's term image:
//   codes  [2 chunks][96 rows][128 B], 128-byte swizzled (row = 16 k + h), the MMA's B operand
//   sfb    [8 K-steps][32 lanes][4 words]: word c of (ks, lane) holds the scale bytes of row
//          lane + 32 c for the four 16-channel blocks of K-step ks -- the image that
//          tcgen05.cp (32x128b, replicated to the four lane quarters) copies into the TMEM
//          scale-factor columns 4 ks .. 4 ks + 3; rows 96..127 are zero
//   p_0    int32: term k carries the factor 2^-(p_0 + 2 k)
// Each term's residual is taken from the codes actually chosen, so the reciprocal and the
// rounding used to choose them need not be exact: the bound on what remains holds either way.
__global__ void __launch_bounds__(512) q_terms_kernel(const uint16_t* __restrict__ q,
                                                      unsigned char* __restrict__ terms) {
  grid_dep_wait();
  grid_dep_launch();  // the attention CTAs allocate TMEM and set up while the terms are made
  __shared__ uint32_t wmax[16];
  const int qi = blockIdx.x, tid = threadIdx.x, h = tid >> 5, g = tid & 31;
  unsigned char* img = terms + (size_t)qi * kTermsBytes;
  const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)qi * kHq + h) * kDkv + 16 * g);
  const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float r[16];
  uint32_t mb = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    r[2 * i] = bf16lo(w[i]);
    r[2 * i + 1] = bf16hi(w[i]);
    mb = max(mb, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  }
  mb = __reduce_max_sync(0xffffffffu, mb);
  if ((tid & 31) == 0) wmax[tid >> 5] = mb;
  // zero the words of rows 96..127 (c = 3)
  if (tid < 256) reinterpret_cast<uint32_t*>(img + kQbBytes)[((tid & 7) * 32 + (tid >> 3)) * 4 + 3] = 0u;
  __syncthreads();
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = max(m, wmax[i]);
  // p_0: max |q| x 2^p_0 in [2^7, 2^8); all scales then stay below 2^8 / 6
  const int gexp = (int)(m >> 7) - 127;
  const int p0 = m == 0 ? 0 : max(-126, min(117, 7 - gexp));
  if (tid == 0) *reinterpret_cast<int32_t*>(img + kTermsP0) = p0;
#pragma unroll
  for (int k = 0; k < kTerms; ++k) {
    const float f = pow2i(p0 + 2 * k), fi = pow2i(-(p0 + 2 * k));
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(r[i]));
    amax *= f;
    // smallest E4M3 scale s with amax / s <= 6 (no code saturates)
    const float target = amax * (1.0f / 6.0f);
    uint32_t sb = e4m3_encode(target);
    if (e4m3_decode(sb) < target && sb < 0x7Eu) ++sb;
    const float s = e4m3_decode(sb);
    uint32_t cw[2] = {0u, 0u};
    if (s > 0.0f) {
      const float inv = f * __frcp_rn(s);  // y / s = r * f / s
      const float back = s * fi;           // code value -> residual units
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint16_t b16;
        asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
            : "=h"(b16)
            : "f"(r[2 * j + 1] * inv), "f"(r[2 * j] * inv));
        const uint32_t b = b16 & 0xFFu;
        cw[j >> 2] |= b << (8 * (j & 3));
        const uint32_t hv = e2m1x2_to_f16x2(b);
        const __half2 hh = *reinterpret_cast<const __half2*>(&hv);
        const float2 fv = __half22float2(hh);
        r[2 * j] = fmaf(-fv.x, back, r[2 * j]);
        r[2 * j + 1] = fmaf(-fv.y, back, r[2 * j + 1]);
      }
    }
    const int row = 16 * k + h;
    const int chunk = g >> 4, unit = (g & 15) >> 1;
    *reinterpret_cast<uint2*>(img + chunk * kQbChunk + row * 128 + ((unit ^ (row & 7)) << 4) +
                              8 * (g & 1)) = make_uint2(cw[0], cw[1]);
    const int lane = row & 31, c = row >> 5, ks = g >> 2, kb = g & 3;
    img[kQbBytes + (((ks * 32 + lane) * 4 + c) << 2) + kb] = (unsigned char)sb;
  }
}

// ------------------------------------------------------------ attention ------------

// 1D bulk copy global -> shared, completion counted on `bar` (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(saddr(bar))
               : "memory");
}
// Descriptor of a 32-row x 16-byte scale-factor block (8-row core matrices 128 B apart, no swizzle).
__device__ __forceinline__ uint64_t desc_sf(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// Copy one 32 x 16-byte block into 4 TMEM columns of every lane quarter.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t ta, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(ta));
}

// One CTA per (query, split of its selected entries), tiles of 128 entries, every warp
// taking part in every phase; two CTAs per SM interleave, so one CTA's weighted sum runs
// while the other gathers, waits for its logits or runs its softmax.
//   gather:   cp.async, 16 lanes per 256-byte code row (stored 128-byte swizzled, the MMA's
//             A layout) and two per 32-byte scale row; a 2-stage ring one tile ahead;
//   logits:   warps 0-3 write the tile's scale factors into TMEM (each its lane quarter),
//             one thread issues the 8 block-scaled MMAs (K = 512);
//   softmax:  thread (w, l) takes token 32 (w % 4) + l and heads 8 (w / 4) .. + 7: the six
//             term columns weighted by 2^-p_k, fp32 in the exp2 domain with a lazily moved
//             reference max (it moves, and the output is rescaled, only when a logit exceeds
//             it by more than 2^8); P stored as hi = f16(p) and lo = f16(p - hi), the
//             normaliser summed from p in fp32;
//   O += P . c_hat: warp w owns channels 64 w .. + 63 (mma.sync m16n8k16, codes dequantised
//             once into operand registers, hi and lo parts of P on the same operands).
__global__ void __launch_bounds__(kThreads, 2)
    attn_nvf4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                     const int32_t* __restrict__ idx, Geom geo, const int32_t* __restrict__ q_seq,
                     int32_t topk, int32_t split_len, float kq, const unsigned char* __restrict__ terms,
                     float* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
                     float* __restrict__ part_ml, int32_t* st) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qi = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
  const int jbeg = split * split_len;
  const int ecount = max(0, min(topk, jbeg + split_len) - jbeg);
  const int ntiles = (ecount + kTile - 1) / kTile;

  if (tid == 0) {
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.t_full, 1);
    mbar_init(&sm.fin, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&sm.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // ---- resolve the selected entries to physical rows, and gather the first tile ----
  // Done before the dependency wait, so that it overlaps the term kernel: the indices, the
  // page table and the cache are inputs of this call, and every kernel before the term
  // kernel in the stream has completed by now (the term kernel lets this one launch only
  // after its own dependency wait).  Nothing global is written before the wait.
  int b = __ldg(q_seq + qi);
  int n_ctx = 0;
  if (b < 0 || b >= geo.num_seqs) {
    if (tid == 0) report(st, CSA2_DEV_BAD_QSEQ);
    b = 0;
  } else {
    n_ctx = min(max(0, __ldg(geo.seq_lens + b)), geo.max_pages * kPage);
  }
  const int32_t* idx_q = idx + (int64_t)qi * topk + jbeg;
  constexpr int kPer = kMaxSplit / kThreads;  // entries resolved per thread
  static_assert(kMaxSplit % kThreads == 0, "whole entries per thread");
  {
    int32_t s_of[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      s_of[i] = e < ecount ? __ldg(idx_q + e) : -1;
    }
    int32_t pg_of[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int32_t s = s_of[i];
      pg_of[i] = (s >= 0 && s < n_ctx) ? __ldg(geo.page_table + (int64_t)b * geo.max_pages + (s >> 6)) : -1;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      if (e >= ecount) continue;
      const int32_t s = s_of[i], pg = pg_of[i];
      int32_t slot = -1;
      if (s >= 0 && s < n_ctx) {
        if (pg >= 0 && pg < geo.num_pages) slot = pg * kPage + (s & (kPage - 1));
        else report(st, CSA2_DEV_BAD_PAGE);
      } else if (s != -1) {
        report(st, CSA2_DEV_BAD_INDEX);
      }
      sm.slot[e] = slot;
    }
  }
  tc_before();
  __syncthreads();  // barriers, TMEM address and every slot visible
  tc_after();
  const uint32_t tmem = sm.tmem;

  // gather tile t (entries t * 128 ..): codes by half-warps (16 pieces of a 256-byte row),
  // scales two pieces per row; every slot is read before any copy
  auto gather = [&](int t) {
    const uint32_t stg = saddr(sm.stage[t & 1]);
    const int e0 = t * kTile;
    const int piece = lane & 15, hi = lane >> 4;
    int32_t rs[4], ss;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = e0 + 16 * k + 2 * warp + hi;  // rows 16 k + 2 w + hi
      rs[k] = e < ecount ? sm.slot[e] : -1;
    }
    {
      const int e = e0 + (tid >> 1);
      ss = e < ecount ? sm.slot[e] : -1;
    }
    const uint32_t cbase = stg + (piece >> 3) * kChunk;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = 16 * k + 2 * warp + hi;
      cp_async16(cbase + row * 128 + (((piece & 7) ^ (row & 7)) << 4),
                 codes + (rs[k] >= 0 ? (int64_t)rs[k] * kCodeRow : 0) + 16 * piece, rs[k] >= 0);
    }
#pragma unroll
    for (int k = 4; k < 8; ++k) {
      const int row = 16 * k + 2 * warp + hi;
      const int e = e0 + row;
      const int32_t r = e < ecount ? sm.slot[e] : -1;
      cp_async16(cbase + row * 128 + (((piece & 7) ^ (row & 7)) << 4),
                 codes + (r >= 0 ? (int64_t)r * kCodeRow : 0) + 16 * piece, r >= 0);
    }
    const int srow = tid >> 1, pc = tid & 1;
    cp_async16(stg + kStageCodes + srow * kScaleRow + 16 * pc,
               scales + (ss >= 0 ? (int64_t)ss * kScaleRow : 0) + 16 * pc, ss >= 0);
  };
  if (ntiles > 0) gather(0);
  cp_commit();

  grid_dep_wait();  // the term kernel's output is read from here on
  // ---- the query's terms (B operand, its scale-factor image, p_0) ----
  if (tid == 0) {
    const unsigned char* img = terms + (size_t)qi * kTermsBytes;
    mbar_expect_tx(&sm.t_full, kQbBytes + kSfbBytes + 16);
    bulk_g2s(saddr(sm.qb), img, kQbBytes, &sm.t_full);
    bulk_g2s(saddr(sm.sfb), img + kQbBytes, kSfbBytes, &sm.t_full);
    bulk_g2s(saddr(&sm.p0[0]), img + kTermsP0, 16, &sm.t_full);
  }
  // B scale factors into TMEM once the terms have landed
  bool ok = mbar_wait(&sm.abort, &sm.t_full, 0, st);
  if (tid == 0 && ok) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) tmem_cp_sf(tmem + kColSfb + 4 * ks, desc_sf(saddr(sm.sfb) + 512 * ks));
  }
  float wt[kTerms];
  {
    const int p0 = sm.p0[0];
#pragma unroll
    for (int k = 0; k < kTerms; ++k) wt[k] = kq * pow2i(max(-126, -(p0 + 2 * k)));
  }

  // softmax ownership: token 32 (w % 4) + lane, heads hb .. hb + 7
  const int tok = 32 * (warp & 3) + lane, hb = 8 * (warp >> 2);
  const uint32_t qlane = (uint32_t)(32 * (warp & 3)) << 16;
  float m_ref[8], lp[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    m_ref[h] = -INFINITY;
    lp[h] = 0.0f;
  }
  // weighted-sum ownership (see the output-phase comment below)
  const int gq = lane >> 2, iq = lane & 3;
  const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lhi = lane >> 4;
  const int unit0 = 2 * (warp & 3) + (gq >> 2), boff = (4 * gq) & 15;
  const uint32_t off_e = (warp >> 2) * kChunk + 256 * iq + ((unit0 ^ (2 * iq)) << 4) + boff;
  const uint32_t off_o = (warp >> 2) * kChunk + 256 * iq + 128 + ((unit0 ^ (2 * iq + 1)) << 4) + boff;
  const uint32_t off_s = kStageCodes + 64 * iq + 4 * warp + (gq >> 1);
  const uint32_t off_p = lrow * kPRow + 16 * lhi;
  float oacc[8][4];
#pragma unroll
  for (int x = 0; x < 8; ++x) oacc[x][0] = oacc[x][1] = oacc[x][2] = oacc[x][3] = 0.0f;
  bool mma_issued = false;

  // Every thread runs every iteration and every barrier, whatever its waits returned: a
  // wait that expires raises sm.abort, after which the other waits return at once and no
  // further MMA is issued.
  for (int t = 0; t < ntiles; ++t) {
    cp_wait<0>();     // this thread's copies of tile t have landed
    __syncthreads();  // everyone's; and the weighted sum of tile t - 1 is done with its stage
    // ---- logits: scale factors of tile t into TMEM, then the MMAs ----
    if (warp < 4) {
      const unsigned char* sc = sm.stage[t & 1] + kStageCodes;
      uint32_t r[32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint4 a = *reinterpret_cast<const uint4*>(sc + (lane + 32 * cc) * kScaleRow);
        const uint4 bb = *reinterpret_cast<const uint4*>(sc + (lane + 32 * cc) * kScaleRow + 16);
        r[0 + cc] = a.x; r[4 + cc] = a.y; r[8 + cc] = a.z; r[12 + cc] = a.w;
        r[16 + cc] = bb.x; r[20 + cc] = bb.y; r[24 + cc] = bb.z; r[28 + cc] = bb.w;
      }
      tmem_st32(tmem + qlane + kColSfa, r);
      tmem_wait_st();
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    if (tid == 0 && !sm.abort) {
      tc_after();
      const uint32_t a0 = saddr(sm.stage[t & 1]), b0 = saddr(sm.qb);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_nvf4(tmem + kColS, desc_sw128(a0 + (ks >> 2) * kChunk) + 2 * (ks & 3),
                 desc_sw128(b0 + (ks >> 2) * kQbChunk) + 2 * (ks & 3), tmem + kColSfa + 4 * ks,
                 tmem + kColSfb + 4 * ks, ks > 0 ? 1u : 0u);
      mma_commit(&sm.s_full);
      mma_issued = true;
    }
    // the next tile's gather is issued while the MMAs run (the other stage is free: the
    // weighted sum of tile t - 1 finished before the barrier at the top)
    if (t + 1 < ntiles) gather(t + 1);
    cp_commit();
    ok &= mbar_wait(&sm.abort, &sm.s_full, (uint32_t)(t & 1), st);
    tc_after();
    // ---- softmax of token tok, heads hb .. hb + 7 ----
    float z[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) z[h] = 0.0f;
#pragma unroll
    for (int k = 0; k < kTerms; ++k) {
      uint32_t d[8];
      tmem_ld8(tmem + qlane + kColS + 16 * k + hb, d);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 8; ++h) z[h] = fmaf(wt[k], __uint_as_float(d[h]), z[h]);
    }
    const int e = t * kTile + tok;
    const bool valid = e < ecount && sm.slot[e] >= 0;
    bool exceed = false;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      z[h] = valid ? z[h] : -INFINITY;
      exceed |= z[h] > m_ref[h] + kRescaleGap;
    }
    tc_before();
    const bool rescale = __syncthreads_or(exceed) != 0;
    if (rescale) {
      // tile max of each head: butterfly over the warp, then over the warps of the head half
      float v[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        v[h] = z[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[h] = fmaxf(v[h], __shfl_xor_sync(0xffffffffu, v[h], o));
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < 8; ++h) sm.red[warp][h] = v[h];
      }
      __syncthreads();
      const int w0 = 4 * (warp >> 2);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float mt = fmaxf(fmaxf(sm.red[w0][h], sm.red[w0 + 1][h]), fmaxf(sm.red[w0 + 2][h], sm.red[w0 + 3][h]));
        const float mu = m_ref[h];
        float mn = mu;
        if (mu == -INFINITY || mt > mu + kRescaleGap) mn = fmaxf(mu, mt);
        const float al = (mn != mu) ? ex2(mu - mn) : 1.0f;
        m_ref[h] = mn;
        lp[h] *= al;
        if (warp < 8 && (warp & 3) == 0 && lane == 0) sm.alpha[hb + h] = al;
      }
    }
    // P hi / lo of token tok for heads hb .. hb + 7
    unsigned char* pb = sm.p[0] + 2 * tok;
    unsigned char* pl = sm.p[1] + 2 * tok;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float mh = m_ref[h] == -INFINITY ? 0.0f : m_ref[h];
      const float pv = ex2(z[h] - mh);
      const __half ph = __float2half_rn(pv);
      const __half plo = __float2half_rn(pv - __half2float(ph));
      lp[h] += pv;
      *reinterpret_cast<__half*>(pb + (hb + h) * kPRow) = ph;
      *reinterpret_cast<__half*>(pl + (hb + h) * kPRow) = plo;
    }
    __syncthreads();  // P (and alpha) complete
    // ---- O += P . c_hat ----
    // Thread (gq, iq) of warp w: heads gq and gq + 8, channels 64 w + 16 iq + x and + 8
    // (x = 0..7); per 16-token k-step it reads tile rows 16 ks + 2 iq + {0, 1, 8, 9} at 4
    // code bytes 4 gq .. of the warp's 32-byte slice, whose swizzled offsets are fixed per
    // thread (the row index modulo 8 does not depend on ks), and their scale bytes of group
    // 4 w + gq / 2.
    if (rescale) {
      const float a_lo = sm.alpha[gq], a_hi = sm.alpha[gq + 8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        oacc[x][0] *= a_lo;
        oacc[x][1] *= a_lo;
        oacc[x][2] *= a_hi;
        oacc[x][3] *= a_hi;
      }
    }
    const unsigned char* stg = sm.stage[t & 1];
    const uint32_t pbs = saddr(sm.p[0]) + off_p, pls = saddr(sm.p[1]) + off_p;
#pragma unroll
    for (int ks = 0; ks < kTile / 16; ++ks) {
      uint32_t a[4], al[4];
      ldmatrix_x4(a, pbs + 32 * ks);
      ldmatrix_x4(al, pls + 32 * ks);
      const uint32_t x0 = *reinterpret_cast<const uint32_t*>(stg + off_e + 2048 * ks);
      const uint32_t x1 = *reinterpret_cast<const uint32_t*>(stg + off_o + 2048 * ks);
      const uint32_t x8 = *reinterpret_cast<const uint32_t*>(stg + off_e + 2048 * ks + 1024);
      const uint32_t x9 = *reinterpret_cast<const uint32_t*>(stg + off_o + 2048 * ks + 1024);
      const unsigned char* sp = stg + off_s + 512 * ks;
      const uint32_t s01 = e4m3x2_to_f16x2(sp[0] | ((uint32_t)sp[32] << 8));
      const uint32_t s89 = e4m3x2_to_f16x2(sp[256] | ((uint32_t)sp[288] << 8));
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
        const uint32_t bl0 = hmul2(L01[p], s01), bl1 = hmul2(L89[p], s89);
        const uint32_t bh0 = hmul2(H01[p], s01), bh1 = hmul2(H89[p], s89);
        mma16816(oacc[2 * p], a, bl0, bl1);
        mma16816(oacc[2 * p + 1], a, bh0, bh1);
        mma16816(oacc[2 * p], al, bl0, bl1);
        mma16816(oacc[2 * p + 1], al, bh0, bh1);
      }
    }
  }
  cp_wait<0>();
  // ---- normaliser and reference max of each head ----
#pragma unroll
  for (int h = 0; h < 8; ++h) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp[h] += __shfl_xor_sync(0xffffffffu, lp[h], o);
  }
  __syncthreads();  // sm.red free; every warp done with P and the stages
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < 8; ++h) sm.red[warp][h] = lp[h];
  }
  if ((warp & 3) == 0 && lane == 0) {
#pragma unroll
    for (int h = 0; h < 8; ++h) sm.m_fin[hb + h] = m_ref[h];
  }
  __syncthreads();
  if (tid < kHq) {
    const int w0 = 4 * (tid >> 3), h = tid & 7;
    sm.l_fin[tid] = (sm.red[w0][h] + sm.red[w0 + 1][h]) + (sm.red[w0 + 2][h] + sm.red[w0 + 3][h]);
  }
  __syncthreads();
  // ---- output: thread (gq, iq) holds heads gq, gq + 8 at channels 64 w + 16 iq + x
  // (x = 0..7) in oacc[x][0 / 2] and + 8 in oacc[x][1 / 3] ----
  const float m_lo = sm.m_fin[gq], m_hi = sm.m_fin[gq + 8];
  const float l_lo = sm.l_fin[gq], l_hi = sm.l_fin[gq + 8];
  const int ch = 64 * warp + 16 * iq;
  if (nsplit == 1) {
    const float il = l_lo > 0.0f ? 1.0f / l_lo : 0.0f, ih = l_hi > 0.0f ? 1.0f / l_hi : 0.0f;
    float* o_lo = out + ((int64_t)qi * kHq + gq) * kDkv + ch;
    float* o_hi = out + ((int64_t)qi * kHq + gq + 8) * kDkv + ch;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      reinterpret_cast<float4*>(o_lo)[u] = make_float4(oacc[4 * u][0] * il, oacc[4 * u + 1][0] * il, oacc[4 * u + 2][0] * il, oacc[4 * u + 3][0] * il);
      reinterpret_cast<float4*>(o_lo + 8)[u] = make_float4(oacc[4 * u][1] * il, oacc[4 * u + 1][1] * il, oacc[4 * u + 2][1] * il, oacc[4 * u + 3][1] * il);
      reinterpret_cast<float4*>(o_hi)[u] = make_float4(oacc[4 * u][2] * ih, oacc[4 * u + 1][2] * ih, oacc[4 * u + 2][2] * ih, oacc[4 * u + 3][2] * ih);
      reinterpret_cast<float4*>(o_hi + 8)[u] = make_float4(oacc[4 * u][3] * ih, oacc[4 * u + 1][3] * ih, oacc[4 * u + 2][3] * ih, oacc[4 * u + 3][3] * ih);
    }
    if (lse != nullptr && warp == 0 && iq == 0) {
      lse[(int64_t)qi * kHq + gq] = l_lo > 0.0f ? m_lo * 0.6931471805599453f + logf(l_lo) : -INFINITY;
      lse[(int64_t)qi * kHq + gq + 8] = l_hi > 0.0f ? m_hi * 0.6931471805599453f + logf(l_hi) : -INFINITY;
    }
  } else {
    const int64_t ps = (int64_t)qi * nsplit + split;
    float* o_lo = part_o + (ps * kHq + gq) * kDkv + ch;
    float* o_hi = part_o + (ps * kHq + gq + 8) * kDkv + ch;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      reinterpret_cast<float4*>(o_lo)[u] = make_float4(oacc[4 * u][0], oacc[4 * u + 1][0], oacc[4 * u + 2][0], oacc[4 * u + 3][0]);
      reinterpret_cast<float4*>(o_lo + 8)[u] = make_float4(oacc[4 * u][1], oacc[4 * u + 1][1], oacc[4 * u + 2][1], oacc[4 * u + 3][1]);
      reinterpret_cast<float4*>(o_hi)[u] = make_float4(oacc[4 * u][2], oacc[4 * u + 1][2], oacc[4 * u + 2][2], oacc[4 * u + 3][2]);
      reinterpret_cast<float4*>(o_hi + 8)[u] = make_float4(oacc[4 * u][3], oacc[4 * u + 1][3], oacc[4 * u + 2][3], oacc[4 * u + 3][3]);
    }
    if (warp == 0 && iq == 0) {
      float* ml = part_ml + ps * 2 * kHq;
      ml[gq] = m_lo;
      ml[gq + 8] = m_hi;
      ml[kHq + gq] = l_lo;
      ml[kHq + gq + 8] = l_hi;
    }
  }
  (void)ok;
  if (tid == 0 && mma_issued) {  // every MMA issued has completed before TMEM is freed
    mma_commit(&sm.fin);
    (void)mbar_drain(&sm.fin, 0);
  }
  tc_before();
  __syncthreads();
  if (warp == 0) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace nvf4

int attn_splits(int32_t num_q, int32_t topk, int num_sms);
int attn_split_len(int32_t topk, int splits);
cudaError_t launch_attn_combine(const float* part_o, const float* part_ml, int nsplit, int32_t num_q,
                                float* out, float* lse, const int32_t* span_count, int32_t span_len,
                                int32_t chunk, cudaStream_t s);

// Splits of the selected set: at most 512 entries (4 tiles) per CTA, as for the MXFP4 path.
static int nvf4_splits(int32_t num_q, int32_t topk, int num_sms, int* split_len) {
  int splits = attn_splits(num_q, topk, num_sms);
  *split_len = attn_split_len(topk, splits);
  splits = (topk + *split_len - 1) / *split_len;
  return splits < 1 ? 1 : splits;
}

size_t attn_nvf4_workspace_bytes(int32_t num_q, int32_t topk, int num_sms) {
  int split_len = 0;
  const int splits = nvf4_splits(num_q, topk, num_sms, &split_len);
  const size_t terms = (size_t)num_q * nvf4::kTermsBytes;
  const size_t parts = splits <= 1 ? 0 : (size_t)num_q * splits * (kHq * kDkv + 2 * kHq) * sizeof(float);
  return terms + parts;
}

cudaError_t launch_attn_nvf4(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                             const int32_t* idx, const csa2_pages& pg, float* out, float* lse,
                             int32_t num_q, const int32_t* q_seq, int32_t topk, float softmax_scale,
                             void* ws, int32_t* st, cudaStream_t s, int num_sms) {
  using namespace nvf4;
  int split_len = 0;
  const int splits = nvf4_splits(num_q, topk, num_sms, &split_len);
  unsigned char* terms = reinterpret_cast<unsigned char*>(ws);
  float* part_o = reinterpret_cast<float*>(terms + (size_t)num_q * kTermsBytes);
  float* part_ml = part_o + (size_t)num_q * splits * kHq * kDkv;
  cudaError_t e = launch_pdl(q_terms_kernel, dim3(num_q), dim3(512), 0, s, q, terms);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  Geom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  const float kq = softmax_scale * 1.4426950408889634f;  // logits in the exp2 domain
  e = launch_pdl(attn_nvf4_kernel, dim3(splits, num_q), dim3(kThreads), kSmemBytes, s, codes, scales, idx, g,
                 q_seq, topk, split_len, kq, (const unsigned char*)terms, out, lse, part_o, part_ml, st);
  if (e != cudaSuccess) return e;
  if (splits > 1) e = launch_attn_combine(part_o, part_ml, splits, num_q, out, lse, nullptr, 1, 1, s);
  return e;
}

}  // namespace csa2
