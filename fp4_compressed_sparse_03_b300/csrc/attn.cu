// Gather-dequantise sparse attention over the selected FP4 latent rows.
//
// zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮": the main KV is stored as
// FP4 E2M1 and dequantised before attention; tech-report digest (jiwasawa.github.io),
// "Reuse Mode": sparse attention runs directly over the inherited top-K entries.
// MQA over the shared latent: K = V = c_hat (512 channels), 16 query heads.
//
// One CTA (8 warps, one per SM) handles one (query, split) pair: up to `split_len`
// selected entries in tiles of 128 tokens, on the 5th-generation tensor cores:
//   1. cp.async gathers the tile's 128 x (256 B codes + 32 B scales) into a 2-stage
//      staging ring (1D bulk copies were measured slower: the copy engine took ~50
//      cycles per 256-byte row);
//   2. the warps dequantise the tile into an f16 tile C [128 tokens][512 channels]
//      laid out as eight 128-byte-swizzled [128][64] chunks (E2M1 x E4M3 is exact in
//      f16: at most 6 significant bits, magnitudes 2^-10 .. 2688);
//   3. S^T = C . Q^T: tcgen05.mma M=128 (tokens) x N=16 (heads) x K=512, C K-major,
//      fp32 accumulator in TMEM;
//   4. fp32 softmax in the exp2 domain with a lazily moved reference max per head: the
//      reference only moves (and the TMEM accumulator is rescaled) when a tile's max
//      exceeds it by more than 2^8, so every weight is at most 2^8;
//   5. O^T += C^T . P^T: M=128 (channels) x N=16 (heads) x K=128 (tokens) per 128-channel
//      block, reading the same C tile as an MN-major operand; P^T is f16, and the
//      normaliser sums the same f16-rounded weights.
// Steps 5 (tile t) and 2-3 (tile t+1) are pipelined by 128-channel chunk pairs: block
// j of the P.C product commits its own mbarrier, the next tile's chunk pair j is
// dequantised as soon as block j is done, and its logit MMAs are issued right after.
// Q is converted to f16 after a per-query power-of-two prescale (exact for every
// value within 2^28 of the largest |q|); the scale is undone in the logit factor.
// Several splits per query are merged by a log-sum-exp combine kernel.
#include <cstddef>

#include "tcgen05.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;   // 8 warps
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTile = 128;           // tokens per tile = UMMA M
constexpr int kRawStages = 2;        // cp.async staging ring
constexpr int kMaxSplit = 1024;      // selected entries per CTA at most
constexpr int kChunkBytes = kTile * 128;        // one 64-channel chunk of C: 16 KB
constexpr int kCBytes = (kDkv / 64) * kChunkBytes;  // 128 KB
constexpr int kQChunk = kHq * 128;              // one 64-channel chunk of Q: 2 KB
constexpr int kQBytes = (kDkv / 64) * kQChunk;  // 16 KB
constexpr int kPBytes = (kTile / 64) * kQChunk; // P^T [16 heads][128 tokens]: 4 KB
constexpr int kRawCodeBytes = kTile * kCodeRow;             // 32 KB
constexpr int kRawBytes = kRawCodeBytes + kTile * kScaleRow;  // 36 KB
constexpr uint32_t kTmemCols = 128;  // S^T at columns 0..15, O^T blocks at 32 + 16 j
constexpr uint32_t kOCol = 32;
constexpr float kRescaleGap = 8.0f;  // log2 units

constexpr int kPairs = kDkv / 128;  // 128-channel chunk pairs = O^T blocks

struct AttnCtl {
  alignas(16) float red_max[kHq][4];  // read back as float4 per head
  alignas(16) float red_sum[kHq][4];
  uint64_t bar_s, bar_fin;
  uint64_t bar_pv[kPairs];  // block j of the current tile's P.C product (and all before it)
  uint32_t tmem;
  volatile int abort;
  uint32_t qmax[kAttnWarps];
  int32_t slot[kMaxSplit];  // physical row of each selected entry, -1 if skipped
};
static_assert(offsetof(AttnCtl, red_max) % 16 == 0 && offsetof(AttnCtl, red_sum) % 16 == 0,
              "per-head reductions are read as float4");
static_assert(offsetof(AttnCtl, bar_s) % 8 == 0 && offsetof(AttnCtl, bar_pv) % 8 == 0,
              "mbarriers need 8-byte alignment");
constexpr size_t kAttnSmem = 1024 + kCBytes + kQBytes + kPBytes + kRawStages * kRawBytes + sizeof(AttnCtl);
static_assert(kAttnSmem <= 232448, "sparse attention needs more than 227 KB of shared memory");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// 2^x by the MUFU ex2 instruction (flushes subnormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait on an mbarrier phase that ignores the CTA's abort flag (used to drain).
__device__ __forceinline__ bool mbar_drain(uint64_t* b, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try(b, parity)) return true;
  return false;
}

struct AttnGeom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t max_pages;
  int32_t num_pages;
  int32_t num_seqs;
};

// Gather the codes and scales of the tile starting at local entry `e0` into `stage`:
// thread -> row tid / 2; the two threads of a row take the 16-byte parts of even and odd
// index (16 code parts, then 2 scale parts), so each pair of lanes moves 32 contiguous bytes.
// Codes are staged chunk-pair-major, [pair j][row][64 B] (code bytes 64 j .. 64 j + 63 of
// each row), so that the dequantiser's four rows per load instruction are contiguous;
// scales are staged [row][32 B].
__device__ __forceinline__ void issue_tile(unsigned char* stage, int e0, int ecount,
                                           const int32_t* slot, const uint8_t* __restrict__ codes,
                                           const uint8_t* __restrict__ scales) {
  const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
  const int e = e0 + r;
  const int32_t sl = e < ecount ? slot[e] : -1;
  if (sl < 0) return;
  const uint8_t* src = codes + (int64_t)sl * kCodeRow;
  unsigned char* dst = stage + r * 64;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int part = 2 * j + h;  // bytes 16 part .. +15 = pair part / 4, offset 16 (part % 4)
    cp_async16(dst + (part >> 2) * (kTile * 64) + 16 * (part & 3), src + 16 * part);
  }
  cp_async16(stage + kRawCodeBytes + r * kScaleRow + 16 * h, scales + (int64_t)sl * kScaleRow + 16 * h);
}
static_assert(kAttnThreads == 2 * kTile, "issue_tile maps two threads to each row of a tile");

// Staged tile -> chunks 2j, 2j + 1 (channels 128 j .. 128 j + 127) of the f16 tile C.
// Lane -> (row sub-index lane / 8, scale group 8 j + lane % 8 = 16 channels = code bytes
// 64 j + 8 (lane % 8) .. +7); warp w takes rows 4 (w + 8 i) + lane / 8, i = 0..3, so each
// 8-byte load instruction reads 256 contiguous staged bytes.  The
// group's 16 channels are units 2 (lane % 4), +1 of chunk 2 j + (lane % 8) / 4, stored at
// unit u ^ (row % 8); lanes of the odd chunk store their two units in the opposite
// order, so each quarter-warp store phase covers all eight units of a 128-byte row
// segment.  All loads are issued before any store.  Invalid rows become zeros.
__device__ __forceinline__ void dequant_pair(const unsigned char* stage, unsigned char* Cs, int j,
                                             int e0, int ecount, const int32_t* slot, int warp,
                                             int lane) {
  constexpr int kIter = kTile / (4 * kAttnWarps);  // 4
  const unsigned char* rc = stage;
  const unsigned char* rs = stage + kRawCodeBytes;
  const int l8 = lane & 7, rsub = lane >> 3;
  const int ch = 2 * j + (l8 >> 2), u0 = 2 * (l8 & 3), swap = l8 >> 2;
  unsigned char* cbase = Cs + ch * kChunkBytes;
  uint2 cw[kIter];
  uint32_t sb[kIter];
  bool ok[kIter];
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int r = 4 * (warp + kAttnWarps * i) + rsub;
    const int e = e0 + r;
    ok[i] = e < ecount && slot[e] >= 0;
    cw[i] = *reinterpret_cast<const uint2*>(rc + j * (kTile * 64) + r * 64 + 8 * l8);
    sb[i] = rs[r * kScaleRow + 8 * j + l8];
  }
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int r = 4 * (warp + kAttnWarps * i) + rsub;
    uint32_t hv[8];
    if (ok[i]) {
      uint32_t s2;
      const uint16_t sp = (uint16_t)(sb[i] | (sb[i] << 8));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"(sp));
      const uint32_t w[2] = {cw[i].x, cw[i].y};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t c2 = e2m1x2_to_f16x2((w[k >> 2] >> (8 * (k & 3))) & 0xFFu);
        const __half2 x = __hmul2(*reinterpret_cast<const __half2*>(&c2),
                                  *reinterpret_cast<const __half2*>(&s2));
        hv[k] = *reinterpret_cast<const uint32_t*>(&x);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) hv[k] = 0u;
    }
    unsigned char* row = cbase + r * 128;
    const int x7 = r & 7;
    const uint4 a = make_uint4(hv[0], hv[1], hv[2], hv[3]), c = make_uint4(hv[4], hv[5], hv[6], hv[7]);
    if (swap) {
      *reinterpret_cast<uint4*>(row + (((u0 + 1) ^ x7) << 4)) = c;
      *reinterpret_cast<uint4*>(row + ((u0 ^ x7) << 4)) = a;
    } else {
      *reinterpret_cast<uint4*>(row + ((u0 ^ x7) << 4)) = a;
      *reinterpret_cast<uint4*>(row + (((u0 + 1) ^ x7) << 4)) = c;
    }
  }
}

// Butterfly over the warp: lane l ends with the reduction, over all 32 lanes, of value
// (l >> 2) & 7 of the 8 each lane holds.
template <bool kMax>
__device__ __forceinline__ float warp_reduce8(float (&v)[8], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 16;
    const float send = hi ? v[i] : v[i + 4];
    const float keep = hi ? v[i + 4] : v[i];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 8;
    const float send = hi ? v[i] : v[i + 2];
    const float keep = hi ? v[i + 2] : v[i];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  {
    const bool hi = lane & 4;
    const float send = hi ? v[0] : v[1];
    const float keep = hi ? v[1] : v[0];
    v[0] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  float x = v[0];
  x = op(x, __shfl_xor_sync(0xffffffffu, x, 2));
  x = op(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return x;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ codes,
                       const uint8_t* __restrict__ scales, const int32_t* __restrict__ idx,
                       AttnGeom g, const int32_t* __restrict__ q_seq, int32_t topk, int32_t split_len,
                       float softmax_scale, float* __restrict__ out, float* __restrict__ lse,
                       float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* Cs = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* Qs = Cs + kCBytes;
  unsigned char* Ps = Qs + kQBytes;
  unsigned char* raw = Ps + kPBytes;
  AttnCtl& ctl = *reinterpret_cast<AttnCtl*>(raw + kRawStages * kRawBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sp = warp & 3;   // TMEM sub-partition: lanes 32 sp .. 32 sp + 31
  const int hg = warp >> 2;  // heads 8 hg .. 8 hg + 7 in the softmax; O blocks 2 hg, 2 hg + 1
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

  // Q is loaded first: its latency overlaps the index and page-table loads below
  const uint4* qv = reinterpret_cast<const uint4*>(q + (int64_t)qi * kHq * kDkv);
  uint4 qr[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) qr[k] = __ldg(qv + tid + kAttnThreads * k);

  // ---- resolve the selected entries to physical rows: the first two tiles first ----
  auto resolve = [&](int e) {
    const int s = __ldg(idx_q + e);
    int32_t slot = -1;
    if (s >= 0 && s < n_ctx) {
      const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (s >> 6));
      if (pg >= 0 && pg < g.num_pages) slot = pg * kPage + (s & (kPage - 1));
      else report(st, CSA2_DEV_BAD_PAGE);
    } else if (s != -1) {
      report(st, CSA2_DEV_BAD_INDEX);
    }
    ctl.slot[e] = slot;
  };
  const int e_first = min(ecount, kRawStages * kTile);
  for (int e = tid; e < e_first; e += kAttnThreads) resolve(e);
  if (tid == 0) {
    mbar_init(&ctl.bar_s, 1);
    for (int j = 0; j < kPairs; ++j) mbar_init(&ctl.bar_pv[j], 1);
    mbar_init(&ctl.bar_fin, 1);
    ctl.abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&ctl.tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem;

  // start the first gathers, then resolve the remaining entries while they land
#pragma unroll
  for (int i = 0; i < kRawStages; ++i) {
    if (i < ntiles) issue_tile(raw + i * kRawBytes, i * kTile, ecount, ctl.slot, codes, scales);
    cp_async_commit();
  }
  for (int e = e_first + tid; e < ecount; e += kAttnThreads) resolve(e);

  // ---- Q: max |q| -> power-of-two prescale -> f16 chunks (the barrier below also
  // publishes the remaining slots) ----
  uint32_t mx = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w[4] = {qr[k].x, qr[k].y, qr[k].z, qr[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) ctl.qmax[warp] = mx;
  __syncthreads();
  uint32_t mxa = 0;
#pragma unroll
  for (int w = 0; w < kAttnWarps; ++w) mxa = max(mxa, ctl.qmax[w]);
  int sh = 0;
  if (mxa != 0) {
    const int e = (int)((mxa >> 7) & 0xFF) - 127;  // bf16 exponent of max |q|
    sh = max(-126, min(126, 14 - e));
  }
  const float pre = __uint_as_float((uint32_t)(127 + sh) << 23);   // 2^sh
  const float post = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
  const float kq = softmax_scale * 1.4426950408889634f * post;  // logits in the exp2 domain
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = tid + kAttnThreads * k;  // 8 channels 8i .. 8i + 7
    const int hd = (8 * i) / kDkv, c = (8 * i) % kDkv;
    const uint32_t w[4] = {qr[k].x, qr[k].y, qr[k].z, qr[k].w};
    uint32_t hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 h = __floats2half2_rn(bf16lo(w[e]) * pre, bf16hi(w[e]) * pre);
      hv[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const int u = (c & 63) >> 3;
    *reinterpret_cast<uint4*>(Qs + (c >> 6) * kQChunk + hd * 128 + ((u ^ (hd & 7)) << 4)) =
        make_uint4(hv[0], hv[1], hv[2], hv[3]);
  }
  fence_proxy_async_smem();

  // per-head reference max (log2 units) and normaliser, identical in every thread
  float m_used[kHq], l_run[kHq];
#pragma unroll
  for (int h = 0; h < kHq; ++h) {
    m_used[h] = -INFINITY;
    l_run[h] = 0.0f;
  }
  const uint32_t idesc_s = umma_idesc_f16(kTile, kHq, false, false, false);
  const uint32_t idesc_o = umma_idesc_f16(128, kHq, false, true, false);
  const uint32_t cs_addr = smem_u32(Cs), qs_addr = smem_u32(Qs), ps_addr = smem_u32(Ps);
  const int tt = 32 * sp + lane;  // this thread's token row of the S tile

  // Build C for tile u from its staged rows, chunk pair by chunk pair, issuing the logit
  // MMAs of each pair as soon as it is written.  For u > 0, pair j is overwritten only
  // after block j of tile u - 1's P.C product has completed.  Returns false on abort.
  auto build_tile = [&](int u) -> bool {
    unsigned char* stage = raw + (u % kRawStages) * kRawBytes;
    if (u > 0) {  // tile u + 1 goes into the stage tile u - 1 has released
      if (u + 1 < ntiles)
        issue_tile(raw + ((u + 1) % kRawStages) * kRawBytes, (u + 1) * kTile, ecount, ctl.slot,
                   codes, scales);
      cp_async_commit();
    }
    cp_async_wait<1>();  // every group but the newest has landed: tile u is staged
    const uint32_t par = (uint32_t)((u - 1) & 1);
    if (tid == 0 && u > 0) (void)mbar_wait(&ctl.abort, &ctl.bar_pv[0], par, st);
    __syncthreads();
    if (ctl.abort) return false;
    for (int j = 0; j < kPairs; ++j) {
      dequant_pair(stage, Cs, j, u * kTile, ecount, ctl.slot, warp, lane);
      fence_proxy_async_smem();
      if (tid == 0 && u > 0 && j + 1 < kPairs)
        (void)mbar_wait(&ctl.abort, &ctl.bar_pv[j + 1], par, st);
      __syncthreads();
      if (ctl.abort) return false;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int kc = 2 * j + c2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(tmem, umma_desc_sw128(cs_addr + kc * kChunkBytes, 16, 1024) + 2 * kk,
                     umma_desc_sw128(qs_addr + kc * kQChunk, 16, 1024) + 2 * kk, idesc_s,
                     (kc | kk) != 0 ? 1u : 0u);
        }
      }
    }
    if (tid == 0) umma_commit(&ctl.bar_s);
    return true;
  };

  bool ok = ntiles == 0 || build_tile(0);
  for (int t = 0; ok && t < ntiles; ++t) {
    // ---- wait for S^T of tile t ----
    if (tid == 0) (void)mbar_wait(&ctl.abort, &ctl.bar_s, (uint32_t)(t & 1), st);
    __syncthreads();
    if (ctl.abort) break;
    tc_fence_after();

    // ---- softmax: thread -> token tt, heads 8 hg .. 8 hg + 7 ----
    uint32_t sr[8];
    tmem_ld8(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(8 * hg), sr);
    const int e = t * kTile + tt;
    const bool valid = e < ecount && ctl.slot[e] >= 0;
    float s[8], v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s[i] = valid ? __uint_as_float(sr[i]) * kq : -INFINITY;
      v[i] = s[i];
    }
    const int hl = (lane >> 2) & 7;
    const float wmax = warp_reduce8<true>(v, lane);
    if ((lane & 3) == 0) ctl.red_max[8 * hg + hl][sp] = wmax;
    __syncthreads();
    float alpha[kHq];
    bool moved = false;
#pragma unroll
    for (int h = 0; h < kHq; ++h) {
      const float4 r = *reinterpret_cast<const float4*>(ctl.red_max[h]);
      const float mt = fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w));
      const float mu = m_used[h];
      float mn = mu;
      if (mu == -INFINITY || mt > mu + kRescaleGap) mn = fmaxf(mu, mt);
      alpha[h] = 1.0f;
      if (mn != mu) {  // uniform: every thread holds the same reference maxima
        alpha[h] = ex2(mu - mn);
        moved = true;
      }
      m_used[h] = mn;
    }
    const int tk = tt & 63, pu = tk >> 3;
    unsigned char* prow = Ps + (tt >> 6) * kQChunk;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float mh = hg ? m_used[8 + i] : m_used[i];
      if (mh == -INFINITY) mh = 0.0f;  // no valid entry yet: every s is -inf as well
      const __half ph = __float2half_rn(ex2(s[i] - mh));  // 2^-inf = 0 for skipped entries
      *reinterpret_cast<__half*>(prow + (8 * hg + i) * 128 + ((pu ^ i) << 4) + (tk & 7) * 2) = ph;
      v[i] = __half2float(ph);
    }
    const float wsum = warp_reduce8<false>(v, lane);
    if ((lane & 3) == 0) ctl.red_sum[8 * hg + hl][sp] = wsum;
    if (moved && t > 0) {  // move the accumulated O^T to the new reference
      uint32_t o[32];
      const uint32_t ta = tmem + ((uint32_t)(32 * sp) << 16) + kOCol + (uint32_t)(32 * hg);
      tmem_ld32(ta, o);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha[i & 15]);
      tmem_st32(ta, o);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kHq; ++h) {
      const float4 r = *reinterpret_cast<const float4*>(ctl.red_sum[h]);
      l_run[h] = l_run[h] * alpha[h] + ((r.x + r.y) + (r.z + r.w));
    }

    // ---- O^T += C^T . P^T, one 128-channel block at a time, one barrier per block ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < kPairs; ++j) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_f16(tmem + kOCol + 16 * j,
                   umma_desc_sw128(cs_addr + 2 * j * kChunkBytes + kk * 2048, kChunkBytes, 1024),
                   umma_desc_sw128(ps_addr + (kk >> 2) * kQChunk, 16, 1024) + 2 * (kk & 3),
                   idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&ctl.bar_pv[j]);
      }
    }
    if (t + 1 < ntiles) ok = build_tile(t + 1);
  }
  cp_async_wait<0>();
  if (tid == 0) {
    if (ntiles > 0 && !ctl.abort)
      (void)mbar_wait(&ctl.abort, &ctl.bar_pv[kPairs - 1], (uint32_t)((ntiles - 1) & 1), st);
    // every MMA this thread issued has completed before TMEM is read or released
    umma_commit(&ctl.bar_fin);
    (void)mbar_drain(&ctl.bar_fin, 0, 1u << 20);
  }
  __syncthreads();
  tc_fence_after();
  const bool have = ntiles > 0 && !ctl.abort;

  // ---- epilogue: thread -> channel 128 j + 32 sp + lane of blocks j = 2 hg, 2 hg + 1 ----
  uint32_t o[32];
  if (have) {
    tmem_ld32(tmem + ((uint32_t)(32 * sp) << 16) + kOCol + (uint32_t)(32 * hg), o);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = 0u;
  }
  if (nsplit == 1) {
    float* ob = out + (int64_t)qi * kHq * kDkv;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int h = i & 15, ch = 128 * (2 * hg + (i >> 4)) + 32 * sp + lane;
      const float l = l_run[h];
      ob[h * kDkv + ch] = l > 0.f ? __uint_as_float(o[i]) / l : 0.f;
    }
    if (lse != nullptr) {
#pragma unroll
      for (int h = 0; h < kHq; ++h)
        if (tid == h)
          lse[(int64_t)qi * kHq + h] =
              l_run[h] > 0.f ? m_used[h] * 0.6931471805599453f + logf(l_run[h]) : -INFINITY;
    }
  } else {
    float* ob = part_o + ((int64_t)qi * nsplit + split) * kHq * kDkv;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int h = i & 15, ch = 128 * (2 * hg + (i >> 4)) + 32 * sp + lane;
      ob[h * kDkv + ch] = __uint_as_float(o[i]);
    }
    float* ml = part_ml + ((int64_t)qi * nsplit + split) * 2 * kHq;
#pragma unroll
    for (int h = 0; h < kHq; ++h)
      if (tid == h) {
        ml[h] = m_used[h];
        ml[kHq + h] = l_run[h];
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the splits of each (query, head): out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           int nsplit, float* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int qi = blockIdx.x, h = blockIdx.y;
  __shared__ float wgt[64];
  __shared__ float inv;
  const float* ml = part_ml + (int64_t)qi * nsplit * 2 * kHq;
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
  // 128 threads x 4 channels
  const float4* po = reinterpret_cast<const float4*>(part_o + ((int64_t)qi * nsplit * kHq + h) * kDkv);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  int s = 0;
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

// Splits per query: the count that minimises (waves of one CTA per SM) x (tiles per
// CTA + a fixed start-up cost of ~2 tiles), with at most kMaxSplit entries per CTA.
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
    const int64_t waves = (ctas + num_sms - 1) / num_sms;
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

size_t attn_smem_bytes() { return kAttnSmem; }

cudaError_t launch_attn(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                        const int32_t* idx, const csa2_pages& pg, float* out, float* lse,
                        int32_t num_q, const int32_t* q_seq, int32_t topk, float softmax_scale,
                        void* ws, int32_t* st, cudaStream_t s, int num_sms) {
  AttnGeom g{pg.seq_lens, pg.page_table, pg.max_pages_per_seq, pg.num_pages, pg.num_seqs};
  int splits = attn_splits(num_q, topk, num_sms);
  const int split_len = attn_split_len(topk, splits);
  splits = (topk + split_len - 1) / split_len;
  if (splits < 1) splits = 1;
  const size_t smem = attn_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  float* part_o = reinterpret_cast<float*>(ws);
  float* part_ml = part_o + (int64_t)num_q * splits * kHq * kDkv;
  dim3 grid(splits, num_q);
  sparse_attn_kernel<<<grid, kAttnThreads, smem, s>>>(q, codes, scales, idx, g, q_seq, topk,
                                                      split_len, softmax_scale, out, lse, part_o,
                                                      part_ml, st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (splits > 1) {
    attn_combine_kernel<<<dim3(num_q, kHq), 128, 0, s>>>(part_o, part_ml, splits, out, lse);
    e = cudaGetLastError();
  }
  return e;
}

size_t attn_workspace_bytes(int32_t num_q, int32_t topk, int num_sms) {
  int splits = attn_splits(num_q, topk, num_sms);
  const int split_len = attn_split_len(topk, splits);
  splits = (topk + split_len - 1) / split_len;
  if (splits <= 1) return 0;
  return (size_t)num_q * splits * (kHq * kDkv + 2 * kHq) * sizeof(float);
}

}  // namespace csa2
