// Gather-dequantise sparse attention over the selected FP4 latent rows.
//
// zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮": the main KV is stored as
// FP4 E2M1 and dequantised before attention; tech-report digest (jiwasawa.github.io),
// "Reuse Mode": sparse attention runs directly over the inherited top-K entries.
// MQA over the shared latent: K = V = c_hat (512 channels), 16 query heads.
//
// One CTA (4 warps) handles one (query, split) pair: up to `split_len` selected
// entries in tiles of 64 tokens.  Per tile:
//   1. cp.async gathers 32 x (256 B codes + 32 B scales) into a 4-stage staging ring;
//   2. S = Q . C^T on tensor cores (m16n8k16, 16 heads = M), fp32 accumulation, with
//      the dequantisation fused in: each lane turns its token's 4-byte code word into
//      its B fragments (E2M1 x E4M3 is exact in f16: at most 6 significant bits,
//      magnitudes 2^-10 .. 2688) and also stores them into the f16 tile C;
//   3. fp32 online softmax in the exp2 domain;
//   4. O += P . C on tensor cores, each warp owning 128 output channels.
// Q is converted to f16 after a per-query power-of-two prescale (exact for every
// value within 2^28 of the largest |q|); the scale is undone in the logit factor.
// Several splits per query are merged by a log-sum-exp combine kernel.
#include "common.cuh"

namespace csa2 {

constexpr int kAttnThreads = 128;   // 4 warps
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTile = 32;            // tokens per tile
constexpr int kStages = 4;           // cp.async staging ring
constexpr int kMaxSplit = 1024;      // selected entries per CTA at most
constexpr int kRowH = kDkv + 8;      // f16 elements per padded Q / C row (1040 B)
constexpr int kPRow = kTile + 8;     // f16 per padded P row
constexpr int kSRow = kTile + 4;     // fp32 per padded S row
constexpr int kCodeStride = kCodeRow + 16;  // padded staging row: conflict-free code reads
constexpr int kStageBytes = kTile * (kCodeStride + kScaleRow);  // 9728

struct AttnSmem {
  __half qs[kHq][kRowH];
  __half cs[kTile][kRowH];
  unsigned char stage[kStages][kStageBytes];
  float ss[kHq][kSRow];
  __half ps[kHq][kPRow];
  int32_t slot[kMaxSplit];           // physical row of each selected entry, -1 if skipped
  float m_run[kHq], l_run[kHq], alpha[kHq];
  uint32_t red[kAttnWarps];
};

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

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct AttnGeom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t max_pages;
  int32_t num_pages;
  int32_t num_seqs;
};

// Issue the gathers of the tile starting at local entry `e0` into staging buffer `sb`.
__device__ __forceinline__ void issue_tile(AttnSmem& sm, int sb, int e0, int ecount,
                                           const uint8_t* __restrict__ codes,
                                           const uint8_t* __restrict__ scales) {
  unsigned char* stage = sm.stage[sb];
  for (int ch = threadIdx.x; ch < kTile * 18; ch += kAttnThreads) {
    const int tok = ch / 18, part = ch - tok * 18;
    const int e = e0 + tok;
    const int32_t slot = e < ecount ? sm.slot[e] : -1;
    if (slot >= 0) {
      if (part < 16)
        cp_async16(stage + tok * kCodeStride + part * 16, codes + (int64_t)slot * kCodeRow + part * 16);
      else
        cp_async16(stage + kTile * kCodeStride + tok * kScaleRow + (part - 16) * 16,
                   scales + (int64_t)slot * kScaleRow + (part - 16) * 16);
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads, 2)
    sparse_attn_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ codes,
                       const uint8_t* __restrict__ scales, const int32_t* __restrict__ idx,
                       AttnGeom g, const int32_t* __restrict__ q_seq, int32_t topk, int32_t split_len,
                       float softmax_scale, float* __restrict__ out, float* __restrict__ lse,
                       float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

  // ---- resolve every selected entry of this split to its physical row ----
  for (int e = tid; e < ecount; e += kAttnThreads) {
    const int s = __ldg(idx_q + e);
    int32_t slot = -1;
    if (s >= 0 && s < n_ctx) {
      const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (s >> 6));
      if (pg >= 0 && pg < g.num_pages) slot = pg * kPage + (s & (kPage - 1));
      else report(st, CSA2_DEV_BAD_PAGE);
    } else if (s != -1) {
      report(st, CSA2_DEV_BAD_INDEX);
    }
    sm.slot[e] = slot;
  }
  if (tid < kHq) {
    sm.m_run[tid] = -INFINITY;
    sm.l_run[tid] = 0.0f;
  }
  __syncthreads();

  // start the first gathers before touching Q
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) issue_tile(sm, s, s * kTile, ecount, codes, scales);
    cp_async_commit();
  }

  // ---- Q: max |q| -> power-of-two prescale -> f16 ----
  const uint16_t* qq = q + (int64_t)qi * kHq * kDkv;
  uint32_t mx = 0;
  for (int i = tid; i < kHq * kDkv / 8; i += kAttnThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(qq) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) sm.red[warp] = mx;
  __syncthreads();
  uint32_t mxa = 0;
  for (int w = 0; w < kAttnWarps; ++w) mxa = max(mxa, sm.red[w]);
  int sh = 0;
  if (mxa != 0) {
    const int e = (int)((mxa >> 7) & 0xFF) - 127;  // bf16 exponent of max |q|
    sh = max(-126, min(126, 14 - e));
  }
  const float pre = __uint_as_float((uint32_t)(127 + sh) << 23);   // 2^sh
  const float post = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
  const float kq = softmax_scale * 1.4426950408889634f * post;  // logits in the exp2 domain
  for (int i = tid; i < kHq * kDkv / 8; i += kAttnThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(qq) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 h = __floats2half2_rn(bf16lo(w[e]) * pre, bf16hi(w[e]) * pre);
      hv[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const int hd = (8 * i) / kDkv, c = (8 * i) % kDkv;
    *reinterpret_cast<uint4*>(&sm.qs[hd][c]) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
  }

  float acc[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.0f;

  const int gq = lane >> 2, cq = lane & 3;
  const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix and row served by this lane
  for (int t = 0; t < ntiles; ++t) {
    const int sb = t % kStages;
    cp_async_wait<kStages - 2>();
    __syncthreads();  // tile t staged; previous tile's readers of cs / ps are done
    {
      const int nt = t + kStages - 1;
      if (nt < ntiles) issue_tile(sm, nt % kStages, nt * kTile, ecount, codes, scales);
      cp_async_commit();
    }
    // ---- S = Q . C^T with fused dequantisation: warp w -> tokens 8w .. 8w+7 ----
    // Lane (gq, cq) serves token gq of the warp.  For channel block p (32 channels,
    // k-steps 2p and 2p + 1) its k-slots {2cq, 2cq+1, 2cq+8, 2cq+9} map to channels
    // 32p + 8cq + {0..3} (k-step 2p) and 32p + 8cq + {4..7} (k-step 2p + 1), so one
    // 4-byte code word gives its B fragments and the A fragments of Q come from 16-byte
    // reads of head rows gq and gq + 8 at the same channels.
    const unsigned char* stage = sm.stage[sb];
    const int e0 = t * kTile;
    {
      const int tok = 8 * warp + gq;
      const bool tv = (e0 + tok < ecount) && sm.slot[e0 + tok] >= 0;
      const unsigned char* crow = stage + tok * kCodeStride;
      const unsigned char* srow = stage + kTile * kCodeStride + tok * kScaleRow;
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int p = 0; p < kDkv / 32; ++p) {
        const int ch = 32 * p + 8 * cq;
        const uint4 qa = *reinterpret_cast<const uint4*>(&sm.qs[gq][ch]);
        const uint4 qb = *reinterpret_cast<const uint4*>(&sm.qs[gq + 8][ch]);
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        if (tv) {
          const uint32_t cw = *reinterpret_cast<const uint32_t*>(crow + ch / 2);
          const __half2 s2 = __float2half2_rn(e4m3_decode(srow[ch >> 4]));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t h2 = e2m1x2_to_f16x2((cw >> (8 * k)) & 0xFFu);
            const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), s2);
            h[k] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        *reinterpret_cast<uint4*>(&sm.cs[tok][ch]) = make_uint4(h[0], h[1], h[2], h[3]);
        const uint32_t a0[4] = {qa.x, qb.x, qa.y, qb.y}, a1[4] = {qa.z, qb.z, qa.w, qb.w};
        mma_f16(d0, a0, h[0], h[1]);
        mma_f16(d1, a1, h[2], h[3]);
      }
      // d: heads gq (0..1) and gq + 8 (2..3), tokens 8w + 2cq, 8w + 2cq + 1
      const int tk = 8 * warp + 2 * cq;
      const bool v0 = (e0 + tk < ecount) && sm.slot[e0 + tk] >= 0;
      const bool v1 = (e0 + tk + 1 < ecount) && sm.slot[e0 + tk + 1] >= 0;
      sm.ss[gq][tk] = v0 ? (d0[0] + d1[0]) * kq : -INFINITY;
      sm.ss[gq][tk + 1] = v1 ? (d0[1] + d1[1]) * kq : -INFINITY;
      sm.ss[gq + 8][tk] = v0 ? (d0[2] + d1[2]) * kq : -INFINITY;
      sm.ss[gq + 8][tk + 1] = v1 ? (d0[3] + d1[3]) * kq : -INFINITY;
    }
    __syncthreads();

    // ---- online softmax: warp w -> heads 4w .. 4w+3, lane -> token ----
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const int h = 4 * warp + hh;
      const float s0 = sm.ss[h][lane];
      float tmax = s0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_old = sm.m_run[h];
      const float m_new = fmaxf(m_old, tmax);
      const float al = (m_new == -INFINITY) ? 1.0f : exp2f(m_old - m_new);
      const __half p0 = __float2half_rn((s0 == -INFINITY) ? 0.0f : exp2f(s0 - m_new));
      sm.ps[h][lane] = p0;
      // the normaliser sums the same f16-rounded weights the P.C product uses, so the
      // output stays an exact weighted average of the rows
      float ps = __half2float(p0);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      __syncwarp();
      if (lane == 0) {
        sm.m_run[h] = m_new;
        sm.l_run[h] = sm.l_run[h] * al + ps;
        sm.alpha[h] = al;
      }
    }
    __syncthreads();

    // ---- O += P . C: warp w -> channels 128w .. 128w+127 ----
    {
      const float al0 = sm.alpha[gq], al1 = sm.alpha[gq + 8];
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        acc[n][0] *= al0;
        acc[n][1] *= al0;
        acc[n][2] *= al1;
        acc[n][3] *= al1;
      }
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, &sm.ps[(lm & 1) * 8 + lr][16 * ks + (lm >> 1) * 8]);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t bb[4];
          // matrices: (tok 0-7, ch n0), (tok 8-15, ch n0), (tok 0-7, ch n0+8), (tok 8-15, ch n0+8)
          ldsm_x4_t(bb, &sm.cs[16 * ks + (lm & 1) * 8 + lr][128 * warp + 16 * np + (lm >> 1) * 8]);
          mma_f16(acc[2 * np], a, bb[0], bb[1]);
          mma_f16(acc[2 * np + 1], a, bb[2], bb[3]);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- epilogue ----
  const float l0 = sm.l_run[gq], l1 = sm.l_run[gq + 8];
  if (nsplit == 1) {
    const float i0 = l0 > 0.f ? 1.0f / l0 : 0.f, i1 = l1 > 0.f ? 1.0f / l1 : 0.f;
    float* o = out + (int64_t)qi * kHq * kDkv;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int ch = 128 * warp + 8 * n + 2 * cq;
      *reinterpret_cast<float2*>(o + gq * kDkv + ch) = make_float2(acc[n][0] * i0, acc[n][1] * i0);
      *reinterpret_cast<float2*>(o + (gq + 8) * kDkv + ch) = make_float2(acc[n][2] * i1, acc[n][3] * i1);
    }
    if (lse != nullptr && tid < kHq) {
      const float l = sm.l_run[tid];
      lse[(int64_t)qi * kHq + tid] =
          l > 0.f ? sm.m_run[tid] * 0.6931471805599453f + logf(l) : -INFINITY;
    }
  } else {
    float* o = part_o + ((int64_t)qi * nsplit + split) * kHq * kDkv;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int ch = 128 * warp + 8 * n + 2 * cq;
      *reinterpret_cast<float2*>(o + gq * kDkv + ch) = make_float2(acc[n][0], acc[n][1]);
      *reinterpret_cast<float2*>(o + (gq + 8) * kDkv + ch) = make_float2(acc[n][2], acc[n][3]);
    }
    if (tid < kHq) {
      float* ml = part_ml + ((int64_t)qi * nsplit + split) * 2 * kHq;
      ml[tid] = sm.m_run[tid];
      ml[kHq + tid] = sm.l_run[tid];
    }
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

// Splits per query: the count that minimises (waves of two CTAs per SM) x (tiles per
// CTA + a fixed start-up cost of ~4 tiles), with at most kMaxSplit entries per CTA.
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
    const int64_t waves = (ctas + 2 * num_sms - 1) / (2 * num_sms);
    const double cost = (double)waves * (per + 4);
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

size_t attn_smem_bytes() { return sizeof(AttnSmem); }

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
