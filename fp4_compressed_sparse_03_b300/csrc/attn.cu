// Gather-dequantise sparse attention over the selected FP4 latent rows.
//
// zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮": the main KV is stored as
// FP4 E2M1 and dequantised before attention; tech-report digest (jiwasawa.github.io),
// "Reuse Mode": sparse attention runs directly over the inherited top-K entries.
// MQA over the shared latent: K = V = c_hat (512 channels), 16 query heads.
//
// One CTA (8 warps) handles one (query, split) pair: up to `split_len` selected
// entries in tiles of 64 tokens.  Per tile:
//   1. cp.async gathers 64 x (256 B codes + 32 B scales) into a 3-stage staging ring;
//   2. the tile is dequantised once into f16 in shared memory (E2M1 x E4M3 is exact
//      in f16: at most 6 significant bits, magnitudes 2^-10 .. 2688);
//   3. S = Q . C^T on tensor cores (m16n8k16, 16 heads = M), fp32 accumulation;
//   4. fp32 online softmax in the exp2 domain;
//   5. O += P . C on tensor cores, each warp owning 64 output channels.
// Q is converted to f16 after a per-query power-of-two prescale (exact for every
// value within 2^28 of the largest |q|); the scale is undone in the logit factor.
// Several splits per query are merged by a log-sum-exp combine kernel.
#include "common.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;
constexpr int kTile = 64;
constexpr int kStages = 3;
constexpr int kRowH = kDkv + 8;        // f16 elements per padded Q / C row (1040 B)
constexpr int kPRow = kTile + 8;       // f16 per padded P row
constexpr int kSRow = kTile + 4;       // fp32 per padded S row
constexpr int kStageBytes = kTile * (kCodeRow + kScaleRow);  // 18432

struct AttnSmem {
  __half qs[kHq][kRowH];
  __half cs[kTile][kRowH];
  unsigned char stage[kStages][kStageBytes];
  float ss[kHq][kSRow];
  __half ps[kHq][kPRow];
  int valid[kStages][kTile];
  float m_run[kHq], l_run[kHq], alpha[kHq];
  uint32_t red[kAttnThreads / 32];
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

// Issue the gathers of tile `tile` (entries j0 + 64*tile ...) into staging buffer `sb`.
__device__ __forceinline__ void issue_tile(AttnSmem& sm, int sb, const int32_t* __restrict__ idx_q,
                                           int jbeg, int jend, const uint8_t* __restrict__ codes,
                                           const uint8_t* __restrict__ scales, const AttnGeom& g,
                                           int b, int n_ctx, int32_t* st) {
  unsigned char* stage = sm.stage[sb];
  for (int ch = threadIdx.x; ch < kTile * 18; ch += kAttnThreads) {
    const int tok = ch / 18, part = ch - tok * 18;
    const int j = jbeg + tok;
    int valid = 0;
    int64_t slot = 0;
    if (j < jend) {
      const int s = __ldg(idx_q + j);
      if (s >= 0 && s < n_ctx) {
        const int32_t pg = __ldg(g.page_table + (int64_t)b * g.max_pages + (s >> 6));
        if (pg >= 0 && pg < g.num_pages) {
          valid = 1;
          slot = (int64_t)pg * kPage + (s & (kPage - 1));
        } else if (part == 0) {
          report(st, CSA2_DEV_BAD_PAGE);
        }
      } else if (s != -1 && part == 0) {
        report(st, CSA2_DEV_BAD_INDEX);
      }
    }
    if (part == 0) sm.valid[sb][tok] = valid;
    if (valid) {
      if (part < 16)
        cp_async16(stage + tok * kCodeRow + part * 16, codes + slot * kCodeRow + part * 16);
      else
        cp_async16(stage + kTile * kCodeRow + tok * kScaleRow + (part - 16) * 16,
                   scales + slot * kScaleRow + (part - 16) * 16);
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ codes,
                       const uint8_t* __restrict__ scales, const int32_t* __restrict__ idx,
                       AttnGeom g, const int32_t* __restrict__ q_seq, int32_t topk, int32_t split_len,
                       float softmax_scale, float* __restrict__ out, float* __restrict__ lse,
                       float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qi = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
  const int jbeg0 = split * split_len;
  const int jend = min(topk, jbeg0 + split_len);
  const int ntiles = jend > jbeg0 ? (jend - jbeg0 + kTile - 1) / kTile : 0;
  int b = __ldg(q_seq + qi);
  int n_ctx = 0;
  if (b < 0 || b >= g.num_seqs) {
    if (tid == 0) report(st, CSA2_DEV_BAD_QSEQ);
    b = 0;
  } else {
    n_ctx = __ldg(g.seq_lens + b);
  }
  const int32_t* idx_q = idx + (int64_t)qi * topk;

  // start the first gathers before touching Q
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) issue_tile(sm, s, idx_q, jbeg0 + s * kTile, jend, codes, scales, g, b, n_ctx, st);
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
  if (tid < kHq) {
    sm.m_run[tid] = -INFINITY;
    sm.l_run[tid] = 0.0f;
  }
  __syncthreads();
  uint32_t mxa = 0;
  for (int w = 0; w < kAttnThreads / 32; ++w) mxa = max(mxa, sm.red[w]);
  int sh = 0;
  if (mxa != 0) {
    const int e = (int)((mxa >> 7) & 0xFF) - 127;  // bf16 exponent of max |q|
    sh = max(-126, min(126, 14 - e));
  }
  const float pre = __uint_as_float((uint32_t)(127 + sh) << 23);   // 2^sh
  const float post = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
  const float kq = softmax_scale * 1.4426950408889634f * post;  // logits in the exp2 domain
  for (int i = tid; i < kHq * kDkv / 2; i += kAttnThreads) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(qq) + i);
    const __half2 h = __floats2half2_rn(bf16lo(w) * pre, bf16hi(w) * pre);
    const int hd = (2 * i) / kDkv, c = (2 * i) % kDkv;
    *reinterpret_cast<__half2*>(&sm.qs[hd][c]) = h;
  }

  float acc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.0f;

  const int gq = lane >> 2, cq = lane & 3;
  for (int t = 0; t < ntiles; ++t) {
    const int sb = t % kStages;
    cp_async_wait<kStages - 2>();
    __syncthreads();  // tile t staged; previous tile's readers of cs / ps are done
    {
      const int nt = t + kStages - 1;
      if (nt < ntiles)
        issue_tile(sm, nt % kStages, idx_q, jbeg0 + nt * kTile, jend, codes, scales, g, b, n_ctx, st);
      cp_async_commit();
    }
    // ---- dequantise: (token, 16-channel group) units ----
    const unsigned char* stage = sm.stage[sb];
    for (int uidx = tid; uidx < kTile * 32; uidx += kAttnThreads) {
      const int tok = uidx >> 5, grp = uidx & 31;
      uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
      if (sm.valid[sb][tok]) {
        const uint2 cw = *reinterpret_cast<const uint2*>(stage + tok * kCodeRow + grp * 8);
        const float s = e4m3_decode(stage[kTile * kCodeRow + tok * kScaleRow + grp]);
        const __half2 s2 = __float2half2_rn(s);
        uint32_t r[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t byte = ((k < 4 ? cw.x : cw.y) >> (8 * (k & 3))) & 0xFFu;
          const uint32_t h2 = e2m1x2_to_f16x2(byte);
          const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), s2);
          r[k] = *reinterpret_cast<const uint32_t*>(&v);
        }
        o0 = make_uint4(r[0], r[1], r[2], r[3]);
        o1 = make_uint4(r[4], r[5], r[6], r[7]);
      }
      uint4* dst = reinterpret_cast<uint4*>(&sm.cs[tok][grp * 16]);
      dst[0] = o0;
      dst[1] = o1;
    }
    __syncthreads();

    // ---- S = Q . C^T: warp w -> tokens 8w .. 8w+7, all 512 channels ----
    {
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const int tok0 = 8 * warp;
#pragma unroll 4
      for (int kk = 0; kk < kDkv / 16; kk += 2) {
        uint32_t a0[4], a1[4], bb[4];
        {
          const int m = lane >> 3, r = lane & 7;
          ldsm_x4(a0, &sm.qs[(m & 1) * 8 + r][16 * kk + (m >> 1) * 8]);
          ldsm_x4(a1, &sm.qs[(m & 1) * 8 + r][16 * (kk + 1) + (m >> 1) * 8]);
          ldsm_x4(bb, &sm.cs[tok0 + r][16 * kk + m * 8]);
        }
        mma_f16(d, a0, bb[0], bb[1]);
        mma_f16(d, a1, bb[2], bb[3]);
      }
      // d0,d1: head gq, tokens 2cq, 2cq+1; d2,d3: head gq+8
      const int tk = tok0 + 2 * cq;
      const bool v0 = sm.valid[sb][tk], v1 = sm.valid[sb][tk + 1];
      sm.ss[gq][tk] = v0 ? d[0] * kq : -INFINITY;
      sm.ss[gq][tk + 1] = v1 ? d[1] * kq : -INFINITY;
      sm.ss[gq + 8][tk] = v0 ? d[2] * kq : -INFINITY;
      sm.ss[gq + 8][tk + 1] = v1 ? d[3] * kq : -INFINITY;
    }
    __syncthreads();

    // ---- online softmax: warp w -> heads 2w, 2w+1 ----
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * warp + hh;
      const float s0 = sm.ss[h][lane], s1 = sm.ss[h][lane + 32];
      float tmax = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_old = sm.m_run[h];
      const float m_new = fmaxf(m_old, tmax);
      const float al = (m_new == -INFINITY) ? 1.0f : exp2f(m_old - m_new);
      const float p0 = (s0 == -INFINITY) ? 0.0f : exp2f(s0 - m_new);
      const float p1 = (s1 == -INFINITY) ? 0.0f : exp2f(s1 - m_new);
      sm.ps[h][lane] = __float2half_rn(p0);
      sm.ps[h][lane + 32] = __float2half_rn(p1);
      float ps = p0 + p1;
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

    // ---- O += P . C: warp w -> channels 64w .. 64w+63 ----
    {
      const float al0 = sm.alpha[gq], al1 = sm.alpha[gq + 8];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        acc[n][0] *= al0;
        acc[n][1] *= al0;
        acc[n][2] *= al1;
        acc[n][3] *= al1;
      }
      const int m = lane >> 3, r = lane & 7;
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, &sm.ps[(m & 1) * 8 + r][16 * ks + (m >> 1) * 8]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bb[4];
          // matrices: (tok 0-7, ch n0), (tok 8-15, ch n0), (tok 0-7, ch n0+8), (tok 8-15, ch n0+8)
          ldsm_x4_t(bb, &sm.cs[16 * ks + (m & 1) * 8 + r][64 * warp + 16 * np + (m >> 1) * 8]);
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
    for (int n = 0; n < 8; ++n) {
      const int ch = 64 * warp + 8 * n + 2 * cq;
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
    for (int n = 0; n < 8; ++n) {
      const int ch = 64 * warp + 8 * n + 2 * cq;
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

// Merge the splits of each query: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           int nsplit, float* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int qi = blockIdx.x;
  __shared__ float wgt[64][kHq];
  __shared__ float inv[kHq];
  const float* ml = part_ml + (int64_t)qi * nsplit * 2 * kHq;
  if (threadIdx.x < kHq) {
    const int h = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[s * 2 * kHq + h]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float m = ml[s * 2 * kHq + h], l = ml[s * 2 * kHq + kHq + h];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      wgt[s][h] = w;
      L += w * l;
    }
    inv[h] = L > 0.f ? 1.0f / L : 0.f;
    if (lse) lse[(int64_t)qi * kHq + h] = L > 0.f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
  }
  __syncthreads();
  const float4* po = reinterpret_cast<const float4*>(part_o + (int64_t)qi * nsplit * kHq * kDkv);
  float4* o = reinterpret_cast<float4*>(out + (int64_t)qi * kHq * kDkv);
  for (int i = threadIdx.x; i < kHq * kDkv / 4; i += blockDim.x) {
    const int h = (4 * i) / kDkv;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nsplit; ++s) {
      const float w = wgt[s][h];
      if (w == 0.f) continue;
      const float4 v = po[(int64_t)s * kHq * kDkv / 4 + i];
      a.x += w * v.x;
      a.y += w * v.y;
      a.z += w * v.z;
      a.w += w * v.w;
    }
    const float iv = inv[h];
    o[i] = make_float4(a.x * iv, a.y * iv, a.z * iv, a.w * iv);
  }
}

int attn_splits(int32_t num_q, int32_t topk, int num_sms) {
  const int max_splits = std::max(1, std::min(64, (topk + kTile - 1) / kTile));
  int want = (2 * num_sms + num_q - 1) / std::max(1, num_q);
  return std::max(1, std::min(max_splits, want));
}

int attn_split_len(int32_t topk, int splits) {
  int len = (topk + splits - 1) / splits;
  return (len + kTile - 1) / kTile * kTile;
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
    attn_combine_kernel<<<num_q, 256, 0, s>>>(part_o, part_ml, splits, out, lse);
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
