// CED write path: C = H . W on the 5th-generation tensor cores, quantised on write.
//
// Tech-report digest (jiwasawa.github.io), section "Causal Encoder-Decoder (CED)
// アーキテクチャ", equation C_l = H_{L/2} W_l^KV: every decoder layer's global KV is
// a projection of the encoder's final hidden state.  ai2.x.ezic.info blog, section
// "KVを捨てる、共有する、作り直す": the KV is held as FP4 E2M1 with one E4M3 scale per
// 16 channels.
//
// Kernel design (sm_103a):
//   - persistent CTAs, one per SM, 128 x 256 output tiles (bf16 operands, fp32
//     accumulation), K consumed in 64-wide blocks through a 4-stage TMA ring
//     (128-byte swizzle, both operands K-major); for T <= 128 (one M-tile: the weight
//     stream is the whole cost) 128 x 128 tiles through 3 stages of two K-blocks, and
//     for T <= 64 through 4 such stages holding only H's 64 real rows;
//   - warp 0 lane 0 issues TMA, warp 1 lane 0 issues tcgen05.mma (M=128, N=256 or 128,
//     K=16) into one of two TMEM accumulators, warps 2..5 run the epilogue of the
//     previous tile while the next one accumulates;
//   - epilogue: tcgen05.ld 32 columns of one row per thread, then per 16-channel block
//     amax -> E4M3(amax/6) -> E2M1(x/s) packed codes + scale byte (latent
//     projections), or bf16 RNE (indexer-key projections), stored at the token's slot;
//   - tile order: groups of 16 M-tiles swept across all N-tiles, so the A tiles of a
//     group stay in L2 while the B slices stream;
//   - any T: rows of the last M-tile beyond T are zero-filled by the TMA load and not
//     stored (decode-time append writes T = one token per sequence);
//   - every mbarrier wait is bounded; on expiry the CTA raises CSA2_DEV_TIMEOUT, stops
//     issuing, waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include "async.cuh"

namespace csa2 {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int kThreads = 192;                   // 6 warps
constexpr int kGroupM = 16;

// Output tile width BN, TMA ring depth, K-blocks of 64 per stage (KSUB) and A rows loaded
// per K-block (AROWS).  Prefill-sized T: 256 columns, 4 stages of 48 KB.  A single M-tile
// (T <= 128, e.g. decode-time append of one token per sequence) is bound by streaming the
// weights: 128 columns double the CTAs that stream them, and stages of two adjacent
// K-blocks read 256 contiguous bytes of each weight row at a time.  With T <= 64 only 64
// rows of H are loaded per K-block (8 KB instead of 16): the MMA still has M = 128, and its
// A rows 64..127 read whatever follows in the stage (the next A block, or the first B
// block); those accumulator rows are never stored.  The smem saved holds a fourth stage,
// so a third more of the weights is in flight.  A stage is all its A blocks, then all its
// B blocks.
template <int BN, int STAGES, int KSUB, int AROWS = BM>
struct KvCfg {
  static constexpr int A_SUB = AROWS * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int A_PART = KSUB * A_SUB;  // offset of the B blocks in a stage
  static constexpr int STAGE_BYTES = KSUB * (A_SUB + B_BYTES);
  static_assert(AROWS == BM || A_PART + B_BYTES >= KSUB * A_SUB + (BM - AROWS) * BK * 2,
                "the MMA's overread of the last A block stays inside the stage");
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
  struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t fin;
    uint32_t tmem_base;
    volatile int abort;
  };
  static constexpr size_t smem_bytes() { return (size_t)STAGES * STAGE_BYTES + sizeof(Bars) + 1024; }
};
static_assert(KvCfg<256, 4, 1>::smem_bytes() <= 232448 && KvCfg<128, 6, 1>::smem_bytes() <= 232448 &&
                  KvCfg<128, 3, 2>::smem_bytes() <= 232448 && KvCfg<128, 4, 2, 64>::smem_bytes() <= 232448 &&
                  KvCfg<128, 8, 1, 64>::smem_bytes() <= 232448,
              "write-path ring exceeds 227 KB of shared memory");

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
  const uint64_t addr = saddr(p);
  uint64_t d = 0;
  d |= (addr & 0x3FFFFull) >> 4;      // start address, bits 0-13
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;             // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;             // swizzle mode: 128 B
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  uint32_t d = 0;
  d |= 1u << 4;                      // D format: f32
  d |= 1u << 7;                      // A format: bf16
  d |= 1u << 10;                     // B format: bf16
  d |= (uint32_t)(n >> 3) << 17;     // N / 8
  d |= (uint32_t)(m >> 4) << 24;     // M / 16
  return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct WriteParams {
  uint8_t* codes;
  uint8_t* scales;
  uint16_t* k_idx;
  const int32_t* slot_of_token;
  int64_t num_slots;
  int32_t T, d_model, n_kv_proj, n_idx_proj, n_out;
  int32_t* st;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& m, int& n) {
  const int per_group = kGroupM * num_n;
  const int grp = tile / per_group;
  const int first_m = grp * kGroupM;
  const int gm = min(kGroupM, num_m - first_m);
  const int r = tile - grp * per_group;
  n = r / gm;
  m = first_m + (r - n * gm);
}

}  // namespace

template <int BN, int STAGES, int KSUB, int AROWS>
__global__ void __launch_bounds__(kThreads, 1)
    kv_write_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    WriteParams p) {
  using Cfg = KvCfg<BN, STAGES, KSUB, AROWS>;
  constexpr int A_SUB = Cfg::A_SUB, A_PART = Cfg::A_PART, B_BYTES = Cfg::B_BYTES;
  using Bars = typename Cfg::Bars;
  constexpr int STAGE_BYTES = Cfg::STAGE_BYTES;
  constexpr int kTmemCols = Cfg::kTmemCols;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(base + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 128);
    }
    mbar_init(&bars->fin, 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(&bars->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars->tmem_base;

  const int num_m = (p.T + BM - 1) / BM;
  const int num_n = (p.n_out + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int kblocks = p.d_model / BK;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    uint32_t issued_mask = 0, last_par = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      int m, n;
      tile_coords(tile, num_m, num_n, m, n);
      for (int kb = 0; kb < kblocks; kb += KSUB) {  // kblocks is a multiple of KSUB
        if (!mbar_wait(&bars->abort, &bars->empty[stage], phase ^ 1u, p.st)) {
          ok = false;
          break;
        }
        unsigned char* sa = base + stage * STAGE_BYTES;
        mbar_expect_tx(&bars->full[stage], STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < KSUB; ++j) {
          tma_load_2d(sa + j * A_SUB, &tmA, &bars->full[stage], (kb + j) * BK, m * BM);
          tma_load_2d(sa + A_PART + j * B_BYTES, &tmB, &bars->full[stage], (kb + j) * BK, n * BN);
        }
        issued_mask |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // make sure no copy of ours is still landing in shared memory
    for (int s = 0; s < STAGES; ++s)
      if (issued_mask & (1u << s))
        (void)mbar_wait(&bars->abort, &bars->full[s], (last_par >> s) & 1u, p.st, 1u << 20);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_bf16(BM, BN);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      if (!mbar_wait(&bars->abort, &bars->tempty[acc], acc_phase ^ 1u, p.st)) break;
      fence_after();
      const uint32_t d = tmem + (uint32_t)(acc * BN);
      for (int kb = 0; kb < kblocks; kb += KSUB) {
        if (!mbar_wait(&bars->abort, &bars->full[stage], phase, p.st)) {
          ok = false;
          break;
        }
        fence_after();
#pragma unroll
        for (int j = 0; j < KSUB; ++j) {
          const unsigned char* st_base = base + stage * STAGE_BYTES;
          const uint64_t adesc = sw128_desc(st_base + j * A_SUB);
          const uint64_t bdesc = sw128_desc(st_base + A_PART + j * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                      (kb > 0 || j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars->empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(&bars->tfull[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // wait until every MMA this thread issued has completed
    umma_commit(&bars->fin);
    (void)mbar_wait(&bars->abort, &bars->fin, 0, p.st, 1u << 20);
  } else if (warp >= 2) {
    // ---------------- epilogue: 128 threads, one output row each ----------------
    const int quad = warp & 3;              // TMEM lanes 32*quad .. 32*quad+31
    const int row = 32 * quad + lane;
    const int kv_cols = p.n_kv_proj * kDkv;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int m, n;
      tile_coords(tile, num_m, num_n, m, n);
      if (!mbar_wait(&bars->abort, &bars->tfull[acc], acc_phase, p.st)) break;
      fence_after();
      const int t = m * BM + row;
      const bool in_t = t < p.T;  // rows past T are padding of the last M-tile
      const int32_t slot = in_t ? __ldg(p.slot_of_token + t) : -1;
      const bool slot_ok = in_t && slot >= 0 && slot < p.num_slots;
      if (in_t && !slot_ok) report(p.st, CSA2_DEV_BAD_SLOT);
      const uint32_t tbase = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(acc * BN);
      uint32_t sc[4] = {0, 0, 0, 0};
      const int col0 = n * BN;
      const bool kv_tile = col0 < kv_cols;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tbase + (uint32_t)(32 * ch), r);
        const int col = col0 + 32 * ch;
        if (!slot_ok || col >= p.n_out) continue;
        if (kv_tile) {
          const int proj = col / kDkv, c = col - proj * kDkv;
          uint32_t w[4];
          uint32_t s2 = 0;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(r[16 * g + i]);
            const uint32_t sb = quantize16(x, w[2 * g], w[2 * g + 1]);
            s2 |= sb << (8 * g);
          }
          uint8_t* crow = p.codes + ((int64_t)proj * p.num_slots + slot) * kCodeRow + c / 2;
          *reinterpret_cast<uint4*>(crow) = make_uint4(w[0], w[1], w[2], w[3]);
          const int sidx = (c / kGroup) & (BN / kGroup - 1);  // position within the tile's scales
          sc[sidx >> 2] |= s2 << (8 * (sidx & 3));
        } else {
          const int ic = col - kv_cols;
          const int proj = ic / kDidx, c = ic - proj * kDidx;
          uint32_t h[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            h[i] = f32_to_bf16_rn(__uint_as_float(r[2 * i])) |
                   (f32_to_bf16_rn(__uint_as_float(r[2 * i + 1])) << 16);
          uint4* krow = reinterpret_cast<uint4*>(
              p.k_idx + ((int64_t)proj * p.num_slots + slot) * kDidx + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) krow[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      if (kv_tile && slot_ok) {
        const int proj = col0 / kDkv, c = col0 - proj * kDkv;
        uint8_t* srow = p.scales + ((int64_t)proj * p.num_slots + slot) * kScaleRow + c / kGroup;
        if constexpr (BN == 256)
          *reinterpret_cast<uint4*>(srow) = make_uint4(sc[0], sc[1], sc[2], sc[3]);
        else
          *reinterpret_cast<uint2*>(srow) = make_uint2(sc[0], sc[1]);
      }
      fence_before();
      mbar_arrive(&bars->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

namespace {

template <int BN, int STAGES, int KSUB, int AROWS = BM>
cudaError_t launch_kv_write_cfg(const uint16_t* H, const uint16_t* Wt, const WriteParams& p,
                                cudaStream_t s, int num_sms) {
  CUtensorMap ta, tb;
  if (!make_bf16_map(&ta, H, p.T, p.d_model, BK, AROWS) ||
      !make_bf16_map(&tb, Wt, p.n_out, p.d_model, BK, BN))
    return cudaErrorInvalidValue;
  const size_t smem = KvCfg<BN, STAGES, KSUB, AROWS>::smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kv_write_kernel<BN, STAGES, KSUB, AROWS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = ((p.T + BM - 1) / BM) * ((p.n_out + BN - 1) / BN);
  const int grid = std::max(1, std::min(tiles, num_sms));
  kv_write_kernel<BN, STAGES, KSUB, AROWS><<<grid, kThreads, smem, s>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_write(const uint16_t* H, const uint16_t* Wt, uint8_t* codes, uint8_t* scales,
                            uint16_t* k_idx, int32_t T, int32_t d_model, int32_t n_kv_proj,
                            int32_t n_idx_proj, const int32_t* slot_of_token, int64_t num_slots,
                            int32_t* st, cudaStream_t s, int num_sms) {
  const int32_t n_out = n_kv_proj * kDkv + n_idx_proj * kDidx;
  WriteParams p{codes, scales, k_idx, slot_of_token, num_slots, T, d_model, n_kv_proj, n_idx_proj,
                n_out, st};
  if (T <= BM / 2 && d_model % (2 * BK) == 0) return launch_kv_write_cfg<128, 4, 2, BM / 2>(H, Wt, p, s, num_sms);
  if (T <= BM / 2) return launch_kv_write_cfg<128, 8, 1, BM / 2>(H, Wt, p, s, num_sms);
  if (T <= BM && d_model % (2 * BK) == 0) return launch_kv_write_cfg<128, 3, 2>(H, Wt, p, s, num_sms);
  if (T <= BM) return launch_kv_write_cfg<128, 6, 1>(H, Wt, p, s, num_sms);
  return launch_kv_write_cfg<256, 4, 1>(H, Wt, p, s, num_sms);
}

}  // namespace csa2
