// Shared device helpers of libcsa2 (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kPage = 64;      // tokens per page
constexpr int kDkv = 512;      // latent channels
constexpr int kGroup = 16;     // channels per E4M3 scale
constexpr int kDidx = 128;     // indexer head dim
constexpr int kHidx = 4;       // indexer heads
constexpr int kHq = 16;        // attention query heads
constexpr int kCodeRow = kDkv / 2;      // 256 B of codes per token
constexpr int kScaleRow = kDkv / kGroup;  // 32 B of scales per token
constexpr int kKeyRow = kDidx * 2;      // 256 B of bf16 key per token

// Iteration limit of every bounded spin (mbarrier try_wait loops).  try_wait itself
// suspends for a hardware-chosen interval, so this is seconds of real time.
constexpr uint32_t kSpinLimit = 1u << 26;

// ---- programmatic dependent launch ----
// Every kernel of the index and attention calls begins with grid_dep_wait() and is
// launched by launch_pdl.  The launch may then be processed while the previous kernel in
// the stream is still finishing; the wait (a no-op after an ordinary launch) returns once
// that kernel has completed and its writes are visible, so stream order is unchanged.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream be scheduled before this one completes; that kernel
// still waits (grid_dep_wait) for this one's completion before touching its results.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void report(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

// bf16x2 word -> two fp32 (low half = element 0).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed fp32x2 fused multiply-add (Blackwell FFMA2): acc += a * b lane-wise.
__device__ __forceinline__ void ffma2(unsigned long long& acc, unsigned long long a,
                                      unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo2(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(unsigned long long v) {
  return __uint_as_float((uint32_t)(v >> 32));
}

// ---- FP4 / FP8 conversions (hardware cvt, round-to-nearest-even, saturating) ----

// Two fp32 -> one byte of E2M1 codes: `lo` in bits 0..3, `hi` in bits 4..7.
// The magnitude comes from the hardware conversion of |x|; the sign bit is copied
// from x, so values that round to zero keep their sign.
__device__ __forceinline__ uint32_t e2m1x2_pack(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(fabsf(hi)), "f"(fabsf(lo)));
  uint32_t b = r & 0xFFu;
  b |= (__float_as_uint(lo) >> 31) << 3;
  b |= (__float_as_uint(hi) >> 31) << 7;
  return b;
}

// fp32 -> E4M3 byte (RNE, satfinite).
__device__ __forceinline__ uint32_t e4m3_encode(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// E4M3 byte -> fp32 (exact, via f16).
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  uint32_t h2;
  uint16_t in = (uint16_t)(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// One byte of two E2M1 codes -> f16x2 (low nibble -> low half), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h2;
  uint16_t in = (uint16_t)(byte & 0xFFu);
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
  return h2;
}

// Quantise 16 fp32 channels: returns the E4M3 scale byte and writes 8 code bytes
// (two 32-bit words, channel 2j in the low nibble of byte j).
//   s = E4M3(amax / 6), y = x / decode(s) (IEEE division), code = E2M1(y);
//   decode(s) == 0 -> all codes 0.
__device__ __forceinline__ uint32_t quantize16(const float (&x)[16], uint32_t& w0, uint32_t& w1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t sb = e4m3_encode(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_decode(sb);
  uint32_t w[2] = {0u, 0u};
  if (s > 0.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = e2m1x2_pack(__fdiv_rn(x[2 * j], s), __fdiv_rn(x[2 * j + 1], s));
      w[j >> 2] |= b << (8 * (j & 3));
    }
  }
  w0 = w[0];
  w1 = w[1];
  return sb;
}

// bf16 round-to-nearest-even of an fp32 (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16_rn(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// Slot of logical token t of sequence b; -1 (and a fault bit) when the page id is bad.
__device__ __forceinline__ int64_t token_slot(const int32_t* __restrict__ page_table,
                                              int32_t max_pages, int32_t num_pages, int b, int t,
                                              int32_t* st) {
  const int32_t pg = __ldg(page_table + (int64_t)b * max_pages + (t >> 6));
  if (pg < 0 || pg >= num_pages) {
    report(st, CSA2_DEV_BAD_PAGE);
    return -1;
  }
  return (int64_t)pg * kPage + (t & (kPage - 1));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace csa2
