// Standalone FP4 codec kernels: quantise fp32 latent rows into the paged code/scale
// pools, and dequantise them back.  Format: E2M1 codes, one E4M3 scale per 16
// channels (ai2.x.ezic.info blog, section "KVを捨てる、共有する、作り直す"), and the
// MXFP4 variant with one E8M0 scale per 32 channels.
// Memory-bound: one thread per 16-channel block, 64 B in, 9 B out (per 32-channel block,
// 128 B in, 17 B out, for MXFP4).
#include <algorithm>

#include "common.cuh"

namespace csa2 {

__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ x,
                                                       const int32_t* __restrict__ slot_of_token,
                                                       uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales, int32_t T,
                                                       int32_t D, int64_t num_slots, int32_t* st) {
  const int nb = D / kGroup;
  const int64_t total = (int64_t)T * nb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nb;
    const int j = (int)(i - t * nb);
    const int32_t slot = __ldg(slot_of_token + t);
    if (slot < 0 || slot >= num_slots) {
      report(st, CSA2_DEV_BAD_SLOT);
      continue;
    }
    const float4* src = reinterpret_cast<const float4*>(x + t * D + j * kGroup);
    float v[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 f = __ldcs(src + k);
      v[4 * k] = f.x;
      v[4 * k + 1] = f.y;
      v[4 * k + 2] = f.z;
      v[4 * k + 3] = f.w;
    }
    uint32_t w0, w1;
    const uint32_t sb = quantize16(v, w0, w1);
    *reinterpret_cast<uint2*>(codes + (int64_t)slot * (D / 2) + j * 8) = make_uint2(w0, w1);
    scales[(int64_t)slot * nb + j] = (uint8_t)sb;
  }
}

__global__ void __launch_bounds__(256) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         const int32_t* __restrict__ slot_of_token,
                                                         float* __restrict__ x, int32_t T, int32_t D,
                                                         int64_t num_slots, int32_t* st) {
  const int nb = D / kGroup;
  const int64_t total = (int64_t)T * nb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nb;
    const int j = (int)(i - t * nb);
    const int32_t slot = __ldg(slot_of_token + t);
    float4* dst = reinterpret_cast<float4*>(x + t * D + j * kGroup);
    if (slot < 0 || slot >= num_slots) {
      report(st, CSA2_DEV_BAD_SLOT);
      continue;
    }
    const uint2 w = *reinterpret_cast<const uint2*>(codes + (int64_t)slot * (D / 2) + j * 8);
    const float s = e4m3_decode(scales[(int64_t)slot * nb + j]);
    const uint32_t ws[2] = {w.x, w.y};
    float v[16];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t h2 = e2m1x2_to_f16x2((ws[b >> 2] >> (8 * (b & 3))) & 0xFFu);
      v[2 * b] = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * s;
      v[2 * b + 1] = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * s;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

// ---- MXFP4 variant ----
// Tech-report digest (jiwasawa.github.io), "FP4 メイン KV Cache と SWA Bounded Replay":
// the main KV in the OCP-standard MXFP4 format, E2M1 elements.  Read as OCP MX: one E8M0
// scale per 32 channels, X = 2^(floor(log2 amax) - 2) clamped to 2^-127 .. 2^127 (byte =
// exponent + 127); codes = E2M1_RNE_satfinite(x / X) with the sign kept; a block whose
// amax is 0 gets scale byte 0 and zero codes.  128 B in, 17 B out per block.

// floor(log2 a) of a finite a > 0, from its bits (subnormals included).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = (int)((b >> 23) & 0xFFu);
  if (e != 0) return e - 127;
  return (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
}

// 2^k as a float, k in [-127, 127] (2^-127 is subnormal, exact).
__device__ __forceinline__ float pow2f(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << 22);
}

__global__ void __launch_bounds__(256) quantize_mx_kernel(const float* __restrict__ x,
                                                          const int32_t* __restrict__ slot_of_token,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales, int32_t T,
                                                          int32_t D, int64_t num_slots,
                                                          int32_t* st) {
  const int nb = D / 32;
  const int64_t total = (int64_t)T * nb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nb;
    const int j = (int)(i - t * nb);
    const int32_t slot = __ldg(slot_of_token + t);
    if (slot < 0 || slot >= num_slots) {
      report(st, CSA2_DEV_BAD_SLOT);
      continue;
    }
    const float4* src = reinterpret_cast<const float4*>(x + t * D + j * 32);
    float v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 f = __ldcs(src + k);
      v[4 * k] = f.x;
      v[4 * k + 1] = f.y;
      v[4 * k + 2] = f.z;
      v[4 * k + 3] = f.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    uint32_t sb = 0;
    if (amax > 0.0f) {
      const int se = max(-127, min(127, floor_log2(amax) - 2));
      sb = (uint32_t)(se + 127);
      const float inv = pow2f(-se);  // x * 2^-se is exact: |x / X| < 8
#pragma unroll
      for (int k = 0; k < 16; ++k)
        w[k >> 2] |= e2m1x2_pack(v[2 * k] * inv, v[2 * k + 1] * inv) << (8 * (k & 3));
    }
    *reinterpret_cast<uint4*>(codes + (int64_t)slot * (D / 2) + j * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    scales[(int64_t)slot * nb + j] = (uint8_t)sb;
  }
}

__global__ void __launch_bounds__(256) dequantize_mx_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ scales,
                                                            const int32_t* __restrict__ slot_of_token,
                                                            float* __restrict__ x, int32_t T,
                                                            int32_t D, int64_t num_slots,
                                                            int32_t* st) {
  const int nb = D / 32;
  const int64_t total = (int64_t)T * nb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nb;
    const int j = (int)(i - t * nb);
    const int32_t slot = __ldg(slot_of_token + t);
    if (slot < 0 || slot >= num_slots) {
      report(st, CSA2_DEV_BAD_SLOT);
      continue;
    }
    const uint4 w4 = *reinterpret_cast<const uint4*>(codes + (int64_t)slot * (D / 2) + j * 16);
    const float X = pow2f((int)scales[(int64_t)slot * nb + j] - 127);
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
    float4* dst = reinterpret_cast<float4*>(x + t * D + j * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float v[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = 2 * q + h;
        const uint32_t h2 = e2m1x2_to_f16x2((w[b >> 2] >> (8 * (b & 3))) & 0xFFu);
        v[2 * h] = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * X;
        v[2 * h + 1] = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * X;
      }
      dst[q] = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
}

cudaError_t launch_quantize_mx(const float* x, const int32_t* slot, uint8_t* codes,
                               uint8_t* scales, int32_t T, int32_t D, int64_t num_slots,
                               int32_t* st, cudaStream_t s, int num_sms) {
  const int64_t total = (int64_t)T * (D / 32);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 8));
  quantize_mx_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, slot, codes, scales, T, D, num_slots, st);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_mx(const uint8_t* codes, const uint8_t* scales, const int32_t* slot,
                                 float* x, int32_t T, int32_t D, int64_t num_slots, int32_t* st,
                                 cudaStream_t s, int num_sms) {
  const int64_t total = (int64_t)T * (D / 32);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 8));
  dequantize_mx_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, scales, slot, x, T, D, num_slots, st);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const float* x, const int32_t* slot, uint8_t* codes, uint8_t* scales,
                            int32_t T, int32_t D, int64_t num_slots, int32_t* st, cudaStream_t s,
                            int num_sms) {
  const int64_t total = (int64_t)T * (D / kGroup);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, slot, codes, scales, T, D, num_slots, st);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const int32_t* slot,
                              float* x, int32_t T, int32_t D, int64_t num_slots, int32_t* st,
                              cudaStream_t s, int num_sms) {
  const int64_t total = (int64_t)T * (D / kGroup);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  dequantize_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, scales, slot, x, T, D, num_slots, st);
  return cudaGetLastError();
}

}  // namespace csa2
