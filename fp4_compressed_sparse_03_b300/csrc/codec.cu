// Standalone FP4 codec kernels: quantise fp32 latent rows into the paged code/scale
// pools, and dequantise them back.  Format: E2M1 codes, one E4M3 scale per 16
// channels (ai2.x.ezic.info blog, section "KVを捨てる、共有する、作り直す").
// Memory-bound: one thread per 16-channel block, 64 B in, 9 B out.
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
