// Seeded synthetic inputs: the counter-based generator of csa2_inputs/gen.py in C
// (host, OpenMP threads) and CUDA (device).  Same definition, bit for bit:
//   mix64     SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014)
//   draw(j)   mix64(key + (j + 1) * 0x9E3779B97F4A7C15)
//   normal(i) twelve 16-bit integers from draws 3i..3i+2, S = their sum,
//             value = (2 S - 786420) * 2^-17 (an exact float32)
//   bf16      round-to-nearest-even of the float32 bits
// This file holds no arithmetic of the method; it only fills buffers with draws.
#include <cuda_runtime.h>
#include <omp.h>
#include <string.h>
#include <stdint.h>

#define HD __host__ __device__ __forceinline__

namespace {

HD uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

HD uint64_t draw(uint64_t key, uint64_t j) { return mix64(key + (j + 1) * 0x9E3779B97F4A7C15ull); }

HD float normal(uint64_t key, uint64_t i) {
  int64_t s = 0;
  for (int r = 0; r < 3; ++r) {
    const uint64_t d = draw(key, 3 * i + r);
    s += (int64_t)(d & 0xFFFF) + (int64_t)((d >> 16) & 0xFFFF) + (int64_t)((d >> 32) & 0xFFFF) +
         (int64_t)(d >> 48);
  }
  // |2S - 786420| < 2^20: exact in float32; the power-of-two factor is exact too
  return (float)(2 * s - 786420) * (1.0f / 131072.0f);
}

HD uint16_t bf16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

HD float pow2f(int e) {  // exact 2^e for -126 <= e <= 127
  uint32_t u = (uint32_t)(127 + e) << 23;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

__global__ void fill_bf16_kernel(uint64_t key, uint64_t i0, int64_t n, int pow2, uint16_t* out) {
  const float sc = pow2f(pow2);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v = normal(key, i0 + (uint64_t)i);
    if (pow2) v = __fmul_rn(v, sc);
    out[i] = bf16_rne(v);
  }
}

__global__ void fill_latent_kernel(uint64_t key, int64_t t0, int64_t T, const float* gain,
                                   float* out) {
  const int64_t n = T * 512;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i >> 9;
    const int c = (int)(i & 511);
    out[i] = __fmul_rn(normal(key, (uint64_t)((t0 + t) * 512 + c)), gain[c]);
  }
}

// Indexer keys of every sequence, written straight into the paged key pool:
// pool[(page_table[b][t/64] * 64 + t%64) * 128 + d] = bf16(normal(seq_key[b], t*128 + d)).
__global__ void fill_keys_paged_kernel(const uint64_t* seq_key, const int32_t* seq_lens,
                                       const int32_t* page_table, int32_t max_pages,
                                       int32_t num_seqs, uint16_t* pool) {
  // grid.x: logical pages (all sequences), 128 threads: one token row of 128 dims per 8 threads
  const int64_t gp = blockIdx.x;
  const int b = (int)(gp / max_pages);
  const int p = (int)(gp - (int64_t)b * max_pages);
  if (b >= num_seqs) return;
  const int n = seq_lens[b];
  if (p * 64 >= n) return;
  const int32_t phys = page_table[(int64_t)b * max_pages + p];
  const uint64_t key = seq_key[b];
  for (int e = threadIdx.x; e < 64 * 16; e += blockDim.x) {
    const int r = e >> 4, chunk = e & 15;  // token row r of the page, 8 dims per chunk
    const int t = p * 64 + r;
    if (t >= n) continue;
    uint16_t v[8];
    for (int k = 0; k < 8; ++k) v[k] = bf16_rne(normal(key, (uint64_t)t * 128 + chunk * 8 + k));
    uint4 w;
    w.x = v[0] | ((uint32_t)v[1] << 16);
    w.y = v[2] | ((uint32_t)v[3] << 16);
    w.z = v[4] | ((uint32_t)v[5] << 16);
    w.w = v[6] | ((uint32_t)v[7] << 16);
    *reinterpret_cast<uint4*>(pool + ((int64_t)phys * 64 + r) * 128 + chunk * 8) = w;
  }
}

int blocks_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  if (b > 148 * 64) b = 148 * 64;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace

extern "C" {

// ---------------- host ----------------
void csa2g_fill_bf16_host(uint64_t key, uint64_t i0, int64_t n, int pow2, uint16_t* out) {
  const float sc = pow2f(pow2);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = normal(key, i0 + (uint64_t)i);
    if (pow2) v = v * sc;
    out[i] = bf16_rne(v);
  }
}

void csa2g_fill_latent_host(uint64_t key, int64_t t0, int64_t T, const float* gain, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < T * 512; ++i) {
    const int64_t t = i >> 9;
    const int c = (int)(i & 511);
    out[i] = normal(key, (uint64_t)((t0 + t) * 512 + c)) * gain[c];
  }
}

void csa2g_fill_normal_host(uint64_t key, uint64_t i0, int64_t n, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = normal(key, i0 + (uint64_t)i);
}

// ---------------- device (stream-ordered, asynchronous) ----------------
int csa2g_fill_bf16_dev(uint64_t key, uint64_t i0, int64_t n, int pow2, uint16_t* out,
                        cudaStream_t s) {
  if (n <= 0) return 0;
  fill_bf16_kernel<<<blocks_for(n), 256, 0, s>>>(key, i0, n, pow2, out);
  return (int)cudaGetLastError();
}

int csa2g_fill_latent_dev(uint64_t key, int64_t t0, int64_t T, const float* gain, float* out,
                          cudaStream_t s) {
  if (T <= 0) return 0;
  fill_latent_kernel<<<blocks_for(T * 512), 256, 0, s>>>(key, t0, T, gain, out);
  return (int)cudaGetLastError();
}

int csa2g_fill_keys_paged_dev(const uint64_t* seq_key, const int32_t* seq_lens,
                              const int32_t* page_table, int32_t max_pages, int32_t num_seqs,
                              uint16_t* pool, cudaStream_t s) {
  const int64_t grid = (int64_t)num_seqs * max_pages;
  if (grid <= 0) return 0;
  fill_keys_paged_kernel<<<(unsigned)grid, 128, 0, s>>>(seq_key, seq_lens, page_table, max_pages,
                                                         num_seqs, pool);
  return (int)cudaGetLastError();
}

}  // extern "C"
