// Persistent KV tier: export and import of whole cache pages.
//
// zaikei.co.jp article, opening section: the persistent KV cache used to resume sessions
// lives on SSD or in host memory.  Tech-report digest (jiwasawa.github.io), "FP4 メイン KV
// Cache と SWA Bounded Replay": the sliding-window KV is left out of it, so what persists
// is the global cache -- the FP4 latent pages (codes and scales) and the indexer-key pages.
//
// Packed layout, one record per exported page, in the order of page_ids:
//   codes [64][256] u8 | scales [64][S] u8 | keys [64][128] bf16
// with S = 32 (E4M3 per 16 channels) or 16 (the MXFP4 variant, E8M0 per 32 channels).
// One CTA copies one page with 16-byte loads and stores, every thread issuing all its
// loads (up to 9) before its stores; memory-bound (the record's bytes are read once and
// written once).
#include <algorithm>

#include "common.cuh"

namespace csa2 {

constexpr int kPageThreads = 256;

__host__ __device__ constexpr int64_t page_record_bytes(int scale_row) {
  return (int64_t)kPage * (kCodeRow + scale_row + kDidx * 2);
}

// 16-byte vectors of a record: codes, then scales, then keys.  The pool side of vector i
// lies in one of the page's three regions.
__device__ __forceinline__ uint4* pool_vec(uint8_t* pc, uint8_t* ps, uint8_t* pk, int scale_row,
                                           int i) {
  constexpr int kCodeVecs = kPage * kCodeRow / 16;  // 1024
  const int scale_vecs = kPage * scale_row / 16;    // 128 or 64
  if (i < kCodeVecs) return reinterpret_cast<uint4*>(pc) + i;
  if (i < kCodeVecs + scale_vecs) return reinterpret_cast<uint4*>(ps) + (i - kCodeVecs);
  return reinterpret_cast<uint4*>(pk) + (i - kCodeVecs - scale_vecs);
}

constexpr int kMaxVecs = (int)(page_record_bytes(32) / 16);                   // 2176
constexpr int kVecsPerThread = (kMaxVecs + kPageThreads - 1) / kPageThreads;  // 9

template <bool kExport>
__global__ void __launch_bounds__(kPageThreads) page_copy_kernel(
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, uint8_t* __restrict__ keys,
    int scale_row, int64_t num_pages, const int32_t* __restrict__ page_ids, int32_t n_pages,
    uint8_t* __restrict__ packed, int32_t* st) {
  const int64_t rec = page_record_bytes(scale_row);
  const int nvec = (int)(rec / 16);
  for (int64_t p = blockIdx.x; p < n_pages; p += gridDim.x) {
    const int32_t pg = __ldg(page_ids + p);
    uint4* r = reinterpret_cast<uint4*>(packed + p * rec);
    if (pg < 0 || pg >= num_pages) {
      if (threadIdx.x == 0) report(st, CSA2_DEV_BAD_PAGE);
      if (kExport) {  // a bad page exports as zeros
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) r[i] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    uint8_t* pc = codes + (int64_t)pg * kPage * kCodeRow;
    uint8_t* ps = scales + (int64_t)pg * kPage * scale_row;
    uint8_t* pk = keys + (int64_t)pg * kPage * kDidx * 2;
    // every load of the thread's vectors first, then the stores
    uint4 v[kVecsPerThread];
#pragma unroll
    for (int j = 0; j < kVecsPerThread; ++j) {
      const int i = threadIdx.x + j * kPageThreads;
      if (i < nvec) v[j] = __ldcs(kExport ? pool_vec(pc, ps, pk, scale_row, i) : r + i);
    }
#pragma unroll
    for (int j = 0; j < kVecsPerThread; ++j) {
      const int i = threadIdx.x + j * kPageThreads;
      if (i < nvec) *(kExport ? r + i : pool_vec(pc, ps, pk, scale_row, i)) = v[j];
    }
  }
}

size_t page_export_bytes(int scale_row) { return (size_t)page_record_bytes(scale_row); }

cudaError_t launch_page_copy(bool do_export, uint8_t* codes, uint8_t* scales, uint8_t* keys,
                             int scale_row, int64_t num_pages, const int32_t* page_ids,
                             int32_t n_pages, uint8_t* packed, int32_t* st, cudaStream_t s,
                             int num_sms) {
  const int grid = std::max(1, std::min<int>(n_pages, num_sms * 8));
  if (do_export)
    page_copy_kernel<true><<<grid, kPageThreads, 0, s>>>(codes, scales, keys, scale_row, num_pages,
                                                         page_ids, n_pages, packed, st);
  else
    page_copy_kernel<false><<<grid, kPageThreads, 0, s>>>(codes, scales, keys, scale_row, num_pages,
                                                          page_ids, n_pages, packed, st);
  return cudaGetLastError();
}

}  // namespace csa2
