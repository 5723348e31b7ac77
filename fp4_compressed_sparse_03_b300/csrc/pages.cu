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
// One CTA copies one page with 16-byte loads and stores; memory-bound (the record's bytes
// are read once and written once).
#include <algorithm>

#include "common.cuh"

namespace csa2 {

constexpr int kPageThreads = 256;

__host__ __device__ constexpr int64_t page_record_bytes(int scale_row) {
  return (int64_t)kPage * (kCodeRow + scale_row + kDidx * 2);
}

// Copy `bytes` (a multiple of 16) from src to dst with the CTA's threads.
__device__ __forceinline__ void copy_block(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                           int64_t bytes) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int64_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) d[i] = __ldcs(s + i);
}

template <bool kExport>
__global__ void __launch_bounds__(kPageThreads) page_copy_kernel(
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, uint8_t* __restrict__ keys,
    int scale_row, int64_t num_pages, const int32_t* __restrict__ page_ids, int32_t n_pages,
    uint8_t* __restrict__ packed, int32_t* st) {
  const int64_t rec = page_record_bytes(scale_row);
  for (int64_t i = blockIdx.x; i < n_pages; i += gridDim.x) {
    const int32_t pg = __ldg(page_ids + i);
    uint8_t* r = packed + i * rec;
    uint8_t* rc = r;
    uint8_t* rs = rc + kPage * kCodeRow;
    uint8_t* rk = rs + kPage * scale_row;
    if (pg < 0 || pg >= num_pages) {
      if (threadIdx.x == 0) report(st, CSA2_DEV_BAD_PAGE);
      if (kExport) {  // a bad page exports as zeros
        for (int64_t j = threadIdx.x; j < rec / 16; j += blockDim.x)
          reinterpret_cast<uint4*>(r)[j] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    uint8_t* pc = codes + (int64_t)pg * kPage * kCodeRow;
    uint8_t* ps = scales + (int64_t)pg * kPage * scale_row;
    uint8_t* pk = keys + (int64_t)pg * kPage * kDidx * 2;
    if (kExport) {
      copy_block(rc, pc, kPage * kCodeRow);
      copy_block(rs, ps, kPage * scale_row);
      copy_block(rk, pk, kPage * kDidx * 2);
    } else {
      copy_block(pc, rc, kPage * kCodeRow);
      copy_block(ps, rs, kPage * scale_row);
      copy_block(pk, rk, kPage * kDidx * 2);
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
