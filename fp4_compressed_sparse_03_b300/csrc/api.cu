// libcsa2 C ABI: argument validation, workspace sizing and kernel launches.
// The declarations and their contracts are in include/csa2.h.
#include <algorithm>
#include <cstring>

#include "common.cuh"

namespace csa2 {
cudaError_t launch_quantize(const float*, const int32_t*, uint8_t*, uint8_t*, int32_t, int32_t,
                            int64_t, int32_t*, cudaStream_t, int);
cudaError_t launch_dequantize(const uint8_t*, const uint8_t*, const int32_t*, float*, int32_t,
                              int32_t, int64_t, int32_t*, cudaStream_t, int);
cudaError_t launch_quantize_mx(const float*, const int32_t*, uint8_t*, uint8_t*, int32_t, int32_t,
                               int64_t, int32_t*, cudaStream_t, int);
cudaError_t launch_dequantize_mx(const uint8_t*, const uint8_t*, const int32_t*, float*, int32_t,
                                 int32_t, int64_t, int32_t*, cudaStream_t, int);
cudaError_t launch_score_full(const uint16_t*, const uint16_t*, const int32_t*, int32_t, int32_t,
                              const csa2_pages&, uint32_t*, int64_t, void*, uint32_t*, int32_t*,
                              cudaStream_t, int);
cudaError_t launch_score_reindex(const uint16_t*, const uint16_t*, const int32_t*, int32_t,
                                 const csa2_pages&, const int32_t*, int32_t, uint32_t*, int32_t*,
                                 cudaStream_t, int);
size_t runlist_bytes(int32_t num_q);
int32_t* runlist_order(void* base, int32_t num_q);
cudaError_t launch_select(bool, const uint32_t*, int64_t, const int32_t*, const csa2_pages&,
                          int32_t, const int32_t*, int32_t, int32_t, int32_t*, int32_t*,
                          const uint32_t*, void*, const int32_t*, int32_t*, cudaStream_t, int);
size_t wide_select_bytes(int32_t num_q, int32_t n);
cudaError_t launch_attn(const uint16_t*, const uint8_t*, const uint8_t*, const int32_t*,
                        const csa2_pages&, float*, float*, int32_t, const int32_t*, int32_t, float,
                        void*, int32_t*, cudaStream_t, int, bool);
size_t attn_workspace_bytes(int32_t, int32_t, int);
cudaError_t launch_chunk_attn(const uint16_t*, const uint8_t*, const uint8_t*, const int32_t*,
                              const csa2_pages&, float*, float*, int32_t, const int32_t*, int32_t,
                              int32_t, float, void*, int32_t*, cudaStream_t, int);
size_t chunk_attn_workspace_bytes(int32_t, int32_t, int32_t, int);
int chunk_attn_max_union();
int chunk_attn_max_chunk();
size_t page_export_bytes(int);
cudaError_t launch_page_copy(bool, uint8_t*, uint8_t*, uint8_t*, int, int64_t, const int32_t*,
                             int32_t, uint8_t*, int32_t*, cudaStream_t, int);
cudaError_t launch_kv_write(const uint16_t*, const uint16_t*, uint8_t*, uint8_t*, uint16_t*,
                            int32_t, int32_t, int32_t, int32_t, const int32_t*, int64_t, int32_t*,
                            cudaStream_t, int);
cudaError_t launch_bounded_wait(int, uint32_t, int32_t*, cudaStream_t);
}  // namespace csa2

using namespace csa2;

namespace {

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa2_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return CSA2_OK;
  (void)cudaGetLastError();  // clear a sticky launch-configuration error
  return CSA2_ERR_CUDA;
}

csa2_status check_pages(const csa2_pages* pg) {
  if (pg == nullptr || pg->seq_lens == nullptr || pg->page_table == nullptr)
    return CSA2_ERR_INVALID_ARGUMENT;
  if (pg->page_size != kPage) return CSA2_ERR_UNSUPPORTED;
  if (pg->num_seqs < 1 || pg->max_pages_per_seq < 1 || pg->num_pages < 1)
    return CSA2_ERR_INVALID_ARGUMENT;
  if ((int64_t)pg->max_pages_per_seq * kPage > (int64_t)INT32_MAX / 2) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

}  // namespace

extern "C" {

int32_t csa2_version(void) { return 10000; }

const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARGUMENT: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported geometry";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_DEVICE_FAULT: return "device-detected fault (bad index, page or slot)";
    case CSA2_ERR_TIMEOUT: return "bounded device wait expired";
  }
  return "unknown status";
}

csa2_status csa2_quantize(const float* x, const int32_t* slot_of_token, uint8_t* codes,
                          uint8_t* scales, int32_t T, int32_t D, int64_t num_slots,
                          int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || D <= 0 || num_slots < 0) return CSA2_ERR_INVALID_ARGUMENT;
  if (D % kGroup != 0 || D > 4096) return CSA2_ERR_UNSUPPORTED;
  if (T == 0) return CSA2_OK;
  if (!x || !slot_of_token || !codes || !scales) return CSA2_ERR_INVALID_ARGUMENT;
  if (!al16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_quantize(x, slot_of_token, codes, scales, T, D, num_slots, dev_status,
                                   stream, device_sms()));
}

csa2_status csa2_dequantize(const uint8_t* codes, const uint8_t* scales,
                            const int32_t* slot_of_token, float* x, int32_t T, int32_t D,
                            int64_t num_slots, int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || D <= 0 || num_slots < 0) return CSA2_ERR_INVALID_ARGUMENT;
  if (D % kGroup != 0 || D > 4096) return CSA2_ERR_UNSUPPORTED;
  if (T == 0) return CSA2_OK;
  if (!x || !slot_of_token || !codes || !scales) return CSA2_ERR_INVALID_ARGUMENT;
  if (!al16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_dequantize(codes, scales, slot_of_token, x, T, D, num_slots, dev_status,
                                     stream, device_sms()));
}

csa2_status csa2_quantize_mx(const float* x, const int32_t* slot_of_token, uint8_t* codes,
                             uint8_t* scales, int32_t T, int32_t D, int64_t num_slots,
                             int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || D <= 0 || num_slots < 0) return CSA2_ERR_INVALID_ARGUMENT;
  if (D % 32 != 0 || D > 4096) return CSA2_ERR_UNSUPPORTED;
  if (T == 0) return CSA2_OK;
  if (!x || !slot_of_token || !codes || !scales) return CSA2_ERR_INVALID_ARGUMENT;
  if (!al16(x) || !al16(codes)) return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_quantize_mx(x, slot_of_token, codes, scales, T, D, num_slots,
                                      dev_status, stream, device_sms()));
}

csa2_status csa2_dequantize_mx(const uint8_t* codes, const uint8_t* scales,
                               const int32_t* slot_of_token, float* x, int32_t T, int32_t D,
                               int64_t num_slots, int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || D <= 0 || num_slots < 0) return CSA2_ERR_INVALID_ARGUMENT;
  if (D % 32 != 0 || D > 4096) return CSA2_ERR_UNSUPPORTED;
  if (T == 0) return CSA2_OK;
  if (!x || !slot_of_token || !codes || !scales) return CSA2_ERR_INVALID_ARGUMENT;
  if (!al16(x) || !al16(codes)) return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_dequantize_mx(codes, scales, slot_of_token, x, T, D, num_slots,
                                        dev_status, stream, device_sms()));
}

// Scores (one 32-bit key per candidate) followed, at a 256-byte boundary, by the FULL
// scorer's run list (the REINDEX work list is arithmetic).
static size_t scores_bytes(csa2_mode mode, int32_t num_q, int32_t max_pages_per_seq,
                           int32_t pool_size) {
  const size_t n = mode == CSA2_FULL ? (size_t)std::max(0, max_pages_per_seq) * kPage
                                     : (size_t)std::max(0, pool_size);
  return ((size_t)num_q * n * sizeof(uint32_t) + 255) / 256 * 256;
}

// The run list's span in the workspace, rounded to 256 B so that what follows it (the
// selection histograms, cleared with 16-byte stores) stays aligned.
static size_t runlist_span(int32_t num_q) { return (runlist_bytes(num_q) + 255) / 256 * 256; }

// FULL: per-query selection histograms (2048 bins) written by the scorer
static size_t hist_bytes(csa2_mode mode, int32_t num_q) {
  return mode == CSA2_FULL ? ((size_t)num_q * 2048 * sizeof(uint32_t) + 255) / 256 * 256 : 0;
}

// FULL over contexts beyond 2^18 tokens: candidate lists of the wide selection
static size_t wide_bytes(csa2_mode mode, int32_t num_q, int32_t max_pages_per_seq) {
  if (mode != CSA2_FULL) return 0;
  const int64_t n = (int64_t)std::max(0, max_pages_per_seq) * kPage;
  return (wide_select_bytes(num_q, (int32_t)std::min<int64_t>(n, INT32_MAX)) + 255) / 256 * 256;
}

size_t csa2_index_workspace_size(csa2_mode mode, int32_t num_q, int32_t max_pages_per_seq,
                                 int32_t pool_size) {
  if (num_q <= 0 || (mode != CSA2_FULL && mode != CSA2_REINDEX)) return 0;
  return scores_bytes(mode, num_q, max_pages_per_seq, pool_size) +
         (mode == CSA2_FULL ? runlist_span(num_q) : 0) + hist_bytes(mode, num_q) +
         wide_bytes(mode, num_q, max_pages_per_seq);
}

csa2_status csa2_index(csa2_mode mode, const uint16_t* q_idx, const uint16_t* k_idx, int32_t* pool,
                       int32_t topk, int32_t* out_idx, const csa2_pages* pages,
                       const csa2_index_args* args, cudaStream_t stream) {
  if (args == nullptr || out_idx == nullptr || topk < 1) return CSA2_ERR_INVALID_ARGUMENT;
  if (args->num_q < 1 || args->q_seq == nullptr) return CSA2_ERR_INVALID_ARGUMENT;
  if (mode == CSA2_REUSE) {
    if (args->inherit_idx == nullptr) return CSA2_ERR_INVALID_ARGUMENT;
    if (args->inherit_idx == out_idx) return CSA2_OK;
    return from_cuda(cudaMemcpyAsync(out_idx, args->inherit_idx,
                                     (size_t)args->num_q * topk * sizeof(int32_t),
                                     cudaMemcpyDeviceToDevice, stream));
  }
  if (mode != CSA2_FULL && mode != CSA2_REINDEX) return CSA2_ERR_INVALID_ARGUMENT;
  csa2_status ps = check_pages(pages);
  if (ps != CSA2_OK) return ps;
  if (!q_idx || !k_idx || !al16(q_idx) || !al16(k_idx)) return CSA2_ERR_INVALID_ARGUMENT;
  if (args->max_q_per_seq < 1 || args->max_q_per_seq > 4) return CSA2_ERR_UNSUPPORTED;
  const int32_t P = args->pool_size;
  const size_t need = csa2_index_workspace_size(mode, args->num_q, pages->max_pages_per_seq, P);
  if (args->workspace == nullptr || args->workspace_bytes < need || !al16(args->workspace))
    return CSA2_ERR_INVALID_ARGUMENT;
  if (args->num_q > 65535) return CSA2_ERR_UNSUPPORTED;  // grid.y of the selection
  const int sms = device_sms();
  uint32_t* ws = static_cast<uint32_t*>(args->workspace);
  cudaError_t e;
  if (mode == CSA2_FULL) {
    if (pool != nullptr && P < 1) return CSA2_ERR_INVALID_ARGUMENT;
    const int64_t stride = (int64_t)pages->max_pages_per_seq * kPage;
    void* rl = static_cast<char*>(args->workspace) +
               scores_bytes(mode, args->num_q, pages->max_pages_per_seq, P);
    uint32_t* hist = reinterpret_cast<uint32_t*>(static_cast<char*>(rl) + runlist_span(args->num_q));
    void* wide = wide_bytes(mode, args->num_q, pages->max_pages_per_seq) == 0
                     ? nullptr
                     : static_cast<void*>(reinterpret_cast<char*>(hist) + hist_bytes(mode, args->num_q));
    e = launch_score_full(q_idx, k_idx, args->q_seq, args->num_q, args->max_q_per_seq, *pages, ws,
                          stride, rl, hist, args->dev_status, stream, sms);
    if (e != cudaSuccess) return from_cuda(e);
    e = launch_select(false, ws, stride, args->q_seq, *pages, args->num_q, nullptr,
                      pool ? P : 0, topk, out_idx, pool, hist, wide, runlist_order(rl, args->num_q),
                      args->dev_status, stream, sms);
    return from_cuda(e);
  }
  // REINDEX
  if (pool == nullptr || P < 1) return CSA2_ERR_INVALID_ARGUMENT;
  e = launch_score_reindex(q_idx, k_idx, args->q_seq, args->num_q, *pages, pool, P, ws,
                           args->dev_status, stream, sms);
  if (e != cudaSuccess) return from_cuda(e);
  e = launch_select(true, ws, P, args->q_seq, *pages, args->num_q, pool, P, topk, out_idx, nullptr,
                    nullptr, nullptr, nullptr, args->dev_status, stream, sms);
  return from_cuda(e);
}

size_t csa2_attn_workspace_size(int32_t num_q, int32_t topk) {
  if (num_q <= 0 || topk <= 0) return 0;
  return attn_workspace_bytes(num_q, topk, device_sms());
}

// csa2_sparse_attn and its MXFP4 variant: the same checks, the scale format chosen by `mx`.
static csa2_status sparse_attn_call(bool mx, const uint16_t* q, const uint8_t* codes,
                                    const uint8_t* scales, const int32_t* idx,
                                    const csa2_pages* pages, float* out, float* lse, int32_t num_q,
                                    const int32_t* q_seq, int32_t topk, float softmax_scale,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    cudaStream_t stream) {
  if (num_q < 1 || topk < 1 || !q || !codes || !scales || !idx || !out || !q_seq)
    return CSA2_ERR_INVALID_ARGUMENT;
  csa2_status ps = check_pages(pages);
  if (ps != CSA2_OK) return ps;
  if (!al16(q) || !al16(codes) || !al16(scales) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return CSA2_ERR_INVALID_ARGUMENT;
  if (!(softmax_scale == softmax_scale)) return CSA2_ERR_INVALID_ARGUMENT;
  if (num_q > 65535 || topk > CSA2_ATTN_MAX_TOPK) return CSA2_ERR_UNSUPPORTED;
  const int sms = device_sms();
  const size_t need = attn_workspace_bytes(num_q, topk, sms);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !al16(workspace)))
    return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_attn(q, codes, scales, idx, *pages, out, lse, num_q, q_seq, topk,
                               softmax_scale, workspace, dev_status, stream, sms, mx));
}

csa2_status csa2_sparse_attn(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                             const int32_t* idx, const csa2_pages* pages, float* out, float* lse,
                             int32_t num_q, const int32_t* q_seq, int32_t topk, float softmax_scale,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             cudaStream_t stream) {
  return sparse_attn_call(false, q, codes, scales, idx, pages, out, lse, num_q, q_seq, topk,
                          softmax_scale, workspace, workspace_bytes, dev_status, stream);
}

csa2_status csa2_sparse_attn_mx(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                                const int32_t* idx, const csa2_pages* pages, float* out,
                                float* lse, int32_t num_q, const int32_t* q_seq, int32_t topk,
                                float softmax_scale, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, cudaStream_t stream) {
  return sparse_attn_call(true, q, codes, scales, idx, pages, out, lse, num_q, q_seq, topk,
                          softmax_scale, workspace, workspace_bytes, dev_status, stream);
}

static bool chunk_args_ok(int32_t num_q, int32_t chunk, int32_t topk) {
  return num_q >= 1 && chunk >= 1 && topk >= 1 && num_q % chunk == 0;
}

static bool chunk_args_supported(int32_t num_q, int32_t chunk, int32_t topk) {
  return chunk <= chunk_attn_max_chunk() && (int64_t)chunk * topk <= chunk_attn_max_union() &&
         num_q / chunk <= 65535;
}

size_t csa2_chunk_attn_workspace_size(int32_t num_q, int32_t chunk, int32_t topk) {
  if (!chunk_args_ok(num_q, chunk, topk) || !chunk_args_supported(num_q, chunk, topk)) return 0;
  return chunk_attn_workspace_bytes(num_q, chunk, topk, device_sms());
}

csa2_status csa2_sparse_attn_chunked(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                                     const int32_t* idx, const csa2_pages* pages, float* out,
                                     float* lse, int32_t num_q, const int32_t* q_seq, int32_t chunk,
                                     int32_t topk, float softmax_scale, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_status,
                                     cudaStream_t stream) {
  if (!chunk_args_ok(num_q, chunk, topk) || !q || !codes || !scales || !idx || !out || !q_seq)
    return CSA2_ERR_INVALID_ARGUMENT;
  csa2_status ps = check_pages(pages);
  if (ps != CSA2_OK) return ps;
  if (!al16(q) || !al16(codes) || !al16(scales) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return CSA2_ERR_INVALID_ARGUMENT;
  if (!(softmax_scale == softmax_scale)) return CSA2_ERR_INVALID_ARGUMENT;
  if (!chunk_args_supported(num_q, chunk, topk)) return CSA2_ERR_UNSUPPORTED;
  const int sms = device_sms();
  const size_t need = chunk_attn_workspace_bytes(num_q, chunk, topk, sms);
  if (workspace == nullptr || workspace_bytes < need || !al16(workspace))
    return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_chunk_attn(q, codes, scales, idx, *pages, out, lse, num_q, q_seq, chunk,
                                     topk, softmax_scale, workspace, dev_status, stream, sms));
}

csa2_status csa2_kv_write(const uint16_t* H, const uint16_t* Wt, uint8_t* codes, uint8_t* scales,
                          uint16_t* k_idx, int32_t T, int32_t d_model, int32_t n_kv_proj,
                          int32_t n_idx_proj, const int32_t* slot_of_token, int64_t num_slots,
                          int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || d_model <= 0 || n_kv_proj < 0 || n_idx_proj < 0 || num_slots < 0)
    return CSA2_ERR_INVALID_ARGUMENT;
  if (n_kv_proj + n_idx_proj == 0 || T == 0) return CSA2_OK;
  if (!H || !Wt || !slot_of_token) return CSA2_ERR_INVALID_ARGUMENT;
  if (n_kv_proj > 0 && (!codes || !scales)) return CSA2_ERR_INVALID_ARGUMENT;
  if (n_idx_proj > 0 && !k_idx) return CSA2_ERR_INVALID_ARGUMENT;
  if (!al16(H) || !al16(Wt) || (codes && (reinterpret_cast<uintptr_t>(codes) & 7u)) ||
      (k_idx && !al16(k_idx)))
    return CSA2_ERR_INVALID_ARGUMENT;
  if (d_model % 64 != 0) return CSA2_ERR_UNSUPPORTED;
  return from_cuda(launch_kv_write(H, Wt, codes, scales, k_idx, T, d_model, n_kv_proj, n_idx_proj,
                                   slot_of_token, num_slots, dev_status, stream, device_sms()));
}

size_t csa2_page_export_bytes(int32_t scale_row_bytes) {
  if (scale_row_bytes != 32 && scale_row_bytes != 16) return 0;
  return page_export_bytes(scale_row_bytes);
}

static csa2_status page_copy_call(bool do_export, const uint8_t* codes, const uint8_t* scales,
                                  const uint16_t* keys, int32_t scale_row_bytes, int64_t num_pages,
                                  const int32_t* page_ids, int32_t n_pages, const uint8_t* packed,
                                  int32_t* dev_status, cudaStream_t stream) {
  if (n_pages < 0 || num_pages < 0) return CSA2_ERR_INVALID_ARGUMENT;
  if (scale_row_bytes != 32 && scale_row_bytes != 16) return CSA2_ERR_UNSUPPORTED;
  if (n_pages == 0) return CSA2_OK;
  if (!codes || !scales || !keys || !page_ids || !packed) return CSA2_ERR_INVALID_ARGUMENT;
  if (!al16(codes) || !al16(scales) || !al16(keys) || !al16(packed))
    return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_page_copy(do_export, const_cast<uint8_t*>(codes),
                                    const_cast<uint8_t*>(scales),
                                    reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(keys)),
                                    scale_row_bytes, num_pages, page_ids, n_pages,
                                    const_cast<uint8_t*>(packed), dev_status, stream, device_sms()));
}

csa2_status csa2_export_pages(const uint8_t* codes, const uint8_t* scales, const uint16_t* keys,
                              int32_t scale_row_bytes, int64_t num_pages, const int32_t* page_ids,
                              int32_t n_pages, uint8_t* packed, int32_t* dev_status,
                              cudaStream_t stream) {
  return page_copy_call(true, codes, scales, keys, scale_row_bytes, num_pages, page_ids, n_pages,
                        packed, dev_status, stream);
}

csa2_status csa2_import_pages(const uint8_t* packed, int32_t scale_row_bytes,
                              const int32_t* page_ids, int32_t n_pages, int64_t num_pages,
                              uint8_t* codes, uint8_t* scales, uint16_t* keys, int32_t* dev_status,
                              cudaStream_t stream) {
  return page_copy_call(false, codes, scales, keys, scale_row_bytes, num_pages, page_ids, n_pages,
                        packed, dev_status, stream);
}

csa2_status csa2_read_status(int32_t* dev_status, int32_t* host_bits, cudaStream_t stream) {
  if (dev_status == nullptr) return CSA2_ERR_INVALID_ARGUMENT;
  int32_t bits = 0;
  cudaError_t e = cudaMemcpyAsync(&bits, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return from_cuda(e);
  if (host_bits) *host_bits = bits;
  if (bits & CSA2_DEV_TIMEOUT) return CSA2_ERR_TIMEOUT;
  if (bits) return CSA2_ERR_DEVICE_FAULT;
  return CSA2_OK;
}

csa2_status csa2_check_bounded_wait(int32_t arrive, uint32_t limit, int32_t* dev_status,
                                    cudaStream_t stream) {
  if (dev_status == nullptr || limit < 1 || limit > (1u << 20)) return CSA2_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_bounded_wait(arrive != 0, limit, dev_status, stream));
}

}  // extern "C"
