// csa2_sparse_attn_static: the read path with its split-softmax partials held in a
// fixed device array of this library instead of caller-provided workspace.
//
// For callers that cannot allocate device memory around the call: plain C clients of
// the ABI that hold no device allocator of their own, and decode loops that must not
// call cudaMalloc / cudaFree while kernels are in flight, because those calls can
// synchronise the device and stall the whole step.
//
// The partials of every split (16 x 512 fp32 output rows plus the running max and sum
// of each head) are written in full by the attention kernel before the combine kernel
// reads them, so nothing in the array has to start at zero and no clearing pass runs.
// The array is shared by every call on a device: calls that overlap in time (on two
// streams, or from two host threads) race on it.  Being a module global, its 16 MiB are
// reserved on every device where the module of this file is loaded: under lazy module
// loading (the CUDA default) at the first call of this entry point on the device (the
// module holds no kernel, only the array), and under CUDA_MODULE_LOADING=EAGER at
// context creation, whether or not this entry point is ever called.
#include <cuda.h>

#include <mutex>

#include "csa2.h"

static __device__ __align__(256) unsigned char g_attn_scratch[CSA2_ATTN_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// Per device: the context the address was resolved in, and the address.  A context that
// was destroyed and recreated (cudaDeviceReset) reloads this module at a new address, so
// the address is resolved again whenever the current context differs from the recorded one.
CUcontext g_scratch_ctx[kMaxDevices] = {};
void* g_scratch_ptr[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  }
  return fn;
}

// Device address of g_attn_scratch in the current device's current context, resolved on
// the first call made in that context.
csa2_status scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return CSA2_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return CSA2_ERR_UNSUPPORTED;
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return CSA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  // cudaGetSymbolAddress makes the device's primary context current if none is
  // (a first runtime call), so the context is read after it when it is resolved
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return CSA2_ERR_CUDA;
  if (g_scratch_ptr[dev] == nullptr || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return CSA2_ERR_CUDA;
    }
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return CSA2_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return CSA2_OK;
}

}  // namespace

extern "C" csa2_status csa2_sparse_attn_static(const uint16_t* q, const uint8_t* codes,
                                                const uint8_t* scales, const int32_t* idx,
                                                const csa2_pages* pages, float* out, float* lse,
                                                int32_t num_q, const int32_t* q_seq, int32_t topk,
                                                float softmax_scale, int32_t* dev_status,
                                                cudaStream_t stream) {
  if (num_q < 1 || topk < 1) return CSA2_ERR_INVALID_ARGUMENT;
  if (topk > CSA2_ATTN_MAX_TOPK) return CSA2_ERR_UNSUPPORTED;
  if (csa2_attn_workspace_size(num_q, topk) > (size_t)CSA2_ATTN_STATIC_SCRATCH_BYTES)
    return CSA2_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const csa2_status s = scratch_of_current_device(&scratch);
  if (s != CSA2_OK) return s;
  return csa2_sparse_attn(q, codes, scales, idx, pages, out, lse, num_q, q_seq, topk,
                          softmax_scale, scratch, (size_t)CSA2_ATTN_STATIC_SCRATCH_BYTES,
                          dev_status, stream);
}
