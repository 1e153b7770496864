// noalloc.cu -- forward entry point for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: code that runs while a CUDA graph
// is being captured (an allocation there is not allowed), plugins inside a host
// framework that owns every device allocation through its own pool, and
// latency-critical loops where an allocation's implicit synchronisation is not
// acceptable.  nsa_sel_attn_fwd_noalloc serves them: it runs the same forward as
// nsa_sel_attn_fwd, but its scratch (index tensors and partial outputs) lives in
// the fixed array below, which is part of the library image.  Every GPU that
// loads the library holds this array until the process exits.
#include <mutex>

#include "common.cuh"

namespace {

// Fixed scratch of the no-allocation forward (NSA_NOALLOC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_noalloc_scratch[NSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the context the address was looked up in, and the address.  A new
// primary context (after cudaDeviceReset, say) loads the module again and the
// array may move, so the lookup is repeated whenever the current context changes.
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};
void *g_scratch_addr[kMaxDevices] = {nullptr};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// Device address of the array in the current context.  The name g_noalloc_scratch
// in host code is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with the device (and its context) current.
nsa_status scratch_for_current_device(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NSA_ERR_CUDA;
  static const CtxGetCurrentFn ctx_get = nsa::driver_entry<CtxGetCurrentFn>("cuCtxGetCurrent");
  if (!ctx_get) return NSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  CUcontext ctx = nullptr;
  if (ctx_get(&ctx) != CUDA_SUCCESS) return NSA_ERR_CUDA;
  if (ctx == nullptr || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    // The lookup also makes the device's primary context current if none was.
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return NSA_ERR_CUDA;
    if (ctx_get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return NSA_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *addr = g_scratch_addr[dev];
  return NSA_OK;
}

}  // namespace

extern "C" {

nsa_status nsa_sel_attn_fwd_noalloc(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                                    const void *v, const int32_t *sel_idx,
                                    const int32_t *cu_seqlens, float scale, void *out,
                                    float *lse, nsa_stream_t stream) {
  size_t need = 0;
  nsa_status st = nsa_sel_attn_workspace_size(dims, &need, nullptr);
  if (st != NSA_OK) return st;
  if (need > static_cast<size_t>(NSA_NOALLOC_SCRATCH_BYTES)) return NSA_ERR_WORKSPACE;
  void *scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != NSA_OK) return st;
  // The forward clears the status word itself and writes every index entry and
  // every partial row it later reads, so nothing else needs zeroing here.
  return nsa_sel_attn_fwd(dims, q, k, v, sel_idx, cu_seqlens, scale, out, lse, scratch,
                          static_cast<size_t>(NSA_NOALLOC_SCRATCH_BYTES), stream);
}

// Status word of the fixed scratch: the same word, at the same place, that
// nsa_sel_attn_get_status reads in a caller-provided workspace.
nsa_status nsa_sel_attn_fwd_noalloc_status(const nsa_sel_attn_dims *dims, nsa_stream_t stream,
                                           int32_t *bits) {
  size_t need = 0;
  nsa_status st = nsa_sel_attn_workspace_size(dims, &need, nullptr);
  if (st != NSA_OK) return st;
  if (need > static_cast<size_t>(NSA_NOALLOC_SCRATCH_BYTES)) return NSA_ERR_WORKSPACE;
  void *scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != NSA_OK) return st;
  return nsa_sel_attn_get_status(dims, scratch, stream, bits);
}

}  // extern "C"
