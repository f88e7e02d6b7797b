// noalloc.cu - attn_bwd_noalloc: the key pass and the dQ pass with their dS
// scratch in a static device array, for callers that may not allocate
// device memory while they run (see include/attn.h for who and why).
//
// The array below is a host-side stand-in in host code, not a device
// address: host code must never hand its name to a kernel.  Its device
// address is looked up with cudaGetSymbolAddress, with the device current,
// the first time a call runs in a device's context, and cached per context:
// a device reset (or a released and re-created primary context) loads the
// module again, possibly at another address, so a new context looks the
// address up again.  A failed lookup is not cached.
#include <mutex>

#include "attn_internal.h"

namespace css {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// Unique id of the calling thread's current context (0 if none or unknown).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id = 0;  // context the cached address belongs to
  uint8_t* ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_slots_mu;

// Device address of the scratch in the current device's current context.
int scratch_address(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_slots_mu);
  ScratchSlot& slot = g_slots[dev];
  if (id == 0 || slot.ptr == nullptr || slot.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (p == nullptr) return ATTN_ERR_CUDA;
    slot.ptr = static_cast<uint8_t*>(p);
    slot.ctx_id = id;
  }
  *out = slot.ptr;
  return ATTN_OK;
}

}  // namespace
}  // namespace css

using namespace css;

extern "C" ATTN_API int attn_bwd_noalloc(const attn_shape* shape, const uint16_t* q,
                                         const uint16_t* k, const uint16_t* vt,
                                         const uint16_t* dout, const float* lse,
                                         const float* delta, float* dq, float* dk, float* dvt,
                                         void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!q || !k || !vt || !dout || !lse || !delta || !dq || !dk || !dvt) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(dq) || !aligned16(dk) || !aligned16(dvt))
    return ATTN_ERR_ALIGN;
  // The kernels keep a K/V head's whole query group together, so one K/V
  // head's share of the dS tiles must fit the array.
  Dims one = d;
  one.kv_count = 1;
  const size_t per_head = workspace_bytes_for(one);
  if (per_head > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH_LIMIT;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  uint8_t* ws = nullptr;
  if ((rc = scratch_address(&ws)) != ATTN_OK) return rc;
  const int fit = static_cast<int>(ATTN_NOALLOC_SCRATCH_BYTES / per_head);
  const int end = d.kv_begin + d.kv_count;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int h0 = d.kv_begin; h0 < end; h0 += fit) {
    Dims c = d;
    c.kv_begin = h0;
    c.kv_count = end - h0 < fit ? end - h0 : fit;
    if ((rc = launch_bwd_keys(c, ctx, q, k, vt, dout, lse, delta, ws, dk, dvt, st)) != ATTN_OK)
      return rc;
    if ((rc = launch_bwd_queries(c, ctx, k, ws, dq, st)) != ATTN_OK) return rc;
  }
  return ATTN_OK;
}
