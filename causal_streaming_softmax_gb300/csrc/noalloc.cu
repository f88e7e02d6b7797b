// noalloc.cu - attn_bwd_noalloc: the key pass and the dQ pass with their dS
// scratch in a static device array, for callers that may not allocate
// device memory while they run (see include/attn.h for who and why).
//
// The array below is a host-side stand-in in host code, not a device
// address: host code must never hand its name to a kernel.  Its device
// address is looked up with cudaGetSymbolAddress once per device (with that
// device current) and cached; that pointer is what the kernels receive.
#include <mutex>

#include "attn_internal.h"

namespace css {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  std::once_flag once;
  cudaError_t status = cudaErrorUnknown;
  uint8_t* ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the scratch on the current device.
int scratch_address(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  ScratchSlot& slot = g_slots[dev];
  std::call_once(slot.once, [&slot] {
    void* p = nullptr;
    slot.status = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    slot.ptr = static_cast<uint8_t*>(p);
  });
  if (slot.status != cudaSuccess || slot.ptr == nullptr) return ATTN_ERR_CUDA;
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
