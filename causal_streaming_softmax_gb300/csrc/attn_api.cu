// attn_api.cu - the C ABI: host-side admission checks, per-device context,
// tensor-map encoding, and dispatch to the kernel launchers.
#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "attn_internal.h"
#include "sm103.cuh"

namespace css {
namespace {

__device__ uint32_t g_device_error;

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

constexpr int kMaxDevices = 64;
struct DevState {
  std::once_flag once;
  int status = ATTN_ERR_CUDA;
  uint32_t* err = nullptr;
  int sm_count = 0;
};
DevState g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int device_context(DevCtx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  DevState& s = g_dev[dev];
  std::call_once(s.once, [&s, dev] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      s.status = ATTN_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      s.status = ATTN_ERR_DEVICE;
      return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      s.status = ATTN_ERR_CUDA;
      return;
    }
    s.err = static_cast<uint32_t*>(p);
    s.sm_count = sms;
    s.status = ATTN_OK;
  });
  if (s.status != ATTN_OK) return s.status;
  ctx->err = s.err;
  ctx->sm_count = s.sm_count;
  ctx->wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  return ATTN_OK;
}

// Admission checks (the pages' admission predicate, adapted: 64-bit offsets).
int validate_shape(const attn_shape* s, Dims* d) {
  if (!s) return ATTN_ERR_NULL;
  if (s->batch < 1 || s->batch > 65535) return ATTN_ERR_SHAPE;
  if (s->seq < 64 || s->seq % 64 != 0 || s->seq > (1 << 22)) return ATTN_ERR_SHAPE;
  if (s->heads < 1 || s->heads > 65535 || s->kv_heads < 1) return ATTN_ERR_SHAPE;
  if (s->heads % s->kv_heads != 0) return ATTN_ERR_SHAPE;
  if (s->head_dim != 64) return ATTN_ERR_SHAPE;
  if (s->causal != 0 && s->causal != 1) return ATTN_ERR_SHAPE;
  if (s->v_rows != 0 && s->v_rows != 1) return ATTN_ERR_SHAPE;
  if (!(s->scale > 0.0f) || !isfinite(s->scale)) return ATTN_ERR_SHAPE;
  int begin = s->head_begin, count = s->head_count;
  if (begin < 0 || count < 0) return ATTN_ERR_SHAPE;
  if (count == 0) {
    if (begin != 0) return ATTN_ERR_SHAPE;
    count = s->kv_heads;
  }
  if (begin + count > s->kv_heads) return ATTN_ERR_SHAPE;
  d->B = s->batch;
  d->T = s->seq;
  d->H = s->heads;
  d->Hkv = s->kv_heads;
  d->G = s->heads / s->kv_heads;
  d->causal = s->causal;
  d->lens = s->seq_lens;
  d->scale = s->scale;
  d->c = static_cast<float>(static_cast<double>(s->scale) / 0.69314718055994530942);
  d->kv_begin = begin;
  d->kv_count = count;
  d->nt = (s->seq + kTile - 1) / kTile;
  d->npairs = s->causal ? (long long)d->nt * (d->nt + 1) / 2 : (long long)d->nt * d->nt;
  d->v_rows = s->v_rows;
  d->ws_heads = 0;
  d->ws_h0 = 0;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t workspace_bytes_for(const Dims& d) {
  return (size_t)d.B * (size_t)(d.kv_count * d.G) * (size_t)d.npairs * kDsTileBytes;
}

namespace {
thread_local cudaError_t t_last_cuda_error = cudaSuccess;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  t_last_cuda_error = e;
  return ATTN_ERR_CUDA;
}

bool encode_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace css

using namespace css;

extern "C" {

int attn_version(void) { return 100; }

const char* attn_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* attn_error_string(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_SHAPE: return "shape outside the admission rules";
    case ATTN_ERR_NULL: return "a required pointer is null";
    case ATTN_ERR_ALIGN: return "a buffer is not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace smaller than required";
    case ATTN_ERR_CUDA: return "a CUDA call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
    case ATTN_ERR_DEVICE: return "the current device is not sm_103";
    case ATTN_ERR_SCRATCH_LIMIT: return "problem exceeds the static scratch of attn_bwd_noalloc";
    default: return "unknown error";
  }
}

void attn_set_wait_limit_ns(uint64_t limit_ns) {
  uint64_t v = limit_ns ? limit_ns : kDefaultWaitNs;
  if (v < ATTN_MIN_WAIT_LIMIT_NS) v = ATTN_MIN_WAIT_LIMIT_NS;
  g_wait_ns.store(v, std::memory_order_relaxed);
}

uint64_t attn_wait_limit_ns(void) { return g_wait_ns.load(std::memory_order_relaxed); }

size_t attn_bwd_workspace_bytes(const attn_shape* shape) {
  Dims d;
  if (validate_shape(shape, &d) != ATTN_OK) return 0;
  return workspace_bytes_for(d);
}

int attn_fwd(const attn_shape* shape, const uint16_t* q, const uint16_t* k, const uint16_t* vt,
             uint16_t* o, float* lse, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!q || !k || !vt || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_fwd(d, ctx, q, k, vt, o, lse, static_cast<cudaStream_t>(stream));
}

int attn_row_terms(const attn_shape* shape, const uint16_t* o, const uint16_t* dout,
                   float* delta, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!o || !dout || !delta) return ATTN_ERR_NULL;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(delta)) return ATTN_ERR_ALIGN;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_row_terms(d, ctx, o, dout, delta, static_cast<cudaStream_t>(stream));
}

int attn_bwd_keys(const attn_shape* shape, const uint16_t* q, const uint16_t* k,
                  const uint16_t* vt, const uint16_t* dout, const float* lse,
                  const float* delta, void* ds_ws, size_t ws_bytes, float* dk, float* dvt,
                  void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  // no workspace at all (null, 0 bytes): dS is not stored
  const bool store = !(ds_ws == nullptr && ws_bytes == 0);
  if (!q || !k || !vt || !dout || !lse || !delta || (store && !ds_ws) || !dk || !dvt)
    return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(ds_ws) || !aligned16(dk) || !aligned16(dvt))
    return ATTN_ERR_ALIGN;
  if (store && ws_bytes < workspace_bytes_for(d)) return ATTN_ERR_WORKSPACE;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_bwd_keys(d, ctx, q, k, vt, dout, lse, delta, static_cast<uint8_t*>(ds_ws), dk,
                         dvt, static_cast<cudaStream_t>(stream));
}

int attn_bwd_queries_fused(const attn_shape* shape, const uint16_t* q, const uint16_t* k,
                           const uint16_t* vt, const uint16_t* dout, const uint16_t* o,
                           const float* lse, float* delta, float* dq, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!q || !k || !vt || !dout || !o || !lse || !delta || !dq) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(dout) || !aligned16(o) ||
      !aligned16(lse) || !aligned16(delta) || !aligned16(dq))
    return ATTN_ERR_ALIGN;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_bwd_fused_q(d, ctx, q, k, vt, dout, o, lse, delta, dq,
                            static_cast<cudaStream_t>(stream));
}

int attn_bwd_queries(const attn_shape* shape, const uint16_t* k, const void* ds_ws,
                     size_t ws_bytes, float* dq, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!k || !ds_ws || !dq) return ATTN_ERR_NULL;
  if (!aligned16(k) || !aligned16(ds_ws) || !aligned16(dq)) return ATTN_ERR_ALIGN;
  if (ws_bytes < workspace_bytes_for(d)) return ATTN_ERR_WORKSPACE;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_bwd_queries(d, ctx, k, static_cast<const uint8_t*>(ds_ws), dq,
                            static_cast<cudaStream_t>(stream));
}

int attn_bwd_queries_rotated(const attn_shape* shape, const uint16_t* k, const void* ds_ws,
                             size_t ws_bytes, const float* cos_tab, const float* sin_tab,
                             uint16_t* dq_out, int64_t ld, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!k || !ds_ws || !cos_tab || !sin_tab || !dq_out) return ATTN_ERR_NULL;
  if (ld < (int64_t)d.H * 64 || ld % 8 != 0) return ATTN_ERR_SHAPE;
  if (!aligned16(k) || !aligned16(ds_ws) || !aligned16(cos_tab) || !aligned16(sin_tab) ||
      !aligned16(dq_out))
    return ATTN_ERR_ALIGN;
  if (ws_bytes < workspace_bytes_for(d)) return ATTN_ERR_WORKSPACE;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_bwd_queries(d, ctx, k, static_cast<const uint8_t*>(ds_ws), nullptr,
                            static_cast<cudaStream_t>(stream), cos_tab, sin_tab, dq_out, ld);
}

namespace {
// Checks a caller's projection block for `heads` heads of 64 columns.
int projection_from(const attn_projection* p, int heads, Projection* out) {
  if (!p || (!p->f32 && !p->bf16)) return ATTN_ERR_NULL;
  if (p->ld < (int64_t)heads * 64 || p->ld % 8 != 0) return ATTN_ERR_SHAPE;
  if (!aligned16(p->f32) || !aligned16(p->bf16)) return ATTN_ERR_ALIGN;
  *out = Projection{p->f32, p->bf16, p->ld};
  return ATTN_OK;
}
}  // namespace

int attn_bwd_keys_projected(const attn_shape* shape, const uint16_t* q, const uint16_t* k,
                            const uint16_t* vt, const uint16_t* dout, const float* lse,
                            const float* delta, void* ds_ws, size_t ws_bytes,
                            const attn_projection* dk_out, const attn_projection* dv_out,
                            void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  const bool store = !(ds_ws == nullptr && ws_bytes == 0);
  if (!q || !k || !vt || !dout || !lse || !delta || (store && !ds_ws)) return ATTN_ERR_NULL;
  Projection pk, pv;
  if ((rc = projection_from(dk_out, d.Hkv, &pk)) != ATTN_OK) return rc;
  if ((rc = projection_from(dv_out, d.Hkv, &pv)) != ATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(ds_ws))
    return ATTN_ERR_ALIGN;
  if (store && ws_bytes < workspace_bytes_for(d)) return ATTN_ERR_WORKSPACE;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_bwd_keys(d, ctx, q, k, vt, dout, lse, delta, static_cast<uint8_t*>(ds_ws),
                         nullptr, nullptr, static_cast<cudaStream_t>(stream), pk, pv);
}

int attn_bwd_queries_projected(const attn_shape* shape, const uint16_t* k, const void* ds_ws,
                               size_t ws_bytes, const attn_projection* dq_out, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!k || !ds_ws) return ATTN_ERR_NULL;
  Projection pq;
  if ((rc = projection_from(dq_out, d.H, &pq)) != ATTN_OK) return rc;
  if (!aligned16(k) || !aligned16(ds_ws)) return ATTN_ERR_ALIGN;
  if (ws_bytes < workspace_bytes_for(d)) return ATTN_ERR_WORKSPACE;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  return launch_bwd_queries(d, ctx, k, static_cast<const uint8_t*>(ds_ws), nullptr,
                            static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, 0, pq);
}

int attn_last_device_error(void* stream) {
  DevCtx ctx;
  int rc = device_context(&ctx);
  if (rc != ATTN_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v == 0) return ATTN_OK;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_ERR_DEVICE_TIMEOUT;
}

int attn_selftest_arith(const float* x, uint32_t* packed, float* e2, int n, void* stream) {
  if (n < 0 || (n & 1)) return ATTN_ERR_SHAPE;
  if (n > 0 && (!x || !packed || !e2)) return ATTN_ERR_NULL;
  DevCtx ctx;
  int rc = device_context(&ctx);
  if (rc != ATTN_OK) return rc;
  rc = launch_arith_probe(x, packed, e2, n, static_cast<cudaStream_t>(stream));
  if (rc != ATTN_OK) return rc;
  return cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
}

int attn_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  DevCtx ctx;
  int rc = device_context(&ctx);
  if (rc != ATTN_OK) return rc;
  rc = launch_wait_probe(ctx, limit_ns ? limit_ns : 1000000ull, static_cast<cudaStream_t>(stream));
  if (rc != ATTN_OK) return rc;
  return attn_last_device_error(stream);
}

}  // extern "C"
