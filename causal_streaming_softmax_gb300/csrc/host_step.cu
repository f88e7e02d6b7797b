// host_step.cu - attn_step_host: one whole forward + backward from host
// memory to host memory, with the copies overlapped with the kernels.
//
// The kernels run in order on the caller's stream: forward, row terms, key
// pass, then the dQ pass in two K/V-head halves (the stored order); or
// forward, the fused query pass in two halves (it forms D), then the key pass
// storing no dS (the fused order).  The fused order is taken when the caller
// gives no workspace, and also when dQ is large: the host link then bounds
// the step, and the fused order has dQ ready before the key pass, so dQ's
// copy back runs under the key pass instead of after the last kernel.
// Measured end to end on GB300 (ms per step, stored / fused order): dQ of
// 0.25 MiB 0.044 / 0.046, 2 MiB 0.111 / 0.119, 32 MiB 0.677 / 0.598,
// 128 MiB 5.50 / 5.27, 256 MiB 8.22 / 7.56; the switch sits at 8 MiB.
//
// A second stream, owned by the library (one per device), carries the copies
// that need not wait for the whole chain:
//   dO goes in after Q, K and V^T (so it never slows their copy) while the
//   forward runs; O and L come back while the backward runs; dK and dV^T
//   come back while the dQ pass runs (stored path); dQ comes back in halves,
//   each while later kernels run.  Only Q, K, V^T in and the last outputs
//   out are exposed.  The caller's stream waits for the side stream at the end,
//   so everything is complete once the caller's stream is.
#include <mutex>

#include "attn_internal.h"

namespace css {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kEvents = 6;
constexpr size_t kFusedOrderDqBytes = size_t(8) << 20;

struct StepStreams {
  std::once_flag once;
  cudaError_t status = cudaErrorUnknown;
  cudaStream_t side = nullptr;
  cudaEvent_t ev[kEvents] = {};
  std::mutex mu;  // the events are reused: one enqueue at a time per device
};
StepStreams g_step[kMaxDevices];

int step_streams(int dev, StepStreams** out) {
  StepStreams& ss = g_step[dev];
  std::call_once(ss.once, [&ss] {
    ss.status = cudaStreamCreateWithFlags(&ss.side, cudaStreamNonBlocking);
    for (int i = 0; i < kEvents && ss.status == cudaSuccess; ++i)
      ss.status = cudaEventCreateWithFlags(&ss.ev[i], cudaEventDisableTiming);
  });
  if (ss.status != cudaSuccess) return cuda_status(ss.status);
  *out = &ss;
  return ATTN_OK;
}

// The fused order: no workspace (null, 0 bytes), or 8 MiB of dQ or more.
bool fused_order(const Dims& d, const attn_device_buffers* dev) {
  const size_t dq_total = (size_t)d.B * d.H * d.T * 64 * 4;
  return (dev->ws == nullptr && dev->ws_bytes == 0) || dq_total >= kFusedOrderDqBytes;
}

// Copies rows [h0, h0 + nh) of every batch of a [B][H][row_bytes] tensor.
cudaError_t copy_heads(void* dst, const void* src, int B, int H, int h0, int nh, size_t row_bytes,
                       cudaMemcpyKind kind, cudaStream_t st) {
  const size_t pitch = (size_t)H * row_bytes;
  const size_t off = (size_t)h0 * row_bytes;
  return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + off, pitch,
                           static_cast<const uint8_t*>(src) + off, pitch, (size_t)nh * row_bytes,
                           (size_t)B, kind, st);
}

}  // namespace
}  // namespace css

using namespace css;

extern "C" ATTN_API int attn_step_host(const attn_shape* shape, const attn_device_buffers* dev,
                                       const uint16_t* h_q, const uint16_t* h_k,
                                       const uint16_t* h_vt, const uint16_t* h_dout,
                                       uint16_t* h_o, float* h_lse, float* h_dq, float* h_dk,
                                       float* h_dvt, void* stream) {
  Dims d;
  int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (d.kv_begin != 0 || d.kv_count != d.Hkv) return ATTN_ERR_SHAPE;  // whole problems only
  if (!dev || !h_q || !h_k || !h_vt || !h_dout || !h_o || !h_lse || !h_dq || !h_dk || !h_dvt)
    return ATTN_ERR_NULL;
  const bool fused = fused_order(d, dev);
  if (!dev->q || !dev->k || !dev->vt || !dev->dout || !dev->o || !dev->lse || !dev->delta ||
      (!fused && !dev->ws) || !dev->dq || !dev->dk || !dev->dvt)
    return ATTN_ERR_NULL;
  if (!aligned16(dev->q) || !aligned16(dev->k) || !aligned16(dev->vt) ||
      !aligned16(dev->dout) || !aligned16(dev->o) || !aligned16(dev->lse) ||
      !aligned16(dev->delta) || !aligned16(dev->ws) || !aligned16(dev->dq) ||
      !aligned16(dev->dk) || !aligned16(dev->dvt))
    return ATTN_ERR_ALIGN;
  if (!fused && dev->ws_bytes < workspace_bytes_for(d)) return ATTN_ERR_WORKSPACE;
  DevCtx ctx;
  if ((rc = device_context(&ctx)) != ATTN_OK) return rc;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return ATTN_ERR_CUDA;
  StepStreams* ss = nullptr;
  if ((rc = step_streams(device, &ss)) != ATTN_OK) return rc;

  const size_t B = d.B, H = d.H, Hkv = d.Hkv, T = d.T;
  const size_t q_bytes = B * H * T * 64 * 2, kv_bytes = B * Hkv * T * 64 * 2;
  const size_t o_bytes = B * T * H * 64 * 2, lse_bytes = B * H * T * 4;
  const size_t dk_bytes = B * Hkv * T * 64 * 4;
  const size_t dq_row = T * 64 * 4;  // one query head's dQ
  cudaStream_t main = static_cast<cudaStream_t>(stream), side = ss->side;
  cudaEvent_t* ev = ss->ev;
  uint8_t* ws = static_cast<uint8_t*>(dev->ws);
  std::lock_guard<std::mutex> lock(ss->mu);

#define CK(x)                                \
  do {                                       \
    const cudaError_t e_ = (x);              \
    if (e_ != cudaSuccess) return cuda_status(e_); \
  } while (0)
#define RC(x)                          \
  do {                                 \
    const int r_ = (x);                \
    if (r_ != ATTN_OK) return r_;      \
  } while (0)

  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  CK(cudaMemcpyAsync(dev->q, h_q, q_bytes, h2d, main));
  CK(cudaMemcpyAsync(dev->k, h_k, kv_bytes, h2d, main));
  CK(cudaMemcpyAsync(dev->vt, h_vt, kv_bytes, h2d, main));
  CK(cudaEventRecord(ev[0], main));
  CK(cudaStreamWaitEvent(side, ev[0], 0));
  CK(cudaMemcpyAsync(dev->dout, h_dout, q_bytes, h2d, side));
  CK(cudaEventRecord(ev[1], side));

  RC(launch_fwd(d, ctx, dev->q, dev->k, dev->vt, dev->o, dev->lse, main));
  CK(cudaEventRecord(ev[2], main));
  CK(cudaStreamWaitEvent(side, ev[2], 0));
  CK(cudaMemcpyAsync(h_o, dev->o, o_bytes, d2h, side));
  CK(cudaMemcpyAsync(h_lse, dev->lse, lse_bytes, d2h, side));

  CK(cudaStreamWaitEvent(main, ev[1], 0));
  const int halves = d.Hkv >= 2 ? 2 : 1;
  // the dQ pass in two K/V-head halves; the first half's dQ comes back while
  // the rest of the backward runs
  auto dq_half = [&](int part, int& kv0, bool last) -> int {
    Dims c = d;
    c.kv_begin = kv0;
    c.kv_count = (d.Hkv * (part + 1)) / halves - kv0;
    c.ws_heads = d.H;
    c.ws_h0 = kv0 * d.G;
    int r = fused ? launch_bwd_fused_q(c, ctx, dev->q, dev->k, dev->vt, dev->dout, dev->o,
                                       dev->lse, dev->delta, dev->dq, main)
                  : launch_bwd_queries(c, ctx, dev->k, ws, dev->dq, main);
    if (r != ATTN_OK) return r;
    cudaError_t e;
    if (!last) {
      if ((e = cudaEventRecord(ev[4], main)) != cudaSuccess) return cuda_status(e);
      if ((e = cudaStreamWaitEvent(side, ev[4], 0)) != cudaSuccess) return cuda_status(e);
    }
    e = copy_heads(h_dq, dev->dq, d.B, d.H, c.kv_begin * d.G, c.kv_count * d.G, dq_row, d2h,
                   last ? main : side);
    if (e != cudaSuccess) return cuda_status(e);
    kv0 += c.kv_count;
    return ATTN_OK;
  };
  int kv0 = 0;
  if (fused) {
    // the fused query pass forms D itself, then the key pass (no dS store)
    for (int part = 0; part < halves; ++part) RC(dq_half(part, kv0, false));
    RC(launch_bwd_keys(d, ctx, dev->q, dev->k, dev->vt, dev->dout, dev->lse, dev->delta,
                       nullptr, dev->dk, dev->dvt, main));
    CK(cudaMemcpyAsync(h_dk, dev->dk, dk_bytes, d2h, main));
    CK(cudaMemcpyAsync(h_dvt, dev->dvt, dk_bytes, d2h, main));
  } else {
    RC(launch_row_terms(d, ctx, dev->o, dev->dout, dev->delta, main));
    RC(launch_bwd_keys(d, ctx, dev->q, dev->k, dev->vt, dev->dout, dev->lse, dev->delta, ws,
                       dev->dk, dev->dvt, main));
    CK(cudaEventRecord(ev[3], main));
    CK(cudaStreamWaitEvent(side, ev[3], 0));
    CK(cudaMemcpyAsync(h_dk, dev->dk, dk_bytes, d2h, side));
    CK(cudaMemcpyAsync(h_dvt, dev->dvt, dk_bytes, d2h, side));
    for (int part = 0; part < halves; ++part) RC(dq_half(part, kv0, part + 1 == halves));
  }
  CK(cudaEventRecord(ev[5], side));
  CK(cudaStreamWaitEvent(main, ev[5], 0));
#undef CK
#undef RC
  return ATTN_OK;
}

extern "C" ATTN_API int attn_step_host_order(const attn_shape* shape,
                                             const attn_device_buffers* dev) {
  Dims d;
  const int rc = validate_shape(shape, &d);
  if (rc != ATTN_OK) return rc;
  if (!dev) return ATTN_ERR_NULL;
  return fused_order(d, dev) ? ATTN_STEP_FUSED : ATTN_STEP_STORED;
}
