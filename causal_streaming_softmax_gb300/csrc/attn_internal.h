// attn_internal.h - what the host API hands the kernel launchers: the
// validated shape with its derived sizes, and per-device context.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace css {

// Tile edge shared by every kernel: 128 queries by 128 keys.  The dS
// workspace is a sequence of such tiles (32 KiB of binary16 each).
constexpr int kTile = 128;
constexpr uint32_t kDsTileBytes = kTile * kTile * 2;

struct Dims {
  int B, T, H, Hkv, G;
  int causal;
  const int32_t* lens;  // device [B] or null
  float scale;          // natural scale s
  float c;              // fp32(s / ln 2)
  int kv_begin;         // head chunk (backward calls)
  int kv_count;
  int nt;               // ceil(T / 128)
  long long npairs;     // workspace tiles per query head
  int v_rows;           // V given as rows [B][Hkv][T][64] (else V^T [B][Hkv][64][T])
  int ws_heads;         // query heads per batch in the workspace layout (0: kv_count * G)
  int ws_h0;            // layout index of the chunk's first query head
  // workspace tile index of (query tile i, key tile j)
  __host__ __device__ long long pair(int i, int j) const {
    return causal ? (long long)i * (i + 1) / 2 + j : (long long)i * nt + j;
  }
};

// A token-major block of a projection gradient: element (b, t, head, c) at
// [(b T + t) ld + 64 head + c]; a null pointer is not written.
struct Projection {
  float* f32;
  uint16_t* bf16;
  long long ld;
  __host__ __device__ bool on() const { return f32 != nullptr || bf16 != nullptr; }
};

struct DevCtx {
  uint32_t* err;     // device error word
  uint64_t wait_ns;  // bounded-wait limit
  int sm_count;
};

// Host-side admission checks of a shape (ATTN_OK or an ATTN_ERR_ code) and
// the derived sizes.
int validate_shape(const attn_shape* s, Dims* d);
// The current device's context (error word, SM count, wait limit); fails
// with ATTN_ERR_DEVICE on anything but sm_103.
int device_context(DevCtx* ctx);
// Bytes of the dS workspace for a validated shape and its head chunk.
size_t workspace_bytes_for(const Dims& d);
bool aligned16(const void* p);

// Encodes a rank-3 binary16 tiled tensor map with the 128-byte swizzle.
// dims/strides as cuTensorMapEncodeTiled takes them (strides in bytes of
// dims 1 and 2), box = {box0, box1, 1}.
bool encode_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1);

// ATTN_OK when `e` is cudaSuccess; otherwise records e for
// attn_last_cuda_error on this host thread and returns ATTN_ERR_CUDA.
int cuda_status(cudaError_t e);

// Launches `kernel` with programmatic stream serialization: it may start
// while the previous kernel in `stream` finishes (every kernel of the path
// calls griddep_wait before touching global memory).  Returns the launch's
// status.
template <typename... P, typename... A>
inline cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
  const cudaError_t last = cudaGetLastError();  // takes the launch error off the thread
  return e != cudaSuccess ? e : last;
}

int launch_fwd(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
               const uint16_t* vt, uint16_t* o, float* lse, cudaStream_t stream);
int launch_row_terms(const Dims& d, const DevCtx& ctx, const uint16_t* o, const uint16_t* dout,
                     float* delta, cudaStream_t stream);
int launch_bwd_keys(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
                    const uint16_t* vt, const uint16_t* dout, const float* lse,
                    const float* delta, uint8_t* ws, float* dk, float* dvt,
                    cudaStream_t stream,
                    Projection pk = {}, Projection pv = {});
int launch_bwd_fused_q(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
                       const uint16_t* vt, const uint16_t* dout, const uint16_t* o,
                       const float* lse, float* delta, float* dq, cudaStream_t stream);
int launch_bwd_queries(const Dims& d, const DevCtx& ctx, const uint16_t* k, const uint8_t* ws,
                       float* dq, cudaStream_t stream, const float* cos_t = nullptr,
                       const float* sin_t = nullptr, uint16_t* rot_out = nullptr,
                       long long ld = 0, Projection pq = {});
int launch_wait_probe(const DevCtx& ctx, uint64_t limit_ns, cudaStream_t stream);
int launch_arith_probe(const float* x, uint32_t* packed, float* e2, int n, cudaStream_t stream);

}  // namespace css
