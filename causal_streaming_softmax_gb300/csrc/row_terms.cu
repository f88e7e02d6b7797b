// row_terms.cu - D = rowsum(dO * O) per query row, and the bounded-wait probe.
//
// Method: streamingAttentionRowTermsOrderedUncheckedSM86 (page 1 header and
// definition): the backward pass's row terms, D_i = sum_d dO_id O_id from the
// stored binary16 O and dO, summed in binary32, written [head][T].  Rows at
// or past a sequence's length get D = 0.
//
// Memory-bound: eight threads share a row, each reading 16 bytes of dO (row
// r of [B][H][T][64]) and 16 bytes of O (token-major [B][T][H*64]); a
// three-step butterfly inside the eight-lane group forms the sum.
#include <math.h>

#include "attn_internal.h"
#include "sm103.cuh"

namespace css {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 8;  // T is a multiple of 64

__device__ __forceinline__ float dot8(uint4 a, uint4 b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    acc = fmaf(f16_bits_to_f32((uint16_t)(aw[u] & 0xFFFFu)),
               f16_bits_to_f32((uint16_t)(bw[u] & 0xFFFFu)), acc);
    acc = fmaf(f16_bits_to_f32((uint16_t)(aw[u] >> 16)), f16_bits_to_f32((uint16_t)(bw[u] >> 16)),
               acc);
  }
  return acc;
}

// Grid (T / 32, H, B): a block takes 32 consecutive rows of one (batch,
// head), so no thread divides by a runtime size.
__global__ void __launch_bounds__(kThreads)
    row_terms_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                     float* __restrict__ delta, int T, int H, const int32_t* __restrict__ lens) {
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 3);
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int part = threadIdx.x & 7;
  const size_t row = ((size_t)b * H + h) * T + t;  // [B][H][T]
  const uint4 dv = __ldg(reinterpret_cast<const uint4*>(dout + row * 64) + part);
  const uint4 ov =
      __ldg(reinterpret_cast<const uint4*>(o + (((size_t)b * T + t) * H + h) * 64) + part);
  float acc = dot8(dv, ov);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  if (part == 0) {
    int len = T;
    if (lens) {
      len = lens[b];
      len = len < 0 ? 0 : (len > T ? T : len);
    }
    delta[row] = t < len ? acc : 0.f;
  }
}

// One block waits on a barrier that nothing completes, with a short limit:
// the wait must give up, record the timeout and let the kernel return.
__global__ void wait_probe_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl w{err, limit_ns, &abort_flag};
    (void)mbar_wait(smem_u32(&bar), 0, w);
  }
  __syncthreads();
}

// The binary16 packing and the exponential exactly as the kernels use them.
__global__ void arith_probe_kernel(const float* __restrict__ x, uint32_t* __restrict__ packed,
                                   float* __restrict__ e2, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) e2[i] = ex2_approx(x[i]);
  if (2 * i + 1 < n) packed[i] = pack_f16x2(x[2 * i], x[2 * i + 1]);
}

}  // namespace

int launch_arith_probe(const float* x, uint32_t* packed, float* e2, int n, cudaStream_t stream) {
  if (n <= 0) return ATTN_OK;
  arith_probe_kernel<<<(n + 255) / 256, 256, 0, stream>>>(x, packed, e2, n);
  return cuda_status(cudaGetLastError());
}

int launch_row_terms(const Dims& d, const DevCtx& ctx, const uint16_t* o, const uint16_t* dout,
                     float* delta, cudaStream_t stream) {
  (void)ctx;
  if (d.H > 65535 || d.B > 65535) return ATTN_ERR_SHAPE;
  dim3 grid(d.T / kRowsPerBlock, d.H, d.B);
  return cuda_status(launch_dependent(row_terms_kernel, grid, dim3(kThreads), 0, stream, o, dout,
                                     delta, d.T, d.H, d.lens));
}

int launch_wait_probe(const DevCtx& ctx, uint64_t limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(ctx.err, limit_ns);
  return cuda_status(cudaGetLastError());
}

}  // namespace css
