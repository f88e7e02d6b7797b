// bwd_queries.cu - the dQ pass: one 128-query tile of one query head per
// CTA, dQ = s * sum over the visible key tiles of dS K, dS read back from the
// workspace the key pass filled.
//
// Method (StreamingAttentionSM86.alpha, streamingAttentionQueryFromScores
// section and the page-1 header of the split backward): for each key tile up
// to the diagonal, dQ += dS K with dS taken from the stored dS^T read
// transposed; the epilogue scales by s and stores binary32 rows, or (the
// pages' other epilogues) turns dQ back by the inverse half-split rotation
// into bfloat16 token-major rows, or writes a token-major block of a fused
// projection gradient in binary32 and bfloat16 (a template parameter picks
// one, so each variant carries only its own code).
//
// GB300 design: warp 4 copies each workspace tile (32 KiB, already in the
// shared-memory image the tensor core reads) with one bulk copy and K's tile
// with TMA, through a 2-stage ring (two CTAs per SM); warp 5 issues dQ += dS K with dS as an
// MN-major A operand (queries along the 128-byte rows) and K as an MN-major
// B operand; warps 0-3 scale and store.  The pass is bound by reading dS
// from HBM.
#include <math.h>

#include <mutex>

#include "attn_internal.h"
#include "epilogue.cuh"
#include "sm103.cuh"

namespace css {
namespace {

constexpr int kBM = 128;  // queries per CTA
constexpr int kBN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr int kStages = 2;  // two CTAs share an SM: one's epilogue overlaps the other's loads
constexpr uint32_t kKTileBytes = 16384;
constexpr uint32_t kStageBytes = kDsTileBytes + kKTileBytes;  // dS^T image, then K tile
constexpr uint32_t kSmemBar = kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kSmemBar + 128 + 1024;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kIdesc = idesc_f16_f32(128, 64, 1, 1);  // dS (MN-major) x K (MN-major)

enum { BAR_FULL = 0, BAR_EMPTY = kStages, BAR_DONE = 2 * kStages, BAR_COUNT };
static_assert(BAR_COUNT * 8 <= 128, "barrier area");

struct QueriesArgs {
  Dims d;
  const uint8_t* ws;
  float* dq;
  // inverse half-split rotation epilogue (rot_out non-null): cos and sin
  // tables [T][32], bfloat16 output row p of head h at rot_out[p * ld + 64 h]
  const float* cos_t;
  const float* sin_t;
  uint16_t* rot_out;
  long long ld;
  uint32_t* err;
  uint64_t wait_ns;
  Projection pq;  // token-major dQ block instead of dq (when on)
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// EPI: 0 binary32 dQ rows [B][H][T][64]; 1 the inverse half-split rotation
// to bfloat16 token-major; 2 the projection-fused token-major block.
template <int EPI>
__global__ void __launch_bounds__(kThreads, 2)
    bwd_queries_kernel(const __grid_constant__ CUtensorMap tm_k, const QueriesArgs a) {
  griddep_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar0 = sbase + kSmemBar;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

  const Dims& d = a.d;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h_local = blockIdx.x;
  const int h = d.kv_begin * d.G + h_local;
  const int kv = h / d.G;
  const int it = (int)gridDim.y - 1 - (int)blockIdx.y;  // heaviest causal tiles first
  const int b = blockIdx.z;
  const int T = d.T;
  const int Hc = d.ws_heads ? d.ws_heads : d.kv_count * d.G;
  const long long tile0 = ((long long)b * Hc + d.ws_h0 + h_local) * d.npairs;

  WaitCtl wc{a.err, a.wait_ns, &s_abort};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(BAR_FULL + s), 1);
      mbar_init(BAR(BAR_EMPTY + s), 1);
    }
    mbar_init(BAR(BAR_DONE), 1);
    fence_mbarrier_init();
  }
  if (warp == 5) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  griddep_wait();
  int len = T;
  if (d.lens) {
    len = d.lens[b];
    len = len < 0 ? 0 : (len > T ? T : len);
  }
  const int q0 = it * kBM;
  int n_kt = 0;
  if (q0 < len) n_kt = d.causal ? it + 1 : (len + kBN - 1) / kBN;

  if (warp == 4) {
    // ---------------- producer: workspace tile (bulk) + K tile (TMA) ----------------
    if (lane == 0 && n_kt > 0) {
      tma_prefetch_desc(&tm_k);
      const int kvplane = b * d.Hkv + kv;
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait(BAR(BAR_EMPTY + s), ((j / kStages) - 1) & 1, wc)) break;
        const uint32_t st = sbase + s * kStageBytes;
        mbar_arrive_expect_tx(BAR(BAR_FULL + s), kStageBytes);
        // dS is read once: evict it first, so the K tiles every query tile
        // reads again stay in L2
        bulk_load_hint(st, a.ws + (size_t)(tile0 + d.pair(it, j)) * kDsTileBytes, kDsTileBytes,
                       BAR(BAR_FULL + s), l2_policy_evict_first());
        tma_load_3d(st + kDsTileBytes, &tm_k, BAR(BAR_FULL + s), 0, j * kBN, kvplane);
        issued = j + 1;
      }
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
        drain_wait(BAR(BAR_FULL + j % kStages), (j / kStages) & 1);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && n_kt > 0) {
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(BAR(BAR_FULL + s), (j / kStages) & 1, wc)) break;
        tc_fence_after();
        const uint32_t ds_s = sbase + s * kStageBytes;
        const uint32_t k_s = ds_s + kDsTileBytes;
        // reduction over the tile's 128 keys, 16 rows (2 KiB) per step, in
        // both operands; dS's two 64-query blocks are 16 KiB apart
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem, sdesc_sw128(ds_s + kk * 2048, 16384, 1024),
                 sdesc_sw128(k_s + kk * 2048, 8192, 1024), kIdesc, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(BAR(BAR_EMPTY + s));
      }
      mma_commit(BAR(BAR_DONE));
    }
  } else {
    // ---------------- epilogue: dQ = s * sum ----------------
    const int q = q0 + threadIdx.x;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t r0[32], r1[32];
    // the whole warp waits together, so the warp-aligned tensor-memory load
    // below runs converged; if the wait gave up, the load is skipped (the
    // device error word already records the timeout)
    if (n_kt > 0 && mbar_wait_warp(BAR(BAR_DONE), 0, wc)) {
      tc_fence_after();
      tmem_ld32x2_wait(tmem + lane_base, tmem + lane_base + 32, r0, r1);
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) r0[u] = r1[u] = 0u;  // no visible key: dQ = 0
    }
    if (EPI == 2 && q < T) {
      // projection-fused epilogue: row q of head h, token-major
      store_projection_row(a.pq, ((size_t)b * T + q) * a.pq.ld + 64 * (size_t)h, r0, r1, d.scale,
                           true);
    } else if (EPI == 0 && q < T) {
      float4* dst = reinterpret_cast<float4*>(a.dq + (((size_t)b * d.H + h) * T + q) * 64);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        dst[u] = make_float4(as_f(r0[4 * u]) * d.scale, as_f(r0[4 * u + 1]) * d.scale,
                             as_f(r0[4 * u + 2]) * d.scale, as_f(r0[4 * u + 3]) * d.scale);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        dst[8 + u] = make_float4(as_f(r1[4 * u]) * d.scale, as_f(r1[4 * u + 1]) * d.scale,
                                 as_f(r1[4 * u + 2]) * d.scale, as_f(r1[4 * u + 3]) * d.scale);
    } else if (EPI == 1 && q < T) {
      // dQ turned back by the inverse half-split rotation of position q:
      // column c < 32 pairs with c + 32; out_c = x_c cos + x_{c+32} sin,
      // out_{c+32} = x_{c+32} cos - x_c sin, each product of the sine
      // rounded before the fused multiply-add; then packed to bfloat16
      const float4* cr = reinterpret_cast<const float4*>(a.cos_t + (size_t)q * 32);
      const float4* sr = reinterpret_cast<const float4*>(a.sin_t + (size_t)q * 32);
      uint32_t lo[16], hi[16];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 cv = __ldg(cr + u), sv = __ldg(sr + u);
        const float co[4] = {cv.x, cv.y, cv.z, cv.w}, si[4] = {sv.x, sv.y, sv.z, sv.w};
        float o1[4], o2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x1 = __fmul_rn(as_f(r0[4 * u + e]), d.scale);
          const float x2 = __fmul_rn(as_f(r1[4 * u + e]), d.scale);
          o1[e] = fmaf(x1, co[e], __fmul_rn(x2, si[e]));
          o2[e] = fmaf(x2, co[e], -__fmul_rn(x1, si[e]));
        }
        lo[2 * u] = pack_bf16x2(o1[0], o1[1]);
        lo[2 * u + 1] = pack_bf16x2(o1[2], o1[3]);
        hi[2 * u] = pack_bf16x2(o2[0], o2[1]);
        hi[2 * u + 1] = pack_bf16x2(o2[2], o2[3]);
      }
      uint4* dst = reinterpret_cast<uint4*>(a.rot_out + ((size_t)b * T + q) * a.ld + 64 * h);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        dst[u] = make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
        dst[4 + u] = make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    if (n_kt > 0) drain_wait(BAR(BAR_DONE), 0);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef BAR
}

}  // namespace

int launch_bwd_queries(const Dims& d, const DevCtx& ctx, const uint16_t* k, const uint8_t* ws,
                       float* dq, cudaStream_t stream, const float* cos_t, const float* sin_t,
                       uint16_t* rot_out, long long ld, Projection pq) {
  CUtensorMap tk;
  const uint64_t T = (uint64_t)d.T;
  if (!encode_tmap_3d(&tk, k, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, kBN))
    return ATTN_ERR_CUDA;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_status[64];
  std::call_once(attr_once[dev & 63], [dev] {
    cudaError_t e = cudaFuncSetAttribute(bwd_queries_kernel<0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_queries_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_queries_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    attr_status[dev & 63] = e;
  });
  if (attr_status[dev & 63] != cudaSuccess) return cuda_status(attr_status[dev & 63]);
  QueriesArgs args{d, ws, dq, cos_t, sin_t, rot_out, ld, ctx.err, ctx.wait_ns, pq};
  dim3 grid(d.kv_count * d.G, d.nt, d.B);
  auto* kernel = pq.on() ? bwd_queries_kernel<2>
                         : (rot_out != nullptr ? bwd_queries_kernel<1> : bwd_queries_kernel<0>);
  return cuda_status(
      launch_dependent(kernel, grid, dim3(kThreads), kSmemBytes, stream, tk, args));
}

}  // namespace css
