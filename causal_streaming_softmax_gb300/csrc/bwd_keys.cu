// bwd_keys.cu - the key pass of the backward: one 128-key tile of one K/V
// head per CTA, walking every query head of the head's group and every
// 128-query tile that can see the keys.
//
// Method (StreamingAttentionSM86.alpha, key launch streamingAttentionKeySM86
// and the page-1 header of the split backward): with L and D of the queries,
//   S^T = K Q^T, P^T = 2^(S^T c - L), dP^T = V dO^T, dS^T = P^T (dP^T - D),
//   dV += P^T dO, dK += dS^T Q,
// P^T and dS^T rounded to binary16 before their products (score-gradient
// packing in skTileBody); dS^T is also stored for the dQ pass (the shared
// pass's sksStoreScoreGradients), so S, P and dP are formed once.  The
// epilogue writes dK = s * sum (binary32 rows) and dV^T unscaled.
//
// GB300 design: warps 0-3 one thread per key row (tensor-memory lane),
// warp 4 TMA producer (K and V^T once, Q / dO / L / D per step through a
// 2-stage ring), warp 5 MMA issuer.  The group's query heads are summed in
// the tensor-memory accumulators of dK and dV (no atomics, fixed order).
// dS^T goes through shared memory in the 128-byte-swizzled image that both
// the dK product here (K-major A) and the dQ pass (MN-major A) read, and is
// copied to the workspace by one bulk store per step.
// Tensor memory: S^T 0-127, dP^T 128-255, P^T 256-319 (binary16 pairs),
// dK 320-383, dV 384-447.
#include <math.h>

#include <mutex>

#include "attn_internal.h"
#include "sm103.cuh"

namespace css {
namespace {

constexpr int kBK = 128;  // keys per CTA
constexpr int kBQ = 128;  // queries per step
constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kTileB = 16384;  // 128 rows x 128 B
constexpr uint32_t kSmemK = 0;
constexpr uint32_t kSmemV = kTileB;  // V^T: two 64-key halves of 64 rows x 128 B
constexpr uint32_t kSmemStage0 = 2 * kTileB;
constexpr uint32_t kStageQ = 0, kStageDO = kTileB, kStageL = 2 * kTileB, kStageD = 2 * kTileB + 512;
constexpr uint32_t kStageBytes = 2 * kTileB + 2048;  // keeps every stage 1024-aligned
constexpr uint32_t kSmemDS0 = kSmemStage0 + kStages * kStageBytes;
constexpr uint32_t kSmemBar = kSmemDS0 + 2 * kDsTileBytes;
constexpr uint32_t kSmemBytes = kSmemBar + 256 + 1024;

constexpr uint32_t kColST = 0, kColDPT = 128, kColPT = 256, kColDK = 320, kColDV = 384;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_f16_f32(128, 128, 0, 0);   // K (K-major) x Q (K-major)
constexpr uint32_t kIdescDP = idesc_f16_f32(128, 128, 1, 0);  // V (MN-major) x dO (K-major)
constexpr uint32_t kIdescAcc = idesc_f16_f32(128, 64, 0, 1);  // P^T/dS^T x dO/Q (MN-major)

enum {
  BAR_KV = 0,
  BAR_Q_FULL = 1,
  BAR_Q_EMPTY = BAR_Q_FULL + kStages,
  BAR_S_FULL = BAR_Q_EMPTY + kStages,
  BAR_P_READY,
  BAR_DS_FREE,                     // [2] the dK product has read dS^T buffer b
  BAR_DS_STORED = BAR_DS_FREE + 2,  // [2] the bulk store has read dS^T buffer b
  BAR_DONE = BAR_DS_STORED + 2,
  BAR_COUNT
};
static_assert(BAR_COUNT * 8 <= 256, "barrier area");

struct KeysArgs {
  Dims d;
  const float* lse;
  const float* delta;
  uint8_t* ws;
  float* dk;
  float* dvt;
  uint32_t* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

static __device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_keys_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_vt,
                    const __grid_constant__ CUtensorMap tm_do, const KeysArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar0 = sbase + kSmemBar;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

  const Dims& d = a.d;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kv = d.kv_begin + blockIdx.x;
  const int jt = blockIdx.y;  // key tile; low tiles see the most queries (heaviest first)
  const int b = blockIdx.z;
  const int T = d.T;
  int len = T;
  if (d.lens) {
    len = d.lens[b];
    len = len < 0 ? 0 : (len > T ? T : len);
  }
  const int k0 = jt * kBK;
  const int i_lo = d.causal ? jt : 0;
  int i_hi = (len + kBQ - 1) / kBQ;
  if (k0 >= len) i_hi = i_lo;
  const int n_i = i_hi > i_lo ? i_hi - i_lo : 0;
  const int n_steps = d.G * n_i;

  WaitCtl wc{a.err, a.wait_ns, &s_abort};

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(BAR(BAR_KV), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(BAR_Q_FULL + s), 1);
      mbar_init(BAR(BAR_Q_EMPTY + s), 1);
    }
    mbar_init(BAR(BAR_S_FULL), 1);
    mbar_init(BAR(BAR_P_READY), 128);
    for (int u = 0; u < 2; ++u) {
      mbar_init(BAR(BAR_DS_FREE + u), 1);
      mbar_init(BAR(BAR_DS_STORED + u), 1);
    }
    mbar_init(BAR(BAR_DONE), 1);
    fence_mbarrier_init();
  }
  if (warp == 5) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_steps > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      tma_prefetch_desc(&tm_do);
      const int kvplane = b * d.Hkv + kv;
      mbar_arrive_expect_tx(BAR(BAR_KV), 2 * kTileB);
      tma_load_3d(sbase + kSmemK, &tm_k, BAR(BAR_KV), 0, k0, kvplane);
      tma_load_3d(sbase + kSmemV, &tm_vt, BAR(BAR_KV), k0, 0, kvplane);
      tma_load_3d(sbase + kSmemV + 8192, &tm_vt, BAR(BAR_KV), k0 + 64, 0, kvplane);
      int issued = 0;
      for (int n = 0; n < n_steps; ++n) {
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait(BAR(BAR_Q_EMPTY + s), ((n / kStages) - 1) & 1, wc)) break;
        const int g = n / n_i;
        const int i = i_lo + n % n_i;
        const int qplane = b * d.H + kv * d.G + g;
        const int rows = min(kBQ, T - i * kBQ);
        const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
        mbar_arrive_expect_tx(BAR(BAR_Q_FULL + s), 2 * kTileB + 2 * rows * 4);
        tma_load_3d(st + kStageQ, &tm_q, BAR(BAR_Q_FULL + s), 0, i * kBQ, qplane);
        tma_load_3d(st + kStageDO, &tm_do, BAR(BAR_Q_FULL + s), 0, i * kBQ, qplane);
        const size_t lo = (size_t)qplane * T + (size_t)i * kBQ;
        bulk_load(st + kStageL, a.lse + lo, rows * 4, BAR(BAR_Q_FULL + s));
        bulk_load(st + kStageD, a.delta + lo, rows * 4, BAR(BAR_Q_FULL + s));
        issued = n + 1;
      }
      drain_wait(BAR(BAR_KV), 0, a.wait_ns);
      for (int n = (issued > kStages ? issued - kStages : 0); n < issued; ++n)
        drain_wait(BAR(BAR_Q_FULL + n % kStages), (n / kStages) & 1, a.wait_ns);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0 && n_steps > 0) {
      const uint32_t k_s = sbase + kSmemK, v_s = sbase + kSmemV;
      bool ok = mbar_wait(BAR(BAR_KV), 0, wc);
      for (int n = 0; ok && n < n_steps; ++n) {
        const int s = n % kStages;
        if (!mbar_wait(BAR(BAR_Q_FULL + s), (n / kStages) & 1, wc)) break;
        tc_fence_after();
        const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
        const uint32_t q_s = st + kStageQ, do_s = st + kStageDO;
        // S^T = K Q^T (reduction over d: four K=16 steps of 32 B)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + kColST, sdesc_sw128(k_s + kk * 32, 16, 1024),
                 sdesc_sw128(q_s + kk * 32, 16, 1024), kIdescS, kk > 0);
        // dP^T = V dO^T: V read MN-major from the V^T tile (keys along the
        // 128-byte rows, two 64-key blocks 8 KiB apart; a K step = 16 rows)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + kColDPT, sdesc_sw128(v_s + kk * 2048, 8192, 1024),
                 sdesc_sw128(do_s + kk * 32, 16, 1024), kIdescDP, kk > 0);
        mma_commit(BAR(BAR_S_FULL));
        if (!mbar_wait(BAR(BAR_P_READY), n & 1, wc)) break;
        tc_fence_after();
        const uint32_t ds_s = sbase + kSmemDS0 + (n & 1) * kDsTileBytes;
        // dV += P^T dO and dK += dS^T Q: reduction over the step's 128
        // queries (eight K=16 steps); dO and Q read MN-major (d along rows).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColDV, tmem + kColPT + kk * 8, sdesc_sw128(do_s + kk * 2048, 8192, 1024),
                 kIdescAcc, (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kColDK, sdesc_sw128(ds_s + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(q_s + kk * 2048, 8192, 1024), kIdescAcc, (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(BAR(BAR_Q_EMPTY + s));
        mma_commit(BAR(BAR_DS_FREE + (n & 1)));
      }
      mma_commit(BAR(BAR_DONE));
    }
  } else {
    // ---------------- score gradients: thread = key row ----------------
    const int kr = threadIdx.x;
    const int key = k0 + kr;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c = d.c;
    const int h_local0 = (kv - d.kv_begin) * d.G;
    const int Hc = d.kv_count * d.G;
    bool ok = true;
    for (int n = 0; n < n_steps; ++n) {
      const int s = n % kStages;
      const int g = n / n_i;
      const int i = i_lo + n % n_i;
      const uint32_t ds_s = sbase + kSmemDS0 + (n & 1) * kDsTileBytes;
      if (n >= 2) {
        // dS^T buffer n%2 was last filled at step n-2: wait until the dK
        // product and the bulk store of that step have both read it
        if (!mbar_wait(BAR(BAR_DS_FREE + (n & 1)), ((n >> 1) - 1) & 1, wc) ||
            !mbar_wait(BAR(BAR_DS_STORED + (n & 1)), ((n >> 1) - 1) & 1, wc)) {
          ok = false;
          break;
        }
      }
      if (!mbar_wait(BAR(BAR_S_FULL), n & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint8_t* stg = sgen + kSmemStage0 + s * kStageBytes;
      const float* Ls = reinterpret_cast<const float*>(stg + kStageL);
      const float* Ds = reinterpret_cast<const float*>(stg + kStageD);
      const int q0 = i * kBQ;
      const bool need_mask = (d.causal && q0 < k0 + kBK) || (q0 + kBQ > len) || (k0 + kBK > len);
      // query (local index) ql is valid for this key iff qlo <= ql < qhi
      const int qlo = (d.causal ? key : 0) - q0;
      const int qhi = (key < len ? len : 0) - q0;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sv[32], dv[32];
        tmem_ld32x2_wait(tmem + lane_base + kColST + ch * 32, tmem + lane_base + kColDPT + ch * 32,
                         sv, dv);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int ql = ch * 32 + e;
          float p0 = ex2_approx(fmaf(as_f(sv[e]), c, -Ls[ql]));
          float p1 = ex2_approx(fmaf(as_f(sv[e + 1]), c, -Ls[ql + 1]));
          float d0 = p0 * (as_f(dv[e]) - Ds[ql]);
          float d1 = p1 * (as_f(dv[e + 1]) - Ds[ql + 1]);
          if (need_mask) {
            if (ql < qlo || ql >= qhi) p0 = 0.f, d0 = 0.f;
            if (ql + 1 < qlo || ql + 1 >= qhi) p1 = 0.f, d1 = 0.f;
          }
          pp[e >> 1] = pack_f16x2(p0, p1);
          dd[e >> 1] = pack_f16x2(d0, d1);
        }
        tmem_st16(tmem + lane_base + kColPT + ch * 16, pp);
        // dS^T row kr, queries 32ch..32ch+31: 64-query block ch/2, chunks
        // (ch%2)*4 .. +3 of the swizzled 128-byte row
        const uint32_t rowbase = ds_s + (ch >> 1) * 16384;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(rowbase + sw128_offset(kr, (ch & 1) * 4 + u), dd[4 * u], dd[4 * u + 1],
                       dd[4 * u + 2], dd[4 * u + 3]);
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_shared();
      mbar_arrive(BAR(BAR_P_READY));
      if (threadIdx.x == 0) {
        // every row of dS^T is in shared memory once all 128 threads arrived
        if (!mbar_wait(BAR(BAR_P_READY), n & 1, wc)) {
          ok = false;
          break;
        }
        const long long tile =
            ((long long)b * Hc + h_local0 + g) * d.npairs + d.pair(i, jt);
        bulk_store(a.ws + (size_t)tile * kDsTileBytes, ds_s, kDsTileBytes);
        bulk_commit();
        if (n >= 1) {
          // at most this step's store still reads shared memory: the
          // previous step's buffer is free for step n+1
          bulk_wait_read<1>();
          mbar_arrive(BAR(BAR_DS_STORED + ((n - 1) & 1)));
        }
      }
    }
    if (threadIdx.x == 0) bulk_wait_all<0>();

    // ---------------- epilogue: dK = s * sum (rows), dV^T (columns) ----------------
    const bool store = key < T;
    float* dkrow = a.dk + (((size_t)b * d.Hkv + kv) * T + key) * 64;
    float* dvcol = a.dvt + ((size_t)b * d.Hkv + kv) * 64 * (size_t)T + key;
    if (n_steps > 0) {
      ok = ok && mbar_wait(BAR(BAR_DONE), 0, wc);
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32x2_wait(tmem + lane_base + kColDK, tmem + lane_base + kColDK + 32, r0, r1);
      if (store) {
        float4* dst = reinterpret_cast<float4*>(dkrow);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(as_f(r0[4 * u]) * d.scale, as_f(r0[4 * u + 1]) * d.scale,
                               as_f(r0[4 * u + 2]) * d.scale, as_f(r0[4 * u + 3]) * d.scale);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[8 + u] = make_float4(as_f(r1[4 * u]) * d.scale, as_f(r1[4 * u + 1]) * d.scale,
                                   as_f(r1[4 * u + 2]) * d.scale, as_f(r1[4 * u + 3]) * d.scale);
      }
      tmem_ld32x2_wait(tmem + lane_base + kColDV, tmem + lane_base + kColDV + 32, r0, r1);
      if (store) {
#pragma unroll
        for (int u = 0; u < 32; ++u) dvcol[(size_t)u * T] = as_f(r0[u]);
#pragma unroll
        for (int u = 0; u < 32; ++u) dvcol[(size_t)(32 + u) * T] = as_f(r1[u]);
      }
    } else if (store) {
      float4* dst = reinterpret_cast<float4*>(dkrow);
#pragma unroll
      for (int u = 0; u < 16; ++u) dst[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 64; ++u) dvcol[(size_t)u * T] = 0.f;
    }
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    if (n_steps > 0) drain_wait(BAR(BAR_DONE), 0, a.wait_ns);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef BAR
}

}  // namespace

int launch_bwd_keys(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
                    const uint16_t* vt, const uint16_t* dout, const float* lse,
                    const float* delta, uint8_t* ws, float* dk, float* dvt,
                    cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t T = (uint64_t)d.T;
  if (!encode_tmap_3d(&tq, q, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBQ) ||
      !encode_tmap_3d(&tdo, dout, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBQ) ||
      !encode_tmap_3d(&tk, k, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, kBK) ||
      !encode_tmap_3d(&tv, vt, T, 64, (uint64_t)d.B * d.Hkv, T * 2, T * 128, 64, 64))
    return ATTN_ERR_CUDA;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(bwd_keys_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  KeysArgs args{d, lse, delta, ws, dk, dvt, ctx.err, ctx.wait_ns};
  dim3 grid(d.kv_count, d.nt, d.B);
  bwd_keys_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, tdo, args);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace css
