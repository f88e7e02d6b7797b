// bwd_fused_q.cu - the fused query pass: dQ for one 128-query tile of one
// query head per CTA, with S, P, dP and dS recomputed from Q, K, V, dO, L and
// D instead of read back from a stored dS.
//
// Method (StreamingAttentionSM86.alpha, backward-pass header: the query
// launch streamingAttentionQuerySM86, which forms D for its rows from dO and
// the forward's O, writes it for the key launch, then walks the query tile's
// key tiles up to the diagonal as the forward does, forms P, dP and dS again
// and keeps dQ = s * sum_j dS_j K_j):
//   D = rowsum(dO * O), S = Q K^T, P = 2^(S c - L), dP = dO V^T,
//   dS = P (dP - D), dQ += dS K,
// dS rounded to binary16 before its product, as in the key pass.  It trades
// two recomputed products per tile pair for the dS workspace, whose size and
// traffic grow as T^2: the key pass then runs without storing dS.
//
// GB300 design.
//   warps 0-15  score gradients, thread = query row (tensor-memory lane);
//               warp group w (warps 4w..4w+3) takes keys 32w..32w+31 of a key
//               tile (sixteen warps measured 10% faster than eight warps of
//               two 32-key chunks each)
//   warp 16     TMA producer: Q and dO once, then per key tile K and V^T
//               through a 4-stage ring
//   warps 17-19 MMA issuers: S = Q K^T, dP = dO V^T (A = Q / dO copied into
//               tensor memory once, B = the K tile K-major / the V^T tile as
//               an MN-major V), dQ += dS K (A = dS from tensor memory, B = the
//               K tile MN-major)
// A query row's L and D are per-thread scalars; warps 4-7, which copy dO
// into tensor memory, form D from it and the row's O (binary16 widened,
// binary32 sum) and hand it to the other warps through shared memory.  The S and dP buffer is
// released once the score-gradient warps hold their columns in registers,
// so the next tile's products run during their arithmetic; dS goes into one
// of two pair buffers, which gives dQ += dS K a tile to finish.
//
// Tensor memory (512 columns): Q 0-31, dO 32-63 (binary16 pairs); S 64-191,
// dP 192-319; dS pair buffer b at 320+64b (keys 2i, 2i+1 in column i);
// dQ 448-511, columns 16w..16w+15 read back by warp group w.
#include <math.h>

#include <mutex>

#include "attn_internal.h"
#include "sm103.cuh"

namespace css {
namespace {

constexpr int kBM = 128;  // queries per CTA
constexpr int kBN = 128;  // keys per tile
constexpr int kThreads = 640;
constexpr int kStages = 4;
constexpr uint32_t kSmemQ = 0, kSmemDO = 16384;
constexpr uint32_t kSmemStage0 = 32768;
constexpr uint32_t kStK = 0, kStVT = 16384;  // V^T: two 64-key halves of 64 rows x 128 B
constexpr uint32_t kStageBytes = 32768;
constexpr uint32_t kSmemBar = kSmemStage0 + kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kSmemBar + 256 + 1024;

constexpr uint32_t kColQ = 0, kColDO = 32, kColS = 64, kColDP = 192, kColDS = 320, kColDQ = 448;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_f16_f32(128, 128, 0, 0);   // Q (tmem) x K (K-major)
constexpr uint32_t kIdescDP = idesc_f16_f32(128, 128, 0, 1);  // dO (tmem) x V (MN-major, from V^T)
constexpr uint32_t kIdescDPR = idesc_f16_f32(128, 128, 0, 0); // dO (tmem) x V rows (K-major)
constexpr uint32_t kIdescDQ = idesc_f16_f32(128, 64, 0, 1);   // dS (tmem) x K (MN-major)

enum {
  BAR_QD_FULL = 0,                      // Q and dO tiles landed
  BAR_QD_TMEM,                          // Q, dO in tensor memory, D in shared (256 threads)
  BAR_KV_FULL,                          // [stage] K and V^T landed
  BAR_KV_EMPTY = BAR_KV_FULL + kStages, // [stage] dQ += dS K of the tile done
  BAR_S_FULL = BAR_KV_EMPTY + kStages,  // S and dP of the tile done (2 commits)
  BAR_LOADED,                           // S and dP are in registers (512 threads)
  BAR_P_READY,                          // [2] dS of pair buffer b written (512 threads)
  BAR_PK_FREE = BAR_P_READY + 2,        // [2] dQ += dS K has read pair buffer b
  BAR_DONE = BAR_PK_FREE + 2,           // dQ complete
  BAR_COUNT
};
static_assert(BAR_COUNT * 8 <= 256, "barrier area");

struct FusedArgs {
  Dims d;
  const uint16_t* o;
  const float* lse;
  float* delta;
  float* dq;
  uint32_t* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// dS = P (dP - D) with P = 2^(S c - L) for 32 keys of one query row, packed
// to binary16 pairs.  MASK zeroes the keys outside [0, lim) (local indices).
template <bool MASK>
__device__ __forceinline__ void score_gradients(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                                float c, float L, float D, int lim,
                                                uint32_t (&dd)[16]) {
  const float2 c2 = make_float2(c, c), nl = make_float2(-L, -L), nd = make_float2(-D, -D);
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float2 t = __ffma2_rn(make_float2(as_f(sv[e]), as_f(sv[e + 1])), c2, nl);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASK) {
      if (e >= lim) p.x = 0.f;
      if (e + 1 >= lim) p.y = 0.f;
    }
    const float2 g = __fadd2_rn(make_float2(as_f(dv[e]), as_f(dv[e + 1])), nd);
    const float2 ds = __fmul2_rn(p, g);
    dd[e >> 1] = pack_f16x2(ds.x, ds.y);
  }
}

// 20 warps on four schedulers allow 96 registers a thread.
__global__ void __launch_bounds__(kThreads, 1)
    bwd_fused_q_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_vt,
                       const __grid_constant__ CUtensorMap tm_do, const FusedArgs a) {
  griddep_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_D[kBM];

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar0 = sbase + kSmemBar;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

  const Dims& d = a.d;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = d.kv_begin * d.G + blockIdx.x;
  const int kv = h / d.G;
  const int it = (int)gridDim.y - 1 - (int)blockIdx.y;  // heaviest causal tiles first
  const int b = blockIdx.z;
  const int T = d.T;

  WaitCtl wc{a.err, a.wait_ns, &s_abort};

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(BAR(BAR_QD_FULL), 1);
    mbar_init(BAR(BAR_QD_TMEM), 256);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(BAR_KV_FULL + s), 1);
      mbar_init(BAR(BAR_KV_EMPTY + s), 1);
    }
    mbar_init(BAR(BAR_S_FULL), 2);
    mbar_init(BAR(BAR_LOADED), 512);
    for (int u = 0; u < 2; ++u) {
      mbar_init(BAR(BAR_P_READY + u), 512);
      mbar_init(BAR(BAR_PK_FREE + u), 1);
    }
    mbar_init(BAR(BAR_DONE), 1);
    fence_mbarrier_init();
  }
  if (warp == 17) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
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
  if (d.causal && n_kt * kBN > len) n_kt = (len + kBN - 1) / kBN;

  if (warp == 16) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_kt > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      tma_prefetch_desc(&tm_do);
      const int qplane = b * d.H + h;
      const int kvplane = b * d.Hkv + kv;
      mbar_arrive_expect_tx(BAR(BAR_QD_FULL), 32768);
      tma_load_3d(sbase + kSmemQ, &tm_q, BAR(BAR_QD_FULL), 0, q0, qplane);
      tma_load_3d(sbase + kSmemDO, &tm_do, BAR(BAR_QD_FULL), 0, q0, qplane);
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait(BAR(BAR_KV_EMPTY + s), ((j / kStages) - 1) & 1, wc)) break;
        const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
        mbar_arrive_expect_tx(BAR(BAR_KV_FULL + s), kStageBytes);
        tma_load_3d(st + kStK, &tm_k, BAR(BAR_KV_FULL + s), 0, j * kBN, kvplane);
        if (d.v_rows) {
          tma_load_3d(st + kStVT, &tm_vt, BAR(BAR_KV_FULL + s), 0, j * kBN, kvplane);  // as K
        } else {
          tma_load_3d(st + kStVT, &tm_vt, BAR(BAR_KV_FULL + s), j * kBN, 0, kvplane);
          tma_load_3d(st + kStVT + 8192, &tm_vt, BAR(BAR_KV_FULL + s), j * kBN + 64, 0, kvplane);
        }
        issued = j + 1;
      }
      drain_wait(BAR(BAR_QD_FULL), 0);
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
        drain_wait(BAR(BAR_KV_FULL + j % kStages), (j / kStages) & 1);
    }
  } else if (warp >= 17) {
    // ---------------- MMA issuers ----------------
    const int role = warp - 17;  // 0: S = Q K^T, 1: dP = dO V^T, 2: dQ += dS K
    if (lane == 0 && n_kt > 0) {
      bool ok = true;
      if (role < 2) {
        ok = mbar_wait(BAR(BAR_QD_TMEM), 0, wc);
        const uint32_t a_col = role == 0 ? kColQ : kColDO;
        const uint32_t dcol = tmem + (role == 0 ? kColS : kColDP);
        for (int j = 0; ok && j < n_kt; ++j) {
          const int s = j % kStages;
          if (!mbar_wait(BAR(BAR_KV_FULL + s), (j / kStages) & 1, wc)) break;
          // the score-gradient warps hold tile j-1's S and dP in registers
          if (j >= 1 && !mbar_wait(BAR(BAR_LOADED), (j - 1) & 1, wc)) break;
          tc_fence_after();
          const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
          // reduction over d: four K=16 steps.  K: 32 B along its K-major
          // rows; V from V^T: 16 rows of d (2 KiB) a step, its two 64-key
          // halves 8 KiB apart
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // V given as rows is K-major like K
            const uint64_t bdesc =
                role == 0   ? sdesc_sw128(st + kStK + kk * 32, 16, 1024)
                : d.v_rows ? sdesc_sw128(st + kStVT + kk * 32, 16, 1024)
                           : sdesc_sw128(st + kStVT + kk * 2048, 8192, 1024);
            const uint32_t idesc = role == 0 ? kIdescS : (d.v_rows ? kIdescDPR : kIdescDP);
            mma_ts(dcol, tmem + a_col + kk * 8, bdesc, idesc, kk > 0);
          }
          mma_commit(BAR(BAR_S_FULL));
        }
      } else {
        for (int j = 0; ok && j < n_kt; ++j) {
          const int s = j % kStages;
          const int pb = j & 1;
          if (!mbar_wait(BAR(BAR_P_READY + pb), (j >> 1) & 1, wc)) break;
          tc_fence_after();
          const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
          // reduction over the tile's 128 keys: 16 K rows (2 KiB) a step
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + kColDQ, tmem + kColDS + 64 * pb + 8 * kk,
                   sdesc_sw128(st + kStK + kk * 2048, 8192, 1024), kIdescDQ,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(BAR(BAR_PK_FREE + pb));
          mma_commit(BAR(BAR_KV_EMPTY + s));
        }
        mma_commit(BAR(BAR_DONE));
      }
    }
  } else {
    // ---------------- score gradients: thread = query row ----------------
    const int wg = warp >> 2;  // keys 32wg..32wg+31 of each tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q = q0 + r;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float c = d.c;
    const bool row_ok = q < len;
    // keys below `lim` are valid for this row
    int lim = row_ok ? len : 0;
    if (d.causal) lim = min(lim, q + 1);
    const size_t lrow = ((size_t)b * d.H + h) * T + q;
    const float L = row_ok ? a.lse[lrow] : 0.f;
    bool ok = true;
    if (n_kt > 0 && wg < 2) {
      // the row's O for D, loaded while Q and dO are on their way
      uint4 ov[8];
      if (wg == 1 && row_ok) {
        const uint4* orow =
            reinterpret_cast<const uint4*>(a.o + (((size_t)b * T + q) * d.H + h) * 64);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) ov[ch] = __ldg(orow + ch);
      }
      // Q (warps 0-3) or dO (warps 4-7) row r into tensor memory as A operands
      ok = mbar_wait_warp(BAR(BAR_QD_FULL), 0, wc);
      uint32_t w[32];
      const uint8_t* src = sgen + (wg == 0 ? kSmemQ : kSmemDO);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + sw128_offset(r, ch));
        w[4 * ch] = v.x, w[4 * ch + 1] = v.y, w[4 * ch + 2] = v.z, w[4 * ch + 3] = v.w;
      }
      tmem_st32(tmem + lane_base + (wg == 0 ? kColQ : kColDO), w);
      if (wg == 1) {
        // row terms D = rowsum(dO * O) from the stored binary16 O
        float D = 0.f;
        if (row_ok) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};  // four chains, summed at the end
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint32_t ow[4] = {ov[ch].x, ov[ch].y, ov[ch].z, ov[ch].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t dw = w[4 * ch + u];
              acc[u] = fmaf(f16_bits_to_f32((uint16_t)(dw & 0xFFFFu)),
                            f16_bits_to_f32((uint16_t)(ow[u] & 0xFFFFu)), acc[u]);
              acc[u] = fmaf(f16_bits_to_f32((uint16_t)(dw >> 16)),
                            f16_bits_to_f32((uint16_t)(ow[u] >> 16)), acc[u]);
            }
          }
          D = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        s_D[r] = D;
        if (q < T) a.delta[lrow] = D;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(BAR_QD_TMEM));
    } else if (n_kt == 0 && wg == 1 && q < T) {
      a.delta[lrow] = 0.f;  // no row of this tile sees a key
    }
    // every score-gradient warp takes its row's D from shared memory
    if (n_kt > 0 && !mbar_wait_warp(BAR(BAR_QD_TMEM), 0, wc)) ok = false;
    const float D = n_kt > 0 ? s_D[r] : 0.f;
    for (int j = 0; ok && j < n_kt; ++j) {
      const int pb = j & 1;
      const int k0 = j * kBN + 32 * wg;  // this thread's first key
      // S and dP of tile j done; pair buffer pb last read by dQ += dS K of
      // tile j-2: one vote for both, bounded waits only when one is not ready
      {
        const bool f1 = mbar_try_wait(BAR(BAR_S_FULL), j & 1);
        const bool f2 = j < 2 || mbar_try_wait(BAR(BAR_PK_FREE + pb), ((j >> 1) - 1) & 1);
        if (!__all_sync(0xffffffffu, f1 && f2)) {
          if (!mbar_wait_warp(BAR(BAR_S_FULL), j & 1, wc)) {
            ok = false;
            break;
          }
          if (j >= 2 && !mbar_wait_warp(BAR(BAR_PK_FREE + pb), ((j >> 1) - 1) & 1, wc)) {
            ok = false;
            break;
          }
        }
      }
      tc_fence_after();
      {
        uint32_t sv[32], dv[32];
        const uint32_t col = 32 * wg;
        tmem_ld32x2_wait(tmem + lane_base + kColS + col, tmem + lane_base + kColDP + col, sv, dv);
        tc_fence_before();
        mbar_arrive(BAR(BAR_LOADED));
        const int lim_local = lim - k0;
        uint32_t dd[16];
        if (lim_local < 32)
          score_gradients<true>(sv, dv, c, L, D, lim_local, dd);
        else
          score_gradients<false>(sv, dv, c, L, D, lim_local, dd);
        tmem_st16(tmem + lane_base + kColDS + 64 * pb + 16 * wg, dd);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(BAR_P_READY + pb));
    }

    // ---------------- epilogue: dQ = s * sum; warp group w takes columns 32w.. ----------------
    if (q < T) {
      float* dst = a.dq + lrow * 64 + 16 * wg;
      if (n_kt > 0) {
        ok = mbar_wait_warp(BAR(BAR_DONE), 0, wc) && ok;
        tc_fence_after();
        uint32_t r0[16];
        // ok is warp-uniform; after a wait gave up the load is skipped
        if (ok) {
          tmem_ld16_wait(tmem + lane_base + kColDQ + 16 * wg, r0);
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) r0[u] = 0u;
        }
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          d4[u] = make_float4(as_f(r0[4 * u]) * d.scale, as_f(r0[4 * u + 1]) * d.scale,
                              as_f(r0[4 * u + 2]) * d.scale, as_f(r0[4 * u + 3]) * d.scale);
      } else {
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int u = 0; u < 4; ++u) d4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else if (n_kt > 0) {
      ok = mbar_wait_warp(BAR(BAR_DONE), 0, wc) && ok;
    }
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    if (n_kt > 0) drain_wait(BAR(BAR_DONE), 0);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef BAR
}


// ---------------------------------------------------------------------------
// The same pass with persistent CTAs.  Each CTA walks its share of the work
// units (one 128-query tile of one query head), heaviest first in snake order
// over the list (CTA c of G takes units c, 2G-1-c, 2G+c, ...), keeping its
// tensor memory, barriers and K/V^T ring from one unit to the next.  The
// producer loads the next unit's Q, dO and O tiles into the other of two
// shared-memory buffers while the current unit runs; at the end of a unit's
// key tiles, warps 0-7 put the next unit's Q and dO into tensor memory and
// form its D (from the shared O and dO tiles) before the current unit's dQ
// epilogue, so the next unit's first S and dP run during that epilogue.  The
// per-tile work is the non-persistent kernel's, in the same order: the
// results are the same bits.  Used when the shape has no per-sequence
// lengths (every unit then has at least one key tile) and at least two units
// per SM.
// ---------------------------------------------------------------------------
constexpr int kStagesP = 3;
constexpr uint32_t kQdoBytes = 3 * 16384;  // Q, dO, O tiles of one unit
constexpr uint32_t kSmemRingP = 2 * kQdoBytes;
constexpr uint32_t kSmemBarP = kSmemRingP + kStagesP * kStageBytes;
constexpr uint32_t kSmemBytesP = kSmemBarP + 256 + 1024;
static_assert(kSmemBytesP + 3072 <= 232448, "shared memory of the persistent pass");

enum {
  PB_QD_FULL = 0,                          // [buffer] Q, dO, O tiles landed
  PB_QD_FREE = PB_QD_FULL + 2,             // [buffer] read into tensor memory / D (256 threads)
  PB_QD_TMEM = PB_QD_FREE + 2,             // the unit's Q, dO in tensor memory, D shared (256)
  PB_KV_FULL,                              // [stage] K and V^T landed
  PB_KV_EMPTY = PB_KV_FULL + kStagesP,     // [stage] dQ += dS K of the tile done
  PB_S_FULL = PB_KV_EMPTY + kStagesP,      // S and dP of the tile done (2 commits)
  PB_LOADED,                               // S and dP are in registers (512 threads)
  PB_P_READY,                              // [2] dS of pair buffer b written (512 threads)
  PB_PK_FREE = PB_P_READY + 2,             // [2] dQ += dS K has read pair buffer b
  PB_DONE = PB_PK_FREE + 2,                // the unit's dQ complete
  PB_DQ_FREE,                              // the epilogue has read dQ (512 threads)
  PB_MMA_DONE,                             // every MMA of the CTA done (3 issuer commits)
  PB_COUNT
};
static_assert(PB_COUNT * 8 <= 256, "barrier area");

struct FusedUnit {
  int h, b, it, q0, n_kt;
};

// Units: head of the chunk fastest, then query tiles from the last (longest
// causal rows), then batch entries.
__device__ __forceinline__ FusedUnit fused_unit_at(const Dims& d, int u) {
  FusedUnit w;
  const int hc = d.kv_count * d.G;
  w.h = d.kv_begin * d.G + u % hc;
  const int r = u / hc;
  w.it = d.nt - 1 - r % d.nt;
  w.b = r / d.nt;
  w.q0 = w.it * kBM;
  w.n_kt = d.causal ? w.it + 1 : d.nt;
  return w;
}

// The i-th unit of this CTA (snake order over the list), or -1 past the end.
__device__ __forceinline__ int fused_unit_index(int units, int i) {
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const long long u = (long long)i * G + ((i & 1) ? (G - 1 - c) : c);
  return u < units ? (int)u : -1;
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_fused_q_persistent(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_vt,
                           const __grid_constant__ CUtensorMap tm_do,
                           const __grid_constant__ CUtensorMap tm_o, const FusedArgs a, int units) {
  griddep_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_D[2][kBM];
  __shared__ float s_L[2][kBM];

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar0 = sbase + kSmemBarP;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

  const Dims& d = a.d;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = d.T;

  WaitCtl wc{a.err, a.wait_ns, &s_abort};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int u = 0; u < 2; ++u) {
      mbar_init(BAR(PB_QD_FULL + u), 1);
      mbar_init(BAR(PB_QD_FREE + u), 256);
    }
    mbar_init(BAR(PB_QD_TMEM), 256);
    for (int s = 0; s < kStagesP; ++s) {
      mbar_init(BAR(PB_KV_FULL + s), 1);
      mbar_init(BAR(PB_KV_EMPTY + s), 1);
    }
    mbar_init(BAR(PB_S_FULL), 2);
    mbar_init(BAR(PB_LOADED), 512);
    for (int u = 0; u < 2; ++u) {
      mbar_init(BAR(PB_P_READY + u), 512);
      mbar_init(BAR(PB_PK_FREE + u), 1);
    }
    mbar_init(BAR(PB_DONE), 1);
    mbar_init(BAR(PB_DQ_FREE), 512);
    mbar_init(BAR(PB_MMA_DONE), 3);
    fence_mbarrier_init();
  }
  if (warp == 17) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  griddep_wait();

  if (warp == 16) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_o);
      int kt = 0, nq = 0;  // key tiles issued, Q/dO/O buffers issued
      bool ok = true;
      // Q, dO and O of the CTA's i-th unit into buffer i & 1, once the unit
      // that used it before (i - 2) has read it
      auto issue_qdo = [&](int i) -> bool {
        const int u = fused_unit_index(units, i);
        if (u < 0) return true;
        const FusedUnit w = fused_unit_at(d, u);
        const int ub = i & 1;
        if (i >= 2 && !mbar_wait(BAR(PB_QD_FREE + ub), ((i >> 1) - 1) & 1, wc)) return false;
        const uint32_t buf = sbase + ub * kQdoBytes;
        const int qplane = w.b * d.H + w.h;
        mbar_arrive_expect_tx(BAR(PB_QD_FULL + ub), kQdoBytes);
        tma_load_3d(buf, &tm_q, BAR(PB_QD_FULL + ub), 0, w.q0, qplane);
        tma_load_3d(buf + 16384, &tm_do, BAR(PB_QD_FULL + ub), 0, w.q0, qplane);
        tma_load_3d(buf + 32768, &tm_o, BAR(PB_QD_FULL + ub), w.h * 64, w.q0, w.b);
        nq = i + 1;
        return true;
      };
      ok = issue_qdo(0);
      for (int i = 0; ok; ++i) {
        const int u = fused_unit_index(units, i);
        if (u < 0) break;
        const FusedUnit w = fused_unit_at(d, u);
        if (!(ok = issue_qdo(i + 1))) break;
        const int kvplane = w.b * d.Hkv + w.h / d.G;
        for (int j = 0; j < w.n_kt; ++j, ++kt) {
          const int s = kt % kStagesP;
          if (kt >= kStagesP &&
              !mbar_wait(BAR(PB_KV_EMPTY + s), ((kt / kStagesP) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + kSmemRingP + s * kStageBytes;
          mbar_arrive_expect_tx(BAR(PB_KV_FULL + s), kStageBytes);
          tma_load_3d(st + kStK, &tm_k, BAR(PB_KV_FULL + s), 0, j * kBN, kvplane);
          if (d.v_rows) {
            tma_load_3d(st + kStVT, &tm_vt, BAR(PB_KV_FULL + s), 0, j * kBN, kvplane);
          } else {
            tma_load_3d(st + kStVT, &tm_vt, BAR(PB_KV_FULL + s), j * kBN, 0, kvplane);
            tma_load_3d(st + kStVT + 8192, &tm_vt, BAR(PB_KV_FULL + s), j * kBN + 64, 0,
                        kvplane);
          }
        }
      }
      // every copy this thread issued has landed before the CTA ends
      for (int i = (nq > 2 ? nq - 2 : 0); i < nq; ++i)
        drain_wait(BAR(PB_QD_FULL + (i & 1)), (i >> 1) & 1);
      for (int k = (kt > kStagesP ? kt - kStagesP : 0); k < kt; ++k)
        drain_wait(BAR(PB_KV_FULL + k % kStagesP), (k / kStagesP) & 1);
    }
  } else if (warp >= 17) {
    // ---------------- MMA issuers ----------------
    const int role = warp - 17;  // 0: S = Q K^T, 1: dP = dO V^T, 2: dQ += dS K
    if (lane == 0) {
      bool ok = true;
      int kt = 0;  // key tiles of this CTA so far (ring stage, pair buffer, phases)
      for (int i = 0; ok; ++i) {
        const int u = fused_unit_index(units, i);
        if (u < 0) break;
        const int n_kt = fused_unit_at(d, u).n_kt;
        if (role < 2) {
          // the unit's Q and dO are in tensor memory
          if (!mbar_wait(BAR(PB_QD_TMEM), i & 1, wc)) break;
          const uint32_t a_col = role == 0 ? kColQ : kColDO;
          const uint32_t dcol = tmem + (role == 0 ? kColS : kColDP);
          for (int j = 0; j < n_kt; ++j, ++kt) {
            const int s = kt % kStagesP;
            if (!mbar_wait(BAR(PB_KV_FULL + s), (kt / kStagesP) & 1, wc) ||
                (kt >= 1 && !mbar_wait(BAR(PB_LOADED), (kt - 1) & 1, wc))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = sbase + kSmemRingP + s * kStageBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc =
                  role == 0   ? sdesc_sw128(st + kStK + kk * 32, 16, 1024)
                  : d.v_rows ? sdesc_sw128(st + kStVT + kk * 32, 16, 1024)
                             : sdesc_sw128(st + kStVT + kk * 2048, 8192, 1024);
              const uint32_t idesc = role == 0 ? kIdescS : (d.v_rows ? kIdescDPR : kIdescDP);
              mma_ts(dcol, tmem + a_col + kk * 8, bdesc, idesc, kk > 0);
            }
            mma_commit(BAR(PB_S_FULL));
          }
        } else {
          for (int j = 0; j < n_kt; ++j, ++kt) {
            const int s = kt % kStagesP;
            const int pb = kt & 1;
            if (!mbar_wait(BAR(PB_P_READY + pb), (kt >> 1) & 1, wc) ||
                // the unit's first product overwrites dQ: the previous
                // unit's epilogue must have read it
                (j == 0 && i >= 1 && !mbar_wait(BAR(PB_DQ_FREE), (i - 1) & 1, wc))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = sbase + kSmemRingP + s * kStageBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + kColDQ, tmem + kColDS + 64 * pb + 8 * kk,
                     sdesc_sw128(st + kStK + kk * 2048, 8192, 1024), kIdescDQ,
                     (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(BAR(PB_PK_FREE + pb));
            mma_commit(BAR(PB_KV_EMPTY + s));
          }
          if (ok) mma_commit(BAR(PB_DONE));
        }
      }
      mma_commit(BAR(PB_MMA_DONE));  // all of this thread's products, for the exit
    }
  } else {
    // ---------------- score gradients: thread = query row ----------------
    const int wg = warp >> 2;  // keys 32wg..32wg+31 of each tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float c = d.c;
    bool ok = true;
    // Warps 0-7: the i-th unit's Q (warps 0-3) or dO (warps 4-7) row r into
    // tensor memory as A operands; warps 4-7 also form the row's D from the
    // shared dO and O tiles (binary16 widened, binary32 sum, as the
    // non-persistent kernel does) and write it, and put the row's L in
    // shared memory (so no unit starts with a global load).
    auto prepare = [&](int i) -> bool {
      const int u = fused_unit_index(units, i);
      if (u < 0) return true;
      const FusedUnit w = fused_unit_at(d, u);
      const int ub = i & 1;
      const int qn = w.q0 + r;
      const float Ln = (wg == 1 && qn < T) ? a.lse[((size_t)w.b * d.H + w.h) * T + qn] : 0.f;
      if (!mbar_wait_warp(BAR(PB_QD_FULL + ub), (i >> 1) & 1, wc)) return false;
      const uint8_t* buf = sgen + ub * kQdoBytes;
      uint32_t wv[32];
      const uint8_t* src = buf + (wg == 0 ? 0 : 16384);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + sw128_offset(r, ch));
        wv[4 * ch] = v.x, wv[4 * ch + 1] = v.y, wv[4 * ch + 2] = v.z, wv[4 * ch + 3] = v.w;
      }
      tmem_st32(tmem + lane_base + (wg == 0 ? kColQ : kColDO), wv);
      if (wg == 1) {
        const int q = w.q0 + r;
        float D = 0.f;
        if (q < T) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};  // four chains, summed at the end
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 ov = *reinterpret_cast<const uint4*>(buf + 32768 + sw128_offset(r, ch));
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t dw = wv[4 * ch + e];
              acc[e] = fmaf(f16_bits_to_f32((uint16_t)(dw & 0xFFFFu)),
                            f16_bits_to_f32((uint16_t)(ow[e] & 0xFFFFu)), acc[e]);
              acc[e] = fmaf(f16_bits_to_f32((uint16_t)(dw >> 16)),
                            f16_bits_to_f32((uint16_t)(ow[e] >> 16)), acc[e]);
            }
          }
          D = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          a.delta[((size_t)w.b * d.H + w.h) * T + q] = D;
        }
        s_D[ub][r] = D;
        s_L[ub][r] = Ln;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(PB_QD_FREE + ub));
      mbar_arrive(BAR(PB_QD_TMEM));
      return true;
    };
    if (wg < 2) ok = prepare(0);
    int kt = 0;  // key tiles of this CTA so far
    for (int i = 0; ok; ++i) {
      const int u = fused_unit_index(units, i);
      if (u < 0) break;
      const FusedUnit w = fused_unit_at(d, u);
      const int q = w.q0 + r;
      const bool row_ok = q < T;
      // keys below `lim` are valid for this row
      int lim = row_ok ? T : 0;
      if (d.causal) lim = min(lim, q + 1);
      const size_t lrow = ((size_t)w.b * d.H + w.h) * T + q;
      // the unit's Q, dO are in tensor memory and its D and L in shared memory
      if (!mbar_wait_warp(BAR(PB_QD_TMEM), i & 1, wc)) {
        ok = false;
        break;
      }
      const float D = s_D[i & 1][r];
      const float L = s_L[i & 1][r];
      for (int j = 0; j < w.n_kt; ++j, ++kt) {
        const int pb = kt & 1;
        const int k0 = j * kBN + 32 * wg;  // this thread's first key
        {
          const bool f1 = mbar_try_wait(BAR(PB_S_FULL), kt & 1);
          const bool f2 = kt < 2 || mbar_try_wait(BAR(PB_PK_FREE + pb), ((kt >> 1) - 1) & 1);
          if (!__all_sync(0xffffffffu, f1 && f2)) {
            if (!mbar_wait_warp(BAR(PB_S_FULL), kt & 1, wc) ||
                (kt >= 2 && !mbar_wait_warp(BAR(PB_PK_FREE + pb), ((kt >> 1) - 1) & 1, wc))) {
              ok = false;
              break;
            }
          }
        }
        tc_fence_after();
        {
          uint32_t sv[32], dv[32];
          const uint32_t col = 32 * wg;
          tmem_ld32x2_wait(tmem + lane_base + kColS + col, tmem + lane_base + kColDP + col, sv,
                           dv);
          tc_fence_before();
          mbar_arrive(BAR(PB_LOADED));
          const int lim_local = lim - k0;
          uint32_t dd[16];
          if (lim_local < 32)
            score_gradients<true>(sv, dv, c, L, D, lim_local, dd);
          else
            score_gradients<false>(sv, dv, c, L, D, lim_local, dd);
          tmem_st16(tmem + lane_base + kColDS + 64 * pb + 16 * wg, dd);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(PB_P_READY + pb));
      }
      if (!ok) break;
      // the next unit's Q and dO go into tensor memory (its S and dP can then
      // run) before this unit's epilogue
      if (wg < 2 && !prepare(i + 1)) {
        ok = false;
        break;
      }
      // ---------------- epilogue: dQ = s * sum; warp group w takes columns 16w.. ----------------
      if (!mbar_wait_warp(BAR(PB_DONE), i & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r0[16];
      tmem_ld16_wait(tmem + lane_base + kColDQ + 16 * wg, r0);
      tc_fence_before();
      mbar_arrive(BAR(PB_DQ_FREE));  // the next unit's first product may overwrite dQ
      if (row_ok) {
        float4* d4 = reinterpret_cast<float4*>(a.dq + lrow * 64 + 16 * wg);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          d4[e] = make_float4(as_f(r0[4 * e]) * d.scale, as_f(r0[4 * e + 1]) * d.scale,
                              as_f(r0[4 * e + 2]) * d.scale, as_f(r0[4 * e + 3]) * d.scale);
      }
    }
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    // every product of this CTA has completed before its tensor memory is freed
    drain_wait(BAR(PB_MMA_DONE), 0);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef BAR
}

}  // namespace

int launch_bwd_fused_q(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
                       const uint16_t* vt, const uint16_t* dout, const uint16_t* o,
                       const float* lse, float* delta, float* dq, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t T = (uint64_t)d.T;
  if (!encode_tmap_3d(&tq, q, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBM) ||
      !encode_tmap_3d(&tdo, dout, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBM) ||
      !encode_tmap_3d(&tk, k, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, kBN) ||
      !(d.v_rows ? encode_tmap_3d(&tv, vt, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, 128)
                  : encode_tmap_3d(&tv, vt, T, 64, (uint64_t)d.B * d.Hkv, T * 2, T * 128, 64, 64)))
    return ATTN_ERR_CUDA;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_status[64];
  std::call_once(attr_once[dev & 63], [dev] {
    attr_status[dev & 63] = cudaFuncSetAttribute(
        bwd_fused_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_status[dev & 63] != cudaSuccess) return cuda_status(attr_status[dev & 63]);
  FusedArgs args{d, o, lse, delta, dq, ctx.err, ctx.wait_ns};
  const long long units = (long long)d.kv_count * d.G * d.nt * d.B;
  // Persistent (one CTA per SM walking its share of the units) when there are
  // no per-sequence lengths and at least two units per SM: the next unit's
  // loads and set-up then overlap the current one.  Measured on GB300: T =
  // 4096, 32 heads (1024 units) 129 -> 117 us, T = 16384 (4096 units)
  // 1.516 -> 1.476 ms; with at most one unit per SM (T = 128 and T = 1024
  // workloads) the persistent kernel was 2-3 us slower.
  if (d.lens == nullptr && units >= 2LL * ctx.sm_count) {
    if (units > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    CUtensorMap to;
    if (!encode_tmap_3d(&to, o, (uint64_t)d.H * 64, T, (uint64_t)d.B, (uint64_t)d.H * 128,
                        T * d.H * 128, 64, kBM))
      return ATTN_ERR_CUDA;
    static std::once_flag pattr_once[64];
    static cudaError_t pattr_status[64];
    std::call_once(pattr_once[dev & 63], [dev] {
      pattr_status[dev & 63] = cudaFuncSetAttribute(
          bwd_fused_q_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytesP);
    });
    if (pattr_status[dev & 63] != cudaSuccess) return cuda_status(pattr_status[dev & 63]);
    const long long ctas = units < ctx.sm_count ? units : ctx.sm_count;
    return cuda_status(launch_dependent(bwd_fused_q_persistent, dim3((unsigned)ctas),
                                        dim3(kThreads), kSmemBytesP, stream, tq, tk, tv, tdo, to,
                                        args, (int)units));
  }
  dim3 grid(d.kv_count * d.G, d.nt, d.B);
  return cuda_status(launch_dependent(bwd_fused_q_kernel, grid, dim3(kThreads), kSmemBytes, stream,
                                     tq, tk, tv, tdo, args));
}

}  // namespace css
