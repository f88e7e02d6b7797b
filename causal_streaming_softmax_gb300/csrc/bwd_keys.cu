// bwd_keys.cu - the key pass of the backward: one 128-key tile of one K/V
// head per CTA, walking every query head of the head's group and every
// 64-query half of each 128-query tile that can see the keys.
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
// GB300 design.
//   warps 0-7   score gradients, thread = key row (tensor-memory lane); warps
//               0-3 take queries 0-31 of a step, warps 4-7 queries 32-63
//   warp 8      TMA producer: K and V^T once, then per step a 64-query tile
//               of Q and dO and their L and D, through an 8-stage ring
//   warps 9-12  MMA issuers, one per product chain: S^T, dP^T, dV, dK
//   warp 13     store: one 16 KiB bulk store of each step's dS^T
// Every MMA reads its A operand from tensor memory and its B operand (a Q or
// dO tile, 8 KiB) from shared memory: K and V are copied into tensor memory
// once.  The score-gradient warps load a step's S^T and dP^T into registers
// and release the buffer at once, so the next step's S^T and dP^T run while
// they compute; they write P^T and dS^T as binary16 pairs into one of two
// separate buffers, which dV and dK read, so the accumulation of a step has
// two steps to finish.  With those latencies off the loop, a step costs the
// score-gradient work.  The four product chains are issued by four warps.
// dK and dV sum the group's query heads in tensor memory (no atomics, fixed
// order).  dS^T also goes to shared memory (three buffers) in the
// 128-byte-swizzled image the dQ pass reads; the store warp copies it into
// the workspace, so no score-gradient warp ever waits for a store.  Without a
// workspace (the fused query pass recomputes dS) the staging and the store
// are skipped.
//
// Tensor memory (512 columns): K 0-31, V 32-63 (binary16 pairs), S^T 64-127,
// dP^T 128-191; pair buffer b at 192+64b: P^T of queries 32w..32w+31 at
// 16w..16w+15, dS^T likewise at 32+16w; dK 320-383, dV 384-447.
#include <math.h>

#include <mutex>

#include "attn_internal.h"
#include "epilogue.cuh"
#include "sm103.cuh"

namespace css {
namespace {

constexpr int kBK = 128;  // keys per CTA
constexpr int kBQ = 64;   // queries per step
constexpr int kThreads = 448;
constexpr int kStages = 8;
constexpr uint32_t kSmemK = 0;                // K tile: 128 rows x 128 B
constexpr uint32_t kSmemV = 16384;            // V^T: two 64-key halves of 64 rows x 128 B
constexpr uint32_t kSmemStage0 = 32768;
constexpr uint32_t kStQ = 0, kStDO = 8192, kStL = 16384, kStD = 16640;
constexpr uint32_t kStageBytes = 17408;       // a multiple of 1024
constexpr uint32_t kSmemDS0 = kSmemStage0 + kStages * kStageBytes;
constexpr uint32_t kDSHalf = 16384;           // one 64-query half of a workspace tile
constexpr int kDSBufs = 3;                    // shared dS^T staging buffers
constexpr uint32_t kSmemBar = kSmemDS0 + kDSBufs * kDSHalf;
constexpr uint32_t kSmemBytes = kSmemBar + 256 + 1024;

constexpr uint32_t kColK = 0, kColV = 32, kColS = 64, kColDP = 128, kColPK = 192;
constexpr uint32_t kColDK = 320, kColDV = 384;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_f16_f32(128, 64, 0, 0);    // A (tmem) x Q / dO (K-major)
constexpr uint32_t kIdescAcc = idesc_f16_f32(128, 64, 0, 1);  // P^T / dS^T (tmem) x dO / Q (MN-major)

// Tensor-memory column (within the 32 P^T or dS^T columns of a pair buffer)
// of the binary16 pairs of queries 16kk..16kk+15.
__host__ __device__ constexpr uint32_t packed_col(int kk) { return 8 * kk; }

enum {
  BAR_KV_FULL = 0,
  BAR_KV_TMEM,                          // K and V in tensor memory (256 threads)
  BAR_Q_FULL,                           // [stage] Q, dO, L, D landed
  BAR_Q_EMPTY = BAR_Q_FULL + kStages,   // [stage] dV and dK of the step are done (2 commits)
  BAR_S_FULL = BAR_Q_EMPTY + kStages,   // S^T and dP^T of the step are done (2 commits)
  BAR_LOADED,                           // S^T and dP^T are in registers (256 threads)
  BAR_P_READY,                          // [2] P^T / dS^T of pair buffer b written (256 threads)
  BAR_PK_FREE = BAR_P_READY + 2,        // [2] dV and dK have read pair buffer b (2 commits)
  BAR_DS_STORED = BAR_PK_FREE + 2,      // [3] the bulk store has read shared dS^T buffer b
  BAR_DONE = BAR_DS_STORED + kDSBufs,   // dK and dV complete (2 commits)
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
  Projection pk, pv;  // token-major dK / dV blocks instead of dk, dvt (when on)
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// One key row's step for 32 queries: P = 2^(S c - L) and dS = P (dP - D),
// both packed to binary16 pairs (P for dV, dS for dK and the workspace); dS
// takes P unrounded.  MASK zeroes P, so also dS, outside [qlo, qhi) (local
// query indices).  Both formulas sit in one basic block, so the compiler can
// interleave one pair's exponentials with another pair's score-gradient
// arithmetic (separate blocks cost 5% of the kernel); dP - D is one FFMA2
// with factor -1, which rounds exactly as the subtraction.
template <bool MASK>
__device__ __forceinline__ void step_math(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                          const float4* __restrict__ L4,
                                          const float4* __restrict__ D4, float c, int qlo,
                                          int qhi, uint32_t (&pp)[16], uint32_t (&dd)[16]) {
  const float2 c2 = make_float2(c, c);
  const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 l = L4[u];
    const float4 dl = D4[u];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 4 * u + 2 * h;
      const float2 nl = h ? make_float2(-l.z, -l.w) : make_float2(-l.x, -l.y);
      const float2 d2 = h ? make_float2(dl.z, dl.w) : make_float2(dl.x, dl.y);
      const float2 t = __ffma2_rn(make_float2(as_f(sv[e]), as_f(sv[e + 1])), c2, nl);
      float2 q = make_float2(ex2_approx(t.x), ex2_approx(t.y));
      if (MASK) {
        if (e < qlo || e >= qhi) q.x = 0.f;
        if (e + 1 < qlo || e + 1 >= qhi) q.y = 0.f;
      }
      pp[e >> 1] = pack_f16x2(q.x, q.y);
      const float2 g = __ffma2_rn(d2, m1, make_float2(as_f(dv[e]), as_f(dv[e + 1])));
      const float2 ds = __fmul2_rn(q, g);
      dd[e >> 1] = pack_f16x2(ds.x, ds.y);
    }
  }
}

// 14 warps put four on a scheduler, which caps a thread at 128 registers.
// STORE: dS^T is kept in the workspace (fixed per launch, so the step loop
// carries only its own waits).
template <bool STORE>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_keys_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_vt,
                    const __grid_constant__ CUtensorMap tm_do, const KeysArgs a) {
  griddep_launch_dependents();
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

  WaitCtl wc{a.err, a.wait_ns, &s_abort};

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(BAR(BAR_KV_FULL), 1);
    mbar_init(BAR(BAR_KV_TMEM), 256);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(BAR_Q_FULL + s), 1);
      mbar_init(BAR(BAR_Q_EMPTY + s), 2);
    }
    mbar_init(BAR(BAR_S_FULL), 2);
    mbar_init(BAR(BAR_LOADED), 256);
    for (int u = 0; u < 2; ++u) {
      mbar_init(BAR(BAR_P_READY + u), 256);
      mbar_init(BAR(BAR_PK_FREE + u), 2);
    }
    for (int u = 0; u < kDSBufs; ++u) mbar_init(BAR(BAR_DS_STORED + u), 1);
    mbar_init(BAR(BAR_DONE), 2);
    fence_mbarrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
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
  const int k0 = jt * kBK;
  const int i_lo = d.causal ? jt : 0;
  int i_hi = (len + kTile - 1) / kTile;
  if (k0 >= len) i_hi = i_lo;
  const int n_i = i_hi > i_lo ? i_hi - i_lo : 0;
  // 64-query halves per query head: the second half of a tile that starts at
  // or past T holds no row and is skipped (its rows are never stored).
  const bool half_tail = n_i > 0 && (i_hi - 1) * kTile + kBQ >= T;
  const int per_g = n_i > 0 ? 2 * n_i - (half_tail ? 1 : 0) : 0;
  const int n_steps = d.G * per_g;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_steps > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      tma_prefetch_desc(&tm_do);
      const int kvplane = b * d.Hkv + kv;
      mbar_arrive_expect_tx(BAR(BAR_KV_FULL), 32768);
      tma_load_3d(sbase + kSmemK, &tm_k, BAR(BAR_KV_FULL), 0, k0, kvplane);
      if (d.v_rows) {
        tma_load_3d(sbase + kSmemV, &tm_vt, BAR(BAR_KV_FULL), 0, k0, kvplane);  // V rows, as K
      } else {
        tma_load_3d(sbase + kSmemV, &tm_vt, BAR(BAR_KV_FULL), k0, 0, kvplane);
        tma_load_3d(sbase + kSmemV + 8192, &tm_vt, BAR(BAR_KV_FULL), k0 + 64, 0, kvplane);
      }
      int issued = 0, g = 0, rem = 0;
      for (int n = 0; n < n_steps; ++n) {
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait(BAR(BAR_Q_EMPTY + s), ((n / kStages) - 1) & 1, wc)) break;
        const int q0 = (i_lo + (rem >> 1)) * kTile + (rem & 1) * kBQ;
        const int qplane = b * d.H + kv * d.G + g;
        const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
        mbar_arrive_expect_tx(BAR(BAR_Q_FULL + s), 2 * 8192 + 2 * kBQ * 4);
        tma_load_3d(st + kStQ, &tm_q, BAR(BAR_Q_FULL + s), 0, q0, qplane);
        tma_load_3d(st + kStDO, &tm_do, BAR(BAR_Q_FULL + s), 0, q0, qplane);
        const size_t lo = (size_t)qplane * T + (size_t)q0;
        bulk_load(st + kStL, a.lse + lo, kBQ * 4, BAR(BAR_Q_FULL + s));
        bulk_load(st + kStD, a.delta + lo, kBQ * 4, BAR(BAR_Q_FULL + s));
        issued = n + 1;
        if (++rem == per_g) rem = 0, ++g;
      }
      drain_wait(BAR(BAR_KV_FULL), 0);
      for (int n = (issued > kStages ? issued - kStages : 0); n < issued; ++n)
        drain_wait(BAR(BAR_Q_FULL + n % kStages), (n / kStages) & 1);
    }
  } else if (warp == 13) {
    // ---------------- store: dS^T of each step into the workspace ----------------
    // (no workspace: dS is not kept, for a dQ pass that recomputes it)
    if (STORE && lane == 0 && n_steps > 0) {
      const int Hc = d.ws_heads ? d.ws_heads : d.kv_count * d.G;
      const int h_local0 = d.ws_h0 + (kv - d.kv_begin) * d.G;
      int g = 0, rem = 0;
      for (int n = 0; n < n_steps; ++n) {
        // every row of the step's dS^T is in shared memory (and fenced for
        // the async proxy) once all 256 score-gradient threads arrived
        if (!mbar_wait(BAR(BAR_P_READY + (n & 1)), (n >> 1) & 1, wc)) break;
        const int it = i_lo + (rem >> 1);
        const int hq = rem & 1;
        const long long tile = ((long long)b * Hc + h_local0 + g) * d.npairs + d.pair(it, jt);
        if (++rem == per_g) rem = 0, ++g;
        bulk_store(a.ws + (size_t)tile * kDsTileBytes + (size_t)hq * kDSHalf,
                   sbase + kSmemDS0 + (n % kDSBufs) * kDSHalf, kDSHalf);
        bulk_commit();
        if (n >= 1) {
          // at most this step's store still reads shared memory: the previous
          // step's buffer is free for step n + 2
          bulk_wait_read<1>();
          mbar_arrive(BAR(BAR_DS_STORED + (n - 1) % kDSBufs));
        }
      }
      bulk_wait_all<0>();
    }
  } else if (warp >= 9) {
    // ---------------- MMA issuers: one thread per product chain ----------------
    const int role = warp - 9;  // 0: S^T = K Q^T, 1: dP^T = V dO^T, 2: dV += P^T dO, 3: dK += dS^T Q
    if (lane == 0 && n_steps > 0) {
      bool ok = true;
      if (role < 2) {
        ok = mbar_wait(BAR(BAR_KV_TMEM), 0, wc);
        const uint32_t a_col = role == 0 ? kColK : kColV;
        const uint32_t b_off = role == 0 ? kStQ : kStDO;
        const uint32_t d = tmem + (role == 0 ? kColS : kColDP);
        for (int n = 0; ok && n < n_steps; ++n) {
          const int s = n % kStages;
          if (!mbar_wait(BAR(BAR_Q_FULL + s), (n / kStages) & 1, wc)) break;
          // the score-gradient warps hold step n-1's S^T and dP^T in registers
          if (n >= 1 && !mbar_wait(BAR(BAR_LOADED), (n - 1) & 1, wc)) break;
          tc_fence_after();
          const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
          // reduction over d: four K=16 steps of 32 B
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(d, tmem + a_col + kk * 8, sdesc_sw128(st + b_off + kk * 32, 16, 1024), kIdescS,
                   kk > 0);
          mma_commit(BAR(BAR_S_FULL));
        }
      } else {
        const uint32_t d = tmem + (role == 2 ? kColDV : kColDK);
        const uint32_t b_off = role == 2 ? kStDO : kStQ;
        for (int n = 0; ok && n < n_steps; ++n) {
          const int s = n % kStages;
          const int pb = n & 1;
          if (!mbar_wait(BAR(BAR_P_READY + pb), (n >> 1) & 1, wc)) break;
          tc_fence_after();
          const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
          // P^T (dV) or dS^T (dK) of pair buffer pb
          const uint32_t a_base = tmem + kColPK + 64 * pb + (role == 2 ? 0 : 32);
          // reduction over the step's 64 queries: 16 rows (2 KiB) of the
          // MN-major dO / Q tile per K step
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(d, a_base + packed_col(kk), sdesc_sw128(st + b_off + kk * 2048, 8192, 1024),
                   kIdescAcc, (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(BAR(BAR_PK_FREE + pb));
          mma_commit(BAR(BAR_Q_EMPTY + s));
        }
        mma_commit(BAR(BAR_DONE));
      }
    }
  } else {
    // ---------------- score gradients: thread = key row ----------------
    const int wg = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int key = k0 + r;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float c = d.c;
    bool ok = true;
    if (n_steps > 0) {
      // K (warps 0-3) or V (warps 4-7) row r into tensor memory as A operands
      ok = mbar_wait_warp(BAR(BAR_KV_FULL), 0, wc);
      uint32_t w[32];
      if (wg == 0 || d.v_rows) {
        // K, or V given as rows: row r of the tile, eight 16-byte chunks
        const uint8_t* tile = sgen + (wg == 0 ? kSmemK : kSmemV);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_offset(r, ch));
          w[4 * ch] = v.x, w[4 * ch + 1] = v.y, w[4 * ch + 2] = v.z, w[4 * ch + 3] = v.w;
        }
      } else {
        // V^T tile: row = d, 64 keys per 128-byte row, keys 64-127 in the second half
        const uint8_t* vt = sgen + kSmemV + (r >> 6) * 8192;
        const int kc = (r & 63) >> 3, kb = (r & 7) * 2;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const uint32_t lo =
              *reinterpret_cast<const uint16_t*>(vt + sw128_offset(2 * u, kc) + kb);
          const uint32_t hi =
              *reinterpret_cast<const uint16_t*>(vt + sw128_offset(2 * u + 1, kc) + kb);
          w[u] = lo | (hi << 16);
        }
      }
      tmem_st32(tmem + lane_base + (wg == 0 ? kColK : kColV), w);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(BAR_KV_TMEM));
    }
    int rem_c = 0;
    for (int n = 0; ok && n < n_steps; ++n) {
      const int s = n % kStages;
      const int pb = n & 1;
      const int rem = rem_c;
      if (++rem_c == per_g) rem_c = 0;
      const int it = i_lo + (rem >> 1);
      const int hq = rem & 1;
      const int qb = it * kTile + hq * kBQ + 32 * wg;  // this thread's first query
      if (!mbar_wait_warp(BAR(BAR_S_FULL), n & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this thread's S^T and dP^T columns into registers, then the buffer
      // is free for the next step's products
      uint32_t sv[32], dv[32];
      tmem_ld32x2_wait(tmem + lane_base + kColS + 32 * wg, tmem + lane_base + kColDP + 32 * wg,
                       sv, dv);
      tc_fence_before();
      mbar_arrive(BAR(BAR_LOADED));

      const uint8_t* stg = sgen + kSmemStage0 + s * kStageBytes;
      const float4* L4 = reinterpret_cast<const float4*>(stg + kStL) + 8 * wg;
      const float4* D4 = reinterpret_cast<const float4*>(stg + kStD) + 8 * wg;
      const bool need_mask =
          (d.causal && qb < k0 + kBK - 1) || (qb + 32 > len) || (k0 + kBK > len);
      const int qlo = (d.causal ? key : 0) - qb;
      const int qhi = (key < len ? len : 0) - qb;
      uint32_t pp[16], dd[16];
      if (need_mask)
        step_math<true>(sv, dv, L4, D4, c, qlo, qhi, pp, dd);
      else
        step_math<false>(sv, dv, L4, D4, c, qlo, qhi, pp, dd);
      // pair buffer pb was last read by dV and dK of step n-2; with the
      // store, shared dS^T buffer n % 3 was last filled at step n-3 and its
      // bulk store must have read it.  Both are almost always free: one vote
      // covers both checks, and the bounded waits run only when one is not.
      const int dsbuf = n % kDSBufs;
      if (!STORE) {
        if (n >= 2 && !mbar_wait_warp(BAR(BAR_PK_FREE + pb), ((n >> 1) - 1) & 1, wc)) {
          ok = false;
          break;
        }
      } else {
        const bool f1 = n < 2 || mbar_try_wait(BAR(BAR_PK_FREE + pb), ((n >> 1) - 1) & 1);
        const bool f2 =
            n < kDSBufs || mbar_try_wait(BAR(BAR_DS_STORED + dsbuf), ((n / kDSBufs) - 1) & 1);
        if (!__all_sync(0xffffffffu, f1 && f2)) {
          if (n >= 2 && !mbar_wait_warp(BAR(BAR_PK_FREE + pb), ((n >> 1) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          if (n >= kDSBufs &&
              !mbar_wait_warp(BAR(BAR_DS_STORED + dsbuf), ((n / kDSBufs) - 1) & 1, wc)) {
            ok = false;
            break;
          }
        }
      }
      tc_fence_after();
      const uint32_t pk = kColPK + 64 * pb + 16 * wg;
      tmem_st16(tmem + lane_base + pk, pp);
      tmem_st16(tmem + lane_base + pk + 32, dd);

      if (STORE) {
        // dS^T row r, queries 32wg..32wg+31 of this 64-query half: chunks 4wg..4wg+3
        const uint32_t dsb = sbase + kSmemDS0 + dsbuf * kDSHalf;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(dsb + sw128_offset(r, 4 * wg + u), dd[4 * u], dd[4 * u + 1],
                       dd[4 * u + 2], dd[4 * u + 3]);
        fence_proxy_async_shared();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(BAR_P_READY + pb));
    }



    // ---------------- epilogue: dK = s * sum (rows), dV^T (columns) ----------------
    const bool store = key < T;
    uint32_t r0[32], r1[32];
    // ok is warp-uniform (every wait above is taken by the whole warp); the
    // epilogue wait is too, so the warp-aligned load runs converged, and it
    // is skipped once any wait gave up
    if (n_steps > 0 && ok && mbar_wait_warp(BAR(BAR_DONE), 0, wc)) {
      tc_fence_after();
      const uint32_t col = wg == 0 ? kColDK : kColDV;
      tmem_ld32x2_wait(tmem + lane_base + col, tmem + lane_base + col + 32, r0, r1);
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) r0[u] = r1[u] = 0u;
    }
    if (store && a.pk.on()) {
      // projection-fused epilogue: row `key` of dK (scaled) or dV, token-major
      const Projection& pr = wg == 0 ? a.pk : a.pv;
      store_projection_row(pr, ((size_t)b * T + key) * pr.ld + 64 * (size_t)kv, r0, r1, d.scale,
                           wg == 0);
    } else if (store && wg == 0) {
      float4* dst = reinterpret_cast<float4*>(a.dk + (((size_t)b * d.Hkv + kv) * T + key) * 64);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        dst[u] = make_float4(as_f(r0[4 * u]) * d.scale, as_f(r0[4 * u + 1]) * d.scale,
                             as_f(r0[4 * u + 2]) * d.scale, as_f(r0[4 * u + 3]) * d.scale);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        dst[8 + u] = make_float4(as_f(r1[4 * u]) * d.scale, as_f(r1[4 * u + 1]) * d.scale,
                                 as_f(r1[4 * u + 2]) * d.scale, as_f(r1[4 * u + 3]) * d.scale);
    } else if (store) {
      float* dvcol = a.dvt + ((size_t)b * d.Hkv + kv) * 64 * (size_t)T + key;
#pragma unroll
      for (int u = 0; u < 32; ++u) dvcol[(size_t)u * T] = as_f(r0[u]);
#pragma unroll
      for (int u = 0; u < 32; ++u) dvcol[(size_t)(32 + u) * T] = as_f(r1[u]);
    }
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    if (n_steps > 0) drain_wait(BAR(BAR_DONE), 0);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef BAR
}

}  // namespace

int launch_bwd_keys(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
                    const uint16_t* vt, const uint16_t* dout, const float* lse,
                    const float* delta, uint8_t* ws, float* dk, float* dvt,
                    cudaStream_t stream, Projection pk, Projection pv) {
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t T = (uint64_t)d.T;
  if (!encode_tmap_3d(&tq, q, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBQ) ||
      !encode_tmap_3d(&tdo, dout, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBQ) ||
      !encode_tmap_3d(&tk, k, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, kBK) ||
      !(d.v_rows ? encode_tmap_3d(&tv, vt, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, 128)
                  : encode_tmap_3d(&tv, vt, T, 64, (uint64_t)d.B * d.Hkv, T * 2, T * 128, 64, 64)))
    return ATTN_ERR_CUDA;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_status[64];
  std::call_once(attr_once[dev & 63], [dev] {
    attr_status[dev & 63] = cudaFuncSetAttribute(
        bwd_keys_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (attr_status[dev & 63] == cudaSuccess)
      attr_status[dev & 63] = cudaFuncSetAttribute(
          bwd_keys_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_status[dev & 63] != cudaSuccess) return cuda_status(attr_status[dev & 63]);
  KeysArgs args{d, lse, delta, ws, dk, dvt, ctx.err, ctx.wait_ns, pk, pv};
  dim3 grid(d.kv_count, d.nt, d.B);
  return cuda_status(
      ws != nullptr ? launch_dependent(bwd_keys_kernel<true>, grid, dim3(kThreads), kSmemBytes,
                                       stream, tq, tk, tv, tdo, args)
                    : launch_dependent(bwd_keys_kernel<false>, grid, dim3(kThreads), kSmemBytes,
                                       stream, tq, tk, tv, tdo, args));
}

}  // namespace css
