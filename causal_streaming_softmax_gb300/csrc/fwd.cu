// fwd.cu - forward pass: causal (or length-masked) attention as a streaming
// normalised sum, two 128-query tiles of one query head per CTA.
//
// Method (StreamingAttentionSM86.alpha, forward module header and the
// "one key tile" / epilogue sections): for every key tile up to the
// diagonal, S = Q K^T; t = S c in base 2; m' = max(m, rowmax t);
// alpha = 2^(m - m'); P = 2^(t - m'); l = alpha l + sum P (binary32, P
// unrounded); O = alpha O + f16(P) V.  Output O / l (binary16, token-major)
// and L = m + log2 l (binary32).
//
// GB300 design (not the pages' SM86 register kernel).  A work unit is 256
// queries of one head as two 128-row tiles, A and B, that share every K/V
// tile and ping-pong on the exponential unit.  The units are listed longest
// causal rows first; a CTA walks a share of them in snake order (CTA c of G
// takes units c, 2G-1-c, 2G+c, ...), with tensor memory, barriers and the
// K/V ring carried over from one unit to the next, and the next unit's Q and
// first K/V tiles loading while the current unit finishes.  The launch picks
// G: one CTA per SM (persistent) when there are few units per SM and no
// per-sequence lengths, else one CTA per unit.
//   warps 0-3   softmax of tile A, one thread per query row (= TMEM lane)
//   warps 4-7   softmax of tile B
//   warp 8      TMA producer: each unit's Q (two buffers), then its K and
//               V^T (or V rows) tiles through a 3-stage ring
//   warps 9-11  MMA issuers: S_A = Q_A K^T and S_B = Q_B K^T (warp 9),
//               O_A += P_A V (warp 10), O_B += P_B V (warp 11): independent
//               chains get their own warps, so one chain waiting on its
//               barrier never holds back another's issue.
// Tensor memory (512 columns): S_A 0-127, S_B 128-255 (binary32), P_A
// 256-319, P_B 320-383 (binary16 pairs), O_A 384-447, O_B 448-511.  Since P
// has its own columns, S of the next key tile is computed as soon as the
// softmax has read S, while O += P V of this tile runs.
#include <math.h>

#include <mutex>

#include "attn_internal.h"
#include "sm103.cuh"

namespace css {
namespace {

constexpr int kBM = 128;   // rows per query tile
constexpr int kBN = 128;   // keys per key tile
constexpr int kStages = 3;
constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = 128 * 128;         // 128 rows x 128 B
constexpr uint32_t kStageBytes = 2 * kTileBytes;   // K tile, then V^T as two 64-key halves
constexpr uint32_t kSmemQ = 0;                     // [buffer] Q_A, then Q_B
constexpr uint32_t kSmemStage0 = 4 * kTileBytes;
constexpr uint32_t kSmemBar = kSmemStage0 + kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kSmemBar + 256 + 1024;  // barriers + 1024-B alignment slack

constexpr uint32_t kColS = 0;    // + 128 * tile
constexpr uint32_t kColP = 256;  // + 64 * tile
constexpr uint32_t kColO = 384;  // + 64 * tile
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_f16_f32(128, 128, 0, 0);  // Q (K-major) x K (K-major)
constexpr uint32_t kIdescO = idesc_f16_f32(128, 64, 0, 0);   // P (tmem) x V^T (K-major)
constexpr uint32_t kIdescOR = idesc_f16_f32(128, 64, 0, 1);  // P (tmem) x V rows (MN-major)

enum {
  BAR_Q = 0,                             // [Q buffer] the unit's Q tiles landed
  BAR_Q_FREE = BAR_Q + 2,                // [Q buffer] every S = Q K^T of its unit done
  BAR_KV_FULL = BAR_Q_FREE + 2,
  BAR_KV_EMPTY = BAR_KV_FULL + kStages,  // [stage] both O += P V of the key tile done (2 commits)
  BAR_S_FULL = BAR_KV_EMPTY + kStages,   // [tile] S of the tile computed
  BAR_S_FREE = BAR_S_FULL + 2,           // [tile] softmax has read S (128 threads)
  BAR_P_FULL = BAR_S_FREE + 2,           // [tile] P written and O rescaled (128 threads)
  BAR_P_FREE = BAR_P_FULL + 2,           // [tile] O += P V done (P may be overwritten)
  BAR_O_DONE = BAR_P_FREE + 2,           // [tile] every O += P V of the tile's unit done
  BAR_O_FREE = BAR_O_DONE + 2,           // [tile] the epilogue has read O (128 threads)
  BAR_MMA_DONE = BAR_O_FREE + 2,         // every MMA of the CTA done (3 issuer commits)
  BAR_COUNT
};
static_assert(BAR_COUNT * 8 <= 256, "barrier area");

struct FwdArgs {
  int T, H, Hkv, G, causal, v_rows;
  int B, nqb, units;  // batch, 256-query blocks per head, work units (H * nqb * B)
  const int32_t* lens;
  float c;
  uint16_t* o;
  float* lse;
  uint32_t* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// Number of 128-key tiles that query rows [q0, q0 + 128) see.
__device__ __forceinline__ int key_tiles(int q0, int len, int causal) {
  if (q0 >= len) return 0;
  const int kend = causal ? min(len, q0 + kBM) : len;
  return (kend + kBN - 1) / kBN;
}

// The row's maximum raw score over one 128-key tile in tensor memory.  MASK
// sets the columns at or past `lim` (local key index) to -inf first.  The
// raw bits of columns 96-127 are kept in `keep` for the exponential pass, so
// that pass reads tensor memory three times instead of four and releases S
// a quarter of its work earlier.
template <bool MASK>
__device__ __forceinline__ float tile_row_max(uint32_t t_s, int lim, uint32_t (&keep)[32]) {
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t v0[32], v1[32];
    tmem_ld32x2_wait(t_s + half * 64, t_s + half * 64 + 32, v0, v1);
    if (half == 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) keep[i] = v1[i];
    }
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0 = as_f(v0[e]), x1 = as_f(v0[e + 1]), y0 = as_f(v1[e]), y1 = as_f(v1[e + 1]);
      if (MASK) {
        const int cb = half * 64 + e;
        if (cb >= lim) x0 = -INFINITY;
        if (cb + 1 >= lim) x1 = -INFINITY;
        if (cb + 32 >= lim) y0 = -INFINITY;
        if (cb + 33 >= lim) y1 = -INFINITY;
      }
      if (e & 2) {
        m0 = fmax3(m0, x0, x1);
        m1 = fmax3(m1, y0, y1);
      } else {
        m2 = fmax3(m2, x0, x1);
        m3 = fmax3(m3, y0, y1);
      }
    }
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// P = 2^(S c - m') for one 128-key tile as binary16 pairs in registers (the
// lower key in the low half); returns the row sum of the unrounded binary32 P.
// Columns 96-127 come from `keep`; after its last read of S (columns 64-95)
// it arrives on `s_free`.
template <bool MASK>
__device__ __forceinline__ float tile_exp(uint32_t t_s, float c, float neg_m, int lim,
                                          uint32_t s_free, uint32_t (&pk)[64],
                                          const uint32_t (&keep)[32]) {
  const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
  float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
  for (int qtr = 0; qtr < 4; ++qtr) {
    uint32_t v[32];
    if (qtr < 3) {
      tmem_ld32_wait(t_s + qtr * 32, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = keep[(qtr - 3) * 32 + i];
    }
    if (qtr == 2) {
      tc_fence_before();
      mbar_arrive(s_free);
    }
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float2 x = make_float2(as_f(v[e]), as_f(v[e + 1]));
      if (MASK) {
        const int cb = qtr * 32 + e;
        if (cb >= lim) x.x = -INFINITY;
        if (cb + 1 >= lim) x.y = -INFINITY;
      }
      const float2 tx = __ffma2_rn(x, c2, nm2);
      const float2 ex = make_float2(ex2_approx(tx.x), ex2_approx(tx.y));
      if (e & 2)
        a0 = __fadd2_rn(a0, ex);
      else
        a1 = __fadd2_rn(a1, ex);
      // key k of the tile goes to packed word k / 2
      pk[qtr * 16 + (e >> 1)] = pack_f16x2(ex.x, ex.y);
    }
  }
  const float2 s01 = __fadd2_rn(a0, a1);
  return s01.x + s01.y;
}

// Stores the 64 packed words of P (128 keys) into the row's P columns.
__device__ __forceinline__ void store_p(uint32_t t_p, const uint32_t (&pk)[64]) {
  const uint32_t(&w0)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]);
  const uint32_t(&w1)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]);
  tmem_st32(t_p, w0);
  tmem_st32(t_p + 32, w1);
}

// One work unit: 256 queries (query tiles A and B) of one head of one batch
// entry, and the number of key tiles each tile sees.
struct Unit {
  int h, b, kv, len, q0, n_a, n_b, n_kt;
};

// Units are listed head fastest, then the 256-query blocks from the last
// (longest causal rows) to the first, then batch entries.
__device__ __forceinline__ Unit unit_at(const FwdArgs& a, int u) {
  Unit w;
  w.h = u % a.H;
  const int r = u / a.H;
  const int qb = a.nqb - 1 - r % a.nqb;
  w.b = r / a.nqb;
  w.kv = w.h / a.G;
  w.len = a.T;
  if (a.lens) {
    const int l = a.lens[w.b];
    w.len = l < 0 ? 0 : (l > a.T ? a.T : l);
  }
  w.q0 = qb * 2 * kBM;
  w.n_a = key_tiles(w.q0, w.len, a.causal);
  w.n_b = key_tiles(w.q0 + kBM, w.len, a.causal);
  w.n_kt = max(w.n_a, w.n_b);
  return w;
}

// The i-th unit of this CTA (snake order over the list), or -1 past the end.
__device__ __forceinline__ int unit_index(const FwdArgs& a, int i) {
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const long long u = (long long)i * G + ((i & 1) ? (G - 1 - c) : c);
  return u < a.units ? (int)u : -1;
}

// 12 warps: three per scheduler, so up to 168 registers per thread.
// VROWS: V given as rows [B][Hkv][T][64] (else V^T), fixed at compile time
// so that each layout's kernel carries only its own addressing.
template <bool VROWS>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_vt, const FwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  griddep_launch_dependents();

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar0 = sbase + kSmemBar;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.T;

  WaitCtl wc{a.err, a.wait_ns, &s_abort};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int q = 0; q < 2; ++q) {
      mbar_init(BAR(BAR_Q + q), 1);
      mbar_init(BAR(BAR_Q_FREE + q), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(BAR_KV_FULL + s), 1);
      mbar_init(BAR(BAR_KV_EMPTY + s), 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(BAR_S_FULL + t), 1);
      mbar_init(BAR(BAR_S_FREE + t), 128);
      mbar_init(BAR(BAR_P_FULL + t), 128);
      mbar_init(BAR(BAR_P_FREE + t), 1);
      mbar_init(BAR(BAR_O_DONE + t), 1);
      mbar_init(BAR(BAR_O_FREE + t), 128);
    }
    mbar_init(BAR(BAR_MMA_DONE), 3);
    fence_mbarrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  griddep_wait();

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      int kt = 0, nq = 0;  // key tiles loaded so far, units with work so far
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int u = unit_index(a, i);
        if (u < 0) break;
        const Unit w = unit_at(a, u);
        if (w.n_kt == 0) continue;
        const int qplane = w.b * a.H + w.h;
        const int kvplane = w.b * a.Hkv + w.kv;
        const int qbuf = nq & 1;
        // this Q buffer was last read by the S products of unit nq - 2
        if (nq >= 2 && !mbar_wait(BAR(BAR_Q_FREE + qbuf), ((nq >> 1) - 1) & 1, wc)) break;
        // a tile with no visible key is never computed, so its Q is not loaded
        const uint32_t q_s = sbase + kSmemQ + qbuf * 2 * kTileBytes;
        mbar_arrive_expect_tx(BAR(BAR_Q + qbuf), ((w.n_a > 0) + (w.n_b > 0)) * kTileBytes);
        if (w.n_a > 0) tma_load_3d(q_s, &tm_q, BAR(BAR_Q + qbuf), 0, w.q0, qplane);
        if (w.n_b > 0) tma_load_3d(q_s + kTileBytes, &tm_q, BAR(BAR_Q + qbuf), 0, w.q0 + kBM, qplane);
        ++nq;
        for (int j = 0; j < w.n_kt; ++j, ++kt) {
          const int s = kt % kStages;
          if (kt >= kStages && !mbar_wait(BAR(BAR_KV_EMPTY + s), ((kt / kStages) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + kSmemStage0 + s * kStageBytes;
          mbar_arrive_expect_tx(BAR(BAR_KV_FULL + s), kStageBytes);
          tma_load_3d(st, &tm_k, BAR(BAR_KV_FULL + s), 0, j * kBN, kvplane);
          if (VROWS) {
            tma_load_3d(st + kTileBytes, &tm_vt, BAR(BAR_KV_FULL + s), 0, j * kBN, kvplane);
          } else {
            tma_load_3d(st + kTileBytes, &tm_vt, BAR(BAR_KV_FULL + s), j * kBN, 0, kvplane);
            tma_load_3d(st + kTileBytes + 8192, &tm_vt, BAR(BAR_KV_FULL + s), j * kBN + 64, 0,
                        kvplane);
          }
        }
      }
      // no copy may still be landing when the CTA exits (matters only when a
      // wait gave up): wait for the last fill of each Q buffer and stage
      for (int q = 0; q < 2 && q < nq; ++q) {
        const int uses = (nq - q + 1) / 2;  // fills of buffer q
        drain_wait(BAR(BAR_Q + q), (uses - 1) & 1);
      }
      for (int k = (kt > kStages ? kt - kStages : 0); k < kt; ++k)
        drain_wait(BAR(BAR_KV_FULL + k % kStages), (k / kStages) & 1);
    }
  } else if (warp >= 9) {
    // ---------------- MMA issuers: one thread per product chain ----------------
    if (lane == 0) {
      bool ok = true;
      if (warp == 9) {
        // S_A and S_B for each key tile, in that order
        int kt = 0, nq = 0, ns[2] = {0, 0};
        for (int i = 0; ok; ++i) {
          const int u = unit_index(a, i);
          if (u < 0) break;
          const Unit w = unit_at(a, u);
          if (w.n_kt == 0) continue;
          const int qbuf = nq & 1;
          if (!mbar_wait(BAR(BAR_Q + qbuf), (nq >> 1) & 1, wc)) break;
          const uint32_t q_base = sbase + kSmemQ + qbuf * 2 * kTileBytes;
          for (int j = 0; ok && j < w.n_kt; ++j, ++kt) {
            const int s = kt % kStages;
            if (!mbar_wait(BAR(BAR_KV_FULL + s), (kt / kStages) & 1, wc)) {
              ok = false;
              break;
            }
            const uint32_t k_s = sbase + kSmemStage0 + s * kStageBytes;
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
              if (j >= (t ? w.n_b : w.n_a)) continue;
              // the softmax has read this tile's previous S
              if (ns[t] > 0 && !mbar_wait(BAR(BAR_S_FREE + t), (ns[t] - 1) & 1, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t q_s = q_base + t * kTileBytes;
              // S = Q K^T over d = 64: four K=16 steps inside the 128-byte atom
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(tmem + kColS + 128 * t, sdesc_sw128(q_s + kk * 32, 16, 1024),
                       sdesc_sw128(k_s + kk * 32, 16, 1024), kIdescS, kk > 0);
              mma_commit(BAR(BAR_S_FULL + t));
              ++ns[t];
            }
          }
          if (!ok) break;
          mma_commit(BAR(BAR_Q_FREE + qbuf));  // the unit's Q buffer may be refilled
          ++nq;
        }
      } else {
        const int t = warp - 10;
        int kt = 0, npv = 0, no = 0;
        for (int i = 0; ok; ++i) {
          const int u = unit_index(a, i);
          if (u < 0) break;
          const Unit w = unit_at(a, u);
          if (w.n_kt == 0) continue;
          const int n_t = t ? w.n_b : w.n_a;
          // walks every loaded key tile so that each stage gets both commits;
          // for a key tile this query tile does not see, the commit waits
          // until the tile has been loaded, so that it counts toward that
          // tile's use of the stage and not toward an earlier one
          for (int j = 0; j < w.n_kt; ++j, ++kt) {
            const int s = kt % kStages;
            if (j >= n_t) {
              if (!mbar_wait(BAR(BAR_KV_FULL + s), (kt / kStages) & 1, wc)) {
                ok = false;
                break;
              }
            } else {
              if (!mbar_wait(BAR(BAR_P_FULL + t), npv & 1, wc)) {
                ok = false;
                break;
              }
              // the unit's first product overwrites O: the previous unit's
              // epilogue must have read it
              if (j == 0 && no > 0 && !mbar_wait(BAR(BAR_O_FREE + t), (no - 1) & 1, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t v_s = sbase + kSmemStage0 + s * kStageBytes + kTileBytes;
              // O += P V over the tile's 128 keys: eight K=16 steps; keys 0-63
              // in the first V^T half, 64-127 in the second
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts(tmem + kColO + 64 * t, tmem + kColP + 64 * t + kk * 8,
                       VROWS ? sdesc_sw128(v_s + kk * 2048, 8192, 1024)
                                : sdesc_sw128(v_s + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                       VROWS ? kIdescOR : kIdescO,
                       (j > 0 || kk > 0) ? 1u : 0u);
              mma_commit(BAR(BAR_P_FREE + t));
              ++npv;
            }
            mma_commit(BAR(BAR_KV_EMPTY + s));
          }
          if (!ok) break;
          if (n_t > 0) {
            mma_commit(BAR(BAR_O_DONE + t));
            ++no;
          }
        }
      }
      // every MMA this thread issued is done once this arrives
      mma_commit(BAR(BAR_MMA_DONE));
    }
  } else {
    // ---------------- softmax: thread = query row of tile t ----------------
    const int t = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + kColS + 128 * t;
    const uint32_t t_p = tmem + lane_base + kColP + 64 * t;
    const uint32_t t_o = tmem + lane_base + kColO + 64 * t;
    const float c = a.c;
    int ns = 0, npv = 0, no = 0;  // S tiles read, P tiles written, units finished
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int u = unit_index(a, i);
      if (u < 0) break;
      int qt0, n_t, len;
      {
        const Unit w = unit_at(a, u);
        qt0 = w.q0 + t * kBM;
        n_t = t ? w.n_b : w.n_a;
        len = w.len;
      }
      const int qrow = qt0 + row;
      const bool row_ok = qrow < len;
      // keys below `lim` are valid for this row
      int lim = row_ok ? len : 0;
      if (a.causal) lim = min(lim, qrow + 1);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n_t; ++j) {
        if (!mbar_wait_warp(BAR(BAR_S_FULL + t), ns & 1, wc)) {
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        const int k0 = j * kBN;
        const bool need_mask =
            (a.causal && k0 + kBN - 1 > qt0) || (k0 + kBN > len) || (qt0 + kBM > len);
        const int lim_local = lim - k0;

        // pass 1: the row's maximum raw score over the tile
        uint32_t keep[32];
        const float mx = need_mask ? tile_row_max<true>(t_s, lim_local, keep)
                                   : tile_row_max<false>(t_s, lim_local, keep);
        // c > 0, so max(S) c is the maximum of the scaled scores.
        const float m_new = fmaxf(m, mx * c);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_use);
        // pass 2: P = 2^(S c - m') and its row sum, P kept in registers
        uint32_t pk[64];
        const float sum = need_mask ? tile_exp<true>(t_s, c, -m_use, lim_local,
                                                     BAR(BAR_S_FREE + t), pk, keep)
                                    : tile_exp<false>(t_s, c, -m_use, lim_local,
                                                      BAR(BAR_S_FREE + t), pk, keep);
        // P of the previous key tile has been read by its O += P V (and O is
        // final for the rescale below): only now is P overwritten
        if (npv > 0 && !mbar_wait_warp(BAR(BAR_P_FREE + t), (npv - 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        store_p(t_p, pk);
        l = l * alpha + sum;
        m = m_new;

        // O *= alpha.  Skipped for a warp whose rows all keep their maximum,
        // which leaves O unchanged exactly.
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t o0[32], o1[32];
          tmem_ld32x2_wait(t_o, t_o + 32, o0, o1);
          const float2 al = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 x = __fmul2_rn(make_float2(as_f(o0[e]), as_f(o0[e + 1])), al);
            const float2 y = __fmul2_rn(make_float2(as_f(o1[e]), as_f(o1[e + 1])), al);
            o0[e] = __float_as_uint(x.x), o0[e + 1] = __float_as_uint(x.y);
            o1[e] = __float_as_uint(y.x), o1[e + 1] = __float_as_uint(y.y);
          }
          tmem_st32(t_o, o0);
          tmem_st32(t_o + 32, o1);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(BAR_P_FULL + t));
        ++npv;
      }
      if (!ok) break;

      // ---------------- epilogue: O / l, L = m + log2 l ----------------
      const int uh = u % a.H, ub = (u / a.H) / a.nqb;
      uint16_t* orow = a.o + ((size_t)((size_t)ub * T + qrow) * a.H + uh) * 64;
      float* lrow = a.lse + ((size_t)ub * a.H + uh) * T + qrow;
      if (n_t > 0) {
        if (!mbar_wait_warp(BAR(BAR_O_DONE + t), no & 1, wc)) {
          ok = false;
          break;
        }
        ++no;
        tc_fence_after();
        uint32_t o0[32], o1[32];
        tmem_ld32x2_wait(t_o, t_o + 32, o0, o1);
        // O is in registers: the next unit's first product may overwrite it
        tc_fence_before();
        mbar_arrive(BAR(BAR_O_FREE + t));
        const bool valid = row_ok && l > 0.f;
        const float inv = valid ? 1.0f / l : 0.f;
        if (qrow < T) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_f16x2(as_f(o0[8 * q + 0]) * inv, as_f(o0[8 * q + 1]) * inv),
                                pack_f16x2(as_f(o0[8 * q + 2]) * inv, as_f(o0[8 * q + 3]) * inv),
                                pack_f16x2(as_f(o0[8 * q + 4]) * inv, as_f(o0[8 * q + 5]) * inv),
                                pack_f16x2(as_f(o0[8 * q + 6]) * inv, as_f(o0[8 * q + 7]) * inv));
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[4 + q] =
                make_uint4(pack_f16x2(as_f(o1[8 * q + 0]) * inv, as_f(o1[8 * q + 1]) * inv),
                           pack_f16x2(as_f(o1[8 * q + 2]) * inv, as_f(o1[8 * q + 3]) * inv),
                           pack_f16x2(as_f(o1[8 * q + 4]) * inv, as_f(o1[8 * q + 5]) * inv),
                           pack_f16x2(as_f(o1[8 * q + 6]) * inv, as_f(o1[8 * q + 7]) * inv));
          *lrow = valid ? m + lg2_approx(l) : -INFINITY;
        }
      } else if (qrow < T) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        *lrow = -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    // every MMA of this CTA has completed before its tensor memory is freed
    drain_wait(BAR(BAR_MMA_DONE), 0);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef BAR
}

}  // namespace

int launch_fwd(const Dims& d, const DevCtx& ctx, const uint16_t* q, const uint16_t* k,
               const uint16_t* vt, uint16_t* o, float* lse, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  const uint64_t T = (uint64_t)d.T;
  // Q [B*H][T][64], K [B*Hkv][T][64]: boxes of 128 rows x 64 values.
  if (!encode_tmap_3d(&tq, q, 64, T, (uint64_t)d.B * d.H, 128, T * 128, 64, kBM) ||
      !encode_tmap_3d(&tk, k, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, kBN) ||
      // V^T [B*Hkv][64][T]: boxes of 64 keys x 64 rows; V rows: 128 keys x 64
      !(d.v_rows ? encode_tmap_3d(&tv, vt, 64, T, (uint64_t)d.B * d.Hkv, 128, T * 128, 64, 128)
                  : encode_tmap_3d(&tv, vt, T, 64, (uint64_t)d.B * d.Hkv, T * 2, T * 128, 64, 64)))
    return ATTN_ERR_CUDA;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_status[64];
  std::call_once(attr_once[dev & 63], [dev] {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    attr_status[dev & 63] = e;
  });
  if (attr_status[dev & 63] != cudaSuccess) return cuda_status(attr_status[dev & 63]);
  const int nqb = (d.T + 2 * kBM - 1) / (2 * kBM);
  const long long units = (long long)d.H * nqb * d.B;
  if (units > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  FwdArgs args{d.T, d.H, d.Hkv, d.G, d.causal, d.v_rows, d.B, nqb, (int)units, d.lens, d.c, o,
               lse, ctx.err, ctx.wait_ns};
  // Persistent (one CTA per SM walking its share of the units) when there are
  // few units per SM and no per-sequence lengths: the per-unit start-up and
  // tail then overlap the neighbouring units, and the snake order balances
  // the known causal work.  Otherwise one CTA per unit, which the hardware
  // schedules as SMs free up (better for many units or unknown lengths).
  // Measured on GB300: T = 4096, 32 heads (512 units) 92.8 -> 88.8 us
  // persistent; T = 16384 (1024 units) and the 16-sequence length-masked
  // batch (2048 units) were 2% and 9% faster with one CTA per unit.
  const bool persistent = d.lens == nullptr && units <= 4LL * ctx.sm_count;
  dim3 grid((unsigned)(persistent && units > ctx.sm_count ? ctx.sm_count : units));
  cudaError_t e;
  if (d.v_rows)
    e = launch_dependent(fwd_kernel<true>, grid, dim3(kThreads), kSmemBytes, stream, tq, tk, tv,
                         args);
  else
    e = launch_dependent(fwd_kernel<false>, grid, dim3(kThreads), kSmemBytes, stream, tq, tk, tv,
                         args);
  return cuda_status(e);
}

}  // namespace css
