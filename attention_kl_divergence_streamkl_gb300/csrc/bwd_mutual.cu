// Attention-KL backward for the mutual case: both distributions train, so the
// loss L = sum_i g_i KL_i sends gradients to Q1, K1 (setting 2, P2 held fixed)
// and to Q2, K2 (setting 1, P1 held fixed) at once.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "recompute strategy" and its two settings.  Neither setting's gradient
// depends on the other side's parameters, so the mutual gradient is the pair
// of single-setting gradients; what the two settings share is the recompute:
// both need S1 and S2 of every tile pair.  These blocks read the two logit
// tiles once and produce both dS tiles from them (make_ds_row_mutual), where
// running the settings one after the other computes every logit tile twice.
//
// Two kinds of block, like the separate single-setting path's two kernels (no
// atomics), run as one launch (bwd_mutual_kernel):
//
// dQ blocks: a block owns 128 query rows (Q1, Q2 stationary) and streams key tiles:
//     S1 = Q1 K1^T, then S2 = Q2 K2^T     both into TMEM columns [0, 128)
//     dS1, dS2 packed to bf16 into TMEM   [128, 192), [192, 256)
//     dQ1 += dS1 K1, dQ2 += dS2 K2        A = dS in TMEM, B = K read MN-major -> [256, 256 + D), [384, 384 + D)
// The 512 TMEM columns hold no second logit region, so S1 and S2 take turns in
// one: the dS warps copy S1 into registers and release it, S2 is written over
// it.  The key tiles (K1(j), K2(j), each held from its logits MMA to its dQ MMA)
// go through one 5-slot ring in the order K1(0), K2(0), K1(1), ...
//   warps 0-15  dS warps: thread = query row (lane quarter = warp % 4), group g = warp / 4
//               takes key columns [32g, 32g + 32); at the end they write dQ1 and dQ2
//   warp 16     TMA producer        warp 17  TMEM owner, issuer of the logits MMAs
//   warp 18     issuer of the gradient MMAs: dQ1(j) at once, dQ2(j) once S2(j + 1) is queued
//
// dK blocks: a block owns 128 keys (K1, K2 stationary) and streams query tiles as
// the M operand of the logits MMA, so a dS thread owns a query row:
//     S1 = Q1 K1^T -> [0, 128), S2 = Q2 K2^T -> [128, 256)
//     dS1, then dS2, to one shared-memory buffer as dS[query][key]
//     dK1 += dS1^T Q1, dK2 += dS2^T Q2    A = dS read MN-major (M = keys), B = Q read MN-major
//                                         -> [256, 256 + D), [384, 384 + D)
// Shared memory holds K1, K2, one dS buffer and a 4-slot ring of query tiles
// (Q1(j), Q2(j), ...): the two query tiles of the tile being reduced and the
// two of the next.  The dS warps store dS1, copy S1 of the next tile while dK1's
// MMA runs, then store dS2.
//   warps 0-15  dS warps (then: thread = key row, group g = d columns [32g, 32g + 32) of dK1, dK2)
//   warp 16     TMA producer        warp 17  TMEM owner and MMA issuer
#include "common.cuh"
#include "ds_math.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int DS_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int GRAD_WARP = 18;  // dQ blocks: issuer of the gradient MMAs
constexpr int THREADS = 20 * 32;
constexpr int kRegsDs = 104, kRegsOther = 64;  // 512 * 104 + 128 * 64 = 640 * 96 registers at launch
constexpr uint32_t kTmemCols = 512;
constexpr int kOneBlockPerSmSmem = 120 * 1024;  // a block owns all 512 TMEM columns

__device__ __forceinline__ void setmaxnreg_inc_ds() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
}
__device__ __forceinline__ void setmaxnreg_dec_other() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

// Row of 8 scaled fp32 accumulator values per uint4: bf16(scale * v).
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&v)[32], float scale) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t* src = &v[q * 8];
    uint4 o;
    o.x = pack_bf16(__uint_as_float(src[0]) * scale, __uint_as_float(src[1]) * scale);
    o.y = pack_bf16(__uint_as_float(src[2]) * scale, __uint_as_float(src[3]) * scale);
    o.z = pack_bf16(__uint_as_float(src[4]) * scale, __uint_as_float(src[5]) * scale);
    o.w = pack_bf16(__uint_as_float(src[6]) * scale, __uint_as_float(src[7]) * scale);
    reinterpret_cast<uint4*>(dst)[q] = o;
  }
}

// The row's folded values (ds_math.cuh): nA, setting 1's nB, setting 2's nB, g.
struct RowVals {
  float nA, nB2, nB1, G;
};
__device__ __forceinline__ RowVals row_vals(const float* lse1, const float* lse2, const float* klv, const float* gv,
                                            size_t o) {
  const float l1v = lse1[o], l2v = lse2[o];
  return RowVals{-l1v * kLog2e, -l2v * kLog2e, -(l1v - l2v + klv[o]), gv[o]};
}

// ============================================================================ dQ blocks
namespace mdq {
constexpr int BX = 128, BY = 128, SLOTS = 5;
constexpr uint32_t kColS = 0, kColDS1 = 128, kColDS2 = 192, kColG1 = 256, kColG2 = 384;

template <int D>
struct Smem {
  static constexpr int TILE = 128 * D * 2;  // one 128-row bf16 tile, D/64 halves of 16 KiB
  static constexpr int OFF_X1 = 0;
  static constexpr int OFF_X2 = TILE;
  static constexpr int OFF_Y = 2 * TILE;  // key-tile ring [SLOTS]
  static constexpr int OFF_BAR = OFF_Y + SLOTS * TILE;
  // x_full, y_full[5], y_empty[5], s_full, s_free, ds_full, ds_free, g_done, s2_issued; then the TMEM base
  // address slot and the abort flag
  static constexpr int BAR_SLOT = 8 * 17;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");
}  // namespace mdq

// Block `blk` of the dQ grid (head-major, the last query tiles first).
template <int D>
__device__ __forceinline__ void dq_mutual_block(const Problem& p, const float* __restrict__ lse1,
                                                const float* __restrict__ lse2, const float* __restrict__ klv,
                                                const float* __restrict__ gv, __nv_bfloat16* __restrict__ dq1,
                                                __nv_bfloat16* __restrict__ dq2, int* status, const CUtensorMap& mq1,
                                                const CUtensorMap& mq2, const CUtensorMap& mk1, const CUtensorMap& mk2,
                                                const unsigned blk) {
  using namespace mdq;
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_xt = (p.NQ + BX - 1) / BX;
  // heads in order, the last query tiles (the most keys when causal) first within a head
  const int bh = (int)(blk / n_xt);
  const int mh = bh % p.H, mb = bh / p.H;
  const int xt = n_xt - 1 - (int)(blk % n_xt);
  const int x0 = xt * BX;
  const int y_end = p.causal ? min(p.NK, min(p.NQ, x0 + BX) - 1 + p.off + 1) : p.NK;  // keys the last row sees
  const int n_yt = (y_end + BY - 1) / BY;
  const int n_items = 2 * n_yt;  // ring items: K1(j) = 2j, K2(j) = 2j + 1

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t x_full = bar, y_full = bar + 8, y_empty = bar + 48, s_full = bar + 88, s_free = bar + 96,
                 ds_full = bar + 104, ds_free = bar + 112, g_done = bar + 120, s2_issued = bar + 128,
                 slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);

  if (threadIdx.x == 0) {
    mbar_init(x_full, 1);
    mbar_init(s2_issued, 1);
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(y_full + 8 * s, 1);
      mbar_init(y_empty + 8 * s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, DS_WARPS);
    mbar_init(ds_full, DS_WARPS);
    mbar_init(ds_free, 1);
    mbar_init(g_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_BAR + L::BAR_SLOT);

  if (warp >= DS_WARPS) {
    setmaxnreg_dec_other();
    if (warp == PRODUCER_WARP) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        mbar_arrive_expect_tx(x_full, 2 * L::TILE);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(sb + L::OFF_X1 + h * BX * 128, &mq1, x_full, h * 64, x0, mh, mb);
          tma_load_4d(sb + L::OFF_X2 + h * BX * 128, &mq2, x_full, h * 64, x0, mh, mb);
        }
        int issued = 0;
        for (int i = 0; i < n_items; ++i) {
          const int s = i % SLOTS;
          if (i >= SLOTS && !mbar_wait(y_empty + 8 * s, ((i / SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(y_full + 8 * s, L::TILE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_Y + s * L::TILE + h * BY * 128, (i & 1) ? &mk2 : &mk1, y_full + 8 * s, h * 64,
                        (i >> 1) * BY, mh, mb);
          issued = i + 1;
        }
        // copies that may still be landing: the Q tiles and the last SLOTS ring items
        mbar_drain(x_full, 0, status);
        for (int i = max(0, issued - SLOTS); i < issued; ++i)
          mbar_drain(y_full + 8 * (i % SLOTS), (i / SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------------ MMA issuer: logits
      // S1(j) once the dS warps have copied S2(j - 1) out of the region, S2(j) once they hold S1(j);
      // s_free completes twice per key tile: S1(j) copied (2j), S2(j) copied (2j + 1)
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16(BX, BY, false, false);
        const uint64_t x1d = sdesc_sw128(sb + L::OFF_X1, 0, 1024), x2d = sdesc_sw128(sb + L::OFF_X2, 0, 1024);
        bool ok = mbar_wait(x_full, 0, status, abort_flag);
        for (int i = 0; ok && i < n_items; ++i) {
          const int t = i & 1, s = i % SLOTS;
          if (!mbar_wait(y_full + 8 * s, (i / SLOTS) & 1, status, abort_flag)) break;
          if (i >= 1 && !mbar_wait(s_free, (i - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          const uint64_t xd = t ? x2d : x1d;
          const uint64_t yd = sdesc_sw128(sb + L::OFF_Y + s * L::TILE, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;  // BX == BY: same half stride
            mma_ss(tmem + kColS, sdesc_add(xd, off), sdesc_add(yd, off), id_s, ks > 0);
          }
          mma_commit(s_full);
          if (t) mbar_arrive(s2_issued);  // S2(j) is in the tensor pipe's queue
        }
      }
      __syncwarp();
    } else if (warp == GRAD_WARP) {
      // ------------------------------------------------------------------ MMA issuer: gradients
      // dQ1(j) as soon as dS(j) is in TMEM, so it runs while the dS warps copy S1(j + 1); dQ2(j) once
      // S2(j + 1) is queued, so the logits the dS warps wait for come first (pipe order S1(j + 1),
      // dQ1(j), S2(j + 1), dQ2(j)).
      if (lane == 0) {
        constexpr uint32_t id_g = idesc_bf16(BX, D, false, true);
        bool ok = true;
        for (int j = 0; ok && j < n_yt; ++j) {
          if (!mbar_wait(ds_full, j & 1, status, abort_flag)) break;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int i = 2 * j + t, s = i % SLOTS;
            if (t && j + 1 < n_yt && !mbar_wait(s2_issued, (j + 1) & 1, status, abort_flag)) {
              ok = false;
              break;
            }
            // K_t(j) has landed (its logits MMA read it); waited here too so that this thread's MMAs are
            // ordered after the copy
            if (!mbar_wait(y_full + 8 * s, (i / SLOTS) & 1, status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // A = dS_t packed in TMEM (16 keys = 8 columns per k-step); B = K_t read MN-major
            const uint64_t yd = sdesc_sw128(sb + L::OFF_Y + s * L::TILE, BY * 128, 1024);
            const uint32_t g_col = t ? kColG2 : kColG1, ds_col = t ? kColDS2 : kColDS1;
#pragma unroll
            for (int ks = 0; ks < BY / 16; ++ks)
              mma_ts(tmem + g_col, tmem + ds_col + 8 * ks, sdesc_add(yd, ks * 2048), id_g, j > 0 || ks > 0);
            mma_commit(y_empty + 8 * s);
          }
          if (ok) mma_commit(ds_free);
        }
        mma_commit(g_done);
        mbar_drain(g_done, 0, status);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc_ds();
    // ------------------------------------------------------------------ dS warps
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int xidx = x0 + r;
    const float c = p.c;
    RowVals v{0.f, 0.f, 0.f, 0.f};
    if (xidx < p.NQ) v = row_vals(lse1, lse2, klv, gv, (size_t)bh * p.NQ + xidx);
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tcol = tmem + lane_base + kColS + grp * 32;
    bool ok = true;
    for (int j = 0; j < n_yt; ++j) {
      ok = mbar_wait_warp(s_full, 0, status, abort_flag);  // S1(j): completion 2j
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      uint32_t s1[32];
      tmem_ld32(tcol, s1);
      tmem_ld_wait();
      reg_fence32(s1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      const int ylo = j * BY + grp * 32;  // key columns ylo.., query row xidx
      const bool masked = (ylo + 31 >= p.NK) || (xidx >= p.NQ) || (p.causal && ylo + 31 > xidx + p.off);
      ok = mbar_wait_warp(s_full, 1, status, abort_flag);  // S2(j): completion 2j + 1
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      uint32_t pk1[16], pk2[16];
      // S2 in two halves of 16 columns; the region is released once both are in registers
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t s2[16];
        tmem_ld16(tcol + 16 * h, s2);
        tmem_ld_wait();
        reg_fence16(s2);
        if (h == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
        }
        if (masked)
          make_ds_row_mutual<true, 16>(s1 + 16 * h, s2, pk1 + 8 * h, pk2 + 8 * h, c, p.scale, v.nA, v.nB2, v.nB1,
                                       v.G, visible_keys<16>(xidx, ylo + 16 * h, p.NQ, p.NK, p.off, p.causal));
        else
          make_ds_row_mutual<false, 16>(s1 + 16 * h, s2, pk1 + 8 * h, pk2 + 8 * h, c, p.scale, v.nA, v.nB2, v.nB1,
                                        v.G, 0u);
      }
      reg_fence16(pk1);
      reg_fence16(pk2);
      // the dS columns are free once the gradient MMAs of tile j - 1 are done
      if (j >= 1) {
        ok = mbar_wait_warp(ds_free, (j - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!ok) break;
      }
      tc_fence_after();
      tmem_st16(tmem + lane_base + kColDS1 + 16 * grp, pk1);
      tmem_st16(tmem + lane_base + kColDS2 + 16 * grp, pk2);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // ---- dQ1, dQ2 = scale * accumulators, to bf16: group g writes d columns [32g, 32g + 32)
    const bool got = ok && mbar_wait_warp(g_done, 0, status, abort_flag);
    __syncwarp();
    if (got && grp * 32 < D) {
      tc_fence_after();
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        uint32_t acc[32];
        tmem_ld32(tmem + lane_base + (t ? kColG2 : kColG1) + grp * 32, acc);
        tmem_ld_wait();
        reg_fence32(acc);
        if (xidx < p.NQ)
          store_row32((t ? dq2 : dq1) + row_offset(bh, p.H, xidx, p.qs_b, p.qs_h, p.qs_n) + grp * 32, acc, p.scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================================ dK blocks
namespace mdk {
constexpr int BK = 128, BQ = 128, SLOTS = 4;
constexpr uint32_t kColSA = 0, kColSB = 128, kColG1 = 256, kColG2 = 384;

template <int D>
struct Smem {
  static constexpr int TK = BK * D * 2, TQ = BQ * D * 2;
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = TK;
  static constexpr int OFF_Q = 2 * TK;                   // query-tile ring [SLOTS]
  static constexpr int OFF_DS = OFF_Q + SLOTS * TQ;      // dS[query][key] bf16: 2 halves of [128 queries][128 B]
  static constexpr int OFF_BAR = OFF_DS + BQ * BK * 2;
  // k_full, q_full[4], q_empty[4], sa_full, sa_free, sb_full, sb_free, ds_full, ds_free, g_done; then the
  // TMEM base address slot and the abort flag
  static constexpr int BAR_SLOT = 8 * 16;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");
}  // namespace mdk

// Block `blk` of the dK grid (head-major, the first key tiles first).
template <int D>
__device__ __forceinline__ void dk_mutual_block(const Problem& p, const float* __restrict__ lse1,
                                                const float* __restrict__ lse2, const float* __restrict__ klv,
                                                const float* __restrict__ gv, __nv_bfloat16* __restrict__ dk1,
                                                __nv_bfloat16* __restrict__ dk2, int* status, const CUtensorMap& mk1,
                                                const CUtensorMap& mk2, const CUtensorMap& mq1, const CUtensorMap& mq2,
                                                const unsigned blk) {
  using namespace mdk;
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heads in order; within a head the first key tiles (seen by the most queries when causal) first
  const int n_kt_all = (p.NK + BK - 1) / BK;
  const int bh = (int)(blk / n_kt_all);
  const int mh = bh % p.H, mb = bh / p.H;
  const int k0 = (int)(blk % n_kt_all) * BK;
  const int q_begin = p.causal ? max(0, k0 - p.off) / BQ * BQ : 0;
  const int n_qt = (p.NQ - q_begin + BQ - 1) / BQ;
  const int n_items = 2 * n_qt;  // ring items: Q1(j) = 2j, Q2(j) = 2j + 1

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t k_full = bar, q_full = bar + 8, q_empty = bar + 40, sa_full = bar + 72, sa_free = bar + 80,
                 sb_full = bar + 88, sb_free = bar + 96, ds_full = bar + 104, ds_free = bar + 112, g_done = bar + 120,
                 slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(q_full + 8 * s, 1);
      mbar_init(q_empty + 8 * s, 1);
    }
    mbar_init(sa_full, 1);
    mbar_init(sa_free, DS_WARPS);
    mbar_init(sb_full, 1);
    mbar_init(sb_free, DS_WARPS);
    mbar_init(ds_full, DS_WARPS);
    mbar_init(ds_free, 1);
    mbar_init(g_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_BAR + L::BAR_SLOT);

  if (warp >= DS_WARPS) {
    setmaxnreg_dec_other();
    if (warp == PRODUCER_WARP) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        mbar_arrive_expect_tx(k_full, 2 * L::TK);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(sb + L::OFF_K1 + h * BK * 128, &mk1, k_full, h * 64, k0, mh, mb);
          tma_load_4d(sb + L::OFF_K2 + h * BK * 128, &mk2, k_full, h * 64, k0, mh, mb);
        }
        int issued = 0;
        for (int i = 0; i < n_items; ++i) {
          const int s = i % SLOTS;
          if (i >= SLOTS && !mbar_wait(q_empty + 8 * s, ((i / SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(q_full + 8 * s, L::TQ);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_Q + s * L::TQ + h * BQ * 128, (i & 1) ? &mq2 : &mq1, q_full + 8 * s, h * 64,
                        q_begin + (i >> 1) * BQ, mh, mb);
          issued = i + 1;
        }
        mbar_drain(k_full, 0, status);
        for (int i = max(0, issued - SLOTS); i < issued; ++i)
          mbar_drain(q_full + 8 * (i % SLOTS), (i / SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16(BQ, BK, false, false);
        constexpr uint32_t id_g = idesc_bf16(BK, D, true, true);
        const uint64_t k1d = sdesc_sw128(sb + L::OFF_K1, 0, 1024), k2d = sdesc_sw128(sb + L::OFF_K2, 0, 1024);
        const uint64_t dsm = sdesc_sw128(sb + L::OFF_DS, BQ * 128, 1024);  // dS^T: M = keys, MN-major
        bool ok = mbar_wait(k_full, 0, status, abort_flag);
        // ds_full and ds_free complete twice per query tile: dS1(j) (2j), then dS2(j) (2j + 1)
        for (int j = 0; ok && j <= n_qt; ++j) {
          if (j < n_qt) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int i = 2 * j + t, s = i % SLOTS;
              const uint32_t s_free = t ? sb_free : sa_free;
              if (!mbar_wait(q_full + 8 * s, (i / SLOTS) & 1, status, abort_flag)) {
                ok = false;
                break;
              }
              if (j >= 1 && !mbar_wait(s_free, (j - 1) & 1, status, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t qd = sdesc_sw128(sb + L::OFF_Q + s * L::TQ, 0, 1024);
              const uint64_t kd = t ? k2d : k1d;
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;  // BQ == BK: same half stride
                mma_ss(tmem + (t ? kColSB : kColSA), sdesc_add(qd, off), sdesc_add(kd, off), id_s, ks > 0);
              }
              mma_commit(t ? sb_full : sa_full);
            }
            if (!ok) break;
          }
          if (j >= 1) {
            const int jj = j - 1;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int i = 2 * jj + t, s = i % SLOTS;
              if (!mbar_wait(ds_full, t, status, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              // dK_t += dS_t^T Q_t: A = dS[query][key] read MN-major (M = keys), B = Q_t read MN-major
              const uint64_t qod = sdesc_sw128(sb + L::OFF_Q + s * L::TQ, BQ * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < BQ / 16; ++ks)
                mma_ss(tmem + (t ? kColG2 : kColG1), sdesc_add(dsm, ks * 2048), sdesc_add(qod, ks * 2048), id_g,
                       jj > 0 || ks > 0);
              mma_commit(q_empty + 8 * s);
              mma_commit(ds_free);
            }
            if (!ok) break;
          }
        }
        mma_commit(g_done);
        mbar_drain(g_done, 0, status);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc_ds();
    // ------------------------------------------------------------------ dS warps
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const float c = p.c;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tcol = tmem + lane_base + grp * 32;
    const uint32_t dsb = sb + L::OFF_DS;
    // this row's folded values for query tile j (loaded one tile ahead)
    auto fetch = [&](int j) {
      const int q = q_begin + j * BQ + r;
      if (j < n_qt && q < p.NQ) return row_vals(lse1, lse2, klv, gv, (size_t)bh * p.NQ + q);
      return RowVals{0.f, 0.f, 0.f, 0.f};
    };
    auto store_ds = [&](const uint32_t(&pk)[16]) {
#pragma unroll
      for (int cch = 0; cch < 4; ++cch) {
        const uint32_t dst = sw128<BQ>(dsb, r, grp * 4 + cch);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk[4 * cch]), "r"(pk[4 * cch + 1]),
                     "r"(pk[4 * cch + 2]), "r"(pk[4 * cch + 3])
                     : "memory");
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    };
    // S1(j) is copied out before the loop body of tile j: for j >= 1 while dK1(j - 1)'s MMA, which the
    // dS warps wait for before they can store dS2(j - 1), is running
    uint32_t s1[32];  // this thread's 32 columns of S1 of the current tile
    auto copy_s1 = [&](int j) {
      const bool got = mbar_wait_warp(sa_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!got) return false;
      tc_fence_after();
      tmem_ld32(tcol + kColSA, s1);
      tmem_ld_wait();
      reg_fence32(s1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sa_free);
      return true;
    };
    RowVals v = fetch(0);
    bool ok = n_qt > 0 && copy_s1(0);
    for (int j = 0; ok && j < n_qt; ++j) {
      const RowVals vn = fetch(j + 1);
      const int q = q_begin + j * BQ + r;
      const int kg = k0 + grp * 32;
      const bool masked = (kg + 31 >= p.NK) || (q >= p.NQ) || (p.causal && kg + 31 > q + p.off);
      ok = mbar_wait_warp(sb_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      uint32_t pk1[16], pk2[16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t s2[16];
        tmem_ld16(tcol + kColSB + 16 * h, s2);
        tmem_ld_wait();
        reg_fence16(s2);
        if (h == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sb_free);
        }
        if (masked)
          make_ds_row_mutual<true, 16>(s1 + 16 * h, s2, pk1 + 8 * h, pk2 + 8 * h, c, p.scale, v.nA, v.nB2, v.nB1,
                                       v.G, visible_keys<16>(q, kg + 16 * h, p.NQ, p.NK, p.off, p.causal));
        else
          make_ds_row_mutual<false, 16>(s1 + 16 * h, s2, pk1 + 8 * h, pk2 + 8 * h, c, p.scale, v.nA, v.nB2, v.nB1,
                                        v.G, 0u);
      }
      reg_fence16(pk1);
      reg_fence16(pk2);
      // the dS buffer is free once the previous dK MMA (dK2 of tile j - 1) is done
      if (j >= 1) {
        ok = mbar_wait_warp(ds_free, 1, status, abort_flag);  // completion 2j - 1
        __syncwarp();
        if (!ok) break;
      }
      store_ds(pk1);
      if (j + 1 < n_qt && !(ok = copy_s1(j + 1))) break;  // S1(j + 1) was issued before dK1(j)
      ok = mbar_wait_warp(ds_free, 0, status, abort_flag);  // completion 2j: dK1 of tile j done
      __syncwarp();
      if (!ok) break;
      store_ds(pk2);
      v = vn;
    }
    // ---- dK1, dK2 out: thread = key row k0 + r, group g writes d columns [32g, 32g + 32)
    const bool got = ok && mbar_wait_warp(g_done, 0, status, abort_flag);
    __syncwarp();
    const int key = k0 + r;
    if (got && grp * 32 < D) {
      tc_fence_after();
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        uint32_t acc[32];
        tmem_ld32(tmem + lane_base + (t ? kColG2 : kColG1) + grp * 32, acc);
        tmem_ld_wait();
        reg_fence32(acc);
        if (key < p.NK)
          store_row32((t ? dk2 : dk1) + row_offset(bh, p.H, key, p.ks_b, p.ks_h, p.ks_n) + grp * 32, acc, p.scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Both grids in one launch: blocks [0, n_first) are the first kind's, the rest the other's (dq_first picks
// which comes first: the kind whose blocks walk more tiles).  The grids share no data; with few query tiles
// the dQ grid has few, long blocks and the dK grid many short ones that fill the SMs the former leave idle.
template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_mutual_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                      const float* __restrict__ klv, const float* __restrict__ gv, __nv_bfloat16* __restrict__ dq1,
                      __nv_bfloat16* __restrict__ dk1, __nv_bfloat16* __restrict__ dq2,
                      __nv_bfloat16* __restrict__ dk2, int* status, const __grid_constant__ CUtensorMap mq1,
                      const __grid_constant__ CUtensorMap mq2, const __grid_constant__ CUtensorMap mk1,
                      const __grid_constant__ CUtensorMap mk2, const unsigned n_first, const int dq_first) {
  const unsigned b = blockIdx.x;
  const bool is_dq = dq_first ? b < n_first : b >= n_first;
  const unsigned blk = b < n_first ? b : b - n_first;
  if (is_dq)
    dq_mutual_block<D>(p, lse1, lse2, klv, gv, dq1, dq2, status, mq1, mq2, mk1, mk2, blk);
  else
    dk_mutual_block<D>(p, lse1, lse2, klv, gv, dk1, dk2, status, mk1, mk2, mq1, mq2, blk);
}

template <int D>
cudaError_t mutual_d(const Problem& p, const BwdIn& in, void* dq1, void* dk1, void* dq2, void* dk2, int* status,
                     cudaStream_t st) {
  CUtensorMap mq1, mq2, mk1, mk2;
  if (!encode_q_map(&mq1, in.q1, p, 128) || !encode_q_map(&mq2, in.q2, p, 128) ||
      !encode_k_map(&mk1, in.k1, p, 128) || !encode_k_map(&mk2, in.k2, p, 128))
    return cudaErrorInvalidValue;
  int smem = kOneBlockPerSmSmem;
  if (mdq::Smem<D>::BYTES > smem) smem = mdq::Smem<D>::BYTES;
  if (mdk::Smem<D>::BYTES > smem) smem = mdk::Smem<D>::BYTES;
  auto kern = bwd_mutual_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long dq_blocks = (long long)p.BH * ((p.NQ + mdq::BX - 1) / mdq::BX);
  const long long dk_blocks = (long long)p.BH * ((p.NK + mdk::BK - 1) / mdk::BK);
  const int dq_first = p.NK >= p.NQ;  // a dQ block walks the keys, a dK block the queries
  kern<<<(unsigned)(dq_blocks + dk_blocks), THREADS, smem, st>>>(
      p, in.lse1, in.lse2, in.kl, in.g, static_cast<__nv_bfloat16*>(dq1), static_cast<__nv_bfloat16*>(dk1),
      static_cast<__nv_bfloat16*>(dq2), static_cast<__nv_bfloat16*>(dk2), status, mq1, mq2, mk1, mk2,
      (unsigned)(dq_first ? dq_blocks : dk_blocks), dq_first);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_mutual(const Problem& p, const BwdIn& in, void* dq1, void* dk1, void* dq2, void* dk2,
                              int* status, cudaStream_t st) {
  if (p.D == 64) return mutual_d<64>(p, in, dq1, dk1, dq2, dk2, status, st);
  return mutual_d<128>(p, in, dq1, dk1, dq2, dk2, status, st);
}

}  // namespace skl
