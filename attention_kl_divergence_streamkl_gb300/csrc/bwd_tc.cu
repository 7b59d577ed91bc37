// Recompute-based attention-KL backward on the 5th-generation tensor cores:
// the separate-path dQ and dK kernels.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "recompute strategy": only KL, LSE1, LSE2 are kept; the backward rebuilds
// P_t = exp(S_t - LSE_t) tile by tile.  Setting 1 (P1 fixed) optimises Q2/K2,
// setting 2 (P2 fixed) optimises Q1/K1; the dS arithmetic (ds_math.cuh) is the
// fused kernel's.  dQ = scale dS K_opt, dK = scale dS^T Q_opt.
//
// In both kernels the 128 TMEM lanes of the logits are queries, so a dS thread
// owns a query row and holds its folded LSE1, LSE2, g, KL in registers.
//
// dQ kernel (dq_block): a block owns 128 query rows X (Q1, Q2 stationary) and
// streams key tiles Y:
//     S1 = X1 Y1^T, S2 = X2 Y2^T          (tcgen05, both operands K-major in smem)
//     dS from S1, S2 and the row's values, packed to bf16 into TMEM
//     G += dS Y_opt                       (tcgen05, A = dS in TMEM, B = Y_opt
//                                          read MN-major from the same smem tile)
// so dS never leaves the SM.  TMEM (512 columns): S1 [0,128), S2 [128,256),
// dS double buffer [256,320) / [320,384) (bf16 pairs), G [384, 384 + D).  The
// logits are single-buffered: the dS warps copy their columns into registers
// (in two halves) and release them, so S of the next tile is computed while
// they work.
//   warps 0-15  dS warps: thread = query row (lane quarter = warp % 4), group g = warp / 4
//               takes columns [32g, 32g + 32) of each key tile; then they write dQ out
//   warp 16     TMA producer: X once; Y_opt (read by the gradient MMA, so held until
//               it is done) through three slots, the other Y tile through two
//   warp 17     TMEM owner and MMA issuer; issues S(j) before G += dS(j-1)
// Warpgroup 4 gives registers to the dS warpgroups (setmaxnreg).
//
// The dK kernel (dk_block, below) keeps 128 keys stationary and streams
// query tiles as the M operand of the logits MMA; see its own comment.  When
// both gradients are wanted the two grids run as one launch (bwd_dqdk_kernel).
// A dQ block walks the key tiles and a dK block the query tiles, so with few
// query tiles the dQ grid has few, long blocks and the dK grid many short ones:
// in one launch the dK blocks fill the SMs the dQ blocks leave idle.
#include "common.cuh"
#include "ds_math.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BX = 128;  // stationary query rows (MMA M)
constexpr int BY = 128;  // streamed keys per tile (MMA N of S, K of the gradient MMA)
constexpr int DS_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int QOPT_WARP = 18;  // dK kernel: producer of the Q_opt tiles
constexpr int THREADS = 20 * 32;
constexpr int kRegsDs = 104, kRegsOther = 64;  // 512 * 104 + 128 * 64 = 640 * 96 registers at launch
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS1 = 0, kColS2 = 128, kColDS = 256, kColG = 384;
constexpr int YO_SLOTS = 3, YT_SLOTS = 2;

template <int D>
struct Smem {
  static constexpr int TILE = 128 * D * 2;  // one 128-row bf16 tile, D/64 halves of 16 KiB
  static constexpr int OFF_X1 = 0;
  static constexpr int OFF_X2 = TILE;
  static constexpr int OFF_YO = 2 * TILE;               // Y_opt slots [YO_SLOTS]
  static constexpr int OFF_YT = OFF_YO + YO_SLOTS * TILE;  // the other Y tile, slots [YT_SLOTS]
  static constexpr int OFF_BAR = OFF_YT + YT_SLOTS * TILE;
  // x_full, yo_full[3], yo_empty[3], yt_full[2], yt_empty[2], s_full, s_free, ds_full[2], ds_free[2],
  // g_done; then the TMEM base address slot and the abort flag
  static constexpr int BAR_SLOT = 8 * 18;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ void setmaxnreg_inc_ds() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
}
__device__ __forceinline__ void setmaxnreg_dec_other() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

// One block of the dQ kernel: block `blk` of the dQ grid (head-major, the last query tiles first).
template <int D, int SETTING>
__device__ __forceinline__ void dq_block(const Problem& p, const float* __restrict__ lse1,
                                         const float* __restrict__ lse2, const float* __restrict__ klv,
                                         const float* __restrict__ gv, __nv_bfloat16* __restrict__ out, int* status,
                                         const CUtensorMap& mx1, const CUtensorMap& mx2, const CUtensorMap& my1,
                                         const CUtensorMap& my2, const unsigned blk) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NX = p.NQ, NY = p.NK;
  const int n_xt = (NX + BX - 1) / BX;
  // heads in order (the blocks in flight share one head's K tiles in L2), longest blocks (the last query
  // tiles) first within a head
  const int bh = (int)(blk / n_xt);
  const int mh = bh % p.H, mb = bh / p.H;  // head and batch coordinates of the tensor maps
  const int xt = n_xt - 1 - (int)(blk % n_xt);
  const int x0 = xt * BX;
  const int y_end = p.causal ? min(NY, min(NX, x0 + BX) - 1 + p.off + 1) : NY;  // keys the last row sees
  const int n_yt = (y_end + BY - 1) / BY;

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t x_full = bar, yo_full = bar + 8, yo_empty = bar + 32, yt_full = bar + 56, yt_empty = bar + 72,
                 s_full = bar + 88, s_free = bar + 96, ds_full = bar + 104, ds_free = bar + 120, g_done = bar + 136,
                 slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);

  if (threadIdx.x == 0) {
    mbar_init(x_full, 1);
    for (int s = 0; s < YO_SLOTS; ++s) {
      mbar_init(yo_full + 8 * s, 1);
      mbar_init(yo_empty + 8 * s, 1);
    }
    for (int s = 0; s < YT_SLOTS; ++s) {
      mbar_init(yt_full + 8 * s, 1);
      mbar_init(yt_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ds_full + 8 * b, DS_WARPS);
      mbar_init(ds_free + 8 * b, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, DS_WARPS);
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
          tma_load_4d(sb + L::OFF_X1 + h * BX * 128, &mx1, x_full, h * 64, x0, mh, mb);
          tma_load_4d(sb + L::OFF_X2 + h * BX * 128, &mx2, x_full, h * 64, x0, mh, mb);
        }
        // Y_opt is Y2 in setting 1 (Q2 or K2), Y1 in setting 2
        const CUtensorMap* mopt = SETTING == 1 ? &my2 : &my1;
        const CUtensorMap* moth = SETTING == 1 ? &my1 : &my2;
        int issued = 0, issued_t = 0;
        for (int j = 0; j < n_yt; ++j) {
          const int so = j % YO_SLOTS, st = j % YT_SLOTS;
          if (j >= YO_SLOTS && !mbar_wait(yo_empty + 8 * so, ((j / YO_SLOTS) - 1) & 1, status, abort_flag)) break;
          const int y0 = j * BY;
          mbar_arrive_expect_tx(yo_full + 8 * so, L::TILE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_YO + so * L::TILE + h * BY * 128, mopt, yo_full + 8 * so, h * 64, y0, mh, mb);
          issued = j + 1;
          if (j >= YT_SLOTS && !mbar_wait(yt_empty + 8 * st, ((j / YT_SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(yt_full + 8 * st, L::TILE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_YT + st * L::TILE + h * BY * 128, moth, yt_full + 8 * st, h * 64, y0, mh, mb);
          issued_t = j + 1;
        }
        // copies that may still be landing: the last YO_SLOTS Y_opt tiles and YT_SLOTS other tiles
        mbar_drain(x_full, 0, status);
        for (int j = max(0, issued - YO_SLOTS); j < issued; ++j)
          mbar_drain(yo_full + 8 * (j % YO_SLOTS), (j / YO_SLOTS) & 1, status);
        for (int j = max(0, issued_t - YT_SLOTS); j < issued_t; ++j)
          mbar_drain(yt_full + 8 * (j % YT_SLOTS), (j / YT_SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16(BX, BY, false, false);
        constexpr uint32_t id_g = idesc_bf16(BX, D, false, true);
        const uint64_t x1d = sdesc_sw128(sb + L::OFF_X1, 0, 1024), x2d = sdesc_sw128(sb + L::OFF_X2, 0, 1024);
        bool ok = mbar_wait(x_full, 0, status, abort_flag);
        for (int j = 0; ok && j <= n_yt; ++j) {
          if (j < n_yt) {
            const int so = j % YO_SLOTS, st = j % YT_SLOTS;
            if (!mbar_wait(yo_full + 8 * so, (j / YO_SLOTS) & 1, status, abort_flag)) break;
            if (!mbar_wait(yt_full + 8 * st, (j / YT_SLOTS) & 1, status, abort_flag)) break;
            if (j >= 1 && !mbar_wait(s_free, (j - 1) & 1, status, abort_flag)) break;
            tc_fence_after();
            const uint32_t yo = sb + L::OFF_YO + so * L::TILE, yt = sb + L::OFF_YT + st * L::TILE;
            const uint64_t y1d = sdesc_sw128(SETTING == 1 ? yt : yo, 0, 1024);
            const uint64_t y2d = sdesc_sw128(SETTING == 1 ? yo : yt, 0, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;  // BX == BY: same half stride
              mma_ss(tmem + kColS1, sdesc_add(x1d, off), sdesc_add(y1d, off), id_s, ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
              mma_ss(tmem + kColS2, sdesc_add(x2d, off), sdesc_add(y2d, off), id_s, ks > 0);
            }
            mma_commit(s_full);
            mma_commit(yt_empty + 8 * st);  // the other Y tile is read only by these MMAs
          }
          if (j >= 1) {
            const int jj = j - 1, b = jj & 1;
            if (!mbar_wait(ds_full + 8 * b, (jj >> 1) & 1, status, abort_flag)) break;
            tc_fence_after();
            // A = dS packed in TMEM (16 Y rows = 8 columns per k-step); B = Y_opt read MN-major
            const uint64_t yod = sdesc_sw128(sb + L::OFF_YO + (jj % YO_SLOTS) * L::TILE, BY * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < BY / 16; ++ks)
              mma_ts(tmem + kColG, tmem + kColDS + 64 * b + 8 * ks, sdesc_add(yod, ks * 2048), id_g, jj > 0 || ks > 0);
            mma_commit(yo_empty + 8 * (jj % YO_SLOTS));
            mma_commit(ds_free + 8 * b);
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
    const int xidx = x0 + r;
    const float c = p.c;
    float nAr = 0.f, nBr = 0.f, Gr = 0.f;  // the row's folded values
    if (xidx < p.NQ) {
      const size_t o = (size_t)bh * p.NQ + xidx;
      const float l1v = lse1[o], l2v = lse2[o];
      nAr = -l1v * kLog2e;
      nBr = SETTING == 1 ? -l2v * kLog2e : -(l1v - l2v + klv[o]);
      Gr = gv[o];
    }
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tcol = tmem + lane_base + grp * 32;
    bool ok = true;
    for (int j = 0; j < n_yt; ++j) {
      const int b = j & 1;
      ok = mbar_wait_warp(s_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const int ylo = j * BY + grp * 32;  // key columns ylo.., query row xidx
      const bool masked = (ylo + 31 >= p.NK) || (xidx >= p.NQ) || (p.causal && ylo + 31 > xidx + p.off);
      uint32_t pk[16];
      // Two halves of 16 columns: the second half is read after the first is
      // computed, and the logits' TMEM is released once both are in registers.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[16], bb[16];
        tmem_ld16(tcol + kColS1 + 16 * h, a);
        tmem_ld16(tcol + kColS2 + 16 * h, bb);
        tmem_ld_wait();
        reg_fence16(a);
        reg_fence16(bb);
        if (h == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
        }
        const int y = ylo + 16 * h;
        if (masked)
          make_ds_row<SETTING, true, 16>(a, bb, pk + 8 * h, c, p.scale, nAr, nBr, Gr,
                                         visible_keys<16>(xidx, y, p.NQ, p.NK, p.off, p.causal));
        else
          make_ds_row<SETTING, false, 16>(a, bb, pk + 8 * h, c, p.scale, nAr, nBr, Gr, 0u);
        if (h == 0)  // first half final before the second half is read
          asm volatile("" : "+r"(pk[0]), "+r"(pk[1]), "+r"(pk[2]), "+r"(pk[3]), "+r"(pk[4]), "+r"(pk[5]),
                       "+r"(pk[6]), "+r"(pk[7])::"memory");
      }
      reg_fence16(pk);
      // dS buffer b is free once the gradient MMA of tile j - 2 is done
      if (j >= 2) {
        ok = mbar_wait_warp(ds_free + 8 * b, ((j >> 1) - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!ok) break;
      }
      tc_fence_after();
      tmem_st16(tmem + lane_base + kColDS + 64 * b + 16 * grp, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full + 8 * b);
    }
    // ---- G = sum dS Y_opt, scaled, to bf16: group g writes d columns [32g, 32g + 32)
    const bool got = ok && mbar_wait_warp(g_done, 0, status, abort_flag);
    __syncwarp();
    if (got && grp * 32 < D) {
      tc_fence_after();
      uint32_t g0[32];
      tmem_ld32(tmem + lane_base + kColG + grp * 32, g0);
      tmem_ld_wait();
      reg_fence32(g0);
      if (xidx < NX) {
        __nv_bfloat16* dst = out + row_offset(bh, p.H, xidx, p.qs_b, p.qs_h, p.qs_n) + grp * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t* src = &g0[v * 8];
          uint4 o;
          o.x = pack_bf16(__uint_as_float(src[0]) * p.scale, __uint_as_float(src[1]) * p.scale);
          o.y = pack_bf16(__uint_as_float(src[2]) * p.scale, __uint_as_float(src[3]) * p.scale);
          o.z = pack_bf16(__uint_as_float(src[4]) * p.scale, __uint_as_float(src[5]) * p.scale);
          o.w = pack_bf16(__uint_as_float(src[6]) * p.scale, __uint_as_float(src[7]) * p.scale);
          reinterpret_cast<uint4*>(dst)[v] = o;
        }
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

// ---------------------------------------------------------------------------
// The dK kernel.  A block owns 128 keys (K1, K2 stationary in smem) and streams
// 128-query tiles, but computes the logits with the query tile as the MMA's M
// operand, so the 128 TMEM lanes are queries: a dS thread owns a query row and
// holds its folded values in registers (no shared-memory loads in the dS loop).
// dS goes to smem as dS[query][key] and dK += dS^T Q_opt reads it MN-major, so
// the dK accumulator has the keys on its lanes.
//   S_a = Q_a K_a^T, S_b = Q_b K_b^T   SS, K-major, TMEM [0, 128) and [128, 256) (lanes = queries)
//   dK += dS^T Q_opt                   SS: A = dS read MN-major (M = keys), B = Q_opt MN-major -> [256, 256 + D)
//   warps 0-15  dS warps: thread = query row, group g = key columns [32g, 32g + 32);
//               at the end, thread = key row, group g = d columns [32g, 32g + 32) of dK
//   warp 16     TMA producer: K1, K2 once, then the other Q tile through two slots
//   warp 17     TMEM owner and MMA issuer
//   warp 18     TMA producer of Q_opt (two slots, held until the dK MMA)
namespace dkk {
constexpr int BK = 128, BQ = 128, SLOTS = 2;
constexpr uint32_t kColSA = 0, kColSB = 128, kColG = 256;

template <int D>
struct Smem {
  static constexpr int TK = BK * D * 2, TQ = BQ * D * 2;
  static constexpr int OFF_KA = 0;                       // the other K (K1 in setting 1, K2 in setting 2)
  static constexpr int OFF_KB = TK;                      // K_opt
  static constexpr int OFF_QO = 2 * TK;                  // Q_opt slots
  static constexpr int OFF_QT = OFF_QO + SLOTS * TQ;     // the other Q tile's slots
  static constexpr int OFF_DS = OFF_QT + SLOTS * TQ;     // dS[query][key] bf16: 2 halves of [128 queries][128 B]
  static constexpr int OFF_BAR = OFF_DS + BQ * BK * 2;
  // k_full, qo_full[2], qo_empty[2], qt_full[2], qt_empty[2], sa_full, sa_free, sb_full, sb_free,
  // ds_full, ds_free, g_done; then the TMEM base address slot and the abort flag
  static constexpr int BAR_SLOT = 16 * 8;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");
}  // namespace dkk

// One block of the dK kernel: block `blk` of the dK grid (head-major, the first key tiles first).
template <int D, int SETTING>
__device__ __forceinline__ void dk_block(const Problem& p, const float* __restrict__ lse1,
                                         const float* __restrict__ lse2, const float* __restrict__ klv,
                                         const float* __restrict__ gv, __nv_bfloat16* __restrict__ dk_out, int* status,
                                         const CUtensorMap& mk1, const CUtensorMap& mk2, const CUtensorMap& mq1,
                                         const CUtensorMap& mq2, const unsigned blk) {
  using dkk::BK;
  using dkk::BQ;
  using dkk::SLOTS;
  using L = dkk::Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heads in order (the blocks in flight share one head's Q tiles in L2); within a head the first key
  // tiles, which see the most queries, first
  const int n_kt_all = (p.NK + BK - 1) / BK;
  const int bh = (int)(blk / n_kt_all);
  const int mh = bh % p.H, mb = bh / p.H;  // head and batch coordinates of the tensor maps
  const int kt = (int)(blk % n_kt_all);
  const int k0 = kt * BK;
  const int q_begin = p.causal ? max(0, k0 - p.off) / BQ * BQ : 0;
  const int n_qt = (p.NQ - q_begin + BQ - 1) / BQ;

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t k_full = bar, qo_full = bar + 8, qo_empty = bar + 24, qt_full = bar + 40, qt_empty = bar + 56,
                 sa_full = bar + 72, sa_free = bar + 80, sb_full = bar + 88, sb_free = bar + 96, ds_full = bar + 104,
                 ds_free = bar + 112, g_done = bar + 120, slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(qo_full + 8 * s, 1);
      mbar_init(qo_empty + 8 * s, 1);
      mbar_init(qt_full + 8 * s, 1);
      mbar_init(qt_empty + 8 * s, 1);
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
          tma_load_4d(sb + L::OFF_KA + h * BK * 128, SETTING == 1 ? &mk1 : &mk2, k_full, h * 64, k0, mh, mb);
          tma_load_4d(sb + L::OFF_KB + h * BK * 128, SETTING == 1 ? &mk2 : &mk1, k_full, h * 64, k0, mh, mb);
        }
        const CUtensorMap* mqa = SETTING == 1 ? &mq1 : &mq2;
        int issued = 0;
        for (int j = 0; j < n_qt; ++j) {
          const int s = j % SLOTS;
          if (j >= SLOTS && !mbar_wait(qt_empty + 8 * s, ((j / SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(qt_full + 8 * s, L::TQ);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_QT + s * L::TQ + h * BQ * 128, mqa, qt_full + 8 * s, h * 64, q_begin + j * BQ, mh, mb);
          issued = j + 1;
        }
        mbar_drain(k_full, 0, status);
        for (int j = max(0, issued - SLOTS); j < issued; ++j)
          mbar_drain(qt_full + 8 * (j % SLOTS), (j / SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == QOPT_WARP) {
      // ------------------------------------------------------------------ TMA producer of Q_opt
      if (lane == 0) {
        const CUtensorMap* mqb = SETTING == 1 ? &mq2 : &mq1;
        int issued = 0;
        for (int j = 0; j < n_qt; ++j) {
          const int s = j % SLOTS;
          if (j >= SLOTS && !mbar_wait(qo_empty + 8 * s, ((j / SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(qo_full + 8 * s, L::TQ);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_QO + s * L::TQ + h * BQ * 128, mqb, qo_full + 8 * s, h * 64, q_begin + j * BQ, mh, mb);
          issued = j + 1;
        }
        for (int j = max(0, issued - SLOTS); j < issued; ++j)
          mbar_drain(qo_full + 8 * (j % SLOTS), (j / SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16(BQ, BK, false, false);
        constexpr uint32_t id_g = idesc_bf16(BK, D, true, true);
        const uint64_t kad = sdesc_sw128(sb + L::OFF_KA, 0, 1024), kbd = sdesc_sw128(sb + L::OFF_KB, 0, 1024);
        const uint64_t dsm = sdesc_sw128(sb + L::OFF_DS, BQ * 128, 1024);  // dS^T: M = keys, MN-major
        bool ok = mbar_wait(k_full, 0, status, abort_flag);
        for (int j = 0; ok && j <= n_qt; ++j) {
          if (j < n_qt) {
            const int s = j % SLOTS;
            if (!mbar_wait(qt_full + 8 * s, (j / SLOTS) & 1, status, abort_flag)) break;
            if (j >= 1 && !mbar_wait(sa_free, (j - 1) & 1, status, abort_flag)) break;
            tc_fence_after();
            const uint64_t qad = sdesc_sw128(sb + L::OFF_QT + s * L::TQ, 0, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;  // BQ == BK: same half stride
              mma_ss(tmem + dkk::kColSA, sdesc_add(qad, off), sdesc_add(kad, off), id_s, ks > 0);
            }
            mma_commit(sa_full);
            mma_commit(qt_empty + 8 * s);  // the other Q tile is read only by S_a
            if (!mbar_wait(qo_full + 8 * s, (j / SLOTS) & 1, status, abort_flag)) break;
            if (j >= 1 && !mbar_wait(sb_free, (j - 1) & 1, status, abort_flag)) break;
            tc_fence_after();
            const uint64_t qbd = sdesc_sw128(sb + L::OFF_QO + s * L::TQ, 0, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
              mma_ss(tmem + dkk::kColSB, sdesc_add(qbd, off), sdesc_add(kbd, off), id_s, ks > 0);
            }
            mma_commit(sb_full);
          }
          if (j >= 1) {
            const int jj = j - 1, s = jj % SLOTS;
            if (!mbar_wait(ds_full, jj & 1, status, abort_flag)) break;
            tc_fence_after();
            // dK += dS^T Q_opt: A = dS[query][key] read MN-major (M = keys), B = Q_opt read MN-major
            const uint64_t qod = sdesc_sw128(sb + L::OFF_QO + s * L::TQ, BQ * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < BQ / 16; ++ks)
              mma_ss(tmem + dkk::kColG, sdesc_add(dsm, ks * 2048), sdesc_add(qod, ks * 2048), id_g, jj > 0 || ks > 0);
            mma_commit(qo_empty + 8 * s);
            mma_commit(ds_free);
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
    auto fetch = [&](int j, float& a, float& b, float& g) {
      const int q = q_begin + j * BQ + r;
      a = b = g = 0.f;
      if (j < n_qt && q < p.NQ) {
        const size_t o = (size_t)bh * p.NQ + q;
        const float l1v = lse1[o], l2v = lse2[o];
        a = -l1v * kLog2e;
        b = SETTING == 1 ? -l2v * kLog2e : -(l1v - l2v + klv[o]);
        g = gv[o];
      }
    };
    float nAr, nBr, Gr, nA2, nB2, G2;
    fetch(0, nAr, nBr, Gr);
    bool ok = true;
    for (int j = 0; j < n_qt; ++j) {
      fetch(j + 1, nA2, nB2, G2);
      const int q = q_begin + j * BQ + r;
      ok = mbar_wait_warp(sa_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      uint32_t held[32];  // this thread's 32 columns of S_a
      tmem_ld32(tcol + dkk::kColSA, held);
      tmem_ld_wait();
      reg_fence32(held);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sa_free);
      const int kg = k0 + grp * 32;
      const bool masked = (kg + 31 >= p.NK) || (q >= p.NQ) || (p.causal && kg + 31 > q + p.off);
      uint32_t pk[16];
      ok = mbar_wait_warp(sb_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t half[16];
        tmem_ld16(tcol + dkk::kColSB + 16 * h, half);
        tmem_ld_wait();
        reg_fence16(half);
        if (h == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sb_free);
        }
        const uint32_t(&ha)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&held[16 * h]);
        auto run = [&](const uint32_t(&s1)[16], const uint32_t(&s2)[16]) {
          if (masked)
            make_ds_row<SETTING, true, 16>(s1, s2, pk + 8 * h, c, p.scale, nAr, nBr, Gr,
                                           visible_keys<16>(q, kg + 16 * h, p.NQ, p.NK, p.off, p.causal));
          else
            make_ds_row<SETTING, false, 16>(s1, s2, pk + 8 * h, c, p.scale, nAr, nBr, Gr, 0u);
        };
        if (SETTING == 1)
          run(ha, half);  // S_a = S1, S_b = S2
        else
          run(half, ha);  // S_a = S2, S_b = S1
        if (h == 0)  // first half final before the second half is read
          asm volatile("" : "+r"(pk[0]), "+r"(pk[1]), "+r"(pk[2]), "+r"(pk[3]), "+r"(pk[4]), "+r"(pk[5]),
                       "+r"(pk[6]), "+r"(pk[7])::"memory");
      }
      reg_fence16(pk);
      // dS smem is free once the dK MMA of the previous tile is done
      if (j >= 1) {
        ok = mbar_wait_warp(ds_free, (j - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!ok) break;
      }
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
      nAr = nA2;
      nBr = nB2;
      Gr = G2;
    }
    // ---- dK out: thread = key row k0 + r, group g writes d columns [32g, 32g + 32)
    const bool got = ok && mbar_wait_warp(g_done, 0, status, abort_flag);
    __syncwarp();
    const int key = k0 + r;
    if (got && grp * 32 < D) {
      tc_fence_after();
      uint32_t g0[32];
      tmem_ld32(tmem + lane_base + dkk::kColG + grp * 32, g0);
      tmem_ld_wait();
      reg_fence32(g0);
      if (key < p.NK) {
        __nv_bfloat16* dst = dk_out + row_offset(bh, p.H, key, p.ks_b, p.ks_h, p.ks_n) + grp * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t* src = &g0[v * 8];
          uint4 o;
          o.x = pack_bf16(__uint_as_float(src[0]) * p.scale, __uint_as_float(src[1]) * p.scale);
          o.y = pack_bf16(__uint_as_float(src[2]) * p.scale, __uint_as_float(src[3]) * p.scale);
          o.z = pack_bf16(__uint_as_float(src[4]) * p.scale, __uint_as_float(src[5]) * p.scale);
          o.w = pack_bf16(__uint_as_float(src[6]) * p.scale, __uint_as_float(src[7]) * p.scale);
          reinterpret_cast<uint4*>(dst)[v] = o;
        }
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

template <int D, int SETTING>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dq_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                  const float* __restrict__ klv, const float* __restrict__ gv, __nv_bfloat16* __restrict__ out,
                  int* status, const __grid_constant__ CUtensorMap mq1, const __grid_constant__ CUtensorMap mq2,
                  const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mk2) {
  dq_block<D, SETTING>(p, lse1, lse2, klv, gv, out, status, mq1, mq2, mk1, mk2, blockIdx.x);
}

template <int D, int SETTING>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dk_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                  const float* __restrict__ klv, const float* __restrict__ gv, __nv_bfloat16* __restrict__ dk_out,
                  int* status, const __grid_constant__ CUtensorMap mq1, const __grid_constant__ CUtensorMap mq2,
                  const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mk2) {
  dk_block<D, SETTING>(p, lse1, lse2, klv, gv, dk_out, status, mk1, mk2, mq1, mq2, blockIdx.x);
}

// The dQ and the dK grids in one launch: blocks [0, n_first) are the first kind's, the rest the other's
// (dq_first picks which comes first: the kind whose blocks walk more tiles).  The two kinds share no data, so
// the short blocks of one fill the SMs the long blocks of the other leave free -- with few query tiles the dQ
// grid alone has a block per head.
template <int D, int SETTING>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dqdk_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                    const float* __restrict__ klv, const float* __restrict__ gv, __nv_bfloat16* __restrict__ dq_out,
                    __nv_bfloat16* __restrict__ dk_out, int* status, const __grid_constant__ CUtensorMap mq1,
                    const __grid_constant__ CUtensorMap mq2, const __grid_constant__ CUtensorMap mk1,
                    const __grid_constant__ CUtensorMap mk2, const unsigned n_first, const int dq_first) {
  const unsigned b = blockIdx.x;
  const bool is_dq = dq_first ? b < n_first : b >= n_first;
  const unsigned blk = b < n_first ? b : b - n_first;
  if (is_dq)
    dq_block<D, SETTING>(p, lse1, lse2, klv, gv, dq_out, status, mq1, mq2, mk1, mk2, blk);
  else
    dk_block<D, SETTING>(p, lse1, lse2, klv, gv, dk_out, status, mk1, mk2, mq1, mq2, blk);
}

constexpr int kOneBlockPerSmSmem = 120 * 1024;  // a block owns all 512 TMEM columns

template <int D, int SETTING>
cudaError_t launch_sep(const Problem& p, const BwdIn& in, void* dq, void* dk, int* status, cudaStream_t st) {
  static_assert(BX == 128 && BY == 128 && dkk::BK == 128 && dkk::BQ == 128, "one box height for every map");
  CUtensorMap mq1, mq2, mk1, mk2;
  if (!encode_q_map(&mq1, in.q1, p, 128) || !encode_q_map(&mq2, in.q2, p, 128) ||
      !encode_k_map(&mk1, in.k1, p, 128) || !encode_k_map(&mk2, in.k2, p, 128))
    return cudaErrorInvalidValue;
  const long long dq_blocks = (long long)p.BH * ((p.NQ + BX - 1) / BX);
  const long long dk_blocks = (long long)p.BH * ((p.NK + dkk::BK - 1) / dkk::BK);
  auto* dq_out = static_cast<__nv_bfloat16*>(dq);
  auto* dk_out = static_cast<__nv_bfloat16*>(dk);
  int smem = kOneBlockPerSmSmem;
  if (dq && Smem<D>::BYTES > smem) smem = Smem<D>::BYTES;
  if (dk && dkk::Smem<D>::BYTES > smem) smem = dkk::Smem<D>::BYTES;
  cudaError_t e;
  if (dq && dk) {
    auto kern = bwd_dqdk_kernel<D, SETTING>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    const int dq_first = p.NK >= p.NQ;  // a dQ block walks the keys, a dK block the queries
    kern<<<(unsigned)(dq_blocks + dk_blocks), THREADS, smem, st>>>(p, in.lse1, in.lse2, in.kl, in.g, dq_out, dk_out,
                                                                   status, mq1, mq2, mk1, mk2,
                                                                   (unsigned)(dq_first ? dq_blocks : dk_blocks),
                                                                   dq_first);
  } else if (dq) {
    auto kern = bwd_dq_kernel<D, SETTING>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    kern<<<(unsigned)dq_blocks, THREADS, smem, st>>>(p, in.lse1, in.lse2, in.kl, in.g, dq_out, status, mq1, mq2, mk1,
                                                     mk2);
  } else if (dk) {
    auto kern = bwd_dk_kernel<D, SETTING>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    kern<<<(unsigned)dk_blocks, THREADS, smem, st>>>(p, in.lse1, in.lse2, in.kl, in.g, dk_out, status, mq1, mq2, mk1,
                                                     mk2);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t separate_d(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, int* status,
                       cudaStream_t st) {
  return setting == 1 ? launch_sep<D, 1>(p, in, dq, dk, status, st) : launch_sep<D, 2>(p, in, dq, dk, status, st);
}

}  // namespace

cudaError_t launch_bwd_separate(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, int* status,
                                cudaStream_t st) {
  if (p.D == 64) return separate_d<64>(p, setting, in, dq, dk, status, st);
  return separate_d<128>(p, setting, in, dq, dk, status, st);
}

}  // namespace skl
