// Recompute-based attention-KL backward on the 5th-generation tensor cores:
// the separate-path dQ and dK kernels.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "recompute strategy": only KL, LSE1, LSE2 are kept; the backward rebuilds
// P_t = exp(S_t - LSE_t) tile by tile.  Setting 1 (P1 fixed) optimises Q2/K2,
// setting 2 (P2 fixed) optimises Q1/K1; the dS arithmetic (ds_math.cuh) is the
// fused kernel's.  dQ = scale dS K_opt, dK = scale dS^T Q_opt.
//
// One kernel template serves both separate kernels.  A block owns a stationary
// tile X of 128 rows (query rows for dQ, keys for dK) on the 128 TMEM lanes and
// streams tiles Y of 128 rows of the other side:
//     S1 = X1 Y1^T, S2 = X2 Y2^T          (tcgen05, both operands K-major in smem)
//     dS from S1, S2 and the folded per-query values, packed to bf16 into TMEM
//     G += dS Y_opt                       (tcgen05, A = dS in TMEM, B = Y_opt
//                                          read MN-major from the same smem tile)
// so dS never leaves the SM.  TMEM (512 columns): S1 [0,128), S2 [128,256),
// dS double buffer [256,320) / [320,384) (bf16 pairs), G [384, 384 + D).  The
// logits are single-buffered: the dS warps copy their columns into registers
// (in two halves) and release them, so S of the next tile is computed while
// they work.
//   warps 0-15  dS warps: thread = X row (lane quarter = warp % 4), group g = warp / 4
//               takes columns [32g, 32g + 32) of each Y tile; then they write G out
//   warp 16     TMA producer: X once; Y_opt (read by the gradient MMA, so held until
//               it is done) through three slots, the other Y tile through two
//   warp 17     TMEM owner and MMA issuer; issues S(j) before G += dS(j-1)
//   warp 18     (dK kernel) stages the per-query values of each Y tile in smem
// Warpgroup 4 gives registers to the dS warpgroups (setmaxnreg).
#include "common.cuh"
#include "ds_math.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BX = 128;  // stationary rows (MMA M)
constexpr int BY = 128;  // streamed rows per tile (MMA N of S, K of the gradient MMA)
constexpr int DS_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int VALS_WARP = 18;
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
  static constexpr int OFF_VALS = OFF_YT + YT_SLOTS * TILE;  // [3][BY] fp32 (dK kernel), one tile
  static constexpr int OFF_BAR = OFF_VALS + 3 * BY * 4;
  // x_full, yo_full[3], yo_empty[3], yt_full[2], yt_empty[2], s_full, s_free, v_full, v_free, ds_full[2],
  // ds_free[2], g_done; then the TMEM base address slot and the abort flag
  static constexpr int BAR_SLOT = 8 * 20;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ void setmaxnreg_inc_ds() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
}
__device__ __forceinline__ void setmaxnreg_dec_other() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

template <int D, int SETTING, bool KSTAT>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_tc_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                  const float* __restrict__ klv, const float* __restrict__ gv, __nv_bfloat16* __restrict__ out,
                  int* status, const __grid_constant__ CUtensorMap mx1, const __grid_constant__ CUtensorMap mx2,
                  const __grid_constant__ CUtensorMap my1, const __grid_constant__ CUtensorMap my2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // X side: queries (dQ) or keys (dK); Y side: the other
  const int NX = KSTAT ? p.NK : p.NQ, NY = KSTAT ? p.NQ : p.NK;
  const int n_xt = (NX + BX - 1) / BX;
  const int bh = blockIdx.x % p.BH;
  // longest blocks first: for dQ the last query tiles, for dK the first key tiles
  const int xt = KSTAT ? (int)(blockIdx.x / p.BH) : n_xt - 1 - (int)(blockIdx.x / p.BH);
  const int x0 = xt * BX;
  int y_begin = 0, y_end = NY;
  if (p.causal) {
    if (KSTAT) y_begin = max(0, x0 - p.off) / BY * BY;            // first query that sees key x0
    else y_end = min(p.NK, min(p.NQ, x0 + BX) - 1 + p.off + 1);  // keys the last row sees
  }
  const int y_first = y_begin / BY;
  const int n_yt = (y_end - y_begin + BY - 1) / BY;

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t x_full = bar, yo_full = bar + 8, yo_empty = bar + 32, yt_full = bar + 56, yt_empty = bar + 72,
                 s_full = bar + 88, s_free = bar + 96, v_full = bar + 104, v_free = bar + 112, ds_full = bar + 120,
                 ds_free = bar + 136, g_done = bar + 152, slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);
  float* vals = reinterpret_cast<float*>(smem + L::OFF_VALS);

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
    mbar_init(v_full, 1);
    mbar_init(v_free, DS_WARPS);
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
          tma_load_3d(sb + L::OFF_X1 + h * BX * 128, &mx1, x_full, h * 64, x0, bh);
          tma_load_3d(sb + L::OFF_X2 + h * BX * 128, &mx2, x_full, h * 64, x0, bh);
        }
        // Y_opt is Y2 in setting 1 (Q2 or K2), Y1 in setting 2
        const CUtensorMap* mopt = SETTING == 1 ? &my2 : &my1;
        const CUtensorMap* moth = SETTING == 1 ? &my1 : &my2;
        int issued = 0, issued_t = 0;
        for (int j = 0; j < n_yt; ++j) {
          const int so = j % YO_SLOTS, st = j % YT_SLOTS;
          if (j >= YO_SLOTS && !mbar_wait(yo_empty + 8 * so, ((j / YO_SLOTS) - 1) & 1, status, abort_flag)) break;
          const int y0 = (y_first + j) * BY;
          mbar_arrive_expect_tx(yo_full + 8 * so, L::TILE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(sb + L::OFF_YO + so * L::TILE + h * BY * 128, mopt, yo_full + 8 * so, h * 64, y0, bh);
          issued = j + 1;
          if (j >= YT_SLOTS && !mbar_wait(yt_empty + 8 * st, ((j / YT_SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(yt_full + 8 * st, L::TILE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(sb + L::OFF_YT + st * L::TILE + h * BY * 128, moth, yt_full + 8 * st, h * 64, y0, bh);
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
    } else if (warp == VALS_WARP && KSTAT) {
      // ------------------------------------------------------------------ per-query values (dK kernel)
      // Loads for tile j are issued before waiting for the dS warps to release the
      // previous tile's values, so their latency overlaps that wait.
      constexpr int PER = BY / 32;
      float a[PER], b[PER], g[PER];
      auto fetch = [&](int j) {
        const int q0 = (y_first + j) * BY;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const int q = q0 + lane + 32 * k;
          const bool in = q < p.NQ;
          const size_t o = (size_t)bh * p.NQ + (in ? q : 0);
          const float l1v = in ? lse1[o] : 0.f, l2v = in ? lse2[o] : 0.f;
          a[k] = -l1v * kLog2e;
          b[k] = SETTING == 1 ? -l2v * kLog2e : -(l1v - l2v + (in ? klv[o] : 0.f));
          g[k] = in ? gv[o] : 0.f;
        }
      };
      if (n_yt > 0) fetch(0);
      for (int j = 0; j < n_yt; ++j) {
        const bool ok = j == 0 || mbar_wait(v_free, (j - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          vals[lane + 32 * k] = a[k];
          vals[BY + lane + 32 * k] = b[k];
          vals[2 * BY + lane + 32 * k] = g[k];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(v_full);
        if (j + 1 < n_yt) fetch(j + 1);
      }
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
    float nAr = 0.f, nBr = 0.f, Gr = 0.f;  // dQ kernel: the row's folded values
    if (!KSTAT && xidx < p.NQ) {
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
      ok = mbar_wait(s_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const int ylo = (y_first + j) * BY + grp * 32;
      bool masked;
      if (KSTAT)  // query columns ylo.., key row xidx
        masked = (ylo + 31 >= p.NQ) || (xidx >= p.NK) || (p.causal && xidx > ylo + p.off);
      else  // key columns ylo.., query row xidx
        masked = (ylo + 31 >= p.NK) || (xidx >= p.NQ) || (p.causal && ylo + 31 > xidx + p.off);
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
        } else if (KSTAT) {
          ok = mbar_wait(v_full, j & 1, status, abort_flag);
          __syncwarp();
          if (!ok) break;
        }
        const int y = ylo + 16 * h;
        if (KSTAT) {
          const float* vh = vals + grp * 32 + 16 * h;
          if (masked)
            make_ds_cols<SETTING, true, 16, BY>(a, bb, pk + 8 * h, c, p.scale, vh,
                                                visible_queries<16>(xidx, y, p.NQ, p.NK, p.off, p.causal));
          else
            make_ds_cols<SETTING, false, 16, BY>(a, bb, pk + 8 * h, c, p.scale, vh, 0u);
        } else {
          if (masked)
            make_ds_row<SETTING, true, 16>(a, bb, pk + 8 * h, c, p.scale, nAr, nBr, Gr,
                                           visible_keys<16>(xidx, y, p.NQ, p.NK, p.off, p.causal));
          else
            make_ds_row<SETTING, false, 16>(a, bb, pk + 8 * h, c, p.scale, nAr, nBr, Gr, 0u);
        }
        if (h == 0)  // first half final before the second half is read
          asm volatile("" : "+r"(pk[0]), "+r"(pk[1]), "+r"(pk[2]), "+r"(pk[3]), "+r"(pk[4]), "+r"(pk[5]),
                       "+r"(pk[6]), "+r"(pk[7])::"memory");
      }
      if (!ok) break;
      reg_fence16(pk);
      if (KSTAT) {
        __syncwarp();
        if (lane == 0) mbar_arrive(v_free);
      }
      // dS buffer b is free once the gradient MMA of tile j - 2 is done
      if (j >= 2) {
        ok = mbar_wait(ds_free + 8 * b, ((j >> 1) - 1) & 1, status, abort_flag);
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
    const bool got = ok && mbar_wait(g_done, 0, status, abort_flag);
    __syncwarp();
    if (got && grp * 32 < D) {
      tc_fence_after();
      uint32_t g0[32];
      tmem_ld32(tmem + lane_base + kColG + grp * 32, g0);
      tmem_ld_wait();
      reg_fence32(g0);
      if (xidx < NX) {
        __nv_bfloat16* dst = out + ((size_t)bh * NX + xidx) * D + grp * 32;
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

constexpr int kOneBlockPerSmSmem = 120 * 1024;  // a block owns all 512 TMEM columns

template <int D, int SETTING, bool KSTAT>
cudaError_t launch_one(const Problem& p, const BwdIn& in, void* out, int* status, cudaStream_t st) {
  const void* x1 = KSTAT ? in.k1 : in.q1;
  const void* x2 = KSTAT ? in.k2 : in.q2;
  const void* y1 = KSTAT ? in.q1 : in.k1;
  const void* y2 = KSTAT ? in.q2 : in.k2;
  const int NX = KSTAT ? p.NK : p.NQ, NY = KSTAT ? p.NQ : p.NK;
  CUtensorMap mx1, mx2, my1, my2;
  if (!encode_tile_map(&mx1, x1, D, NX, p.BH, BX) || !encode_tile_map(&mx2, x2, D, NX, p.BH, BX) ||
      !encode_tile_map(&my1, y1, D, NY, p.BH, BY) || !encode_tile_map(&my2, y2, D, NY, p.BH, BY))
    return cudaErrorInvalidValue;
  const int smem = Smem<D>::BYTES > kOneBlockPerSmSmem ? Smem<D>::BYTES : kOneBlockPerSmSmem;
  auto kern = bwd_tc_kernel<D, SETTING, KSTAT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.BH * ((NX + BX - 1) / BX);
  kern<<<(unsigned)blocks, THREADS, smem, st>>>(p, in.lse1, in.lse2, in.kl, in.g, static_cast<__nv_bfloat16*>(out),
                                                status, mx1, mx2, my1, my2);
  return cudaGetLastError();
}

template <int D>
cudaError_t separate_d(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, int* status,
                       cudaStream_t st) {
  if (dq) {
    cudaError_t e = setting == 1 ? launch_one<D, 1, false>(p, in, dq, status, st)
                                 : launch_one<D, 2, false>(p, in, dq, status, st);
    if (e != cudaSuccess) return e;
  }
  if (!dk) return cudaSuccess;
  return setting == 1 ? launch_one<D, 1, true>(p, in, dk, status, st) : launch_one<D, 2, true>(p, in, dk, status, st);
}

}  // namespace

cudaError_t launch_bwd_separate(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, int* status,
                                cudaStream_t st) {
  if (p.D == 64) return separate_d<64>(p, setting, in, dq, dk, status, st);
  return separate_d<128>(p, setting, in, dq, dk, status, st);
}

}  // namespace skl
