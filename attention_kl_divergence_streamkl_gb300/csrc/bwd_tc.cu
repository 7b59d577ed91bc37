// Recompute-based attention-KL backward on the 5th-generation tensor cores:
// the separate-path dQ and dK kernels.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "recompute strategy": only KL, LSE1, LSE2 are kept; the backward rebuilds
// P_t = exp(S_t - LSE_t) tile by tile.  Setting 1 (P1 fixed) optimises Q2/K2,
// setting 2 (P2 fixed) optimises Q1/K1; section 手法 3 "numerical stability":
// the setting-2 log ratio is taken from logits and the saved LSEs.  With
// L = sum_i g_i KL_i (chain rule, derived):
//     setting 1:  dS2 = g (P2 - P1)
//     setting 2:  dS1 = g P1 (r - KL),  r = (S1 - LSE1) - (S2 - LSE2)
//     dQ = scale dS K_opt,   dK = scale dS^T Q_opt.
//
// One kernel template serves both separate kernels.  A block owns a stationary
// tile X of 128 rows (query rows for dQ, keys for dK) on the 128 TMEM lanes and
// streams tiles Y of 128 rows of the other side:
//     S1 = X1 Y1^T, S2 = X2 Y2^T          (tcgen05, both operands K-major in smem)
//     dS from S1, S2 and the saved row values, packed to bf16 into TMEM
//     G += dS Y_opt                       (tcgen05, A = dS in TMEM, B = Y_opt
//                                          read MN-major from the same smem tile)
// so dS never leaves the SM.  TMEM (512 columns): S1 [0,128), S2 [128,256),
// dS double buffer [256,320) / [320,384) (bf16 pairs), G [384, 384 + D).
//   warp 8      TMA producer (and, for dK, the per-query LSE/g/KL values)
//   warp 9      TMEM owner and MMA issuer; issues S(j) before G += dS(j-1) so
//               the tensor pipe computes the next logits while dS is built
//   warps 0-7   two groups of 4 warps, thread = X row, group g takes columns
//               [64g, 64g + 64) of each Y tile; then they write G out.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BX = 128;  // stationary rows (MMA M)
constexpr int BY = 128;  // streamed rows per tile (MMA N of S, K of the gradient MMA)
constexpr int SOFTMAX_WARPS = 8;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 10 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS1 = 0, kColS2 = 128, kColDS = 256, kColG = 384;

template <int D>
struct Smem {
  static constexpr int TILE = 128 * D * 2;  // one 128-row bf16 tile, D/64 halves of 16 KiB
  static constexpr int OFF_X1 = 0;
  static constexpr int OFF_X2 = TILE;
  static constexpr int OFF_Y = 2 * TILE;  // stage s: Y1, Y2
  static constexpr int STAGE = 2 * TILE;
  static constexpr int OFF_VALS = OFF_Y + 2 * STAGE;  // [2 stages][4][128] fp32 (dK kernel)
  static constexpr int OFF_BAR = OFF_VALS + 2 * 4 * BY * 4;
  // x_full, y_full[2], y_empty[2], s_full, s_free, ds_full[2], ds_free[2], g_done, slot, abort
  static constexpr int BYTES = OFF_BAR + 8 * 12 + 16 + 1024;
};


// dS for one thread's 64 columns; values are packed as bf16 pairs into pk[32].
// KSTAT: X rows are keys and Y rows are queries (per-column row values).
// Arithmetic on column pairs uses the packed fp32 instructions.
template <int SETTING, bool KSTAT, bool MASKED>
__device__ __forceinline__ void make_ds(uint32_t (&a0)[32], uint32_t (&a1)[32], uint32_t (&b0)[32],
                                        uint32_t (&b1)[32], uint32_t (&pk)[32], float c, const float* vals,
                                        float L1r, float L2r, float Gr, float KLr, int xidx, int y0, int nx, int ny,
                                        int off, int causal) {
  const float2 cc = make_float2(c, c);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const int col = h * 32 + i;
      const uint32_t* A = h == 0 ? a0 : a1;
      const uint32_t* Bv = h == 0 ? b0 : b1;
      const float2 s1 = make_float2(__uint_as_float(A[i]), __uint_as_float(A[i + 1]));
      const float2 s2 = make_float2(__uint_as_float(Bv[i]), __uint_as_float(Bv[i + 1]));
      float2 L1 = make_float2(L1r, L1r), L2 = make_float2(L2r, L2r), G = make_float2(Gr, Gr);
      float2 KL = make_float2(KLr, KLr);
      if (KSTAT) {
        L1 = *reinterpret_cast<const float2*>(vals + col);
        L2 = *reinterpret_cast<const float2*>(vals + BY + col);
        G = *reinterpret_cast<const float2*>(vals + 2 * BY + col);
        if (SETTING == 2) KL = *reinterpret_cast<const float2*>(vals + 3 * BY + col);
      }
      const float2 x1 = ffma2(s1, cc, make_float2(-L1.x, -L1.y));
      float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
      if (MASKED) {
        const int y = y0 + col;  // streamed index: key (dQ kernel) or query (dK kernel)
        bool keep[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = KSTAT ? y + e : xidx, k = KSTAT ? xidx : y + e;
          const int nq = KSTAT ? ny : nx, nk = KSTAT ? nx : ny;
          keep[e] = q < nq && k < nk && (!causal || k <= q + off);
        }
        p1.x = keep[0] ? p1.x : 0.f;
        p1.y = keep[1] ? p1.y : 0.f;
        if (SETTING == 1) {
          const float2 x2 = ffma2(s2, cc, make_float2(-L2.x, -L2.y));
          const float2 p2 = make_float2(keep[0] ? ex2(x2.x) : 0.f, keep[1] ? ex2(x2.y) : 0.f);
          const float2 ds = fmul2(G, fsub2(p2, p1));
          pk[col / 2] = pack_bf16(ds.x, ds.y);
          continue;
        }
      } else if (SETTING == 1) {
        const float2 x2 = ffma2(s2, cc, make_float2(-L2.x, -L2.y));
        const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
        const float2 ds = fmul2(G, fsub2(p2, p1));
        pk[col / 2] = pack_bf16(ds.x, ds.y);
        continue;
      }
      if (SETTING == 2) {
        // r = ln2 ((s1 - s2) c - (L1 - L2));  dS1 = g p1 (r - KL)
        const float2 r = fmul2(make_float2(kLn2, kLn2), ffma2(fsub2(s1, s2), cc, fsub2(L2, L1)));
        const float2 ds = fmul2(fmul2(G, p1), fsub2(r, KL));
        pk[col / 2] = pack_bf16(ds.x, ds.y);
      }
    }
  }
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
  const uint32_t x_full = bar, y_full = bar + 8, y_empty = bar + 24, s_full = bar + 40, s_free = bar + 48,
                 ds_full = bar + 56, ds_free = bar + 72, g_done = bar + 88, slot = bar + 96;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 100);

  if (threadIdx.x == 0) {
    mbar_init(x_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(y_full + 8 * s, KSTAT ? 32 : 1);
      mbar_init(y_empty + 8 * s, 1);
      mbar_init(ds_full + 8 * s, SOFTMAX_WARPS);
      mbar_init(ds_free + 8 * s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, SOFTMAX_WARPS);
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
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_BAR + 96);

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(x_full, 2 * L::TILE);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(sb + L::OFF_X1 + h * BX * 128, &mx1, x_full, h * 64, x0, bh);
        tma_load_3d(sb + L::OFF_X2 + h * BX * 128, &mx2, x_full, h * 64, x0, bh);
      }
    }
    int issued = 0;
    for (int j = 0; j < n_yt; ++j) {
      const int s = j & 1;
      const bool free_ok = j < 2 || mbar_wait(y_empty + 8 * s, ((j >> 1) - 1) & 1, status, abort_flag);
      __syncwarp();
      if (!free_ok) break;
      const int y0 = (y_first + j) * BY;
      const uint32_t yb = sb + L::OFF_Y + s * L::STAGE;
      if (lane == 0) {
        if (KSTAT) mbar_expect_tx(y_full + 8 * s, 2 * L::TILE);
        else mbar_arrive_expect_tx(y_full + 8 * s, 2 * L::TILE);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(yb + h * BY * 128, &my1, y_full + 8 * s, h * 64, y0, bh);
          tma_load_3d(yb + L::TILE + h * BY * 128, &my2, y_full + 8 * s, h * 64, y0, bh);
        }
      }
      if (KSTAT) {
        // per-query values of this tile, log2 units for the LSEs
        float* vals = reinterpret_cast<float*>(smem + L::OFF_VALS + s * 4 * BY * 4);
#pragma unroll
        for (int k = 0; k < BY / 32; ++k) {
          const int qi = lane + 32 * k, q = y0 + qi;
          const bool in = q < p.NQ;
          const size_t o = (size_t)bh * p.NQ + q;
          vals[qi] = in ? lse1[o] * kLog2e : 0.f;
          vals[BY + qi] = in ? lse2[o] * kLog2e : 0.f;
          vals[2 * BY + qi] = in ? gv[o] : 0.f;
          vals[3 * BY + qi] = (SETTING == 2 && in) ? klv[o] : 0.f;
        }
        mbar_arrive(y_full + 8 * s);
      }
      issued = j + 1;
    }
    if (lane == 0) {
      mbar_drain(x_full, 0, status);
      for (int j = max(0, issued - 2); j < issued; ++j) mbar_drain(y_full + 8 * (j & 1), (j >> 1) & 1, status);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(BX, BY, false, false);
      constexpr uint32_t id_g = idesc_bf16(BX, D, false, true);
      bool ok = mbar_wait(x_full, 0, status, abort_flag);
      for (int j = 0; ok && j <= n_yt; ++j) {
        if (j < n_yt) {
          const int s = j & 1;
          if (!mbar_wait(y_full + 8 * s, (j >> 1) & 1, status, abort_flag)) break;
          if (j >= 1 && !mbar_wait(s_free, (j - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          const uint32_t y1 = sb + L::OFF_Y + s * L::STAGE, y2 = y1 + L::TILE;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
            mma_ss(tmem + kColS1, sdesc_sw128(sb + L::OFF_X1 + off, 0, 1024), sdesc_sw128(y1 + off, 0, 1024), id_s,
                   ks > 0);
          }
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
            mma_ss(tmem + kColS2, sdesc_sw128(sb + L::OFF_X2 + off, 0, 1024), sdesc_sw128(y2 + off, 0, 1024), id_s,
                   ks > 0);
          }
          mma_commit(s_full);
        }
        if (j >= 1) {
          const int jj = j - 1, b = jj & 1;
          if (!mbar_wait(ds_full + 8 * b, (jj >> 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          // B = Y_opt read MN-major: N = D along the 128-byte rows, K = Y rows
          const uint32_t yopt = sb + L::OFF_Y + b * L::STAGE + (SETTING == 1 ? L::TILE : 0);
#pragma unroll
          for (int ks = 0; ks < BY / 16; ++ks)
            mma_ts(tmem + kColG, tmem + kColDS + 64 * b + 8 * ks, sdesc_sw128(yopt + ks * 2048, BY * 128, 1024), id_g,
                   jj > 0 || ks > 0);
          mma_commit(y_empty + 8 * b);
          mma_commit(ds_free + 8 * b);
        }
      }
      mma_commit(g_done);
      mbar_drain(g_done, 0, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dS warps
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int xidx = x0 + r;
    const float c = p.c;
    float L1r = 0.f, L2r = 0.f, Gr = 0.f, KLr = 0.f;
    if (!KSTAT && xidx < p.NQ) {
      const size_t o = (size_t)bh * p.NQ + xidx;
      L1r = lse1[o] * kLog2e;
      L2r = lse2[o] * kLog2e;
      Gr = gv[o];
      if (SETTING == 2) KLr = klv[o];
    }
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    for (int j = 0; j < n_yt; ++j) {
      const int b = j & 1;
      bool got = mbar_wait(s_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t a0[32], a1[32], b0[32], b1[32];
      const uint32_t ta = tmem + lane_base + grp * 64;
      tmem_ld32(ta + kColS1, a0);
      tmem_ld32(ta + kColS1 + 32, a1);
      tmem_ld32(ta + kColS2, b0);
      tmem_ld32(ta + kColS2 + 32, b1);
      tmem_ld_wait();
      reg_fence32(a0);
      reg_fence32(a1);
      reg_fence32(b0);
      reg_fence32(b1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);

      const int y0 = (y_first + j) * BY;
      const float* vals = reinterpret_cast<const float*>(smem + L::OFF_VALS + b * 4 * BY * 4) + grp * 64;
      const int ylo = y0 + grp * 64;
      bool masked;
      if (KSTAT)  // query columns ylo.., key row xidx
        masked = (ylo + 63 >= p.NQ) || (xidx >= p.NK) || (p.causal && xidx > ylo + p.off);
      else  // key columns ylo.., query row xidx
        masked = (ylo + 63 >= p.NK) || (p.causal && ylo + 63 > xidx + p.off);
      uint32_t pk[32];
      if (masked)
        make_ds<SETTING, KSTAT, true>(a0, a1, b0, b1, pk, c, vals, L1r, L2r, Gr, KLr, xidx, ylo, NX, NY, p.off,
                                      p.causal);
      else
        make_ds<SETTING, KSTAT, false>(a0, a1, b0, b1, pk, c, vals, L1r, L2r, Gr, KLr, xidx, ylo, NX, NY, p.off,
                                       p.causal);
      if (j >= 2) {
        got = mbar_wait(ds_free + 8 * b, ((j >> 1) - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!got) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      tmem_st32(tmem + lane_base + kColDS + 64 * b + grp * 32, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full + 8 * b);
    }
    // ---- G = sum dS Y_opt, scaled, to bf16
    bool got = ok && mbar_wait(g_done, 0, status, abort_flag);
    __syncwarp();
    if (got) {
      tc_fence_after();
      constexpr int HALF = D / 2;  // columns of G this group writes
      uint32_t g0[32], g1[32];
      const uint32_t tg = tmem + lane_base + kColG + grp * HALF;
      tmem_ld32(tg, g0);
      if (HALF == 64) tmem_ld32(tg + 32, g1);
      tmem_ld_wait();
      reg_fence32(g0);
      reg_fence32(g1);
      if (xidx < NX) {
        __nv_bfloat16* dst = out + ((size_t)bh * NX + xidx) * D + grp * HALF;
#pragma unroll
        for (int v = 0; v < HALF / 8; ++v) {
          uint4 o;
          const uint32_t* src = v < 4 ? &g0[v * 8] : &g1[(v - 4) * 8];
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
