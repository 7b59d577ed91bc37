// Fused attention-KL backward on the 5th-generation tensor cores.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "kernel fusion": each (query tile, key tile) pair is visited exactly once; dK
// accumulates along the queries inside the block and dQ, which accumulates
// along the keys, is added into an fp32 buffer with atomics -- the path the
// library takes while that buffer fits in L2.  Gradient formulas as in
// bwd_tc.cu (setting 1: dS2 = g (P2 - P1); setting 2: dS1 = g P1 (r - KL)).
//
// Block = one 128-key tile (stationary K1, K2 in smem; keys on the 128 TMEM
// lanes), streaming 64-query tiles Y:
//   S1^T = K1 Q1^T, S2^T = K2 Q2^T    SS, M = 128 keys, N = 64 queries (double-buffered in TMEM)
//   dS^T from S^T and the per-query LSE1, LSE2, g, KL of the tile
//   dK  += dS^T Q_opt                 TS: A = dS^T packed bf16 over S1^T's columns, B = Q_opt MN-major
//   dQp^T = K_opt^T dS                SS: A = K_opt read MN-major (M = D on lanes), B = dS^T in smem
//   dq_acc[q, d] += dQp^T[d, q]       one warp adds 32 consecutive d of one query row (128 B) per red
// TMEM: S^T buffer b at [128b, 128b + 128) (S1^T then S2^T, 64 columns each),
// dK at [256, 256 + D), dQp^T buffer b at [384 + 64b, 448 + 64b).
//   warp 12     TMA producer; its 32 lanes also stage the per-query values
//   warp 13     TMEM owner and MMA issuer (S(j) issued before dK/dQp of tile j-1)
//   warps 0-7   dS warps: thread = key row, group g = query columns [32g, 32g + 32)
//   warps 8-11  dQ warps: thread = column d of dQp^T, reduce-add into dq_acc
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BK = 128;  // keys per block (M of the S and dK MMAs)
constexpr int BQ = 64;   // queries per step
constexpr int STAGES = 3;
constexpr int DS_WARPS = 8;
constexpr int DQ_WARP0 = 8;
constexpr int PRODUCER_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr int THREADS = 14 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDK = 256, kColDQ = 384;

template <int D>
struct Smem {
  static constexpr int KT = BK * D * 2;   // one 128-key tile
  static constexpr int QT = BQ * D * 2;   // one 64-query tile (D/64 halves of 8 KiB)
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = KT;
  static constexpr int OFF_Q = 2 * KT;  // stage s: Q1, Q2
  static constexpr int STAGE = 2 * QT;
  static constexpr int OFF_DS = OFF_Q + STAGES * STAGE;  // [2][128 keys][64 queries] bf16, 16 KiB each
  static constexpr int DS_BYTES = BK * BQ * 2;
  static constexpr int OFF_VALS = OFF_DS + 2 * DS_BYTES;  // [STAGES][4][64] fp32
  static constexpr int OFF_BAR = OFF_VALS + STAGES * 4 * BQ * 4;
  // k_full, y_full[3], y_empty[3], s_full[2], s_free[2], ds_full[2], ds_free[2], dq_full[2], dq_free[2], slot, abort
  static constexpr int BYTES = OFF_BAR + 8 * 19 + 16 + 1024;
};

// Per-query values staged for a tile, three arrays of BQ floats, folded so the
// element loop needs one packed FMA per logit:
//   nA = -LSE1 log2(e)
//   nB = -LSE2 log2(e)                    (setting 1)
//        -(LSE1 - LSE2 + KL)              (setting 2; the log ratio minus KL is then
//                                          scale (S1 - S2) + nB, from logits and LSEs)
//   G  = g
template <int SETTING, bool MASKED>
__device__ __forceinline__ void make_dst(const uint32_t (&a)[32], const uint32_t (&b)[32], uint32_t (&pk)[16],
                                         float c, float scale, const float* vals, int key, int q0, int nq, int nk,
                                         int off, int causal) {
  // thread = one key; 32 query columns q0 .. q0 + 31 with their values in vals[*][0..31]
  const float2 cc = make_float2(c, c), sc = make_float2(scale, scale);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 nA4 = *reinterpret_cast<const float4*>(vals + i);
    const float4 nB4 = *reinterpret_cast<const float4*>(vals + BQ + i);
    const float4 G4 = *reinterpret_cast<const float4*>(vals + 2 * BQ + i);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int k = i + 2 * h;
      const float2 nA = h ? make_float2(nA4.z, nA4.w) : make_float2(nA4.x, nA4.y);
      const float2 nB = h ? make_float2(nB4.z, nB4.w) : make_float2(nB4.x, nB4.y);
      const float2 G = h ? make_float2(G4.z, G4.w) : make_float2(G4.x, G4.y);
      const float2 s1 = make_float2(__uint_as_float(a[k]), __uint_as_float(a[k + 1]));
      const float2 s2 = make_float2(__uint_as_float(b[k]), __uint_as_float(b[k + 1]));
      const float2 x1 = ffma2(s1, cc, nA);
      float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
      bool k0 = true, k1 = true;
      if (MASKED) {
        const int q = q0 + k;
        k0 = q < nq && key < nk && (!causal || key <= q + off);
        k1 = q + 1 < nq && key < nk && (!causal || key <= q + 1 + off);
        p1.x = k0 ? p1.x : 0.f;
        p1.y = k1 ? p1.y : 0.f;
      }
      float2 ds;
      if (SETTING == 1) {
        const float2 x2 = ffma2(s2, cc, nB);
        float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
        if (MASKED) {
          p2.x = k0 ? p2.x : 0.f;
          p2.y = k1 ? p2.y : 0.f;
        }
        ds = fmul2(G, fsub2(p2, p1));
      } else {
        ds = fmul2(fmul2(G, p1), ffma2(sc, fsub2(s1, s2), nB));
      }
      pk[k / 2] = pack_bf16(ds.x, ds.y);
    }
  }
}

template <int D, int SETTING>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_fused_tc_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                        const float* __restrict__ klv, const float* __restrict__ gv,
                        __nv_bfloat16* __restrict__ dk_out, float* __restrict__ dq_acc, int* status,
                        const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mk2,
                        const __grid_constant__ CUtensorMap mq1, const __grid_constant__ CUtensorMap mq2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kt = (p.NK + BK - 1) / BK;
  const int bh = (int)(blockIdx.x / n_kt);  // heads in order (their dq_acc rows stay in L2), ...
  const int kt = (int)(blockIdx.x % n_kt);  // ... and within a head the longest (first) key tiles first
  const int k0 = kt * BK;
  const int q_begin = p.causal ? max(0, k0 - p.off) / BQ * BQ : 0;
  const int n_yt = (p.NQ - q_begin + BQ - 1) / BQ;

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t k_full = bar, y_full = bar + 8, y_empty = bar + 32, s_full = bar + 56, s_free = bar + 72,
                 ds_full = bar + 88, ds_free = bar + 104, dq_full = bar + 120, dq_free = bar + 136,
                 slot = bar + 152;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 156);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(y_full + 8 * s, 32);
      mbar_init(y_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + 8 * b, 1);
      mbar_init(s_free + 8 * b, DS_WARPS);
      mbar_init(ds_full + 8 * b, DS_WARPS);
      mbar_init(ds_free + 8 * b, 1);
      mbar_init(dq_full + 8 * b, 1);
      mbar_init(dq_free + 8 * b, 4);
    }
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
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_BAR + 152);

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(k_full, 2 * L::KT);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(sb + L::OFF_K1 + h * BK * 128, &mk1, k_full, h * 64, k0, bh);
        tma_load_3d(sb + L::OFF_K2 + h * BK * 128, &mk2, k_full, h * 64, k0, bh);
      }
    }
    int issued = 0;
    for (int j = 0; j < n_yt; ++j) {
      const int s = j % STAGES;
      const bool free_ok = j < STAGES || mbar_wait(y_empty + 8 * s, ((j / STAGES) - 1) & 1, status, abort_flag);
      __syncwarp();
      if (!free_ok) break;
      const int q0 = q_begin + j * BQ;
      const uint32_t qb = sb + L::OFF_Q + s * L::STAGE;
      if (lane == 0) {
        mbar_expect_tx(y_full + 8 * s, 2 * L::QT);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(qb + h * BQ * 128, &mq1, y_full + 8 * s, h * 64, q0, bh);
          tma_load_3d(qb + L::QT + h * BQ * 128, &mq2, y_full + 8 * s, h * 64, q0, bh);
        }
      }
      float* vals = reinterpret_cast<float*>(smem + L::OFF_VALS + s * 4 * BQ * 4);
#pragma unroll
      for (int k = 0; k < BQ / 32; ++k) {
        const int qi = lane + 32 * k, q = q0 + qi;
        const bool in = q < p.NQ;
        const size_t o = (size_t)bh * p.NQ + q;
        const float l1v = in ? lse1[o] : 0.f, l2v = in ? lse2[o] : 0.f;
        vals[qi] = -l1v * kLog2e;
        vals[BQ + qi] = SETTING == 1 ? -l2v * kLog2e : -(l1v - l2v + (in ? klv[o] : 0.f));
        vals[2 * BQ + qi] = in ? gv[o] : 0.f;
      }
      mbar_arrive(y_full + 8 * s);
      issued = j + 1;
    }
    if (lane == 0) {
      mbar_drain(k_full, 0, status);
      for (int j = max(0, issued - STAGES); j < issued; ++j)
        mbar_drain(y_full + 8 * (j % STAGES), (j / STAGES) & 1, status);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(BK, BQ, false, false);
      constexpr uint32_t id_dk = idesc_bf16(BK, D, false, true);
      constexpr uint32_t id_dq = idesc_bf16(128, BQ, true, true);
      const uint32_t kopt = sb + (SETTING == 1 ? L::OFF_K2 : L::OFF_K1);
      const uint64_t k1d = sdesc_sw128(sb + L::OFF_K1, 0, 1024), k2d = sdesc_sw128(sb + L::OFF_K2, 0, 1024);
      const uint64_t kod = sdesc_sw128(kopt, D == 128 ? BK * 128 : 0, 1024);
      bool ok = mbar_wait(k_full, 0, status, abort_flag);
      for (int j = 0; ok && j <= n_yt; ++j) {
        if (j < n_yt) {
          const int s = j % STAGES, b = j & 1;
          if (!mbar_wait(y_full + 8 * s, (j / STAGES) & 1, status, abort_flag)) break;
          if (j >= 2 && !mbar_wait(s_free + 8 * b, ((j >> 1) - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          const uint32_t q1 = sb + L::OFF_Q + s * L::STAGE, q2 = q1 + L::QT;
          const uint64_t q1d = sdesc_sw128(q1, 0, 1024), q2d = sdesc_sw128(q2, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t ka = (ks >> 2) * (BK * 128) + (ks & 3) * 32;  // 128-key tile halves
            const uint32_t qa = (ks >> 2) * (BQ * 128) + (ks & 3) * 32;  // 64-query tile halves
            mma_ss(tmem + 128 * b, sdesc_add(k1d, ka), sdesc_add(q1d, qa), id_s, ks > 0);
          }
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t ka = (ks >> 2) * (BK * 128) + (ks & 3) * 32;
            const uint32_t qa = (ks >> 2) * (BQ * 128) + (ks & 3) * 32;
            mma_ss(tmem + 128 * b + 64, sdesc_add(k2d, ka), sdesc_add(q2d, qa), id_s, ks > 0);
          }
          mma_commit(s_full + 8 * b);
        }
        if (j >= 1) {
          const int jj = j - 1, b = jj & 1, s = jj % STAGES;
          if (!mbar_wait(ds_full + 8 * b, (jj >> 1) & 1, status, abort_flag)) break;
          if (jj >= 2 && !mbar_wait(dq_free + 8 * b, ((jj >> 1) - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          // dK += dS^T Q_opt: A = packed dS^T in TMEM (query k-steps 0,1 at columns 128b + 0.., 2,3 at 128b + 32..)
          const uint64_t qod = sdesc_sw128(sb + L::OFF_Q + s * L::STAGE + (SETTING == 1 ? L::QT : 0), BQ * 128, 1024);
#pragma unroll
          for (int ks = 0; ks < BQ / 16; ++ks)
            mma_ts(tmem + kColDK, tmem + 128 * b + (ks >> 1) * 32 + (ks & 1) * 8, sdesc_add(qod, ks * 2048), id_dk,
                   jj > 0 || ks > 0);
          // dQp^T = K_opt^T dS: A = K_opt (keys x d) read MN-major, B = dS^T (keys x queries) MN-major
          const uint64_t dsd = sdesc_sw128(sb + L::OFF_DS + b * L::DS_BYTES, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            mma_ss(tmem + kColDQ + 64 * b, sdesc_add(kod, ks * 2048), sdesc_add(dsd, ks * 2048), id_dq, ks > 0);
          mma_commit(y_empty + 8 * s);
          mma_commit(ds_free + 8 * b);
          mma_commit(dq_full + 8 * b);
        }
      }
      // all MMAs done (the last dq_full commit covers every earlier MMA)
      if (n_yt > 0) mbar_drain(dq_full + 8 * ((n_yt - 1) & 1), ((n_yt - 1) >> 1) & 1, status);
    }
    __syncwarp();
  } else if (warp < DS_WARPS) {
    // ------------------------------------------------------------------ dS warps
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int key = k0 + r;
    const float c = p.c;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    for (int j = 0; j < n_yt; ++j) {
      const int b = j & 1, s = j % STAGES;
      bool got = mbar_wait(s_full + 8 * b, (j >> 1) & 1, status, abort_flag);
      __syncwarp();
      if (!got) break;
      tc_fence_after();
      // the per-query values were staged by the producer lanes: acquire them directly
      got = mbar_wait(y_full + 8 * s, (j / STAGES) & 1, status, abort_flag);
      __syncwarp();
      if (!got) break;
      uint32_t a[32], bb[32];
      const uint32_t ta = tmem + lane_base + 128 * b + grp * 32;
      tmem_ld32(ta, a);
      tmem_ld32(ta + 64, bb);
      tmem_ld_wait();
      reg_fence32(a);
      reg_fence32(bb);
      const int q0 = q_begin + j * BQ + grp * 32;
      const float* vals = reinterpret_cast<const float*>(smem + L::OFF_VALS + s * 4 * BQ * 4) + grp * 32;
      const bool masked = (q0 + 31 >= p.NQ) || (key >= p.NK) || (p.causal && key > q0 + p.off);
      uint32_t pk[16];
      if (masked)
        make_dst<SETTING, true>(a, bb, pk, c, p.scale, vals, key, q0, p.NQ, p.NK, p.off, p.causal);
      else
        make_dst<SETTING, false>(a, bb, pk, c, p.scale, vals, key, q0, p.NQ, p.NK, p.off, p.causal);
      // the smem copy of dS^T (B of the dQ MMA) is free once the dQ MMA of tile j-2 is done
      if (j >= 2) {
        got = mbar_wait(ds_free + 8 * b, ((j >> 1) - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!got) break;
      }
      const uint32_t dsb = sb + L::OFF_DS + b * L::DS_BYTES;
#pragma unroll
      for (int cch = 0; cch < 4; ++cch) {
        const uint32_t dst = sw128<BK>(dsb, r, grp * 4 + cch);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk[4 * cch]), "r"(pk[4 * cch + 1]),
                     "r"(pk[4 * cch + 2]), "r"(pk[4 * cch + 3])
                     : "memory");
      }
      fence_async_smem();
      // packed dS^T over this group's first 16 S1^T columns (already read): A of the dK MMA
      tmem_st16(tmem + lane_base + 128 * b + grp * 32, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(s_free + 8 * b);
        mbar_arrive(ds_full + 8 * b);
      }
    }
    // ---- dK out
    constexpr int HALF = D / 2;
    bool got = mbar_wait(dq_full + 8 * ((n_yt - 1) & 1), ((n_yt - 1) >> 1) & 1, status, abort_flag);
    __syncwarp();
    if (got) {
      tc_fence_after();
      uint32_t g0[32], g1[32];
      const uint32_t tg = tmem + lane_base + kColDK + grp * HALF;
      tmem_ld32(tg, g0);
      if (HALF == 64) tmem_ld32(tg + 32, g1);
      tmem_ld_wait();
      reg_fence32(g0);
      reg_fence32(g1);
      if (key < p.NK) {
        __nv_bfloat16* dst = dk_out + ((size_t)bh * p.NK + key) * D + grp * HALF;
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
  } else {
    // ------------------------------------------------------------------ dQ warps
    const int wq = warp - DQ_WARP0;
    const int d = wq * 32 + lane;  // lane of dQp^T = column d
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    for (int j = 0; j < n_yt; ++j) {
      const int b = j & 1;
      const bool got = mbar_wait(dq_full + 8 * b, (j >> 1) & 1, status, abort_flag);
      __syncwarp();
      if (!got) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(tmem + lane_base + kColDQ + 64 * b, v0);
      tmem_ld32(tmem + lane_base + kColDQ + 64 * b + 32, v1);
      tmem_ld_wait();
      reg_fence32(v0);
      reg_fence32(v1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free + 8 * b);
      if (d < D) {
        const int q0 = q_begin + j * BQ;
        float* base = dq_acc + ((size_t)bh * p.NQ + q0) * D + d;
        const int nrow = min(BQ, p.NQ - q0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < nrow) red_add_f32(base + (size_t)i * D, __uint_as_float(v0[i]));
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (32 + i < nrow) red_add_f32(base + (size_t)(32 + i) * D, __uint_as_float(v1[i]));
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

template <int D, int SETTING>
cudaError_t launch_fused(const Problem& p, const BwdIn& in, void* dk, float* dq_acc, int* status, cudaStream_t st) {
  CUtensorMap mk1, mk2, mq1, mq2;
  if (!encode_tile_map(&mk1, in.k1, D, p.NK, p.BH, BK) || !encode_tile_map(&mk2, in.k2, D, p.NK, p.BH, BK) ||
      !encode_tile_map(&mq1, in.q1, D, p.NQ, p.BH, BQ) || !encode_tile_map(&mq2, in.q2, D, p.NQ, p.BH, BQ))
    return cudaErrorInvalidValue;
  const int smem = Smem<D>::BYTES > kOneBlockPerSmSmem ? Smem<D>::BYTES : kOneBlockPerSmSmem;
  auto kern = bwd_fused_tc_kernel<D, SETTING>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.BH * ((p.NK + BK - 1) / BK);
  kern<<<(unsigned)blocks, THREADS, smem, st>>>(p, in.lse1, in.lse2, in.kl, in.g, static_cast<__nv_bfloat16*>(dk),
                                                dq_acc, status, mk1, mk2, mq1, mq2);
  return cudaGetLastError();
}

// dQ (bf16) = scale * dQ accumulator (fp32); 8 elements per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ out,
                                                         size_t n8, float scale) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a.x * scale, a.y * scale);
    o.y = pack_bf16(a.z * scale, a.w * scale);
    o.z = pack_bf16(b.x * scale, b.y * scale);
    o.w = pack_bf16(b.z * scale, b.w * scale);
    out[i] = o;
  }
}

template <int D>
cudaError_t fused_d(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, float* dq_acc, int* status,
                    cudaStream_t st) {
  const size_t n = (size_t)p.BH * p.NQ * D;
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, n * sizeof(float), st);
  if (e != cudaSuccess) return e;
  e = setting == 1 ? launch_fused<D, 1>(p, in, dk, dq_acc, status, st)
                   : launch_fused<D, 2>(p, in, dk, dq_acc, status, st);
  if (e != cudaSuccess) return e;
  const size_t n8 = n / 8;
  const int blocks = (int)((n8 + 255) / 256 < 4096 ? (n8 + 255) / 256 : 4096);
  dq_convert_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(reinterpret_cast<const float4*>(dq_acc),
                                                             static_cast<uint4*>(dq), n8, p.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, float* dq_acc,
                             int* status, cudaStream_t st) {
  if (p.D == 64) return fused_d<64>(p, setting, in, dq, dk, dq_acc, status, st);
  return fused_d<128>(p, setting, in, dq, dk, dq_acc, status, st);
}

}  // namespace skl
