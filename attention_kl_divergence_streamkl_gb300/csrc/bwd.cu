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
// lanes), streaming 128-query tiles Y.  Every MMA is M = 128, N = 128: on this
// GPU a single-CTA M = 128 MMA costs the same for any N up to 128, so narrower
// tiles only waste the tensor core.
//   S1^T = K1 Q1^T, S2^T = K2 Q2^T    SS, K-major, into TMEM columns [0, 128) and [128, 256)
//   dS^T from S^T and the per-query LSE1, LSE2, g, KL of the tile, written to smem as dS[key][query]
//   dK  += dS^T Q_opt                 SS: A = dS (K-major over queries), B = Q_opt MN-major  -> [256, 256 + D)
//   dQp^T = K_opt^T dS                SS: A = K_opt read MN-major (M = d), B = dS MN-major   -> [384, 512)
//   dq_acc[q, d] += dQp^T[d, q]       one warp adds 32 consecutive d of one query row (128 B) per red
// TMEM holds one S tile, so the dS warps copy their part of S^T into registers
// first and release it: S of the next tile is computed while they work.  The
// same warps drain the previous tile's dQp^T (a 32 x 32 block each) before they
// publish dS, so one barrier tells the MMA issuer that both dS and the dQp^T
// columns are ready.
//   warps 0-15  dS warps: thread = key row (lane quarter = warp % 4), group g = warp / 4
//               takes query columns [32g, 32g + 32); for dQp^T, thread = column d
//   warp 16     TMA producer (K1, K2 once; Q1, Q2 through two stages)
//   warp 17     TMEM owner and MMA issuer (S(j) issued before dK/dQp of tile j-1)
//   warp 18     stages the per-query values of each tile in smem
// Warpgroup 4 gives registers to the dS warpgroups (setmaxnreg).
#include <utility>

#include "common.cuh"
#include "ds_math.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BK = 128;  // keys per block (M of the S and dK MMAs)
constexpr int BQ = 128;  // queries per step (N of the S and dQp MMAs)
constexpr int STAGES = 2;
constexpr int DS_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int VALS_WARP = 18;
constexpr int THREADS = 20 * 32;
constexpr int kRegsDs = 104, kRegsOther = 64;  // 512 * 104 + 128 * 64 = 640 * 96 registers at launch
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS1 = 0, kColS2 = 128, kColDK = 256, kColDQ = 384;

template <int D>
struct Smem {
  static constexpr int KT = BK * D * 2;  // one 128-key tile (D/64 halves of [128][128 B])
  static constexpr int QT = BQ * D * 2;  // one 128-query tile
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = KT;
  static constexpr int OFF_Q = 2 * KT;  // stage s: Q1, Q2
  static constexpr int STAGE = 2 * QT;
  static constexpr int OFF_DS = OFF_Q + STAGES * STAGE;  // dS[key][query] bf16: 2 halves of [128 keys][128 B]
  static constexpr int DS_BYTES = BK * BQ * 2;
  static constexpr int OFF_VALS = OFF_DS + DS_BYTES;  // [3][BQ] fp32, one tile
  static constexpr int OFF_BAR = OFF_VALS + 3 * BQ * 4;
  // mbarriers (8 B each): k_full, y_full[STAGES], y_empty[STAGES], s_full, s_free, v_full, v_free,
  // ds_full, ds_free, all_done; then the TMEM base address slot and the abort flag
  static constexpr int BAR_Y_FULL = 8, BAR_Y_EMPTY = BAR_Y_FULL + 8 * STAGES, BAR_ONE = BAR_Y_EMPTY + 8 * STAGES;
  static constexpr int BAR_SLOT = BAR_ONE + 7 * 8;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ void setmaxnreg_inc_ds() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
}
__device__ __forceinline__ void setmaxnreg_dec_other() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

// red.global.add.f32 at base + OFF bytes: the offset rides in the instruction,
// so a row loop keeps one 64-bit address live instead of one per row.
template <int OFF>
__device__ __forceinline__ void red_add_at(float* base, float a) {
  asm volatile("red.global.add.f32 [%0+%2], %1;" ::"l"(base), "f"(a), "n"(OFF) : "memory");
}
// base[i * D] += v[i] for the rows i < nrow of a 32-row block
template <int D, int... I>
__device__ __forceinline__ void red_rows(float* base, const uint32_t (&v)[32], int nrow,
                                         std::integer_sequence<int, I...>) {
  ((I < nrow ? red_add_at<I * D * 4>(base, __uint_as_float(v[I])) : void()), ...);
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
  const uint32_t k_full = bar, y_full = bar + L::BAR_Y_FULL, y_empty = bar + L::BAR_Y_EMPTY,
                 s_full = bar + L::BAR_ONE, s_free = s_full + 8, v_full = s_full + 16, v_free = s_full + 24,
                 ds_full = s_full + 32, ds_free = s_full + 40, all_done = s_full + 48, slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);
  float* vals = reinterpret_cast<float*>(smem + L::OFF_VALS);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(y_full + 8 * s, 1);
      mbar_init(y_empty + 8 * s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, DS_WARPS);
    mbar_init(v_full, 1);
    mbar_init(v_free, DS_WARPS);
    mbar_init(ds_full, DS_WARPS);
    mbar_init(ds_free, 1);
    mbar_init(all_done, 1);
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
        mbar_arrive_expect_tx(k_full, 2 * L::KT);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(sb + L::OFF_K1 + h * BK * 128, &mk1, k_full, h * 64, k0, bh);
          tma_load_3d(sb + L::OFF_K2 + h * BK * 128, &mk2, k_full, h * 64, k0, bh);
        }
        int issued = 0;
        for (int j = 0; j < n_yt; ++j) {
          const int s = j % STAGES;
          if (j >= STAGES && !mbar_wait(y_empty + 8 * s, ((j / STAGES) - 1) & 1, status, abort_flag)) break;
          const int q0 = q_begin + j * BQ;
          const uint32_t qb = sb + L::OFF_Q + s * L::STAGE;
          mbar_arrive_expect_tx(y_full + 8 * s, 2 * L::QT);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_3d(qb + h * BQ * 128, &mq1, y_full + 8 * s, h * 64, q0, bh);
            tma_load_3d(qb + L::QT + h * BQ * 128, &mq2, y_full + 8 * s, h * 64, q0, bh);
          }
          issued = j + 1;
        }
        mbar_drain(k_full, 0, status);
        for (int j = max(0, issued - STAGES); j < issued; ++j)
          mbar_drain(y_full + 8 * (j % STAGES), (j / STAGES) & 1, status);
      }
      __syncwarp();
    } else if (warp == VALS_WARP) {
      // ------------------------------------------------------------------ per-query values
      // Loads for tile j are issued before waiting for the dS warps to release the
      // previous tile's values, so their latency overlaps that wait.
      constexpr int PER = BQ / 32;
      float a[PER], b[PER], g[PER];
      auto fetch = [&](int j) {
        const int q0 = q_begin + j * BQ;
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
          vals[BQ + lane + 32 * k] = b[k];
          vals[2 * BQ + lane + 32 * k] = g[k];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(v_full);
        if (j + 1 < n_yt) fetch(j + 1);
      }
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16(BK, BQ, false, false);
        constexpr uint32_t id_dk = idesc_bf16(BK, D, false, true);
        constexpr uint32_t id_dq = idesc_bf16(128, BQ, true, true);
        constexpr uint32_t HI = sdesc_sw128_hi(1024);  // every operand: 8-row atoms 1024 B apart
        // low descriptor words; K-major operands have no leading offset, MN-major ones
        // step 64 elements along M/N by one 128-row tile half
        const uint32_t k1l = sdesc_sw128_lo(sb + L::OFF_K1, 0), k2l = sdesc_sw128_lo(sb + L::OFF_K2, 0);
        const uint32_t kol = sdesc_sw128_lo(sb + (SETTING == 1 ? L::OFF_K2 : L::OFF_K1), D == 128 ? BK * 128 : 0);
        const uint32_t dskl = sdesc_sw128_lo(sb + L::OFF_DS, 0);         // dS as A of dK (K-major over queries)
        const uint32_t dsml = sdesc_sw128_lo(sb + L::OFF_DS, BK * 128);  // dS as B of dQp (MN-major over queries)
        bool ok = mbar_wait(k_full, 0, status, abort_flag);
        for (int j = 0; ok && j <= n_yt; ++j) {
          if (j < n_yt) {
            const int s = j % STAGES;
            if (!mbar_wait(y_full + 8 * s, (j / STAGES) & 1, status, abort_flag)) break;
            if (j >= 1 && !mbar_wait(s_free, (j - 1) & 1, status, abort_flag)) break;
            tc_fence_after();
            const uint32_t q1l = sdesc_sw128_lo(sb + L::OFF_Q + s * L::STAGE, 0), q2l = q1l + (L::QT >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t ka = ((ks >> 2) * (BK * 128) + (ks & 3) * 32) >> 4;  // 128-key tile halves
              const uint32_t qa = ((ks >> 2) * (BQ * 128) + (ks & 3) * 32) >> 4;  // 128-query tile halves
              mma_ss_lohi(tmem + kColS1, k1l + ka, HI, q1l + qa, HI, id_s, ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t ka = ((ks >> 2) * (BK * 128) + (ks & 3) * 32) >> 4;
              const uint32_t qa = ((ks >> 2) * (BQ * 128) + (ks & 3) * 32) >> 4;
              mma_ss_lohi(tmem + kColS2, k2l + ka, HI, q2l + qa, HI, id_s, ks > 0);
            }
            mma_commit(s_full);
          }
          if (j >= 1) {
            const int jj = j - 1, s = jj % STAGES;
            // dS(jj) in smem, and dQp^T of tile jj - 1 drained from TMEM
            if (!mbar_wait(ds_full, jj & 1, status, abort_flag)) break;
            tc_fence_after();
            // dK += dS^T Q_opt: A = dS[key][query] K-major (query k-steps), B = Q_opt read MN-major
            const uint32_t qol =
                sdesc_sw128_lo(sb + L::OFF_Q + s * L::STAGE + (SETTING == 1 ? L::QT : 0), BQ * 128);
#pragma unroll
            for (int ks = 0; ks < BQ / 16; ++ks)
              mma_ss_lohi(tmem + kColDK, dskl + (((ks >> 2) * (BK * 128) + (ks & 3) * 32) >> 4), HI,
                          qol + ks * (2048 >> 4), HI, id_dk, jj > 0 || ks > 0);
            // dQp^T = K_opt^T dS: A = K_opt (keys x d) read MN-major, B = dS (keys x queries) MN-major
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              mma_ss_lohi(tmem + kColDQ, kol + ks * (2048 >> 4), HI, dsml + ks * (2048 >> 4), HI, id_dq, ks > 0);
            mma_commit(y_empty + 8 * s);
            mma_commit(ds_free);
          }
        }
        // every MMA done: arrives on all_done (waited by the dK epilogue and below)
        mma_commit(all_done);
        mbar_drain(all_done, 0, status);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc_ds();
    // ------------------------------------------------------------------ dS warps
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int key = k0 + r;
    const int d = r;  // as the reader of dQp^T, lane r holds column d = r
    const float c = p.c;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t dsb = sb + L::OFF_DS;
    // dq_acc[q, d] += dQp^T[d, q] for this warp's 32 queries [32 grp, 32 grp + 32) of tile jt
    auto add_dq = [&](int jt, const uint32_t(&v)[32]) {
      const int q0 = q_begin + jt * BQ + grp * 32;
      if (d < D) {
        float* base = dq_acc + ((size_t)bh * p.NQ + q0) * D + d;
        red_rows<D>(base, v, min(32, p.NQ - q0), std::make_integer_sequence<int, 32>{});
      }
    };
    for (int j = 0; j < n_yt; ++j) {
      bool got = mbar_wait(s_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!got) break;
      tc_fence_after();
      const int q0 = q_begin + j * BQ + grp * 32;
      const bool masked = (q0 + 31 >= p.NQ) || (key >= p.NK) || (p.causal && key > q0 + p.off);
      uint32_t pk[16];
      // Two halves of 16 query columns: the second half is read after the first
      // is computed, and TMEM is released once both are in registers.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[16], bb[16];
        tmem_ld16(tmem + lane_base + kColS1 + grp * 32 + 16 * h, a);
        tmem_ld16(tmem + lane_base + kColS2 + grp * 32 + 16 * h, bb);
        tmem_ld_wait();
        reg_fence16(a);
        reg_fence16(bb);
        if (h == 1) {
          // S of this tile is in registers: the next tile's S MMA may overwrite TMEM
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
        } else {
          got = mbar_wait(v_full, j & 1, status, abort_flag);
          __syncwarp();
          if (!got) break;
        }
        const float* vh = vals + grp * 32 + 16 * h;
        if (masked)
          make_ds_cols<SETTING, true, 16, BQ>(a, bb, pk + 8 * h, c, p.scale, vh,
                                              visible_queries<16>(key, q0 + 16 * h, p.NQ, p.NK, p.off, p.causal));
        else
          make_ds_cols<SETTING, false, 16, BQ>(a, bb, pk + 8 * h, c, p.scale, vh, 0u);
        if (h == 0)  // first half final before the second half is read
          asm volatile("" : "+r"(pk[0]), "+r"(pk[1]), "+r"(pk[2]), "+r"(pk[3]), "+r"(pk[4]), "+r"(pk[5]),
                       "+r"(pk[6]), "+r"(pk[7])::"memory");
      }
      if (!got) break;
      // dS is final here: keeps the compiler from sinking its arithmetic below the
      // TMEM read of dQp^T, where S and the dQp^T block would both be live
      reg_fence16(pk);
      __syncwarp();
      if (lane == 0) mbar_arrive(v_free);
      // The dK and dQp MMAs of the previous tile are done: dS smem is free and
      // that tile's dQp^T is complete in TMEM.  Read this warp's block of it
      // before publishing dS(j), which lets the next dQp MMA overwrite it.
      if (j >= 1) {
        got = mbar_wait(ds_free, (j - 1) & 1, status, abort_flag);
        __syncwarp();
        if (!got) break;
      }
#pragma unroll
      for (int cch = 0; cch < 4; ++cch) {
        const uint32_t dst = sw128<BK>(dsb, r, grp * 4 + cch);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk[4 * cch]), "r"(pk[4 * cch + 1]),
                     "r"(pk[4 * cch + 2]), "r"(pk[4 * cch + 3])
                     : "memory");
      }
      fence_async_smem();
      uint32_t v[32];
      if (j >= 1) {
        tc_fence_after();
        tmem_ld32(tmem + lane_base + kColDQ + grp * 32, v);
        tmem_ld_wait();
        reg_fence32(v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      if (j >= 1) add_dq(j - 1, v);
    }
    // ---- last tile's dQp^T, then dK out (group g writes d columns [32g, 32g + 32))
    const bool done = mbar_wait(all_done, 0, status, abort_flag);
    __syncwarp();
    if (done) {
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + kColDQ + grp * 32, v);
      tmem_ld_wait();
      reg_fence32(v);
      add_dq(n_yt - 1, v);
    }
    if (done && grp * 32 < D) {
      uint32_t g0[32];
      tmem_ld32(tmem + lane_base + kColDK + grp * 32, g0);
      tmem_ld_wait();
      reg_fence32(g0);
      if (key < p.NK) {
        __nv_bfloat16* dst = dk_out + ((size_t)bh * p.NK + key) * D + grp * 32;
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
