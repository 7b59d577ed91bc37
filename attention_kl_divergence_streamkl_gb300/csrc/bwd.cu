// Recompute-based attention-KL backward, both settings.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "recompute strategy": only KL, LSE1 and LSE2 are kept from the forward; the
// backward rebuilds P_t = exp(S_t - LSE_t) tile by tile from Q, K and the saved
// LSE.  Setting 1 holds P1 fixed and optimises the student side (Q2, K2);
// setting 2 holds P2 fixed and optimises Q1, K1.  Section 手法 3 "numerical
// stability": the setting-2 log ratio is formed from the logits and the saved
// LSEs, never from log of probabilities.  The gradient of L = sum_i g_i KL_i
// with respect to the logits is (derived by the chain rule):
//     setting 1:  dS2 = g_i (P2 - P1)
//     setting 2:  dS1 = g_i P1 (r - KL_i),  r = (S1 - LSE1) - (S2 - LSE2)
// and for the optimised pair dQ = scale dS K, dK = scale dS^T Q.
//
// This file holds the fused path (section 手法 2 "kernel fusion"): each
// (query tile, key tile) pair is visited once from a key-stationary block, dK
// accumulates in registers and the dQ contribution is added into an fp32
// buffer with vector atomics, which the library uses while that buffer fits in
// L2.  The separate path (a query-stationary dQ kernel and a key-stationary dK
// kernel on tcgen05) is in bwd_tc.cu.
#include "common.cuh"
#include "kernels.h"

namespace skl {
namespace {

constexpr int CONSUMERS = 8;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int STAGES = 2;

// ============================================================================
// dK kernel (and fused dK + dQ-atomics): one block per (b*h, 128-key tile),
// streams 64-row query tiles together with their LSE1, LSE2, g, KL values.
// ============================================================================
constexpr int KBK = 128;
constexpr int KBQ = 64;

template <int D, bool FUSED>
struct DkSmem {
  static constexpr int K_BYTES = KBK * D * 2;
  static constexpr int Q_BYTES = KBQ * D * 2;
  static constexpr int V_BYTES = 4 * KBQ * 4;  // lse1', lse2', g, kl per query row
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = K_BYTES;
  static constexpr int OFF_STAGE = 2 * K_BYTES;
  static constexpr int STAGE_BYTES = 2 * Q_BYTES + V_BYTES;  // every term a multiple of 1024
  static constexpr int OFF_DS = OFF_STAGE + STAGES * STAGE_BYTES;
  static constexpr int DS_BYTES = FUSED ? KBK * KBQ * 2 : 0;  // bf16 dS^T [128 keys][64 queries]
  static constexpr int OFF_BAR = OFF_DS + 2 * DS_BYTES;
  static constexpr int BYTES = OFF_BAR + 8 + 16 * STAGES + 16 + 1024;
};

template <int D, int SETTING, bool FUSED>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dk_kernel(const Problem p, const float* __restrict__ lse1, const float* __restrict__ lse2,
                  const float* __restrict__ klv, const float* __restrict__ gv, __nv_bfloat16* __restrict__ dk_out,
                  float* __restrict__ dq_acc, int* status, const __grid_constant__ CUtensorMap mq1,
                  const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mq2,
                  const __grid_constant__ CUtensorMap mk2) {
  using L = DkSmem<D, FUSED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int kt = blockIdx.y;
  const int kb0 = kt * KBK;
  const int n_qt = (p.NQ + KBQ - 1) / KBQ;
  const int qs = p.causal ? max(0, kb0 - p.off) / KBQ : 0;
  const int n_it = n_qt - qs;

  const uint32_t bar_k = sb + L::OFF_BAR;
  const uint32_t bar_full = bar_k + 8;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 + 16 * STAGES);
  if (threadIdx.x == 0) {
    mbar_init(bar_k, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 32);  // 32 producer lanes store row values; lane 0 also posts the TMA bytes
      mbar_init(bar_empty + 8 * s, CONSUMERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == CONSUMERS) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_k, 2 * L::K_BYTES);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(sb + L::OFF_K1 + h * KBK * 128, &mk1, bar_k, h * 64, kb0, bh);
        tma_load_3d(sb + L::OFF_K2 + h * KBK * 128, &mk2, bar_k, h * 64, kb0, bh);
      }
    }
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % STAGES;
      if (it >= STAGES && !mbar_wait(bar_empty + 8 * s, ((it / STAGES) - 1) & 1, status, abort_flag)) break;
      const int q0 = (qs + it) * KBQ;
      const uint32_t st_base = sb + L::OFF_STAGE + s * L::STAGE_BYTES;
      if (lane == 0) {
        mbar_expect_tx(bar_full + 8 * s, 2 * L::Q_BYTES);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(st_base + h * KBQ * 128, &mq1, bar_full + 8 * s, h * 64, q0, bh);
          tma_load_3d(st_base + L::Q_BYTES + h * KBQ * 128, &mq2, bar_full + 8 * s, h * 64, q0, bh);
        }
      }
      float* vals = reinterpret_cast<float*>(smem + L::OFF_STAGE + s * L::STAGE_BYTES + 2 * L::Q_BYTES);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int qi = lane + half * 32;
        const int q = q0 + qi;
        const bool in = q < p.NQ;
        const size_t o = (size_t)bh * p.NQ + q;
        vals[qi] = in ? lse1[o] * kLog2e : 0.f;
        vals[KBQ + qi] = in ? lse2[o] * kLog2e : 0.f;
        vals[2 * KBQ + qi] = in ? gv[o] : 0.f;
        vals[3 * KBQ + qi] = (SETTING == 2 && in) ? klv[o] : 0.f;
      }
      mbar_arrive(bar_full + 8 * s);
      issued = it + 1;
    }
    if (lane == 0) {
      mbar_drain(bar_k, 0, status);
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        mbar_drain(bar_full + 8 * (it % STAGES), (it / STAGES) & 1, status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const float c = p.c;
  const int key0 = kb0 + warp * 16 + g;  // this thread's keys: key0, key0 + 8
  float dk[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) dk[n][j] = 0.f;

  bool ok = mbar_wait(bar_k, 0, status, abort_flag);
  const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int acol = lane >> 4;
  const int brow = (lane & 7) + (lane >> 4) * 8;
  const int bcol = (lane >> 3) & 1;
  const int trow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int tcol = lane >> 4;

  for (int it = 0; ok && it < n_it; ++it) {
    const int s = it % STAGES;
    if (!mbar_wait(bar_full + 8 * s, (it / STAGES) & 1, status, abort_flag)) {
      ok = false;
      break;
    }
    const int q0 = (qs + it) * KBQ;
    const uint32_t qb1 = sb + L::OFF_STAGE + s * L::STAGE_BYTES;
    const uint32_t qb2 = qb1 + L::Q_BYTES;
    const float* vals = reinterpret_cast<const float*>(smem + L::OFF_STAGE + s * L::STAGE_BYTES + 2 * L::Q_BYTES);

    // S^T = K Q^T for this warp's 16 keys and the 64 queries of the tile
    float s1[8][4], s2[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) s1[n][j] = s2[n][j] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a1[4], a2[4];
      ldsm_x4(sw128<KBK>(sb + L::OFF_K1, arow, 2 * ks + acol), a1);
      ldsm_x4(sw128<KBK>(sb + L::OFF_K2, arow, 2 * ks + acol), a2);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldsm_x4(sw128<KBQ>(qb1, np * 16 + brow, 2 * ks + bcol), b);
        mma16816(s1[2 * np], a1, b[0], b[1]);
        mma16816(s1[2 * np + 1], a1, b[2], b[3]);
        ldsm_x4(sw128<KBQ>(qb2, np * 16 + brow, 2 * ks + bcol), b);
        mma16816(s2[2 * np], a2, b[0], b[1]);
        mma16816(s2[2 * np + 1], a2, b[2], b[3]);
      }
    }
    const bool need_mask =
        (q0 + KBQ > p.NQ) || (kb0 + KBK > p.NK) || (p.causal && kb0 + KBK - 1 > q0 + p.off);
    uint32_t af[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      float ds[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = key0 + (j >> 1) * 8;
        const int qi = n * 8 + 2 * t + (j & 1);
        const int q = q0 + qi;
        const bool keep = !need_mask || (q < p.NQ && key < p.NK && (!p.causal || key <= q + p.off));
        const float L1 = vals[qi], L2 = vals[KBQ + qi], G = vals[2 * KBQ + qi];
        const float p1 = keep ? ex2(fmaf(s1[n][j], c, -L1)) : 0.f;
        if (SETTING == 1) {
          const float p2 = keep ? ex2(fmaf(s2[n][j], c, -L2)) : 0.f;
          ds[j] = G * (p2 - p1);
        } else {
          const float r = kLn2 * fmaf(s1[n][j] - s2[n][j], c, L2 - L1);
          ds[j] = G * p1 * (r - vals[3 * KBQ + qi]);
        }
      }
      af[n >> 1][2 * (n & 1) + 0] = pack_bf16(ds[0], ds[1]);
      af[n >> 1][2 * (n & 1) + 1] = pack_bf16(ds[2], ds[3]);
    }
    const uint32_t dsb = sb + L::OFF_DS + (it & 1) * L::DS_BYTES;
    if (FUSED) {
      // dS^T (keys x queries) to shared memory for the dQ contraction
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const uint32_t a0 = sw128<KBK>(dsb, warp * 16 + g, n) + 4 * t;
        const uint32_t a8 = sw128<KBK>(dsb, warp * 16 + g + 8, n) + 4 * t;
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(a0), "r"(af[n >> 1][2 * (n & 1)]) : "memory");
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(a8), "r"(af[n >> 1][2 * (n & 1) + 1]) : "memory");
      }
    }
    // dK += dS^T Q_opt
    const uint32_t qopt = SETTING == 1 ? qb2 : qb1;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b[4];
        ldsm_x4_t(sw128<KBQ>(qopt, kk * 16 + trow, 2 * np + tcol), b);
        mma16816(dk[2 * np], af[kk], b[0], b[1]);
        mma16816(dk[2 * np + 1], af[kk], b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    if (FUSED) {
      // dQ partial = dS (64 queries x 128 keys) K_opt (128 keys x D): each warp
      // owns 16 queries x D/2 columns; results go to the fp32 buffer atomically.
      named_bar_sync(1, CONSUMERS * 32);
      const int qg = warp >> 1, dh = warp & 1;
      const uint32_t kopt = sb + (SETTING == 1 ? L::OFF_K2 : L::OFF_K1);
      float pq[D / 16][4];
#pragma unroll
      for (int n = 0; n < D / 16; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) pq[n][j] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KBK / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4_t(sw128<KBK>(dsb, kk * 16 + (lane & 7) + (lane >> 4) * 8, 2 * qg + ((lane >> 3) & 1)), a);
#pragma unroll
        for (int np = 0; np < D / 32; ++np) {
          uint32_t b[4];
          ldsm_x4_t(sw128<KBK>(kopt, kk * 16 + trow, dh * (D / 16) + 2 * np + tcol), b);
          mma16816(pq[2 * np], a, b[0], b[1]);
          mma16816(pq[2 * np + 1], a, b[2], b[3]);
        }
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int q = q0 + qg * 16 + g + hr * 8;
        if (q < p.NQ) {
          float* dst = dq_acc + ((size_t)bh * p.NQ + q) * D + dh * (D / 2) + 2 * t;
#pragma unroll
          for (int n = 0; n < D / 16; ++n) red_add_v2(dst + n * 8, pq[n][2 * hr], pq[n][2 * hr + 1]);
        }
      }
    }
  }
  if (!ok) return;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int key = key0 + hr * 8;
    if (key < p.NK) {
      __nv_bfloat16* dst = dk_out + ((size_t)bh * p.NK + key) * D + 2 * t;
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<uint32_t*>(dst + n * 8) =
            pack_bf16(dk[n][2 * hr] * p.scale, dk[n][2 * hr + 1] * p.scale);
    }
  }
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

// FUSED = false is the separate-path dK form of the same loop; only the fused
// form is launched (the separate path runs on tcgen05, bwd_tc.cu).
template <int D, int SETTING, bool FUSED>
cudaError_t launch_dk(const Problem& p, const BwdIn& in, void* dk, float* dq_acc, int* status, cudaStream_t st) {
  CUtensorMap mq1, mk1, mq2, mk2;
  if (!encode_tile_map(&mq1, in.q1, D, p.NQ, p.BH, KBQ) || !encode_tile_map(&mq2, in.q2, D, p.NQ, p.BH, KBQ) ||
      !encode_tile_map(&mk1, in.k1, D, p.NK, p.BH, KBK) || !encode_tile_map(&mk2, in.k2, D, p.NK, p.BH, KBK))
    return cudaErrorInvalidValue;
  const int smem = DkSmem<D, FUSED>::BYTES;
  auto kern = bwd_dk_kernel<D, SETTING, FUSED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.BH, (p.NK + KBK - 1) / KBK), THREADS, smem, st>>>(
      p, in.lse1, in.lse2, in.kl, in.g, static_cast<__nv_bfloat16*>(dk), dq_acc, status, mq1, mk1, mq2, mk2);
  return cudaGetLastError();
}

template <int D>
cudaError_t fused_d(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, float* dq_acc, int* status,
                    cudaStream_t st) {
  const size_t n = (size_t)p.BH * p.NQ * D;
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, n * sizeof(float), st);
  if (e != cudaSuccess) return e;
  e = setting == 1 ? launch_dk<D, 1, true>(p, in, dk, dq_acc, status, st)
                   : launch_dk<D, 2, true>(p, in, dk, dq_acc, status, st);
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
