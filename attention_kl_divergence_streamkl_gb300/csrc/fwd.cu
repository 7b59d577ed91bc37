// One-pass attention-KL forward.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 1
// "online formulation": each query row keeps five running scalars -- the two
// running maxima m1, m2, the two unnormalised exponential sums l1, l2 and the
// weighted logit-difference accumulator acc -- while key tiles stream through
// on-chip memory; the row result is KL = acc/l1 + LSE2 - LSE1 with
// LSE_t = m_t + log l_t, and key tiles wholly past the causal boundary are
// never visited.
//
// Update rules used here (derived; the pages name the scalars but print no
// update equations), per key tile, in log2 units x = c * (q . k), c = scale*log2 e:
//     m1' = max(m1, max_j x1_j)          a1 = 2^(m1 - m1')
//     l1  = a1 l1  + sum_j 2^(x1_j - m1')
//     acc = a1 acc + sum_j 2^(x1_j - m1') (q1.k1_j - q2.k2_j)
//     m2', l2 likewise from x2
// and at the end LSE_t = ln2 (m_t + log2 l_t), KL = scale acc / l1 + LSE2 - LSE1.
//
// Layout: one CTA per (b*h, 128-row query tile); 8 consumer warps own 16 rows
// each, one producer warp feeds K1/K2 tiles of 64 keys through a 2-stage TMA
// ring (128-byte swizzle).  The logits come from bf16 mma.sync into fp32
// registers.  Query tiles are launched longest-first for causal balance.
#include "common.cuh"
#include "kernels.h"

namespace skl {
namespace {

constexpr int BM = 128;
constexpr int BN = 64;
constexpr int STAGES = 2;
constexpr int CONSUMERS = 8;
constexpr int THREADS = (CONSUMERS + 1) * 32;

template <int D>
struct Smem {
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int K_BYTES = BN * D * 2;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = Q_BYTES;
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int STAGE_BYTES = 2 * K_BYTES;
  static constexpr int OFF_BAR = OFF_K + STAGES * STAGE_BYTES;
  // bar_q, full[STAGES], empty[STAGES], abort flag
  static constexpr int BYTES = OFF_BAR + 8 + 16 * STAGES + 16 + 1024;
};

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_kernel(const Problem p, float* __restrict__ out_kl, float* __restrict__ out_lse1,
               float* __restrict__ out_lse2, int* status, const __grid_constant__ CUtensorMap mq1,
               const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mq2,
               const __grid_constant__ CUtensorMap mk2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int qt = gridDim.y - 1 - blockIdx.y;  // longest causal tiles first
  const int q0 = qt * BM;
  const int q_last = min(p.NQ, q0 + BM) - 1;
  const int kend = p.causal ? min(p.NK, q_last + p.off + 1) : p.NK;
  const int n_kt = (kend + BN - 1) / BN;

  const uint32_t bar_q = sb + L::OFF_BAR;
  const uint32_t bar_full = bar_q + 8;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 + 16 * STAGES);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, CONSUMERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == CONSUMERS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&mq1);
      prefetch_tensormap(&mk1);
      prefetch_tensormap(&mq2);
      prefetch_tensormap(&mk2);
      mbar_arrive_expect_tx(bar_q, 2 * L::Q_BYTES);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(sb + L::OFF_Q1 + h * BM * 128, &mq1, bar_q, h * 64, q0, bh);
        tma_load_3d(sb + L::OFF_Q2 + h * BM * 128, &mq2, bar_q, h * 64, q0, bh);
      }
      int issued = 0;
      for (int it = 0; it < n_kt; ++it) {
        const int s = it % STAGES;
        if (it >= STAGES && !mbar_wait(bar_empty + 8 * s, ((it / STAGES) - 1) & 1, status, abort_flag)) break;
        const uint32_t kb = sb + L::OFF_K + s * L::STAGE_BYTES;
        mbar_arrive_expect_tx(bar_full + 8 * s, L::STAGE_BYTES);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(kb + h * BN * 128, &mk1, bar_full + 8 * s, h * 64, it * BN, bh);
          tma_load_3d(kb + L::K_BYTES + h * BN * 128, &mk2, bar_full + 8 * s, h * 64, it * BN, bh);
        }
        issued = it + 1;
      }
      // Do not leave while copies may still land in this block's shared memory.
      mbar_drain(bar_q, 0, status);
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        mbar_drain(bar_full + 8 * (it % STAGES), (it / STAGES) & 1, status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int row0 = q0 + warp * 16 + g;  // this thread's rows: row0, row0 + 8
  const float c = p.c;
  float m1[2] = {kNegInf, kNegInf}, m2[2] = {kNegInf, kNegInf};
  float l1[2] = {0.f, 0.f}, l2[2] = {0.f, 0.f}, acc[2] = {0.f, 0.f};
  bool ok = mbar_wait(bar_q, 0, status, abort_flag);

  const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int acol = lane >> 4;
  const int brow = (lane & 7) + (lane >> 4) * 8;
  const int bcol = (lane >> 3) & 1;

  for (int it = 0; ok && it < n_kt; ++it) {
    const int s = it % STAGES;
    if (!mbar_wait(bar_full + 8 * s, (it / STAGES) & 1, status, abort_flag)) {
      ok = false;
      break;
    }
    const uint32_t kb1 = sb + L::OFF_K + s * L::STAGE_BYTES;
    const uint32_t kb2 = kb1 + L::K_BYTES;
    float s1[8][4], s2[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) s1[n][j] = s2[n][j] = 0.f;

#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a1[4], a2[4];
      ldsm_x4(sw128<BM>(sb + L::OFF_Q1, arow, 2 * ks + acol), a1);
      ldsm_x4(sw128<BM>(sb + L::OFF_Q2, arow, 2 * ks + acol), a2);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldsm_x4(sw128<BN>(kb1, np * 16 + brow, 2 * ks + bcol), b);
        mma16816(s1[2 * np], a1, b[0], b[1]);
        mma16816(s1[2 * np + 1], a1, b[2], b[3]);
        ldsm_x4(sw128<BN>(kb2, np * 16 + brow, 2 * ks + bcol), b);
        mma16816(s2[2 * np], a2, b[0], b[1]);
        mma16816(s2[2 * np + 1], a2, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    // ---- online update of the five scalars for rows row0 and row0 + 8
    const int kbase = it * BN;
    const bool need_mask = (kbase + BN > p.NK) || (p.causal && kbase + BN - 1 > q0 + p.off);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = row0 + hr * 8;
      float v1[16], v2[16], d[16];
      float mx1 = kNegInf, mx2 = kNegInf;
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = n * 2 + e;
          v1[i] = s1[n][2 * hr + e];
          v2[i] = s2[n][2 * hr + e];
          d[i] = v1[i] - v2[i];
          if (need_mask) {
            const int key = kbase + n * 8 + 2 * t + e;
            const bool keep = key < p.NK && (!p.causal || key <= row + p.off);
            if (!keep) {
              v1[i] = kNegInf;
              v2[i] = kNegInf;
              d[i] = 0.f;
            }
          }
          mx1 = fmaxf(mx1, v1[i]);
          mx2 = fmaxf(mx2, v2[i]);
        }
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      mx2 = fmaxf(mx2, __shfl_xor_sync(0xffffffffu, mx2, 1));
      mx2 = fmaxf(mx2, __shfl_xor_sync(0xffffffffu, mx2, 2));
      const float n1 = fmaxf(m1[hr], mx1 * c);
      const float n2 = fmaxf(m2[hr], mx2 * c);
      const float b1 = n1 == kNegInf ? 0.f : n1;  // all keys masked so far: weights stay 0
      const float b2 = n2 == kNegInf ? 0.f : n2;
      const float a1 = ex2(m1[hr] - b1);
      const float a2 = ex2(m2[hr] - b2);
      float sl1 = 0.f, sl2 = 0.f, sacc = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p1 = ex2(fmaf(v1[i], c, -b1));
        const float p2 = ex2(fmaf(v2[i], c, -b2));
        sl1 += p1;
        sl2 += p2;
        sacc = fmaf(p1, d[i], sacc);
      }
      l1[hr] = fmaf(l1[hr], a1, sl1);
      acc[hr] = fmaf(acc[hr], a1, sacc);
      l2[hr] = fmaf(l2[hr], a2, sl2);
      m1[hr] = n1;
      m2[hr] = n2;
    }
  }
  if (!ok) return;

  // ---- epilogue: the quad shares the running maxima, so sums simply add
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    float L1 = l1[hr], L2 = l2[hr], A = acc[hr];
    L1 += __shfl_xor_sync(0xffffffffu, L1, 1);
    L1 += __shfl_xor_sync(0xffffffffu, L1, 2);
    L2 += __shfl_xor_sync(0xffffffffu, L2, 1);
    L2 += __shfl_xor_sync(0xffffffffu, L2, 2);
    A += __shfl_xor_sync(0xffffffffu, A, 1);
    A += __shfl_xor_sync(0xffffffffu, A, 2);
    const int row = row0 + hr * 8;
    if (t == 0 && row < p.NQ) {
      const float lse1 = (m1[hr] + log2f(L1)) * kLn2;
      const float lse2 = (m2[hr] + log2f(L2)) * kLn2;
      const size_t o = (size_t)bh * p.NQ + row;
      out_lse1[o] = lse1;
      out_lse2[o] = lse2;
      out_kl[o] = p.scale * (A / L1) + lse2 - lse1;
    }
  }
}

template <int D>
cudaError_t launch_fwd_d(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                         float* kl, float* lse1, float* lse2, int* status, cudaStream_t st) {
  CUtensorMap mq1, mk1, mq2, mk2;
  if (!encode_tile_map(&mq1, q1, D, p.NQ, p.BH, BM) || !encode_tile_map(&mq2, q2, D, p.NQ, p.BH, BM) ||
      !encode_tile_map(&mk1, k1, D, p.NK, p.BH, BN) || !encode_tile_map(&mk2, k2, D, p.NK, p.BH, BN))
    return cudaErrorInvalidValue;
  const int smem = Smem<D>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.BH, (p.NQ + BM - 1) / BM);
  fwd_kernel<D><<<grid, THREADS, smem, st>>>(p, kl, lse1, lse2, status, mq1, mk1, mq2, mk2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                       float* kl, float* lse1, float* lse2, int* status, cudaStream_t st) {
  if (p.D == 64) return launch_fwd_d<64>(p, q1, k1, q2, k2, kl, lse1, lse2, status, st);
  return launch_fwd_d<128>(p, q1, k1, q2, k2, kl, lse1, lse2, status, st);
}

}  // namespace skl
