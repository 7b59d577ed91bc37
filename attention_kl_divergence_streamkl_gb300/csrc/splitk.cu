// Split-K attention-KL forward for few query rows (decode).
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 3
// "Split-K variant": when N_Q is small (autoregressive decoding, N_Q = 1) the
// key dimension is divided across thread blocks so that the SMs stay busy.
// The pages leave the merge implicit; the plain reading is the exact merge of
// the five running scalars of each key range (derived):
//     M1 = max_s m1_s,  l1 = sum_s l1_s 2^(m1_s - M1),  acc = sum_s acc_s 2^(m1_s - M1)
//     M2 = max_s m2_s,  l2 = sum_s l2_s 2^(m2_s - M2)
// followed by the usual closing step of the forward.
//
// The work is HBM-bound: every key byte is read once.  A block owns one
// (b*h, key range); a producer warp streams 64-key tiles of K1 and K2 (16 KiB
// each at D = 128) through a 3-stage TMA ring, and 4 consumer warps each take
// 16 keys of a tile with the keys on the MMA M dimension and the (at most 16)
// queries on N, so a tile costs a handful of mma.sync per warp.  Each thread
// keeps the running scalars of its queries and rescales only when a new
// maximum exceeds the reference by more than 2^8 (exact: l1 and acc share m1).
#include <atomic>

#include "../../include/streamkl.h"
#include "common.cuh"
#include "kernels.h"

// Fixed scratch of the allocation-free Split-K entry point: the partial states
// of every split live here instead of in a caller-provided workspace.  Every
// GPU that loads the library holds it until the process exits.
static __device__ __align__(256) float g_splitk_noalloc_scratch[STREAMKL_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace skl {
namespace {

constexpr int BN = kSplitKTile;  // 64 keys per stage
constexpr int STAGES = 3;
constexpr int CONSUMERS = 4;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int QROWS = 16;  // queries padded to 16
constexpr float kLazy = 8.0f;  // log2 units

template <int D>
struct Smem {
  static constexpr int Q_BYTES = QROWS * D * 2;
  static constexpr int K_BYTES = BN * D * 2;
  static constexpr int OFF_K = 0;
  static constexpr int STAGE_BYTES = 2 * K_BYTES;
  static constexpr int OFF_Q1 = STAGES * STAGE_BYTES;
  static constexpr int OFF_Q2 = OFF_Q1 + Q_BYTES;
  static constexpr int OFF_RED = OFF_Q2 + Q_BYTES;  // [CONSUMERS][QROWS][5] fp32
  static constexpr int OFF_BAR = OFF_RED + CONSUMERS * QROWS * 5 * 4;
  static constexpr int BYTES = OFF_BAR + 16 * STAGES + 16 + 1024;
};

struct State {
  float m1, m2, l1, l2, acc;
};

__device__ __forceinline__ void merge_into(State& a, const State& b) {
  const float M1 = fmaxf(a.m1, b.m1), M2 = fmaxf(a.m2, b.m2);
  if (M1 != kNegInf) {
    const float wa = ex2(a.m1 - M1), wb = ex2(b.m1 - M1);
    a.l1 = a.l1 * wa + b.l1 * wb;
    a.acc = a.acc * wa + b.acc * wb;
  }
  if (M2 != kNegInf) {
    const float wa = ex2(a.m2 - M2), wb = ex2(b.m2 - M2);
    a.l2 = a.l2 * wa + b.l2 * wb;
  }
  a.m1 = M1;
  a.m2 = M2;
}

__device__ __forceinline__ State shfl_state(const State& s, int mask) {
  State o;
  o.m1 = __shfl_xor_sync(0xffffffffu, s.m1, mask);
  o.m2 = __shfl_xor_sync(0xffffffffu, s.m2, mask);
  o.l1 = __shfl_xor_sync(0xffffffffu, s.l1, mask);
  o.l2 = __shfl_xor_sync(0xffffffffu, s.l2, mask);
  o.acc = __shfl_xor_sync(0xffffffffu, s.acc, mask);
  return o;
}

// Lazy online step for one query and two candidate keys (a, b).
__device__ __forceinline__ void step2(State& st, float x1a, float x1b, float x2a, float x2b, float da, float db,
                                      bool va, bool vb) {
  // x*: logits in log2 units (-inf when masked); d*: raw q1.k1 - q2.k2
  const float t1 = fmaxf(x1a, x1b), t2 = fmaxf(x2a, x2b);
  if (t1 > st.m1 + kLazy) {
    const float al = ex2(st.m1 - t1);
    st.l1 *= al;
    st.acc *= al;
    st.m1 = t1;
  }
  if (t2 > st.m2 + kLazy) {
    const float al = ex2(st.m2 - t2);
    st.l2 *= al;
    st.m2 = t2;
  }
  const float p1a = va ? ex2(x1a - st.m1) : 0.f, p1b = vb ? ex2(x1b - st.m1) : 0.f;
  const float p2a = va ? ex2(x2a - st.m2) : 0.f, p2b = vb ? ex2(x2b - st.m2) : 0.f;
  st.l1 += p1a + p1b;
  st.l2 += p2a + p2b;
  st.acc = fmaf(p1a, da, fmaf(p1b, db, st.acc));
}

template <int D>
__global__ void __launch_bounds__(THREADS)
    splitk_partial_kernel(const Problem p, const __nv_bfloat16* __restrict__ q1, const __nv_bfloat16* __restrict__ q2,
                          float* __restrict__ partials, int* status, const __grid_constant__ CUtensorMap mk1,
                          const __grid_constant__ CUtensorMap mk2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int mh = bh % p.H, mb = bh / p.H;  // head and batch coordinates of the tensor maps
  const int split = blockIdx.y, S = gridDim.y;
  const int T = (p.NK + BN - 1) / BN;
  const int t_begin = (int)(((long long)split * T) / S);
  const int t_end = (int)(((long long)(split + 1) * T) / S);
  const int n_t = t_end - t_begin;

  const uint32_t bar_full = sb + L::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 16 * STAGES);

  // Query rows go to shared memory with plain loads (zero past N_Q), in the
  // same swizzled layout the TMA tiles use.
  {
    const int chunks = QROWS * (D / 8);
    for (int i = threadIdx.x; i < 2 * chunks; i += THREADS) {
      const int which = i / chunks, rem = i % chunks;
      const int r = rem / (D / 8), ch = rem % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < p.NQ) {
        const __nv_bfloat16* src = (which == 0 ? q1 : q2) + row_offset(bh, p.H, r, p.qs_b, p.qs_h, p.qs_n) + ch * 8;
        v = *reinterpret_cast<const uint4*>(src);
      }
      const uint32_t dst = sw128<QROWS>(sb + (which == 0 ? L::OFF_Q1 : L::OFF_Q2), r, ch);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, CONSUMERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == CONSUMERS) {
    if (lane == 0) {
      prefetch_tensormap(&mk1);
      prefetch_tensormap(&mk2);
      int issued = 0;
      for (int it = 0; it < n_t; ++it) {
        const int s = it % STAGES;
        if (it >= STAGES && !mbar_wait(bar_empty + 8 * s, ((it / STAGES) - 1) & 1, status, abort_flag)) break;
        const uint32_t kb = sb + L::OFF_K + s * L::STAGE_BYTES;
        const int y = (t_begin + it) * BN;
        mbar_arrive_expect_tx(bar_full + 8 * s, L::STAGE_BYTES);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(kb + h * BN * 128, &mk1, bar_full + 8 * s, h * 64, y, mh, mb);
          tma_load_4d(kb + L::K_BYTES + h * BN * 128, &mk2, bar_full + 8 * s, h * 64, y, mh, mb);
        }
        issued = it + 1;
      }
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        mbar_drain(bar_full + 8 * (it % STAGES), (it / STAGES) & 1, status);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const float c = p.c;
  // B fragments of Q1^T and Q2^T (both 8-query n-tiles) for every k-step.
  uint32_t qb1[D / 16][4], qb2[D / 16][4];
  {
    const int qrow = (lane & 7) + (lane >> 4) * 8;
    const int qcol = (lane >> 3) & 1;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      ldsm_x4(sw128<QROWS>(sb + L::OFF_Q1, qrow, 2 * ks + qcol), qb1[ks]);
      ldsm_x4(sw128<QROWS>(sb + L::OFF_Q2, qrow, 2 * ks + qcol), qb2[ks]);
    }
  }
  const int nt_count = p.NQ > 8 ? 2 : 1;
  State st[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) st[nt][e] = State{kNegInf, kNegInf, 0.f, 0.f, 0.f};

  const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int acol = lane >> 4;
  bool ok = true;
  for (int it = 0; it < n_t; ++it) {
    const int s = it % STAGES;
    if (!mbar_wait(bar_full + 8 * s, (it / STAGES) & 1, status, abort_flag)) {
      ok = false;
      break;
    }
    const uint32_t kb1 = sb + L::OFF_K + s * L::STAGE_BYTES;
    const uint32_t kb2 = kb1 + L::K_BYTES;
    float c1[2][4], c2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) c1[nt][j] = c2[nt][j] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a1[4], a2[4];
      ldsm_x4(sw128<BN>(kb1, arow, 2 * ks + acol), a1);
      ldsm_x4(sw128<BN>(kb2, arow, 2 * ks + acol), a2);
      mma16816(c1[0], a1, qb1[ks][0], qb1[ks][1]);
      mma16816(c2[0], a2, qb2[ks][0], qb2[ks][1]);
      if (nt_count == 2) {
        mma16816(c1[1], a1, qb1[ks][2], qb1[ks][3]);
        mma16816(c2[1], a2, qb2[ks][2], qb2[ks][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    const int ka = (t_begin + it) * BN + warp * 16 + g, kb = ka + 8;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt < nt_count) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = nt * 8 + 2 * t + e;
          const bool va = ka < p.NK && (!p.causal || ka <= q + p.off);
          const bool vb = kb < p.NK && (!p.causal || kb <= q + p.off);
          const float s1a = c1[nt][e], s1b = c1[nt][2 + e];
          const float s2a = c2[nt][e], s2b = c2[nt][2 + e];
          step2(st[nt][e], va ? s1a * c : kNegInf, vb ? s1b * c : kNegInf, va ? s2a * c : kNegInf,
                vb ? s2b * c : kNegInf, va ? s1a - s2a : 0.f, vb ? s1b - s2b : 0.f, va, vb);
        }
      }
    }
  }
  // A block that gave up writes nothing; the status word reports it.
  if (!ok) return;

  // ---- reduce: across the 8 lanes that share t (different keys), then across warps
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) merge_into(st[nt][e], shfl_state(st[nt][e], m));
      if (g == 0) {
        float* r = red + (warp * QROWS + nt * 8 + 2 * t + e) * 5;
        r[0] = st[nt][e].m1;
        r[1] = st[nt][e].m2;
        r[2] = st[nt][e].l1;
        r[3] = st[nt][e].l2;
        r[4] = st[nt][e].acc;
      }
    }
  named_bar_sync(1, CONSUMERS * 32);
  if (warp == 0 && lane < p.NQ) {
    const float* r = red + lane * 5;
    State a{r[0], r[1], r[2], r[3], r[4]};
    for (int w = 1; w < CONSUMERS; ++w) {
      const float* o = red + (w * QROWS + lane) * 5;
      merge_into(a, State{o[0], o[1], o[2], o[3], o[4]});
    }
    float* dst = partials + (((size_t)bh * p.NQ + lane) * S + split) * 5;
    dst[0] = a.m1;
    dst[1] = a.m2;
    dst[2] = a.l1;
    dst[3] = a.l2;
    dst[4] = a.acc;
  }
}

// One warp merges the S partial states of one (b*h, query) row.  Partial s of
// row `row` starts at partials + row * row_stride + s * part_stride (floats):
// [row][split][5] for the Split-K splits, [part][row][5] for key shards.  A part
// whose keys the row does not see (m = -inf, l = acc = 0) adds nothing.
__global__ void __launch_bounds__(256) splitk_combine_kernel(const Problem p, int S, const float* __restrict__ partials,
                                                             long long row_stride, long long part_stride,
                                                             float* __restrict__ out_kl,
                                                             float* __restrict__ out_lse1,
                                                             float* __restrict__ out_lse2) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.BH * p.NQ) return;
  const float* ps = partials + (size_t)row * row_stride;
  float M1 = kNegInf, M2 = kNegInf;
  for (int s = lane; s < S; s += 32) {
    M1 = fmaxf(M1, ps[s * part_stride + 0]);
    M2 = fmaxf(M2, ps[s * part_stride + 1]);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    M1 = fmaxf(M1, __shfl_xor_sync(0xffffffffu, M1, m));
    M2 = fmaxf(M2, __shfl_xor_sync(0xffffffffu, M2, m));
  }
  float l1 = 0.f, l2 = 0.f, acc = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float* q = ps + s * part_stride;
    const float w1 = ex2(q[0] - M1);  // 2^-inf = 0 for a part that saw no key
    const float w2 = ex2(q[1] - M2);
    l1 = fmaf(q[2], w1, l1);
    acc = fmaf(q[4], w1, acc);
    l2 = fmaf(q[3], w2, l2);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    l1 += __shfl_xor_sync(0xffffffffu, l1, m);
    l2 += __shfl_xor_sync(0xffffffffu, l2, m);
    acc += __shfl_xor_sync(0xffffffffu, acc, m);
  }
  if (lane == 0) {
    const float lse1 = (M1 + log2f(l1)) * kLn2;
    const float lse2 = (M2 + log2f(l2)) * kLn2;
    out_lse1[row] = lse1;
    out_lse2[row] = lse2;
    out_kl[row] = p.scale * (acc / l1) + lse2 - lse1;
  }
}

template <int D>
cudaError_t launch_d(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2, int splits,
                     float* partials, float* kl, float* lse1, float* lse2, int* status, cudaStream_t st) {
  CUtensorMap mk1, mk2;
  if (!encode_k_map(&mk1, k1, p, BN) || !encode_k_map(&mk2, k2, p, BN))
    return cudaErrorInvalidValue;
  const int smem = Smem<D>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(splitk_partial_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  splitk_partial_kernel<D><<<dim3(p.BH, splits), THREADS, smem, st>>>(
      p, static_cast<const __nv_bfloat16*>(q1), static_cast<const __nv_bfloat16*>(q2), partials, status, mk1, mk2);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = p.BH * p.NQ;
  splitk_combine_kernel<<<(rows + 7) / 8, 256, 0, st>>>(p, splits, partials, (long long)splits * 5, 5, kl, lse1,
                                                        lse2);
  return cudaGetLastError();
}

}  // namespace

int splitk_key_tiles(const Problem& p) { return (p.NK + BN - 1) / BN; }

// In host code the name g_splitk_noalloc_scratch is only a host-side stand-in;
// the kernels need its device address, which the runtime gives per device.  It
// is looked up once per device, with that device current, and kept.
cudaError_t splitk_noalloc_scratch(float** out) {
  constexpr int kMaxDevices = 64;
  static std::atomic<float*> table[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  float* p = table[dev].load(std::memory_order_acquire);
  if (!p) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_splitk_noalloc_scratch);
    if (e != cudaSuccess) return e;
    p = static_cast<float*>(addr);
    table[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

// Split count for BH heads of `key_tiles` tiles on `num_sms` SMs: minimises
// waves x (tiles per block + a fixed per-block cost), where a wave is one
// block on each of kSplitKCtasPerSm slots per SM.
int splitk_plan(int BH, int key_tiles, int num_sms) {
  if (key_tiles <= 1) return 1;
  const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * kSplitKCtasPerSm;
  const long long overhead = 2;  // tiles' worth of prologue/epilogue per block
  int best = 1;
  long long best_cost = -1;
  const int max_s = key_tiles < 4096 ? key_tiles : 4096;
  for (int s = 1; s <= max_s; ++s) {
    const long long blocks = (long long)BH * s;
    const long long waves = (blocks + slots - 1) / slots;
    const long long per = (key_tiles + s - 1) / s;
    const long long cost = waves * (per + overhead);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

cudaError_t launch_merge_partials(const Problem& p, int parts, const float* partials, float* kl, float* lse1,
                                  float* lse2, cudaStream_t st) {
  const long long rows = (long long)p.BH * p.NQ;
  if (rows == 0) return cudaSuccess;
  splitk_combine_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(p, parts, partials, 5, rows * 5, kl, lse1, lse2);
  return cudaGetLastError();
}

cudaError_t launch_splitk(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                          int splits, float* partials, float* kl, float* lse1, float* lse2, int* status,
                          cudaStream_t st) {
  if (p.D == 64) return launch_d<64>(p, q1, k1, q2, k2, splits, partials, kl, lse1, lse2, status, st);
  return launch_d<128>(p, q1, k1, q2, k2, splits, partials, kl, lse1, lse2, status, st);
}

}  // namespace skl
