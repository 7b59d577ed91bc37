// One-pass attention-KL forward on the 5th-generation tensor cores.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 1
// "online formulation": each query row keeps five running scalars (the running
// maxima m1, m2, the unnormalised exponential sums l1, l2 and the weighted
// logit-difference accumulator acc) while key tiles stream through on-chip
// memory; the row result is KL = acc/l1 + LSE2 - LSE1 with LSE_t = m_t + log l_t,
// and key tiles wholly past the causal boundary are never visited.
//
// Update rules (derived; the pages name the scalars but print no equations), in
// log2 units x = c (q . k), c = scale log2(e), for the keys j of a tile:
//     if max_j x1_j > m1 + 8:  a = 2^(m1 - max_j x1_j); l1 *= a; acc *= a; m1 = max_j x1_j
//     l1  += sum_j 2^(x1_j - m1)
//     acc += sum_j 2^(x1_j - m1) (q1.k1_j - q2.k2_j)
//     m2, l2 likewise from x2
// The maximum is only moved when it grows by more than 2^8 (terms stay <= 256,
// far from fp32 overflow); this is exact because l1 and acc share m1.  Once a
// row has finite maxima, a tile is first summed against them without taking its
// own maximum: if every term stays below 2^64 (the tile's sums show it, inf
// included) the sums are kept, else the tile is redone with its maximum as
// above.  At the end LSE_t = ln2 (m_t + log2 l_t) and KL = scale acc / l1 +
// LSE2 - LSE1 -- or, for a key shard of a longer sequence, the five scalars
// themselves are written out, to be merged with the other shards' (the
// exact merge of the Split-K variant, section 手法 3).
//
// Block layout (a block walks 128-row query tiles, "items"; key tiles of 128):
//   warp 8      TMA producer: an item's Q1, Q2 once the previous item's MMAs are done, then its K1/K2
//               tiles through 2 stages (stage and barrier phases count tiles across items)
//   warp 9      TMEM owner (512 columns) and MMA issuer (one thread):
//               S1 = Q1 K1^T and S2 = Q2 K2^T, M = N = 128, bf16 -> fp32 in
//               TMEM, double-buffered (buffer b: S1 at 256b, S2 at 256b + 128)
//   warps 0-7   two softmax warpgroups; thread = query row (TMEM lane), group
//               g takes columns [64g, 64g + 64) of every tile and keeps its own
//               five scalars; the groups merge in the epilogue.
// Items are ordered head by head, longest causal tile first.  With many items
// per SM each block takes one (the hardware's block scheduler then balances the
// triangle); with few, one block per SM walks them, alternating the direction
// of each round so that long and short items even out.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int SOFTMAX_WARPS = 8;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 10 * 32;
constexpr float kLazy = 8.0f;
constexpr float kFastSumLimit = 18446744073709551616.0f;  // 2^64
constexpr uint32_t kTmemCols = 512;
constexpr int kOneBlockPerSmSmem = 120 * 1024;
constexpr long long kMaxPersistentRounds = 32;
constexpr long long kMaxPersistentKeyTiles = 64;

template <int D>
struct Smem {
  static constexpr int Q_BYTES = BM * D * 2;  // one 128-row tile, D/64 halves of 16 KiB
  static constexpr int K_BYTES = BN * D * 2;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = Q_BYTES;
  static constexpr int OFF_K = 2 * Q_BYTES;  // stage s: K1 at OFF_K + s*STAGE, K2 after it
  static constexpr int STAGE = 2 * K_BYTES;
  static constexpr int OFF_MERGE = OFF_K + 2 * STAGE;  // [2][5][128] fp32 from group 1 (by item parity)
  static constexpr int OFF_BAR = OFF_MERGE + 2 * 5 * BM * 4;
  // bar_q, full[2], empty[2], sfull[2], sfree[2], qempty, tmem slot, abort flag
  static constexpr int BYTES = OFF_BAR + 8 * 10 + 16 + 1024;
};

struct Row5 {
  float m1, m2, l1, l2, acc;
};

// Masked logits are set to this finite sentinel (not -inf) in both S1 and S2:
// their weight 2^(c*sentinel - m) is exactly 0 and their difference S1 - S2 is
// exactly 0, so the packed arithmetic below needs no per-element selects.
constexpr float kMaskedLogit = -1.0e30f;

template <bool MASKED>
__device__ __forceinline__ void online_update(Row5& st, uint32_t (&a0)[32], uint32_t (&a1)[32], uint32_t (&b0)[32],
                                              uint32_t (&b1)[32], float c, int key0, int row_lim, int nk) {
  // a*: raw S1 = q1.k1 (64 columns), b*: raw S2; key0 = key index of column 0
  if (MASKED) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const int key = key0 + i;
      const bool keep = key < nk && key <= row_lim;
      uint32_t& s1 = i < 32 ? a0[i] : a1[i - 32];
      uint32_t& s2 = i < 32 ? b0[i] : b1[i - 32];
      if (!keep) {
        s1 = __float_as_uint(kMaskedLogit);
        s2 = __float_as_uint(kMaskedLogit);
      }
    }
  }
  const float2 cc = make_float2(c, c);
  // sums of 2^(c s - m) over the 64 columns against the maxima m1, m2
  auto tile_sums = [&](float m1, float m2, float2& l1, float2& l2, float2& acc) {
    const float2 n1 = make_float2(-m1, -m1), n2 = make_float2(-m2, -m2);
    l1 = l2 = acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const uint32_t* A = h == 0 ? a0 : a1;
        const uint32_t* Bv = h == 0 ? b0 : b1;
        const float2 s1 = make_float2(__uint_as_float(A[i]), __uint_as_float(A[i + 1]));
        const float2 s2 = make_float2(__uint_as_float(Bv[i]), __uint_as_float(Bv[i + 1]));
        const float2 x1 = ffma2(s1, cc, n1), x2 = ffma2(s2, cc, n2);
        const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
        const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
        l1 = fadd2(l1, p1);
        l2 = fadd2(l2, p2);
        acc = ffma2(p1, fsub2(s1, s2), acc);
      }
    }
  };
  float2 l1, l2, acc;
  if (st.m1 != kNegInf && st.m2 != kNegInf) {
    tile_sums(st.m1, st.m2, l1, l2, acc);
    const float t1 = l1.x + l1.y, t2 = l2.x + l2.y;
    if (t1 < kFastSumLimit && t2 < kFastSumLimit) {  // false for inf and NaN too
      st.l1 += t1;
      st.l2 += t2;
      st.acc += acc.x + acc.y;
      return;
    }
  }
  float mx1 = kMaskedLogit, mx2 = kMaskedLogit;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    mx1 = fmax3(mx1, __uint_as_float(a0[i]), __uint_as_float(a1[i]));
    mx2 = fmax3(mx2, __uint_as_float(b0[i]), __uint_as_float(b1[i]));
  }
  if (MASKED && mx1 == kMaskedLogit) return;  // every column of this tile is masked for this row
  const float t1 = mx1 * c, t2 = mx2 * c;
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
  tile_sums(st.m1, st.m2, l1, l2, acc);
  st.l1 += l1.x + l1.y;
  st.l2 += l2.x + l2.y;
  st.acc += acc.x + acc.y;
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_tc_kernel(const Problem p, float* __restrict__ out_kl, float* __restrict__ out_lse1,
                  float* __restrict__ out_lse2, float* __restrict__ out_part, int* status,
                  const __grid_constant__ CUtensorMap mq1,
                  const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mq2,
                  const __grid_constant__ CUtensorMap mk2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (p.NQ + BM - 1) / BM;
  const int items = p.BH * n_qt;
  // Item `it`: heads in order, so the blocks in flight share one head's K tiles in L2; within a head the
  // longest causal tiles first.  Block b takes the items b, b + gridDim.x, ...
  // round r of the block's walk: left to right in even rounds, right to left in odd ones, so that a block
  // that took one of the longest items of a round takes one of the shortest of the next
  auto item_at = [&](int r) {
    return r * (int)gridDim.x + ((r & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };
  auto item_of = [&](int it, int& bh, int& qt, int& n_kt) {
    bh = it / n_qt;
    qt = n_qt - 1 - it % n_qt;
    const int q_last = min(p.NQ, qt * BM + BM) - 1;
    const int kend = p.causal ? min(p.NK, q_last + p.off + 1) : p.NK;
    n_kt = kend > 0 ? (kend + BN - 1) / BN : 0;
  };

  const uint32_t bar_q = sb + L::OFF_BAR;
  const uint32_t bar_full = bar_q + 8;     // [2]
  const uint32_t bar_empty = bar_q + 24;   // [2]
  const uint32_t bar_sfull = bar_q + 40;   // [2]
  const uint32_t bar_sfree = bar_q + 56;   // [2]
  const uint32_t bar_qempty = bar_q + 72;  // Q tiles free again: the item's MMAs are done
  const uint32_t tmem_slot = bar_q + 80;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 84);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sfull + 8 * s, 1);
      mbar_init(bar_sfree + 8 * s, SOFTMAX_WARPS);
    }
    mbar_init(bar_qempty, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_BAR + 80);

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      prefetch_tensormap(&mq1);
      prefetch_tensormap(&mk1);
      prefetch_tensormap(&mq2);
      prefetch_tensormap(&mk2);
      int T = 0, k = 0;  // tiles and items issued by this block
      bool ok = true;
      for (int rr = 0, it = item_at(0); ok && it < items; it = item_at(++rr)) {
        int bh, qt, n_kt;
        item_of(it, bh, qt, n_kt);
        const int mh = bh % p.H, mb = bh / p.H;
        if (k >= 1 && !mbar_wait(bar_qempty, (k - 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(bar_q, 2 * L::Q_BYTES);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(sb + L::OFF_Q1 + h * BM * 128, &mq1, bar_q, h * 64, qt * BM, mh, mb);
          tma_load_4d(sb + L::OFF_Q2 + h * BM * 128, &mq2, bar_q, h * 64, qt * BM, mh, mb);
        }
        ++k;
        for (int j = 0; j < n_kt; ++j) {
          const int s = T & 1;
          if (T >= 2 && !mbar_wait(bar_empty + 8 * s, ((T >> 1) - 1) & 1, status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t kb = sb + L::OFF_K + s * L::STAGE;
          mbar_arrive_expect_tx(bar_full + 8 * s, L::STAGE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(kb + h * BN * 128, &mk1, bar_full + 8 * s, h * 64, j * BN, mh, mb);
            tma_load_4d(kb + L::K_BYTES + h * BN * 128, &mk2, bar_full + 8 * s, h * 64, j * BN, mh, mb);
          }
          ++T;
        }
      }
      // copies that may still be landing: the last item's Q tiles and the last two K stages
      if (k > 0) mbar_drain(bar_q, (k - 1) & 1, status);
      for (int t = max(0, T - 2); t < T; ++t) mbar_drain(bar_full + 8 * (t & 1), (t >> 1) & 1, status);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
      const uint64_t q1d = sdesc_sw128(sb + L::OFF_Q1, 0, 1024), q2d = sdesc_sw128(sb + L::OFF_Q2, 0, 1024);
      int T = 0, k = 0;
      bool ok = true;
      for (int rr = 0, it = item_at(0); ok && it < items; it = item_at(++rr), ++k) {
        int bh, qt, n_kt;
        item_of(it, bh, qt, n_kt);
        if (!mbar_wait(bar_q, k & 1, status, abort_flag)) break;
        for (int j = 0; j < n_kt; ++j) {
          const int s = T & 1;
          if (!mbar_wait(bar_full + 8 * s, (T >> 1) & 1, status, abort_flag) ||
              (T >= 2 && !mbar_wait(bar_sfree + 8 * s, ((T >> 1) - 1) & 1, status, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb1 = sb + L::OFF_K + s * L::STAGE, kb2 = kb1 + L::K_BYTES;
          const uint32_t d1 = tmem + s * 256, d2 = d1 + 128;
          const uint64_t k1d = sdesc_sw128(kb1, 0, 1024), k2d = sdesc_sw128(kb2, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (BM * 128) + (ks & 3) * 32;  // BM == BN: same half stride
            mma_ss(d1, sdesc_add(q1d, off), sdesc_add(k1d, off), idesc, ks > 0);
          }
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (BM * 128) + (ks & 3) * 32;
            mma_ss(d2, sdesc_add(q2d, off), sdesc_add(k2d, off), idesc, ks > 0);
          }
          mma_commit(bar_sfull + 8 * s);
          mma_commit(bar_empty + 8 * s);
          ++T;
        }
        if (ok) mma_commit(bar_qempty);  // this item's MMAs done: the producer may load the next Q tiles
      }
      // the last commit completes once every MMA issued here has finished
      if (T > 0) mbar_drain(bar_sfull + 8 * ((T - 1) & 1), ((T - 1) >> 1) & 1, status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax groups
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;  // row within the tile = TMEM lane
    const float c = p.c;
    int T = 0, k = 0;
    bool ok = true;
    for (int rr = 0, it = item_at(0); ok && it < items; it = item_at(++rr), ++k) {
      int bh, qt, n_kt;
      item_of(it, bh, qt, n_kt);
      const int row = qt * BM + r;
      const int row_lim = row + p.off;  // last key this row keeps when causal
      Row5 st{kNegInf, kNegInf, 0.f, 0.f, 0.f};
      for (int j = 0; j < n_kt; ++j, ++T) {
        const int s = T & 1;
        const bool got = mbar_wait_warp(bar_sfull + 8 * s, (T >> 1) & 1, status, abort_flag);
        __syncwarp();
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(wq * 32) << 16) + s * 256 + grp * 64;
        uint32_t a0[32], a1[32], b0[32], b1[32];
        tmem_ld32(ta, a0);
        tmem_ld32(ta + 32, a1);
        tmem_ld32(ta + 128, b0);
        tmem_ld32(ta + 160, b1);
        tmem_ld_wait();
        reg_fence32(a0);
        reg_fence32(a1);
        reg_fence32(b0);
        reg_fence32(b1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree + 8 * s);
        const int key0 = j * BN + grp * 64;
        const bool masked = (key0 + 63 >= p.NK) || (p.causal && key0 + 63 > row_lim);
        if (masked)
          online_update<true>(st, a0, a1, b0, b1, c, key0, p.causal ? row_lim : 0x7fffffff, p.NK);
        else
          online_update<false>(st, a0, a1, b0, b1, c, key0, 0, p.NK);
      }
      // ---- merge the two column groups, then the closing step of the forward
      float* mrg = reinterpret_cast<float*>(smem + L::OFF_MERGE) + (k & 1) * 5 * BM;
      if (grp == 1 && ok) {
        mrg[0 * BM + r] = st.m1;
        mrg[1 * BM + r] = st.m2;
        mrg[2 * BM + r] = st.l1;
        mrg[3 * BM + r] = st.l2;
        mrg[4 * BM + r] = st.acc;
      }
      // every softmax warp reaches this barrier once per item; a warp whose wait gave up makes them all stop
      if (named_bar_any(1, SOFTMAX_WARPS * 32, !ok)) break;
      if (grp == 0 && !*abort_flag && row < p.NQ) {
        const float om1 = mrg[r], om2 = mrg[BM + r], ol1 = mrg[2 * BM + r], ol2 = mrg[3 * BM + r],
                    oacc = mrg[4 * BM + r];
        const float M1 = fmaxf(st.m1, om1), M2 = fmaxf(st.m2, om2);
        // both groups empty only for a row that sees no key of a shard
        const float wa1 = M1 == kNegInf ? 0.f : ex2(st.m1 - M1), wb1 = M1 == kNegInf ? 0.f : ex2(om1 - M1);
        const float wa2 = M2 == kNegInf ? 0.f : ex2(st.m2 - M2), wb2 = M2 == kNegInf ? 0.f : ex2(om2 - M2);
        const float l1 = st.l1 * wa1 + ol1 * wb1, acc = st.acc * wa1 + oacc * wb1;
        const float l2 = st.l2 * wa2 + ol2 * wb2;
        const size_t o = (size_t)bh * p.NQ + row;
        if (out_part) {  // the row's five scalars over this shard's keys: m in log2 units, acc unscaled
          float* d = out_part + o * 5;
          d[0] = M1;
          d[1] = M2;
          d[2] = l1;
          d[3] = l2;
          d[4] = acc;
        } else {
          const float lse1 = (M1 + log2f(l1)) * kLn2;
          const float lse2 = (M2 + log2f(l2)) * kLn2;
          out_lse1[o] = lse1;
          out_lse2[o] = lse2;
          out_kl[o] = p.scale * (acc / l1) + lse2 - lse1;
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

template <int D>
cudaError_t launch_d(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2, float* kl,
                     float* lse1, float* lse2, float* part, int* status, cudaStream_t st) {
  CUtensorMap mq1, mk1, mq2, mk2;
  if (!encode_q_map(&mq1, q1, p, BM) || !encode_q_map(&mq2, q2, p, BM) ||
      !encode_k_map(&mk1, k1, p, BN) || !encode_k_map(&mk2, k2, p, BN))
    return cudaErrorInvalidValue;
  // A block owns all 512 TMEM columns: ask for enough shared memory that a
  // second block never shares the SM (it would only wait in tcgen05.alloc).
  const int smem = Smem<D>::BYTES > kOneBlockPerSmSmem ? Smem<D>::BYTES : kOneBlockPerSmSmem;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long items = (long long)p.BH * ((p.NQ + BM - 1) / BM);
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // Short items in few rounds per SM: one block per SM walks them (the per-block set-up is paid once, and an
  // item's closing step overlaps the next item's loads).  Otherwise one block per item, so that the hardware's
  // block scheduler balances the causal triangle and the blocks in flight stay on one head.  Measured: the
  // static walk is 6-8% faster on B2 H32 N4096 (32 key tiles, 13.5 rounds), 5% slower on B1 H4 N64K causal
  // (512 key tiles, 13.5 rounds) and 2% slower on B1 H32 N64K causal (108 rounds).
  const long long rounds = (items + sms - 1) / sms;
  const long long key_tiles = (p.NK + BN - 1) / BN;
  const bool walk = rounds <= kMaxPersistentRounds && key_tiles <= kMaxPersistentKeyTiles;
  const long long blocks = walk ? (items < sms ? items : sms) : items;
  fwd_tc_kernel<D><<<(unsigned)blocks, THREADS, smem, st>>>(p, kl, lse1, lse2, part, status, mq1, mk1, mq2, mk2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                       float* kl, float* lse1, float* lse2, int* status, cudaStream_t st) {
  if (p.D == 64) return launch_d<64>(p, q1, k1, q2, k2, kl, lse1, lse2, nullptr, status, st);
  return launch_d<128>(p, q1, k1, q2, k2, kl, lse1, lse2, nullptr, status, st);
}

cudaError_t launch_fwd_partials(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                                float* partials, int* status, cudaStream_t st) {
  if (p.D == 64) return launch_d<64>(p, q1, k1, q2, k2, nullptr, nullptr, nullptr, partials, status, st);
  return launch_d<128>(p, q1, k1, q2, k2, nullptr, nullptr, nullptr, partials, status, st);
}

}  // namespace skl
