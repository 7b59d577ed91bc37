// Fused attention-KL backward on the 5th-generation tensor cores.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), section 手法 2
// "kernel fusion": each (query tile, key tile) pair is visited exactly once.
// Here the query tile is stationary: dQ accumulates in TMEM along the keys, and
// the dK partial of each key tile is added into an fp32 buffer with atomics,
// which stay cheap while the rows being accumulated sit in L2.  For long key
// sequences the host runs the kernel once per key range sized to keep them
// there, summing dQ over the ranges in fp32 (KeyRange below).  dS arithmetic in
// ds_math.cuh (setting 1: dS2 = g (P2 - P1); setting 2: dS1 = g P1 (r - KL)).
//
// Block = one 128-query tile (stationary Q1, Q2 in smem; queries on the 128 TMEM
// lanes), streaming 128-key tiles.  Every MMA is M = 128, N = 128 (a single-CTA
// M128 K16 MMA runs 48 cycles at N = 64 and 64 at N = 128, the full tensor rate):
//   S_a = Q_a K_a^T, then S_b = Q_b K_b^T  SS, K-major, both into TMEM columns [0, 128);
//                                          b = opt (2 in setting 1, 1 in setting 2), a = the other
//   dS from S and the row's folded LSE1, LSE2, g, KL; to smem as dS[query][key]
//   dQ   += dS K_opt                    SS: A = dS (K-major over keys), B = K_opt MN-major  -> [128, 128 + D)
//   dKp^T = Q_opt^T dS                  SS: A = Q_opt read MN-major (M = d), B = dS MN-major -> [256 + 128 b, ...)
//   dk_acc[key, d] += dKp^T[d, key]     staged in smem 32 keys at a time, added by a TMA bulk tensor
//                                       reduction (cp.reduce.async.bulk.tensor .add.f32)
// Two threads issue the MMAs, each from its own warp: one the logits S_a(j),
// S_b(j) of every key tile, the other the gradient MMAs dQ(j), dKp(j) once dS(j)
// is in shared memory.  A tcgen05.mma takes a single issuing thread several
// tens of cycles to issue, close to the 64 cycles an M128 N128 K16 MMA runs,
// so one thread that also waits on every hand-off leaves the tensor pipe idle;
// two threads on different SMSPs keep it fed, and a gradient MMA waiting for
// its dK buffer no longer holds up the next tile's logits.  The gradient thread
// issues dKp(j) only once S_b(j + 1) is queued (pipe order S_a(j + 1), dQ(j),
// S_b(j + 1), dKp(j)), so the logits the dS warps wait for come first.
// The dS warps copy S_a into registers (in setting 1 they turn it into P1 while
// S_b is in flight), S_b is written over it and read in two halves.  A thread
// owns a query row, so its per-query values sit in registers
// and the dS loop issues no shared-memory loads.  dKp^T is double-buffered so
// the dK warps have two tile periods per tile.  They read it from TMEM, write
// each 32-key chunk into a shared buffer as [key][d] fp32 and one thread adds
// the chunk into the fp32 accumulator with a TMA bulk reduction: 64 KB of
// dK partial per tile would otherwise take 512 warp-wide red.global
// instructions through the load/store path, which measured 14% of the kernel
// (a timing-only copy without them ran B1 H32 N64K causal in 50.6 against
// 59.4 ms; plain stores in their place cost as much as the reductions).  The
// chunk buffers take the second slot of the other K tile's ring (B1 H32:
// 59.4 -> 58.1 ms; setting 2 at H8 14.87 -> 14.16).
//   warps 0-15  dS warps: thread = query row (lane quarter = warp % 4), group g = warp / 4
//               takes key columns [32g, 32g + 32); at the end they write dQ
//   warp 16     TMA producer: Q1, Q2 once, the other K tile through one slot
//   warp 17     TMEM owner and issuer of the logits MMAs
//   warp 18     TMA producer of K_opt (two slots, each held until the gradient MMAs)
//   warp 19     issuer of the gradient MMAs
//   warps 20-27 dK warps: thread = column d of dKp^T (lane quarter = warp % 4), warps
//               20-23 take keys [0, 64) of a tile and 24-27 keys [64, 128), each group
//               with its own 16 KB chunk buffer
// Warpgroups 4-6 give registers to the dS warpgroups (setmaxnreg).
#include <algorithm>

#include "common.cuh"
#include "ds_math.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skl {
namespace {

constexpr int BQ = 128;  // queries per block (M of the S and dQ MMAs)
constexpr int BK = 128;  // keys per step (N of the S and dKp MMAs)
constexpr int SLOTS = 2;     // K_opt slots
constexpr int KT_SLOTS = 1;  // slots of the other K tile
constexpr int STG_ROWS = 32; // keys per staged dK chunk
constexpr int DS_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int KOPT_WARP = 18;
constexpr int GRAD_WARP = 19;
constexpr int DK_WARP0 = 20;
constexpr int DK_WARPS = 8;
constexpr int THREADS = 28 * 32;
constexpr int kRegsDs = 80, kRegsOther = 56;  // 512 * 80 + 384 * 56 <= 896 * 72 registers at launch
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDQ = 128, kColDK = 256;  // dKp^T buffer b at kColDK + 128 b

template <int D>
struct Smem {
  static constexpr int TQ = BQ * D * 2;  // one 128-row tile (D/64 halves of [128][128 B])
  static constexpr int TK = BK * D * 2;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = TQ;
  static constexpr int OFF_KO = 2 * TQ;              // K_opt slots
  static constexpr int OFF_KT = OFF_KO + SLOTS * TK;  // the other K tile's slots
  static constexpr int STG = STG_ROWS * D * 4;        // one staged dK chunk: [32 keys][D] fp32
  static constexpr int OFF_STG = OFF_KT + KT_SLOTS * TK;  // two chunk buffers (one per dK warp group)
  static constexpr int OFF_DS = OFF_STG + 2 * STG;    // dS[query][key] bf16: 2 halves of [128 queries][128 B]
  static constexpr int DS_BYTES = BQ * BK * 2;
  static constexpr int OFF_BAR = OFF_DS + DS_BYTES;
  // mbarriers (8 B each): q_full, ko_full[2], ko_empty[2] (S_b and dQ both arrive), kt_full[2] and
  // kt_empty[2] (the first KT_SLOTS used), sa_full, sa_free, sb_full, sb_free, ds_full, ds_free, dk_full[2], dk_free[2],
  // all_done, sb_issued; then the TMEM base address slot and the abort flag
  static constexpr int BAR_SLOT = 21 * 8;
  static constexpr int BYTES = OFF_BAR + BAR_SLOT + 16 + 1024;
};
static_assert(Smem<128>::BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ void setmaxnreg_inc_ds() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
}
__device__ __forceinline__ void setmaxnreg_dec_other() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

// One launch covers the key tiles [jt0, jt1) and the query tiles from qt_min on
// (those that see a key of the range).  dK partials go to the range's rows of
// dk_acc ([B*H][dk_rows][D] fp32, row = key - 128 jt0).  dQ: DQ_BF16 writes the
// finished bf16 gradient (the range is every key), DQ_STORE / DQ_ADD store or
// add the unscaled fp32 sum over the range into dq_acc ([B*H][N_Q][D]).
enum { DQ_BF16 = 0, DQ_STORE = 1, DQ_ADD = 2 };
struct KeyRange {
  int jt0, jt1, qt_min, dq_mode, dk_rows;
  float* dq_acc;
};

template <int D, int SETTING>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_fused_tc_kernel(const Problem p, const KeyRange kr, const float* __restrict__ lse1,
                        const float* __restrict__ lse2, const float* __restrict__ klv,
                        const float* __restrict__ gv, __nv_bfloat16* __restrict__ dq_out,
                        float* __restrict__ dk_acc, int* status,
                        const __grid_constant__ CUtensorMap mq1, const __grid_constant__ CUtensorMap mq2,
                        const __grid_constant__ CUtensorMap mk1, const __grid_constant__ CUtensorMap mk2,
                        const __grid_constant__ CUtensorMap mdk) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (p.NQ + BQ - 1) / BQ;
  const int n_qt_r = n_qt - kr.qt_min;                   // query tiles that see this key range
  const int bh = (int)(blockIdx.x / n_qt_r);             // heads in order (their dk_acc rows stay in L2), ...
  const int qt = n_qt - 1 - (int)(blockIdx.x % n_qt_r);  // ... and within a head the longest (last) query tiles first
  const int mh = bh % p.H, mb = bh / p.H;  // head and batch coordinates of the tensor maps
  const int q0 = qt * BQ;
  const int q_last = min(p.NQ, q0 + BQ) - 1;
  const int kend = min(p.causal ? min(p.NK, q_last + p.off + 1) : p.NK, kr.jt1 * BK);
  const int n_kt = (kend + BK - 1) / BK - kr.jt0;  // >= 1: qt >= qt_min sees key 128 jt0
  const int kbase = kr.jt0 * BK;                   // first key of the range; local tile j = keys kbase + 128 j

  const uint32_t bar = sb + L::OFF_BAR;
  const uint32_t q_full = bar, ko_full = bar + 8, ko_empty = bar + 24, kt_full = bar + 40, kt_empty = bar + 56,
                 sa_full = bar + 72, sa_free = bar + 80, sb_full = bar + 88, sb_free = bar + 96, ds_full = bar + 104,
                 ds_free = bar + 112, dk_full = bar + 120, dk_free = bar + 136, all_done = bar + 152, sb_issued = bar + 160,
                 slot = bar + L::BAR_SLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + L::BAR_SLOT + 4);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(ko_full + 8 * s, 1);
      mbar_init(ko_empty + 8 * s, 2);
      mbar_init(kt_full + 8 * s, 1);
      mbar_init(kt_empty + 8 * s, 1);
    }
    mbar_init(sa_full, 1);
    mbar_init(sa_free, DS_WARPS);
    mbar_init(sb_full, 1);
    mbar_init(sb_free, DS_WARPS);
    mbar_init(ds_full, DS_WARPS);
    mbar_init(ds_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(dk_full + 8 * b, 1);
      mbar_init(dk_free + 8 * b, DK_WARPS);
    }
    mbar_init(all_done, 1);
    mbar_init(sb_issued, 1);
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

  // opt side: 2 in setting 1 (dQ2, dK2), 1 in setting 2; "a" is the other side
  constexpr int OFF_QA = SETTING == 1 ? L::OFF_Q1 : L::OFF_Q2, OFF_QB = SETTING == 1 ? L::OFF_Q2 : L::OFF_Q1;

  if (warp >= DS_WARPS) {
    setmaxnreg_dec_other();
    if (warp == PRODUCER_WARP) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, 2 * L::TQ);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(sb + L::OFF_Q1 + h * BQ * 128, &mq1, q_full, h * 64, q0, mh, mb);
          tma_load_4d(sb + L::OFF_Q2 + h * BQ * 128, &mq2, q_full, h * 64, q0, mh, mb);
        }
        const CUtensorMap* mka = SETTING == 1 ? &mk1 : &mk2;
        int issued = 0;
        for (int j = 0; j < n_kt; ++j) {
          const int s = j % KT_SLOTS;
          if (j >= KT_SLOTS && !mbar_wait(kt_empty + 8 * s, ((j / KT_SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(kt_full + 8 * s, L::TK);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_KT + s * L::TK + h * BK * 128, mka, kt_full + 8 * s, h * 64, kbase + j * BK, mh,
                        mb);
          issued = j + 1;
        }
        mbar_drain(q_full, 0, status);
        for (int j = max(0, issued - KT_SLOTS); j < issued; ++j)
          mbar_drain(kt_full + 8 * (j % KT_SLOTS), (j / KT_SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == KOPT_WARP) {
      // ------------------------------------------------------------------ TMA producer of K_opt
      // A stream of its own: its slots free only after the gradient MMAs, and the
      // other K tile must not wait behind it.
      if (lane == 0) {
        const CUtensorMap* mkb = SETTING == 1 ? &mk2 : &mk1;
        int issued = 0;
        for (int j = 0; j < n_kt; ++j) {
          const int s = j % SLOTS;
          if (j >= SLOTS && !mbar_wait(ko_empty + 8 * s, ((j / SLOTS) - 1) & 1, status, abort_flag)) break;
          mbar_arrive_expect_tx(ko_full + 8 * s, L::TK);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sb + L::OFF_KO + s * L::TK + h * BK * 128, mkb, ko_full + 8 * s, h * 64, kbase + j * BK, mh,
                        mb);
          issued = j + 1;
        }
        for (int j = max(0, issued - SLOTS); j < issued; ++j)
          mbar_drain(ko_full + 8 * (j % SLOTS), (j / SLOTS) & 1, status);
      }
      __syncwarp();
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------------ MMA issuer: logits
      // S_a(j) once the dS warps have read S_b(j - 1) out of the shared region,
      // S_b(j) once they hold S_a(j).
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16(BQ, BK, false, false);
        const uint64_t qad = sdesc_sw128(sb + OFF_QA, 0, 1024), qbd = sdesc_sw128(sb + OFF_QB, 0, 1024);
        bool ok = mbar_wait(q_full, 0, status, abort_flag);
        for (int j = 0; ok && j < n_kt; ++j) {
          const int s = j % SLOTS, st = j % KT_SLOTS;
          if (!mbar_wait(kt_full + 8 * st, (j / KT_SLOTS) & 1, status, abort_flag)) break;
          if (j >= 1 && !mbar_wait(sb_free, (j - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          const uint64_t kad = sdesc_sw128(sb + L::OFF_KT + st * L::TK, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;  // BQ == BK: same half stride
            mma_ss(tmem + kColS, sdesc_add(qad, off), sdesc_add(kad, off), id_s, ks > 0);
          }
          mma_commit(sa_full);
          mma_commit(kt_empty + 8 * st);  // the other K tile is read only by S_a
          if (!mbar_wait(sa_free, j & 1, status, abort_flag)) break;
          if (!mbar_wait(ko_full + 8 * s, (j / SLOTS) & 1, status, abort_flag)) break;
          tc_fence_after();
          const uint64_t kbd = sdesc_sw128(sb + L::OFF_KO + s * L::TK, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
            mma_ss(tmem + kColS, sdesc_add(qbd, off), sdesc_add(kbd, off), id_s, ks > 0);
          }
          mma_commit(sb_full);
          mma_commit(ko_empty + 8 * s);  // first of the two arrivals that free K_opt(j)
          mbar_arrive(sb_issued);        // S_b(j) is in the tensor pipe's queue
        }
      }
      __syncwarp();
    } else if (warp == GRAD_WARP) {
      // ------------------------------------------------------------------ MMA issuer: gradients
      // dQ(j) and dKp(j) once dS(j) is in shared memory; dKp(j) also waits for
      // its TMEM buffer (tile j - 2's) to be drained by the dK warps, and for the
      // logits thread to have issued S_b(j + 1), so that the pipe runs S_a(j + 1),
      // dQ(j), S_b(j + 1), dKp(j): the dS warps, which wait for S_b after copying
      // S_a, find it behind one gradient MMA instead of two (measured: B1 H32 N64K
      // causal 62.3 -> 59.8 ms; holding dQ(j) back as well made it 71.2 ms).
      if (lane == 0) {
        constexpr uint32_t id_dq = idesc_bf16(BQ, D, false, true);
        constexpr uint32_t id_dk = idesc_bf16(128, BK, true, true);
        const uint64_t qod = sdesc_sw128(sb + OFF_QB, D == 128 ? BQ * 128 : 0, 1024);  // Q_opt as MN-major A
        const uint64_t dsk = sdesc_sw128(sb + L::OFF_DS, 0, 1024);         // dS as A of dQ (K-major over keys)
        const uint64_t dsm = sdesc_sw128(sb + L::OFF_DS, BQ * 128, 1024);  // dS as B of dKp (MN-major over keys)
        bool ok = mbar_wait(q_full, 0, status, abort_flag);
        for (int j = 0; ok && j < n_kt; ++j) {
          const int s = j % SLOTS, b = j & 1;
          if (!mbar_wait(ds_full, j & 1, status, abort_flag)) break;
          // K_opt(j) has landed (S_b(j) read it before dS(j) existed); waited here too so that this
          // thread's MMAs are ordered after the copy
          if (!mbar_wait(ko_full + 8 * s, (j / SLOTS) & 1, status, abort_flag)) break;
          tc_fence_after();
          // dQ += dS K_opt: A = dS[query][key] K-major (key k-steps), B = K_opt read MN-major
          const uint64_t kod = sdesc_sw128(sb + L::OFF_KO + s * L::TK, BK * 128, 1024);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            mma_ss(tmem + kColDQ, sdesc_add(dsk, (ks >> 2) * (BQ * 128) + (ks & 3) * 32), sdesc_add(kod, ks * 2048),
                   id_dq, j > 0 || ks > 0);
          mma_commit(ko_empty + 8 * s);  // second arrival: K_opt(j) was read by S_b(j) and this dQ
          if (j + 1 < n_kt && !mbar_wait(sb_issued, (j + 1) & 1, status, abort_flag)) break;
          // dKp^T buffer b was drained (tile j - 2) by the dK warps
          if (j >= 2 && !mbar_wait(dk_free + 8 * b, ((j >> 1) - 1) & 1, status, abort_flag)) break;
          tc_fence_after();
          // dKp^T = Q_opt^T dS: A = Q_opt (queries x d) read MN-major, B = dS (queries x keys) MN-major
#pragma unroll
          for (int ks = 0; ks < BQ / 16; ++ks)
            mma_ss(tmem + kColDK + 128 * b, sdesc_add(qod, ks * 2048), sdesc_add(dsm, ks * 2048), id_dk, ks > 0);
          mma_commit(ds_free);
          mma_commit(dk_full + 8 * b);
        }
        // every gradient MMA done: arrives on all_done (waited by the dQ epilogue and below)
        mma_commit(all_done);
        mbar_drain(all_done, 0, status);
      }
      __syncwarp();
    } else if (warp >= DK_WARP0) {
      // ------------------------------------------------------------------ dK warps
      // Group h (warps 20-23: keys [0, 64) of a tile, warps 24-27: keys [64, 128)) stages each 32-key chunk of
      // the dKp^T tile in its own shared buffer as [key][d] fp32 and one thread adds the chunk into dk_acc with
      // a TMA bulk tensor reduction (rows past the range's end are clipped by the map).
      const int wq = (warp - DK_WARP0) & 3, half = (warp - DK_WARP0) >> 2;
      const int d = wq * 32 + lane;  // lane of dKp^T = column d
      const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
      const uint32_t stg = sb + L::OFF_STG + half * L::STG;
      const bool leader = wq == 0 && lane == 0;
      for (int j = 0; j < n_kt; ++j) {
        const int b = j & 1;
        const bool got = mbar_wait_warp(dk_full + 8 * b, (j >> 1) & 1, status, abort_flag);
        // the group's four warps stop together (they share named barriers below)
        if (named_bar_any(2 + half, 128, !got)) break;
        tc_fence_after();
#pragma unroll 1
        for (int cb = 2 * half; cb < 2 * half + 2; ++cb) {  // this group's half of the keys
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kColDK + 128 * b + 32 * cb, v);
          tmem_ld_wait();
          reg_fence32(v);
          if (cb == 2 * half + 1) {
            // this warp's half of the dKp^T tile has been read: once all eight warps have, the
            // dKp MMA of tile j + 2 may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dk_free + 8 * b);
          }
          // the group's buffer is free once the previous reduction from it has read it
          if (leader) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          named_bar_sync(2 + half, 128);
          if (d < D) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg + (uint32_t)(i * D + d) * 4), "r"(v[i]) : "memory");
          }
          fence_async_smem();
          named_bar_sync(2 + half, 128);
          const int row0 = j * BK + 32 * cb;  // first accumulator row of the chunk within the head
          if (leader && row0 < kr.dk_rows) {  // a chunk wholly past the range's rows has nothing to add
            asm volatile(
                "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                ::"l"(reinterpret_cast<uint64_t>(&mdk)), "r"(0), "r"(row0), "r"(bh), "r"(stg)
                : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      }
      if (leader) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
  } else {
    setmaxnreg_inc_ds();
    // ------------------------------------------------------------------ dS warps
    const int grp = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int row = q0 + r;
    const float c = p.c;
    float nAr = 0.f, nBr = 0.f, Gr = 0.f;  // the row's folded values
    if (row < p.NQ) {
      const size_t o = (size_t)bh * p.NQ + row;
      const float l1v = lse1[o], l2v = lse2[o];
      nAr = -l1v * kLog2e;
      nBr = SETTING == 1 ? -l2v * kLog2e : -(l1v - l2v + klv[o]);
      Gr = gv[o];
    }
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tcol = tmem + lane_base + kColS + grp * 32;
    const uint32_t dsb = sb + L::OFF_DS;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      ok = mbar_wait_warp(sa_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      uint32_t held[32];  // this thread's 32 columns of S_a
      tmem_ld32(tcol, held);
      tmem_ld_wait();
      reg_fence32(held);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sa_free);
      const int kg = kbase + j * BK + grp * 32;
      const bool masked = (kg + 31 >= p.NK) || (row >= p.NQ) || (p.causal && kg + 31 > row + p.off);
      const uint32_t vis = masked ? visible_keys<16>(row, kg, p.NQ, p.NK, p.off, p.causal) |
                                        (visible_keys<16>(row, kg + 16, p.NQ, p.NK, p.off, p.causal) << 16)
                                  : ~0u;
      if (SETTING == 1) {
        // P1 needs S_a (= S1) alone: computed in place while S_b is computed
        if (masked)
          p1_row<true, 32>(held, c, nAr, vis);
        else
          p1_row<false, 32>(held, c, nAr, 0u);
      }
      uint32_t pk[16];
      ok = mbar_wait_warp(sb_full, j & 1, status, abort_flag);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      // S_b in two halves of 16 columns; TMEM is released once both are in registers
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t half[16];
        tmem_ld16(tcol + 16 * h, half);
        tmem_ld_wait();
        reg_fence16(half);
        if (h == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sb_free);
        }
        const uint32_t(&ha)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&held[16 * h]);
        if (SETTING == 1) {  // S_b = S2; held = P1
          if (masked)
            ds1_from_p1<true, 16>(half, ha, pk + 8 * h, c, nBr, Gr, vis >> (16 * h));
          else
            ds1_from_p1<false, 16>(half, ha, pk + 8 * h, c, nBr, Gr, 0u);
        } else {  // S_a = S2, S_b = S1
          if (masked)
            make_ds_row<SETTING, true, 16>(half, ha, pk + 8 * h, c, p.scale, nAr, nBr, Gr, vis >> (16 * h));
          else
            make_ds_row<SETTING, false, 16>(half, ha, pk + 8 * h, c, p.scale, nAr, nBr, Gr, 0u);
        }
        if (h == 0)  // first half final before the second half is read
          asm volatile("" : "+r"(pk[0]), "+r"(pk[1]), "+r"(pk[2]), "+r"(pk[3]), "+r"(pk[4]), "+r"(pk[5]),
                       "+r"(pk[6]), "+r"(pk[7])::"memory");
      }
      reg_fence16(pk);
      // dS smem is free once the dQ and dKp MMAs of the previous tile are done
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
    }
    // ---- dQ out: group g writes d columns [32g, 32g + 32)
    const bool done = mbar_wait_warp(all_done, 0, status, abort_flag);
    __syncwarp();
    if (done && grp * 32 < D) {
      tc_fence_after();
      uint32_t g0[32];
      tmem_ld32(tmem + lane_base + kColDQ + grp * 32, g0);
      tmem_ld_wait();
      reg_fence32(g0);
      if (row < p.NQ && kr.dq_mode == DQ_BF16) {
        __nv_bfloat16* dst = dq_out + row_offset(bh, p.H, row, p.qs_b, p.qs_h, p.qs_n) + grp * 32;
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
      } else if (row < p.NQ) {
        float4* dst = reinterpret_cast<float4*>(kr.dq_acc + ((size_t)bh * p.NQ + row) * D + grp * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          float4 o = make_float4(__uint_as_float(g0[4 * v]), __uint_as_float(g0[4 * v + 1]),
                                 __uint_as_float(g0[4 * v + 2]), __uint_as_float(g0[4 * v + 3]));
          if (kr.dq_mode == DQ_ADD) {
            const float4 a = dst[v];
            o.x += a.x;
            o.y += a.y;
            o.z += a.z;
            o.w += a.w;
          }
          dst[v] = o;
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
cudaError_t launch_fused(const Problem& p, const KeyRange& kr, const BwdIn& in, void* dq, float* dk_acc, int* status,
                         cudaStream_t st) {
  CUtensorMap mq1, mq2, mk1, mk2;
  if (!encode_q_map(&mq1, in.q1, p, BQ) || !encode_q_map(&mq2, in.q2, p, BQ) ||
      !encode_k_map(&mk1, in.k1, p, BK) || !encode_k_map(&mk2, in.k2, p, BK))
    return cudaErrorInvalidValue;
  const int smem = Smem<D>::BYTES > kOneBlockPerSmSmem ? Smem<D>::BYTES : kOneBlockPerSmSmem;
  auto kern = bwd_fused_tc_kernel<D, SETTING>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.BH * ((p.NQ + BQ - 1) / BQ - kr.qt_min);
  CUtensorMap mdk;
  if (!encode_rows_f32_map(&mdk, dk_acc, D, kr.dk_rows, p.BH, STG_ROWS)) return cudaErrorInvalidValue;
  kern<<<(unsigned)blocks, THREADS, smem, st>>>(p, kr, in.lse1, in.lse2, in.kl, in.g,
                                                static_cast<__nv_bfloat16*>(dq), dk_acc, status, mq1, mq2, mk1, mk2,
                                                mdk);
  return cudaGetLastError();
}

// out row (row0 + r) of head bh = bf16(scale * acc[bh][r]) for r < nrows, with
// the output's strides (sb, sh, sn); acc holds acc_rows fp32 rows of D per head.
// One thread converts 8 values.
template <int D>
__global__ void __launch_bounds__(256)
    acc_convert_kernel(const float4* __restrict__ acc, __nv_bfloat16* __restrict__ out, const int H,
                       const int acc_rows, const int row0, const int nrows, const long long sb, const long long sh,
                       const long long sn, const float scale, const size_t n8) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const size_t rr = i / (D / 8);
    const int d = (int)(i % (D / 8)) * 8;
    const int bh = (int)(rr / (size_t)nrows), r = (int)(rr % (size_t)nrows);
    const size_t a = (((size_t)bh * acc_rows + r) * D + d) / 4;
    const float4 x = acc[a], y = acc[a + 1];
    uint4 o;
    o.x = pack_bf16(x.x * scale, x.y * scale);
    o.y = pack_bf16(x.z * scale, x.w * scale);
    o.z = pack_bf16(y.x * scale, y.y * scale);
    o.w = pack_bf16(y.z * scale, y.w * scale);
    *reinterpret_cast<uint4*>(out + row_offset(bh, H, row0 + r, sb, sh, sn) + d) = o;
  }
}

template <int D>
cudaError_t convert_rows(const float* acc, void* out, const Problem& p, int acc_rows, int row0, int nrows, long long sb,
                         long long sh, long long sn, cudaStream_t st) {
  const size_t n8 = (size_t)p.BH * nrows * (D / 8);
  if (n8 == 0) return cudaSuccess;
  const int blocks = (int)((n8 + 255) / 256 < 4096 ? (n8 + 255) / 256 : 4096);
  acc_convert_kernel<D><<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                                static_cast<__nv_bfloat16*>(out), p.H, acc_rows, row0, nrows, sb, sh,
                                                sn, p.scale, n8);
  return cudaGetLastError();
}

// First query tile whose rows see key k0 (causal: row i keeps keys j <= i + off).
int first_qtile(const Problem& p, long long k0) {
  if (!p.causal) return 0;
  const long long need = k0 - p.off;  // the tile's last row must reach this
  if (need <= 0) return 0;
  return (int)((need + 1 + BQ - 1) / BQ - 1);
}

template <int D>
cudaError_t fused_d(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, float* ws, int range_tiles,
                    int* status, cudaStream_t st, float* dq_f32) {
  const int n_kt = (p.NK + BK - 1) / BK;
  const int n_ranges = (n_kt + range_tiles - 1) / range_tiles;
  const int dk_rows = std::min(range_tiles * BK, p.NK);
  float* dk_acc = ws;
  float* dq_acc = dq_f32 ? dq_f32 : (n_ranges > 1 ? ws + (size_t)p.BH * dk_rows * D : nullptr);
  if (dq_f32) {
    // every range adds into the caller's buffer: query tiles that see no key of these keys stay zero
    cudaError_t e = cudaMemsetAsync(dq_f32, 0, (size_t)p.BH * p.NQ * D * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  for (int r = 0; r < n_ranges; ++r) {
    const int jt0 = r * range_tiles, jt1 = std::min(n_kt, jt0 + range_tiles);
    const int k0 = jt0 * BK, nk = std::min(p.NK, jt1 * BK) - k0;
    cudaError_t e = cudaMemsetAsync(dk_acc, 0, (size_t)p.BH * dk_rows * D * sizeof(float), st);
    if (e != cudaSuccess) return e;
    const int dq_mode = dq_f32 ? DQ_ADD : (n_ranges == 1 ? DQ_BF16 : (r == 0 ? DQ_STORE : DQ_ADD));
    const KeyRange kr{jt0, jt1, first_qtile(p, k0), dq_mode, dk_rows, dq_acc};
    e = setting == 1 ? launch_fused<D, 1>(p, kr, in, dq, dk_acc, status, st)
                     : launch_fused<D, 2>(p, kr, in, dq, dk_acc, status, st);
    if (e != cudaSuccess) return e;
    e = convert_rows<D>(dk_acc, dk, p, dk_rows, k0, nk, p.ks_b, p.ks_h, p.ks_n, st);
    if (e != cudaSuccess) return e;
  }
  if (!dq_f32 && n_ranges > 1) return convert_rows<D>(dq_acc, dq, p, p.NQ, 0, p.NQ, p.qs_b, p.qs_h, p.qs_n, st);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_fused(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, float* workspace,
                             int range_tiles, int* status, cudaStream_t st, float* dq_f32) {
  if (p.D == 64) return fused_d<64>(p, setting, in, dq, dk, workspace, range_tiles, status, st, dq_f32);
  return fused_d<128>(p, setting, in, dq, dk, workspace, range_tiles, status, st, dq_f32);
}

// Zeroes rows [0, nrows) of every head of a bf16 [B, H, N, D] view with strides (sb, sh, sn): one thread
// writes 8 values.
template <int D>
__global__ void __launch_bounds__(256)
    zero_rows_kernel(__nv_bfloat16* __restrict__ out, const int H, const int nrows, const long long sb,
                     const long long sh, const long long sn, const size_t n8) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const size_t rr = i / (D / 8);
    const int d = (int)(i % (D / 8)) * 8;
    const int bh = (int)(rr / (size_t)nrows), r = (int)(rr % (size_t)nrows);
    *reinterpret_cast<uint4*>(out + row_offset(bh, H, r, sb, sh, sn) + d) = make_uint4(0, 0, 0, 0);
  }
}

template <int D>
cudaError_t zero_k_rows(const Problem& p, void* dk, cudaStream_t st) {
  const size_t n8 = (size_t)p.BH * p.NK * (D / 8);
  if (n8 == 0) return cudaSuccess;
  const int blocks = (int)((n8 + 255) / 256 < 4096 ? (n8 + 255) / 256 : 4096);
  zero_rows_kernel<D><<<blocks, 256, 0, st>>>(static_cast<__nv_bfloat16*>(dk), p.H, p.NK, p.ks_b, p.ks_h, p.ks_n,
                                             n8);
  return cudaGetLastError();
}

cudaError_t launch_zero_k_rows(const Problem& p, void* dk, cudaStream_t st) {
  return p.D == 64 ? zero_k_rows<64>(p, dk, st) : zero_k_rows<128>(p, dk, st);
}

cudaError_t launch_rows_to_bf16(const Problem& p, const float* acc, void* out, cudaStream_t st) {
  if (p.D == 64) return convert_rows<64>(acc, out, p, p.NQ, 0, p.NQ, p.qs_b, p.qs_h, p.qs_n, st);
  return convert_rows<128>(acc, out, p, p.NQ, 0, p.NQ, p.qs_b, p.qs_h, p.qs_n, st);
}

int fused_first_qtile(const Problem& p, long long k0) { return first_qtile(p, k0); }

}  // namespace skl
