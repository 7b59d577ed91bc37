// Element-wise dS of the attention-KL backward, shared by the fused and the
// separate tcgen05 kernels.
//
// StreamKL technical summary (gist.science/ja/paper/2606.20005), sections 手法 2
// "recompute strategy" (P_t = exp(S_t - LSE_t) rebuilt per tile) and 手法 3
// "numerical stability" (the setting-2 log ratio from logits and saved LSEs).
// With L = sum_i g_i KL_i (chain rule, derived):
//     setting 1:  dS2 = g (P2 - P1)
//     setting 2:  dS1 = g P1 (r - KL),  r = (S1 - LSE1) - (S2 - LSE2)
// Per-query values are folded so that each logit needs one packed FMA, in log2
// units (c = scale log2(e)):
//     nA = -LSE1 log2(e)
//     nB = -LSE2 log2(e)                 (setting 1)
//          -(LSE1 - LSE2 + KL)           (setting 2: r - KL = scale (S1 - S2) + nB)
//     G  = g
// so P1 = 2^(c S1 + nA), P2 = 2^(c S2 + nB).
#pragma once

#include "common.cuh"

namespace skl {

// Bit k set iff key column k0 + k (k < N <= 16) is seen by query `q`.
template <int N>
__device__ __forceinline__ uint32_t visible_keys(int q, int k0, int nq, int nk, int off, int causal) {
  if (q >= nq) return 0u;
  const int kend = causal ? min(nk, q + off + 1) : nk;
  const int hi = min(max(kend - k0, 0), N);
  return hi > 0 ? (1u << hi) - 1u : 0u;
}

// One dS element pair from the two logit pairs and the folded values; with
// MASKED, an element whose bit in `visible` (at position k, k + 1) is clear is 0.
template <int SETTING, bool MASKED>
__device__ __forceinline__ uint32_t ds_pair(float2 s1, float2 s2, float2 cc, float2 sc, float2 nA, float2 nB,
                                            float2 G, uint32_t visible, int k) {
  const float2 x1 = ffma2(s1, cc, nA);
  float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
  bool k0 = true, k1 = true;
  if (MASKED) {
    k0 = (visible >> k) & 1u;
    k1 = (visible >> (k + 1)) & 1u;
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
  return pack_bf16(ds.x, ds.y);
}

// Thread = one query row with its folded values (nA, nB, G), N key columns.
template <int SETTING, bool MASKED, int N>
__device__ __forceinline__ void make_ds_row(const uint32_t (&a)[N], const uint32_t (&b)[N], uint32_t* pk, float c,
                                            float scale, float nAr, float nBr, float Gr, uint32_t visible) {
  const float2 cc = make_float2(c, c), sc = make_float2(scale, scale);
  const float2 nA = make_float2(nAr, nAr), nB = make_float2(nBr, nBr), G = make_float2(Gr, Gr);
#pragma unroll
  for (int k = 0; k < N; k += 2) {
    const float2 s1 = make_float2(__uint_as_float(a[k]), __uint_as_float(a[k + 1]));
    const float2 s2 = make_float2(__uint_as_float(b[k]), __uint_as_float(b[k + 1]));
    pk[k / 2] = ds_pair<SETTING, MASKED>(s1, s2, cc, sc, nA, nB, G, visible, k);
  }
}

// Setting 1 in two steps, for kernels that receive S1 before S2.  First, in
// place: P1 for N columns of S1 (0 where the key is not visible).
template <bool MASKED, int N>
__device__ __forceinline__ void p1_row(uint32_t (&s)[N], float c, float nAr, uint32_t visible) {
  const float2 cc = make_float2(c, c), nA = make_float2(nAr, nAr);
#pragma unroll
  for (int k = 0; k < N; k += 2) {
    const float2 x1 = ffma2(make_float2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), cc, nA);
    float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
    if (MASKED) {
      p1.x = (visible >> k) & 1u ? p1.x : 0.f;
      p1.y = (visible >> (k + 1)) & 1u ? p1.y : 0.f;
    }
    s[k] = __float_as_uint(p1.x);
    s[k + 1] = __float_as_uint(p1.y);
  }
}

// Then dS2 = g (P2 - P1) for N columns, from S2 and the first step's P1 (the
// same operations as ds_pair, so identical distributions give exact zeros).
template <bool MASKED, int N>
__device__ __forceinline__ void ds1_from_p1(const uint32_t (&s2)[N], const uint32_t* p1v, uint32_t* pk, float c,
                                            float nBr, float Gr, uint32_t visible) {
  const float2 cc = make_float2(c, c), nB = make_float2(nBr, nBr), G = make_float2(Gr, Gr);
#pragma unroll
  for (int k = 0; k < N; k += 2) {
    const float2 x2 = ffma2(make_float2(__uint_as_float(s2[k]), __uint_as_float(s2[k + 1])), cc, nB);
    float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
    if (MASKED) {
      p2.x = (visible >> k) & 1u ? p2.x : 0.f;
      p2.y = (visible >> (k + 1)) & 1u ? p2.y : 0.f;
    }
    const float2 ds = fmul2(G, fsub2(p2, make_float2(__uint_as_float(p1v[k]), __uint_as_float(p1v[k + 1]))));
    pk[k / 2] = pack_bf16(ds.x, ds.y);
  }
}

// Both settings at once (the mutual case, where Q1/K1 and Q2/K2 all train):
// dS1 = g P1 (r - KL) and dS2 = g (P2 - P1) from one read of the two logit
// tiles, with the folded values nA, nB2 = -LSE2 log2(e) (setting 1's nB) and
// nB1 = -(LSE1 - LSE2 + KL) (setting 2's nB).  The operations are ds_pair's of
// each setting, so each output is bit-identical to that setting's dS.
template <bool MASKED, int N>
__device__ __forceinline__ void make_ds_row_mutual(const uint32_t* a, const uint32_t (&b)[N], uint32_t* pk1,
                                                   uint32_t* pk2, float c, float scale, float nAr, float nB2r,
                                                   float nB1r, float Gr, uint32_t visible) {
  const float2 cc = make_float2(c, c), sc = make_float2(scale, scale);
  const float2 nA = make_float2(nAr, nAr), nB2 = make_float2(nB2r, nB2r), nB1 = make_float2(nB1r, nB1r);
  const float2 G = make_float2(Gr, Gr);
#pragma unroll
  for (int k = 0; k < N; k += 2) {
    const float2 s1 = make_float2(__uint_as_float(a[k]), __uint_as_float(a[k + 1]));
    const float2 s2 = make_float2(__uint_as_float(b[k]), __uint_as_float(b[k + 1]));
    const float2 x1 = ffma2(s1, cc, nA), x2 = ffma2(s2, cc, nB2);
    float2 p1 = make_float2(ex2(x1.x), ex2(x1.y)), p2 = make_float2(ex2(x2.x), ex2(x2.y));
    if (MASKED) {
      const bool k0 = (visible >> k) & 1u, k1 = (visible >> (k + 1)) & 1u;
      p1.x = k0 ? p1.x : 0.f;
      p1.y = k1 ? p1.y : 0.f;
      p2.x = k0 ? p2.x : 0.f;
      p2.y = k1 ? p2.y : 0.f;
    }
    const float2 d2 = fmul2(G, fsub2(p2, p1));
    const float2 d1 = fmul2(fmul2(G, p1), ffma2(sc, fsub2(s1, s2), nB1));
    pk1[k / 2] = pack_bf16(d1.x, d1.y);
    pk2[k / 2] = pack_bf16(d2.x, d2.y);
  }
}

}  // namespace skl
