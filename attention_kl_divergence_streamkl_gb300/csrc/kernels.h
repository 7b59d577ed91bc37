// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace skl {

// A validated problem.  Logits are handled in log2 units: c = scale * log2(e).
struct Problem {
  int B, H, NQ, NK, D;
  int BH;
  int causal;
  int off;      // NK - NQ: row i keeps key j iff j <= i + off (causal)
  float scale;  // softmax scale applied to Q K^T
  float c;      // scale * log2(e)
  // element strides of Q1/Q2 (and dQ) and of K1/K2 (and dK) along b, h, n; d is contiguous
  long long qs_b, qs_h, qs_n, ks_b, ks_h, ks_n;
};

// Element offset of row n of head (b, h) = bh in a tensor with strides (sb, sh, sn).
__host__ __device__ inline long long row_offset(int bh, int H, long long n, long long sb, long long sh, long long sn) {
  return (long long)(bh / H) * sb + (long long)(bh % H) * sh + n * sn;
}

// Builds a 4-D TMA map {d, n, h, b} over a bf16 [B, H, N, D] view with the given
// element strides (d contiguous), a {64, box_rows, 1, 1} box and the 128-byte
// swizzle.  Returns false if the driver rejects it.
bool encode_tile_map(CUtensorMap* map, const void* base, int D, int N, int H, int B, long long sn, long long sh,
                     long long sb, int box_rows);
// A 3-D TMA map {d, row, bh} over an fp32 [BH][rows][D] accumulator, a {D, box_rows, 1} box, no swizzle
// (for bulk reductions into it).
bool encode_rows_f32_map(CUtensorMap* map, float* base, int D, int rows, int BH, int box_rows);
// The maps of Q1/Q2 and K1/K2 of a problem.
inline bool encode_q_map(CUtensorMap* map, const void* base, const Problem& p, int box_rows) {
  return encode_tile_map(map, base, p.D, p.NQ, p.H, p.B, p.qs_n, p.qs_h, p.qs_b, box_rows);
}
inline bool encode_k_map(CUtensorMap* map, const void* base, const Problem& p, int box_rows) {
  return encode_tile_map(map, base, p.D, p.NK, p.H, p.B, p.ks_n, p.ks_h, p.ks_b, box_rows);
}

// ---- forward (one CTA per 128-row query tile) -------------------------------
cudaError_t launch_fwd(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                       float* kl, float* lse1, float* lse2, int* status, cudaStream_t st);
// The same forward over one key shard (p.off already shifted by the shard's
// first key): the five scalars of every row, fp32 [B*H*N_Q][5] (m1, m2 in log2
// units, l1, l2, acc unscaled), instead of KL and LSE.
cudaError_t launch_fwd_partials(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                                float* partials, int* status, cudaStream_t st);
// Merges `parts` partial sets laid out [part][B*H*N_Q][5] into KL, LSE1, LSE2.
cudaError_t launch_merge_partials(const Problem& p, int parts, const float* partials, float* kl, float* lse1,
                                  float* lse2, cudaStream_t st);

// ---- Split-K forward ---------------------------------------------------------
constexpr int kSplitKTile = 64;        // keys per pipeline stage
constexpr int kSplitKCtasPerSm = 2;    // resident blocks per SM the planner assumes
int splitk_key_tiles(const Problem& p);
int splitk_plan(int BH, int key_tiles, int num_sms);
cudaError_t launch_splitk(const Problem& p, const void* q1, const void* k1, const void* q2, const void* k2,
                          int splits, float* partials, float* kl, float* lse1, float* lse2, int* status,
                          cudaStream_t st);
// Device address (current device) of the fixed scratch of the allocation-free entry point.
cudaError_t splitk_noalloc_scratch(float** out);

// ---- backward ------------------------------------------------------------------
struct BwdIn {
  const void *q1, *k1, *q2, *k2;
  const float *lse1, *lse2, *kl, *g;
};
// setting 1: dq/dk are dQ2/dK2; setting 2: dQ1/dK1.  The separate path skips a NULL output; with both
// outputs its dQ and dK grids run as one launch.
cudaError_t launch_bwd_separate(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, int* status,
                                cudaStream_t st);
// Fused backward over key ranges of range_tiles 128-key tiles (all keys when
// range_tiles >= the tile count).  workspace: the fp32 dK rows of one range
// ([B*H][min(128 range_tiles, N_K)][D]), then, with more than one range, the
// fp32 dQ accumulator ([B*H][N_Q][D]).
// With dq_f32 non-null, dQ is not written to dq: the unscaled fp32 sum over
// this launch's keys goes to dq_f32 ([B*H][N_Q][D], zeroed first), and the
// workspace holds only the dK rows of one range.
cudaError_t launch_bwd_fused(const Problem& p, int setting, const BwdIn& in, void* dq, void* dk, float* workspace,
                             int range_tiles, int* status, cudaStream_t st, float* dq_f32 = nullptr);
// Both settings' gradients in one recompute (the mutual case): dQ1, dK1 (setting 2) and dQ2, dK2
// (setting 1), each written with its input's strides; the dQ and the dK blocks in one launch, no workspace.
cudaError_t launch_bwd_mutual(const Problem& p, const BwdIn& in, void* dq1, void* dk1, void* dq2, void* dk2,
                              int* status, cudaStream_t st);
// dK = 0 for every key row of every head, written with K's strides (a backward with no query rows).
cudaError_t launch_zero_k_rows(const Problem& p, void* dk, cudaStream_t st);
// out row n of head bh = bf16(scale * acc[bh][n]) for n < N_Q, with Q's strides.
cudaError_t launch_rows_to_bf16(const Problem& p, const float* acc, void* out, cudaStream_t st);
// First 128-query tile whose rows see key k0.
int fused_first_qtile(const Problem& p, long long k0);

// ---- test hook ------------------------------------------------------------------
cudaError_t launch_wait_timeout_probe(int timeout_us, int* status, cudaStream_t st);

}  // namespace skl
