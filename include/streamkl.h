/*
 * libstreamkl — fused attention KL divergence for one GB300 GPU (sm_103a).
 *
 * For every (batch b, head h, query row i) the library computes
 *
 *     S_t = scale * Q_t K_t^T,  P_t = row-softmax(S_t)   (t = 1 teacher, t = 2 student)
 *     KL_i = sum_j P1_ij (log P1_ij - log P2_ij)           i.e. KL(P1 || P2)
 *     LSE_t,i = log sum_j exp(S_t,ij)
 *
 * over the keys j that the (optional) causal mask keeps, without ever writing
 * an N_Q x N_K matrix to memory.  The forward is the one-pass online
 * formulation with five running scalars per row (m1, m2, l1, l2, acc) and the
 * closing identity KL = acc/l1 + LSE2 - LSE1 (StreamKL technical summary,
 * gist.science/ja/paper/2606.20005, section 手法 1 "online formulation").  The
 * backward rebuilds P_t = exp(S_t - LSE_t) tile by tile from Q, K and the saved
 * LSE (section 手法 2 "recompute strategy") in the two settings named there.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Q_t are [B, H, N_Q, D] and K_t are [B, H, N_K, D], bf16, DEVICE
 *   pointers, 16-byte aligned, contiguous unless the shape's strides say
 *   otherwise (see streamkl_shape).  D is 64 or 128.
 * - Row outputs and inputs (KL, LSE1, LSE2, g) are fp32 [B, H, N_Q], device.
 * - Gradient outputs are bf16 in the layout of the tensor they belong to.
 * - scale <= 0 selects 1/sqrt(D).  causal != 0 keeps key j for row i iff
 *   j <= i + N_K - N_Q (bottom-right alignment); causal with N_Q > N_K is
 *   rejected so that no row is left without keys.
 * - The caller owns every buffer; the library allocates no device memory.
 *   Scratch memory is passed in as a workspace whose size is queried first.
 *   The one exception is streamkl_fwd_splitk_noalloc, whose scratch is a
 *   fixed static device array inside the library.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *   asynchronous on it.  Argument errors are returned synchronously before
 *   anything is launched.  Launch failures return STREAMKL_ERR_CUDA.
 * - Device-side waits are bounded.  A wait that runs out sets a device status
 *   word instead of hanging; streamkl_check_device_status() reads it.
 * - No C++ exception crosses this interface.
 */
#ifndef STREAMKL_H
#define STREAMKL_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  STREAMKL_OK = 0,
  STREAMKL_ERR_INVALID = 1,     /* bad shape, null/misaligned pointer, causal with N_Q > N_K */
  STREAMKL_ERR_UNSUPPORTED = 2, /* valid but not handled (e.g. D not in {64,128}, Split-K N_Q > 16) */
  STREAMKL_ERR_WORKSPACE = 3,   /* workspace pointer missing, misaligned or too small */
  STREAMKL_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, memset, tensor map) */
  STREAMKL_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (reported by check_device_status) */
  STREAMKL_ERR_SCRATCH_LIMIT = 6 /* needs more than the fixed scratch of streamkl_fwd_splitk_noalloc */
} streamkl_status;

/*
 * Problem shape.  scale <= 0 means 1/sqrt(D).
 *
 * q_stride_* and k_stride_* are ELEMENT strides along b, h and n of the
 * logical [B, H, N, D] views of Q1/Q2 and of K1/K2 (D itself is contiguous).
 * All three zero selects the contiguous [B, H, N, D] layout; otherwise each is
 * positive and a multiple of 8 (16 bytes), n's stride is at least D, and both
 * tensors of a pair (Q1 and Q2, K1 and K2) share the strides.  A [B, N, H, D]
 * tensor, as many attention implementations store it, is passed without a
 * copy as strides (N*H*D, D, H*D).  Gradient outputs (dQ, dK) are written
 * with the strides of the input they belong to, so those strides must not
 * make two rows overlap (inputs are only read and may overlap); row-shaped
 * tensors (KL, LSE, g) stay contiguous [B, H, N_Q].
 */
typedef struct {
  int B, H, NQ, NK, D;
  float scale;
  int causal;
  long long q_stride_b, q_stride_h, q_stride_n;
  long long k_stride_b, k_stride_h, k_stride_n;
} streamkl_shape;

/* Backward path selection (the adaptive rule of section 手法 2 "kernel fusion"). */
typedef enum {
  STREAMKL_BWD_AUTO = 0,     /* the rule of streamkl_bwd_select */
  STREAMKL_BWD_FUSED = 1,    /* one pass over each QK tile pair, dQ on chip, dK by atomics into fp32 */
  STREAMKL_BWD_SEPARATE = 2, /* a Q-stationary dQ kernel and a K-stationary dK kernel */
  STREAMKL_BWD_DQ_ONLY = 3,  /* separate path, dQ kernel only (dK pointer may be NULL) */
  STREAMKL_BWD_DK_ONLY = 4   /* separate path, dK kernel only (dQ pointer may be NULL) */
} streamkl_bwd_mode;

/* Largest N_Q the Split-K forward takes. */
#define STREAMKL_SPLITK_MAX_NQ 16

/*
 * Forward: KL, LSE1, LSE2 [B,H,N_Q] fp32 from bf16 Q1, K1, Q2, K2.
 * (technical summary, 手法 1 "online formulation": five running scalars,
 *  KL = acc/l1 + LSE2 - LSE1, whole key tiles past the causal boundary skipped.)
 * One CTA owns a tile of query rows and streams every key tile it needs.
 */
streamkl_status streamkl_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                             streamkl_shape s, float* kl, float* lse1, float* lse2, void* stream);

/*
 * Split-K forward for few query rows (decode, N_Q <= STREAMKL_SPLITK_MAX_NQ).
 * (technical summary, 手法 3 "Split-K variant": the key dimension is divided
 *  over thread blocks so that a small N_Q still fills the SMs.)
 * Each of `num_splits` blocks per (b, h) reduces a contiguous key range to the
 * five partial scalars per row; a second kernel merges them.  num_splits = 0
 * picks a count that fills the GPU.  Workspace: fp32 [B,H,N_Q,splits,5], size
 * from streamkl_fwd_splitk_workspace(), 16-byte aligned, contents ignored.
 */
streamkl_status streamkl_fwd_splitk_workspace(streamkl_shape s, int num_splits, size_t* bytes);
streamkl_status streamkl_fwd_splitk(const void* q1, const void* k1, const void* q2, const void* k2,
                                    streamkl_shape s, int num_splits, void* workspace,
                                    size_t workspace_bytes, float* kl, float* lse1, float* lse2,
                                    void* stream);
/*
 * The split count num_splits = 0 resolves to, for a GPU with `num_sms` SMs
 * (num_sms <= 0: the current device).  It minimises waves x (tiles per block
 * + a fixed per-block cost); with num_sms > 0 it is a pure host computation.
 */
streamkl_status streamkl_fwd_splitk_plan(streamkl_shape s, int num_sms, int* num_splits);

/*
 * Split-K forward that allocates nothing and takes no workspace.  The paper
 * has no counterpart of this entry point; it exists for callers that cannot
 * call cudaMalloc or hand out scratch memory -- code that runs inside a host
 * application or serving runtime owning all device memory, or a decode loop
 * whose memory budget is fixed before it starts.  The caller still passes the
 * inputs and outputs.
 *
 * The per-split partial states live in one static device array of
 * STREAMKL_NOALLOC_SCRATCH_BYTES built into the library; every GPU that loads
 * the library keeps it until the process exits.  A problem whose partials
 * (B*H*N_Q*splits*5 floats) do not fit returns STREAMKL_ERR_SCRATCH_LIMIT with
 * nothing launched.  All calls share that array and it keeps the last call's
 * contents: a call that completes writes every partial it then reads, so
 * nothing needs clearing.  If one of its bounded waits runs out, a partial
 * block stops without writing and the merge reads what an earlier call left
 * there, so the outputs are valid only when streamkl_check_device_status
 * returns STREAMKL_OK afterwards.  Calls that overlap on the GPU -- on
 * different streams, or from different host threads -- race on the array
 * and must be serialised by the caller.
 * The first call on a device looks up the array's device address with that
 * device current (once per device); make that first call before any stream
 * capture.  Results equal streamkl_fwd_splitk's for the same num_splits.
 */
#define STREAMKL_NOALLOC_SCRATCH_BYTES (4u << 20)
streamkl_status streamkl_fwd_splitk_noalloc(const void* q1, const void* k1, const void* q2, const void* k2,
                                            streamkl_shape s, int num_splits, float* kl, float* lse1,
                                            float* lse2, void* stream);

/*
 * Key shards (context parallelism): the keys of a long sequence split into
 * contiguous ranges, e.g. one per GPU, every range seen by every query row.
 * (technical summary, 手法 3 "Split-K variant": a key range reduces to five
 *  scalars per row and ranges merge exactly; the pages split over thread
 *  blocks, here the same algebra splits over devices.)
 *
 * In each of these calls s.NK is the shard's key count and K1, K2 point at the
 * shard's rows (any strides the shape allows, so a row slice of a larger
 * [B, H, N, D] tensor is passed as is), which are the keys at global positions
 * [key_offset, key_offset + s.NK) of a sequence of nk_total keys.  The causal
 * frontier is the global one: row i keeps global key j iff
 * j <= i + nk_total - N_Q; rows that see none of the shard's keys are allowed.
 * Requires 0 <= key_offset, key_offset + s.NK <= nk_total, and, when causal,
 * N_Q <= nk_total.
 *
 * streamkl_fwd_partials: the five scalars of every row over the shard's keys,
 *   fp32 [B, H, N_Q, 5] = (m1, m2, l1, l2, acc): m_t the reference maximum of
 *   scale * log2(e) * q_t.k_t, l_t = sum 2^(that - m_t), acc = sum of
 *   2^(...1 - m1) (q1.k1 - q2.k2) (unscaled).  A row with no visible key gets
 *   (-inf, -inf, 0, 0, 0).
 * streamkl_merge_partials: KL, LSE1, LSE2 [B, H, N_Q] from num_parts such
 *   partial sets stored one after the other, [num_parts][B, H, N_Q, 5] (what
 *   an all-gather of every shard's partials produces).  Only B, H, N_Q, D and
 *   the scale of s are used.  Every row must see a key in some part.
 * streamkl_bwd_keyshard: the backward (setting 1 or 2, as streamkl_bwd_s1 /
 *   streamkl_bwd_s2) over the shard's keys, given the merged LSE1, LSE2, KL of
 *   the whole sequence: the shard's dK rows (bf16, K's layout, complete since
 *   every query row is here) and this shard's unscaled contribution to dQ,
 *   fp32 [B, H, N_Q, D] contiguous, 16-byte aligned, overwritten.  Summing the
 *   dq_partial of all shards (an all-reduce) gives the full unscaled dQ.
 *   Workspace (16-byte aligned) from streamkl_bwd_keyshard_workspace: the fused
 *   path's fp32 dK rows of one key range.
 * streamkl_dq_from_partial: bf16 dQ = scale * dq_partial, written with the Q
 *   strides of s (the full problem's shape).
 */
streamkl_status streamkl_fwd_partials(const void* q1, const void* k1, const void* q2, const void* k2,
                                      streamkl_shape s, long long key_offset, long long nk_total, float* partials,
                                      void* stream);
streamkl_status streamkl_merge_partials(const float* partials, int num_parts, streamkl_shape s, float* kl,
                                        float* lse1, float* lse2, void* stream);
streamkl_status streamkl_bwd_keyshard_workspace(streamkl_shape s, long long key_offset, long long nk_total,
                                                size_t* bytes);
streamkl_status streamkl_bwd_keyshard(int setting, const void* q1, const void* k1, const void* q2, const void* k2,
                                      streamkl_shape s, long long key_offset, long long nk_total, const float* lse1,
                                      const float* lse2, const float* kl, const float* g, float* dq_partial,
                                      void* dk, void* workspace, size_t workspace_bytes, void* stream);
streamkl_status streamkl_dq_from_partial(const float* dq_partial, streamkl_shape s, void* dq, void* stream);

/*
 * Backward workspace for the current device (0 bytes for the separate path).
 * The fused path adds dK partials (TMA bulk fp32 reductions) into an
 * accumulator that the library zeroes; they stay cheap while the rows being
 * accumulated sit in L2.  Its blocks run head by head, so the live rows are one head's keys times
 * the heads a wave of blocks spans.  When all N_K keys fit that way, one
 * launch covers them and the workspace is the fp32 [B,H,N_K,D] dK accumulator
 * (dQ stays on chip).  Otherwise the keys are split into ranges whose live rows
 * fit in half the L2, each range one launch, and the workspace is the fp32
 * [B,H,range,D] dK rows of one range followed by an fp32 [B,H,N_Q,D] dQ
 * accumulator.  streamkl_bwd_fused_plan gives the same figures for any L2
 * size.  The environment variable STREAMKL_FUSED_KEY_TILES, a positive count of
 * 128-key tiles, fixes the range length instead (for testing and tuning).
 */
streamkl_status streamkl_bwd_workspace(streamkl_shape s, int bwd_mode, size_t* bytes);
/*
 * Which path AUTO takes (pure host rule, no device; 0 for an invalid shape or
 * num_sms <= 0): the fused path (over key ranges when N_K is long; see
 * streamkl_bwd_fused_plan), except the separate kernels when a head has at
 * most eight 128-row query tiles and the fused path would either need more
 * than one key range or launch fewer blocks (B*H*query tiles) than num_sms --
 * a key tile is then reused by few query tiles, the separate kernels' extra
 * recompute costs less than the fused path's dK atomics and per-range dQ round
 * trips, and the separate dK grid's many short blocks fill the SMs its few
 * long dQ blocks leave free (the two grids run as one launch).  This is the
 * "separate kernels under contention" rule of section 手法 2 "kernel fusion",
 * with the thresholds measured on GB300.
 */
int streamkl_bwd_select(streamkl_shape s, size_t l2_bytes, int num_sms);
/*
 * The fused path's plan on a device with `l2_bytes` of L2 and `num_sms` SMs
 * (pure host rule, no device): the number of key ranges (launches) and the
 * workspace bytes, as described at streamkl_bwd_workspace.
 */
streamkl_status streamkl_bwd_fused_plan(streamkl_shape s, size_t l2_bytes, int num_sms, int* key_ranges,
                                        size_t* workspace_bytes);

/*
 * Setting 1: P1 held fixed, Q2/K2 optimised (standard distillation).
 * (technical summary, 手法 2 "recompute strategy", setting 1.)
 * Rebuilds P_t = exp(S_t - LSE_t); dS2 = g_i (P2 - P1); writes
 * dQ2 = scale dS2 K2 and dK2 = scale dS2^T Q2 (bf16).  g is dLoss/dKL_i, fp32
 * [B,H,N_Q] (a mean over rows is g = 1/N_Q).  lse1/lse2 are the forward's.
 */
streamkl_status streamkl_bwd_s1(const void* q1, const void* k1, const void* q2, const void* k2,
                                streamkl_shape s, const float* lse1, const float* lse2,
                                const float* g, void* dq2, void* dk2, int bwd_mode,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Setting 2: P2 held fixed, Q1/K1 optimised.
 * (technical summary, 手法 2, setting 2; 手法 3 "numerical stability": the log
 *  ratio comes from logits and stored LSEs, never from log of probabilities.)
 * r = (S1 - LSE1) - (S2 - LSE2); dS1 = g_i P1 (r - KL_i); writes
 * dQ1 = scale dS1 K1 and dK1 = scale dS1^T Q1 (bf16).  kl is the forward's.
 */
streamkl_status streamkl_bwd_s2(const void* q1, const void* k1, const void* q2, const void* k2,
                                streamkl_shape s, const float* lse1, const float* lse2,
                                const float* kl, const float* g, void* dq1, void* dk1, int bwd_mode,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * The mutual case: Q1, K1, Q2, K2 all optimised (both distributions train).
 * (technical summary, 手法 2 "recompute strategy", settings 1 and 2.)
 * P2 does not depend on Q1/K1 nor P1 on Q2/K2, so the gradients of
 * L = sum_i g_i KL_i are setting 2's (dQ1, dK1) and setting 1's (dQ2, dK2).
 * bwd_mode:
 *   STREAMKL_BWD_SEPARATE  the mutual kernels: S1 and S2 of each tile pair are
 *                          rebuilt once and both dS tiles formed from them
 *                          (dQ blocks and dK blocks in one launch, no atomics,
 *                          no workspace); dS1 and dS2 are bit-identical to the
 *                          single settings', and so are the four outputs to
 *                          those of streamkl_bwd_s2 / streamkl_bwd_s1 with
 *                          STREAMKL_BWD_SEPARATE.
 *   STREAMKL_BWD_FUSED     one fused pass per setting (setting 1, then setting
 *                          2), sharing the workspace of streamkl_bwd_workspace.
 *   STREAMKL_BWD_AUTO      as streamkl_bwd_mutual_select decides.
 * Arguments are those of streamkl_bwd_s2 (kl is required) with four bf16
 * outputs, each [B,H,N,D] with the strides of its input (dq1: q1's strides,
 * dk2: k2's, ...), all four non-NULL and 16-byte aligned.  Work runs on
 * `stream`.  With N_Q = 0 both dK are written as zeros.  Errors:
 * STREAMKL_ERR_INVALID for a bad shape, pointer or mode (DQ_ONLY / DK_ONLY are
 * refused), STREAMKL_ERR_WORKSPACE when the fused passes are chosen and the
 * workspace is missing or smaller than streamkl_bwd_mutual_workspace's,
 * STREAMKL_ERR_UNSUPPORTED for D not in {64, 128}; nothing is launched then.
 */
streamkl_status streamkl_bwd_mutual(const void* q1, const void* k1, const void* q2, const void* k2,
                                    streamkl_shape s, const float* lse1, const float* lse2,
                                    const float* kl, const float* g, void* dq1, void* dk1,
                                    void* dq2, void* dk2, int bwd_mode, void* workspace,
                                    size_t workspace_bytes, void* stream);
/*
 * AUTO's choice for the mutual case (pure host rule; the arguments match
 * streamkl_bwd_select's): STREAMKL_BWD_SEPARATE (the mutual kernels) when a
 * head has at most 64 query tiles of 128 rows, else STREAMKL_BWD_FUSED (a
 * fused pass per setting) -- the threshold measured on GB300.  0 for an
 * invalid shape or num_sms <= 0.
 */
int streamkl_bwd_mutual_select(streamkl_shape s, size_t l2_bytes, int num_sms);
/* Workspace bytes streamkl_bwd_mutual needs in `bwd_mode` on the current device (0 for the mutual kernels). */
streamkl_status streamkl_bwd_mutual_workspace(streamkl_shape s, int bwd_mode, size_t* bytes);

/* Text for a status code (static storage). */
const char* streamkl_status_string(streamkl_status st);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns STREAMKL_ERR_TIMEOUT if a bounded wait ran out since
 * the last check, STREAMKL_ERR_CUDA if the sync failed, else STREAMKL_OK.
 *
 * The status word is one flag per device for the whole process, shared by
 * every caller, stream and thread that uses the library: a timeout on any
 * stream sets it, and the first check afterwards -- from whichever thread --
 * reports and clears it.  Callers that share a device and each want to see
 * their own timeouts must serialise their checks (or agree on one checker).
 */
streamkl_status streamkl_check_device_status(void* stream);

/*
 * Test hook for the timeout path: launches one block that waits on a barrier
 * nobody arrives at, giving up after `timeout_us` microseconds (clamped to
 * [1, 1000000]) and recording STREAMKL_ERR_TIMEOUT in the status word.
 */
streamkl_status streamkl_debug_wait_timeout(int timeout_us, void* stream);

/* Library version, major*10000 + minor*100 + patch. */
int streamkl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* STREAMKL_H */
