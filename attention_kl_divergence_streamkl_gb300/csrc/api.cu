// C-ABI of libstreamkl: argument validation, path selection and launches.
// The operations are declared and documented in include/streamkl.h.
#include <cstdlib>
#include <algorithm>
#include <math.h>
#include <stdint.h>

#include "../../include/streamkl.h"
#include "common.cuh"
#include "kernels.h"

// Device status word: bounded waits that run out OR bits into it.
__device__ int g_streamkl_status;

namespace skl {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn resolve_encode_fn() {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<EncodeTiledFn>(ptr);
  return nullptr;
}

EncodeTiledFn encode_fn() {
  // Resolved once, by a function-local static: C++ runs its initialiser
  // exactly once even when several host threads arrive here together.
  static const EncodeTiledFn fn = resolve_encode_fn();
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Maximum key/query tiles along grid.y.
constexpr long long kMaxGridY = 65535;
constexpr int kMaxRows = 1 << 30;

// Element strides of a [B, H, N, D] view: all zero selects the contiguous
// layout; otherwise each is positive and a multiple of 8 elements (16 bytes, the
// TMA stride granule), and a row holds at least D elements.
bool strides_ok(long long sb, long long sh, long long sn, int H, int N, int D, long long* ob, long long* oh,
                long long* on) {
  if (sb == 0 && sh == 0 && sn == 0) {
    *on = D;
    *oh = (long long)N * D;
    *ob = (long long)H * N * D;
    return true;
  }
  if (sb <= 0 || sh <= 0 || sn < D) return false;
  if (sb % 8 || sh % 8 || sn % 8) return false;
  if (sb >= (1ll << 38) || sh >= (1ll << 38) || sn >= (1ll << 38)) return false;  // TMA strides below 2^40 bytes
  *ob = sb;
  *oh = sh;
  *on = sn;
  return true;
}

streamkl_status validate(const streamkl_shape& s, Problem* p) {
  if (s.B <= 0 || s.H <= 0 || s.NQ < 0 || s.NK <= 0 || s.D <= 0) return STREAMKL_ERR_INVALID;
  if (!(s.scale == s.scale) || isinf(s.scale)) return STREAMKL_ERR_INVALID;
  if (s.causal && s.NQ > s.NK) return STREAMKL_ERR_INVALID;
  if (s.NQ > kMaxRows || s.NK > kMaxRows) return STREAMKL_ERR_UNSUPPORTED;
  if ((long long)s.B * s.H > 0x7fffffffLL) return STREAMKL_ERR_UNSUPPORTED;
  if (s.D != 64 && s.D != 128) return STREAMKL_ERR_UNSUPPORTED;
  if ((s.NQ + 127LL) / 128 > kMaxGridY || (s.NK + 127LL) / 128 > kMaxGridY) return STREAMKL_ERR_UNSUPPORTED;
  // one-dimensional grids of (query tiles + key tiles) blocks per head must fit a grid's x extent (and the
  // kernels' int block arithmetic)
  if ((long long)s.B * s.H * ((s.NQ + 127LL) / 128 + (s.NK + 127LL) / 128) > 0x7fffffffLL)
    return STREAMKL_ERR_UNSUPPORTED;
  p->B = s.B;
  p->H = s.H;
  p->NQ = s.NQ;
  p->NK = s.NK;
  p->D = s.D;
  p->BH = s.B * s.H;
  p->causal = s.causal ? 1 : 0;
  p->off = s.NK - s.NQ;
  p->scale = s.scale > 0.f ? s.scale : 1.0f / sqrtf((float)s.D);
  p->c = p->scale * kLog2e;
  if (!strides_ok(s.q_stride_b, s.q_stride_h, s.q_stride_n, s.H, s.NQ, s.D, &p->qs_b, &p->qs_h, &p->qs_n) ||
      !strides_ok(s.k_stride_b, s.k_stride_h, s.k_stride_n, s.H, s.NK, s.D, &p->ks_b, &p->ks_h, &p->ks_n))
    return STREAMKL_ERR_INVALID;
  return STREAMKL_OK;
}

// A key shard: s.NK keys at global positions [key_offset, key_offset + NK) of a
// sequence of nk_total keys, every query row of the problem.  The causal
// frontier is the global one (row i keeps global key j <= i + nk_total - N_Q),
// which for the shard's local keys is j_local <= i + off with the offset below;
// it may be negative (rows that see none of the shard's keys).
streamkl_status validate_shard(streamkl_shape s, long long key_offset, long long nk_total, Problem* p) {
  if (key_offset < 0 || nk_total <= 0 || nk_total > kMaxRows || s.NK <= 0 || key_offset + s.NK > nk_total)
    return STREAMKL_ERR_INVALID;
  if (s.causal && s.NQ > nk_total) return STREAMKL_ERR_INVALID;
  const int causal = s.causal;
  s.causal = 0;
  const streamkl_status v = validate(s, p);
  if (v != STREAMKL_OK) return v;
  p->causal = causal ? 1 : 0;
  p->off = (int)(nk_total - s.NQ - key_offset);
  return STREAMKL_OK;
}

bool inputs_ok(const void* q1, const void* k1, const void* q2, const void* k2) {
  return q1 && k1 && q2 && k2 && aligned16(q1) && aligned16(k1) && aligned16(q2) && aligned16(k2);
}

bool rows_ok(const float* a) { return a && (reinterpret_cast<uintptr_t>(a) & 3u) == 0; }

streamkl_status status_ptr(int** out) {
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_streamkl_status) != cudaSuccess) return STREAMKL_ERR_CUDA;
  return STREAMKL_OK;
}

streamkl_status from_cuda(cudaError_t e) { return e == cudaSuccess ? STREAMKL_OK : STREAMKL_ERR_CUDA; }

// The fused path adds dK partials into the fp32 buffer with atomics; they stay
// cheap while the rows being accumulated stay in L2.  Its blocks run head by
// head (all query tiles of one (b, h) before the next), so the live part of the
// buffer is the dK rows of the heads that are in flight at once: one head's
// N_K x D fp32 rows times the heads a full wave of blocks spans.
size_t live_acc_bytes(const Problem& p, int num_sms) {
  const long long query_tiles = (p.NQ + 127) / 128;  // blocks per head
  const long long heads_in_flight = (num_sms + query_tiles - 1) / query_tiles + 1;
  const long long heads = heads_in_flight < p.BH ? heads_in_flight : p.BH;
  return (size_t)p.NK * p.D * sizeof(float) * (size_t)heads;
}

// The same for one key range of `tiles` 128-key tiles: its dK rows times the
// heads in flight, counted with the fewest query tiles any range has (the last
// range's, under a causal mask).
size_t live_range_bytes(const Problem& p, int tiles, int num_sms) {
  const long long n_kt = (p.NK + 127) / 128, n_qt = (p.NQ + 127) / 128;
  const long long ranges = (n_kt + tiles - 1) / tiles;
  const long long keys = std::min<long long>((long long)tiles * 128, p.NK);
  const long long query_tiles = std::max<long long>(1, n_qt - fused_first_qtile(p, (ranges - 1) * tiles * 128));
  const long long heads_in_flight = (num_sms + query_tiles - 1) / query_tiles + 1;
  const long long heads = heads_in_flight < p.BH ? heads_in_flight : p.BH;
  return (size_t)keys * p.D * sizeof(float) * (size_t)heads;
}

// Key tiles per launch of the fused backward.  Its dK partials go into an fp32
// buffer through atomics, which stay cheap while the rows being accumulated
// stay in L2: all keys in one launch when their live rows fit, else the longest
// key range whose live rows fit in half the L2 (the K tiles streamed for those
// heads share it), with dQ summed over the ranges in fp32.  A positive integer
// in the environment variable STREAMKL_FUSED_KEY_TILES overrides the choice.
int fused_range_tiles(const Problem& p, size_t l2_bytes, int num_sms) {
  const int n_kt = (p.NK + 127) / 128;
  if (const char* e = std::getenv("STREAMKL_FUSED_KEY_TILES")) {
    const long v = std::strtol(e, nullptr, 10);
    if (v > 0) return (int)std::min<long>(v, n_kt);
  }
  if (live_acc_bytes(p, num_sms) <= l2_bytes) return n_kt;
  for (int n = 2;; ++n) {
    const int tiles = (n_kt + n - 1) / n;
    if (tiles <= 1 || live_range_bytes(p, tiles, num_sms) <= l2_bytes / 2) return std::max(tiles, 1);
  }
}

size_t fused_workspace_bytes(const Problem& p, int range_tiles) {
  const long long n_kt = (p.NK + 127) / 128;
  const size_t dk_rows = (size_t)std::min<long long>((long long)range_tiles * 128, p.NK);
  size_t bytes = (size_t)p.BH * dk_rows * p.D * sizeof(float);
  if (range_tiles < n_kt) bytes += (size_t)p.BH * p.NQ * p.D * sizeof(float);
  return bytes;
}

// AUTO takes the fused path (over key ranges it keeps its atomics in L2 for any
// N_K) unless a head has at most kSeparateMaxQTiles query tiles and the fused
// path would either need more than one key range or leave SMs idle (fewer
// fused blocks, one per query tile, than SMs).  A key tile is then reused by
// few query tiles, so the fused kernel's one visit per tile pair saves little,
// while its dK atomics and per-range dQ round trips cost more than the separate
// kernels' second recompute -- and the separate path's dK grid, many short
// blocks, fills the SMs that its few long dQ blocks leave free, both grids in
// one launch (the "separate kernels under contention" rule of the technical
// summary, section 手法 2 "kernel fusion").
// Measured, ms for setting 1's backward, separate against fused: B1 H8
// N_K=64K non-causal N_Q=256 0.70 / 1.16, N_Q=512 0.71 / 1.16, N_Q=1024 0.76 /
// 1.17, N_Q=2048 1.39 / 1.25, N_Q=4096 2.64 / 2.33; B1 H32 N_Q=128 N_K=64K 0.84 /
// 1.74; one key range: B1 H32 N_Q=512 N_K=4096 causal (128 fused blocks) 0.13 /
// 0.17, B1 H32 N_Q=1024 N_K=8192 (256 fused blocks) 0.40 / 0.32.
constexpr int kSeparateMaxQTiles = 8;
int resolve_bwd_mode(const Problem& p, int mode, size_t l2_bytes, int num_sms) {
  if (mode != STREAMKL_BWD_AUTO) return mode;
  const int n_qt = (p.NQ + 127) / 128, n_kt = (p.NK + 127) / 128;
  const bool idle_sms = (long long)p.BH * n_qt < num_sms;
  if (n_qt <= kSeparateMaxQTiles && (idle_sms || fused_range_tiles(p, l2_bytes, num_sms) < n_kt))
    return STREAMKL_BWD_SEPARATE;
  return STREAMKL_BWD_FUSED;
}

// The mutual case (both settings' gradients): AUTO takes the mutual kernels
// (one recompute of each logit tile pair for both settings, reported as
// STREAMKL_BWD_SEPARATE) when a head has at most kMutualMaxQTiles query tiles,
// else one fused pass per setting.  Measured, ms for both settings' backward
// (mutual against two fused passes): B1 H32 N_Q=128 N_K=64K non-causal 1.15 /
// 3.52; B1 H8 N_K=64K non-causal N_Q=1024 1.10 / 2.33, N_Q=8192 7.63 / 8.36,
// N_Q=16384 15.1 / 14.6; causal B2 H32 N4096 1.18 / 1.25 (non-causal 2.08 /
// 2.08), B1 H8 N8K 0.59 / 0.65, N16K 2.02 / 1.99, N32K 7.60 / 7.25, N64K 29.9 /
// 29.0; B1 H2 N512K causal 508 / 492.
constexpr int kMutualMaxQTiles = 64;
int resolve_mutual_mode(const Problem& p, int mode, size_t l2_bytes, int num_sms) {
  (void)l2_bytes;
  (void)num_sms;
  if (mode != STREAMKL_BWD_AUTO) return mode;
  return (p.NQ + 127) / 128 <= kMutualMaxQTiles ? STREAMKL_BWD_SEPARATE : STREAMKL_BWD_FUSED;
}

streamkl_status device_l2_bytes(size_t* out) {
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
  *out = (size_t)l2;
  return STREAMKL_OK;
}

streamkl_status device_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
  if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
  return STREAMKL_OK;
}

// Bounded wait on a barrier that nothing arrives at: exercises the timeout path.
__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, &abort_flag, limit_ns);
}

}  // namespace

bool encode_rows_f32_map(CUtensorMap* map, float* base, int D, int rows, int BH, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)rows * D * 4};
  const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)box_rows, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tile_map(CUtensorMap* map, const void* base, int D, int N, int H, int B, long long sn, long long sh,
                     long long sb, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)sn * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  const cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_wait_timeout_probe(int timeout_us, int* status, cudaStream_t st) {
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>((unsigned long long)timeout_us * 1000ull, status);
  return cudaGetLastError();
}

}  // namespace skl

using namespace skl;

extern "C" {

int streamkl_version(void) { return 100; }

const char* streamkl_status_string(streamkl_status st) {
  switch (st) {
    case STREAMKL_OK: return "ok";
    case STREAMKL_ERR_INVALID: return "invalid argument";
    case STREAMKL_ERR_UNSUPPORTED: return "unsupported shape or option";
    case STREAMKL_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case STREAMKL_ERR_CUDA: return "CUDA call failed";
    case STREAMKL_ERR_TIMEOUT: return "device-side wait timed out";
    case STREAMKL_ERR_SCRATCH_LIMIT: return "problem needs more than the fixed no-allocation scratch";
  }
  return "unknown status";
}

streamkl_status streamkl_fwd(const void* q1, const void* k1, const void* q2, const void* k2, streamkl_shape s,
                             float* kl, float* lse1, float* lse2, void* stream) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (p.NQ == 0) return STREAMKL_OK;
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(kl) || !rows_ok(lse1) || !rows_ok(lse2)) return STREAMKL_ERR_INVALID;
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  return from_cuda(launch_fwd(p, q1, k1, q2, k2, kl, lse1, lse2, status, static_cast<cudaStream_t>(stream)));
}

streamkl_status streamkl_fwd_splitk_plan(streamkl_shape s, int num_sms, int* num_splits) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (!num_splits) return STREAMKL_ERR_INVALID;
  if (num_sms <= 0 && (v = device_sms(&num_sms)) != STREAMKL_OK) return v;
  int sp = splitk_plan(p.BH, splitk_key_tiles(p), num_sms);
  *num_splits = sp > (int)kMaxGridY ? (int)kMaxGridY : sp;
  return STREAMKL_OK;
}

streamkl_status streamkl_fwd_splitk_workspace(streamkl_shape s, int num_splits, size_t* bytes) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (!bytes || num_splits < 0 || num_splits > kMaxGridY) return STREAMKL_ERR_INVALID;
  if (p.NQ > STREAMKL_SPLITK_MAX_NQ) return STREAMKL_ERR_UNSUPPORTED;
  if (num_splits == 0 && (v = streamkl_fwd_splitk_plan(s, 0, &num_splits)) != STREAMKL_OK) return v;
  *bytes = (size_t)p.BH * p.NQ * num_splits * 5 * sizeof(float);
  return STREAMKL_OK;
}

streamkl_status streamkl_fwd_splitk(const void* q1, const void* k1, const void* q2, const void* k2,
                                    streamkl_shape s, int num_splits, void* workspace, size_t workspace_bytes,
                                    float* kl, float* lse1, float* lse2, void* stream) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (p.NQ > STREAMKL_SPLITK_MAX_NQ) return STREAMKL_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > kMaxGridY) return STREAMKL_ERR_INVALID;
  if (p.NQ == 0) return STREAMKL_OK;
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(kl) || !rows_ok(lse1) || !rows_ok(lse2)) return STREAMKL_ERR_INVALID;
  if (num_splits == 0 && (v = streamkl_fwd_splitk_plan(s, 0, &num_splits)) != STREAMKL_OK) return v;
  const size_t need = (size_t)p.BH * p.NQ * num_splits * 5 * sizeof(float);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return STREAMKL_ERR_WORKSPACE;
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  return from_cuda(launch_splitk(p, q1, k1, q2, k2, num_splits, static_cast<float*>(workspace), kl, lse1, lse2,
                                 status, static_cast<cudaStream_t>(stream)));
}

streamkl_status streamkl_fwd_splitk_noalloc(const void* q1, const void* k1, const void* q2, const void* k2,
                                            streamkl_shape s, int num_splits, float* kl, float* lse1, float* lse2,
                                            void* stream) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (p.NQ > STREAMKL_SPLITK_MAX_NQ) return STREAMKL_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > kMaxGridY) return STREAMKL_ERR_INVALID;
  if (p.NQ == 0) return STREAMKL_OK;
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(kl) || !rows_ok(lse1) || !rows_ok(lse2)) return STREAMKL_ERR_INVALID;
  if (num_splits == 0 && (v = streamkl_fwd_splitk_plan(s, 0, &num_splits)) != STREAMKL_OK) return v;
  const size_t need = (size_t)p.BH * p.NQ * num_splits * 5 * sizeof(float);
  if (need > STREAMKL_NOALLOC_SCRATCH_BYTES) return STREAMKL_ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  if (splitk_noalloc_scratch(&scratch) != cudaSuccess) return STREAMKL_ERR_CUDA;
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  return from_cuda(launch_splitk(p, q1, k1, q2, k2, num_splits, scratch, kl, lse1, lse2, status,
                                 static_cast<cudaStream_t>(stream)));
}

streamkl_status streamkl_fwd_partials(const void* q1, const void* k1, const void* q2, const void* k2,
                                      streamkl_shape s, long long key_offset, long long nk_total, float* partials,
                                      void* stream) {
  Problem p;
  streamkl_status v = validate_shard(s, key_offset, nk_total, &p);
  if (v != STREAMKL_OK) return v;
  if (p.NQ == 0) return STREAMKL_OK;
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(partials)) return STREAMKL_ERR_INVALID;
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  return from_cuda(launch_fwd_partials(p, q1, k1, q2, k2, partials, status, static_cast<cudaStream_t>(stream)));
}

streamkl_status streamkl_merge_partials(const float* partials, int num_parts, streamkl_shape s, float* kl,
                                        float* lse1, float* lse2, void* stream) {
  Problem p;
  s.causal = 0;  // only B, H, N_Q, D and the scale matter here
  if (s.NK <= 0) s.NK = 1;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (num_parts < 1) return STREAMKL_ERR_INVALID;
  if (p.NQ == 0) return STREAMKL_OK;
  if (!rows_ok(partials) || !rows_ok(kl) || !rows_ok(lse1) || !rows_ok(lse2)) return STREAMKL_ERR_INVALID;
  return from_cuda(launch_merge_partials(p, num_parts, partials, kl, lse1, lse2, static_cast<cudaStream_t>(stream)));
}

streamkl_status streamkl_bwd_keyshard_workspace(streamkl_shape s, long long key_offset, long long nk_total,
                                                size_t* bytes) {
  Problem p;
  streamkl_status v = validate_shard(s, key_offset, nk_total, &p);
  if (v != STREAMKL_OK) return v;
  if (!bytes) return STREAMKL_ERR_INVALID;
  size_t l2 = 0;
  int sms = 0;
  if ((v = device_l2_bytes(&l2)) != STREAMKL_OK || (v = device_sms(&sms)) != STREAMKL_OK) return v;
  const int tiles = fused_range_tiles(p, l2, sms);
  *bytes = (size_t)p.BH * std::min<long long>((long long)tiles * 128, p.NK) * p.D * sizeof(float);
  return STREAMKL_OK;
}

streamkl_status streamkl_bwd_keyshard(int setting, const void* q1, const void* k1, const void* q2, const void* k2,
                                      streamkl_shape s, long long key_offset, long long nk_total, const float* lse1,
                                      const float* lse2, const float* kl, const float* g, float* dq_partial,
                                      void* dk, void* workspace, size_t workspace_bytes, void* stream) {
  Problem p;
  streamkl_status v = validate_shard(s, key_offset, nk_total, &p);
  if (v != STREAMKL_OK) return v;
  if (setting != 1 && setting != 2) return STREAMKL_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!dk || !aligned16(dk)) return STREAMKL_ERR_INVALID;
  if (p.NQ == 0) return from_cuda(launch_zero_k_rows(p, dk, st));
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(lse1) || !rows_ok(lse2) || !rows_ok(g)) return STREAMKL_ERR_INVALID;
  if (setting == 2 && !rows_ok(kl)) return STREAMKL_ERR_INVALID;
  if (!dq_partial || !aligned16(dq_partial)) return STREAMKL_ERR_INVALID;
  if (!workspace || !aligned16(workspace)) return STREAMKL_ERR_WORKSPACE;
  size_t l2 = 0;
  int sms = 0;
  if ((v = device_l2_bytes(&l2)) != STREAMKL_OK || (v = device_sms(&sms)) != STREAMKL_OK) return v;
  const int range_tiles = fused_range_tiles(p, l2, sms);
  const size_t need = (size_t)p.BH * std::min<long long>((long long)range_tiles * 128, p.NK) * p.D * sizeof(float);
  if (workspace_bytes < need) return STREAMKL_ERR_WORKSPACE;
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  BwdIn in{q1, k1, q2, k2, lse1, lse2, kl, g};
  return from_cuda(launch_bwd_fused(p, setting, in, nullptr, dk, static_cast<float*>(workspace), range_tiles, status,
                                    st, dq_partial));
}

streamkl_status streamkl_dq_from_partial(const float* dq_partial, streamkl_shape s, void* dq, void* stream) {
  Problem p;
  s.causal = 0;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (p.NQ == 0) return STREAMKL_OK;
  if (!dq_partial || !aligned16(dq_partial) || !dq || !aligned16(dq)) return STREAMKL_ERR_INVALID;
  return from_cuda(launch_rows_to_bf16(p, dq_partial, dq, static_cast<cudaStream_t>(stream)));
}

int streamkl_bwd_select(streamkl_shape s, size_t l2_bytes, int num_sms) {
  Problem p;
  if (validate(s, &p) != STREAMKL_OK || num_sms <= 0) return 0;
  return resolve_bwd_mode(p, STREAMKL_BWD_AUTO, l2_bytes, num_sms);
}

streamkl_status streamkl_bwd_fused_plan(streamkl_shape s, size_t l2_bytes, int num_sms, int* key_ranges,
                                        size_t* workspace_bytes) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (num_sms <= 0 || !key_ranges || !workspace_bytes) return STREAMKL_ERR_INVALID;
  const int tiles = fused_range_tiles(p, l2_bytes, num_sms);
  const int n_kt = (p.NK + 127) / 128;
  *key_ranges = (n_kt + tiles - 1) / tiles;
  *workspace_bytes = fused_workspace_bytes(p, tiles);
  return STREAMKL_OK;
}

streamkl_status streamkl_bwd_workspace(streamkl_shape s, int bwd_mode, size_t* bytes) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (!bytes || bwd_mode < 0 || bwd_mode > STREAMKL_BWD_DK_ONLY) return STREAMKL_ERR_INVALID;
  *bytes = 0;
  if (bwd_mode == STREAMKL_BWD_AUTO || bwd_mode == STREAMKL_BWD_FUSED) {
    size_t l2 = 0;
    int sms = 0;
    if ((v = device_l2_bytes(&l2)) != STREAMKL_OK || (v = device_sms(&sms)) != STREAMKL_OK) return v;
    if (resolve_bwd_mode(p, bwd_mode, l2, sms) == STREAMKL_BWD_FUSED)
      *bytes = fused_workspace_bytes(p, fused_range_tiles(p, l2, sms));
  }
  return STREAMKL_OK;
}

static streamkl_status bwd_common(int setting, const void* q1, const void* k1, const void* q2, const void* k2,
                                  streamkl_shape s, const float* lse1, const float* lse2, const float* kl,
                                  const float* g, void* dq, void* dk, int bwd_mode, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (bwd_mode < 0 || bwd_mode > STREAMKL_BWD_DK_ONLY) return STREAMKL_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool want_dq = bwd_mode != STREAMKL_BWD_DK_ONLY;
  const bool want_dk = bwd_mode != STREAMKL_BWD_DQ_ONLY;
  if (want_dk && (!dk || !aligned16(dk))) return STREAMKL_ERR_INVALID;
  if (p.NQ == 0) {
    // no query rows: the loss is an empty sum, so dK is zero (written with dK's strides)
    return want_dk ? from_cuda(launch_zero_k_rows(p, dk, st)) : STREAMKL_OK;
  }
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(lse1) || !rows_ok(lse2) || !rows_ok(g))
    return STREAMKL_ERR_INVALID;
  if (want_dq && (!dq || !aligned16(dq))) return STREAMKL_ERR_INVALID;
  if (setting == 2 && !rows_ok(kl)) return STREAMKL_ERR_INVALID;
  int range_tiles = 0;
  if (bwd_mode == STREAMKL_BWD_FUSED && (!workspace || !aligned16(workspace))) return STREAMKL_ERR_WORKSPACE;
  if (bwd_mode == STREAMKL_BWD_AUTO || bwd_mode == STREAMKL_BWD_FUSED) {
    size_t l2 = 0;
    int sms = 0;
    if ((v = device_l2_bytes(&l2)) != STREAMKL_OK || (v = device_sms(&sms)) != STREAMKL_OK) return v;
    bwd_mode = resolve_bwd_mode(p, bwd_mode, l2, sms);
    range_tiles = fused_range_tiles(p, l2, sms);
  }
  if (bwd_mode == STREAMKL_BWD_FUSED) {
    if (!workspace || !aligned16(workspace)) return STREAMKL_ERR_WORKSPACE;
    if (workspace_bytes < fused_workspace_bytes(p, range_tiles)) return STREAMKL_ERR_WORKSPACE;
  }
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  BwdIn in{q1, k1, q2, k2, lse1, lse2, kl, g};
  if (bwd_mode == STREAMKL_BWD_FUSED)
    return from_cuda(
        launch_bwd_fused(p, setting, in, dq, dk, static_cast<float*>(workspace), range_tiles, status, st));
  return from_cuda(launch_bwd_separate(p, setting, in, want_dq ? dq : nullptr, want_dk ? dk : nullptr, status, st));
}

streamkl_status streamkl_bwd_s1(const void* q1, const void* k1, const void* q2, const void* k2, streamkl_shape s,
                                const float* lse1, const float* lse2, const float* g, void* dq2, void* dk2,
                                int bwd_mode, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(1, q1, k1, q2, k2, s, lse1, lse2, nullptr, g, dq2, dk2, bwd_mode, workspace, workspace_bytes,
                    stream);
}

streamkl_status streamkl_bwd_s2(const void* q1, const void* k1, const void* q2, const void* k2, streamkl_shape s,
                                const float* lse1, const float* lse2, const float* kl, const float* g, void* dq1,
                                void* dk1, int bwd_mode, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(2, q1, k1, q2, k2, s, lse1, lse2, kl, g, dq1, dk1, bwd_mode, workspace, workspace_bytes, stream);
}

int streamkl_bwd_mutual_select(streamkl_shape s, size_t l2_bytes, int num_sms) {
  Problem p;
  if (validate(s, &p) != STREAMKL_OK || num_sms <= 0) return 0;
  return resolve_mutual_mode(p, STREAMKL_BWD_AUTO, l2_bytes, num_sms);
}

static bool mutual_mode_ok(int mode) {
  return mode == STREAMKL_BWD_AUTO || mode == STREAMKL_BWD_FUSED || mode == STREAMKL_BWD_SEPARATE;
}

streamkl_status streamkl_bwd_mutual_workspace(streamkl_shape s, int bwd_mode, size_t* bytes) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (!bytes || !mutual_mode_ok(bwd_mode)) return STREAMKL_ERR_INVALID;
  *bytes = 0;
  if (bwd_mode == STREAMKL_BWD_SEPARATE) return STREAMKL_OK;
  size_t l2 = 0;
  int sms = 0;
  if ((v = device_l2_bytes(&l2)) != STREAMKL_OK || (v = device_sms(&sms)) != STREAMKL_OK) return v;
  if (resolve_mutual_mode(p, bwd_mode, l2, sms) == STREAMKL_BWD_FUSED)
    *bytes = fused_workspace_bytes(p, fused_range_tiles(p, l2, sms));
  return STREAMKL_OK;
}

streamkl_status streamkl_bwd_mutual(const void* q1, const void* k1, const void* q2, const void* k2,
                                    streamkl_shape s, const float* lse1, const float* lse2, const float* kl,
                                    const float* g, void* dq1, void* dk1, void* dq2, void* dk2, int bwd_mode,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  Problem p;
  streamkl_status v = validate(s, &p);
  if (v != STREAMKL_OK) return v;
  if (!mutual_mode_ok(bwd_mode)) return STREAMKL_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!dk1 || !aligned16(dk1) || !dk2 || !aligned16(dk2)) return STREAMKL_ERR_INVALID;
  if (p.NQ == 0) {  // an empty sum: both dK are zero
    cudaError_t e = launch_zero_k_rows(p, dk1, st);
    return from_cuda(e != cudaSuccess ? e : launch_zero_k_rows(p, dk2, st));
  }
  if (!inputs_ok(q1, k1, q2, k2) || !rows_ok(lse1) || !rows_ok(lse2) || !rows_ok(kl) || !rows_ok(g))
    return STREAMKL_ERR_INVALID;
  if (!dq1 || !aligned16(dq1) || !dq2 || !aligned16(dq2)) return STREAMKL_ERR_INVALID;
  if (bwd_mode == STREAMKL_BWD_FUSED && (!workspace || !aligned16(workspace))) return STREAMKL_ERR_WORKSPACE;
  int range_tiles = 0;
  if (bwd_mode != STREAMKL_BWD_SEPARATE) {
    size_t l2 = 0;
    int sms = 0;
    if ((v = device_l2_bytes(&l2)) != STREAMKL_OK || (v = device_sms(&sms)) != STREAMKL_OK) return v;
    bwd_mode = resolve_mutual_mode(p, bwd_mode, l2, sms);
    range_tiles = fused_range_tiles(p, l2, sms);
  }
  if (bwd_mode == STREAMKL_BWD_FUSED) {
    if (!workspace || !aligned16(workspace)) return STREAMKL_ERR_WORKSPACE;
    if (workspace_bytes < fused_workspace_bytes(p, range_tiles)) return STREAMKL_ERR_WORKSPACE;
  }
  int* status = nullptr;
  if ((v = status_ptr(&status)) != STREAMKL_OK) return v;
  BwdIn in{q1, k1, q2, k2, lse1, lse2, kl, g};
  if (bwd_mode == STREAMKL_BWD_SEPARATE) return from_cuda(launch_bwd_mutual(p, in, dq1, dk1, dq2, dk2, status, st));
  // one fused pass per setting, one after the other on the stream, sharing the workspace
  float* ws = static_cast<float*>(workspace);
  cudaError_t e = launch_bwd_fused(p, 1, in, dq2, dk2, ws, range_tiles, status, st);
  return from_cuda(e != cudaSuccess ? e : launch_bwd_fused(p, 2, in, dq1, dk1, ws, range_tiles, status, st));
}

streamkl_status streamkl_check_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return STREAMKL_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_streamkl_status, sizeof(int)) != cudaSuccess) return STREAMKL_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_streamkl_status, &zero, sizeof(int)) != cudaSuccess) return STREAMKL_ERR_CUDA;
  return (h & kStatusTimeout) ? STREAMKL_ERR_TIMEOUT : STREAMKL_OK;
}

streamkl_status streamkl_debug_wait_timeout(int timeout_us, void* stream) {
  if (timeout_us < 1) timeout_us = 1;
  if (timeout_us > 1000000) timeout_us = 1000000;
  int* status = nullptr;
  streamkl_status v = status_ptr(&status);
  if (v != STREAMKL_OK) return v;
  return from_cuda(launch_wait_timeout_probe(timeout_us, status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
