// Internal declarations shared by the kernels and the C-ABI layer of libkvq.so.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kGroup = KVQ_INT4_GROUP;
// 1 / sqrt(D) and sqrt(D) of the head dims the kernels are built for (64, 128, 256)
__host__ __device__ constexpr float inv_sqrt_dim(int d) { return d == 256 ? 0.0625f : (d == 128 ? 0.08838834764831845f : 0.125f); }
__host__ __device__ constexpr float sqrt_dim(int d) { return d == 256 ? 16.0f : (d == 128 ? 11.313708498984760f : 8.0f); }

// Count of kernel launches made by this library (kvq_kernel_launches); every launcher calls
// note_launch() after a launch that the runtime accepted.
void note_launch();

// ------------------------------------------------------------------------ quantize
struct QuantSide {
  uint8_t* rows;
  __half* aux;
  const float* bounds;
  const float* centroids;
  const int8_t* signs;
  const float* qjl;  // KVQ_FMT_CODEBOOK_QJL: projection [KVQ_QJL_DIM][D]
  const int32_t* outl;  // KVQ_FMT_CODEBOOK_OUTLIER: outlier channels [Hkv][KVQ_OUTLIER_CHANNELS]
  int fmt, bits, row_bytes;
};

struct QuantParams {
  const uint16_t* x[2];  // K, V inputs [T][Hkv][D] fp16 (either may be null)
  QuantSide side[2];
  const int32_t* slots;
  int num_tokens, hkv, page_size, num_slots;
  int page_shift;             // log2(page_size) when it is a power of two, else -1
  int kind_first, num_kinds;  // kinds present: [kind_first, kind_first + num_kinds)
  long long num_vectors;      // num_kinds * num_tokens * hkv
  // re-encode of stored fp16 rows (kvq_requantize) instead of new vectors: the source
  // pool's K and V rows (rotated fp16, same page size and kv heads) and slots
  const uint8_t* src_rows[2];
  const int32_t* src_slots;
  int src_num_slots;
};

cudaError_t launch_quantize(const QuantParams& p, int head_dim, cudaStream_t stream);
// Outlier channels of every kv head (kvq_outlier_calibrate): one block per head.
cudaError_t launch_outlier_calibrate(const uint16_t* k, int num_tokens, int hkv, int head_dim, int32_t* out,
                                     cudaStream_t stream);
// Re-encode: one warp per vector, every destination format.
cudaError_t launch_requantize(const QuantParams& p, int head_dim, cudaStream_t stream);

// ------------------------------------------------------------------------ decode
// Kernel family of a decode tier (chosen per tier on the host).
enum TierKind { TIER_GENERIC = 0, TIER_GQA = 1, TIER_CB = 2 };
// The 256-byte counter block at the end of the decode workspace (cleared once per call):
// ints [0, KVQ_MAX_TIERS) codebook work counters, kErrorWord the call's device error word
// (the OR of the KVQ_DEVERR_* bits any of its kernels raised), kGqaCounter the fused fp16 /
// fp8 + INT4 kernel's work counter.
constexpr int kErrorWord = 32, kGqaCounter = 40;

// ------------------------------------------------------------------------ index checks
// Every decode kernel reads lengths and block-table entries from device memory the host
// never sees, so it checks them itself before using them: a length outside
// [0, max_pages * page_size] is clamped into it, a page outside [0, num_pages) is skipped,
// and either raises its KVQ_DEVERR_* bit in *bits (the kernels OR the bits into the call's
// error word).  Host-callable, so a CPU test can drive them with out-of-range values.
__host__ __device__ __forceinline__ int checked_len(int len, int max_pages, int page_size, int* bits) {
  const long long cap = (long long)max_pages * page_size;
  if (len < 0 || (long long)len > cap) {
    *bits |= KVQ_DEVERR_SEQ_LEN;
    return len < 0 ? 0 : (int)cap;
  }
  return len;
}
// true when the page may be read; false (and the bit raised) when it lies outside the pool
__host__ __device__ __forceinline__ bool page_in_pool(int phys, int num_pages, int* bits) {
  if (phys < 0 || phys >= num_pages) {
    *bits |= KVQ_DEVERR_PAGE_INDEX;
    return false;
  }
  return true;
}
// Split-K chunks of one sequence that hold tokens (len already checked), never more than
// the plan made for the tier.
__host__ __device__ __forceinline__ int splits_holding_tokens(int len, int chunk, int num_splits) {
  const int n = (len + chunk - 1) / chunk;
  return n < num_splits ? n : num_splits;
}
// Whether slot `off` of logical page `lp` holds one of a chunk's tokens (those before
// t_end): it must lie inside the page -- a page size that is no multiple of the tokens a
// warp step covers leaves the last step's upper lanes past the page, on the next (page,
// kv head) block's rows -- and before the chunk's end.
__host__ __device__ __forceinline__ bool slot_holds_token(int lp, int off, int page_size, int t_end) {
  return off < page_size && (long long)lp * page_size + off < t_end;
}

struct DecTier {
  const uint8_t* k_rows;
  const uint8_t* v_rows;
  const __half* k_aux;
  const __half* v_aux;
  const float* k_cent;
  const float* v_cent;
  const float* k_qjl;  // KVQ_FMT_CODEBOOK_QJL keys: projection [KVQ_QJL_DIM][D]
  const int32_t* k_outl;  // KVQ_FMT_CODEBOOK_OUTLIER keys: outlier channels [Hkv][8]
  const int32_t* block_table;
  const int32_t* seq_lens;
  int k_fmt, v_fmt, k_bits, v_bits, k_row_bytes, v_row_bytes;
  int kind;  // TierKind
  int num_pages;  // pages in the pool (block-table entries must lie below)
  int max_pages, split_begin, num_splits, chunk;
};

struct DecParams {
  DecTier tier[KVQ_MAX_TIERS];
  int num_tiers;
  const __half* q;
  const int8_t* k_signs;
  const int8_t* v_signs;
  float* out;
  float* ws_acc;  // [B][Hq][S][D]
  float* ws_ml;   // [B][Hq][S][2]  (running max in log2 units, sum of exp2)
  float* ws_pq;   // [B][Hq][KVQ_QJL_DIM] projected queries when a tier's keys carry a sketch
  float* ws_min;  // [B][Hq][S] lowest score of each tier-0 split (written when spike != null)
  int* spike;     // [B][Hq] spike flags, or null
  int* err;       // the call's device error word (KVQ_DEVERR_* bits), zero at launch
  int* status;    // where the combine pass copies the error word, or null
  int gate;       // score-gated value loading
  int batch, hq, hkv, page_size, total_splits;
};

constexpr float kGateLog2 = 23.083120654223414f;  // KVQ_SCORE_GATE_NATS * log2(e): scores are base-2

// Split-K launchers: each runs the tiers of its family (DecTier::kind) and skips the rest.
// Generic kernel, every format pair: one launch per tier.
cudaError_t launch_decode(const DecParams& p, int head_dim, int group, cudaStream_t stream);
// Fused tensor-core decode for head_dim 128, 1, 2 or 4 query heads per kv head, tiers stored
// as fp16/fp16 or fp8-E4M3/INT4-g32 (one launch for all of them).  `counter`: one int of
// device scratch, zero at launch.
bool gqa_fast_supported(int head_dim, int group, int k_fmt, int v_fmt);
int gqa_max_chunk_tokens();
// trigger: a codebook split-K launch follows and may start on SMs this grid leaves idle.
cudaError_t launch_decode_gqa(const DecParams& p, int* counter, cudaStream_t stream, bool trigger);
// Fused tensor-core decode over codebook tiers (codebook K and V), head_dim 128 or 256,
// 1, 2 or 4 query heads per kv head; one launch per tier (after one projection launch when
// a tier's keys carry a sketch).  `counters`: the 256-byte counter block, zero at launch
// (ints [0, KVQ_MAX_TIERS) work counters; the error word is DecParams::err).
bool cb_fast_supported(int head_dim, int group, int k_fmt, int v_fmt);
// after_split_k: a split-K launch of this call precedes; the codebook grids then run as its
// programmatic dependents (overlapping its tail) and complete only after it.
cudaError_t launch_decode_cb(const DecParams& p, int head_dim, int* counters, cudaStream_t stream,
                             bool after_split_k);
cudaError_t launch_combine(const DecParams& p, int head_dim, cudaStream_t stream);

// ------------------------------------------------------------------------ device helpers
__device__ __forceinline__ float fp8e4m3_to_float(uint32_t byte) {
  // exact: every E4M3 value is an fp16 value; the hardware conversion takes two bytes
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)byte));
  return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFF)));
}

// Two floats -> two E4M3 bytes (lo = first element), nearest-even, saturating.
__device__ __forceinline__ uint32_t float2_to_fp8x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace kvq
