/*
 * kvq.h -- rotate-then-quantize KV-cache compression and decode attention that reads
 * the compressed cache directly.  C ABI of libkvq.so (CUDA, sm_103a / GB300).
 *
 * The method (sources named by page title and section):
 *   - "Shrinking the LLM KV Cache by 8x on CPU: The Engineering Behind AdapTQ",
 *     "The Math Fix: Hadamard Accelerated Rotation (HAR)": a random sign flip and a
 *     Fast Walsh-Hadamard Transform spread outlier energy over all coordinates before
 *     scalar quantisation; "Engineering the Hot Path": the query is rotated once and
 *     the attention loop never expands the cache back to full precision.
 *   - "I Ported a Google Research Paper to Apple Silicon" (VeloxQuant-MLX), "Stage 1:
 *     Random Rotation" (x~ = H diag(s) x / sqrt(d)), "Stage 2: Lloyd-Max Scalar
 *     Quantization" (unit norm, fp16 norm, nearest Lloyd-Max centroid per coordinate),
 *     "The Bit-Packing Problem" (little-endian bit stream per vector).
 *   - "FoveatedKV", "The VR headset thing" (a near tier of fp16 tokens and a far tier of
 *     fp8 E4M3 keys and INT4 values, all in one softmax) and "Making it fast" (one fused
 *     split-K dispatch over both tiers, query pre-scaled by 1/sqrt(D), online softmax
 *     computing each exp once).
 *   - "XQuant KV Cache Rematerialization", step 4: scores = q K^T / sqrt(d), softmax,
 *     times V -- the result every entry point below must reproduce.
 *
 * Conventions that hold for every function:
 *   - Pointers are DEVICE pointers unless the comment says "host".
 *   - The caller owns every buffer.  The library allocates nothing, keeps no mutable
 *     global state besides a kernel-launch counter (kvq_kernel_launches) and a per-device
 *     note of the kernels whose shared-memory limit it has raised (both atomic;
 *     kvq_decode_attention_noalloc, at the end, adds its scratch array), never
 *     synchronises, and is safe to call from several threads.
 *   - GPU work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and ordered with the caller's other work on that stream.
 *   - Arguments are checked on the host before anything is launched; a failed check
 *     returns a status != KVQ_OK and launches nothing.  A launch failure returns
 *     KVQ_ERR_CUDA.  Faults inside a kernel surface at the caller's next synchronisation.
 *   - fp16 data is passed as raw IEEE binary16 bits (uint16_t).
 *   - Inputs must be finite.  Outputs must not alias inputs.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_API __attribute__((visibility("default")))

#define KVQ_MAX_TIERS 4  /* decode attends over at most this many tiers at once */
#define KVQ_MAX_SPLITS 1024  /* split-K chunks per sequence, summed over the tiers */
#define KVQ_INT4_GROUP 32 /* coordinates sharing one fp16 scale in KVQ_FMT_INT4_G32 */
#define KVQ_QJL_DIM 128   /* rows m of the residual sketch's projection (KVQ_FMT_CODEBOOK_QJL) */
#define KVQ_OUTLIER_CHANNELS 8  /* outlier channels per kv head (KVQ_FMT_CODEBOOK_OUTLIER) */

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, misaligned buffer       */
  KVQ_ERR_UNSUPPORTED = 2,        /* valid but not built: head_dim, bits, format pair */
  KVQ_ERR_WORKSPACE_TOO_SMALL = 3,
  KVQ_ERR_CUDA = 4                /* a CUDA launch or runtime call failed            */
} kvq_status;

/* How the rows of one side (K or V) of a tier are stored.  Every format stores the
 * ROTATED vector x~ = H diag(s) x / sqrt(D) of the fp16 input x.
 *   KVQ_FMT_CODEBOOK : b-bit indices (b = 2, 3, 4) of the nearest centroid of
 *                      u = sqrt(D) x~ / ||x~||, packed little-endian (element j in bits
 *                      j*b .. j*b+b-1 of the row's bit stream, bit k of the stream is
 *                      bit k%8 of byte k/8); side data: fp16 ||x~|| per row.  Decodes
 *                      to ||x~||_fp16 * C[idx] / sqrt(D).
 *   KVQ_FMT_FP16     : x~ rounded to fp16 (near tier).
 *   KVQ_FMT_FP8_E4M3 : x~ rounded to OCP fp8 E4M3, nearest-even, saturating at +-448
 *                      (far-tier keys).
 *   KVQ_FMT_INT4_G32 : per 32 consecutive coordinates, s = fp16(max|x~| / 7) and
 *                      q = clamp(rint(x~ / s), -7, 7) stored as the nibble q + 8
 *                      (even coordinate in the low nibble); side data: the fp16 scales
 *                      (far-tier values).
 *   KVQ_FMT_CODEBOOK_QJL (keys only; VeloxQuant-MLX page, "Stage 3: QJL Residual
 *                      Correction" -- TurboQuantProd): the KVQ_FMT_CODEBOOK row, then
 *                      KVQ_QJL_DIM sign bits z_j = [ (S r~)_j >= 0 ] of the residual
 *                      r~ = x~ - (the decoded x~) under the cache's projection S
 *                      (k_qjl), LSB-first; side data: fp16 [2] = (||x~||, ||r~||).
 *                      Decode adds ||r~|| sqrt(pi/2) / KVQ_QJL_DIM * sum_j (2 z_j - 1)
 *                      <S_j, q~> to the key's inner product with the rotated query q~
 *                      (the unbiased estimator of <q~, r~>).
 *   KVQ_FMT_CODEBOOK_OUTLIER (keys only; VeloxQuant-MLX page, "Outlier Two-Stream
 *                      Cache"): the kv head's KVQ_OUTLIER_CHANNELS outlier channels c_j
 *                      (k_outliers, indices of the UNROTATED vector, e.g. from
 *                      kvq_outlier_calibrate) are stored as int8 with a per-token scale,
 *                      s = fp16(max_j |x_cj| / 127), q_j = clamp(rint(x_cj / s), -127,
 *                      127); the rest of the vector, those channels set to zero, is
 *                      rotated and stored as a KVQ_FMT_CODEBOOK row.  Side data: 4 +
 *                      KVQ_OUTLIER_CHANNELS bytes per row = fp16 norm, fp16 s, then the
 *                      int8 q_j in channel-list order.  Decode adds sum_j q[c_j] q_j s
 *                      (unrotated query) to the inlier inner product.
 * Rounding decisions are taken on float32 values. */
typedef enum kvq_format {
  KVQ_FMT_CODEBOOK = 0,
  KVQ_FMT_FP16 = 1,
  KVQ_FMT_FP8_E4M3 = 2,
  KVQ_FMT_INT4_G32 = 3,
  KVQ_FMT_CODEBOOK_QJL = 4,
  KVQ_FMT_CODEBOOK_OUTLIER = 5
} kvq_format;

/* One tier of a paged cache.  A token of a sequence at position t lives in physical
 * page block_table[t / page_size] at slot t % page_size; "slot" = page * page_size +
 * offset addresses the pool directly.
 *   rows : uint8 [num_pages][num_kv_heads][page_size][row_bytes], 16-byte aligned
 *   aux  : fp16  [num_pages][num_kv_heads][page_size]          (codebook: norms)
 *          fp16  [num_pages][num_kv_heads][page_size][2]        (codebook + sketch:
 *                                                                norm, residual norm)
 *          fp16  [num_pages][num_kv_heads][page_size][D/32]     (INT4: group scales)
 *          uint8 [num_pages][num_kv_heads][page_size][12]       (codebook + outlier
 *                                                                stream, 16-byte aligned)
 *          unused (may be NULL) for fp16 / fp8.
 * row_bytes / aux bytes per row come from kvq_row_bytes().  Codebook tables are fp32:
 * centroids [2^bits] increasing, bounds [2^bits - 1] with centroids[i] < bounds[i] <
 * centroids[i+1]; a coordinate gets the index #{i : u > bounds[i]}.  Signs are the
 * Rademacher diagonal, int8 +1/-1 [num_kv_heads][head_dim]; every tier attended in one
 * decode call must use the same K signs and the same V signs. */
typedef struct kvq_cache {
  int32_t head_dim;     /* D: 64, 128 or 256; keys with an outlier stream 128 or 256, keys
                           with a sketch are appended at 128 or 256 and decoded at 128;
                           anything else returns KVQ_ERR_UNSUPPORTED */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t page_size;    /* tokens per page, >= 1; 16 is the size the fused decode kernels
                           take, any other decodes on the generic kernel (a decode of keys
                           with a sketch or an outlier stream needs 16, else
                           KVQ_ERR_UNSUPPORTED; appends take any size) */
  int32_t num_pages;    /* pages in the pool */
  int32_t k_format;     /* kvq_format of keys   */
  int32_t v_format;     /* kvq_format of values */
  int32_t k_bits;       /* 2, 3 or 4 when k_format is a codebook format, else ignored */
  int32_t v_bits;
  void* k_rows;
  void* v_rows;
  void* k_aux;
  void* v_aux;
  const float* k_centroids; /* codebook format only */
  const float* k_bounds;
  const float* v_centroids;
  const float* v_bounds;
  const int8_t* k_signs;
  const int8_t* v_signs;
  const float* k_qjl;       /* KVQ_FMT_CODEBOOK_QJL keys only: the projection S, fp32
                               [KVQ_QJL_DIM][head_dim] (iid N(0,1) entries), 16-byte
                               aligned; the same for every tier attended together */
  const int32_t* k_outliers; /* KVQ_FMT_CODEBOOK_OUTLIER keys only: int32
                               [num_kv_heads][KVQ_OUTLIER_CHANNELS] distinct channels in
                               [0, head_dim), 16-byte aligned */
} kvq_cache;

/* One tier as seen by a decode call: the cache plus each sequence's pages and length.
 *   block_table : int32 [batch][max_pages]; entries past a sequence's length unused
 *   seq_lens    : int32 [batch], 0 <= seq_lens[b] <= max_pages * page_size           */
typedef struct kvq_tier_view {
  const kvq_cache* cache; /* host pointer */
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t max_pages;
} kvq_tier_view;

/* Human-readable name of a status.  Never NULL. */
KVQ_API const char* kvq_status_string(kvq_status status);

/* Number of GPU kernels this library has launched since it was loaded, over every device
 * and stream (host-side count, incremented at each successful launch; memsets are not
 * kernels and are not counted).  No counterpart in the pages: it lets a caller state how
 * many kernels a timed region ran.  Thread-safe; never fails. */
KVQ_API uint64_t kvq_kernel_launches(void);

/* Bytes of one stored row and of its side data (host outputs) for a format, code bits
 * and head_dim.  Layouts are those of kvq_format above. */
KVQ_API kvq_status kvq_row_bytes(int32_t format, int32_t bits, int32_t head_dim,
                                 size_t* row_bytes, size_t* aux_bytes);

/* Lloyd-Max codebook for N(0,1) with 2^bits levels (bits 1..8), computed on the host in
 * double precision: boundaries at the midpoints of neighbouring centroids, each centroid
 * the conditional mean of N(0,1) over its cell (VeloxQuant-MLX page, "Stage 2"), the
 * outer cells ending at +-8.  host centroids [2^bits], host bounds [2^bits - 1]. */
KVQ_API kvq_status kvq_lloyd_max_codebook(int32_t bits, double* centroids, double* bounds);

/* Symmetric uniform codebook c_i = (i - (2^bits - 1)/2) * delta with the step delta that
 * minimises the N(0,1) mean squared error; boundaries at midpoints.  Host outputs. */
KVQ_API kvq_status kvq_uniform_codebook(int32_t bits, double* centroids, double* bounds);

/* Rademacher sign vectors of the rotation for one layer (VeloxQuant-MLX page, "Stage 1:
 * Random Rotation": the random +1/-1 diagonal applied before the Walsh-Hadamard transform;
 * AdapTQ page, "The Math Fix": the random sign flip).  Host outputs k_signs and v_signs,
 * int8 [num_kv_heads][head_dim] each, ready to upload as kvq_cache.k_signs / v_signs.
 * Sign j of kv head h on side s (0 keys, 1 values) is +1 if the lowest bit of the first
 * output of a SplitMix64 generator whose state starts at
 *     seed XOR (layer * 2^40 + s * 2^32 + h * 2^16 + j)
 * is 0, else -1 (SplitMix64: state += 0x9E3779B97F4A7C15; z = state; z = (z ^ z >> 30) *
 * 0xBF58476D1CE4E5B9; z = (z ^ z >> 27) * 0x94D049BB133111EB; output z ^ z >> 31).  The
 * same (seed, layer) always gives the same signs.  0 <= layer < 2^24, 1 <= num_kv_heads <=
 * 2^16 (else KVQ_ERR_INVALID_ARGUMENT); head_dim 64, 128 or 256 (else
 * KVQ_ERR_UNSUPPORTED); null outputs: KVQ_ERR_INVALID_ARGUMENT. */
KVQ_API kvq_status kvq_make_signs(uint64_t seed, int32_t layer, int32_t num_kv_heads, int32_t head_dim,
                                  int8_t* k_signs, int8_t* v_signs);

/* float32 tables for the device: centroids32[i] = (float)centroids[i] and bounds32[i] =
 * (float)(((double)centroids32[i] + centroids32[i+1]) / 2).  All host arrays. */
KVQ_API kvq_status kvq_codebook_tables(int32_t bits, const double* centroids,
                                       float* centroids32, float* bounds32);

/* Quantise-and-append: for every token i < num_tokens and kv head h, rotate
 * k[i][h][:] (fp16, [num_tokens][num_kv_heads][head_dim]) with k_signs[h], encode it in
 * cache->k_format and store it at pool slot slot_mapping[i]; the same for v with v_signs.
 * k or v may be NULL to append only the other side (not both, unless num_tokens is 0:
 * an empty append returns KVQ_OK whatever the pointers).  slot_mapping: int32
 * [num_tokens]; a negative slot skips the token; slots >= num_pages * page_size are
 * skipped too.  Two tokens of one call must not share a slot.  k, v: 16-byte aligned.
 * Up to 16384 vectors per side (a decode step) take one launch for both sides; larger
 * appends one launch per side (keys with an outlier stream: one launch). */
KVQ_API kvq_status kvq_quantize_append(const kvq_cache* cache, const uint16_t* k,
                                       const uint16_t* v, int32_t num_tokens,
                                       const int32_t* slot_mapping, void* stream);

/* Move tokens from an fp16 tier into another tier, re-encoding their rows: the recent-token
 * window of FoveatedKV's fused kernel ("Making it fast": the unquantised decode buffer in
 * the same dispatch) and AdapTQ's hybrid execution ("Hybrid Execution: The Best of Both
 * Worlds": short contexts stay unquantised, tokens switch to the quantised path past a
 * threshold).  A caller keeps the newest tokens of each sequence in an fp16 tier (appended
 * with kvq_quantize_append, attended with the other tiers in one kvq_decode_attention call)
 * and moves the oldest ones out with this call once the window is full.
 *   src       : host pointer; both sides KVQ_FMT_FP16 (it stores the rotated vector x~)
 *   src_slots : int32 [num_tokens] pool slots of the tokens in src
 *   dst       : host pointer; any formats; same head_dim, num_kv_heads, page_size and the
 *               same K and V sign vectors as src (else KVQ_ERR_INVALID_ARGUMENT)
 *   dst_slots : int32 [num_tokens] destination slots
 * Token i's K and V rows of every kv head are read at src_slots[i] and written, encoded in
 * dst's formats, at dst_slots[i]: the encode of the stored fp16 x~, with no second
 * rotation (so a codebook row of a moved token can differ from appending the original x
 * directly where the fp16 rounding of x~ crosses a decision boundary).  A token whose src
 * or dst slot is negative or out of range is skipped.  src is left unchanged.  A src
 * that is not fp16, or a dst whose keys are KVQ_FMT_CODEBOOK_OUTLIER (its channel split
 * needs the unrotated vector), returns KVQ_ERR_UNSUPPORTED; num_tokens x num_kv_heads above
 * 2^28 returns KVQ_ERR_INVALID_ARGUMENT (split the move). */
KVQ_API kvq_status kvq_requantize(const kvq_cache* src, const int32_t* src_slots,
                                  const kvq_cache* dst, const int32_t* dst_slots,
                                  int32_t num_tokens, void* stream);

/* Calibration of the outlier two-stream cache (VeloxQuant-MLX page, "Outlier Two-Stream
 * Cache", steps 1 and 2): over the first num_tokens tokens of a sequence, the population
 * variance of every channel of every kv head's keys (computed in fp64), and per head the
 * KVQ_OUTLIER_CHANNELS channels of largest variance, largest first, ties to the lower
 * channel.
 *   k          : fp16 [num_tokens][num_kv_heads][head_dim] keys (unrotated), 4-byte aligned
 *   out_idx    : int32 [num_kv_heads][KVQ_OUTLIER_CHANNELS], written
 * head_dim 128 or 256; num_tokens >= 1. */
KVQ_API kvq_status kvq_outlier_calibrate(const uint16_t* k, int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t* out_idx, void* stream);

/* Workspace bytes kvq_decode_attention needs for these tiers and shapes (host output).
 * split_tokens: tokens per split-K chunk (a multiple of page_size), or 0 to let the
 * library choose; pass the same value to kvq_decode_attention.  The chunks of the longest
 * possible sequence (max_pages * page_size tokens per tier), summed over the tiers, may not
 * exceed KVQ_MAX_SPLITS: a smaller split_tokens returns KVQ_ERR_UNSUPPORTED.  With 0 the
 * library sizes chunks for the GPU's item count and lengthens them where a long block table
 * would need more splits (few sequences at long context); chunks of the fused fp16 / fp8
 * kernel stop at 2048 tokens, so its tiers take block tables of at most KVQ_MAX_SPLITS x
 * 2048 tokens in total, other tiers 2^20 tokens a chunk.  A tier on the generic kernel
 * (page sizes other than 16, D = 64, format pairs the fused kernels do not take) takes at
 * most 65535 sequences a call (KVQ_ERR_UNSUPPORTED beyond). */
KVQ_API kvq_status kvq_decode_workspace_size(const kvq_tier_view* tiers, int32_t num_tiers,
                                             int32_t batch, int32_t num_q_heads,
                                             int32_t split_tokens, size_t* bytes);

/* Decode attention for one new query per sequence over all tiers (a split-K pass, then a
 * combine pass).  Each tier goes to the kernel family that fits its formats: fp16/fp16 and
 * fp8/INT4 tiers (D = 128, 1, 2, 4 or 8 query heads per kv head) share one fused launch,
 * codebook tiers (D = 128 or 256; 1, 2 or 4 query heads per kv head, or 8 with plain codes)
 * take one launch each (8 heads run as two 4-head passes over each chunk, the second from
 * L2), anything else (D = 64, other format pairs) the generic kernel, which is much slower
 * (measured on GB300: a 32768-token, batch-32 two-tier cache at D = 64 decodes at ~10% of
 * the HBM copy bandwidth, a D = 64 Llama-7B-shaped codebook layer at ~17%, against ~88% and
 * ~37% on the fused kernels at D = 128):
 *   out[b][h] = softmax_t( q[b][h] . K[t] / sqrt(D) ) V[t]
 * over every cached token t < seq_lens[b] of every tier of kv head h / (Hq / Hkv), where
 * K[t], V[t] are the dequantised cache rows with the rotation undone; keys stored as
 * KVQ_FMT_CODEBOOK_QJL add their sketch's estimate of <q, r> to q . K[t] (one more small
 * launch per call projects every query once).  The query is
 * rotated with the K signs inside the kernel and the result is rotated back with the V
 * signs, so the cache is never expanded.  A sequence with no cached token gives zeros.
 *   tiers : host array [num_tiers], 1..KVQ_MAX_TIERS, same head_dim / num_kv_heads
 *   q     : fp16 [batch][num_q_heads][head_dim]; num_q_heads / num_kv_heads in {1,2,4,8}
 *   out   : fp32 [batch][num_q_heads][head_dim]
 *   workspace : >= kvq_decode_workspace_size() bytes, 256-byte aligned, scratch only. */
KVQ_API kvq_status kvq_decode_attention(const kvq_tier_view* tiers, int32_t num_tiers,
                                        const uint16_t* q, int32_t batch,
                                        int32_t num_q_heads, int32_t split_tokens,
                                        float* out, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Device-side error bits of a decode call.  The kernels check what only the device can see
 * (lengths and block-table entries live in device memory) and never read outside a buffer
 * because of it; a call that raised a bit has a wrong result for the sequences concerned.
 * They reach the caller through kvq_decode_options.status. */
#define KVQ_DEVERR_COPY_TIMEOUT 1 /* a wait for one of the kernel's own bulk copies gave up
                                     after its iteration limit: the work items of that warp
                                     contribute nothing to the result */
#define KVQ_DEVERR_PAGE_INDEX 2   /* a block-table entry outside [0, num_pages): no read is made
                                     through it -- the fused fp16 / fp8 kernel leaves out the
                                     split-K chunk holding it, the codebook kernel reads page 0
                                     in its place, the generic kernel leaves out the page */
#define KVQ_DEVERR_SEQ_LEN 4      /* a seq_lens entry outside [0, max_pages * page_size] (a pool
                                     with num_pages 0 has no room: any length above 0): it is
                                     cut into that range */

/* Options of kvq_decode_attention_ex: two features of the FoveatedKV page's fused kernel
 * ("Making it fast"), and the device error report.  All zero is the plain computation of
 * kvq_decode_attention. */
#define KVQ_SCORE_GATE_NATS 16.0f
typedef struct kvq_decode_options {
  /* Nonzero: score-gated value loading.  A token whose score is more than
   * KVQ_SCORE_GATE_NATS below the running maximum of its split-K chunk (natural-log
   * units: its softmax weight is below exp(-16) of that maximum's) may leave out its value:
   * it still counts in the softmax denominator, but adds nothing to the value sum.  The
   * fused kernels leave out the value work of a 16-token page when every token of it, for
   * every query head of the kv head, qualifies; the generic kernel judges token by token
   * and skips the value row's load.  A running maximum never exceeds the final one, so the
   * output differs from the exact one by at most sum_t w_t |v_t| over the tokens scoring
   * more than 16 nats below the sequence's best (w_t the exact softmax weights). */
  int32_t score_gate;
  /* Optional device int32 [batch][num_q_heads] (4-byte aligned), written when non-NULL:
   * 1 where the best score among the tokens of tiers 1..num_tiers-1 exceeds the worst
   * score among the tokens of tier 0 (a far-tier token outranks a near-tier one -- the
   * page's spike detection), else 0; 0 when tier 0 or the later tiers hold no token of the
   * sequence.  Scores are compared as the kernels compute them (float32). */
  int32_t* spike_flags;
  /* Optional device int32 (4-byte aligned), written when non-NULL by the call's last kernel
   * (stream-ordered, like the output): the OR of the KVQ_DEVERR_* bits the call's kernels
   * raised, 0 when none.  Not written by a call with batch 0 (it launches nothing). */
  int32_t* status;
} kvq_decode_options;

/* kvq_decode_attention with options (NULL options: identical to kvq_decode_attention).
 * Same arguments, workspace and errors, plus: a misaligned spike_flags or status buffer
 * returns KVQ_ERR_INVALID_ARGUMENT. */
KVQ_API kvq_status kvq_decode_attention_ex(const kvq_tier_view* tiers, int32_t num_tiers,
                                           const uint16_t* q, int32_t batch,
                                           int32_t num_q_heads, int32_t split_tokens,
                                           float* out, void* workspace, size_t workspace_bytes,
                                           const kvq_decode_options* options, void* stream);

/* Decode attention for callers that cannot allocate device memory.
 *
 * Same computation, arguments and results as kvq_decode_attention, without the workspace
 * arguments: the split-K scratch is a static device array inside the library, of
 * KVQ_NOALLOC_SCRATCH_BYTES bytes, that every GPU which loads the library holds until the
 * process exits.  This has no counterpart in the pages; it exists for callers that may not
 * call cudaMalloc or any allocating routine -- for example a plugin running inside a
 * serving framework that hands out no device memory, or a serving loop whose memory budget
 * is fixed at start-up and forbids later allocations.  This entry point allocates nothing.
 *
 * The first call made while a given device is current looks up that device's scratch
 * address (cudaGetSymbolAddress) and remembers it.  Under CUDA's lazy module loading that
 * lookup is also what loads the library's device code on that device, and with it the
 * array: the first call may therefore allocate the KVQ_NOALLOC_SCRATCH_BYTES of device
 * memory, and can fail where none is left.  Make one warm-up call per device at start-up,
 * before any stream capture and before the memory budget is fixed.  The remembered address
 * belongs to the device's primary context (the one the CUDA runtime uses).  Shapes needing more than KVQ_NOALLOC_SCRATCH_BYTES of scratch (see
 * kvq_decode_workspace_size) return KVQ_ERR_WORKSPACE_TOO_SMALL and launch nothing.
 * Every call on a device shares the one array and it keeps the last call's contents (each
 * call clears, on its stream, the part that must start at zero); calls whose work overlaps
 * on the GPU (different streams, or different host threads) race on it and must be
 * serialised by the caller. */
#define KVQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_tier_view* tiers, int32_t num_tiers,
                                                const uint16_t* q, int32_t batch,
                                                int32_t num_q_heads, int32_t split_tokens,
                                                float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
