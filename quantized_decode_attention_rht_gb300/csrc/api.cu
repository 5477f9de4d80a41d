// C ABI of libkvq.so: argument checks, split-K planning and kernel launches.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "kvq_internal.cuh"

namespace kvq {
bool decode_supports(int k_fmt, int k_bits, int v_fmt, int v_bits);

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}

namespace {

using namespace kvq;

// Streaming multiprocessors of the current device (the split plan sizes its items from
// it), queried once per device; 152 (GB300) if the query fails.
int device_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvq_status side_bytes(int fmt, int bits, int d, size_t* row, size_t* aux) {
  if (d != 64 && d != 128 && d != 256) return KVQ_ERR_UNSUPPORTED;
  // keys with a sketch or an outlier stream are attended by the codebook kernel only
  // (head_dim 128 or 256)
  if ((fmt == KVQ_FMT_CODEBOOK_QJL || fmt == KVQ_FMT_CODEBOOK_OUTLIER) && d == 64) return KVQ_ERR_UNSUPPORTED;
  switch (fmt) {
    case KVQ_FMT_CODEBOOK:
      if (bits < 2 || bits > 4) return KVQ_ERR_UNSUPPORTED;
      *row = (size_t)d * bits / 8;
      *aux = 2;
      return KVQ_OK;
    case KVQ_FMT_CODEBOOK_OUTLIER:  // inlier codes; norm, outlier scale, int8 outlier values
      if (bits < 2 || bits > 4) return KVQ_ERR_UNSUPPORTED;
      *row = (size_t)d * bits / 8;
      *aux = 4 + KVQ_OUTLIER_CHANNELS;
      return KVQ_OK;
    case KVQ_FMT_CODEBOOK_QJL:  // codes, then the sketch's sign bits; norm + residual norm
      if (bits < 2 || bits > 4) return KVQ_ERR_UNSUPPORTED;
      *row = (size_t)d * bits / 8 + KVQ_QJL_DIM / 8;
      *aux = 4;
      return KVQ_OK;
    case KVQ_FMT_FP16: *row = 2 * (size_t)d; *aux = 0; return KVQ_OK;
    case KVQ_FMT_FP8_E4M3: *row = d; *aux = 0; return KVQ_OK;
    case KVQ_FMT_INT4_G32: *row = d / 2; *aux = 2 * (size_t)(d / KVQ_INT4_GROUP); return KVQ_OK;
    default: return KVQ_ERR_INVALID_ARGUMENT;
  }
}

bool is_codebook(int fmt) {
  return fmt == KVQ_FMT_CODEBOOK || fmt == KVQ_FMT_CODEBOOK_QJL || fmt == KVQ_FMT_CODEBOOK_OUTLIER;
}

// One side of a cache; is_key: the side holds keys (only keys may carry a residual sketch).
kvq_status check_side(const kvq_cache* c, int fmt, int bits, const void* rows, const void* aux,
                      const float* cent, const float* bounds, const int8_t* signs, bool need_bounds,
                      bool is_key) {
  size_t rb, ab;
  kvq_status st = side_bytes(fmt, bits, c->head_dim, &rb, &ab);
  if (st != KVQ_OK) return st;
  if (!rows || !aligned(rows, 16) || !signs) return KVQ_ERR_INVALID_ARGUMENT;
  if (ab && (!aux || !aligned(aux, 2))) return KVQ_ERR_INVALID_ARGUMENT;
  if (is_codebook(fmt) && (!cent || (need_bounds && !bounds))) return KVQ_ERR_INVALID_ARGUMENT;
  if (fmt == KVQ_FMT_CODEBOOK_QJL &&
      (!is_key || !c->k_qjl || !aligned(c->k_qjl, 16) || !aligned(aux, 16)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (fmt == KVQ_FMT_CODEBOOK_OUTLIER &&
      (!is_key || !c->k_outliers || !aligned(c->k_outliers, 16) || !aligned(aux, 16)))
    return KVQ_ERR_INVALID_ARGUMENT;
  return KVQ_OK;
}

kvq_status check_cache(const kvq_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (c->num_kv_heads < 1 || c->page_size < 1 || c->num_pages < 0) return KVQ_ERR_INVALID_ARGUMENT;
  if ((long long)c->num_pages * c->page_size > 0x7FFFFFFFLL) return KVQ_ERR_INVALID_ARGUMENT;
  return KVQ_OK;
}

int side_row_bytes(int fmt, int bits, int d) {
  size_t rb = 0, ab = 0;
  side_bytes(fmt, bits, d, &rb, &ab);
  return (int)rb;
}

// Split-K plan: tokens per chunk for each tier (a multiple of page_size).
struct Plan {
  int chunk[KVQ_MAX_TIERS];
  int splits[KVQ_MAX_TIERS];
  int kind[KVQ_MAX_TIERS];  // TierKind: which kernel family runs the tier
  int total;
};

// Pages of the block table a call may use: none for a pool without pages (every length
// above 0 is then out of range: the kernels see an empty tier and the report says so).
int usable_pages(const kvq_tier_view& t) { return t.cache->num_pages > 0 ? t.max_pages : 0; }

size_t token_bytes(const kvq_cache* c) {
  size_t rk, ak, rv, av;
  side_bytes(c->k_format, c->k_bits, c->head_dim, &rk, &ak);
  side_bytes(c->v_format, c->v_bits, c->head_dim, &rv, &av);
  return rk + ak + rv + av;
}

// The kernel family of one tier: the fused fp16 / fp8 + INT4 kernel, the fused codebook
// kernel, or the generic one.  q16: the queries are 16-byte aligned.
int tier_kind(const kvq_cache* c, int group, int split_tokens, bool q16) {
  const bool ps16 = c->page_size == 16;
  if (ps16 && q16 && split_tokens <= gqa_max_chunk_tokens() &&
      gqa_fast_supported(c->head_dim, group, c->k_format, c->v_format) && aligned(c->k_signs, 16) &&
      aligned(c->v_signs, 16))
    return TIER_GQA;
  if (ps16 && cb_fast_supported(c->head_dim, group, c->k_format, c->v_format) && aligned(c->k_aux, 16) &&
      aligned(c->v_aux, 16))  // bulk copies of the norm runs need 16-byte aligned sources
    return TIER_CB;
  return TIER_GENERIC;
}

kvq_status make_plan(const kvq_tier_view* tiers, int n, int batch, int hq, int split_tokens, bool q16, Plan* plan) {
  const kvq_cache* c0 = tiers[0].cache;
  const int ps = c0->page_size, hkv = c0->num_kv_heads, group = hq / hkv;
  if (split_tokens < 0 || split_tokens % ps) return KVQ_ERR_INVALID_ARGUMENT;
  const int kSms = device_sms();
  // fused kernels: items of about equal bytes, several per warp of a full GPU, sized from
  // the bytes of the tiers their launch covers (a small recent-token window gets small items)
  size_t family_bytes[3] = {0, 0, 0};
  for (int i = 0; i < n; ++i) {
    plan->kind[i] = tier_kind(tiers[i].cache, group, split_tokens, q16);
    // the generic kernel's grid has the sequences in its z and the kv heads in its y extent
    if (plan->kind[i] == TIER_GENERIC && (batch > 65535 || hkv > 65535)) return KVQ_ERR_UNSUPPORTED;
    family_bytes[plan->kind[i]] += (size_t)batch * hkv * usable_pages(tiers[i]) * ps * token_bytes(tiers[i].cache);
  }
  plan->total = 0;
  for (int i = 0; i < n; ++i) {
    const long long max_len = (long long)usable_pages(tiers[i]) * ps;
    const int kind = plan->kind[i];
    int chunk = split_tokens;
    if (chunk == 0 && kind != TIER_GENERIC) {
      // items per SM: enough that the last ones to finish leave little idle time.  The
      // codebook kernel's tensor-core path (groups of 2 and 4) spends more time per byte
      // than its FMA path, so its items carry fewer bytes (measured on GB300: 4-bit G = 1
      // best at 72 items per SM, 3/2-bit G = 4 at 288, the fp16 / fp8 kernel at 64)
      const size_t fb = family_bytes[kind];
      const size_t per_sm = kind == TIER_GQA ? 64 : (group >= 2 ? 288 : 72);
      // a group of 8 on the fused kernels makes two items per chunk (heads 0-3 and 4-7):
      // chunks twice as long keep the item count
      const size_t halves = group == 8 ? 2 : 1;
      const size_t item_bytes = std::max<size_t>(16 << 10, halves * fb / (kSms * per_sm));
      size_t tok = item_bytes / token_bytes(tiers[i].cache);
      // the tensor-core path's time per token hardly depends on the code width, so its small
      // caches get items of a fixed token count rather than bytes (measured on GB300 for
      // 4/4- and 3/2-bit codes: 96-112 tokens best for 4 query heads per kv head, 192 for 2)
      if (kind == TIER_CB && group >= 2)
        tok = std::max<size_t>(group >= 4 ? 112 * halves : 192,
                               halves * fb / (kSms * per_sm) / token_bytes(tiers[i].cache));
      const size_t cap = kind == TIER_GQA ? (size_t)gqa_max_chunk_tokens() : (size_t)1 << 20;
      chunk = (int)std::min<size_t>(cap, std::max<size_t>(ps, tok / ps * ps));
    } else if (chunk == 0) {
      // aim at ~16 CTAs per SM in total, chunks of 256 .. 4096 tokens
      const long long work = (long long)batch * hkv * max_len;
      long long want = work / (kSms * 16) + 1;
      long long c = 256;
      while (c < want && c < 4096) c *= 2;
      chunk = (int)c;
      if (chunk % ps) chunk = (chunk / ps + 1) * ps;
    }
    plan->chunk[i] = chunk;
    plan->splits[i] = max_len == 0 ? 0 : (int)((max_len + chunk - 1) / chunk);
    plan->total += plan->splits[i];
  }
  // Chunks sized for the item count are short where few (sequence, kv head) pairs share a
  // long block table (batch 1 at long context): one sequence would then need more splits
  // than the combine pass holds.  The chunks the library chose double, each within its
  // kernel's longest, until the splits fit; a plan that already fits stays as it is.
  while (split_tokens == 0 && plan->total > KVQ_MAX_SPLITS) {
    bool grew = false;
    plan->total = 0;
    for (int i = 0; i < n; ++i) {
      const long long cap = plan->kind[i] == TIER_GQA ? gqa_max_chunk_tokens()
                                                      : std::max<long long>(ps, (1LL << 20) / ps * ps);
      const long long next = std::min<long long>(cap, 2LL * plan->chunk[i]);
      if (next > plan->chunk[i]) {
        plan->chunk[i] = (int)next;
        grew = true;
      }
      const long long max_len = (long long)usable_pages(tiers[i]) * ps;
      plan->splits[i] = max_len == 0 ? 0 : (int)((max_len + plan->chunk[i] - 1) / plan->chunk[i]);
      plan->total += plan->splits[i];
    }
    if (!grew) break;
  }
  // the combine pass keeps the per-split weights of one output in shared memory
  if (plan->total > KVQ_MAX_SPLITS) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// log2 of a page size that is a power of two, else -1 (the quantize kernels then divide)
int page_shift_of(int page_size) {
  for (int s = 0; s < 31; ++s)
    if ((1 << s) == page_size) return s;
  return -1;
}

kvq_status check_tiers(const kvq_tier_view* tiers, int n, int batch, int hq) {
  if (!tiers || n < 1 || n > KVQ_MAX_TIERS || batch < 0 || hq < 1) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_cache* c0 = tiers[0].cache;
  kvq_status st = check_cache(c0);
  if (st != KVQ_OK) return st;
  if (hq % c0->num_kv_heads) return KVQ_ERR_INVALID_ARGUMENT;
  const int g = hq / c0->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return KVQ_ERR_UNSUPPORTED;
  for (int i = 0; i < n; ++i) {
    const kvq_cache* c = tiers[i].cache;
    if ((st = check_cache(c)) != KVQ_OK) return st;
    if (c->head_dim != c0->head_dim || c->num_kv_heads != c0->num_kv_heads || c->page_size != c0->page_size)
      return KVQ_ERR_INVALID_ARGUMENT;
    if (c->k_signs != c0->k_signs || c->v_signs != c0->v_signs) return KVQ_ERR_INVALID_ARGUMENT;
    if (tiers[i].max_pages < 0 || (tiers[i].max_pages > 0 && (!tiers[i].block_table || !tiers[i].seq_lens)))
      return KVQ_ERR_INVALID_ARGUMENT;
    if (!tiers[i].seq_lens) return KVQ_ERR_INVALID_ARGUMENT;
    if ((st = check_side(c, c->k_format, c->k_bits, c->k_rows, c->k_aux, c->k_centroids, c->k_bounds,
                         c->k_signs, false, true)) != KVQ_OK)
      return st;
    if ((st = check_side(c, c->v_format, c->v_bits, c->v_rows, c->v_aux, c->v_centroids, c->v_bounds,
                         c->v_signs, false, false)) != KVQ_OK)
      return st;
    if (c->k_format == KVQ_FMT_CODEBOOK_QJL) {
      for (int j = 0; j < n; ++j)
        if (tiers[j].cache->k_format == KVQ_FMT_CODEBOOK_QJL && tiers[j].cache->k_qjl != c->k_qjl)
          return KVQ_ERR_INVALID_ARGUMENT;  // one projection for every tier attended together
    } else if (c->k_format == KVQ_FMT_CODEBOOK_OUTLIER) {
      // the codebook kernel family; checked below
    } else if (!decode_supports(c->k_format, c->k_bits, c->v_format, c->v_bits)) {
      return KVQ_ERR_UNSUPPORTED;
    }
  }
  // keys with a residual sketch or an outlier stream run on the fused codebook kernel only
  for (int i = 0; i < n; ++i) {
    const kvq_cache* c = tiers[i].cache;
    if ((c->k_format == KVQ_FMT_CODEBOOK_QJL || c->k_format == KVQ_FMT_CODEBOOK_OUTLIER) &&
        tier_kind(c, g, 0, false) != TIER_CB)
      return KVQ_ERR_UNSUPPORTED;
  }
  return KVQ_OK;
}

bool has_sketch(const kvq_tier_view* tiers, int n) {
  for (int i = 0; i < n; ++i)
    if (tiers[i].cache->k_format == KVQ_FMT_CODEBOOK_QJL) return true;
  return false;
}

// Workspace: partial accumulators [B][Hq][S][D], (max, sum) [B][Hq][S][2], each split's
// lowest score [B][Hq][S] (spike flags), with keys that carry a sketch the projected queries
// [B][Hq][KVQ_QJL_DIM], then the work counters.
size_t workspace_bytes(int batch, int hq, int d, int total_splits, bool sketch) {
  const size_t parts = (size_t)batch * hq * total_splits;
  const size_t pq = sketch ? align_up((size_t)batch * hq * KVQ_QJL_DIM * sizeof(float), 256) : 0;
  return align_up(parts * d * sizeof(float), 256) + align_up(parts * 2 * sizeof(float), 256) +
         align_up(parts * sizeof(float), 256) + pq + 256;
}

}  // namespace

extern "C" {

KVQ_API const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARGUMENT: return "KVQ_ERR_INVALID_ARGUMENT";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "KVQ_ERR_WORKSPACE_TOO_SMALL";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
  }
  return "KVQ_ERR_UNKNOWN";
}

KVQ_API uint64_t kvq_kernel_launches(void) { return kvq::g_launches.load(std::memory_order_relaxed); }

KVQ_API kvq_status kvq_row_bytes(int32_t format, int32_t bits, int32_t head_dim, size_t* row_bytes,
                                 size_t* aux_bytes) {
  if (!row_bytes || !aux_bytes) return KVQ_ERR_INVALID_ARGUMENT;
  return side_bytes(format, bits, head_dim, row_bytes, aux_bytes);
}

namespace {
// The destination sides (K, V) of an append or a re-encode into cache c.
void fill_sides(const kvq_cache* c, QuantParams* p) {
  const int fmts[2] = {c->k_format, c->v_format}, bits[2] = {c->k_bits, c->v_bits};
  void* rows[2] = {c->k_rows, c->v_rows};
  void* aux[2] = {c->k_aux, c->v_aux};
  const float* bnd[2] = {c->k_bounds, c->v_bounds};
  const float* cnt[2] = {c->k_centroids, c->v_centroids};
  const int8_t* sg[2] = {c->k_signs, c->v_signs};
  for (int i = 0; i < 2; ++i) {
    p->side[i].rows = static_cast<uint8_t*>(rows[i]);
    p->side[i].aux = static_cast<__half*>(aux[i]);
    p->side[i].bounds = bnd[i];
    p->side[i].centroids = cnt[i];
    p->side[i].qjl = i == 0 ? c->k_qjl : nullptr;
    p->side[i].outl = i == 0 ? c->k_outliers : nullptr;
    p->side[i].signs = sg[i];
    p->side[i].fmt = fmts[i];
    p->side[i].bits = bits[i];
    p->side[i].row_bytes = side_row_bytes(fmts[i], bits[i], c->head_dim);
  }
}
}  // namespace

KVQ_API kvq_status kvq_outlier_calibrate(const uint16_t* k, int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t* out_idx, void* stream) {
  if (!k || !out_idx || !aligned(k, 4) || !aligned(out_idx, 4) || num_tokens < 1 || num_kv_heads < 1)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (head_dim != 128 && head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  cudaError_t e = launch_outlier_calibrate(k, num_tokens, num_kv_heads, head_dim, out_idx,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API kvq_status kvq_requantize(const kvq_cache* src, const int32_t* src_slots, const kvq_cache* dst,
                                  const int32_t* dst_slots, int32_t num_tokens, void* stream) {
  kvq_status st = check_cache(src);
  if (st != KVQ_OK || (st = check_cache(dst)) != KVQ_OK) return st;
  if (num_tokens < 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (src->k_format != KVQ_FMT_FP16 || src->v_format != KVQ_FMT_FP16) return KVQ_ERR_UNSUPPORTED;
  if (dst->k_format == KVQ_FMT_CODEBOOK_OUTLIER) return KVQ_ERR_UNSUPPORTED;
  if (src->head_dim != dst->head_dim || src->num_kv_heads != dst->num_kv_heads ||
      src->page_size != dst->page_size || src->k_signs != dst->k_signs || src->v_signs != dst->v_signs)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!src->k_rows || !src->v_rows || !aligned(src->k_rows, 16) || !aligned(src->v_rows, 16))
    return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_cache* c = dst;
  if ((st = check_side(c, c->k_format, c->k_bits, c->k_rows, c->k_aux, c->k_centroids, c->k_bounds, c->k_signs,
                       true, true)) != KVQ_OK ||
      (st = check_side(c, c->v_format, c->v_bits, c->v_rows, c->v_aux, c->v_centroids, c->v_bounds, c->v_signs,
                       true, false)) != KVQ_OK)
    return st;
  if (num_tokens == 0) return KVQ_OK;
  if (!src_slots || !dst_slots || !aligned(src_slots, 4) || !aligned(dst_slots, 4)) return KVQ_ERR_INVALID_ARGUMENT;
  QuantParams p;
  memset(&p, 0, sizeof(p));
  fill_sides(dst, &p);
  p.src_rows[0] = static_cast<const uint8_t*>(src->k_rows);
  p.src_rows[1] = static_cast<const uint8_t*>(src->v_rows);
  p.src_slots = src_slots;
  p.src_num_slots = src->num_pages * src->page_size;
  p.slots = dst_slots;
  p.num_tokens = num_tokens;
  p.hkv = dst->num_kv_heads;
  p.page_size = dst->page_size;
  p.page_shift = page_shift_of(dst->page_size);
  p.num_slots = dst->num_pages * dst->page_size;
  p.kind_first = 0;
  p.num_kinds = 2;
  p.num_vectors = 2LL * num_tokens * dst->num_kv_heads;
  if (p.num_slots == 0 || p.src_num_slots == 0) return KVQ_OK;
  if ((long long)num_tokens * dst->num_kv_heads > (1LL << 28)) return KVQ_ERR_INVALID_ARGUMENT;
  cudaError_t e = launch_requantize(p, dst->head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API kvq_status kvq_quantize_append(const kvq_cache* cache, const uint16_t* k, const uint16_t* v,
                                       int32_t num_tokens, const int32_t* slot_mapping, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return KVQ_OK;  // nothing to append (an empty tensor may have no address)
  if (!k && !v) return KVQ_ERR_INVALID_ARGUMENT;
  if (!slot_mapping || !aligned(slot_mapping, 4)) return KVQ_ERR_INVALID_ARGUMENT;
  if ((k && !aligned(k, 16)) || (v && !aligned(v, 16))) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_cache* c = cache;
  if (k && (st = check_side(c, c->k_format, c->k_bits, c->k_rows, c->k_aux, c->k_centroids, c->k_bounds,
                            c->k_signs, true, true)) != KVQ_OK)
    return st;
  if (v && (st = check_side(c, c->v_format, c->v_bits, c->v_rows, c->v_aux, c->v_centroids, c->v_bounds,
                            c->v_signs, true, false)) != KVQ_OK)
    return st;
  QuantParams p;
  memset(&p, 0, sizeof(p));
  p.x[0] = k;
  p.x[1] = v;
  fill_sides(c, &p);
  p.slots = slot_mapping;
  p.num_tokens = num_tokens;
  p.hkv = c->num_kv_heads;
  p.page_size = c->page_size;
  p.page_shift = page_shift_of(c->page_size);
  p.num_slots = c->num_pages * c->page_size;
  p.kind_first = k ? 0 : 1;
  p.num_kinds = (k && v) ? 2 : 1;
  p.num_vectors = (long long)p.num_kinds * num_tokens * c->num_kv_heads;
  if (p.num_slots == 0) return KVQ_OK;
  cudaError_t e = launch_quantize(p, c->head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API kvq_status kvq_decode_workspace_size(const kvq_tier_view* tiers, int32_t num_tiers, int32_t batch,
                                             int32_t num_q_heads, int32_t split_tokens, size_t* bytes) {
  if (!bytes) return KVQ_ERR_INVALID_ARGUMENT;
  kvq_status st = check_tiers(tiers, num_tiers, batch, num_q_heads);
  if (st != KVQ_OK) return st;
  // the plan depends on whether q is 16-byte aligned (the fused fp16 / fp8 kernel loads it in
  // 16-byte pieces): size for the larger of the two, so any valid q fits
  size_t most = 0;
  for (const bool q16 : {true, false}) {
    Plan plan;
    if ((st = make_plan(tiers, num_tiers, batch, num_q_heads, split_tokens, q16, &plan)) != KVQ_OK) return st;
    most = std::max(most, workspace_bytes(batch, num_q_heads, tiers[0].cache->head_dim, plan.total,
                                          has_sketch(tiers, num_tiers)));
  }
  *bytes = most;
  return KVQ_OK;
}

KVQ_API kvq_status kvq_decode_attention(const kvq_tier_view* tiers, int32_t num_tiers, const uint16_t* q,
                                        int32_t batch, int32_t num_q_heads, int32_t split_tokens, float* out,
                                        void* workspace, size_t ws_bytes, void* stream) {
  return kvq_decode_attention_ex(tiers, num_tiers, q, batch, num_q_heads, split_tokens, out, workspace, ws_bytes,
                                 nullptr, stream);
}

KVQ_API kvq_status kvq_decode_attention_ex(const kvq_tier_view* tiers, int32_t num_tiers, const uint16_t* q,
                                           int32_t batch, int32_t num_q_heads, int32_t split_tokens, float* out,
                                           void* workspace, size_t ws_bytes, const kvq_decode_options* options,
                                           void* stream) {
  kvq_status st = check_tiers(tiers, num_tiers, batch, num_q_heads);
  if (st != KVQ_OK) return st;
  if (options && options->spike_flags && !aligned(options->spike_flags, 4)) return KVQ_ERR_INVALID_ARGUMENT;
  if (options && options->status && !aligned(options->status, 4)) return KVQ_ERR_INVALID_ARGUMENT;
  if (batch == 0) return KVQ_OK;
  if (!q || !out || !aligned(q, 4) || !aligned(out, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  const kvq_cache* c0 = tiers[0].cache;
  const int d = c0->head_dim, hkv = c0->num_kv_heads;
  Plan plan;
  if ((st = make_plan(tiers, num_tiers, batch, num_q_heads, split_tokens, aligned(q, 16), &plan)) != KVQ_OK)
    return st;
  const bool sketch = has_sketch(tiers, num_tiers);
  const size_t need = workspace_bytes(batch, num_q_heads, d, plan.total, sketch);
  if (need > 0 && (!workspace || !aligned(workspace, 256))) return KVQ_ERR_INVALID_ARGUMENT;
  if (ws_bytes < need) return KVQ_ERR_WORKSPACE_TOO_SMALL;

  DecParams p;
  memset(&p, 0, sizeof(p));
  p.num_tiers = num_tiers;
  int at = 0;
  for (int i = 0; i < num_tiers; ++i) {
    const kvq_cache* c = tiers[i].cache;
    DecTier& t = p.tier[i];
    t.k_rows = static_cast<const uint8_t*>(c->k_rows);
    t.v_rows = static_cast<const uint8_t*>(c->v_rows);
    t.k_aux = static_cast<const __half*>(c->k_aux);
    t.v_aux = static_cast<const __half*>(c->v_aux);
    t.k_cent = c->k_centroids;
    t.k_qjl = c->k_qjl;
    t.k_outl = c->k_outliers;
    t.v_cent = c->v_centroids;
    t.block_table = tiers[i].block_table;
    t.seq_lens = tiers[i].seq_lens;
    t.k_fmt = c->k_format;
    t.v_fmt = c->v_format;
    t.k_bits = c->k_bits;
    t.v_bits = c->v_bits;
    t.k_row_bytes = side_row_bytes(c->k_format, c->k_bits, d);
    t.v_row_bytes = side_row_bytes(c->v_format, c->v_bits, d);
    t.num_pages = c->num_pages;
    t.max_pages = usable_pages(tiers[i]);
    t.split_begin = at;
    t.num_splits = plan.splits[i];
    t.chunk = plan.chunk[i];
    t.kind = plan.kind[i];
    at += plan.splits[i];
  }
  p.q = reinterpret_cast<const __half*>(q);
  p.k_signs = c0->k_signs;
  p.v_signs = c0->v_signs;
  p.out = out;
  const size_t parts = (size_t)batch * num_q_heads * plan.total;
  p.ws_acc = static_cast<float*>(workspace);
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + align_up(parts * d * sizeof(float), 256));
  p.ws_min = reinterpret_cast<float*>(reinterpret_cast<char*>(p.ws_ml) + align_up(parts * 2 * sizeof(float), 256));
  p.ws_pq = sketch ? reinterpret_cast<float*>(reinterpret_cast<char*>(p.ws_min) + align_up(parts * sizeof(float), 256))
                   : nullptr;
  p.spike = options ? options->spike_flags : nullptr;
  p.status = options ? options->status : nullptr;
  p.gate = options && options->score_gate ? 1 : 0;
  p.batch = batch;
  p.hq = num_q_heads;
  p.hkv = hkv;
  p.page_size = c0->page_size;
  p.total_splits = plan.total;
  // one split-K launch per kernel family present (the fused fp16 / fp8 + INT4 kernel takes
  // all its tiers at once, the codebook and generic kernels one launch per tier), all
  // writing partials into the one workspace, then the combine pass over every tier
  int* counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + need - 256);
  p.err = counters + kErrorWord;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool fam[3] = {false, false, false};
  for (int i = 0; i < num_tiers; ++i) fam[plan.kind[i]] = true;
  cudaError_t e = cudaMemsetAsync(counters, 0, 256, s);  // work counters and the error word
  if (e == cudaSuccess && fam[TIER_GQA]) e = launch_decode_gqa(p, counters + kGqaCounter, s, fam[TIER_CB]);
  if (e == cudaSuccess && fam[TIER_CB]) e = launch_decode_cb(p, d, counters, s, fam[TIER_GQA]);
  if (e == cudaSuccess && fam[TIER_GENERIC]) e = launch_decode(p, d, num_q_heads / hkv, s);
  if (e == cudaSuccess) e = launch_combine(p, d, s);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // extern "C"
