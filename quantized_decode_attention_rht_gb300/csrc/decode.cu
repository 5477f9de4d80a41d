// Split-K decode attention over the packed cache, and the combine pass.
//
// Pass 1 (decode_tier_kernel): one CTA per (split, kv head, sequence) walks a chunk of the
// sequence's pages.  In its prologue it rotates the G = Hq/Hkv queries of the kv head with
// the K signs, x~ = H diag(s) q / sqrt(D) (AdapTQ page, "Engineering the Hot Path": the
// query is rotated once and compared with the stored rotated codes), pre-scaled by
// 1/sqrt(D) (FoveatedKV page, "Making it fast") and by log2(e) so scores come out in base-2
// units.  Per token it dequantises the K row in registers, forms the G scores, updates an
// online softmax (running max / sum, one exp2 per score), and accumulates the value rows,
// still in the rotated domain.  Partials (max, sum, acc[D]) go to the workspace.
// Pass 2 (combine_kernel): one block per (sequence, query head) merges the partials of every
// split of every tier, normalises, and undoes the V rotation, y = s_V * (H y~) / sqrt(D).
//
// Lane layout: LPT lanes share a token, each holding DPL = D/LPT consecutive coordinates
// of the G rotated queries and of the G value accumulators in registers; a warp advances
// TPS = 32/LPT tokens per step.  The four warps of a CTA take alternate pages and merge
// their softmax states at the end.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- storage formats
// 2^x, x <= 0 or -inf (scores in base-2 units relative to a maximum): the hardware
// approximation (relative error below 2^-22), results below 2^-126 flushed to 0.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int BITS>
struct Codebook {
  static constexpr int bits = BITS;
};
struct Fp16 {};
struct Fp8 {};
struct Int4 {};

// Funnel-shifted window over a row: the lane's N words start exactly at bit `bit0`.
template <int N>
__device__ __forceinline__ void load_window(const uint8_t* row, int row_words, int bit0, uint32_t (&w)[N]) {
  const uint32_t* r32 = reinterpret_cast<const uint32_t*>(row);
  const int w0 = bit0 >> 5, sh = bit0 & 31;
  uint32_t raw[N + 1];
#pragma unroll
  for (int i = 0; i <= N; ++i) raw[i] = (w0 + i < row_words) ? __ldg(r32 + w0 + i) : 0u;
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

// Dequantise the lane's DPL coordinates [e0, e0 + DPL) of one row (rotated domain).
// `scale` receives the per-row (codebook: norm / sqrt(D)) or per-group (INT4) factor that
// multiplies every coordinate; it is applied outside the inner loops.
template <class F, int D, int DPL>
struct Row;

template <int BITS, int D, int DPL>
struct Row<Codebook<BITS>, D, DPL> {
  __device__ __forceinline__ static void load(const uint8_t* rows, const __half* aux, size_t rowid,
                                              int row_bytes, int e0, const float* lut,
                                              float (&x)[DPL], float& scale) {
    constexpr int NW = (DPL * BITS + 31) / 32;
    uint32_t w[NW];
    load_window<NW>(rows + rowid * row_bytes, row_bytes / 4, e0 * BITS, w);
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int o = j * BITS;
      uint32_t v = w[o / 32] >> (o % 32);
      if ((o % 32) + BITS > 32) v |= w[o / 32 + 1] << (32 - (o % 32));
      x[j] = lut[v & ((1u << BITS) - 1u)];
    }
    constexpr float inv_sqrt_d = inv_sqrt_dim(D);
    scale = __half2float(aux[rowid]) * inv_sqrt_d;
  }
};

template <int D, int DPL>
struct Row<Fp16, D, DPL> {
  __device__ __forceinline__ static void load(const uint8_t* rows, const __half*, size_t rowid, int row_bytes,
                                              int e0, const float*, float (&x)[DPL], float& scale) {
    const uint2* src = reinterpret_cast<const uint2*>(rows + rowid * row_bytes + 2 * e0);
#pragma unroll
    for (int k = 0; k < DPL / 4; ++k) {
      const uint2 u = __ldg(src + k);
      const __half2 a = *reinterpret_cast<const __half2*>(&u.x);
      const __half2 b = *reinterpret_cast<const __half2*>(&u.y);
      x[4 * k] = __low2float(a);
      x[4 * k + 1] = __high2float(a);
      x[4 * k + 2] = __low2float(b);
      x[4 * k + 3] = __high2float(b);
    }
    scale = 1.0f;
  }
};

template <int D, int DPL>
struct Row<Fp8, D, DPL> {
  __device__ __forceinline__ static void load(const uint8_t* rows, const __half*, size_t rowid, int row_bytes,
                                              int e0, const float*, float (&x)[DPL], float& scale) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(rows + rowid * row_bytes + e0);
#pragma unroll
    for (int k = 0; k < DPL / 4; ++k) {
      const uint32_t u = __ldg(src + k);
      uint32_t h01, h23;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(u & 0xFFFF)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(u >> 16)));
      const __half2 a = *reinterpret_cast<const __half2*>(&h01);
      const __half2 b = *reinterpret_cast<const __half2*>(&h23);
      x[4 * k] = __low2float(a);
      x[4 * k + 1] = __high2float(a);
      x[4 * k + 2] = __low2float(b);
      x[4 * k + 3] = __high2float(b);
    }
    scale = 1.0f;
  }
};

template <int D, int DPL>
struct Row<Int4, D, DPL> {
  __device__ __forceinline__ static void load(const uint8_t* rows, const __half* aux, size_t rowid,
                                              int row_bytes, int e0, const float*, float (&x)[DPL],
                                              float& scale) {
    constexpr int NW = (DPL * 4 + 31) / 32;
    uint32_t w[NW];
    load_window<NW>(rows + rowid * row_bytes, row_bytes / 4, e0 * 4, w);
#pragma unroll
    for (int j = 0; j < DPL; ++j) x[j] = (float)((int)((w[j / 8] >> (4 * (j % 8))) & 0xFu) - 8);
    scale = __half2float(aux[rowid * (D / kGroup) + e0 / kGroup]);
  }
};

template <class F>
__device__ __forceinline__ bool is_codebook() { return false; }
template <>
__device__ __forceinline__ bool is_codebook<Codebook<2>>() { return true; }
template <>
__device__ __forceinline__ bool is_codebook<Codebook<3>>() { return true; }
template <>
__device__ __forceinline__ bool is_codebook<Codebook<4>>() { return true; }

template <int D, int G>
struct Shape {
  static constexpr int DPL = (D / 32 > 32 / G) ? D / 32 : 32 / G;  // coordinates per lane
  static constexpr int LPT = D / DPL;                             // lanes per token
  static constexpr int TPS = 32 / LPT;                            // tokens per warp step
};

// ---------------------------------------------------------------- pass 1
template <int D, int G, class KF, class VF>
__global__ void __launch_bounds__(kWarps * 32) decode_tier_kernel(const DecParams p, int tier_index) {
  using S = Shape<D, G>;
  constexpr int DPL = S::DPL, LPT = S::LPT, TPS = S::TPS;
  const DecTier& T = p.tier[tier_index];
  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  int bits = 0;  // a length out of range is cut into it here and reported by the combine pass
  const int len = checked_len(T.seq_lens[b], T.max_pages, p.page_size, &bits);
  const int t_begin = split * T.chunk;
  if (t_begin >= len) return;  // the combine pass only reads splits that hold tokens
  const int t_end = min(len, t_begin + T.chunk);

  __shared__ float q_s[G][D];
  __shared__ float lut_k[256], lut_v[256];
  __shared__ float w_m[kWarps][G], w_l[kWarps][G], w_mn[kWarps][G];
  __shared__ float w_acc[kWarps][G][D];

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // ---- rotate and pre-scale the group's queries: q' = H (s_K * q) * log2(e) / D
  for (int i = tid; i < G * D; i += kWarps * 32) {
    const int g = i / D, j = i % D;
    const float qv = __half2float(p.q[((size_t)b * p.hq + hk * G + g) * D + j]);
    q_s[g][j] = p.k_signs[hk * D + j] < 0 ? -qv : qv;
  }
  if (is_codebook<KF>()) for (int i = tid; i < 256; i += kWarps * 32) lut_k[i] = i < 16 ? T.k_cent[min(i, (1 << T.k_bits) - 1)] : 0.f;
  if (is_codebook<VF>()) for (int i = tid; i < 256; i += kWarps * 32) lut_v[i] = i < 16 ? T.v_cent[min(i, (1 << T.v_bits) - 1)] : 0.f;
  __syncthreads();
  for (int hs = 1; hs < D; hs <<= 1) {
    for (int i = tid; i < G * D / 2; i += kWarps * 32) {
      const int g = i / (D / 2), k = i % (D / 2);
      const int j = (k / hs) * 2 * hs + (k % hs);
      const float a = q_s[g][j], c = q_s[g][j + hs];
      q_s[g][j] = a + c;
      q_s[g][j + hs] = a - c;
    }
    __syncthreads();
  }
  const int r = lane % LPT, gi = lane / LPT, e0 = r * DPL;
  const bool track = p.spike != nullptr && tier_index == 0;  // lowest score, for spike flags
  float qr[G][DPL], acc[G][DPL], m[G], l[G], mn[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
    mn[g] = INFINITY;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      qr[g][j] = q_s[g][e0 + j] * (kLog2e / (float)D);
      acc[g][j] = 0.f;
    }
  }

  const int p_begin = t_begin / p.page_size, p_end = (t_end + p.page_size - 1) / p.page_size;
  for (int lp = p_begin + warp; lp < p_end; lp += kWarps) {
    const int phys = T.block_table[(size_t)b * T.max_pages + lp];
    int pbits = 0;
    if (!page_in_pool(phys, T.num_pages, &pbits)) {  // warp-uniform: skip the page
      if (lane == 0) atomicOr(p.err, pbits);
      continue;
    }
    const size_t row_base = ((size_t)phys * p.hkv + hk) * p.page_size;
    for (int s0 = 0; s0 < p.page_size; s0 += TPS) {
      const int off = s0 + gi;
      const bool valid = slot_holds_token(lp, off, p.page_size, t_end);
      const size_t rowid = row_base + off;
      float x[DPL], ks = 0.f;
      if (valid) Row<KF, D, DPL>::load(T.k_rows, T.k_aux, rowid, T.k_row_bytes, e0, lut_k, x, ks);
      float sc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
        if (valid) {
#pragma unroll
          for (int j = 0; j < DPL; ++j) a = fmaf(qr[g][j], x[j], a);
        }
#pragma unroll
        for (int o = 1; o < LPT; o <<= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        sc[g] = valid ? a * ks : -INFINITY;
      }
      // online softmax over the TPS tokens of this step
      float pr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = sc[g];
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (mx > m[g]) {
          const float f = exp2_fast(m[g] - mx);  // m = -inf first: f = 0
          l[g] *= f;
#pragma unroll
          for (int j = 0; j < DPL; ++j) acc[g][j] *= f;
          m[g] = mx;
        }
        pr[g] = valid ? exp2_fast(sc[g] - m[g]) : 0.f;
        l[g] += pr[g];
        if (track && valid) mn[g] = fminf(mn[g], sc[g]);
      }
      // score gate: a token far below the running maximum of every head keeps its value
      // row unread; per head, a gated token adds nothing to that head's value sum
      bool need = valid;
      if (p.gate) {
        bool any = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const bool keep = sc[g] - m[g] >= -kGateLog2;
          pr[g] = keep ? pr[g] : 0.f;
          any = any || keep;
        }
        need = need && any;
      }
      if (need) {
        float vs;
        Row<VF, D, DPL>::load(T.v_rows, T.v_aux, rowid, T.v_row_bytes, e0, lut_v, x, vs);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float wgt = pr[g] * vs;
#pragma unroll
          for (int j = 0; j < DPL; ++j) acc[g][j] = fmaf(wgt, x[j], acc[g][j]);
        }
      }
    }
  }
  // ---- merge the token groups of the warp (same running max in every lane)
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) {
      l[g] += __shfl_xor_sync(0xFFFFFFFFu, l[g], o);
      mn[g] = fminf(mn[g], __shfl_xor_sync(0xFFFFFFFFu, mn[g], o));
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[g][j] += __shfl_xor_sync(0xFFFFFFFFu, acc[g][j], o);
    }
  }
  if (gi == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int j = 0; j < DPL; ++j) w_acc[warp][g][e0 + j] = acc[g][j];
      if (r == 0) {
        w_m[warp][g] = m[g];
        w_l[warp][g] = l[g];
        w_mn[warp][g] = mn[g];
      }
    }
  }
  __syncthreads();
  // ---- merge the warps and write this split's partial
  const int split_slot = T.split_begin + split;
  for (int i = tid; i < G * D; i += kWarps * 32) {
    const int g = i / D, j = i % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, w_m[w][g]);
    float a = 0.f, s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (w_m[w][g] == -INFINITY) continue;  // a warp that saw no token
      const float f = exp2_fast(w_m[w][g] - mx);
      a += w_acc[w][g][j] * f;
      s += w_l[w][g] * f;
    }
    const size_t part = ((size_t)b * p.hq + hk * G + g) * p.total_splits + split_slot;
    p.ws_acc[part * D + j] = a;
    if (j == 0) {
      p.ws_ml[2 * part] = mx;
      p.ws_ml[2 * part + 1] = s;
      if (track) {
        float lo = w_mn[0][g];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) lo = fminf(lo, w_mn[w][g]);
        p.ws_min[part] = lo;
      }
    }
  }
}

// ---------------------------------------------------------------- pass 2
// One block of kCombineWarps warps (4, 8 or 16: more where each output has many splits, so
// every warp's chain of loads stays short) per (sequence, query head).  First every thread reads
// the (max, sum) pair of one split (all splits of every tier at once), and the block forms
// the global max and each split's weight exp2(m_s - max); then warp w streams the
// accumulators of splits w, w + kCombineWarps, ... with no dependence between splits (lane
// l holds coordinates [l*D/32, (l+1)*D/32)).  Warp 0 sums the warps, normalises, and
// undoes the V rotation with a Walsh-Hadamard transform (in-register stages for the lane's
// coordinates, shuffles across lanes).  Launched as a programmatic dependent of the split-K
// pass: it waits for that grid's completion before touching the partials.
constexpr int kCombineMaxSplits = KVQ_MAX_SPLITS;  // the plan never makes more splits per output

template <int D, int kCombineWarps>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const DecParams p) {
  constexpr int PER = D / 32;
  __shared__ float s_acc[kCombineWarps][D];
  __shared__ float s_w[kCombineMaxSplits];
  __shared__ int s_part[kCombineMaxSplits];
  __shared__ float s_red[kCombineWarps][2];
  __shared__ float s_spk[kCombineWarps][2];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // partials of the split-K pass are complete
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (p.status && blockIdx.x == 0) {
    // every split-K kernel of the call has completed: their bits are final; block 0 adds
    // the lengths out of range (every kernel cut them into range) and reports
    int bits = 0;
    for (int i = threadIdx.x; i < p.batch * p.num_tiers; i += blockDim.x) {
      const DecTier& T = p.tier[i % p.num_tiers];
      checked_len(T.seq_lens[i / p.num_tiers], T.max_pages, p.page_size, &bits);
    }
    bits = __reduce_or_sync(0xFFFFFFFFu, bits);
    if (lane == 0) s_part[warp] = bits;  // s_part is free until the split list below
    __syncthreads();
    if (threadIdx.x == 0) {
      int all = *reinterpret_cast<volatile int*>(p.err);
      for (int w = 0; w < kCombineWarps; ++w) all |= s_part[w];
      *p.status = all;
    }
    __syncthreads();
  }
  const int pair = blockIdx.x;
  const int b = pair / p.hq, hq = pair % p.hq;
  const int hk = hq / (p.hq / p.hkv);
  const size_t base = ((size_t)b * p.hq + hq) * p.total_splits;
  // ---- splits holding tokens, over every tier: partial indices and (max, sum)
  int n = 0, n0 = 0;  // splits holding tokens; the first n0 are tier 0's
  for (int ti = 0; ti < p.num_tiers; ++ti) {
    const DecTier& T = p.tier[ti];
    int bits = 0;  // the split-K kernels raised any bit already
    const int nt = splits_holding_tokens(checked_len(T.seq_lens[b], T.max_pages, p.page_size, &bits), T.chunk,
                                         T.num_splits);
    for (int s = threadIdx.x; s < nt && n + s < kCombineMaxSplits; s += blockDim.x)
      s_part[n + s] = T.split_begin + s;
    n += nt;
    if (ti == 0) n0 = nt;
  }
  n = min(n, kCombineMaxSplits);  // the plan refuses more splits than this
  __syncthreads();
  float mx = -INFINITY, lsum = 0.f;
  float far_mx = -INFINITY, near_mn = INFINITY;  // spike flags: best far score, worst near score
  for (int s = threadIdx.x; s < n; s += blockDim.x) {
    const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + 2 * (base + s_part[s]));
    s_w[s] = ml.x;
    mx = fmaxf(mx, ml.x);
    if (p.spike) {
      if (s < n0) near_mn = fminf(near_mn, p.ws_min[base + s_part[s]]);
      else far_mx = fmaxf(far_mx, ml.x);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if (lane == 0) s_red[warp][0] = mx;
  if (p.spike) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      far_mx = fmaxf(far_mx, __shfl_xor_sync(0xFFFFFFFFu, far_mx, o));
      near_mn = fminf(near_mn, __shfl_xor_sync(0xFFFFFFFFu, near_mn, o));
    }
    if (lane == 0) {
      s_spk[warp][0] = far_mx;
      s_spk[warp][1] = near_mn;
    }
  }
  __syncthreads();
  mx = s_red[0][0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, s_red[w][0]);
  if (p.spike && threadIdx.x == 0) {
    for (int w = 1; w < kCombineWarps; ++w) {
      far_mx = fmaxf(far_mx, s_spk[w][0]);
      near_mn = fminf(near_mn, s_spk[w][1]);
    }
    p.spike[(size_t)b * p.hq + hq] = (n0 > 0 && n > n0 && far_mx > near_mn) ? 1 : 0;
  }
  __syncthreads();  // s_red is reused below
  for (int s = threadIdx.x; s < n; s += blockDim.x) {
    const float m = s_w[s];
    const float f = m == -INFINITY ? 0.f : exp2_fast(m - mx);  // a split that saw no token: 0
    lsum = fmaf(p.ws_ml[2 * (base + s_part[s]) + 1], f, lsum);
    s_w[s] = f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
  if (lane == 0) s_red[warp][1] = lsum;
  __syncthreads();
  // ---- weighted sum of the accumulators
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
#pragma unroll 4
  for (int s = warp; s < n; s += kCombineWarps) {
    const float f = s_w[s];
    const float* src = p.ws_acc + (base + s_part[s]) * D + lane * PER;
    if constexpr (PER % 4 == 0) {
#pragma unroll
      for (int k = 0; k < PER / 4; ++k) {
        const float4 v = reinterpret_cast<const float4*>(src)[k];
        acc[4 * k] = fmaf(v.x, f, acc[4 * k]);
        acc[4 * k + 1] = fmaf(v.y, f, acc[4 * k + 1]);
        acc[4 * k + 2] = fmaf(v.z, f, acc[4 * k + 2]);
        acc[4 * k + 3] = fmaf(v.w, f, acc[4 * k + 3]);
      }
    } else {  // D = 64: two coordinates per lane
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(v.x, f, acc[0]);
      acc[1] = fmaf(v.y, f, acc[1]);
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) s_acc[warp][lane * PER + k] = acc[k];
  __syncthreads();
  if (warp != 0) return;
  lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) lsum += s_red[w][1];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) a += s_acc[w][lane * PER + k];
    acc[k] = a;
  }
  const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] *= inv;
  // y = s_V * (H y~) / sqrt(D): coordinate index = lane * PER + k
#pragma unroll
  for (int hs = 1; hs < PER; hs <<= 1) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      if ((k & hs) == 0) {
        const float a = acc[k], c = acc[k + hs];
        acc[k] = a + c;
        acc[k + hs] = a - c;
      }
    }
  }
#pragma unroll
  for (int mm = 1; mm < 32; mm <<= 1) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, acc[k], mm);
      acc[k] = (lane & mm) ? (o - acc[k]) : (acc[k] + o);
    }
  }
  constexpr float inv_sqrt_d = inv_sqrt_dim(D);
  const int8_t* sg = p.v_signs + hk * D + lane * PER;
  float* dst = p.out + ((size_t)b * p.hq + hq) * D + lane * PER;
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int k = 0; k < PER / 4; ++k) {
      float4 v;
      v.x = (sg[4 * k] < 0 ? -acc[4 * k] : acc[4 * k]) * inv_sqrt_d;
      v.y = (sg[4 * k + 1] < 0 ? -acc[4 * k + 1] : acc[4 * k + 1]) * inv_sqrt_d;
      v.z = (sg[4 * k + 2] < 0 ? -acc[4 * k + 2] : acc[4 * k + 2]) * inv_sqrt_d;
      v.w = (sg[4 * k + 3] < 0 ? -acc[4 * k + 3] : acc[4 * k + 3]) * inv_sqrt_d;
      reinterpret_cast<float4*>(dst)[k] = v;
    }
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2((sg[0] < 0 ? -acc[0] : acc[0]) * inv_sqrt_d,
                                                  (sg[1] < 0 ? -acc[1] : acc[1]) * inv_sqrt_d);
  }
}

template <int D, int G, class KF, class VF>
cudaError_t launch_tier(const DecParams& p, int ti, cudaStream_t stream) {
  const DecTier& T = p.tier[ti];
  if (T.num_splits == 0) return cudaSuccess;
  dim3 grid(T.num_splits, p.hkv, p.batch);
  decode_tier_kernel<D, G, KF, VF><<<grid, kWarps * 32, 0, stream>>>(p, ti);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int D, int G>
cudaError_t launch_tier_fmt(const DecParams& p, int ti, cudaStream_t stream) {
  const DecTier& T = p.tier[ti];
  const int kf = T.k_fmt, vf = T.v_fmt;
  if (kf == KVQ_FMT_CODEBOOK && vf == KVQ_FMT_CODEBOOK) {
    switch (T.k_bits * 8 + T.v_bits) {
      case 4 * 8 + 4: return launch_tier<D, G, Codebook<4>, Codebook<4>>(p, ti, stream);
      case 4 * 8 + 3: return launch_tier<D, G, Codebook<4>, Codebook<3>>(p, ti, stream);
      case 4 * 8 + 2: return launch_tier<D, G, Codebook<4>, Codebook<2>>(p, ti, stream);
      case 3 * 8 + 4: return launch_tier<D, G, Codebook<3>, Codebook<4>>(p, ti, stream);
      case 3 * 8 + 3: return launch_tier<D, G, Codebook<3>, Codebook<3>>(p, ti, stream);
      case 3 * 8 + 2: return launch_tier<D, G, Codebook<3>, Codebook<2>>(p, ti, stream);
      case 2 * 8 + 4: return launch_tier<D, G, Codebook<2>, Codebook<4>>(p, ti, stream);
      case 2 * 8 + 3: return launch_tier<D, G, Codebook<2>, Codebook<3>>(p, ti, stream);
      case 2 * 8 + 2: return launch_tier<D, G, Codebook<2>, Codebook<2>>(p, ti, stream);
      default: return cudaErrorNotSupported;
    }
  }
  if (kf == KVQ_FMT_FP16 && vf == KVQ_FMT_FP16) return launch_tier<D, G, Fp16, Fp16>(p, ti, stream);
  if (kf == KVQ_FMT_FP8_E4M3 && vf == KVQ_FMT_INT4_G32) return launch_tier<D, G, Fp8, Int4>(p, ti, stream);
  if (kf == KVQ_FMT_FP8_E4M3 && vf == KVQ_FMT_FP16) return launch_tier<D, G, Fp8, Fp16>(p, ti, stream);
  return cudaErrorNotSupported;
}

template <int D>
cudaError_t launch_decode_d(const DecParams& p, int group, cudaStream_t stream) {
  for (int ti = 0; ti < p.num_tiers; ++ti) {
    if (p.tier[ti].kind != TIER_GENERIC) continue;
    cudaError_t e;
    switch (group) {
      case 1: e = launch_tier_fmt<D, 1>(p, ti, stream); break;
      case 2: e = launch_tier_fmt<D, 2>(p, ti, stream); break;
      case 4: e = launch_tier_fmt<D, 4>(p, ti, stream); break;
      case 8: e = launch_tier_fmt<D, 8>(p, ti, stream); break;
      default: e = cudaErrorNotSupported;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool decode_supports(int k_fmt, int k_bits, int v_fmt, int v_bits) {
  if (k_fmt == KVQ_FMT_CODEBOOK && v_fmt == KVQ_FMT_CODEBOOK)
    return k_bits >= 2 && k_bits <= 4 && v_bits >= 2 && v_bits <= 4;
  if (k_fmt == KVQ_FMT_FP16 && v_fmt == KVQ_FMT_FP16) return true;
  if (k_fmt == KVQ_FMT_FP8_E4M3 && (v_fmt == KVQ_FMT_INT4_G32 || v_fmt == KVQ_FMT_FP16)) return true;
  return false;
}

cudaError_t launch_decode(const DecParams& p, int head_dim, int group, cudaStream_t stream) {
  if (head_dim == 64) return launch_decode_d<64>(p, group, stream);
  if (head_dim == 128) return launch_decode_d<128>(p, group, stream);
  if (head_dim == 256) return launch_decode_d<256>(p, group, stream);
  return cudaErrorNotSupported;
}

namespace {

template <int D, int W>
cudaError_t launch_combine_w(const DecParams& p, cudaStream_t stream) {
  // programmatic dependent launch: the grid may be set up while the split-K pass drains
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch * p.hq);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel<D, W>, p);
  if (e == cudaSuccess) note_launch();
  return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int D>
cudaError_t launch_combine_d(const DecParams& p, cudaStream_t stream) {
  // warps per output from the splits one output may have (every tier's); measured on GB300:
  // 171 splits (the append workload) 851.5 -> 836.2 us per call with 16 warps instead of 4,
  // 39 (gqa32k) 332.9 -> 335.0 us with 8
  if (p.total_splits > 128) return launch_combine_w<D, 16>(p, stream);
  if (p.total_splits > 64) return launch_combine_w<D, 8>(p, stream);
  return launch_combine_w<D, 4>(p, stream);
}

}  // namespace

cudaError_t launch_combine(const DecParams& p, int head_dim, cudaStream_t stream) {
  if (p.batch * p.hq == 0) return cudaSuccess;
  if (head_dim == 64) return launch_combine_d<64>(p, stream);
  if (head_dim == 128) return launch_combine_d<128>(p, stream);
  if (head_dim == 256) return launch_combine_d<256>(p, stream);
  return cudaErrorNotSupported;
}

}  // namespace kvq
