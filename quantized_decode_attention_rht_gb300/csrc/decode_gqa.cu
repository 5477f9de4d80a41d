// Fused decode attention for groups of 1, 2, 4 or 8 query heads per kv head, head_dim 128, over
// fp16 tiers (FoveatedKV near tier, or a recent-token window) and fp8-E4M3-key /
// INT4-g32-value tiers (far tier), all of them in one launch ("Making it fast", FoveatedKV
// page: both tiers and the decode buffer in a single dispatch).
//
// Work: items of (tier, sequence, kv head, chunk of pages) with about equal bytes, handed
// to warps from an atomic counter; 12 warps per SM.  Each warp is independent: it owns a
// ring of shared-memory stages filled by a cp.async pipeline (16-byte copies, rows padded
// by 16 bytes so every fragment load below is free of bank conflicts), and writes one
// split-K partial (running max, sum, rotated-domain accumulator) per item.
//
// The query heads of an item (up to G = 4; smaller groups leave zero columns; a group of 8 is
// two items per chunk, heads 0-3 and 4-7, whose second pass reads the chunk's pages from
// L2) form a real
// contraction with every key and value row, done with mma.sync.m16n8k16 (fp16 inputs, fp32
// accumulation):
//   scores  S[16 tokens x 8] = K[16 tokens x 128] . Qt[128 x 8]
//   values  O[16 dims x 8]  += V^T[16 dims x 16 tokens] . Pt[16 tokens x 8]
// The 8 columns are (head, hi/lo): the rotated query q' and the weights p are split into
// an fp16 high part and an fp16 remainder, so the products keep ~22 bits.  fp8 keys become
// fp16 exactly (cvt.rn.f16x2.e4m3x2); INT4 nibbles u are taken straight out of the
// ldmatrix.trans layout and turned into the exact fp16 level u - 8 (nibble | 0x6400 is
// 1024 + u; subtract 1032), and the group scale s goes into the weights, w = p * s, so
//   O_j = sum_t w_tg (u_tj - 8)
// is accumulated directly, with no cancelling correction term.  q' and the weights are
// scaled by powers of two (2^6, 2^8) so their fp16 remainders stay clear of subnormals;
// the scalings are undone exactly in fp32.  Softmax: scores are in base-2 units (q'
// carries log2(e) / D), one exp2 per score, a running max per head; accumulators rescale
// only when the max grows.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int D = 128, G = 4, PS = 16;  // G: query heads one item can carry
constexpr int kWarps = 12;
constexpr int kWarpSmem = 19360;               // per warp: stage ring + block-table slice
constexpr int kMaxPagesPerItem = 128;
constexpr int kBtab = kWarpSmem - 4 * kMaxPagesPerItem;  // page indices of the current item
constexpr int kRing = kBtab;                   // stages; the rotated queries (2 KB) use the
                                               // start of the ring before the stages fill
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQScale = 64.0f;   // q' is stored x 2^6 in the B fragments
constexpr float kWScale = 256.0f;  // weights are stored x 2^8 in the B fragments

// far tier stage: K fp8 16 x 128 B, V INT4 16 x 64 B, scales 16 x 4 fp16 (rows padded)
constexpr int F_KSTR = 144, F_VSTR = 80;
constexpr int F_V = 16 * F_KSTR, F_S = F_V + 16 * F_VSTR, F_STAGE = F_S + 16 * 8;
constexpr int F_STAGES = kRing / F_STAGE;
// near tier stage: K and V fp16 16 x 256 B (rows padded)
constexpr int N_KSTR = 272, N_VSTR = 272;
constexpr int N_V = 16 * N_KSTR, N_STAGE = N_V + 16 * N_VSTR;
constexpr int N_STAGES = kRing / N_STAGE;
static_assert(F_STAGES >= 2 && N_STAGES >= 2, "ring too small");
static_assert(G * D * 4 <= kRing, "query buffer must fit in the ring");

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four E4M3 bytes -> two fp16 pairs (bytes 0,1 -> lo; bytes 2,3 -> hi), exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// fp16 pair holding either the rounded values (hl = 0) or the rounding remainders (hl = 1)
__device__ __forceinline__ uint32_t split_pair(float x, float y, float hl) {
  const uint32_t h = pack_f16x2(x, y);
  const __half2 hh = *reinterpret_cast<const __half2*>(&h);
  const float rx = fmaf(-hl, __low2float(hh), x);
  const float ry = fmaf(-hl, __high2float(hh), y);
  return pack_f16x2(rx, ry);
}

// 2^x, x <= 0 or -inf (scores in base-2 units relative to the running maximum): the
// hardware approximation (relative error below 2^-22), results below 2^-126 flushed to 0.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Lowest score of head c over the page's 16 tokens (lanes g = 0..7 of the same c).
__device__ __forceinline__ float page_min(float a, float b) {
  float v = fminf(a, b);
  v = fminf(v, __shfl_xor_sync(kFull, v, 4));
  v = fminf(v, __shfl_xor_sync(kFull, v, 8));
  return fminf(v, __shfl_xor_sync(kFull, v, 16));
}

// ---------------------------------------------------------------- parameters
struct GqaTier {
  const uint8_t* k_rows;
  const uint8_t* v_rows;
  const __half* v_aux;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int num_pages;  // pages in the pool: block-table entries at or above are skipped
  int far;    // 1: fp8 K + INT4-g32 V; 0: fp16 K + fp16 V
  int first;  // tier 0 of the call (the near tier of spike detection)
  int max_pages, chunk, nchunks, split_begin, item_begin;
};

struct GqaParams {
  GqaTier tier[KVQ_MAX_TIERS];
  int num_tiers;
  const __half* q;
  const int8_t* k_signs;
  float* ws_acc;
  float* ws_ml;
  float* ws_min;  // lowest score per tier-0 split, when spike flags are asked for
  int* counter;
  int* err;       // the call's error word (KVQ_DEVERR_* bits)
  int hq, hkv, total_splits, total_items;
  int group;        // query heads per kv head (1, 2, 4 or 8)
  int halves;       // items per chunk: 2 for a group of 8 (heads 0-3, 4-7), else 1
  int igroup;       // query heads an item carries: min(group, 4); heads igroup.. are idle
  int trigger;      // a codebook split-K launch follows (as a programmatic dependent)
  int gate, spike;  // score-gated value loading; track tier 0's lowest scores
};

// ---------------------------------------------------------------- per-warp pieces

// q' = H (s_K * q) * log2(e) / D for heads h0 .. h0 + 3 of kv head hk, into qbuf[4][128] (fp32).
// Lane l holds head l/8, coordinates (l%8)*16 .. +16: four butterfly stages in registers,
// three across the 8 lanes of the head.
__device__ __forceinline__ void rotate_query(const GqaParams& p, int b, int hk, int h0, float* qbuf, int lane) {
  const int hh = lane >> 3, d0 = (lane & 7) * 16;
  const bool live = hh < p.igroup;  // idle heads get a zero query (zero B columns)
  const uint4* qs =
      reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.hq + hk * p.group + h0 + (live ? hh : 0)) * D + d0);
  uint4 q0 = __ldg(qs), q1 = __ldg(qs + 1);
  if (!live) q0 = q1 = make_uint4(0u, 0u, 0u, 0u);
  const uint4 sg = __ldg(reinterpret_cast<const uint4*>(p.k_signs + hk * D + d0));
  const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const int8_t* sb = reinterpret_cast<const int8_t*>(&sg);
  float y[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float v = __half2float(__ushort_as_half((uint16_t)(qw[e >> 1] >> (16 * (e & 1)))));
    y[e] = sb[e] < 0 ? -v : v;
  }
#pragma unroll
  for (int hs = 1; hs < 16; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if ((e & hs) == 0) {
        const float a = y[e], c = y[e + hs];
        y[e] = a + c;
        y[e + hs] = a - c;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float o = __shfl_xor_sync(kFull, y[e], m);
      y[e] = (lane & m) ? (o - y[e]) : (y[e] + o);
    }
  }
  constexpr float scale = kLog2e / (float)D * kQScale;
  float4* dst = reinterpret_cast<float4*>(qbuf + hh * D + d0);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    dst[k] = make_float4(y[4 * k] * scale, y[4 * k + 1] * scale, y[4 * k + 2] * scale, y[4 * k + 3] * scale);
}

// ------------------------------------------------------------ far tier (fp8 K, INT4-g32 V)
struct Far {
  static constexpr int STAGE = F_STAGE, S = F_STAGES;

  // B fragments of q' for k-step kk: lane (g, c) holds column g = (head g/2, part g%2) at the
  // coordinates 32c + 4kk + {0,1} (b0b1) and {2,3} (b2b3); the key fragments below use the
  // same coordinate order.
  __device__ static void qfrag(const float* qbuf, uint32_t (&qf)[8][2], int g, int c) {
    const float hl = (float)(g & 1);
    const uint32_t base = smem_addr(qbuf + (g >> 1) * D + 32 * c);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint4 v = lds128(base + 16 * kk);
      qf[kk][0] = split_pair(__uint_as_float(v.x), __uint_as_float(v.y), hl);
      qf[kk][1] = split_pair(__uint_as_float(v.z), __uint_as_float(v.w), hl);
    }
  }

  // Per-lane copy plan of one page: chunk i of the K block (128 x 16 B), V block (64 x 16 B)
  // and scale block (8 x 16 B) goes to its padded row in the stage.
  struct Plan {
    uint32_t kd[4], vd[2], sd;
    uint32_t ks[4], vs[2], ss;
  };
  __device__ static void plan(Plan& pl, int lane) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = lane + 32 * j;
      pl.kd[j] = (i >> 3) * F_KSTR + (i & 7) * 16;
      pl.ks[j] = 16 * i;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = lane + 32 * j;
      pl.vd[j] = F_V + (i >> 2) * F_VSTR + (i & 3) * 16;
      pl.vs[j] = 16 * i;
    }
    pl.sd = F_S + 16 * (lane & 7);
    pl.ss = 16 * (lane & 7);
  }
  __device__ static void issue(const GqaTier& T, const Plan& pl, int phys, int hk, int hkv, uint32_t st, int lane) {
    const size_t blk = (size_t)phys * hkv + hk;
    const uint8_t* kb = T.k_rows + blk * (PS * 128);
    const uint8_t* vb = T.v_rows + blk * (PS * 64);
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(T.v_aux + blk * (PS * 4));
#pragma unroll
    for (int j = 0; j < 4; ++j) cp_async16(st + pl.kd[j], kb + pl.ks[j]);
#pragma unroll
    for (int j = 0; j < 2; ++j) cp_async16(st + pl.vd[j], vb + pl.vs[j]);
    if (lane < 8) cp_async16(st + pl.sd, sb + pl.ss);
  }

  struct State {
    float acc[4][2][4];  // [group][m][c0..c3]
    float m, l, mn;
  };

  __device__ static void init(State& s) {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) s.acc[a][m][k] = 0.f;
    }
    s.m = -INFINITY;
    s.l = 0.f;
    s.mn = INFINITY;
  }

  __device__ static void rescale(State& s, float f) {
    s.l *= f;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) s.acc[a][m][k] *= f;
    }
  }

  __device__ static void page(const uint8_t* st, int nvalid, const uint32_t (&qf)[8][2], State& s, int lane,
                              bool track, bool gate, bool live) {
    const int g = lane >> 2, c = lane & 3;
    const uint32_t s0 = smem_addr(st);
    // ---- scores
    const uint4 r0a = lds128(s0 + g * F_KSTR + 32 * c), r0b = lds128(s0 + g * F_KSTR + 32 * c + 16);
    const uint4 r1a = lds128(s0 + (g + 8) * F_KSTR + 32 * c), r1b = lds128(s0 + (g + 8) * F_KSTR + 32 * c + 16);
    const uint32_t w0[8] = {r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
    const uint32_t w1[8] = {r1a.x, r1a.y, r1a.z, r1a.w, r1b.x, r1b.y, r1b.z, r1b.w};
    float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      e4m3x4_to_f16x4(w0[kk], a[0], a[2]);
      e4m3x4_to_f16x4(w1[kk], a[1], a[3]);
      mma16816(sa[kk & 1], a, qf[kk][0], qf[kk][1]);
    }
    constexpr float unq = 1.0f / kQScale;
    float x0 = ((sa[0][0] + sa[0][1]) + (sa[1][0] + sa[1][1])) * unq;  // token g, head c
    float x1 = ((sa[0][2] + sa[0][3]) + (sa[1][2] + sa[1][3])) * unq;  // token g + 8
    // ---- online softmax for head c over the 16 tokens
    const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
    x0 = v0 ? x0 : -INFINITY;
    x1 = v1 ? x1 : -INFINITY;
    float mt = fmaxf(x0, x1);  // the page maximum: needed only above the running one (or for the gate)
    if (gate || __any_sync(kFull, mt > s.m)) {
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
    }
    if (mt > s.m) {
      rescale(s, exp2_fast(s.m - mt));  // first tile: exp2(-inf) = 0
      s.m = mt;
    }
    const float p0 = v0 ? exp2_fast(x0 - s.m) : 0.f;
    const float p1 = v1 ? exp2_fast(x1 - s.m) : 0.f;
    s.l += p0 + p1;
    if (track) s.mn = fminf(s.mn, page_min(v0 ? x0 : INFINITY, v1 ? x1 : INFINITY));
    // score gate: every token of the page, for every live head, far below the running max
    if (gate && __all_sync(kFull, !live || mt - s.m < -kGateLog2)) return;
    // ---- weights w = p * scale (x 2^8) per group for this lane's tokens (g, g+8), head c
    const uint2 sc0 = lds64(s0 + F_S + 8 * g), sc1 = lds64(s0 + F_S + 8 * (g + 8));
    const __half2* h0 = reinterpret_cast<const __half2*>(&sc0);
    const __half2* h1 = reinterpret_cast<const __half2*>(&sc1);
    const float q0 = p0 * kWScale, q1 = p1 * kWScale;
    float w0g[4], w1g[4];
    w0g[0] = q0 * __low2float(h0[0]);
    w0g[1] = q0 * __high2float(h0[0]);
    w0g[2] = q0 * __low2float(h0[1]);
    w0g[3] = q0 * __high2float(h0[1]);
    w1g[0] = q1 * __low2float(h1[0]);
    w1g[1] = q1 * __high2float(h1[0]);
    w1g[2] = q1 * __low2float(h1[1]);
    w1g[3] = q1 * __high2float(h1[1]);
    // (hi, lo) of the pair (token g, token g + 8) per group, then gather the B fragments:
    // lane (g', c') needs head g'/2, part g'%2 at tokens 2c', 2c'+1 (b0b1) and +8 (b2b3),
    // held by lanes (2c', g'/2) and (2c'+1, g'/2).
    const int srcA = 4 * (2 * c) + (g >> 1), srcB = srcA + 4;
    const bool lo_part = g & 1;
    uint32_t bf[4][2];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const uint32_t hi = pack_f16x2(w0g[a], w1g[a]);
      const __half2 hh = *reinterpret_cast<const __half2*>(&hi);
      const uint32_t lo = pack_f16x2(w0g[a] - __low2float(hh), w1g[a] - __high2float(hh));
      const uint32_t ah = __shfl_sync(kFull, hi, srcA), al = __shfl_sync(kFull, lo, srcA);
      const uint32_t bh = __shfl_sync(kFull, hi, srcB), bl = __shfl_sync(kFull, lo, srcB);
      const uint32_t A = lo_part ? al : ah, B = lo_part ? bl : bh;
      bf[a][0] = __byte_perm(A, B, 0x5410);  // (token 2c, token 2c+1)
      bf[a][1] = __byte_perm(A, B, 0x7632);  // (token 2c+8, token 2c+9)
    }
    // ---- values: ldmatrix.trans gives lane (g, c), per group a and token half th, the
    // bytes 2g, 2g+1 of that group's 16-byte chunk for tokens 2c, 2c+1 (+8 th)
    uint32_t R[4][2];
    {
      const int t = lane & 7, mi = lane >> 3;  // address of row t of matrix mi
      uint32_t r[4];
      // matrices: (group 0, th 0), (0, 1), (1, 0), (1, 1)
      ldsm_x4_t(r, s0 + F_V + ((mi & 1) * 8 + t) * F_VSTR + (mi >> 1) * 16);
      R[0][0] = r[0]; R[0][1] = r[1]; R[1][0] = r[2]; R[1][1] = r[3];
      ldsm_x4_t(r, s0 + F_V + ((mi & 1) * 8 + t) * F_VSTR + (2 + (mi >> 1)) * 16);
      R[2][0] = r[0]; R[2][1] = r[1]; R[3][0] = r[2]; R[3][1] = r[3];
    }
    // nibble -> exact fp16 level: (nibble | 0x6400) is 1024 + u (low nibble) or 1024 + 16u
    // (high nibble); subtracting 1032 or 1152 leaves u - 8 or 16 (u - 8)
    const uint32_t magic = 0x64006400u;
    const __half2 off_lo = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    const __half2 off_hi = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    auto lvl = [&](uint32_t bits, __half2 off) {
      __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&bits), off);
      return *reinterpret_cast<uint32_t*>(&h);
    };
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const uint32_t x0s = R[a][0] >> 8, x1s = R[a][1] >> 8;
      uint32_t am[4];
      // m-tile (group a, m = 0): rows g -> coordinate 4g (low nibble of byte 2g),
      // rows g+8 -> 4g+1 (high nibble)
      am[0] = lvl((R[a][0] & 0x000F000Fu) | magic, off_lo);
      am[1] = lvl((R[a][0] & 0x00F000F0u) | magic, off_hi);
      am[2] = lvl((R[a][1] & 0x000F000Fu) | magic, off_lo);
      am[3] = lvl((R[a][1] & 0x00F000F0u) | magic, off_hi);
      mma16816(s.acc[a][0], am, bf[a][0], bf[a][1]);
      // m = 1: coordinates 4g+2, 4g+3 (byte 2g+1)
      am[0] = lvl((x0s & 0x000F000Fu) | magic, off_lo);
      am[1] = lvl((x0s & 0x00F000F0u) | magic, off_hi);
      am[2] = lvl((x1s & 0x000F000Fu) | magic, off_lo);
      am[3] = lvl((x1s & 0x00F000F0u) | magic, off_hi);
      mma16816(s.acc[a][1], am, bf[a][0], bf[a][1]);
    }
  }

  // Partial for head c: acc[32a + 4g + k] = sum_t p_t s_ta (u - 8), relative to the max.
  __device__ static void finish(State& s, float* acc_out, float* ml_out, float* mn_out, int lane, bool live) {
    const int g = lane >> 2;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) s.l += __shfl_xor_sync(kFull, s.l, o);
    if (!live) return;  // an idle head of a group smaller than 4
    constexpr float even = 1.0f / kWScale, odd = 1.0f / (kWScale * 16.0f);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float4 v;
      v.x = (s.acc[a][0][0] + s.acc[a][0][1]) * even;
      v.y = (s.acc[a][0][2] + s.acc[a][0][3]) * odd;
      v.z = (s.acc[a][1][0] + s.acc[a][1][1]) * even;
      v.w = (s.acc[a][1][2] + s.acc[a][1][3]) * odd;
      reinterpret_cast<float4*>(acc_out)[8 * a + g] = v;
    }
    if (g == 0) {
      ml_out[0] = s.m;
      ml_out[1] = s.l;
      if (mn_out) *mn_out = s.mn;
    }
  }
};

// ------------------------------------------------------------ near tier (fp16 K, fp16 V)
struct Near {
  static constexpr int STAGE = N_STAGE, S = N_STAGES;

  // B fragments in the natural coordinate order: b0b1 = 16kk + 2c, +1; b2b3 = +8, +9.
  __device__ static void qfrag(const float* qbuf, uint32_t (&qf)[8][2], int g, int c) {
    const float hl = (float)(g & 1);
    const uint32_t base = smem_addr(qbuf + (g >> 1) * D + 2 * c);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint2 a = lds64(base + 64 * kk), b = lds64(base + 64 * kk + 32);
      qf[kk][0] = split_pair(__uint_as_float(a.x), __uint_as_float(a.y), hl);
      qf[kk][1] = split_pair(__uint_as_float(b.x), __uint_as_float(b.y), hl);
    }
  }

  struct Plan {
    uint32_t d[8], s[8];
  };
  __device__ static void plan(Plan& pl, int lane) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = lane + 32 * j;  // 256 chunks of 16 B per side
      pl.d[j] = (i >> 4) * N_KSTR + (i & 15) * 16;
      pl.s[j] = 16 * i;
    }
  }
  __device__ static void issue(const GqaTier& T, const Plan& pl, int phys, int hk, int hkv, uint32_t st, int lane) {
    const size_t blk = (size_t)phys * hkv + hk;
    const uint8_t* kb = T.k_rows + blk * (PS * 256);
    const uint8_t* vb = T.v_rows + blk * (PS * 256);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cp_async16(st + pl.d[j], kb + pl.s[j]);
      cp_async16(st + N_V + pl.d[j], vb + pl.s[j]);
    }
  }

  struct State {
    float acc[8][4];  // [m-tile][c0..c3]
    float m, l, mn;
  };

  __device__ static void init(State& s) {
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) s.acc[a][k] = 0.f;
    s.m = -INFINITY;
    s.l = 0.f;
    s.mn = INFINITY;
  }

  __device__ static void page(const uint8_t* st, int nvalid, const uint32_t (&qf)[8][2], State& s, int lane,
                              bool track, bool gate, bool live) {
    const int g = lane >> 2, c = lane & 3;
    const uint32_t s0 = smem_addr(st);
    const int t = lane & 7, mi = lane >> 3;
    // ---- scores: ldmatrix gives the A fragments of K[16 tokens x 16 coordinates]
    float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t kaddr = s0 + ((mi & 1) * 8 + t) * N_KSTR + (mi >> 1) * 16;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, kaddr + 32 * kk);
      mma16816(sa[kk & 1], a, qf[kk][0], qf[kk][1]);
    }
    constexpr float unq = 1.0f / kQScale;
    float x0 = ((sa[0][0] + sa[0][1]) + (sa[1][0] + sa[1][1])) * unq;
    float x1 = ((sa[0][2] + sa[0][3]) + (sa[1][2] + sa[1][3])) * unq;
    const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
    x0 = v0 ? x0 : -INFINITY;
    x1 = v1 ? x1 : -INFINITY;
    float mt = fmaxf(x0, x1);  // the page maximum: needed only above the running one (or for the gate)
    if (gate || __any_sync(kFull, mt > s.m)) {
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
    }
    if (mt > s.m) {
      const float f = exp2_fast(s.m - mt);
      s.l *= f;
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int k = 0; k < 4; ++k) s.acc[a][k] *= f;
      s.m = mt;
    }
    const float p0 = v0 ? exp2_fast(x0 - s.m) : 0.f;
    const float p1 = v1 ? exp2_fast(x1 - s.m) : 0.f;
    s.l += p0 + p1;
    if (track) s.mn = fminf(s.mn, page_min(v0 ? x0 : INFINITY, v1 ? x1 : INFINITY));
    if (gate && __all_sync(kFull, !live || mt - s.m < -kGateLog2)) return;  // score gate (see Far)
    const int srcA = 4 * (2 * c) + (g >> 1), srcB = srcA + 4;
    const float q0 = p0 * kWScale, q1 = p1 * kWScale;
    const uint32_t hi = pack_f16x2(q0, q1);
    const __half2 hh = *reinterpret_cast<const __half2*>(&hi);
    const uint32_t lo = pack_f16x2(q0 - __low2float(hh), q1 - __high2float(hh));
    const bool lo_part = g & 1;
    const uint32_t ah = __shfl_sync(kFull, hi, srcA), al = __shfl_sync(kFull, lo, srcA);
    const uint32_t bh = __shfl_sync(kFull, hi, srcB), bl = __shfl_sync(kFull, lo, srcB);
    const uint32_t A = lo_part ? al : ah, B = lo_part ? bl : bh;
    const uint32_t b0 = __byte_perm(A, B, 0x5410), b1 = __byte_perm(A, B, 0x7632);
    // ---- values: ldmatrix.trans gives V^T[16 coordinates x 16 tokens] fragments
    const uint32_t vaddr = s0 + N_V + ((mi >> 1) * 8 + t) * N_VSTR + (mi & 1) * 16;
#pragma unroll
    for (int mt2 = 0; mt2 < 8; ++mt2) {
      uint32_t a[4];
      ldsm_x4_t(a, vaddr + 32 * mt2);
      mma16816(s.acc[mt2], a, b0, b1);
    }
  }

  __device__ static void finish(State& s, float* acc_out, float* ml_out, float* mn_out, int lane, bool live) {
    const int g = lane >> 2;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) s.l += __shfl_xor_sync(kFull, s.l, o);
    if (!live) return;  // an idle head of a group smaller than 4
    constexpr float unw = 1.0f / kWScale;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      acc_out[16 * a + g] = (s.acc[a][0] + s.acc[a][1]) * unw;
      acc_out[16 * a + g + 8] = (s.acc[a][2] + s.acc[a][3]) * unw;
    }
    if (g == 0) {
      ml_out[0] = s.m;
      ml_out[1] = s.l;
      if (mn_out) *mn_out = s.mn;
    }
  }
};

// The partial of an item that contributes nothing (running max -inf, sum 0): what an item
// with a block-table entry outside the pool leaves, so the combine pass reads no stale data.
__device__ __noinline__ void empty_partial(const GqaParams& p, const GqaTier& T, int b, int hk, int h0, int chunk,
                                           int lane, bool track) {
  for (int h = h0; h < h0 + p.igroup; ++h) {
    const size_t part = ((size_t)b * p.hq + hk * p.group + h) * p.total_splits + T.split_begin + chunk;
    for (int j = lane; j < D; j += 32) p.ws_acc[part * D + j] = 0.f;
    if (lane == 0) {
      p.ws_ml[2 * part] = -INFINITY;
      p.ws_ml[2 * part + 1] = 0.f;
      if (track) p.ws_min[part] = INFINITY;
    }
  }
}

// One work item: pages [t0, t1) of sequence b, kv head hk in tier T.
template <class TT>
__device__ __forceinline__ void run_item(const GqaParams& p, const GqaTier& T, int b, int hk, int h0, int chunk,
                                         int t0, int t1, uint8_t* wsm, int lane, bool track) {
  const int g = lane >> 2, c = lane & 3;
  float* qbuf = reinterpret_cast<float*>(wsm);  // the ring is idle between items
  int* btab = reinterpret_cast<int*>(wsm + kBtab);
  const int pg0 = t0 / PS, npg = (t1 + PS - 1) / PS - pg0;
  const int32_t* bt = T.block_table + (size_t)b * T.max_pages + pg0;
  int bits = 0;
  for (int i = lane; i < npg; i += 32) {
    const int e = __ldg(bt + i);
    page_in_pool(e, T.num_pages, &bits);
    btab[i] = e;
  }
  rotate_query(p, b, hk, h0, qbuf, lane);  // its loads overlap the block-table loads above
  __syncwarp();
  uint32_t qf[8][2];
  TT::qfrag(qbuf, qf, g, c);
  typename TT::Plan pl;
  TT::plan(pl, lane);
  __syncwarp();  // the ring is reused for stages below
  if (__any_sync(kFull, bits != 0)) {  // a page outside the pool: the item reads nothing
    if (lane == 0) atomicOr(p.err, KVQ_DEVERR_PAGE_INDEX);
    empty_partial(p, T, b, hk, h0, chunk, lane, track);
    return;
  }
  const uint32_t ring = smem_addr(wsm);
#pragma unroll 1
  for (int s = 0; s < TT::S; ++s) {
    if (s < npg) TT::issue(T, pl, btab[s], hk, p.hkv, ring + s * TT::STAGE, lane);
    cp_commit();
  }
  typename TT::State st;
  TT::init(st);
#pragma unroll 1
  for (int i = 0; i < npg; ++i) {
    cp_wait<TT::S - 1>();
    __syncwarp();
    const int slot = i % TT::S;
    const int nvalid = min(PS, t1 - (pg0 + i) * PS);
    TT::page(wsm + slot * TT::STAGE, nvalid, qf, st, lane, track, p.gate != 0, c < p.igroup);
    __syncwarp();
    if (i + TT::S < npg) TT::issue(T, pl, btab[i + TT::S], hk, p.hkv, ring + slot * TT::STAGE, lane);
    cp_commit();
  }
  cp_wait<0>();
  const bool live = c < p.igroup;
  const size_t part = live ? ((size_t)b * p.hq + hk * p.group + h0 + c) * p.total_splits + T.split_begin + chunk : 0;
  TT::finish(st, p.ws_acc + part * D, p.ws_ml + 2 * part, track ? p.ws_min + part : nullptr, lane, live);
  __syncwarp();
}

__global__ void __launch_bounds__(kWarps * 32, 1) decode_gqa_kernel(const __grid_constant__ GqaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* wsm = smem + warp * kWarpSmem;
  // a codebook split-K grid that follows may start on SMs this grid leaves idle
  if (p.trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int item = 0;
  if (lane == 0) item = atomicAdd(p.counter, 1);
  item = __shfl_sync(kFull, item, 0);
  while (item < p.total_items) {
    int next = 0;
    if (lane == 0) next = atomicAdd(p.counter, 1);
    int ti = 0;
    while (ti + 1 < p.num_tiers && item >= p.tier[ti + 1].item_begin) ++ti;
    const GqaTier& T = p.tier[ti];
    int rem = item - T.item_begin;
    const int chunk = rem % T.nchunks;
    rem /= T.nchunks;
    // a group of 8: every chunk of heads 0-3, then every chunk of heads 4-7, so the second
    // pass over a chunk comes a few items later and finds its pages in L2
    const int half = p.halves == 2 ? (rem & 1) : 0;
    rem = p.halves == 2 ? rem >> 1 : rem;
    const int hk = rem % p.hkv, b = rem / p.hkv;
    int bits = 0;  // a length out of range is cut into it here and reported by the combine pass
    const int len = checked_len(T.seq_lens[b], T.max_pages, PS, &bits);
    const int t0 = chunk * T.chunk;
    if (t0 < len) {
      const int t1 = min(len, t0 + T.chunk);
      const bool track = p.spike && T.first;
      if (T.far) run_item<Far>(p, T, b, hk, 4 * half, chunk, t0, t1, wsm, lane, track);
      else run_item<Near>(p, T, b, hk, 4 * half, chunk, t0, t1, wsm, lane, track);
    }
    item = __shfl_sync(kFull, next, 0);
  }
}

}  // namespace

bool gqa_fast_supported(int head_dim, int group, int k_fmt, int v_fmt) {
  if (head_dim != D || (group != 1 && group != 2 && group != 4 && group != 8)) return false;
  return (k_fmt == KVQ_FMT_FP16 && v_fmt == KVQ_FMT_FP16) || (k_fmt == KVQ_FMT_FP8_E4M3 && v_fmt == KVQ_FMT_INT4_G32);
}

int gqa_max_chunk_tokens() { return kMaxPagesPerItem * PS; }

cudaError_t launch_decode_gqa(const DecParams& dp, int* counter, cudaStream_t stream, bool trigger) {
  constexpr int smem = kWarps * kWarpSmem;
  static std::atomic<bool> configured[64];  // shared-memory limit raised on this device (threads may race: a
                                           // second raise is harmless)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(decode_gqa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  GqaParams p;
  memset(&p, 0, sizeof(p));
  int items = 0, n = 0;
  for (int i = 0; i < dp.num_tiers; ++i) {
    const DecTier& t = dp.tier[i];
    if (t.kind != TIER_GQA) continue;
    GqaTier& g = p.tier[n++];
    g.first = i == 0;
    g.k_rows = t.k_rows;
    g.v_rows = t.v_rows;
    g.v_aux = t.v_aux;
    g.block_table = t.block_table;
    g.seq_lens = t.seq_lens;
    g.num_pages = t.num_pages;
    g.far = t.k_fmt == KVQ_FMT_FP8_E4M3;
    g.max_pages = t.max_pages;
    g.chunk = t.chunk;
    g.nchunks = t.num_splits;
    g.split_begin = t.split_begin;
    g.item_begin = items;
    items += dp.batch * dp.hkv * t.num_splits * (dp.hq / dp.hkv == 8 ? 2 : 1);
  }
  p.num_tiers = n;
  p.group = dp.hq / dp.hkv;
  p.halves = p.group == 8 ? 2 : 1;
  p.igroup = p.group < 4 ? p.group : 4;
  p.trigger = trigger ? 1 : 0;
  p.q = dp.q;
  p.k_signs = dp.k_signs;
  p.ws_acc = dp.ws_acc;
  p.ws_ml = dp.ws_ml;
  p.ws_min = dp.ws_min;
  p.gate = dp.gate;
  p.spike = dp.spike != nullptr;
  p.counter = counter;
  p.err = dp.err;
  p.hq = dp.hq;
  p.hkv = dp.hkv;
  p.total_splits = dp.total_splits;
  p.total_items = items;
  if (items == 0) return cudaSuccess;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int ctas = std::max(1, std::min(sms, (items + kWarps - 1) / kWarps));
  decode_gqa_kernel<<<ctas, kWarps * 32, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace kvq
