// Fused decode attention over codebook tiers (b-bit Lloyd-Max or uniform codes + fp16 norm
// for keys and values), head_dim 128 or 256, 1, 2 or 4 query heads per kv head.
//
// The scores of a key row are q'.k~ with k~_j = (norm / sqrt(D)) C[idx_j] (TurboQuant page,
// "dequantize" step; AdapTQ page, "Engineering the Hot Path": the rotated query meets the
// stored codes directly, through a table of centroids).  Values accumulate in the rotated
// domain the same way and the combine pass undoes the rotation once.
//
// Layout of the work: items of (sequence, kv head, chunk of pages), handed to warps from an
// atomic counter; every warp is independent and writes one split-K partial per item.  A
// warp takes one 16-token page per step.  Its lanes load the packed code bits they need
// straight from HBM into registers (16- and 8-byte coalesced loads, one page ahead) and
// turn them into tensor-core fragments through a centroid table in shared memory:
//
//   scores  S[16 tokens x 8]  = K~[16 tokens x D] . Q[D x 8]        (D/16 mma k-steps)
//   values  O[16 dims x 8]   += V~^T[16 dims x 16 tokens] . W[16 tokens x 8]
//
// with mma.sync.m16n8k16 (fp16 inputs, fp32 accumulation).  The 8 columns are (head,
// hi/lo) pairs; columns of heads >= G are zero.  Centroids are fp32, so every table entry
// holds the fp16 rounding of 256*C and the fp16 rounding of the remainder: each code pair
// is looked up once and feeds two mma (hi and lo), the query and the weights are split the
// same way, and the products keep ~22 bits.
//
// Table: one entry per value of a pair field (2b bits = two codes, first code in the low
// bits), 8 bytes (hi pair, lo pair), replicated for each of the 32 lanes so that a warp's
// 32 lookups hit 32 different bank pairs.  The table sits at a shared address aligned to
// its own size, so the lookup address of lane l is (field << 8) | (l << 3) | base: one
// byte permute (byte fields) or one shift and one logic op from the packed word.
//
// Pair-slot permutations: the dot product does not care in which order its terms are
// summed, so lane (g, c) of the key mma takes the pair slots [c*D/8, (c+1)*D/8) of rows g
// and g+8 (one contiguous run of bits per row) and the query fragments follow the same
// order; the value mma maps its A rows g and g+8 of m-tile mt to the two coordinates of
// pair slot g*D/16 + mt, so a lookup gives both rows and the lane's output coordinates
// come out contiguous.  The value fragments pair two tokens per register, the table pairs
// two coordinates of one token: two byte permutes per register pair swap them.
#include <algorithm>
#include <cstring>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int PS = 16;
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kCScale = 256.0f;  // table entries hold 2^8 C
constexpr float kQScale = 64.0f;   // query fragments hold 2^6 q'
constexpr float kWScale = 8.0f;    // weight fragments hold 2^3 p norm / sqrt(D); with p <= 1
                                   // every fp16 norm stays below the fp16 maximum

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Table lookup.  Not volatile: once the tables are built it is a plain function of its
// address, which leaves the compiler free to overlap lookups with tensor-core work.  Every
// lookup address derives from a value pin()ned after the barrier that ends the build.
__device__ __forceinline__ uint2 lut64(uint32_t a) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t pin(uint32_t x) {
  asm volatile("" : "+r"(x));
  return x;
}
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
typedef unsigned long long u64;
__device__ __forceinline__ u64 lut64x(uint32_t a) {  // as lut64, one 64-bit register
  u64 v;
  asm("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ u64 pk2(float a, float b) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(u64 r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
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

// ---------------------------------------------------------------- parameters
struct CbTier {
  const uint8_t* k_rows;
  const uint8_t* v_rows;
  const __half* k_norm;
  const __half* v_norm;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int max_pages, chunk, nchunks, split_begin;
};

struct CbParams {
  CbTier t;
  const __half* q;
  const int8_t* k_signs;
  const float* k_cent;
  const float* v_cent;
  float* ws_acc;
  float* ws_ml;
  int* counter;
  int hq, hkv, total_splits, total_items, smem_bytes;
};

template <int D, int G, int KB, int VB>
struct Cfg {
  static constexpr int KS = D / 16;             // key mma k-steps; also value m-tiles
  static constexpr int PPT = D / 8;             // key pair slots per lane (index c)
  static constexpr int QPT = D / 16;            // value pair slots per lane (index g)
  static constexpr int KROW = D * KB / 8;       // bytes of a key row
  static constexpr int VROW = D * VB / 8;
  static constexpr int KBYTES = PPT * KB / 4;   // key bits of one lane, in bytes
  static constexpr int VBYTES = QPT * VB / 4;
  static constexpr int KW = KBYTES / 4;         // always whole words
  static constexpr bool VODD = (VBYTES % 4) != 0;  // 3-bit values at D = 128: 6 bytes
  static constexpr int VW = VODD ? 2 : VBYTES / 4;
  static constexpr int KLUT = (1 << (2 * KB)) * 256;  // table bytes (also its alignment)
  static constexpr int VLUT = (1 << (2 * VB)) * 256;
  static constexpr int WARPS = D == 128 ? 12 : 8;
  static constexpr int QBUF = G * D * 4;        // per-warp rotated queries (fp32)
};

// ---------------------------------------------------------------- bit fields

// Lookup address of the pair field that starts at bit o of the lane's words.  Every call
// sits in a fully unrolled loop, so o is a constant and the branches fold away.
template <int BITS2, int NW>
__device__ __forceinline__ uint32_t field_addr(const uint32_t (&w)[NW], int o, uint32_t lanebase) {
  const int i = o / 32, r = o % 32;
  constexpr uint32_t mask = ((1u << BITS2) - 1u) << 8;
  if (BITS2 == 8) {
    // byte r/8 of word i into byte 1; bytes 0, 2, 3 from lanebase (its byte 1 is zero)
    return __byte_perm(w[i], lanebase, 0x7604 | ((r / 8) << 4));
  } else if (r + BITS2 <= 32) {
    const uint32_t x = r >= 8 ? (w[i] >> (r - 8)) : (w[i] << (8 - r));
    return (x & mask) | lanebase;
  } else {
    const uint32_t x = __funnelshift_r(w[i], w[i + 1 < NW ? i + 1 : i], r - 8);
    return (x & mask) | lanebase;
  }
}

// ---------------------------------------------------------------- per-page data of a lane
template <class C>
struct Page {
  uint32_t k[2][C::KW];  // key bits of rows g and g+8
  uint32_t v[4][C::VW];  // value bits of tokens 2c, 2c+1, 2c+8, 2c+9
  uint32_t nk, nv;       // fp16 norms of tokens g (low half) and g+8 (high half)
};

template <int NBYTES, int NW>
__device__ __forceinline__ void load_words(const uint8_t* src, uint32_t (&w)[NW]) {
  if constexpr (NBYTES == 32) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if constexpr (NBYTES == 24) {
    const uint2* s = reinterpret_cast<const uint2*>(src);
    const uint2 a = __ldg(s), b = __ldg(s + 1), c = __ldg(s + 2);
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y; w[4] = c.x; w[5] = c.y;
  } else if constexpr (NBYTES == 16) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else if constexpr (NBYTES == 12) {
    const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
    w[0] = __ldg(s); w[1] = __ldg(s + 1); w[2] = __ldg(s + 2);
  } else if constexpr (NBYTES == 8) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(src));
    w[0] = a.x; w[1] = a.y;
  } else {
    static_assert(NBYTES == 4, "unsupported run length");
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
  }
}

template <class C>
__device__ __forceinline__ void load_page(const CbTier& T, int phys, int hk, int hkv, int g, int c, Page<C>& pg) {
  const size_t blk = (size_t)phys * hkv + hk;  // [page][kv head] block of 16 rows
  const uint8_t* kr = T.k_rows + blk * (PS * C::KROW) + c * C::KBYTES;
  load_words<C::KBYTES>(kr + g * C::KROW, pg.k[0]);
  load_words<C::KBYTES>(kr + (g + 8) * C::KROW, pg.k[1]);
  const uint8_t* vr = T.v_rows + blk * (PS * C::VROW);
  const int tok[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
  if constexpr (!C::VODD) {
#pragma unroll
    for (int i = 0; i < 4; ++i) load_words<C::VBYTES>(vr + tok[i] * C::VROW + g * C::VBYTES, pg.v[i]);
  } else {
    // 6-byte runs at 6g lie in the two aligned words from (6g & ~3); shift them down by
    // 16 bits when g is odd
    const int off = g * C::VBYTES, a = off & ~3, sh = 8 * (off - a);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(vr + tok[i] * C::VROW + a);
      const uint32_t w0 = __ldg(src), w1 = __ldg(src + 1);  // bytes a .. a+7, inside the row
      pg.v[i][0] = __funnelshift_r(w0, w1, sh);
      pg.v[i][1] = __funnelshift_r(w1, 0u, sh);
    }
  }
  const unsigned short* kn = reinterpret_cast<const unsigned short*>(T.k_norm) + blk * PS;
  const unsigned short* vn = reinterpret_cast<const unsigned short*>(T.v_norm) + blk * PS;
  const uint32_t k0 = __ldg(kn + g), k1 = __ldg(kn + g + 8);
  const uint32_t v0 = __ldg(vn + g), v1 = __ldg(vn + g + 8);
  pg.nk = k0 | (k1 << 16);
  pg.nv = v0 | (v1 << 16);
}

// L2 prefetch of the 128-byte lines of one page block (keys, values, both norm runs).
template <class C>
__device__ __forceinline__ void prefetch_page(const CbTier& T, int phys, int hk, int hkv, int lane) {
  constexpr int NK = PS * C::KROW / 128, NV = PS * C::VROW / 128;  // page blocks are whole lines
  const size_t blk = (size_t)phys * hkv + hk;
  for (int j = lane; j < NK + NV + 2; j += 32) {
    const void* a = j < NK ? (const void*)(T.k_rows + blk * (PS * C::KROW) + 128 * j)
                  : j < NK + NV ? (const void*)(T.v_rows + blk * (PS * C::VROW) + 128 * (j - NK))
                  : j == NK + NV ? (const void*)(T.k_norm + blk * PS) : (const void*)(T.v_norm + blk * PS);
    prefetch_l2(a);
  }
}

// ---------------------------------------------------------------- query rotation

// q' = H (s_K * q) * log2(e) / D * 2^6 for the G heads of kv head hk into qbuf[G][D].
// Lane l holds coordinates [l*D/32, (l+1)*D/32) of one head at a time: in-register
// butterfly stages, then five across lanes.
template <int D, int G>
__device__ __forceinline__ void rotate_query(const CbParams& p, int b, int hk, float* qbuf, int lane) {
  constexpr int E = D / 32;
  const int d0 = lane * E;
  const int8_t* sg = p.k_signs + hk * D + d0;
  int8_t s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) s[e] = sg[e];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __half* qs = p.q + ((size_t)b * p.hq + hk * G + h) * D + d0;
    float y[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float v = __half2float(qs[e]);
      y[e] = s[e] < 0 ? -v : v;
    }
#pragma unroll
    for (int hs = 1; hs < E; hs <<= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & hs) == 0) {
          const float a = y[e], c = y[e + hs];
          y[e] = a + c;
          y[e + hs] = a - c;
        }
      }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(kFull, y[e], m);
        y[e] = (lane & m) ? (o - y[e]) : (y[e] + o);
      }
    }
    constexpr float scale = kLog2e / (float)D * kQScale;
#pragma unroll
    for (int e = 0; e < E; ++e) qbuf[h * D + d0 + e] = y[e] * scale;
  }
}

// ---------------------------------------------------------------- one work item

// A work item: chunk `chunk` of sequence b, kv head hk.  `len` is loaded one item ahead and
// `btw` holds the block-table entry of page pg0 + lane of the item.
struct Item {
  int b, hk, chunk, t0, len;
  uint32_t btw;
};

__device__ __forceinline__ Item fetch_item(const CbParams& p, int item, int lane) {
  const CbTier& T = p.t;
  Item it;
  it.chunk = item % T.nchunks;
  const int rem = item / T.nchunks;
  it.hk = rem % p.hkv;
  it.b = rem / p.hkv;
  it.t0 = it.chunk * T.chunk;
  it.len = __ldg(T.seq_lens + it.b);
  const int pg = it.t0 / PS + lane;
  it.btw = pg < T.max_pages ? (uint32_t)__ldg(T.block_table + (size_t)it.b * T.max_pages + pg) : 0u;
  return it;
}

__device__ __forceinline__ int item_pages(const CbTier& T, const Item& it) {
  const int t1 = min(it.len, it.t0 + T.chunk);
  return t1 > it.t0 ? (t1 + PS - 1) / PS - it.t0 / PS : 0;
}

constexpr int kPrefetch = 3;  // pages between the L2 prefetch and the use of a page

template <int D, int G, int KB, int VB>
__device__ __forceinline__ void run_item(const CbParams& p, const Item& it, bool has_next, const Item& nx,
                                         float* qbuf, uint32_t klane, uint32_t vlane, int lane) {
  using C = Cfg<D, G, KB, VB>;
  const CbTier& T = p.t;
  const int b = it.b, hk = it.hk;
  const int t0 = it.t0, t1 = min(it.len, t0 + T.chunk);
  const int pg0 = t0 / PS, npg = (t1 + PS - 1) / PS - pg0;
  const int g = lane >> 2, c = lane & 3;
  // pages of the item that the previous item's tail did not prefetch (a warp's first item)
  for (int x = 0; x < min(kPrefetch, npg); ++x)
    prefetch_page<C>(T, __shfl_sync(kFull, it.btw, x), hk, p.hkv, lane);
  rotate_query<D, G>(p, b, hk, qbuf, lane);
  __syncwarp();
  // query B fragments: column g = (head g/2, part g%2); pair slots c*PPT + 2ks (+1)
  uint32_t qf[C::KS][2];
  const int hB = g >> 1;
  if (hB < G) {
    const float hl = (float)(g & 1);
    const uint32_t base = smem_addr(qbuf + hB * D + 2 * C::PPT * c);
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const uint4 v = lds128(base + 16 * ks);
      qf[ks][0] = split_pair(__uint_as_float(v.x), __uint_as_float(v.y), hl);
      qf[ks][1] = split_pair(__uint_as_float(v.z), __uint_as_float(v.w), hl);
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) qf[ks][0] = qf[ks][1] = 0u;
  }
  __syncwarp();

  float acc[C::KS][4];
#pragma unroll
  for (int i = 0; i < C::KS; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m = -INFINITY, l = 0.f;
  constexpr float kInvD = D == 128 ? 0.08838834764831845f : 0.0625f;  // 1/sqrt(D)
  constexpr float sscale = kInvD / (kQScale * kCScale);
  constexpr float wscale = kWScale * kInvD;
  const int srcA = 4 * (2 * c) + hB, srcB = srcA + 4;
  const bool lo_part = g & 1, live_col = hB < G;

  // block-table entries of pages [wbase, wbase + 32) and [wbase + 32, wbase + 64), one per lane
  const int32_t* bt = T.block_table + (size_t)b * T.max_pages + pg0;
  uint32_t btw0 = it.btw, btw1 = 0;
  int wbase = 0;
  if (npg > 32 && pg0 + 32 + lane < T.max_pages) btw1 = (uint32_t)__ldg(bt + 32 + lane);
  const int n_next = has_next ? item_pages(T, nx) : 0;
  Page<C> cur;
  load_page<C>(T, __shfl_sync(kFull, btw0, 0), hk, p.hkv, g, c, cur);
#pragma unroll 1
  for (int i = 0; i < npg; ++i) {
    if (i + 1 - wbase >= 32) {  // page i + 1 leaves the first window: slide by 32
      btw0 = btw1;
      wbase += 32;
      btw1 = (wbase + 32 + lane < npg) ? (uint32_t)__ldg(bt + wbase + 32 + lane) : 0u;
    }
    Page<C> nxt;
    if (i + 1 < npg) load_page<C>(T, __shfl_sync(kFull, btw0, i + 1 - wbase), hk, p.hkv, g, c, nxt);
    {  // L2 prefetch kPrefetch pages ahead in the warp's stream of pages
      const int x = i + kPrefetch;
      if (x < npg) {
        const int r = x - wbase;
        const uint32_t ph = r < 32 ? __shfl_sync(kFull, btw0, r) : __shfl_sync(kFull, btw1, r - 32);
        prefetch_page<C>(T, ph, hk, p.hkv, lane);
      } else if (x - npg < n_next) {
        prefetch_page<C>(T, __shfl_sync(kFull, nx.btw, x - npg), nx.hk, p.hkv, lane);
      }
    }
    // ---- scores of tokens g and g+8 for head c
    float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const uint2 e0 = lut64(field_addr<2 * KB>(cur.k[0], 2 * KB * (2 * ks), klane));
      const uint2 e1 = lut64(field_addr<2 * KB>(cur.k[1], 2 * KB * (2 * ks), klane));
      const uint2 e2 = lut64(field_addr<2 * KB>(cur.k[0], 2 * KB * (2 * ks + 1), klane));
      const uint2 e3 = lut64(field_addr<2 * KB>(cur.k[1], 2 * KB * (2 * ks + 1), klane));
      const uint32_t ah[4] = {e0.x, e1.x, e2.x, e3.x}, al[4] = {e0.y, e1.y, e2.y, e3.y};
      mma16816(sa[0], ah, qf[ks][0], qf[ks][1]);
      mma16816(sa[1], al, qf[ks][0], qf[ks][1]);
    }
    const __half2 nk = *reinterpret_cast<const __half2*>(&cur.nk);
    const __half2 nv = *reinterpret_cast<const __half2*>(&cur.nv);
    const int tok0 = (pg0 + i) * PS;
    const bool v0 = tok0 + g < t1, v1 = tok0 + g + 8 < t1;
    float x0 = ((sa[0][0] + sa[0][1]) + (sa[1][0] + sa[1][1])) * (__low2float(nk) * sscale);
    float x1 = ((sa[0][2] + sa[0][3]) + (sa[1][2] + sa[1][3])) * (__high2float(nk) * sscale);
    x0 = v0 ? x0 : -INFINITY;
    x1 = v1 ? x1 : -INFINITY;
    // ---- online softmax of head c over the 16 tokens
    float mt = fmaxf(x0, x1);
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
    if (mt > m) {
      const float f = exp2f(m - mt);  // m = -inf at first: f = 0
      l *= f;
#pragma unroll
      for (int a = 0; a < C::KS; ++a)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[a][k] *= f;
      m = mt;
    }
    const float p0 = v0 ? exp2f(x0 - m) : 0.f;
    const float p1 = v1 ? exp2f(x1 - m) : 0.f;
    l += p0 + p1;
    // ---- weight B fragments: column g = (head g/2, part g%2), tokens 2c, 2c+1 | 2c+8, 2c+9
    const float w0 = v0 ? p0 * (__low2float(nv) * wscale) : 0.f;
    const float w1 = v1 ? p1 * (__high2float(nv) * wscale) : 0.f;
    const uint32_t hi = pack_f16x2(w0, w1);
    const __half2 hh = *reinterpret_cast<const __half2*>(&hi);
    const uint32_t lo = pack_f16x2(w0 - __low2float(hh), w1 - __high2float(hh));
    const uint32_t ah = __shfl_sync(kFull, hi, srcA), al = __shfl_sync(kFull, lo, srcA);
    const uint32_t bh = __shfl_sync(kFull, hi, srcB), bl = __shfl_sync(kFull, lo, srcB);
    const uint32_t A = lo_part ? al : ah, B = lo_part ? bl : bh;
    const uint32_t b0 = live_col ? __byte_perm(A, B, 0x5410) : 0u;
    const uint32_t b1 = live_col ? __byte_perm(A, B, 0x7632) : 0u;
    // ---- values: m-tile mt covers pair slot g*QPT + mt of the four tokens
#pragma unroll
    for (int mt2 = 0; mt2 < C::KS; ++mt2) {
      const uint2 r0 = lut64(field_addr<2 * VB>(cur.v[0], 2 * VB * mt2, vlane));
      const uint2 r1 = lut64(field_addr<2 * VB>(cur.v[1], 2 * VB * mt2, vlane));
      const uint2 r2 = lut64(field_addr<2 * VB>(cur.v[2], 2 * VB * mt2, vlane));
      const uint2 r3 = lut64(field_addr<2 * VB>(cur.v[3], 2 * VB * mt2, vlane));
      const uint32_t ah4[4] = {__byte_perm(r0.x, r1.x, 0x5410), __byte_perm(r0.x, r1.x, 0x7632),
                               __byte_perm(r2.x, r3.x, 0x5410), __byte_perm(r2.x, r3.x, 0x7632)};
      const uint32_t al4[4] = {__byte_perm(r0.y, r1.y, 0x5410), __byte_perm(r0.y, r1.y, 0x7632),
                               __byte_perm(r2.y, r3.y, 0x5410), __byte_perm(r2.y, r3.y, 0x7632)};
      mma16816(acc[mt2], ah4, b0, b1);
      mma16816(acc[mt2], al4, b0, b1);
    }
    if (i + 1 < npg) cur = nxt;
  }
  // ---- partial of head c: sum over the 8 lanes of the head, coordinates 2*QPT*g ..
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(kFull, l, o);
  if (c < G) {
    const size_t part = ((size_t)b * p.hq + hk * G + c) * p.total_splits + T.split_begin + it.chunk;
    constexpr float unw = 1.0f / (kWScale * kCScale);
    float4* dst = reinterpret_cast<float4*>(p.ws_acc + part * D + 2 * C::QPT * g);
#pragma unroll
    for (int a = 0; a < C::KS; a += 2)
      dst[a / 2] = make_float4((acc[a][0] + acc[a][1]) * unw, (acc[a][2] + acc[a][3]) * unw,
                               (acc[a + 1][0] + acc[a + 1][1]) * unw, (acc[a + 1][2] + acc[a + 1][3]) * unw);
    if (g == 0) {
      p.ws_ml[2 * part] = m;
      p.ws_ml[2 * part + 1] = l;
    }
  }
}

// ================================================================ one query head per kv head
//
// With G = 1 the key and value work is a matrix-vector product: on the tensor cores six of
// the eight mma columns would idle and the value fragments would need two byte permutes per
// register, so this variant stays on the FMA pipes.  Lane (t, c) takes tokens t and t+8 of
// the page and the coordinates [c D/4, (c+1) D/4) of both; a table entry is the fp32 pair
// (C[first code], C[second code]) and feeds one packed fma.rn.f32x2 -- exact fp32 products,
// no hi/lo split.  Scores: packed partial dot products, summed over the 4 lanes of a token.
// Values: packed accumulators per coordinate pair, summed over the 8 lanes of a coordinate
// block once per item (a reduce-scatter: each lane ends with D/32 coordinates).
//
// Pages reach shared memory through a per-warp ring of STAGES slots filled by TMA bulk
// copies (cp.async.bulk, completion counted in bytes on one mbarrier per slot): one lane
// issues the four copies of a page block (keys, values, key norms, value norms) into the
// slot the warp has just read, STAGES pages ahead of their use, and the stream of pages runs
// on from one item into the next.  The tables: K and V entries interleave in one region
// (K at byte 0, V at byte 128 of each 256-byte entry), 16 lane copies each -- a 64-bit
// shared load is served half a warp at a time, so lanes l and l + 16 share a copy.
template <int D, int KB, int VB>
struct Cfg1 {
  static constexpr int DL = D / 4;              // coordinates per lane and token
  static constexpr int NP = DL / 2;             // pair slots per lane and token
  static constexpr int KROW = D * KB / 8;
  static constexpr int VROW = D * VB / 8;
  static constexpr int KBYTES = DL * KB / 8;
  static constexpr int VBYTES = DL * VB / 8;
  static constexpr int KW = KBYTES / 4;
  static constexpr int VW = VBYTES / 4;
  static constexpr int TABLE = (1 << (2 * (KB > VB ? KB : VB))) * 256;
  static constexpr int KBLK = PS * KROW, VBLK = PS * VROW;
  static constexpr int STAGE = KBLK + VBLK + 64;  // + 16 fp16 key norms + 16 value norms
  static constexpr int STAGES = 3;
  static constexpr int WARPS = D == 128 ? 16 : 8;
  static constexpr int QBUF = D * 4;
  static constexpr int WSM = STAGES * STAGE + QBUF + 16 * ((8 * STAGES + 15) / 16);  // ring, queries, barriers
  static constexpr int SMEM = (TABLE + WARPS * WSM + WSM > 2 * TABLE) ? TABLE + WARPS * WSM + WSM : 2 * TABLE;
};

constexpr int kSpinLimit = 1 << 22;  // try_wait rounds before a slot counts as lost
constexpr int kErrorWord = 32;       // index of the error word in the counter block

__device__ __forceinline__ void mbar_init(uint32_t a, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int NBYTES>
__device__ __forceinline__ void lds_run(uint32_t a, uint32_t* w) {
  if constexpr (NBYTES == 32 || NBYTES == 16) {
#pragma unroll
    for (int h = 0; h < NBYTES / 16; ++h)
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(w[4 * h]), "=r"(w[4 * h + 1]), "=r"(w[4 * h + 2]), "=r"(w[4 * h + 3])
                   : "r"(a + 16 * h));
  } else if constexpr (NBYTES == 24 || NBYTES == 8) {
#pragma unroll
    for (int h = 0; h < NBYTES / 8; ++h)
      asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w[2 * h]), "=r"(w[2 * h + 1]) : "r"(a + 8 * h));
  } else {
    static_assert(NBYTES == 12 || NBYTES == 4, "unsupported run length");
#pragma unroll
    for (int h = 0; h < NBYTES / 4; ++h) asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[h]) : "r"(a + 4 * h));
  }
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

template <int D, int KB, int VB>
struct Run1 {
  using C = Cfg1<D, KB, VB>;
  static constexpr float kInvD = D == 128 ? 0.08838834764831845f : 0.0625f;
  static constexpr float sscale = kInvD / kQScale;

  u64 q2[C::NP];
  u64 acc[C::NP];
  float m, l;

  // Scores, softmax update and value accumulation of one page whose lane words are in
  // k/v and norms in nk0/nk1/nv0/nv1; v0/v1: tokens t and t+8 lie inside the item.
  __device__ __forceinline__ void page(const uint32_t (&k)[2][C::KW], const uint32_t (&v)[2][C::VW], uint32_t nk0,
                                       uint32_t nk1, uint32_t nv0, uint32_t nv1, bool v0, bool v1, uint32_t klane,
                                       uint32_t vlane) {
    u64 s[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int j = 0; j < C::NP; ++j) {
      s[j & 1] = fma2(q2[j], lut64x(field_addr<2 * KB>(k[0], 2 * KB * j, klane)), s[j & 1]);
      s[2 + (j & 1)] = fma2(q2[j], lut64x(field_addr<2 * KB>(k[1], 2 * KB * j, klane)), s[2 + (j & 1)]);
    }
    float a0, b0, a1, b1, e0, f0, e1, f1;
    upk2(s[0], a0, b0);
    upk2(s[1], e0, f0);
    upk2(s[2], a1, b1);
    upk2(s[3], e1, f1);
    float x0 = (a0 + b0) + (e0 + f0), x1 = (a1 + b1) + (e1 + f1);
    x0 += __shfl_xor_sync(kFull, x0, 1);
    x1 += __shfl_xor_sync(kFull, x1, 1);
    x0 += __shfl_xor_sync(kFull, x0, 2);
    x1 += __shfl_xor_sync(kFull, x1, 2);
    x0 = v0 ? x0 * (__half2float(__ushort_as_half((uint16_t)nk0)) * sscale) : -INFINITY;
    x1 = v1 ? x1 * (__half2float(__ushort_as_half((uint16_t)nk1)) * sscale) : -INFINITY;
    float mt = fmaxf(x0, x1);
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
    if (mt > m) {
      const float f = exp2f(m - mt);  // m = -inf at first: f = 0
      l *= f;
      const u64 f2 = pk2(f, f);
#pragma unroll
      for (int j = 0; j < C::NP; ++j) acc[j] = mul2(acc[j], f2);
      m = mt;
    }
    const float p0 = v0 ? exp2f(x0 - m) : 0.f;
    const float p1 = v1 ? exp2f(x1 - m) : 0.f;
    l += p0 + p1;
    const float w0 = v0 ? p0 * (__half2float(__ushort_as_half((uint16_t)nv0)) * kInvD) : 0.f;
    const float w1 = v1 ? p1 * (__half2float(__ushort_as_half((uint16_t)nv1)) * kInvD) : 0.f;
    const u64 W0 = pk2(w0, w0), W1 = pk2(w1, w1);
#pragma unroll
    for (int j = 0; j < C::NP; ++j)
      acc[j] = fma2(W0, lut64x(field_addr<2 * VB>(v[0], 2 * VB * j, vlane)), acc[j]);
#pragma unroll
    for (int j = 0; j < C::NP; ++j)
      acc[j] = fma2(W1, lut64x(field_addr<2 * VB>(v[1], 2 * VB * j, vlane)), acc[j]);
  }
};

// A warp's page stream: ring slots, their barriers, and how far it has issued and consumed.
struct Ring {
  uint32_t slots, bars;  // shared addresses
  int issued, consumed;  // stream positions (pages)
  bool lost;             // a slot wait gave up
};

template <class C>
__device__ __forceinline__ void ring_issue(const CbTier& T, int hkv, Ring& rg, uint32_t phys, int hk, int lane) {
  const int slot = rg.issued % C::STAGES;
  if (lane == 0) {
    const uint32_t dst = rg.slots + slot * C::STAGE, bar = rg.bars + 8 * slot;
    const size_t blk = (size_t)phys * hkv + hk;
    fence_proxy_async();  // the slot's previous page was read through the generic proxy
    mbar_expect_tx(bar, C::STAGE);
    bulk_g2s(dst, T.k_rows + blk * C::KBLK, C::KBLK, bar);
    bulk_g2s(dst + C::KBLK, T.v_rows + blk * C::VBLK, C::VBLK, bar);
    bulk_g2s(dst + C::KBLK + C::VBLK, T.k_norm + blk * PS, 32, bar);
    bulk_g2s(dst + C::KBLK + C::VBLK + 32, T.v_norm + blk * PS, 32, bar);
  }
  ++rg.issued;
}

// Wait until the next page of the stream has landed; returns its slot address.
template <class C>
__device__ __forceinline__ uint32_t ring_wait(Ring& rg, int* err) {
  const int slot = rg.consumed % C::STAGES;
  const uint32_t parity = (rg.consumed / C::STAGES) & 1;
  int n = 0;
  while (!mbar_try_wait(rg.bars + 8 * slot, parity)) {
    if (++n >= kSpinLimit) {
      rg.lost = true;
      atomicExch(err, 1);
      break;
    }
  }
  return rg.slots + slot * C::STAGE;
}

template <int D, int KB, int VB>
__device__ __forceinline__ void run_item1(const CbParams& p, const Item& it, bool has_next, const Item& nx,
                                          float* qbuf, Ring& rg, uint32_t klane, uint32_t vlane, int lane) {
  using C = Cfg1<D, KB, VB>;
  using R = Run1<D, KB, VB>;
  const CbTier& T = p.t;
  const int b = it.b, hk = it.hk;
  const int t0 = it.t0, t1 = min(it.len, t0 + T.chunk);
  const int pg0 = t0 / PS, npg = (t1 + PS - 1) / PS - pg0;
  const int n_next = has_next ? item_pages(T, nx) : 0;
  const int t = lane >> 2, c = lane & 3;
  const int start = rg.consumed;  // stream position of page 0 of this item
  // block-table entries of pages [wbase, wbase + 32) and [wbase + 32, wbase + 64), one per lane
  const int32_t* bt = T.block_table + (size_t)b * T.max_pages + pg0;
  uint32_t btw0 = it.btw, btw1 = 0;
  int wbase = 0;
  if (npg > 32 && pg0 + 32 + lane < T.max_pages) btw1 = (uint32_t)__ldg(bt + 32 + lane);
  // keep STAGES pages of this item and the next in flight
  auto top_up = [&]() {
    while (rg.issued < rg.consumed + C::STAGES && rg.issued - start < npg + n_next) {
      const int o = rg.issued - start;
      if (o < npg) {
        if (o - wbase >= 32) {  // slide the window: pages [wbase + 32, wbase + 96)
          btw0 = btw1;
          wbase += 32;
          btw1 = (wbase + 32 + lane < npg) ? (uint32_t)__ldg(bt + wbase + 32 + lane) : 0u;
        }
        ring_issue<C>(T, p.hkv, rg, __shfl_sync(kFull, btw0, o - wbase), hk, lane);
      } else {
        ring_issue<C>(T, p.hkv, rg, __shfl_sync(kFull, nx.btw, o - npg), nx.hk, lane);
      }
    }
  };
  top_up();
  rotate_query<D, 1>(p, b, hk, qbuf, lane);
  __syncwarp();
  R r;
  {
    const uint32_t base = smem_addr(qbuf + C::DL * c);
#pragma unroll
    for (int j = 0; j < C::NP; j += 2) {
      const uint4 v = lds128(base + 8 * j);
      r.q2[j] = pk2(__uint_as_float(v.x), __uint_as_float(v.y));
      r.q2[j + 1] = pk2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
  }
#pragma unroll
  for (int j = 0; j < C::NP; ++j) r.acc[j] = 0ull;
  r.m = -INFINITY;
  r.l = 0.f;
#pragma unroll 1
  for (int i = 0; i < npg; ++i) {
    const uint32_t st = ring_wait<C>(rg, p.counter + kErrorWord);
    if (rg.lost) return;
    uint32_t k[2][C::KW], v[2][C::VW];
    lds_run<C::KBYTES>(st + t * C::KROW + c * C::KBYTES, k[0]);
    lds_run<C::KBYTES>(st + (t + 8) * C::KROW + c * C::KBYTES, k[1]);
    lds_run<C::VBYTES>(st + C::KBLK + t * C::VROW + c * C::VBYTES, v[0]);
    lds_run<C::VBYTES>(st + C::KBLK + (t + 8) * C::VROW + c * C::VBYTES, v[1]);
    const uint32_t nrm = st + C::KBLK + C::VBLK + 2 * t;
    const uint32_t nk0 = lds_u16(nrm), nk1 = lds_u16(nrm + 16), nv0 = lds_u16(nrm + 32), nv1 = lds_u16(nrm + 48);
    __syncwarp();  // every lane holds its words: the slot may be refilled
    ++rg.consumed;
    top_up();
    const int tok0 = (pg0 + i) * PS;
    r.page(k, v, nk0, nk1, nv0, nv1, tok0 + t < t1, tok0 + t + 8 < t1, klane, vlane);
  }
  // ---- sums over the 8 token lanes of a coordinate block: reduce-scatter on lane bits 4, 3, 2
  float a[C::DL];
#pragma unroll
  for (int j = 0; j < C::NP; ++j) upk2(r.acc[j], a[2 * j], a[2 * j + 1]);
#pragma unroll
  for (int s2 = 0; s2 < 3; ++s2) {
    const int msk = 16 >> s2, n = C::DL >> s2;
    const bool up = lane & msk;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = up ? a[k] : a[k + n / 2];
      const float keep = up ? a[k + n / 2] : a[k];
      a[k] = keep + __shfl_xor_sync(kFull, send, msk);
    }
  }
  float l = r.l;
  l += __shfl_xor_sync(kFull, l, 4);
  l += __shfl_xor_sync(kFull, l, 8);
  l += __shfl_xor_sync(kFull, l, 16);
  const size_t part = ((size_t)b * p.hq + hk) * p.total_splits + T.split_begin + it.chunk;
  const int off = C::DL * c + ((lane >> 4) & 1) * (C::DL / 2) + ((lane >> 3) & 1) * (C::DL / 4) +
                  ((lane >> 2) & 1) * (C::DL / 8);
  float4* dst = reinterpret_cast<float4*>(p.ws_acc + part * D + off);
#pragma unroll
  for (int k = 0; k < C::DL / 8; k += 4) dst[k / 4] = make_float4(a[k], a[k + 1], a[k + 2], a[k + 3]);
  if (lane == 0) {
    p.ws_ml[2 * part] = r.m;
    p.ws_ml[2 * part + 1] = l;
  }
}

// K and V fp32 pair tables, interleaved: entry e, lane copy l (0..15): K at
// base + e*256 + l*8, V at base + e*256 + 128 + l*8.
template <int KB, int VB>
__device__ void build_tables_f32(const float* kc, const float* vc, uint32_t base) {
  constexpr int NK = 1 << (2 * KB), NV = 1 << (2 * VB), N = NK > NV ? NK : NV;
  for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
    const int e = i >> 5, half = (i >> 4) & 1, ln = i & 15;
    const int bits = half ? VB : KB;
    if (e >= (half ? NV : NK)) continue;
    const float* cent = half ? vc : kc;
    const int mask = (1 << bits) - 1;
    sts64(base + e * 256 + half * 128 + ln * 8, __float_as_uint(__ldg(cent + (e & mask))),
          __float_as_uint(__ldg(cent + (e >> bits))));
  }
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(Cfg1<D, KB, VB>::WARPS * 32, 1)
    decode_cb1_kernel(const __grid_constant__ CbParams p) {
  using C = Cfg1<D, KB, VB>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the table sits at a shared address that is a multiple of its size; warp areas fill the
  // space before it first, then follow it
  const uint32_t base = smem_addr(smem);
  const uint32_t a_t = (base + C::TABLE - 1) & ~(uint32_t)(C::TABLE - 1);
  const int nfit = min(C::WARPS, (int)((a_t - base) / C::WSM));
  const uint32_t end = nfit == C::WARPS ? a_t + C::TABLE : a_t + C::TABLE + (C::WARPS - nfit) * C::WSM;
  if (end > base + (uint32_t)p.smem_bytes) return;  // the launcher sizes smem for any base
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t area = warp < nfit ? base + warp * C::WSM : a_t + C::TABLE + (warp - nfit) * C::WSM;
  Ring rg;
  rg.slots = area;
  rg.bars = area + C::STAGES * C::STAGE + C::QBUF;
  rg.issued = rg.consumed = 0;
  rg.lost = false;
  float* qbuf = reinterpret_cast<float*>(smem + (area + C::STAGES * C::STAGE - base));
  if (lane == 0) {
    for (int s2 = 0; s2 < C::STAGES; ++s2) mbar_init(rg.bars + 8 * s2, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  build_tables_f32<KB, VB>(p.k_cent, p.v_cent, a_t);
  __syncthreads();
  const uint32_t klane = pin(a_t | ((lane & 15) << 3)), vlane = pin(a_t | 128 | ((lane & 15) << 3));
  int item = 0, next = 0;
  if (lane == 0) {
    item = atomicAdd(p.counter, 1);
    next = atomicAdd(p.counter, 1);
  }
  item = __shfl_sync(kFull, item, 0);
  next = __shfl_sync(kFull, next, 0);
  Item cur = fetch_item(p, item < p.total_items ? item : 0, lane);
  while (item < p.total_items && !rg.lost) {
    int after = 0;
    if (lane == 0) after = atomicAdd(p.counter, 1);
    const bool has_next = next < p.total_items;
    Item nx = cur;
    if (has_next) {
      nx = fetch_item(p, next, lane);
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q + ((size_t)nx.b * p.hq + nx.hk) * D);
      if (lane < D / 64) prefetch_l2(qrow + 128 * lane);
    }
    if (cur.len > cur.t0) run_item1<D, KB, VB>(p, cur, has_next, nx, qbuf, rg, klane, vlane, lane);
    item = next;
    next = __shfl_sync(kFull, after, 0);
    cur = nx;
  }
  // a warp that gave up on a slot waits (bounded) for whatever it still has in flight
  if (rg.lost) {
    for (; rg.consumed < rg.issued; ++rg.consumed) {
      const int slot = rg.consumed % C::STAGES;
      const uint32_t parity = (rg.consumed / C::STAGES) & 1;
      for (int n = 0; n < kSpinLimit && !mbar_try_wait(rg.bars + 8 * slot, parity); ++n) {
      }
    }
  }
}

// Fill one lane-replicated table at shared address `base`: entry e (pair field), lane l at
// base + e*256 + l*8 = {fp16x2 hi(256 C[e & mask], 256 C[e >> bits]), fp16x2 remainders}.
template <int BITS>
__device__ void build_table(const float* cent, uint32_t base) {
  constexpr int N = 1 << (2 * BITS), mask = (1 << BITS) - 1;
  for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
    const int e = i >> 5, ln = i & 31;
    const float c0 = __ldg(cent + (e & mask)) * kCScale, c1 = __ldg(cent + (e >> BITS)) * kCScale;
    sts64(base + e * 256 + ln * 8, split_pair(c0, c1, 0.f), split_pair(c0, c1, 1.f));
  }
}

template <int D, int G, int KB, int VB>
__global__ void __launch_bounds__(Cfg<D, G, KB, VB>::WARPS * 32, 1)
    decode_cb_kernel(const __grid_constant__ CbParams p) {
  using C = Cfg<D, G, KB, VB>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the tables start at shared addresses that are multiples of their sizes (the larger
  // first); the per-warp query buffers follow them
  const uint32_t base = smem_addr(smem);
  constexpr uint32_t big = C::KLUT >= C::VLUT ? C::KLUT : C::VLUT;
  constexpr uint32_t small = C::KLUT >= C::VLUT ? C::VLUT : C::KLUT;
  const uint32_t a_big = (base + big - 1) & ~(big - 1);
  const uint32_t a_small = a_big + big;
  const uint32_t a_q = a_small + small;
  if (a_q + C::WARPS * C::QBUF > base + (uint32_t)p.smem_bytes) return;  // launcher sizes smem for any base
  const uint32_t a_k = C::KLUT >= C::VLUT ? a_big : a_small;
  const uint32_t a_v = C::KLUT >= C::VLUT ? a_small : a_big;
  build_table<KB>(p.k_cent, a_k);
  build_table<VB>(p.v_cent, a_v);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* qbuf = reinterpret_cast<float*>(smem + (a_q - base) + warp * C::QBUF);
  const uint32_t klane = pin(a_k | (lane << 3)), vlane = pin(a_v | (lane << 3));
  // items: the one in hand, the next (its metadata and queries fetched while this one
  // runs), and the one after (its counter ticket in flight)
  int item = 0, next = 0;
  if (lane == 0) {
    item = atomicAdd(p.counter, 1);
    next = atomicAdd(p.counter, 1);
  }
  item = __shfl_sync(kFull, item, 0);
  next = __shfl_sync(kFull, next, 0);
  Item cur = fetch_item(p, item < p.total_items ? item : 0, lane);
  while (item < p.total_items) {
    int after = 0;
    if (lane == 0) after = atomicAdd(p.counter, 1);
    const bool has_next = next < p.total_items;
    Item nx = cur;
    if (has_next) {
      nx = fetch_item(p, next, lane);
      // the next item's query rows: G * D fp16 = G * D / 64 lines
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q + ((size_t)nx.b * p.hq + nx.hk * G) * D);
      if (lane < G * D / 64) prefetch_l2(qrow + 128 * lane);
    }
    if (cur.len > cur.t0) run_item<D, G, KB, VB>(p, cur, has_next, nx, qbuf, klane, vlane, lane);
    item = next;
    next = __shfl_sync(kFull, after, 0);
    cur = nx;
  }
}

template <int D, int G, int KB, int VB>
cudaError_t launch_cb(const CbParams& p, int sms, cudaStream_t stream) {
  using C = Cfg<D, G, KB, VB>;
  auto kern = decode_cb_kernel<D, G, KB, VB>;
  const int need = (C::KLUT >= C::VLUT ? C::KLUT : C::VLUT) + C::KLUT + C::VLUT + C::WARPS * C::QBUF;
  CbParams q = p;
  q.smem_bytes = need;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int ctas = std::max(1, std::min(sms, (p.total_items + C::WARPS - 1) / C::WARPS));
  kern<<<ctas, C::WARPS * 32, need, stream>>>(q);
  return cudaGetLastError();
}

template <int D, int KB, int VB>
cudaError_t launch_cb1(const CbParams& p, int sms, cudaStream_t stream) {
  using C = Cfg1<D, KB, VB>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  auto kern = decode_cb1_kernel<D, KB, VB>;
  CbParams q = p;
  q.smem_bytes = C::SMEM;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int ctas = std::max(1, std::min(sms, (p.total_items + 2 * C::WARPS - 1) / (2 * C::WARPS)));
  kern<<<ctas, C::WARPS * 32, C::SMEM, stream>>>(q);
  return cudaGetLastError();
}

template <int D, int G, int KB>
cudaError_t launch_vb(const CbParams& p, int vb, int sms, cudaStream_t s) {
  if constexpr (G == 1) {
    switch (vb) {
      case 2: return launch_cb1<D, KB, 2>(p, sms, s);
      case 3: return launch_cb1<D, KB, 3>(p, sms, s);
      default: return launch_cb1<D, KB, 4>(p, sms, s);
    }
  } else {
    switch (vb) {
      case 2: return launch_cb<D, G, KB, 2>(p, sms, s);
      case 3: return launch_cb<D, G, KB, 3>(p, sms, s);
      default: return launch_cb<D, G, KB, 4>(p, sms, s);
    }
  }
}

template <int D, int G>
cudaError_t launch_kb(const CbParams& p, int kb, int vb, int sms, cudaStream_t s) {
  switch (kb) {
    case 2: return launch_vb<D, G, 2>(p, vb, sms, s);
    case 3: return launch_vb<D, G, 3>(p, vb, sms, s);
    default: return launch_vb<D, G, 4>(p, vb, sms, s);
  }
}

template <int D>
cudaError_t launch_g(const CbParams& p, int g, int kb, int vb, int sms, cudaStream_t s) {
  switch (g) {
    case 1: return launch_kb<D, 1>(p, kb, vb, sms, s);
    case 2: return launch_kb<D, 2>(p, kb, vb, sms, s);
    default: return launch_kb<D, 4>(p, kb, vb, sms, s);
  }
}

}  // namespace

bool cb_fast_supported(int head_dim, int group, int k_fmt, int v_fmt) {
  return (head_dim == 128 || head_dim == 256) && (group == 1 || group == 2 || group == 4) &&
         k_fmt == KVQ_FMT_CODEBOOK && v_fmt == KVQ_FMT_CODEBOOK;
}

cudaError_t launch_decode_cb(const DecParams& dp, int head_dim, int* counters, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(counters, 0, 64 * sizeof(int), stream);  // work counters and the error word
  if (e != cudaSuccess) return e;
  const int group = dp.hq / dp.hkv;
  for (int i = 0; i < dp.num_tiers; ++i) {
    const DecTier& t = dp.tier[i];
    CbParams p;
    memset(&p, 0, sizeof(p));
    p.t.k_rows = t.k_rows;
    p.t.v_rows = t.v_rows;
    p.t.k_norm = t.k_aux;
    p.t.v_norm = t.v_aux;
    p.t.block_table = t.block_table;
    p.t.seq_lens = t.seq_lens;
    p.t.max_pages = t.max_pages;
    p.t.chunk = t.chunk;
    p.t.nchunks = t.num_splits;
    p.t.split_begin = t.split_begin;
    p.q = dp.q;
    p.k_signs = dp.k_signs;
    p.k_cent = t.k_cent;
    p.v_cent = t.v_cent;
    p.ws_acc = dp.ws_acc;
    p.ws_ml = dp.ws_ml;
    p.counter = counters + i;
    p.hq = dp.hq;
    p.hkv = dp.hkv;
    p.total_splits = dp.total_splits;
    p.total_items = dp.batch * dp.hkv * t.num_splits;
    if (p.total_items == 0) continue;
    e = head_dim == 128 ? launch_g<128>(p, group, t.k_bits, t.v_bits, sms, stream)
                        : launch_g<256>(p, group, t.k_bits, t.v_bits, sms, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvq
