// Fused decode attention over codebook tiers (b-bit Lloyd-Max or uniform codes + fp16 norm
// for keys and values), head_dim 128 or 256, 1, 2 or 4 query heads per kv head.
//
// The score of a key row is q'.k~ with k~_j = (norm / sqrt(D)) C[idx_j] (TurboQuant page,
// the dequantisation step; AdapTQ page, "Engineering the Hot Path": the rotated query meets
// the stored codes directly, through a table of centroids).  Values accumulate in the
// rotated domain the same way and the combine pass undoes the rotation once.
//
// Work: items of (sequence, kv head, chunk of pages), handed to warps from an atomic
// counter; every warp is independent and writes one split-K partial per item.
//
// Pages reach shared memory through a per-warp ring of STAGES slots filled by TMA bulk
// copies (cp.async.bulk, completion counted in bytes on one mbarrier per slot): one lane
// issues the four copies of a page block (16 key rows, 16 value rows, their 16 key norms and
// 16 value norms) into the slot the warp has just read, STAGES pages ahead of their use, and
// the stream of pages runs on from one item into the next.  Every wait on a slot is bounded.
//
// Codes become numbers through tables in shared memory indexed by a pair field (2b bits =
// two codes, the first code in the low bits).  K and V entries interleave in one region (K
// at byte 0, V at byte 128 of each 256-byte entry) with 16 lane copies each: a 64-bit shared
// load is served half a warp at a time, so lanes l and l + 16 can share a copy while the 16
// lanes of a half-warp always hit 16 different bank pairs.  The region sits at a shared
// address aligned to its size, so the lookup address of lane l is
// (field << 8) | ((l & 15) << 3) | base (+128 for V): one byte permute (byte fields) or one
// shift and one logic op from the packed word.
//
// Two paths share that machinery:
//  * G = 1 (Path1): a matrix-vector product, kept on the FMA pipes.  Lane (t, c) takes
//    tokens t and t+8 of the page and coordinates [c D/4, (c+1) D/4); a table entry is the
//    fp32 pair (C[first], C[second]) and feeds one packed fma.rn.f32x2 -- exact fp32
//    products.  Scores: packed partial dot products summed over the 4 lanes of a token.
//    Values: packed accumulators per coordinate pair, summed over the 8 lanes of a
//    coordinate block once per item (a reduce-scatter: each lane ends with D/32 coords).
//  * G = 2, 4 (PathM): the G heads make a real contraction, done with mma.sync.m16n8k16
//    (fp16 inputs, fp32 accumulation):
//        scores  S[16 tokens x 8]  = K~[16 tokens x D] . Q[D x 8]
//        values  O[16 dims x 8]   += V~^T[16 dims x 16 tokens] . W[16 tokens x 8]
//    The 8 columns are (head, hi/lo); columns of heads >= G are zero.  Table entries hold
//    fp16 of 256 C and fp16 of the remainder, so each code pair feeds two mma (hi, lo); the
//    query and the weights are split the same way, and the products keep ~22 bits.  The
//    dot product does not care in which order its terms are summed, so lane (g, c) of the
//    key mma takes the pair slots [c D/8, (c+1) D/8) of rows g and g+8 and the query
//    fragments follow that order; the value mma maps its A rows g and g+8 of m-tile mt to
//    the two coordinates of pair slot g D/16 + mt, so one lookup gives both rows and the
//    lane's output coordinates come out contiguous.  Value fragments pair two tokens per
//    register, so the value lookups index the same pair table with the codes of two
//    tokens at one coordinate: per page the lane merges the code runs of its token pairs
//    (a shift and a bit select per word) and each entry is then a ready A register pair.
//    With 2-bit values a byte of the merged run covers two m-tiles: where shared memory
//    allows, a quad table (256 byte values x 16 lane copies x 16 bytes) gives both tiles'
//    registers in one 16-byte lookup addressed by one byte permute.
// (Kernel templates shared by decode_cb.cu -- plain codebook keys -- and decode_cb_qjl.cu
// -- keys with a residual sketch -- so the two instance sets compile in parallel.)
#pragma once
#include <algorithm>
#include <atomic>
#include <cstring>

#include "kvq_internal.cuh"

namespace kvq {
namespace cbk {

constexpr int PS = 16;
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kCScale = 256.0f;  // fp16 table entries hold 2^8 C
constexpr float kQScale = 64.0f;   // the rotated queries hold 2^6 q'
constexpr float kWScale = 8.0f;    // weight fragments hold 2^3 p norm / sqrt(D); with p <= 1
                                   // every fp16 norm stays below the fp16 maximum
constexpr int kSpinLimit = 1 << 22;  // try_wait rounds before a slot counts as lost
// KVQ_SPIN_TEST (a test-only build, never the library's): the slot wait polls once with the
// non-blocking test_wait, and a warp polls the first slot of its stream before the copies
// of that slot are issued -- a poll that cannot succeed -- then issues them: the give-up
// path runs on valid data every time, with copies in flight; the drain after a give-up
// keeps the full limit, so every issued copy lands before the CTA exits.
#ifdef KVQ_SPIN_TEST
constexpr int kSlotSpinLimit = 1;
#else
constexpr int kSlotSpinLimit = kSpinLimit;
#endif
typedef unsigned long long u64;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Table lookups.  Not volatile: once the tables are built a lookup is a plain function of
// its address, which leaves the compiler free to overlap lookups with arithmetic.  Every
// lookup address derives from a value pin()ned after the barrier that ends the build.
__device__ __forceinline__ uint2 lut64(uint32_t a) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ u64 lut64x(uint32_t a) {
  u64 v;
  asm("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t pin(uint32_t x) {
  asm volatile("" : "+r"(x));
  return x;
}
__device__ __forceinline__ void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ uint4 lut128(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
__device__ __forceinline__ u64 pk2(float a, float b) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(u64 r, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r)); }
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
// Non-blocking probe of a phase (test builds' slot wait).
__device__ __forceinline__ bool mbar_test_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// NBYTES of packed bits at shared address a (4-byte aligned) into words.
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

// ---------------------------------------------------------------- parameters
struct CbTier {
  const uint8_t* k_rows;
  const uint8_t* v_rows;
  const __half* k_norm;  // keys with a residual sketch: (norm, residual norm) pairs
  const __half* v_norm;
  const float* qjl;      // keys with a residual sketch: projection [KVQ_QJL_DIM][D]
  const int32_t* outl;   // keys with an outlier stream: channels [Hkv][KVQ_OUTLIER_CHANNELS]
  const int32_t* block_table;
  const int32_t* seq_lens;
  int* err;  // the call's error word (KVQ_DEVERR_* bits)
  int num_pages, max_pages, chunk, nchunks, split_begin;
};

struct CbParams {
  CbTier t;
  const __half* q;
  const int8_t* k_signs;
  const float* k_cent;
  const float* v_cent;
  float* ws_acc;
  float* ws_ml;
  float* pq;     // keys with a residual sketch: p' = S q' per query head, [B][Hq][KVQ_QJL_DIM]
  float* ws_min; // lowest score per split, written when `track` (tier 0, spike flags asked for)
  int* counter;  // this launch's work counter
  int hq, hkv, total_splits, total_items, smem_bytes;
  int gate, track;  // score-gated value loading; record the lowest score
  int pdl;          // launched as a programmatic dependent of the previous split-K launch
  int trigger;      // another split-K launch follows: let it start on SMs this grid leaves
};

// Shared-memory plan common to both paths: table region (aligned to its size), the residual
// sketch's +-1 pair table after it (keys with a sketch), then per warp a ring of STAGES page
// slots, a buffer for the rotated queries and the slot barriers.
// Key formats of the codebook kernel: plain codes, codes + residual sign sketch, codes +
// outlier stream.
constexpr int kModePlain = 0, kModeSketch = 1, kModeOutlier = 2;

// Shared memory of a CTA: the table block (quad table if any, pair table, sketch table),
// aligned to its first table's size, and one area per warp.  The alignment may leave up to
// that size - 1 bytes before the block; warp areas fill that gap first, so the worst case
// wastes under one area.
constexpr int block_smem(int qtab, int table, int skt, int warps, int wsm) {
  const int align = qtab ? qtab : table, blk = qtab + table + skt;
  return blk + warps * wsm + wsm > align + blk ? blk + warps * wsm + wsm : align + blk;
}

template <int D, int G, int KB, int VB, int WARPS_, int MODE_, int STAGES_ = 3>
struct Layout {
  static constexpr bool QJL = MODE_ == kModeSketch, OUT = MODE_ == kModeOutlier;
  static constexpr int KCODE = D * KB / 8;                            // code bytes of a key row
  static constexpr int KROW = KCODE + (QJL ? KVQ_QJL_DIM / 8 : 0), VROW = D * VB / 8;
  static constexpr int KBLK = PS * KROW, VBLK = PS * VROW;
  static constexpr int KNORM = PS * (QJL ? 4 : (OUT ? 4 + KVQ_OUTLIER_CHANNELS : 2));  // key side data of a page block
  static constexpr int STAGE = KBLK + VBLK + KNORM + 32;  // + 16 fp16 value norms
  static constexpr int STAGES = STAGES_;
  static constexpr int WARPS = WARPS_;
  static constexpr int TABLE = (1 << (2 * (KB > VB ? KB : VB))) * 256;
  static constexpr int SKT = QJL ? 4 * 256 : 0;  // 4 entries: pairs of sketch signs
  static constexpr int QBUF = G * D * 4;
  static constexpr int QLINES = G * D * 2 / 128;  // fp16 query rows of the group, in lines
  static constexpr int WSM = STAGES * STAGE + QBUF + 16 * ((8 * STAGES + 15) / 16);
  // 2-bit values on the tensor-core path: a quad table indexed by a byte of two pair slots
  // (256 entries x 16 lane copies x 16 bytes) before the pair table, where it fits
  static constexpr int QTAB =
      (G > 1 && VB == 2 && block_smem(65536, TABLE, SKT, WARPS, WSM) <= 227 * 1024) ? 65536 : 0;
  static constexpr int ALIGN = QTAB ? QTAB : TABLE;  // the table block's alignment
  static constexpr int SMEM = block_smem(QTAB, TABLE, SKT, WARPS, WSM);
  static_assert(SMEM <= 227 * 1024, "shared memory budget");

  // Where things go for a dynamic shared-memory window starting at `base`: the table block
  // at a multiple of its alignment (quad table at q, pair table at t), the first `nfit`
  // warp areas in the gap before it, the rest from w on; `end` is one past the last byte.
  struct Placement {
    uint32_t q, t, w, end;
    int nfit;
  };
  __host__ __device__ static Placement place(uint32_t base) {
    Placement pl;
    pl.q = (base + ALIGN - 1) & ~(uint32_t)(ALIGN - 1);
    pl.t = pl.q + QTAB;
    const int gap = (int)((pl.q - base) / WSM);
    pl.nfit = gap < WARPS ? gap : WARPS;
    pl.w = pl.t + TABLE + SKT;
    pl.end = pl.nfit == WARPS ? pl.w : pl.w + (WARPS - pl.nfit) * WSM;
    return pl;
  }
  // Shared address of warp area `warp`.
  __host__ __device__ static uint32_t area(const Placement& pl, uint32_t base, int warp) {
    return warp < pl.nfit ? base + warp * WSM : pl.w + (warp - pl.nfit) * WSM;
  }
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

// Code runs of two tokens a, b (NW words each, VB-bit codes, pair slots of 2 VB bits) merged
// so that pair slot k of x holds (a's code, b's code) of the slot's first coordinate and
// slot k of y those of its second: the pair field then indexes a table entry
// (C[code of a], C[code of b]), i.e. two tokens at one coordinate.
__host__ __device__ constexpr uint32_t first_code_mask(int vb, int word) {
  uint32_t m = 0;
  for (int n = 0; n < 32; ++n)
    if ((32 * word + n) % (2 * vb) < vb) m |= 1u << n;
  return m;
}
template <int VB, int NW>
__device__ __forceinline__ void token_pairs(const uint32_t (&a)[NW], const uint32_t (&b)[NW], uint32_t (&x)[NW],
                                            uint32_t (&y)[NW]) {
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const uint32_t m = first_code_mask(VB, i);
    const uint32_t bu = i > 0 ? __funnelshift_l(b[i - 1], b[i], VB) : (b[i] << VB);       // b one code up
    const uint32_t ad = i + 1 < NW ? __funnelshift_r(a[i], a[i + 1], VB) : (a[i] >> VB);  // a one code down
    x[i] = (a[i] & m) | (bu & ~m);
    y[i] = (ad & m) | (b[i] & ~m);
  }
}

// ---------------------------------------------------------------- query rotation

// q' = H (s_K * q) * log2(e) / D * 2^6 for heads h0 .. h0 + G - 1 of kv head hk (GQ query heads
// per kv head) into qbuf[G][D].
// Lane l holds coordinates [l*D/32, (l+1)*D/32) of one head at a time: in-register
// butterfly stages, then five across lanes.
template <int D, int G, int GQ = G>
__device__ __forceinline__ void rotate_query(const CbParams& p, int b, int hk, int h0, float* qbuf, int lane) {
  constexpr int E = D / 32;
  const int d0 = lane * E;
  const int8_t* sg = p.k_signs + hk * D + d0;
  int8_t s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) s[e] = sg[e];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __half* qs = p.q + ((size_t)b * p.hq + hk * GQ + h0 + h) * D + d0;
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

// ---------------------------------------------------------------- work items, page stream

// A work item: chunk `chunk` of sequence b, kv head hk.  `len` is loaded one item ahead and
// `btw` holds the block-table entry of page t0/16 + lane of the item.
struct Item {
  int b, hk, h0, chunk, t0, len;  // h0: the item's first query head within the kv head's group
  uint32_t btw;
};

// H8: a group of 8 query heads, two items (heads 0-3, 4-7) per chunk.
template <bool H8>
__device__ __forceinline__ Item fetch_item(const CbParams& p, int item, int lane) {
  const CbTier& T = p.t;
  Item it;
  it.chunk = item % T.nchunks;
  int rem = item / T.nchunks;
  // a group of 8: every chunk of heads 0-3, then every chunk of heads 4-7, so the second
  // pass over a chunk comes a few items later and finds its pages in L2
  it.h0 = H8 ? 4 * (rem & 1) : 0;
  rem = H8 ? rem >> 1 : rem;
  it.hk = rem % p.hkv;
  it.b = rem / p.hkv;
  it.t0 = it.chunk * T.chunk;
  // a length past the block table is cut there (the combine pass reports it); a negative
  // one leaves the item empty
  it.len = min(__ldg(T.seq_lens + it.b), T.max_pages * PS);
  const int pg = it.t0 / PS + lane;
  it.btw = pg < T.max_pages ? (uint32_t)__ldg(T.block_table + (size_t)it.b * T.max_pages + pg) : 0u;
  return it;
}

__device__ __forceinline__ int item_pages(const CbTier& T, const Item& it) {
  const int t1 = min(it.len, it.t0 + T.chunk);
  return t1 > it.t0 ? (t1 + PS - 1) / PS - it.t0 / PS : 0;
}

// A warp's page stream: ring slots, their barriers, and how far it has issued and consumed.
struct Ring {
  uint32_t slots, bars;  // shared addresses
  int issued, consumed;  // stream positions (pages)
  bool lost;             // a slot wait gave up
};

// 2^x, x <= 0 or -inf (scores in base-2 units relative to the running maximum): the
// hardware approximation (relative error below 2^-22), results below 2^-126 flushed to 0.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Issues the copies of page `phys`.  A block-table entry outside the pool (warp-uniform
// test, which also catches negative entries) is never read through: page 0 is copied in its
// place (the host gives a pool without pages no work) and the call reports the entry.
template <class L>
__device__ __forceinline__ void ring_issue(const CbTier& T, int hkv, Ring& rg, uint32_t phys, int hk, int lane) {
  if (__builtin_expect(phys >= (uint32_t)T.num_pages, 0)) {
    if (lane == 0) atomicOr(T.err, KVQ_DEVERR_PAGE_INDEX);
    phys = 0;
  }
  const int slot = rg.issued % L::STAGES;
  if (lane == 0) {
    const uint32_t dst = rg.slots + slot * L::STAGE, bar = rg.bars + 8 * slot;
    const size_t blk = (size_t)phys * hkv + hk;
    fence_proxy_async();  // the slot's previous page was read through the generic proxy
    mbar_expect_tx(bar, L::STAGE);
    bulk_g2s(dst, T.k_rows + blk * L::KBLK, L::KBLK, bar);
    bulk_g2s(dst + L::KBLK, T.v_rows + blk * L::VBLK, L::VBLK, bar);
    bulk_g2s(dst + L::KBLK + L::VBLK, T.k_norm + blk * (L::KNORM / 2), L::KNORM, bar);
    bulk_g2s(dst + L::KBLK + L::VBLK + L::KNORM, T.v_norm + blk * PS, 32, bar);
  }
  ++rg.issued;
}

// Wait until the next page of the stream has landed; returns its slot address.
template <class L>
__device__ __forceinline__ uint32_t ring_wait(Ring& rg, int* err, int lane) {
  const int slot = rg.consumed % L::STAGES;
  if (rg.lost) return rg.slots;  // a warp that gave up waits for nothing more
  const uint32_t parity = (rg.consumed / L::STAGES) & 1;
  int n = 0;
#ifdef KVQ_SPIN_TEST
  while (!mbar_test_wait(rg.bars + 8 * slot, parity)) {
#else
  while (!mbar_try_wait(rg.bars + 8 * slot, parity)) {
#endif
    if (++n >= kSlotSpinLimit) {
      rg.lost = true;
      break;
    }
  }
  // A phase seen complete at the first poll is complete for every lane.  After a longer
  // wait, lanes that kept polling agree through a vote: the warp is lost if any gave up.
  if (__builtin_expect(n > 0, 0)) {
    rg.lost = __any_sync(__activemask(), rg.lost);
    if (rg.lost && lane == 0) atomicOr(err, KVQ_DEVERR_COPY_TIMEOUT);
  }
  return rg.slots + slot * L::STAGE;
}



// Feeds the pages of an item (and the first pages of the next one) into the ring, STAGES
// ahead of consumption.  Block-table entries of pages [wbase, wbase + 32) and
// [wbase + 32, wbase + 64) of the item live one per lane.
template <class L>
struct Feeder {
  const CbTier* T;
  const int32_t* bt;
  const Item* nx;
  uint32_t btw0, btw1;
  int wbase, start, npg, n_next, hk, hkv, lane;

  __device__ __forceinline__ void init(const CbParams& p, const Item& it, const Item& nxt, int n_pages, int n_nxt,
                                       const Ring& rg, int ln) {
    T = &p.t;
    nx = &nxt;
    lane = ln;
    hk = it.hk;
    hkv = p.hkv;
    npg = n_pages;
    n_next = n_nxt;
    start = rg.consumed;
    const int pg0 = it.t0 / PS;
    bt = T->block_table + (size_t)it.b * T->max_pages + pg0;
    btw0 = it.btw;
    btw1 = 0u;
    wbase = 0;
    if (npg > 32 && pg0 + 32 + lane < T->max_pages) btw1 = (uint32_t)__ldg(bt + 32 + lane);
  }
  __device__ __forceinline__ void top_up(Ring& rg) {
    while (rg.issued < rg.consumed + L::STAGES && rg.issued - start < npg + n_next && !rg.lost) {
      const int o = rg.issued - start;
      if (o < npg) {
        if (o - wbase >= 32) {  // slide the window by 32 pages
          btw0 = btw1;
          wbase += 32;
          btw1 = (wbase + 32 + lane < npg) ? (uint32_t)__ldg(bt + wbase + 32 + lane) : 0u;
        }
        ring_issue<L>(*T, hkv, rg, __shfl_sync(kFull, btw0, o - wbase), hk, lane);
      } else {
        ring_issue<L>(*T, hkv, rg, __shfl_sync(kFull, nx->btw, o - npg), nx->hk, lane);
      }
    }
  }
};

// ---------------------------------------------------------------- residual sketch
// Keys stored with a residual sign sketch (VeloxQuant-MLX page, "Stage 3: QJL Residual
// Correction"): the score gains ||r~|| sqrt(pi/2) / m * sum_j z_j <S_j, q~>, z_j = +-1.  In
// base-2 score units, with the kernel's scaled query q' (= q~ log2(e) / sqrt(D) * 2^6):
// rnorm * kSketch * sum_j z_j <S_j, q'> with kSketch = sqrt(pi/2) / m / 2^6.  The sign bits
// are a 1-bit code of m "coordinates" with its own query p' = S q': pairs of bits index a
// 4-entry table of (+-1, +-1) like any other code pair.
constexpr float kSketch = 1.2533141373155003f / KVQ_QJL_DIM / kQScale;

// Outlier stream (VeloxQuant-MLX page, "Outlier Two-Stream Cache"): the score gains
// sum_j q[c_j] q_j s, in base-2 score units times log2(e) / sqrt(D).
template <int D>
struct OutlierScale {
  static constexpr float v = D == 128 ? 0.12751743074960564f : 0.09016844005556021f;  // log2(e) / sqrt(D)
};

// Sign-extended int8 k of a 32-bit word, as float.
__device__ __forceinline__ float i8f(uint32_t w, int k) { return (float)(int)(int8_t)(w >> (8 * k)); }

// p' = S q' for every query head, once per call (every split of a head reads it): one block
// of 4 warps per (sequence, kv head); lane l of warp w computes row 32w + l for the G heads.
template <int D, int G>
__global__ void __launch_bounds__(128) project_kernel(const __grid_constant__ CbParams p) {
  static_assert(KVQ_QJL_DIM == 4 * 32, "one row per thread");
  __shared__ __align__(16) float qs[4][G * D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / p.hkv, hk = blockIdx.x - b * p.hkv;
  rotate_query<D, G>(p, b, hk, 0, qs[warp], lane);
  __syncwarp();
  const int j = 32 * warp + lane;
  const float4* srow = reinterpret_cast<const float4*>(p.t.qjl + (size_t)j * D);
  float a[G], c[G];
#pragma unroll
  for (int h = 0; h < G; ++h) a[h] = c[h] = 0.f;
#pragma unroll 8
  for (int e = 0; e < D; e += 4) {
    const float4 sv = __ldg(srow + e / 4);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 qv = *reinterpret_cast<const float4*>(&qs[warp][h * D + e]);
      a[h] = fmaf(sv.x, qv.x, fmaf(sv.y, qv.y, a[h]));
      c[h] = fmaf(sv.z, qv.z, fmaf(sv.w, qv.w, c[h]));
    }
  }
  float* dst = p.pq + ((size_t)b * p.hq + hk * G) * KVQ_QJL_DIM + j;
#pragma unroll
  for (int h = 0; h < G; ++h) dst[h * KVQ_QJL_DIM] = a[h] + c[h];
}

// The +-1 pair table: entry e (two sign bits, first in the low bit), lane copy l at
// base + e * 256 + l * 8: fp32 pairs (FMA path) or {fp16x2 pair, 0} (tensor-core path).
template <bool F32>
__device__ void build_sketch_table(uint32_t base) {
  for (int i = threadIdx.x; i < 4 * 16; i += blockDim.x) {
    const int e = i >> 4, ln = i & 15;
    const float z0 = (e & 1) ? 1.f : -1.f, z1 = (e & 2) ? 1.f : -1.f;
    if (F32) sts64(base + e * 256 + ln * 8, __float_as_uint(z0), __float_as_uint(z1));
    else sts64(base + e * 256 + ln * 8, pack_f16x2(z0, z1), 0u);
  }
}

// ================================================================ G = 1: FMA path
template <int D, int KB, int VB, int MODE>
struct Path1 {
  static constexpr bool QJL = MODE == kModeSketch, OUT = MODE == kModeOutlier;
  using L = Layout<D, 1, KB, VB, D == 128 ? (QJL ? 12 : 16) : 8, MODE>;
  static constexpr int kD = D, kG = 1, kGQ = 1;
  static constexpr bool kH8 = false;
  static constexpr int SNP = KVQ_QJL_DIM / 8;  // sketch sign pairs per lane and token (a quarter of m)
  static constexpr int DL = D / 4;  // coordinates per lane and token
  static constexpr int NP = DL / 2;  // pair slots per lane and token
  static constexpr int KBYTES = DL * KB / 8, VBYTES = DL * VB / 8;
  static constexpr int KW = KBYTES / 4, VW = VBYTES / 4;
  static constexpr float kInvD = D == 128 ? 0.08838834764831845f : 0.0625f;

  // K and V fp32 pair tables: entry e, lane copy l at base + e*256 + l*8 (K) and +128 (V);
  // the sketch table after them.
  __device__ static void build_tables(const float* kc, const float* vc, uint32_t base) {
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
    if (QJL) build_sketch_table<true>(base + L::TABLE);
  }

  __device__ static void run_item(const CbParams& p, const Item& it, bool has_next, const Item& nx, float* qbuf,
                                  Ring& rg, uint32_t klane, uint32_t vlane, uint32_t slane, int lane) {
    const CbTier& T = p.t;
    const int b = it.b, hk = it.hk;
    const int t1 = min(it.len, it.t0 + T.chunk);
    const int pg0 = it.t0 / PS, npg = item_pages(T, it);
    const int t = lane >> 2, c = lane & 3;
    Feeder<L> fd;
    fd.init(p, it, nx, npg, has_next ? item_pages(T, nx) : 0, rg, lane);
#ifdef KVQ_SPIN_TEST
    if (rg.issued == 0) {  // test build: poll the first slot before its copies exist, then
      ring_wait<L>(rg, T.err, lane);  // issue them so that the drain has copies to wait for
      rg.lost = false;
      fd.top_up(rg);
      rg.lost = true;
    }
#endif
    fd.top_up(rg);
    rotate_query<D, 1>(p, b, hk, 0, qbuf, lane);
    __syncwarp();
    u64 q2[NP], acc[NP], p2[QJL ? SNP : 1];
    {
      const uint32_t base = smem_addr(qbuf + DL * c);
#pragma unroll
      for (int j = 0; j < NP; j += 2) {
        const uint4 v = lds128(base + 8 * j);
        q2[j] = pk2(__uint_as_float(v.x), __uint_as_float(v.y));
        q2[j + 1] = pk2(__uint_as_float(v.z), __uint_as_float(v.w));
      }
    }
    if constexpr (QJL) {  // p' = S q'; lane (t, c) keeps the pairs of sketch rows [32c, 32c + 32)
      const float4* src = reinterpret_cast<const float4*>(p.pq + ((size_t)b * p.hq + hk) * KVQ_QJL_DIM + 2 * SNP * c);
#pragma unroll
      for (int j = 0; j < SNP; j += 2) {
        const float4 v = src[j / 2];
        p2[j] = pk2(v.x, v.y);
        p2[j + 1] = pk2(v.z, v.w);
      }
    }
    float qo0 = 0.f, qo1 = 0.f;  // outlier stream: q[c_2c], q[c_2c+1] in score units
    if constexpr (OUT) {
      const int2 ch = __ldg(reinterpret_cast<const int2*>(T.outl + hk * KVQ_OUTLIER_CHANNELS) + c);
      const __half* qrow = p.q + ((size_t)b * p.hq + hk) * D;
      qo0 = __half2float(qrow[ch.x & (D - 1)]) * OutlierScale<D>::v;  // the mask keeps a bad list in bounds
      qo1 = __half2float(qrow[ch.y & (D - 1)]) * OutlierScale<D>::v;
    }
#pragma unroll
    for (int j = 0; j < NP; ++j) acc[j] = 0ull;
    float m = -INFINITY, l = 0.f, mn = INFINITY;
    constexpr float sscale = kInvD / kQScale;
#pragma unroll 1
    for (int i = 0; i < npg; ++i) {
      const uint32_t st = ring_wait<L>(rg, T.err, lane);
      if (rg.lost) break;  // nothing more is read: the item's partial is written empty below
      uint32_t k[2][KW], v[2][VW];
      lds_run<KBYTES>(st + t * L::KROW + c * KBYTES, k[0]);
      lds_run<KBYTES>(st + (t + 8) * L::KROW + c * KBYTES, k[1]);
      lds_run<VBYTES>(st + L::KBLK + t * L::VROW + c * VBYTES, v[0]);
      lds_run<VBYTES>(st + L::KBLK + (t + 8) * L::VROW + c * VBYTES, v[1]);
      uint32_t sw[2][1] = {{0u}, {0u}}, rn0 = 0, rn1 = 0, nk0, nk1, op0 = 0, op1 = 0;
      if constexpr (QJL) {  // sign bits [32c, 32c + 32) of both tokens; (norm, residual norm)
        lds_run<4>(st + t * L::KROW + L::KCODE + 4 * c, sw[0]);
        lds_run<4>(st + (t + 8) * L::KROW + L::KCODE + 4 * c, sw[1]);
        const uint32_t kn = st + L::KBLK + L::VBLK + 4 * t;
        nk0 = lds_u16(kn);
        rn0 = lds_u16(kn + 2);
        nk1 = lds_u16(kn + 32);
        rn1 = lds_u16(kn + 34);
      } else if constexpr (OUT) {  // (norm, scale) and the int8 pair 2c, 2c+1 of both tokens
        const uint32_t kn = st + L::KBLK + L::VBLK + 12 * t;
        nk0 = lds_u16(kn);
        rn0 = lds_u16(kn + 2);
        op0 = lds_u16(kn + 4 + 2 * c);
        nk1 = lds_u16(kn + 96);
        rn1 = lds_u16(kn + 98);
        op1 = lds_u16(kn + 100 + 2 * c);
      } else {
        const uint32_t kn = st + L::KBLK + L::VBLK + 2 * t;
        nk0 = lds_u16(kn);
        nk1 = lds_u16(kn + 16);
      }
      const uint32_t vn = st + L::KBLK + L::VBLK + L::KNORM + 2 * t;
      const uint32_t nv0 = lds_u16(vn), nv1 = lds_u16(vn + 16);
      __syncwarp();  // every lane holds its words: the slot may be refilled
      ++rg.consumed;
      fd.top_up(rg);
      const int tok0 = (pg0 + i) * PS;
      const bool v0 = tok0 + t < t1, v1 = tok0 + t + 8 < t1;
      // ---- scores of tokens t and t+8
      u64 s[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        s[j & 1] = fma2(q2[j], lut64x(field_addr<2 * KB>(k[0], 2 * KB * j, klane)), s[j & 1]);
        s[2 + (j & 1)] = fma2(q2[j], lut64x(field_addr<2 * KB>(k[1], 2 * KB * j, klane)), s[2 + (j & 1)]);
      }
      float a0, b0, a1, b1, e0, f0, e1, f1;
      upk2(s[0], a0, b0);
      upk2(s[1], e0, f0);
      upk2(s[2], a1, b1);
      upk2(s[3], e1, f1);
      // lane partials, each part scaled by its own norm, then summed over the 4 lanes
      float x0 = ((a0 + b0) + (e0 + f0)) * (__half2float(__ushort_as_half((uint16_t)nk0)) * sscale);
      float x1 = ((a1 + b1) + (e1 + f1)) * (__half2float(__ushort_as_half((uint16_t)nk1)) * sscale);
      if constexpr (QJL) {
        u64 z0 = 0ull, z1 = 0ull;
#pragma unroll
        for (int j = 0; j < SNP; ++j) {
          z0 = fma2(p2[j], lut64x(field_addr<2>(sw[0], 2 * j, slane)), z0);
          z1 = fma2(p2[j], lut64x(field_addr<2>(sw[1], 2 * j, slane)), z1);
        }
        float za, zb, zc, zd;
        upk2(z0, za, zb);
        upk2(z1, zc, zd);
        x0 = fmaf(za + zb, __half2float(__ushort_as_half((uint16_t)rn0)) * kSketch, x0);
        x1 = fmaf(zc + zd, __half2float(__ushort_as_half((uint16_t)rn1)) * kSketch, x1);
      }
      if constexpr (OUT) {  // this lane's two of the eight outlier terms, times the token's scale
        x0 = fmaf(fmaf(qo1, i8f(op0, 1), qo0 * i8f(op0, 0)), __half2float(__ushort_as_half((uint16_t)rn0)), x0);
        x1 = fmaf(fmaf(qo1, i8f(op1, 1), qo0 * i8f(op1, 0)), __half2float(__ushort_as_half((uint16_t)rn1)), x1);
      }
      x0 += __shfl_xor_sync(kFull, x0, 1);
      x1 += __shfl_xor_sync(kFull, x1, 1);
      x0 += __shfl_xor_sync(kFull, x0, 2);
      x1 += __shfl_xor_sync(kFull, x1, 2);
      x0 = v0 ? x0 : -INFINITY;
      x1 = v1 ? x1 : -INFINITY;
      // ---- online softmax over the 16 tokens
      // the page maximum matters only where a score rises above the running maximum (and
      // for the gate): one vote settles the usual page, whose maximum is below it
      float mt = fmaxf(x0, x1);
      if (p.gate || __any_sync(kFull, mt > m)) {
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
      }
      if (mt > m) {
        const float f = exp2_fast(m - mt);  // m = -inf at first: f = 0
        l *= f;
        const u64 f2 = pk2(f, f);
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[j] = mul2(acc[j], f2);
        m = mt;
      }
      const float p0 = v0 ? exp2_fast(x0 - m) : 0.f;
      const float p1 = v1 ? exp2_fast(x1 - m) : 0.f;
      l += p0 + p1;
      if (p.track) {
        float lo = fminf(v0 ? x0 : INFINITY, v1 ? x1 : INFINITY);
        lo = fminf(lo, __shfl_xor_sync(kFull, lo, 4));
        lo = fminf(lo, __shfl_xor_sync(kFull, lo, 8));
        mn = fminf(mn, fminf(lo, __shfl_xor_sync(kFull, lo, 16)));
      }
      if (p.gate && mt - m < -kGateLog2) continue;  // score gate: mt is warp-uniform here
      const float w0 = v0 ? p0 * (__half2float(__ushort_as_half((uint16_t)nv0)) * kInvD) : 0.f;
      const float w1 = v1 ? p1 * (__half2float(__ushort_as_half((uint16_t)nv1)) * kInvD) : 0.f;
      const u64 W0 = pk2(w0, w0), W1 = pk2(w1, w1);
      // ---- values of tokens t and t+8
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[j] = fma2(W0, lut64x(field_addr<2 * VB>(v[0], 2 * VB * j, vlane)), acc[j]);
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[j] = fma2(W1, lut64x(field_addr<2 * VB>(v[1], 2 * VB * j, vlane)), acc[j]);
    }
    if (rg.lost) {  // a wait gave up: the item contributes nothing (its partial says so)
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[j] = 0ull;
      m = -INFINITY;
      l = 0.f;
      mn = INFINITY;
    }
    // ---- sums over the 8 token lanes of a coordinate block: reduce-scatter on lane bits 4, 3, 2
    float a[DL];
#pragma unroll
    for (int j = 0; j < NP; ++j) upk2(acc[j], a[2 * j], a[2 * j + 1]);
#pragma unroll
    for (int s2 = 0; s2 < 3; ++s2) {
      const int msk = 16 >> s2, n = DL >> s2;
      const bool up = lane & msk;
#pragma unroll
      for (int k = 0; k < n / 2; ++k) {
        const float send = up ? a[k] : a[k + n / 2];
        const float keep = up ? a[k + n / 2] : a[k];
        a[k] = keep + __shfl_xor_sync(kFull, send, msk);
      }
    }
    l += __shfl_xor_sync(kFull, l, 4);
    l += __shfl_xor_sync(kFull, l, 8);
    l += __shfl_xor_sync(kFull, l, 16);
    const size_t part = ((size_t)b * p.hq + hk) * p.total_splits + T.split_begin + it.chunk;
    const int off = DL * c + ((lane >> 4) & 1) * (DL / 2) + ((lane >> 3) & 1) * (DL / 4) + ((lane >> 2) & 1) * (DL / 8);
    float4* dst = reinterpret_cast<float4*>(p.ws_acc + part * D + off);
#pragma unroll
    for (int k = 0; k < DL / 8; k += 4) dst[k / 4] = make_float4(a[k], a[k + 1], a[k + 2], a[k + 3]);
    if (lane == 0) {
      p.ws_ml[2 * part] = m;
      p.ws_ml[2 * part + 1] = l;
      if (p.track) p.ws_min[part] = mn;
    }
  }
};

// ================================================================ G = 1: 8 lanes a token
// Plain codes, one query head per kv head, at head_dim 256.  The 4-lanes-a-token mapping of
// Path1 holds
// D/4 coordinates of the query pairs and of the value accumulators per lane (~250
// registers at D = 256: 8 warps per SM to hide the table lookups' latency); here lane
// (t, c) takes coordinates [c D/8, (c + 1) D/8) of tokens t, t+4, t+8 and t+12 of the page,
// which halves that state, so more warps fit: at D = 256 12 warps with two ring stages (168
// registers; measured on the append workload: 837 us per decode call with Path1's 8 warps,
// 771 with 11 warps and three stages, 755 with 12 and two).  Same arithmetic as Path1
// (exact fp32 pair products).  At head_dim 128 (2- and 4-bit codes, whose runs are whole
// words) the same mapping measured slower than Path1 on llama7b: 112.6 / 113.6 / 145 us with
// 16 / 20 / 24 warps against 110.7 us (three shuffle stages per score instead of two, and
// 8-byte code runs).
template <int D, int KB, int VB, int WARPS_ = (D == 256 ? 12 : 20), int STAGES_ = (D == 256 ? 2 : 3)>
struct Path1W {
  using L = Layout<D, 1, KB, VB, WARPS_, kModePlain, STAGES_>;
  static constexpr int kD = D, kG = 1, kGQ = 1;
  static constexpr bool kH8 = false;
  static constexpr int LPT = 8, TS = 32 / LPT, TPL = PS / TS;  // lanes a token, token slots, tokens a lane
  static constexpr int DL = D / LPT;                          // coordinates per lane and token
  static constexpr int NP = DL / 2;                           // pair slots per lane and token
  static constexpr int KBYTES = DL * KB / 8, VBYTES = DL * VB / 8;
  static constexpr int KW = KBYTES / 4, VW = VBYTES / 4;
  static constexpr float kInvD = D == 128 ? 0.08838834764831845f : 0.0625f;
  static_assert(KBYTES % 4 == 0 && VBYTES % 4 == 0, "whole-word runs");

  __device__ static void build_tables(const float* kc, const float* vc, uint32_t base) {
    Path1<D, KB, VB, kModePlain>::build_tables(kc, vc, base);
  }

  __device__ static void run_item(const CbParams& p, const Item& it, bool has_next, const Item& nx, float* qbuf,
                                  Ring& rg, uint32_t klane, uint32_t vlane, uint32_t, int lane) {
    const CbTier& T = p.t;
    const int b = it.b, hk = it.hk;
    const int t1 = min(it.len, it.t0 + T.chunk);
    const int pg0 = it.t0 / PS, npg = item_pages(T, it);
    const int t = lane / LPT, c = lane % LPT;
    Feeder<L> fd;
    fd.init(p, it, nx, npg, has_next ? item_pages(T, nx) : 0, rg, lane);
#ifdef KVQ_SPIN_TEST
    if (rg.issued == 0) {  // test build: poll the first slot before its copies exist, then
      ring_wait<L>(rg, T.err, lane);  // issue them so that the drain has copies to wait for
      rg.lost = false;
      fd.top_up(rg);
      rg.lost = true;
    }
#endif
    fd.top_up(rg);
    rotate_query<D, 1>(p, b, hk, 0, qbuf, lane);
    __syncwarp();
    u64 q2[NP], acc[NP];
    {
      const uint32_t base = smem_addr(qbuf + DL * c);
#pragma unroll
      for (int j = 0; j < NP; j += 2) {
        const uint4 v = lds128(base + 8 * j);
        q2[j] = pk2(__uint_as_float(v.x), __uint_as_float(v.y));
        q2[j + 1] = pk2(__uint_as_float(v.z), __uint_as_float(v.w));
      }
    }
#pragma unroll
    for (int j = 0; j < NP; ++j) acc[j] = 0ull;
    float m = -INFINITY, l = 0.f, mn = INFINITY;
    constexpr float sscale = kInvD / kQScale;
#pragma unroll 1
    for (int i = 0; i < npg; ++i) {
      const uint32_t st = ring_wait<L>(rg, T.err, lane);
      if (rg.lost) break;  // nothing more is read: the item's partial is written empty below
      uint32_t k[TPL][KW], v[TPL][VW], nk[TPL], nv[TPL];
#pragma unroll
      for (int r = 0; r < TPL; ++r) {
        const int tok = t + TS * r;
        lds_run<KBYTES>(st + tok * L::KROW + c * KBYTES, k[r]);
        lds_run<VBYTES>(st + L::KBLK + tok * L::VROW + c * VBYTES, v[r]);
        nk[r] = lds_u16(st + L::KBLK + L::VBLK + 2 * tok);
        nv[r] = lds_u16(st + L::KBLK + L::VBLK + L::KNORM + 2 * tok);
      }
      __syncwarp();  // every lane holds its words: the slot may be refilled
      ++rg.consumed;
      fd.top_up(rg);
      const int tok0 = (pg0 + i) * PS;
      // ---- scores of the lane's four tokens, each part scaled by its own norm, then summed
      // over the 8 lanes of a token
      float x[TPL];
#pragma unroll
      for (int r = 0; r < TPL; ++r) {
        u64 s0 = 0ull, s1 = 0ull;
#pragma unroll
        for (int j = 0; j < NP; j += 2) {
          s0 = fma2(q2[j], lut64x(field_addr<2 * KB>(k[r], 2 * KB * j, klane)), s0);
          s1 = fma2(q2[j + 1], lut64x(field_addr<2 * KB>(k[r], 2 * KB * (j + 1), klane)), s1);
        }
        float a0, b0, e0, f0;
        upk2(s0, a0, b0);
        upk2(s1, e0, f0);
        x[r] = ((a0 + b0) + (e0 + f0)) * (__half2float(__ushort_as_half((uint16_t)nk[r])) * sscale);
      }
#pragma unroll
      for (int o = 1; o < LPT; o <<= 1)
#pragma unroll
        for (int r = 0; r < TPL; ++r) x[r] += __shfl_xor_sync(kFull, x[r], o);
      bool val[TPL];
      float mt = -INFINITY;
#pragma unroll
      for (int r = 0; r < TPL; ++r) {
        val[r] = tok0 + t + TS * r < t1;
        x[r] = val[r] ? x[r] : -INFINITY;
        mt = fmaxf(mt, x[r]);
      }
      // ---- online softmax over the 16 tokens: the page maximum matters only where a score
      // rises above the running maximum (and for the gate)
      if (p.gate || __any_sync(kFull, mt > m)) {
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o));
      }
      if (mt > m) {
        const float f = exp2_fast(m - mt);  // m = -inf at first: f = 0
        l *= f;
        const u64 f2 = pk2(f, f);
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[j] = mul2(acc[j], f2);
        m = mt;
      }
      float pr[TPL];
#pragma unroll
      for (int r = 0; r < TPL; ++r) {
        pr[r] = val[r] ? exp2_fast(x[r] - m) : 0.f;
        l += pr[r];
      }
      if (p.track) {
        float lo = INFINITY;
#pragma unroll
        for (int r = 0; r < TPL; ++r) lo = fminf(lo, val[r] ? x[r] : INFINITY);
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) lo = fminf(lo, __shfl_xor_sync(kFull, lo, o));
        mn = fminf(mn, lo);
      }
      if (p.gate && mt - m < -kGateLog2) continue;  // score gate: mt is warp-uniform here
      // ---- values of the lane's four tokens
#pragma unroll
      for (int r = 0; r < TPL; ++r) {
        const float w = val[r] ? pr[r] * (__half2float(__ushort_as_half((uint16_t)nv[r])) * kInvD) : 0.f;
        const u64 W = pk2(w, w);
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[j] = fma2(W, lut64x(field_addr<2 * VB>(v[r], 2 * VB * j, vlane)), acc[j]);
      }
    }
    if (rg.lost) {  // a wait gave up: the item contributes nothing (its partial says so)
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[j] = 0ull;
      m = -INFINITY;
      l = 0.f;
      mn = INFINITY;
    }
    // ---- sums over the 4 token slots of a coordinate block: reduce-scatter on lane bits 4, 3
    float a[DL];
#pragma unroll
    for (int j = 0; j < NP; ++j) upk2(acc[j], a[2 * j], a[2 * j + 1]);
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const int msk = 16 >> s2, n = DL >> s2;
      const bool up = lane & msk;
#pragma unroll
      for (int kk = 0; kk < n / 2; ++kk) {
        const float send = up ? a[kk] : a[kk + n / 2];
        const float keep = up ? a[kk + n / 2] : a[kk];
        a[kk] = keep + __shfl_xor_sync(kFull, send, msk);
      }
    }
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) l += __shfl_xor_sync(kFull, l, o);
    const size_t part = ((size_t)b * p.hq + hk) * p.total_splits + T.split_begin + it.chunk;
    const int off = DL * c + ((lane >> 4) & 1) * (DL / 2) + ((lane >> 3) & 1) * (DL / 4);
    float4* dst = reinterpret_cast<float4*>(p.ws_acc + part * D + off);
#pragma unroll
    for (int kk = 0; kk < DL / 4; kk += 4) dst[kk / 4] = make_float4(a[kk], a[kk + 1], a[kk + 2], a[kk + 3]);
    if (lane == 0) {
      p.ws_ml[2 * part] = m;
      p.ws_ml[2 * part + 1] = l;
      if (p.track) p.ws_min[part] = mn;
    }
  }
};

// ================================================================ G = 2, 4: tensor-core path
// WIDE: 16 warps instead of 12 (register-limited to 128, a few spilled bytes): more warps
// hide more of the path's latency on large caches, fewer items per warp hurt small ones.
// H8 (G = 4 only): 8 query heads per kv head, two items per chunk, heads 0-3 and 4-7.
template <int D, int G, int KB, int VB, int MODE, bool WIDE = false, bool H8 = false>
struct PathM {
  static_assert(!H8 || G == 4, "a group of 8 runs as two items of 4 heads");
  static constexpr bool QJL = MODE == kModeSketch, OUT = MODE == kModeOutlier;
  using L = Layout<D, G, KB, VB, D == 128 ? (QJL ? 10 : (WIDE ? 16 : 12)) : 8, MODE>;
  static constexpr int kD = D, kG = G, GQ = H8 ? 8 : G, kGQ = GQ;
  static constexpr bool kH8 = H8;
  static constexpr int SKS = KVQ_QJL_DIM / 16;  // sketch mma k-steps
  static constexpr int KS = D / 16;            // key mma k-steps; also value m-tiles
  static constexpr int PPT = D / 8;            // key pair slots per lane (index c)
  static constexpr int QPT = D / 16;           // value pair slots per lane (index g)
  static constexpr int KBYTES = PPT * KB / 4;  // key bits of one lane, in bytes
  static constexpr int VBYTES = QPT * VB / 4;
  static constexpr int KW = KBYTES / 4;
  static constexpr bool VODD = (VBYTES % 4) != 0;  // 3-bit values at D = 128: 6 bytes at 6g
  static constexpr int VW = VODD ? 2 : VBYTES / 4;

  // fp16 hi / remainder tables of 256 C: entry e, lane copy l at base + e*256 + l*8 (K) and
  // +128 (V) = {fp16x2 hi(256 C[e & mask], 256 C[e >> bits]), fp16x2 remainders}.
  __device__ static void build_tables(const float* kc, const float* vc, uint32_t base) {
    constexpr int NK = 1 << (2 * KB), NV = 1 << (2 * VB), N = NK > NV ? NK : NV;
    for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
      const int e = i >> 5, half = (i >> 4) & 1, ln = i & 15;
      const int bits = half ? VB : KB;
      if (e >= (half ? NV : NK)) continue;
      const float* cent = half ? vc : kc;
      const int mask = (1 << bits) - 1;
      const float c0 = __ldg(cent + (e & mask)) * kCScale, c1 = __ldg(cent + (e >> bits)) * kCScale;
      sts64(base + e * 256 + half * 128 + ln * 8, split_pair(c0, c1, 0.f), split_pair(c0, c1, 1.f));
    }
    if (QJL) build_sketch_table<false>(base + L::TABLE);
    if constexpr (L::QTAB != 0) {  // entry e, lane copy l at base - QTAB + e*256 + l*16: the
                                   // pair-table entries of e's low and high nibbles
      for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
        const int e = i >> 4, ln = i & 15;
        const float c0 = __ldg(vc + (e & 3)) * kCScale, c1 = __ldg(vc + ((e >> 2) & 3)) * kCScale;
        const float c2 = __ldg(vc + ((e >> 4) & 3)) * kCScale, c3 = __ldg(vc + (e >> 6)) * kCScale;
        sts128(base - L::QTAB + e * 256 + ln * 16, split_pair(c0, c1, 0.f), split_pair(c0, c1, 1.f),
               split_pair(c2, c3, 0.f), split_pair(c2, c3, 1.f));
      }
    }
  }

  __device__ static void run_item(const CbParams& p, const Item& it, bool has_next, const Item& nx, float* qbuf,
                                  Ring& rg, uint32_t klane, uint32_t vlane, uint32_t slane, int lane) {
    const CbTier& T = p.t;
    const int b = it.b, hk = it.hk;
    const int t1 = min(it.len, it.t0 + T.chunk);
    const int pg0 = it.t0 / PS, npg = item_pages(T, it);
    const int g = lane >> 2, c = lane & 3;
    const int h0 = H8 ? it.h0 : 0;  // the item's first query head within its kv head's group
    // quad-table lookup base: the table block starts QTAB below the pair table, which is
    // aligned to its size; lane copy (l & 15) at 16-byte steps
    const uint32_t qlane = pin(((vlane & ~(uint32_t)(L::TABLE - 1)) - L::QTAB) | ((lane & 15) << 4));
    Feeder<L> fd;
    fd.init(p, it, nx, npg, has_next ? item_pages(T, nx) : 0, rg, lane);
#ifdef KVQ_SPIN_TEST
    if (rg.issued == 0) {  // test build: poll the first slot before its copies exist, then
      ring_wait<L>(rg, T.err, lane);  // issue them so that the drain has copies to wait for
      rg.lost = false;
      fd.top_up(rg);
      rg.lost = true;
    }
#endif
    fd.top_up(rg);
    rotate_query<D, G, GQ>(p, b, hk, h0, qbuf, lane);
    __syncwarp();
    // query B fragments: column g = (head g/2, part g%2); pair slots c*PPT + 2ks (+1)
    uint32_t qf[KS][2];
    const int hB = g >> 1;
    if (hB < G) {
      const float hl = (float)(g & 1);
      const uint32_t base = smem_addr(qbuf + hB * D + 2 * PPT * c);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint4 v = lds128(base + 16 * ks);
        qf[ks][0] = split_pair(__uint_as_float(v.x), __uint_as_float(v.y), hl);
        qf[ks][1] = split_pair(__uint_as_float(v.z), __uint_as_float(v.w), hl);
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) qf[ks][0] = qf[ks][1] = 0u;
    }
    // sketch B fragments: p' = S q' of head g/2, rows c*16 + 2ks (+1) pair by pair, as qf
    uint32_t pf[QJL ? SKS : 1][2];
    if constexpr (QJL) {
      if (hB < G) {
        const float hl = (float)(g & 1);
        const float4* src =
            reinterpret_cast<const float4*>(p.pq + ((size_t)b * p.hq + hk * GQ + h0 + hB) * KVQ_QJL_DIM + 32 * c);
#pragma unroll
        for (int ks = 0; ks < SKS; ++ks) {
          const float4 v = src[ks];
          pf[ks][0] = split_pair(v.x, v.y, hl);
          pf[ks][1] = split_pair(v.z, v.w, hl);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < SKS; ++ks) pf[ks][0] = pf[ks][1] = 0u;
      }
    }
    float qo[OUT ? KVQ_OUTLIER_CHANNELS : 1];  // outlier stream: q[c_j] of head c, score units
    if constexpr (OUT) {
      const int32_t* ch = T.outl + hk * KVQ_OUTLIER_CHANNELS;
      const __half* qrow = p.q + ((size_t)b * p.hq + hk * GQ + h0 + (c < G ? c : 0)) * D;
#pragma unroll
      for (int j = 0; j < KVQ_OUTLIER_CHANNELS; ++j)
        qo[j] = c < G ? __half2float(qrow[__ldg(ch + j) & (D - 1)]) * OutlierScale<D>::v : 0.f;
    }
    float acc[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m = -INFINITY, l = 0.f, mn = INFINITY;
    constexpr float kInvD = D == 128 ? 0.08838834764831845f : 0.0625f;
    constexpr float sscale = kInvD / (kQScale * kCScale);
    constexpr float wscale = kWScale * kInvD;
    const int srcA = 4 * (2 * c) + hB, srcB = srcA + 4;
    const bool lo_part = g & 1, live_col = hB < G;
#pragma unroll 1
    for (int i = 0; i < npg; ++i) {
      const uint32_t st = ring_wait<L>(rg, T.err, lane);
      if (rg.lost) break;  // nothing more is read: the item's partial is written empty below
      uint32_t k[2][KW], v[4][VW];
      lds_run<KBYTES>(st + g * L::KROW + c * KBYTES, k[0]);
      lds_run<KBYTES>(st + (g + 8) * L::KROW + c * KBYTES, k[1]);
      const int tok[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
      if constexpr (!VODD) {
#pragma unroll
        for (int r = 0; r < 4; ++r) lds_run<VBYTES>(st + L::KBLK + tok[r] * L::VROW + g * VBYTES, v[r]);
      } else {
        // 6-byte runs at 6g lie in the two 4-byte aligned words from (6g & ~3), inside the
        // row (a is only 4-byte aligned: two 32-bit loads); shift them down by 16 bits when
        // g is odd
        const int off = g * VBYTES, a = off & ~3, sh = 8 * (off - a);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          uint32_t w[2];
          lds_run<4>(st + L::KBLK + tok[r] * L::VROW + a, w);
          lds_run<4>(st + L::KBLK + tok[r] * L::VROW + a + 4, w + 1);
          v[r][0] = __funnelshift_r(w[0], w[1], sh);
          v[r][1] = __funnelshift_r(w[1], 0u, sh);
        }
      }
      uint32_t sw[2][1] = {{0u}, {0u}}, rn0 = 0, rn1 = 0, nk0, nk1;
      uint32_t ow[2][2] = {{0u, 0u}, {0u, 0u}};
      if constexpr (QJL) {  // sign bits [32c, 32c + 32) of rows g, g+8; (norm, residual norm)
        lds_run<4>(st + g * L::KROW + L::KCODE + 4 * c, sw[0]);
        lds_run<4>(st + (g + 8) * L::KROW + L::KCODE + 4 * c, sw[1]);
        const uint32_t kn = st + L::KBLK + L::VBLK + 4 * g;
        nk0 = lds_u16(kn);
        rn0 = lds_u16(kn + 2);
        nk1 = lds_u16(kn + 32);
        rn1 = lds_u16(kn + 34);
      } else if constexpr (OUT) {  // (norm, scale) and the eight int8 of tokens g, g+8
        const uint32_t kn = st + L::KBLK + L::VBLK + 12 * g;
        nk0 = lds_u16(kn);
        rn0 = lds_u16(kn + 2);
        lds_run<4>(kn + 4, ow[0]);
        lds_run<4>(kn + 8, ow[0] + 1);
        nk1 = lds_u16(kn + 96);
        rn1 = lds_u16(kn + 98);
        lds_run<4>(kn + 100, ow[1]);
        lds_run<4>(kn + 104, ow[1] + 1);
      } else {
        const uint32_t kn = st + L::KBLK + L::VBLK + 2 * g;
        nk0 = lds_u16(kn);
        nk1 = lds_u16(kn + 16);
      }
      const uint32_t vn = st + L::KBLK + L::VBLK + L::KNORM + 2 * g;
      const uint32_t nv0 = lds_u16(vn), nv1 = lds_u16(vn + 16);
      __syncwarp();  // every lane holds its words: the slot may be refilled
      ++rg.consumed;
      fd.top_up(rg);
      // ---- scores of tokens g and g+8 for head c
      float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 e0 = lut64(field_addr<2 * KB>(k[0], 2 * KB * (2 * ks), klane));
        const uint2 e1 = lut64(field_addr<2 * KB>(k[1], 2 * KB * (2 * ks), klane));
        const uint2 e2 = lut64(field_addr<2 * KB>(k[0], 2 * KB * (2 * ks + 1), klane));
        const uint2 e3 = lut64(field_addr<2 * KB>(k[1], 2 * KB * (2 * ks + 1), klane));
        const uint32_t ah[4] = {e0.x, e1.x, e2.x, e3.x}, al[4] = {e0.y, e1.y, e2.y, e3.y};
        mma16816(sa[0], ah, qf[ks][0], qf[ks][1]);
        mma16816(sa[1], al, qf[ks][0], qf[ks][1]);
      }
      const int tok0 = (pg0 + i) * PS;
      const bool v0 = tok0 + g < t1, v1 = tok0 + g + 8 < t1;
      float x0 = ((sa[0][0] + sa[0][1]) + (sa[1][0] + sa[1][1])) *
                 (__half2float(__ushort_as_half((uint16_t)nk0)) * sscale);
      float x1 = ((sa[0][2] + sa[0][3]) + (sa[1][2] + sa[1][3])) *
                 (__half2float(__ushort_as_half((uint16_t)nk1)) * sscale);
      if constexpr (QJL) {  // sketch term: the +-1 signs are exact in fp16, one mma per k-step
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < SKS; ++ks) {
          const uint2 e0 = lut64(field_addr<2>(sw[0], 2 * (2 * ks), slane));
          const uint2 e1 = lut64(field_addr<2>(sw[1], 2 * (2 * ks), slane));
          const uint2 e2 = lut64(field_addr<2>(sw[0], 2 * (2 * ks + 1), slane));
          const uint2 e3 = lut64(field_addr<2>(sw[1], 2 * (2 * ks + 1), slane));
          const uint32_t az[4] = {e0.x, e1.x, e2.x, e3.x};
          mma16816(ss, az, pf[ks][0], pf[ks][1]);
        }
        x0 = fmaf(ss[0] + ss[1], __half2float(__ushort_as_half((uint16_t)rn0)) * kSketch, x0);
        x1 = fmaf(ss[2] + ss[3], __half2float(__ushort_as_half((uint16_t)rn1)) * kSketch, x1);
      }
      if constexpr (OUT) {  // the eight outlier terms of head c, times each token's scale
        float o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int j = 0; j < KVQ_OUTLIER_CHANNELS; ++j) {
          o0 = fmaf(qo[j], i8f(ow[0][j / 4], j % 4), o0);
          o1 = fmaf(qo[j], i8f(ow[1][j / 4], j % 4), o1);
        }
        x0 = fmaf(o0, __half2float(__ushort_as_half((uint16_t)rn0)), x0);
        x1 = fmaf(o1, __half2float(__ushort_as_half((uint16_t)rn1)), x1);
      }
      x0 = v0 ? x0 : -INFINITY;
      x1 = v1 ? x1 : -INFINITY;
      // ---- online softmax of head c over the 16 tokens
      // the page maximum matters only where a score rises above the running maximum (and
      // for the gate): one vote settles the usual page, whose maximum is below it
      float mt = fmaxf(x0, x1);
      if (p.gate || __any_sync(kFull, mt > m)) {
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
      }
      if (mt > m) {
        const float f = exp2_fast(m - mt);  // m = -inf at first: f = 0
        l *= f;
#pragma unroll
        for (int a = 0; a < KS; ++a)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) acc[a][kk] *= f;
        m = mt;
      }
      const float p0 = v0 ? exp2_fast(x0 - m) : 0.f;
      const float p1 = v1 ? exp2_fast(x1 - m) : 0.f;
      l += p0 + p1;
      if (p.track) {
        float lo = fminf(v0 ? x0 : INFINITY, v1 ? x1 : INFINITY);
        lo = fminf(lo, __shfl_xor_sync(kFull, lo, 4));
        lo = fminf(lo, __shfl_xor_sync(kFull, lo, 8));
        mn = fminf(mn, fminf(lo, __shfl_xor_sync(kFull, lo, 16)));
      }
      // score gate: every token of the page, for every live head, far below its running max
      if (p.gate && __all_sync(kFull, c >= G || mt - m < -kGateLog2)) continue;
      // ---- weight B fragments: column g = (head g/2, part g%2), tokens 2c, 2c+1 | 2c+8, 2c+9
      const float w0 = v0 ? p0 * (__half2float(__ushort_as_half((uint16_t)nv0)) * wscale) : 0.f;
      const float w1 = v1 ? p1 * (__half2float(__ushort_as_half((uint16_t)nv1)) * wscale) : 0.f;
      const uint32_t hi = pack_f16x2(w0, w1);
      const __half2 hh = *reinterpret_cast<const __half2*>(&hi);
      const uint32_t lo = pack_f16x2(w0 - __low2float(hh), w1 - __high2float(hh));
      const uint32_t ah = __shfl_sync(kFull, hi, srcA), al = __shfl_sync(kFull, lo, srcA);
      const uint32_t bh = __shfl_sync(kFull, hi, srcB), bl = __shfl_sync(kFull, lo, srcB);
      const uint32_t A = lo_part ? al : ah, B = lo_part ? bl : bh;
      const uint32_t b0 = live_col ? __byte_perm(A, B, 0x5410) : 0u;
      const uint32_t b1 = live_col ? __byte_perm(A, B, 0x7632) : 0u;
      // ---- values: m-tile mt covers pair slot g*QPT + mt (rows g, g+8: its two
      // coordinates) of tokens 2c, 2c+1 (columns of a0, a1) and 2c+8, 2c+9 (a2, a3)
      uint32_t x01[VW], y01[VW], x89[VW], y89[VW];
      token_pairs<VB, VW>(v[0], v[1], x01, y01);
      token_pairs<VB, VW>(v[2], v[3], x89, y89);
      if constexpr (L::QTAB != 0) {
        // 2-bit values: byte j of a merged run is pair slots 2j, 2j+1, and one quad-table
        // entry holds the (hi, lo) registers of both m-tiles
#pragma unroll
        for (int j = 0; j < KS / 2; ++j) {
          const uint4 r0 = lut128(field_addr<8>(x01, 8 * j, qlane));
          const uint4 r1 = lut128(field_addr<8>(y01, 8 * j, qlane));
          const uint4 r2 = lut128(field_addr<8>(x89, 8 * j, qlane));
          const uint4 r3 = lut128(field_addr<8>(y89, 8 * j, qlane));
          const uint32_t ah0[4] = {r0.x, r1.x, r2.x, r3.x}, al0[4] = {r0.y, r1.y, r2.y, r3.y};
          const uint32_t ah1[4] = {r0.z, r1.z, r2.z, r3.z}, al1[4] = {r0.w, r1.w, r2.w, r3.w};
          mma16816(acc[2 * j], ah0, b0, b1);
          mma16816(acc[2 * j], al0, b0, b1);
          mma16816(acc[2 * j + 1], ah1, b0, b1);
          mma16816(acc[2 * j + 1], al1, b0, b1);
        }
      } else {
#pragma unroll
        for (int mt2 = 0; mt2 < KS; ++mt2) {
          const uint2 r0 = lut64(field_addr<2 * VB>(x01, 2 * VB * mt2, vlane));
          const uint2 r1 = lut64(field_addr<2 * VB>(y01, 2 * VB * mt2, vlane));
          const uint2 r2 = lut64(field_addr<2 * VB>(x89, 2 * VB * mt2, vlane));
          const uint2 r3 = lut64(field_addr<2 * VB>(y89, 2 * VB * mt2, vlane));
          const uint32_t ah4[4] = {r0.x, r1.x, r2.x, r3.x}, al4[4] = {r0.y, r1.y, r2.y, r3.y};
          mma16816(acc[mt2], ah4, b0, b1);
          mma16816(acc[mt2], al4, b0, b1);
        }
      }
    }
    if (rg.lost) {  // a wait gave up: the item contributes nothing (its partial says so)
#pragma unroll
      for (int i = 0; i < KS; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      m = -INFINITY;
      l = 0.f;
      mn = INFINITY;
    }
    // ---- partial of head c: sum over the 8 lanes of the head, coordinates 2*QPT*g ..
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(kFull, l, o);
    if (c < G) {
      const size_t part = ((size_t)b * p.hq + hk * GQ + h0 + c) * p.total_splits + T.split_begin + it.chunk;
      constexpr float unw = 1.0f / (kWScale * kCScale);
      float4* dst = reinterpret_cast<float4*>(p.ws_acc + part * D + 2 * QPT * g);
#pragma unroll
      for (int a = 0; a < KS; a += 2)
        dst[a / 2] = make_float4((acc[a][0] + acc[a][1]) * unw, (acc[a][2] + acc[a][3]) * unw,
                                 (acc[a + 1][0] + acc[a + 1][1]) * unw, (acc[a + 1][2] + acc[a + 1][3]) * unw);
      if (g == 0) {
        p.ws_ml[2 * part] = m;
        p.ws_ml[2 * part + 1] = l;
        if (p.track) p.ws_min[part] = mn;
      }
    }
  }
};

// ================================================================ the kernel
template <class P>
__global__ void __launch_bounds__(P::L::WARPS * 32, 1) decode_cb_kernel(const __grid_constant__ CbParams p) {
  using L = typename P::L;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the table sits at a shared address that is a multiple of its size; warp areas fill the
  // space before it first, then follow it
  const uint32_t base = smem_addr(smem);
  const typename L::Placement pl = L::place(base);
  const uint32_t a_t = pl.t, end = pl.end;  // pair table (the quad table, if any, just before it)
  // A later split-K launch may start on SMs this grid leaves; whatever depends on this
  // grid's completion also sees the launch before it (the wait at the end).
  if (p.trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (end > base + (uint32_t)p.smem_bytes) {  // the launcher sizes smem for any base
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t area = L::area(pl, base, warp);
  Ring rg;
  rg.slots = area;
  rg.bars = area + L::STAGES * L::STAGE + L::QBUF;
  rg.issued = rg.consumed = 0;
  rg.lost = false;
  float* qbuf = reinterpret_cast<float*>(smem + (area + L::STAGES * L::STAGE - base));
  if (lane == 0) {
    for (int s = 0; s < L::STAGES; ++s) mbar_init(rg.bars + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  P::build_tables(p.k_cent, p.v_cent, a_t);
  __syncthreads();
  const uint32_t klane = pin(a_t | ((lane & 15) << 3)), vlane = pin(a_t | 128 | ((lane & 15) << 3));
  // the sketch table sits at a_t + TABLE, a multiple of its 1 KB size
  const uint32_t slane = pin((a_t + L::TABLE) | ((lane & 15) << 3));
  // items: the one in hand, the next (its metadata and queries fetched while this one
  // runs), and the one after (its counter ticket in flight)
  int item = 0, next = 0;
  if (lane == 0) {
    item = atomicAdd(p.counter, 1);
    next = atomicAdd(p.counter, 1);
  }
  item = __shfl_sync(kFull, item, 0);
  next = __shfl_sync(kFull, next, 0);
  Item cur = fetch_item<P::kH8>(p, item < p.total_items ? item : 0, lane);
  while (item < p.total_items) {
    // a warp whose slot wait gave up keeps taking items but writes empty partials for
    // them: every item gets a partial even if every warp gave up
    int after = 0;
    if (lane == 0) after = atomicAdd(p.counter, 1);
    const bool has_next = next < p.total_items;
    Item nx = cur;
    if (has_next) {
      nx = fetch_item<P::kH8>(p, next, lane);
      const uint8_t* qrow =
          reinterpret_cast<const uint8_t*>(p.q + ((size_t)nx.b * p.hq + nx.hk * P::kGQ + nx.h0) * P::kD);
      if (lane < L::QLINES) prefetch_l2(qrow + 128 * lane);
    }
    // after a wait gave up, the items the warp still takes run to an empty partial at once
    if (cur.len > cur.t0) P::run_item(p, cur, has_next, nx, qbuf, rg, klane, vlane, slane, lane);
    item = next;
    next = __shfl_sync(kFull, after, 0);
    cur = nx;
  }
  // a warp that gave up on a slot waits (bounded) for whatever it still has in flight
  if (rg.lost) {
    for (; rg.consumed < rg.issued; ++rg.consumed) {
      const int slot = rg.consumed % L::STAGES;
      const uint32_t parity = (rg.consumed / L::STAGES) & 1;
      for (int n = 0; n < kSpinLimit && !mbar_try_wait(rg.bars + 8 * slot, parity); ++n) {
      }
    }
  }
  // A programmatic dependent (p.pdl) ran alongside the previous split-K grid, whose partials
  // it does not read; it completes only after that grid has, so whatever depends on this
  // grid's completion (the combine) sees every earlier partial.  Without the attribute
  // there is nothing to wait for.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <class P>
cudaError_t launch_path(const CbParams& p, int sms, cudaStream_t stream) {
  using L = typename P::L;
  auto kern = decode_cb_kernel<P>;
  CbParams q = p;
  q.smem_bytes = L::SMEM;
  static std::atomic<bool> configured[64];  // shared-memory limit raised on this device (threads may race: a
                                           // second raise is harmless)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  const int ctas = std::max(1, std::min(sms, (p.total_items + 2 * L::WARPS - 1) / (2 * L::WARPS)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(L::WARPS * 32);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, q);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int D, int G, int KB, int VB, int MODE>
cudaError_t launch_bits(const CbParams& p, int sms, cudaStream_t s) {
  if constexpr (G == 1 && MODE == kModePlain && D == 256) return launch_path<Path1W<D, KB, VB>>(p, sms, s);
  else if constexpr (G == 1) return launch_path<Path1<D, KB, VB, MODE>>(p, sms, s);
  else return launch_path<PathM<D, G, KB, VB, MODE>>(p, sms, s);
}

template <int D, int G, int KB, int MODE>
cudaError_t launch_vb(const CbParams& p, int vb, int sms, cudaStream_t s) {
  switch (vb) {
    case 2: return launch_bits<D, G, KB, 2, MODE>(p, sms, s);
    case 3: return launch_bits<D, G, KB, 3, MODE>(p, sms, s);
    default: return launch_bits<D, G, KB, 4, MODE>(p, sms, s);
  }
}

template <int D, int G, int MODE>
cudaError_t launch_kb(const CbParams& p, int kb, int vb, int sms, cudaStream_t s) {
  switch (kb) {
    case 2: return launch_vb<D, G, 2, MODE>(p, vb, sms, s);
    case 3: return launch_vb<D, G, 3, MODE>(p, vb, sms, s);
    default: return launch_vb<D, G, 4, MODE>(p, vb, sms, s);
  }
}

// A group of 8 runs the 4-head instances, two items per chunk (CbParams::halves).
template <int D, int MODE>
cudaError_t launch_g(const CbParams& p, int g, int kb, int vb, int sms, cudaStream_t s) {
  switch (g) {
    case 1: return launch_kb<D, 1, MODE>(p, kb, vb, sms, s);
    case 2: return launch_kb<D, 2, MODE>(p, kb, vb, sms, s);
    default: return launch_kb<D, 4, MODE>(p, kb, vb, sms, s);
  }
}

// Plain codes with 8 query heads per kv head (head_dim 128 or 256; `wide`: the 16-warp
// instances at head_dim 128): instantiated in decode_cb_g8.cu.
cudaError_t launch_cb_g8(const CbParams& p, int d, bool wide, int kb, int vb, int sms, cudaStream_t s);
// Keys with a residual sketch (head_dim 128): instantiated in decode_cb_qjl.cu.
cudaError_t launch_cb_qjl(const CbParams& p, int g, int kb, int vb, int sms, cudaStream_t s);
// p' = S q' of every query head into p.pq (batch * hkv blocks), before the sketched tiers.
cudaError_t launch_project_qjl(const CbParams& p, int g, int batch, cudaStream_t s);
// Plain codes at head_dim 128 with 2 or 4 query heads per kv head on 16 warps (large
// caches): instantiated in decode_cb_wide.cu.
cudaError_t launch_cb_wide(const CbParams& p, int g, int kb, int vb, int sms, cudaStream_t s);
// Keys with an outlier stream (head_dim 128 or 256): instantiated in decode_cb_outlier.cu.
cudaError_t launch_cb_outlier(const CbParams& p, int d, int g, int kb, int vb, int sms, cudaStream_t s);

}  // namespace cbk
}  // namespace kvq
