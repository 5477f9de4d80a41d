// Quantise-and-append: fp16 K/V vectors -> rotated, encoded rows in the paged pool.
//
// Each thread holds kCoords = 32 coordinates of one vector (D / 32 neighbouring lanes per vector).
// Steps per vector, as on the pages:
//   1. multiply by the Rademacher signs (a flip of the fp16 sign bit), then the
//      Walsh-Hadamard butterflies, all in registers with packed f32x2 adds: five stages on
//      strided runs of the vector, one transpose through shared memory, the remaining
//      log2(D / 32) stages (AdapTQ page, "The Math Fix"; VeloxQuant-MLX page, "Stage 1");
//   2. codebook format: norm of the rotated vector, fp16 norm, u = sqrt(D) y / ||y||, the
//      index of u's centroid cell, little-endian bit packing (VeloxQuant-MLX page, "Stage 2"
//      and "The Bit-Packing Problem"); fp16 / fp8 E4M3 / INT4-g32 formats: the rotated vector
//      rounded to the format (FoveatedKV page, "The VR headset thing");
//   3. store the row at its pool slot.
// One launch for both sides (K and V blocks in grid rows 0 and 1), each row specialised to
// its side's format so a block holds a single short path; a persistent grid walks the
// vectors; the decision table is built once per block.
// The kernel is HBM-bound: 2*D bytes read and one row (+ side data) written per vector.
//
// (Kernel templates and helpers, shared by quantize.cu -- the per-thread kernel for large
// appends -- and quantize_small.cu -- one warp per vector for small ones -- so the two
// compile in parallel.  Everything here has internal linkage: each unit owns the instances
// it launches.)
#pragma once
#include <algorithm>
#include <atomic>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kCoords = 32;      // coordinates of one vector held by one thread
constexpr int kMaxCells = 160;   // decision cells a table holds (more: count the boundaries)
constexpr int kCellCopies = 16;  // lane copies of every cell: the 16 lanes of a half-warp, which
                                 // one 64-bit shared load serves together, hit 16 different
                                 // bank pairs whatever cells they look up
constexpr int kCellBytes = kMaxCells * kCellCopies * 8;  // dynamic shared memory of a block
typedef unsigned long long u64;

// ---------------------------------------------------------------- packed fp32 helpers
__device__ __forceinline__ u64 pk(float a, float b) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(u64 r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
  u64 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 sub2(u64 a, u64 b) {
  u64 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }

// ---------------------------------------------------------------- decision table
// The code index #{i : u > bounds[i]} through cells of width w (a power of two no larger
// than the smallest gap between boundaries, so a cell holds at most one boundary).  With
// t = u / w, the cell is k = rint(t) (cell k covers t in [k - 1/2, k + 1/2)) and
//   index = count[k] + (t > beta[k]),
// count[k] = boundaries below the cell, beta[k] = the boundary inside it (in units of w) or
// +inf.  When t sits exactly between two cells rint may pick either, and both give the same
// index.  |u| <= sqrt(D), so the table spans every reachable cell and needs no clamping.
// The cells {count (int bits), beta} live in the block's dynamic shared memory, cell k's
// kCellCopies copies in one 128-byte row.
struct Table {
  float inv_w;
  int k0, ncells, nb;  // k0 = lowest cell
  int linear;
  uint32_t cells;      // shared address of the cell rows
  float bounds[16];
  float cent[16];      // centroids (the residual sketch needs the decoded values)
};

__device__ void build_table(Table& t, float2* cells, const float* bounds, const float* cent, int nb,
                            int head_dim) {
  // every thread of the block calls this
  if (threadIdx.x < 16) t.bounds[threadIdx.x] = threadIdx.x < nb ? bounds[threadIdx.x] : INFINITY;
  if (threadIdx.x < 16) t.cent[threadIdx.x] = (cent && threadIdx.x <= nb) ? cent[threadIdx.x] : 0.0f;
  __syncthreads();
  float gap = INFINITY;
  for (int i = 0; i + 1 < nb; ++i) gap = fminf(gap, t.bounds[i + 1] - t.bounds[i]);
  bool ok = nb >= 1 && nb <= 15 && (nb == 1 || (gap > 0.0f && gap >= 1e-3f));
  float w = 1.0f;
  if (ok && nb > 1) {
    int e;
    frexpf(gap, &e);
    w = ldexpf(1.0f, e - 1);  // largest power of two <= gap
  }
  const float inv_w = 1.0f / w;  // exact
  const int kmax = (int)ceilf(sqrtf((float)head_dim) * inv_w) + 1;
  const int ncells = 2 * kmax + 1;
  ok = ok && ncells <= kMaxCells;
  for (int i = threadIdx.x; ok && i < ncells * kCellCopies; i += blockDim.x) {
    const int c = i / kCellCopies;
    const float k = (float)(c - kmax);
    const float lo = (k - 0.5f) * w, hi = (k + 0.5f) * w;  // exact: w a power of two
    int cnt = 0;
    float beta = INFINITY;
    for (int b = 0; b < nb; ++b) {
      if (t.bounds[b] < lo) ++cnt;
      else if (t.bounds[b] < hi) beta = t.bounds[b] * inv_w;
    }
    cells[i] = make_float2(__int_as_float(cnt), beta);
  }
  if (threadIdx.x == 0) {
    t.cells = static_cast<uint32_t>(__cvta_generic_to_shared(cells));
    t.inv_w = ok ? inv_w : 1.0f;  // the fallback compares u against the bounds directly
    t.k0 = -kmax;
    t.ncells = ncells;
    t.nb = nb;
    t.linear = ok ? 0 : 1;
  }
  __syncthreads();
}

// 12582912 = 1.5 * 2^23: adding it rounds t (|t| < 2^22) to the integer held in the low
// mantissa bits, 0x4B400000 + rint(t).
constexpr float kMagic = 12582912.0f;
constexpr uint32_t kMagicBits = 0x4B400000u;

// Code indices of coordinates t = y[e] * scale (scale = sqrt(D) / ||y|| / w), packed
// little-endian and stored (E * BITS / 8 bytes at row).
template <int BITS, int E, bool RESIDUAL = false>
__device__ __forceinline__ void encode_codebook(const Table& tb, float (&y)[E], float scale, uint8_t* row,
                                                bool store, float rscale = 0.f, float dscale = 0.f) {
  constexpr int W = E * BITS / 32;
  uint32_t w[W];
#pragma unroll
  for (int k = 0; k < W; ++k) w[k] = 0;
  const u64 sc2 = pk(scale, scale), mg2 = pk(kMagic, kMagic);
  // cell address = row of cell (bits - kMagicBits - k0), the copy of this lane's half-warp
  // position, in 32-bit shared-space arithmetic
  const uint32_t base = tb.cells - 128u * (kMagicBits + static_cast<uint32_t>(tb.k0)) + 8u * (threadIdx.x & 15u);
  const bool lin = tb.linear;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    float t0, t1, f0, f1;
    upk(mul2(pk(y[e], y[e + 1]), sc2), t0, t1);
    upk(add2(pk(t0, t1), mg2), f0, f1);
    uint32_t i0, i1;
    if (!lin) {
      float2 c0, c1;
      asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(c0.x), "=f"(c0.y) : "r"(base + 128u * __float_as_uint(f0)));
      asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(c1.x), "=f"(c1.y) : "r"(base + 128u * __float_as_uint(f1)));
      i0 = __float_as_uint(c0.x) + (t0 > c0.y ? 1u : 0u);
      i1 = __float_as_uint(c1.x) + (t1 > c1.y ? 1u : 0u);
    } else {  // no table: count the boundaries (in units of w = 1)
      i0 = i1 = 0;
      for (int i = 0; i < tb.nb; ++i) {
        i0 += t0 > tb.bounds[i] ? 1u : 0u;
        i1 += t1 > tb.bounds[i] ? 1u : 0u;
      }
    }
    if constexpr (RESIDUAL) {
      // y <- the rotated residual x~ - x^~ = y / sqrt(D) - norm16 C[idx] / sqrt(D)
      y[e] = fmaf(-dscale, tb.cent[i0], y[e] * rscale);
      y[e + 1] = fmaf(-dscale, tb.cent[i1], y[e + 1] * rscale);
    }
    const int o0 = e * BITS, o1 = (e + 1) * BITS;
    w[o0 / 32] += i0 * (1u << (o0 % 32));  // fields are disjoint: add = or
    if ((o0 % 32) + BITS > 32) w[o0 / 32 + 1] += i0 >> (32 - (o0 % 32));
    w[o1 / 32] += i1 * (1u << (o1 % 32));
    if ((o1 % 32) + BITS > 32) w[o1 / 32 + 1] += i1 >> (32 - (o1 % 32));
  }
  if (store) {  // the lane's run is W words at a multiple of its own size (3 words: of 4 bytes)
    if (W % 4 == 0) {
#pragma unroll
      for (int k = 0; k < W / 4; ++k)
        reinterpret_cast<uint4*>(row)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    } else if (W % 2 == 0) {
#pragma unroll
      for (int k = 0; k < W / 2; ++k) reinterpret_cast<uint2*>(row)[k] = make_uint2(w[2 * k], w[2 * k + 1]);
    } else {
#pragma unroll
      for (int k = 0; k < W; ++k) reinterpret_cast<uint32_t*>(row)[k] = w[k];
    }
  }
}

enum { F_CB = 0, F_F16 = 1, F_F8 = 2, F_I4 = 3, F_CBQ = 4, F_CBO = 5 };

// Residual sign sketch of one vector (VeloxQuant-MLX page, "Stage 3: QJL Residual
// Correction"): r holds the lane's kE coordinates of the rotated residual; the bits
// z_j = [ (S r)_j >= 0 ], j < KVQ_QJL_DIM, go to sign[] (valid in every lane of the group).
// The projection rows are read through L1 (every lane group of the block reads the same
// rows).
template <int TPV, int kE>
__device__ __forceinline__ void residual_sketch(const float* __restrict__ proj, const float (&r)[kE], int sub,
                                                unsigned gmask, uint32_t (&sign)[KVQ_QJL_DIM / 32]) {
  constexpr int D = kE * TPV;
#pragma unroll
  for (int k = 0; k < KVQ_QJL_DIM / 32; ++k) sign[k] = 0u;
#pragma unroll 1
  for (int j0 = 0; j0 < KVQ_QJL_DIM; j0 += 8) {
    float dot[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const float4* row = reinterpret_cast<const float4*>(proj + (size_t)(j0 + jj) * D + sub * kE);
      u64 a0 = pk(0.f, 0.f), a1 = pk(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < kE; e += 4) {
        const float4 s4 = __ldg(row + e / 4);
        a0 = fma2(pk(s4.x, s4.y), pk(r[e], r[e + 1]), a0);
        a1 = fma2(pk(s4.z, s4.w), pk(r[e + 2], r[e + 3]), a1);
      }
      float x0, x1, x2, x3;
      upk(a0, x0, x1);
      upk(a1, x2, x3);
      dot[jj] = (x0 + x1) + (x2 + x3);
    }
#pragma unroll
    for (int m = 1; m < TPV; m <<= 1)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) dot[jj] += __shfl_xor_sync(gmask, dot[jj], m, TPV);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      if (dot[jj] >= 0.f) sign[(j0 + jj) / 32] |= 1u << ((j0 + jj) % 32);
  }
}

// ---------------------------------------------------------------- rotation
// The Walsh-Hadamard transform of D = 32 TPV points is a product of one butterfly stage per
// index bit, and the stages commute, so they may run in any order.  Thread `sub` of a
// vector first loads the runs of R = 32 / TPV coordinates at 32k + R sub (k < TPV): its 32
// values then span every value of index bits 0 .. log2(R) - 1 and log2(R) + log2(TPV) .. ,
// i.e. five of the stages run in its registers.  One transpose through shared memory hands
// thread `sub` the 32 neighbouring coordinates [32 sub, 32 sub + 32), which span the
// remaining log2(TPV) bits: their stages run in registers too, and the result sits where the
// encoders expect it.  No cross-lane shuffle is involved.
//
// The transpose area of a vector is D floats in 16-byte chunks, 8 chunks to a 128-byte row
// (row = index bits 5.., chunk column = bits 2..4).  Column c of row r is stored at column
// c ^ swz(r, v) (v: the vector's position in its warp), which keeps both the writes (one row,
// TPV threads) and the reads (TPV rows, one column each) of every quarter-warp on eight
// different 16-byte bank groups.
template <int TPV>
__device__ __forceinline__ uint32_t swz(int row, int v) {
  if constexpr (TPV == 8) return (uint32_t)row;                  // one vector per quarter-warp
  else if constexpr (TPV == 4) return (uint32_t)(row ^ (5 * (v & 1)));  // two
  else return (uint32_t)((4 * row) ^ (v & 3));                   // four (TPV == 2)
}

// Sign bytes of the thread's 32 coordinates, in the order the loads below use (32 bytes:
// run k, offset r at byte k R + r).
template <int TPV>
__device__ __forceinline__ void load_signs(const int8_t* signs_h, int sub, uint32_t (&sw)[8]) {
  constexpr int R = 32 / TPV;
#pragma unroll
  for (int k = 0; k < TPV; ++k) {
    const int8_t* src = signs_h + 32 * k + R * sub;
    if constexpr (R == 4) {
      sw[k] = __ldg(reinterpret_cast<const uint32_t*>(src));
    } else if constexpr (R == 8) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
      sw[2 * k] = u.x;
      sw[2 * k + 1] = u.y;
    } else {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
      sw[4 * k] = u.x;
      sw[4 * k + 1] = u.y;
      sw[4 * k + 2] = u.z;
      sw[4 * k + 3] = u.w;
    }
  }
}

// y = H (s * x) (unnormalised) of one vector: thread `sub` ends with coordinates
// [32 sub, 32 sub + 32) in y.  xv: the vector's fp16 coordinates; area: the vector's shared
// transpose area; vw: the vector's position in its warp.
template <int TPV>
__device__ __forceinline__ void load_rotate(const uint16_t* xv, const uint32_t (&sw)[8], uint32_t area, int sub,
                                            int vw, unsigned gmask, float (&y)[32]) {
  constexpr int R = 32 / TPV;
  uint32_t xw[16];
#pragma unroll
  for (int k = 0; k < TPV; ++k) {
    const uint16_t* src = xv + 32 * k + R * sub;
    if constexpr (R == 4) {
      const uint2 u = __ldcs(reinterpret_cast<const uint2*>(src));
      xw[2 * k] = u.x;
      xw[2 * k + 1] = u.y;
    } else {
#pragma unroll
      for (int i = 0; i < R / 8; ++i) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(src) + i);
        xw[(k * R) / 2 + 4 * i] = u.x;
        xw[(k * R) / 2 + 4 * i + 1] = u.y;
        xw[(k * R) / 2 + 4 * i + 2] = u.z;
        xw[(k * R) / 2 + 4 * i + 3] = u.w;
      }
    }
  }
  // signs: bytes 2j, 2j+1 (int8 +-1, bit 7 set for -1) -> fp16 sign bits 15, 31 of pair j;
  // the first stage (index bit 0, a pair's two halves) in scalar
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t m = __byte_perm(sw[j >> 1], 0, (j & 1) ? 0x3424 : 0x1404) & 0x80008000u;
    const uint32_t xs = xw[j] ^ m;
    const __half2 h2 = *reinterpret_cast<const __half2*>(&xs);
    const float a = __low2float(h2), c = __high2float(h2);
    y[2 * j] = a + c;
    y[2 * j + 1] = a - c;
  }
  // the other four register stages on f32x2 pairs
#pragma unroll
  for (int hs = 2; hs < 32; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      if ((e & hs) == 0) {
        const u64 a = pk(y[e], y[e + 1]), c = pk(y[e + hs], y[e + hs + 1]);
        upk(add2(a, c), y[e], y[e + 1]);
        upk(sub2(a, c), y[e + hs], y[e + hs + 1]);
      }
    }
  }
  // transpose: run k (coordinates 32k + R sub ..) to row k, columns (R/4) sub ..; then read
  // row sub
  __syncwarp(gmask);  // the group's reads of the previous vector are done
#pragma unroll
  for (int k = 0; k < TPV; ++k) {
#pragma unroll
    for (int q = 0; q < R / 4; ++q) {
      const uint32_t col = ((uint32_t)((R / 4) * sub + q)) ^ swz<TPV>(k, vw);
      const int e = k * R + 4 * q;
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(area + 16u * (8u * k + col)), "f"(y[e]),
                   "f"(y[e + 1]), "f"(y[e + 2]), "f"(y[e + 3])
                   : "memory");
    }
  }
  __syncwarp(gmask);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t col = (uint32_t)j ^ swz<TPV>(sub, vw);
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(y[4 * j]), "=f"(y[4 * j + 1]), "=f"(y[4 * j + 2]), "=f"(y[4 * j + 3])
                 : "r"(area + 16u * (8u * sub + col))
                 : "memory");
  }
  // stages of index bits log2(R) .. 4 (the vector's TPV rows)
#pragma unroll
  for (int hs = R; hs < 32; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      if ((e & hs) == 0) {
        const u64 a = pk(y[e], y[e + 1]), c = pk(y[e + hs], y[e + hs + 1]);
        upk(add2(a, c), y[e], y[e + 1]);
        upk(sub2(a, c), y[e + hs], y[e + hs + 1]);
      }
    }
  }
}

// One vector's TPV lanes: y holds coordinates [sub * kE, (sub + 1) * kE) of the rotated
// vector H s x (unnormalised).  Encodes and stores it.
template <int TPV, int kE, int FMT, int BITS>
__device__ __forceinline__ void quantize_vector(const QuantParams& p, const QuantSide& side, const Table& table,
                                                float (&y)[kE], int token, int h, int sub, unsigned gmask) {
  constexpr int D = kE * TPV;
  constexpr float inv_sqrt_d = inv_sqrt_dim(D);
  constexpr float sqrt_d = sqrt_dim(D);
  const int slot = __ldg(p.slots + token);
  const bool store = slot >= 0 && slot < p.num_slots;
  // y = H s x (unnormalised); the rotated vector is x~ = y / sqrt(D)
  const int slot_c = store ? slot : 0;
  const int page = p.page_shift >= 0 ? slot_c >> p.page_shift : slot_c / p.page_size;
  const size_t prow = ((size_t)page * p.hkv + h) * p.page_size + (slot_c - page * p.page_size);
  uint8_t* row = side.rows + prow * side.row_bytes;

  if constexpr (FMT == F_CB || FMT == F_CBQ) {
    u64 acc = pk(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < kE; e += 2) {
      const u64 v2 = pk(y[e], y[e + 1]);
      acc = fma2(v2, v2, acc);
    }
    float a0, a1;
    upk(acc, a0, a1);
    float ss = a0 + a1;
#pragma unroll
    for (int m = 1; m < TPV; m <<= 1) ss += __shfl_xor_sync(gmask, ss, m, TPV);
    const float ny = sqrtf(ss);
    const float inv = ny > 0.0f ? sqrt_d / ny : 0.0f;  // u = sqrt(D) y / ||y||
    const __half norm16 = __float2half_rn(ny * inv_sqrt_d);
    if constexpr (FMT == F_CB) {
      encode_codebook<BITS, kE>(table, y, inv * table.inv_w, row + sub * (kE * BITS / 8), store);
      if (store && sub == 0) side.aux[prow] = norm16;
    } else {
      // codes, and y <- the residual against the decoded vector (stored fp16 norm)
      encode_codebook<BITS, kE, true>(table, y, inv * table.inv_w, row + sub * (kE * BITS / 8), store, inv_sqrt_d,
                                      __half2float(norm16) * inv_sqrt_d);
      u64 racc = pk(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < kE; e += 2) {
        const u64 v2 = pk(y[e], y[e + 1]);
        racc = fma2(v2, v2, racc);
      }
      float r0, r1;
      upk(racc, r0, r1);
      float rs = r0 + r1;
#pragma unroll
      for (int m = 1; m < TPV; m <<= 1) rs += __shfl_xor_sync(gmask, rs, m, TPV);
      uint32_t sign[KVQ_QJL_DIM / 32];
      residual_sketch<TPV, kE>(side.qjl, y, sub, gmask, sign);
      if (store && sub == 0) {
        uint4* dst = reinterpret_cast<uint4*>(row + D * BITS / 8);
        *dst = make_uint4(sign[0], sign[1], sign[2], sign[3]);
        const __half2 nr = __halves2half2(norm16, __float2half_rn(sqrtf(rs)));
        reinterpret_cast<__half2*>(side.aux)[prow] = nr;
      }
    }
  } else if constexpr (FMT == F_F16) {
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(row) + sub * (kE / 8);
#pragma unroll
      for (int k = 0; k < kE / 8; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 h2 = __floats2half2_rn(y[8 * k + 2 * j] * inv_sqrt_d, y[8 * k + 2 * j + 1] * inv_sqrt_d);
          w[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else if constexpr (FMT == F_F8) {
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(row) + sub * (kE / 16);
#pragma unroll
      for (int k = 0; k < kE / 16; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 16 * k + 4 * j;
          const uint32_t a = float2_to_fp8x2(y[e] * inv_sqrt_d, y[e + 1] * inv_sqrt_d);
          const uint32_t b = float2_to_fp8x2(y[e + 2] * inv_sqrt_d, y[e + 3] * inv_sqrt_d);
          w[j] = a | (b << 16);
        }
        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {  // F_I4: kE / 32 groups of 32 coordinates per thread
    constexpr int NG = kE / kGroup;
    uint32_t w[NG * 4];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < kGroup; ++e) amax = fmaxf(amax, fabsf(y[kGroup * g + e] * inv_sqrt_d));
      const __half s16 = __float2half_rn(amax / 7.0f);
      const float s = __half2float(s16);
      const float r = s > 0.0f ? 1.0f / s : 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) w[4 * g + k] = 0;
#pragma unroll
      for (int e = 0; e < kGroup; ++e) {
        const float xv = y[kGroup * g + e] * inv_sqrt_d;
        // level = rint(x / s): x * (1/s) is within one ulp of the quotient; where that
        // leaves the result next to a half-integer, divide exactly
        float tq = xv * r;
        if (s > 0.0f && fabsf(fabsf(tq - rintf(tq)) - 0.5f) < 1e-5f) tq = xv / s;
        const float q = s > 0.0f ? fminf(fmaxf(rintf(tq), -7.0f), 7.0f) : 0.0f;
        w[4 * g + e / 8] |= (uint32_t)((int)q + 8) << (4 * (e % 8));
      }
      if (store) side.aux[prow * (D / kGroup) + sub * NG + g] = s16;
    }
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(row) + sub * NG;
#pragma unroll
      for (int k = 0; k < NG; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
  }
}

// Appends of at most this many vectors per side take the warp-per-vector kernel.
constexpr long long kSmallMaxVectors = 1 << 14;

// Every vector of one side (kind) that falls to this block (grid-stride over vectors).
template <int TPV, int FMT, int BITS>
__device__ __forceinline__ void quantize_side(const QuantParams& p, int kind, Table& table, float2* cells,
                                              uint32_t xpose) {
  constexpr int kE = kCoords, D = kE * TPV, VPB = kThreads / TPV;
  const QuantSide& side = p.side[kind];
  if constexpr (FMT == F_CB || FMT == F_CBQ)
    build_table(table, cells, side.bounds, side.centroids, (1 << BITS) - 1, D);
  const int lane = threadIdx.x & 31, sub = lane % TPV, vw = lane / TPV;
  const unsigned gmask = (TPV == 32 ? 0xFFFFFFFFu : ((1u << TPV) - 1u)) << (lane - sub);
  const uint32_t area = xpose + (uint32_t)(threadIdx.x / TPV) * (D * 4);
  const int nvec = p.num_tokens * p.hkv;
  const int stride = gridDim.x * VPB;
  const uint16_t* x = p.x[kind];
  // with a stride that is a multiple of the kv heads the head stays fixed and the token
  // advances by stride / hkv: no division in the loop
  const bool fixed = stride % p.hkv == 0;
  const int v0 = blockIdx.x * VPB + threadIdx.x / TPV, dt = stride / p.hkv;
  int token = v0 / p.hkv, h = v0 - token * p.hkv;
  for (int v = v0; v < nvec; v += stride) {
    if (!fixed) {
      token = v / p.hkv;
      h = v - token * p.hkv;
    }
    // the thread's part of its next vector heads for L2 while this one is worked on
    if (v + stride < nvec) prefetch_l2(x + (size_t)(v + stride) * D + sub * kE);
    uint32_t sw[8];  // (reloaded per vector, from L1: holding them across the loop spills)
    load_signs<TPV>(side.signs + (size_t)h * D, sub, sw);
    float y[kE];
    load_rotate<TPV>(x + (size_t)v * D, sw, area, sub, vw, gmask, y);
    quantize_vector<TPV, kE, FMT, BITS>(p, side, table, y, token, h, sub, gmask);
    token += dt;
  }
}

// Resident blocks per SM: 4 (64 registers a thread) where the format's path fits them
// without spills, else 3 (85 registers: the residual sketch, INT4 groups).
constexpr int blocks_per_sm(int f0, int f1) {
  return (f0 == F_CBQ || f0 == F_I4 || f1 == F_CBQ || f1 == F_I4) ? 3 : 4;
}

// Side slot blockIdx.y: (F0, B0) for slot 0, (F1, B1) for slot 1; kind = kind_first + slot.
// Dynamic shared memory of a block: the decision cells (when a side is coded), then the
// transpose areas of its vectors (32 floats a thread).
constexpr int kXposeBytes = kThreads * kCoords * 4;
template <int F0, int F1>
__host__ __device__ constexpr int quant_smem() {
  return ((F0 == F_CB || F0 == F_CBQ || F1 == F_CB || F1 == F_CBQ) ? kCellBytes : 0) + kXposeBytes;
}

template <int TPV, int F0, int B0, int F1, int B1>
__global__ void __launch_bounds__(kThreads, blocks_per_sm(F0, F1)) quantize_kernel(const QuantParams p) {
  __shared__ Table table;
  extern __shared__ __align__(16) float2 cells[];
  const uint32_t xpose =
      static_cast<uint32_t>(__cvta_generic_to_shared(cells)) + (uint32_t)(quant_smem<F0, F1>() - kXposeBytes);
  if (blockIdx.y == 0) quantize_side<TPV, F0, B0>(p, p.kind_first, table, cells, xpose);
  else quantize_side<TPV, F1, B1>(p, p.kind_first + 1, table, cells, xpose);
}

template <int TPV, int F0, int B0, int F1, int B1>
cudaError_t launch_q(const QuantParams& p, int sides, int sms, cudaStream_t stream) {
  constexpr int VPB = kThreads / TPV;
  constexpr int smem = quant_smem<F0, F1>();
  auto kern = quantize_kernel<TPV, F0, B0, F1, B1>;
  static std::atomic<bool> configured[64];  // shared-memory limit raised on this device (a racing
                                           // second raise is harmless)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  const long long nvec = (long long)p.num_tokens * p.hkv;
  const long long need = (nvec + VPB - 1) / VPB;
  long long blocks = std::max<long long>(1, std::min<long long>(need, (long long)sms * blocks_per_sm(F0, F1) / sides));
  // a grid stride (blocks * VPB vectors) that is a multiple of the kv heads keeps every
  // thread on one head, so it loads that head's signs once
  long long per = p.hkv;
  for (long long a = VPB, b = per; b;) {  // per = hkv / gcd(VPB, hkv)
    const long long t = a % b;
    a = b;
    b = t;
    if (!b) per = p.hkv / a;
  }
  if (blocks >= per) blocks = blocks / per * per;
  kern<<<dim3((unsigned)blocks, sides), kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int TPV, int F0, int B0>
cudaError_t launch_single(const QuantParams& p, int sms, cudaStream_t stream) {
  return launch_q<TPV, F0, B0, F0, B0>(p, 1, sms, stream);
}

}  // namespace

// Small appends, every format: one warp per vector (quantize_small.cu).
cudaError_t launch_quantize_small(const QuantParams& p, int head_dim, int sms, cudaStream_t stream);

}  // namespace kvq
