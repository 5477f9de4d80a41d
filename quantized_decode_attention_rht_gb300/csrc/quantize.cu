// Quantise-and-append: fp16 K/V vectors -> rotated, encoded rows in the paged pool.
//
// One vector (token, kv head, K|V) is held by LPV = D/32 consecutive lanes, 32 contiguous
// coordinates per lane.  Steps per vector, as on the pages:
//   1. multiply by the Rademacher signs, then the Walsh-Hadamard butterflies -- five
//      in-register stages over a lane's 32 coordinates and log2(LPV) stages across lanes
//      with shuffles (AdapTQ page, "The Math Fix"; VeloxQuant-MLX page, "Stage 1");
//   2. codebook format: norm of the rotated vector, fp16 norm, u = sqrt(D) y / ||y||, index
//      of the centroid cell of every coordinate, little-endian bit packing (VeloxQuant-MLX
//      page, "Stage 2" and "The Bit-Packing Problem");
//      fp16 / fp8 E4M3 / INT4-g32 formats: the rotated vector rounded to the format
//      (FoveatedKV page, "The VR headset thing");
//   3. store the row at its pool slot.
// The kernel is HBM-bound: 2*D bytes read and one row (+ side data) written per vector.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxCells = 256;

// Decision grid for the codebook index #{i : u > bounds[i]}: cells of width w (a power of
// two no larger than the smallest gap between boundaries) hold at most one boundary, so
// idx = count[cell] + (u > beta[cell]).  floor(u / w) is exact for a power-of-two w.
struct Grid {
  int cell_lo, ncells, nb;
  float inv_w;
  bool linear;  // fall back to counting when the grid would be too large
  float bounds[255];
  int count[kMaxCells];
  float beta[kMaxCells];
};

__device__ void build_grid(Grid& g, const float* bounds, int nb) {
  // single thread; nb <= 15 in practice
  g.nb = nb;
  for (int i = 0; i < nb; ++i) g.bounds[i] = bounds[i];
  float gap = INFINITY;
  for (int i = 0; i + 1 < nb; ++i) gap = fminf(gap, g.bounds[i + 1] - g.bounds[i]);
  g.linear = true;
  if (nb < 1) return;
  float w = 1.0f;
  if (nb > 1) {
    if (!(gap > 0.0f) || gap < 1e-3f) return;
    int e;
    frexpf(gap, &e);          // gap = m * 2^e, m in [0.5, 1)
    w = ldexpf(1.0f, e - 1);  // largest power of two <= gap
  }
  const float inv_w = 1.0f / w;  // exact: power of two
  const int lo = (int)floorf(g.bounds[0] * inv_w);
  const int hi = (int)floorf(g.bounds[nb - 1] * inv_w);
  if (hi - lo + 1 > kMaxCells) return;
  g.cell_lo = lo;
  g.ncells = hi - lo + 1;
  g.inv_w = inv_w;
  for (int c = 0; c < g.ncells; ++c) {
    const float a = (float)(lo + c) * w, b = (float)(lo + c + 1) * w;
    int cnt = 0;
    float beta = INFINITY;
    for (int i = 0; i < nb; ++i) {
      if (g.bounds[i] < a) ++cnt;
      else if (g.bounds[i] < b) beta = g.bounds[i];
    }
    g.count[c] = cnt;
    g.beta[c] = beta;
  }
  g.linear = false;
}

__device__ __forceinline__ uint32_t code_index(const Grid& g, float u) {
  if (g.linear) {
    uint32_t idx = 0;
    for (int i = 0; i < g.nb; ++i) idx += (u > g.bounds[i]) ? 1u : 0u;
    return idx;
  }
  const int c = (int)floorf(u * g.inv_w) - g.cell_lo;
  if (c < 0) return 0;
  if (c >= g.ncells) return (uint32_t)g.nb;
  return (uint32_t)g.count[c] + ((u > g.beta[c]) ? 1u : 0u);
}

// Pack 32 codes of B bits into B little-endian words.
template <int B>
__device__ __forceinline__ void pack32(const uint32_t (&idx)[32], uint32_t (&w)[B]) {
#pragma unroll
  for (int k = 0; k < B; ++k) w[k] = 0;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int o = e * B;
    w[o / 32] |= idx[e] << (o % 32);
    if ((o % 32) + B > 32) w[o / 32 + 1] |= idx[e] >> (32 - (o % 32));
  }
}

template <int LPV>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const QuantParams p) {
  constexpr int D = 32 * LPV;
  __shared__ Grid grids[2];
  if (threadIdx.x < 2) {
    const int kind = threadIdx.x;
    const QuantSide& s = p.side[kind];
    grids[kind].linear = true;
    grids[kind].nb = 0;
    if (s.fmt == KVQ_FMT_CODEBOOK && s.bounds) build_grid(grids[kind], s.bounds, (1 << s.bits) - 1);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int r = lane % LPV;                                   // lane within the vector
  const unsigned gmask = ((LPV == 32) ? 0xFFFFFFFFu : ((1u << LPV) - 1u)) << (lane - r);
  const long long v = (long long)blockIdx.x * (kThreads / LPV) + threadIdx.x / LPV;
  const bool in_range = v < p.num_vectors;
  const long long per_kind = (long long)p.num_tokens * p.hkv;
  const int kind = p.kind_first + (in_range ? (int)(v / per_kind) : 0);
  const long long rem = in_range ? v % per_kind : 0;
  const int token = (int)(rem / p.hkv);
  const int h = (int)(rem % p.hkv);
  const QuantSide& side = p.side[kind];
  const int slot = in_range ? p.slots[token] : -1;
  const bool store = in_range && slot >= 0 && slot < p.num_slots;

  // ---- load 32 fp16 coordinates and the signs; y = s * x
  float y[32];
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.x[kind] + ((size_t)token * p.hkv + h) * D + r * 32);
    const uint4* sg = reinterpret_cast<const uint4*>(side.signs + (size_t)h * D + r * 32);
    uint4 xs[4], ss[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) xs[i] = in_range ? src[i] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 2; ++i) ss[i] = in_range ? sg[i] : make_uint4(0, 0, 0, 0);
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs);
    const int8_t* sb = reinterpret_cast<const int8_t*>(ss);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const uint16_t bits = (uint16_t)(xw[e / 2] >> (16 * (e % 2)));
      const float f = __half2float(__ushort_as_half(bits));
      y[e] = sb[e] < 0 ? -f : f;
    }
  }
  // ---- Walsh-Hadamard butterflies: in-register stages, then across lanes
#pragma unroll
  for (int hs = 1; hs < 32; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      if ((e & hs) == 0) {
        const float a = y[e], b = y[e + hs];
        y[e] = a + b;
        y[e + hs] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < LPV; m <<= 1) {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float o = __shfl_xor_sync(gmask, y[e], m, LPV);
      y[e] = (r & m) ? (o - y[e]) : (y[e] + o);
    }
  }
  // y = H s x (unnormalised); the rotated vector is x~ = y / sqrt(D)
  constexpr float inv_sqrt_d = (D == 256) ? 0.0625f : 0.08838834764831845f;
  constexpr float sqrt_d = (D == 256) ? 16.0f : 11.313708498984760f;

  uint8_t* row = side.rows + ((size_t)(slot / p.page_size) * p.hkv + h) * (size_t)p.page_size * side.row_bytes +
                 (size_t)(slot % p.page_size) * side.row_bytes;
  const size_t aux_row = ((size_t)(slot / p.page_size) * p.hkv + h) * p.page_size + (slot % p.page_size);

  if (side.fmt == KVQ_FMT_CODEBOOK) {
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) ss += __shfl_xor_sync(gmask, ss, m, LPV);
    const float ny = sqrtf(ss);
    const float inv = ny > 0.0f ? sqrt_d / ny : 0.0f;  // u = sqrt(D) y / ||y||
    const Grid& g = grids[kind];
    uint32_t idx[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) idx[e] = code_index(g, y[e] * inv);
    if (store) {
      if (r == 0) side.aux[aux_row] = __float2half_rn(ny * inv_sqrt_d);
      if (side.bits == 4) {
        uint32_t w[4];
        pack32<4>(idx, w);
        reinterpret_cast<uint4*>(row)[r] = make_uint4(w[0], w[1], w[2], w[3]);
      } else if (side.bits == 3) {
        uint32_t w[3];
        pack32<3>(idx, w);
        uint32_t* dst = reinterpret_cast<uint32_t*>(row) + 3 * r;
        dst[0] = w[0]; dst[1] = w[1]; dst[2] = w[2];
      } else {
        uint32_t w[2];
        pack32<2>(idx, w);
        reinterpret_cast<uint2*>(row)[r] = make_uint2(w[0], w[1]);
      }
    }
  } else if (side.fmt == KVQ_FMT_FP16) {
    if (store) {
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint32_t lo = __half_as_ushort(__float2half_rn(y[2 * k] * inv_sqrt_d));
        const uint32_t hi = __half_as_ushort(__float2half_rn(y[2 * k + 1] * inv_sqrt_d));
        w[k] = lo | (hi << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(row) + 4 * r;
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  } else if (side.fmt == KVQ_FMT_FP8_E4M3) {
    if (store) {
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t a = float2_to_fp8x2(y[4 * k] * inv_sqrt_d, y[4 * k + 1] * inv_sqrt_d);
        const uint32_t b = float2_to_fp8x2(y[4 * k + 2] * inv_sqrt_d, y[4 * k + 3] * inv_sqrt_d);
        w[k] = a | (b << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(row) + 2 * r;
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  } else {  // KVQ_FMT_INT4_G32: the lane's 32 coordinates are one group
    float x[32];
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      x[e] = y[e] * inv_sqrt_d;
      amax = fmaxf(amax, fabsf(x[e]));
    }
    const __half s16 = __float2half_rn(amax / 7.0f);
    const float s = __half2float(s16);
    uint32_t idx[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float q = s > 0.0f ? fminf(fmaxf(rintf(x[e] / s), -7.0f), 7.0f) : 0.0f;
      idx[e] = (uint32_t)((int)q + 8);
    }
    if (store) {
      uint32_t w[4];
      pack32<4>(idx, w);
      reinterpret_cast<uint4*>(row)[r] = make_uint4(w[0], w[1], w[2], w[3]);
      side.aux[aux_row * (D / kGroup) + r] = s16;
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const QuantParams& p, int head_dim, cudaStream_t stream) {
  if (p.num_vectors == 0) return cudaSuccess;
  const int lpv = head_dim / 32;
  const long long vpb = kThreads / lpv;
  const long long blocks = (p.num_vectors + vpb - 1) / vpb;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (lpv == 4) quantize_kernel<4><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  else if (lpv == 8) quantize_kernel<8><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace kvq
