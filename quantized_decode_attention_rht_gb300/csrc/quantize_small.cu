// Quantise-and-append for small appends (a decode step's new token of every sequence): one
// warp per vector, D / 32 neighbouring coordinates per lane (D = 64, 128 or 256).
//
// The per-thread kernel of quantize.cuh keeps 32 coordinates of a vector in one thread's
// registers, which is what a prefill chunk of millions of vectors wants; a few hundred
// vectors then occupy a handful of SMs whose warps wait on one long, cold instruction
// stream (and, for keys with a residual sketch, on 16 K multiply-adds per thread).  Here a
// vector's work is spread over a warp: the rotation takes log2(D / 32) register stages and
// five shuffle stages, the norms are warp sums, the codes are packed through a per-warp
// shared buffer, and the residual sketch is a coalesced pass over the projection rows with
// a reduce-scatter.  Same steps, same stored bytes, and the same float32 decisions as the
// per-thread kernel (VeloxQuant-MLX page, "Stage 1", "Stage 2", "Stage 3" and "The
// Bit-Packing Problem"; FoveatedKV page, "The VR headset thing").
#include "quantize.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 8;  // warps (vectors in flight) per block

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, m);
  return x;  // fp32 addition commutes: every lane ends with the same value
}

// y = H (s * x) (unnormalised) for the lane's coordinates [lane * E, lane * E + E).
template <int E>
__device__ __forceinline__ void load_rotate(const uint16_t* src, const int8_t* sg, int lane, float (&y)[E]) {
  uint32_t xw[E / 2], sw[(E + 3) / 4];
  if constexpr (E == 2) {
    xw[0] = __ldg(reinterpret_cast<const uint32_t*>(src) + lane);
    sw[0] = __ldg(reinterpret_cast<const uint16_t*>(sg) + lane);
  } else if constexpr (E == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src) + lane);
    xw[0] = u.x;
    xw[1] = u.y;
    sw[0] = __ldg(reinterpret_cast<const uint32_t*>(sg) + lane);
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    xw[0] = u.x;
    xw[1] = u.y;
    xw[2] = u.z;
    xw[3] = u.w;
    const uint2 s2 = __ldg(reinterpret_cast<const uint2*>(sg) + lane);
    sw[0] = s2.x;
    sw[1] = s2.y;
  }
#pragma unroll
  for (int k = 0; k < E / 2; ++k) {
    // sign bytes 2k, 2k+1 (int8 +-1: bit 7 set for -1) -> fp16 sign bits 15, 31
    const uint32_t m = __byte_perm(sw[k >> 1], 0, (k & 1) ? 0x3424 : 0x1404) & 0x80008000u;
    const uint32_t xv = xw[k] ^ m;
    const __half2 h2 = *reinterpret_cast<const __half2*>(&xv);
    y[2 * k] = __low2float(h2);
    y[2 * k + 1] = __high2float(h2);
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
    const float sgn = (lane & m) ? -1.0f : 1.0f;  // upper lane keeps partner - own
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = fmaf(sgn, y[e], __shfl_xor_sync(0xFFFFFFFFu, y[e], m));
  }
}

// Keys with an outlier stream (VeloxQuant-MLX page, "Outlier Two-Stream Cache"): the
// lane's coordinates of x (unrotated, fp16 -> fp32) with the head's outlier channels c_j
// set to zero; xo[j] = x[c_j] in every lane.  Then y = H (s * x_inlier).
template <int E>
__device__ __forceinline__ void load_split_rotate(const uint16_t* src, const int8_t* sg, const int32_t* outl, int lane,
                                                  float (&y)[E], float (&xo)[KVQ_OUTLIER_CHANNELS]) {
  uint32_t xw[E / 2];
  if constexpr (E == 2) {
    xw[0] = __ldg(reinterpret_cast<const uint32_t*>(src) + lane);
  } else if constexpr (E == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src) + lane);
    xw[0] = u.x;
    xw[1] = u.y;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    xw[0] = u.x;
    xw[1] = u.y;
    xw[2] = u.z;
    xw[3] = u.w;
  }
#pragma unroll
  for (int k = 0; k < E / 2; ++k) {
    const __half2 h2 = *reinterpret_cast<const __half2*>(&xw[k]);
    y[2 * k] = __low2float(h2);
    y[2 * k + 1] = __high2float(h2);
  }
  const int4 c0 = __ldg(reinterpret_cast<const int4*>(outl)), c1 = __ldg(reinterpret_cast<const int4*>(outl) + 1);
  const int ch[KVQ_OUTLIER_CHANNELS] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int j = 0; j < KVQ_OUTLIER_CHANNELS; ++j) {
    float mine = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (lane * E + e == ch[j]) {
        mine = y[e];
        y[e] = 0.f;
      }
    }
    xo[j] = __shfl_sync(0xFFFFFFFFu, mine, (ch[j] / E) & 31);
  }
  alignas(8) int8_t s8[E < 4 ? 4 : E];
  if constexpr (E == 2) {
    *reinterpret_cast<uint16_t*>(s8) = __ldg(reinterpret_cast<const uint16_t*>(sg) + lane);
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint32_t*>(s8) = __ldg(reinterpret_cast<const uint32_t*>(sg) + lane);
  } else {
    *reinterpret_cast<uint2*>(s8) = __ldg(reinterpret_cast<const uint2*>(sg) + lane);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) y[e] = s8[e] < 0 ? -y[e] : y[e];
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
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = fmaf(sgn, y[e], __shfl_xor_sync(0xFFFFFFFFu, y[e], m));
  }
}

// y = x~ for the lane's coordinates, from a stored fp16 row of the rotated vector.
template <int E>
__device__ __forceinline__ void load_row(const uint8_t* row, int lane, float (&y)[E]) {
  uint32_t xw[E / 2];
  if constexpr (E == 2) {
    xw[0] = *reinterpret_cast<const uint32_t*>(row + 4 * lane);
  } else if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + 8 * lane);
    xw[0] = u.x;
    xw[1] = u.y;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(row + 16 * lane);
    xw[0] = u.x;
    xw[1] = u.y;
    xw[2] = u.z;
    xw[3] = u.w;
  }
#pragma unroll
  for (int k = 0; k < E / 2; ++k) {
    const __half2 h2 = *reinterpret_cast<const __half2*>(&xw[k]);
    y[2 * k] = __low2float(h2);
    y[2 * k + 1] = __high2float(h2);
  }
}

// The lane's E fields of `bits` bits each (coordinate order) into the row's little-endian
// bit stream; `buf` is the warp's shared staging area (D * bits / 32 words).
template <int D, int E, int BITS>
__device__ __forceinline__ void store_fields(uint32_t* buf, uint32_t fields, uint8_t* row, int lane) {
  constexpr int W = D * BITS / 32;
  __syncwarp();  // the previous vector's words have been read
  if (lane < W) buf[lane] = 0u;
  __syncwarp();
  const int off = lane * E * BITS, w0 = off / 32, sh = off % 32;
  atomicOr(buf + w0, fields << sh);
  if (sh + E * BITS > 32) atomicOr(buf + w0 + 1, fields >> (32 - sh));
  __syncwarp();
  if constexpr (W % 4 == 0) {
    if (lane < W / 4) reinterpret_cast<uint4*>(row)[lane] = reinterpret_cast<const uint4*>(buf)[lane];
  } else {  // 3-bit rows at D = 64: 24 bytes, 8-byte aligned
    static_assert(W % 2 == 0, "rows are whole 8-byte units");
    if (lane < W / 2) reinterpret_cast<uint2*>(row)[lane] = reinterpret_cast<const uint2*>(buf)[lane];
  }
}

// Residual sign sketch: word k of z_j = [ (S r)_j >= 0 ], rows j in [32k, 32k + 32).  The
// lane's partial dot products of the 32 rows are reduce-scattered over the warp so lane l
// ends with row 32k + l, and a ballot gathers the signs.  (A key's four words come from
// four warps: a decode step's few hundred keys then spread over four times the warps.)
template <int D, int E>
__device__ __forceinline__ uint32_t sketch_word(const float* __restrict__ proj, const float (&r)[E], int lane, int k) {
  {
    float a[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const float4* srow = reinterpret_cast<const float4*>(proj + (size_t)(32 * k + t) * D + lane * E);
      float s = 0.f;
      if constexpr (E == 2) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(srow));
        s = fmaf(v.y, r[1], v.x * r[0]);
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
          const float4 v = __ldg(srow + q);
          s = fmaf(v.x, r[4 * q], s);
          s = fmaf(v.y, r[4 * q + 1], s);
          s = fmaf(v.z, r[4 * q + 2], s);
          s = fmaf(v.w, r[4 * q + 3], s);
        }
      }
      a[t] = s;
    }
#pragma unroll
    for (int s2 = 0; s2 < 5; ++s2) {
      const int msk = 16 >> s2, n = 32 >> s2;
      const bool up = lane & msk;
#pragma unroll
      for (int q = 0; q < n / 2; ++q) {
        const float send = up ? a[q] : a[q + n / 2];
        const float keep = up ? a[q + n / 2] : a[q];
        a[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, msk);
      }
    }
    return __ballot_sync(0xFFFFFFFFu, a[0] >= 0.f);
  }
}

// FROM_ROWS: the vectors are stored fp16 rows of x~ (src, re-encode) rather than new fp16
// inputs x to rotate.  y is H s x (= sqrt(D) x~) for new inputs and x~ itself for stored
// rows; ys maps y to x~.  Codes and the norm direction do not depend on the scale of y.
template <int D, int FMT, int BITS, bool FROM_ROWS>
__device__ __forceinline__ void append_side(const QuantParams& p, const QuantSide& side, const uint16_t* x,
                                            const uint8_t* src, uint32_t* buf) {
  constexpr int E = D / 32;
  constexpr float inv_sqrt_d = inv_sqrt_dim(D);
  constexpr float sqrt_d = sqrt_dim(D);
  constexpr float ys = FROM_ROWS ? 1.0f : inv_sqrt_d;
  constexpr bool CB = FMT == F_CB || FMT == F_CBQ || FMT == F_CBO;
  constexpr int NB = CB ? (1 << BITS) - 1 : 1;
  const int lane = threadIdx.x & 31;
  float bnd[NB];
  if constexpr (CB) {
#pragma unroll
    for (int i = 0; i < NB; ++i) bnd[i] = __ldg(side.bounds + i);
  }
  // keys with a residual sketch: four work units per key, unit u computing sketch word u
  // (each unit repeats the key's short encode; unit 0 stores the codes and norms)
  constexpr int UNITS = FMT == F_CBQ ? KVQ_QJL_DIM / 32 : 1;
  const int nunits = p.num_tokens * p.hkv * UNITS;
  for (int u = blockIdx.x * kWarps + (threadIdx.x >> 5); u < nunits; u += gridDim.x * kWarps) {
    const int v = u / UNITS, part = u - v * UNITS;
    const int token = v / p.hkv, h = v - token * p.hkv;
    const int slot = p.slots[token];
    if (slot < 0 || slot >= p.num_slots) continue;  // warp-uniform
    float y[E], xo[KVQ_OUTLIER_CHANNELS];
    if constexpr (FMT == F_CBO) {
      load_split_rotate<E>(x + (size_t)v * D, side.signs + (size_t)h * D, side.outl + h * KVQ_OUTLIER_CHANNELS,
                           lane, y, xo);
    } else if constexpr (FROM_ROWS) {
      const int ss = p.src_slots[token];
      if (ss < 0 || ss >= p.src_num_slots) continue;
      const size_t srow = ((size_t)(ss / p.page_size) * p.hkv + h) * p.page_size + (ss % p.page_size);
      load_row<E>(src + srow * (2 * D), lane, y);
    } else {
      load_rotate<E>(x + (size_t)v * D, side.signs + (size_t)h * D, lane, y);
    }
    const size_t prow = ((size_t)(slot / p.page_size) * p.hkv + h) * p.page_size + (slot % p.page_size);
    uint8_t* row = side.rows + prow * side.row_bytes;
    if constexpr (CB) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) ss = fmaf(y[e], y[e], ss);
      const float ny = sqrtf(warp_sum(ss));
      const float inv = ny > 0.0f ? sqrt_d / ny : 0.0f;  // u = sqrt(D) y / ||y||
      const __half norm16 = __float2half_rn(ny * ys);
      uint32_t fields = 0u;
      int idx[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float u = y[e] * inv;
        int c = 0;
#pragma unroll
        for (int i = 0; i < NB; ++i) c += u > bnd[i] ? 1 : 0;
        idx[e] = c;
        fields |= (uint32_t)c << (e * BITS);
      }
      if (part == 0) store_fields<D, E, BITS>(buf, fields, row, lane);  // warp-uniform
      if constexpr (FMT == F_CB) {
        if (lane == 0) side.aux[prow] = norm16;
      } else if constexpr (FMT == F_CBO) {
        // the outlier stream: int8 with a per-token scale s = fp16(max |x_cj| / 127)
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < KVQ_OUTLIER_CHANNELS; ++j) amax = fmaxf(amax, fabsf(xo[j]));
        const __half s16 = __float2half_rn(amax / 127.0f);
        const float sc = __half2float(s16);
        uint32_t qw[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < KVQ_OUTLIER_CHANNELS; ++j) {
          const float qv = sc > 0.f ? fminf(fmaxf(rintf(xo[j] / sc), -127.f), 127.f) : 0.f;
          qw[j / 4] |= ((uint32_t)(int)qv & 0xFFu) << (8 * (j % 4));
        }
        if (lane == 0) {
          uint32_t* rec = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(side.aux) +
                                                      prow * (4 + KVQ_OUTLIER_CHANNELS));
          rec[0] = (uint32_t)__half_as_ushort(norm16) | ((uint32_t)__half_as_ushort(s16) << 16);
          rec[1] = qw[0];
          rec[2] = qw[1];
        }
      } else {
        // y <- the rotated residual x~ - x^~ against the decoded vector (stored fp16 norm)
        const float dscale = __half2float(norm16) * inv_sqrt_d;
        float rs = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          y[e] = fmaf(-dscale, __ldg(side.centroids + idx[e]), y[e] * ys);
          rs = fmaf(y[e], y[e], rs);
        }
        const float rn = sqrtf(warp_sum(rs));
        const uint32_t z = sketch_word<D, E>(side.qjl, y, lane, part);
        if (lane == 0) {
          reinterpret_cast<uint32_t*>(row + D * BITS / 8)[part] = z;
          if (part == 0) reinterpret_cast<__half2*>(side.aux)[prow] = __halves2half2(norm16, __float2half_rn(rn));
        }
      }
    } else if constexpr (FMT == F_F16) {
      uint32_t w[E / 2];
#pragma unroll
      for (int k = 0; k < E / 2; ++k) {
        const __half2 h2 = __floats2half2_rn(y[2 * k] * ys, y[2 * k + 1] * ys);
        w[k] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      if constexpr (E == 2) reinterpret_cast<uint32_t*>(row)[lane] = w[0];
      else if constexpr (E == 4) reinterpret_cast<uint2*>(row)[lane] = make_uint2(w[0], w[1]);
      else reinterpret_cast<uint4*>(row)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (FMT == F_F8) {
      if constexpr (E == 2) {
        reinterpret_cast<uint16_t*>(row)[lane] = (uint16_t)float2_to_fp8x2(y[0] * ys, y[1] * ys);
      } else {
        uint32_t w[E / 4];
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
          const int e = 4 * k;
          w[k] = float2_to_fp8x2(y[e] * ys, y[e + 1] * ys) | (float2_to_fp8x2(y[e + 2] * ys, y[e + 3] * ys) << 16);
        }
        if constexpr (E == 4) reinterpret_cast<uint32_t*>(row)[lane] = w[0];
        else reinterpret_cast<uint2*>(row)[lane] = make_uint2(w[0], w[1]);
      }
    } else {  // F_I4: a group of 32 coordinates spans 32 / E neighbouring lanes
      constexpr int LG = kGroup / E;
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(y[e] * ys));
#pragma unroll
      for (int m = 1; m < LG; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
      const __half s16 = __float2half_rn(amax / 7.0f);
      const float s = __half2float(s16);
      const float rcp = s > 0.0f ? 1.0f / s : 0.0f;
      uint32_t nib = 0u;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float xv = y[e] * ys;
        // level = rint(x / s): x * (1/s) is within one ulp of the quotient; where that
        // leaves the result next to a half-integer, divide exactly
        float tq = xv * rcp;
        if (s > 0.0f && fabsf(fabsf(tq - rintf(tq)) - 0.5f) < 1e-5f) tq = xv / s;
        const float q = s > 0.0f ? fminf(fmaxf(rintf(tq), -7.0f), 7.0f) : 0.0f;
        nib |= (uint32_t)((int)q + 8) << (4 * e);
      }
      if constexpr (E == 2) row[lane] = (uint8_t)nib;
      else if constexpr (E == 4) reinterpret_cast<uint16_t*>(row)[lane] = (uint16_t)nib;
      else reinterpret_cast<uint32_t*>(row)[lane] = nib;
      if (lane % LG == 0) side.aux[prow * (D / kGroup) + lane / LG] = s16;
    }
  }
}

template <int D, int FMT, bool FROM_ROWS>
__device__ __forceinline__ void append_bits(const QuantParams& p, const QuantSide& side, const uint16_t* x,
                                            const uint8_t* src, uint32_t* buf) {
  if (side.bits == 4) append_side<D, FMT, 4, FROM_ROWS>(p, side, x, src, buf);
  else if (side.bits == 3) append_side<D, FMT, 3, FROM_ROWS>(p, side, x, src, buf);
  else append_side<D, FMT, 2, FROM_ROWS>(p, side, x, src, buf);
}

// Grid row blockIdx.y = side kind_first + y; the format is a warp-uniform branch (only the
// taken path's instructions are fetched).
template <int D, bool FROM_ROWS>
__global__ void __launch_bounds__(kWarps * 32) append_kernel(const QuantParams p) {
  __shared__ __align__(16) uint32_t words[kWarps][32];
  const int kind = p.kind_first + blockIdx.y;  // 0 or 1
  const QuantSide side = kind ? p.side[1] : p.side[0];
  const uint16_t* x = kind ? p.x[1] : p.x[0];
  const uint8_t* src = kind ? p.src_rows[1] : p.src_rows[0];
  uint32_t* buf = words[threadIdx.x >> 5];
  switch (side.fmt) {
    case KVQ_FMT_CODEBOOK: append_bits<D, F_CB, FROM_ROWS>(p, side, x, src, buf); break;
    case KVQ_FMT_CODEBOOK_QJL: append_bits<D, F_CBQ, FROM_ROWS>(p, side, x, src, buf); break;
    case KVQ_FMT_CODEBOOK_OUTLIER:  // new vectors only (the host refuses a re-encode into it)
      if constexpr (!FROM_ROWS) append_bits<D, F_CBO, false>(p, side, x, src, buf);
      break;
    case KVQ_FMT_FP16: append_side<D, F_F16, 0, FROM_ROWS>(p, side, x, src, buf); break;
    case KVQ_FMT_FP8_E4M3: append_side<D, F_F8, 0, FROM_ROWS>(p, side, x, src, buf); break;
    default: append_side<D, F_I4, 0, FROM_ROWS>(p, side, x, src, buf); break;
  }
}

template <bool FROM_ROWS>
cudaError_t launch_warp_kernel(const QuantParams& p, int head_dim, int sms, cudaStream_t stream) {
  const bool sketch = p.side[0].fmt == KVQ_FMT_CODEBOOK_QJL && p.kind_first == 0;
  const long long nvec = (long long)p.num_tokens * p.hkv * (sketch ? KVQ_QJL_DIM / 32 : 1);  // work units
  const unsigned blocks =
      (unsigned)std::max<long long>(1, std::min<long long>((nvec + kWarps - 1) / kWarps, (long long)sms * 8));
  const dim3 grid(blocks, p.num_kinds);
  if (head_dim == 64) append_kernel<64, FROM_ROWS><<<grid, kWarps * 32, 0, stream>>>(p);
  else if (head_dim == 128) append_kernel<128, FROM_ROWS><<<grid, kWarps * 32, 0, stream>>>(p);
  else append_kernel<256, FROM_ROWS><<<grid, kWarps * 32, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

cudaError_t launch_quantize_small(const QuantParams& p, int head_dim, int sms, cudaStream_t stream) {
  return launch_warp_kernel<false>(p, head_dim, sms, stream);
}

cudaError_t launch_requantize(const QuantParams& p, int head_dim, cudaStream_t stream) {
  if (p.num_tokens == 0) return cudaSuccess;
  if ((long long)p.num_tokens * p.hkv > (1LL << 28)) return cudaErrorInvalidValue;  // four units per sketched key fit an int
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  return launch_warp_kernel<true>(p, head_dim, sms, stream);
}

}  // namespace kvq
