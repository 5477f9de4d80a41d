// Quantise-and-append: host-side dispatch and the per-thread kernel's instances (the
// kernels are in quantize.cuh; small appends go to quantize_small.cu).
#include "quantize.cuh"

namespace kvq {
namespace {

// Large appends: one launch per side, so every SM runs a single side's code path (the
// paths are long; two of them on one SM compete for the instruction cache).
template <int TPV>
cudaError_t launch_tpv(const QuantParams& p, int sms, cudaStream_t stream) {
  for (int kind = p.kind_first; kind < p.kind_first + p.num_kinds; ++kind) {
    QuantParams q = p;
    q.kind_first = kind;
    q.num_kinds = 1;
    const QuantSide& s = p.side[kind];
    cudaError_t e;
    switch (s.fmt) {
      case KVQ_FMT_CODEBOOK:
        e = s.bits == 4 ? launch_single<TPV, F_CB, 4>(q, sms, stream)
                        : (s.bits == 3 ? launch_single<TPV, F_CB, 3>(q, sms, stream)
                                       : launch_single<TPV, F_CB, 2>(q, sms, stream));
        break;
      case KVQ_FMT_CODEBOOK_QJL:
        e = s.bits == 4 ? launch_single<TPV, F_CBQ, 4>(q, sms, stream)
                        : (s.bits == 3 ? launch_single<TPV, F_CBQ, 3>(q, sms, stream)
                                       : launch_single<TPV, F_CBQ, 2>(q, sms, stream));
        break;
      case KVQ_FMT_FP16: e = launch_single<TPV, F_F16, 0>(q, sms, stream); break;
      case KVQ_FMT_FP8_E4M3: e = launch_single<TPV, F_F8, 0>(q, sms, stream); break;
      default: e = launch_single<TPV, F_I4, 0>(q, sms, stream); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_quantize(const QuantParams& p, int head_dim, cudaStream_t stream) {
  if (p.num_vectors == 0) return cudaSuccess;
  if ((long long)p.num_tokens * p.hkv > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // small appends, and keys with an outlier stream (whose channel split the per-thread
  // kernel does not carry), take the warp-per-vector kernel
  const bool outl = p.side[0].fmt == KVQ_FMT_CODEBOOK_OUTLIER && p.kind_first == 0;
  if ((long long)p.num_tokens * p.hkv <= kSmallMaxVectors || outl) return launch_quantize_small(p, head_dim, sms, stream);
  // kCoords coordinates per thread: head_dim / kCoords lanes per vector
  switch (head_dim) {
    case 64: return launch_tpv<64 / kCoords>(p, sms, stream);
    case 128: return launch_tpv<128 / kCoords>(p, sms, stream);
    case 256: return launch_tpv<256 / kCoords>(p, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
