// Calibration of the outlier two-stream cache (VeloxQuant-MLX page, "Outlier Two-Stream
// Cache", steps 1 and 2): per kv head, the population variance of every key channel over
// the calibration tokens, and the KVQ_OUTLIER_CHANNELS channels of largest variance.
//
// One block per kv head, one thread per channel.  The statistics are taken in fp64 (the
// fp16 inputs are exact in it; two passes, mean then squared deviations), so the ranking
// is that of the exact variances except where two of them agree to ~1e-15.  The top
// channels come out of KVQ_OUTLIER_CHANNELS rounds of a block-wide argmax (ties to the
// lower channel).  A one-off step per sequence: it reads num_tokens * Hkv * D fp16 once.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

template <int D>
__global__ void __launch_bounds__(D) calibrate_kernel(const __half* k, int n, int hkv, int32_t* out) {
  __shared__ double s_v[D];
  __shared__ int s_i[D];
  const int h = blockIdx.x, c = threadIdx.x;
  const __half* x = k + (size_t)h * D + c;
  const size_t stride = (size_t)hkv * D;
  double sum = 0.0;
  for (int t = 0; t < n; ++t) sum += (double)__half2float(x[(size_t)t * stride]);
  const double mean = sum / n;
  double ss = 0.0;
  for (int t = 0; t < n; ++t) {
    const double dv = (double)__half2float(x[(size_t)t * stride]) - mean;
    ss = fma(dv, dv, ss);
  }
  double var = ss / n;
  for (int r = 0; r < KVQ_OUTLIER_CHANNELS; ++r) {
    s_v[c] = var;
    s_i[c] = c;
    __syncthreads();
    for (int w = D / 2; w > 0; w >>= 1) {
      if (c < w) {
        const double a = s_v[c], b = s_v[c + w];
        const int ia = s_i[c], ib = s_i[c + w];
        if (b > a || (b == a && ib < ia)) {
          s_v[c] = b;
          s_i[c] = ib;
        }
      }
      __syncthreads();
    }
    const int win = s_i[0];
    if (c == 0) out[h * KVQ_OUTLIER_CHANNELS + r] = win;
    if (c == win) var = -1.0;  // taken; every variance is >= 0
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_outlier_calibrate(const uint16_t* k, int num_tokens, int hkv, int head_dim, int32_t* out,
                                     cudaStream_t stream) {
  const __half* kh = reinterpret_cast<const __half*>(k);
  if (head_dim == 128) calibrate_kernel<128><<<hkv, 128, 0, stream>>>(kh, num_tokens, hkv, out);
  else calibrate_kernel<256><<<hkv, 256, 0, stream>>>(kh, num_tokens, hkv, out);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace kvq
