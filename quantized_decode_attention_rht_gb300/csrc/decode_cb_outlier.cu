// Fused codebook decode: the instances for keys with an outlier stream (VeloxQuant-MLX page,
// "Outlier Two-Stream Cache": int8 outlier channels added to the inlier score).  Kernels in
// decode_cb.cuh.
#include "decode_cb.cuh"

namespace kvq {
namespace cbk {

cudaError_t launch_cb_outlier(const CbParams& p, int d, int g, int kb, int vb, int sms, cudaStream_t s) {
  return d == 128 ? launch_g<128, kModeOutlier>(p, g, kb, vb, sms, s) : launch_g<256, kModeOutlier>(p, g, kb, vb, sms, s);
}

}  // namespace cbk
}  // namespace kvq
