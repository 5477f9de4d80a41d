// Fused codebook decode: the instances for keys with a residual sign sketch (head_dim 128;
// VeloxQuant-MLX page, "Stage 3: QJL Residual Correction").  Kernels in decode_cb.cuh.
#include "decode_cb.cuh"

namespace kvq {
namespace cbk {

cudaError_t launch_cb_qjl(const CbParams& p, int g, int kb, int vb, int sms, cudaStream_t s) {
  return launch_g<128, kModeSketch>(p, g, kb, vb, sms, s);
}

cudaError_t launch_project_qjl(const CbParams& p, int g, int batch, cudaStream_t s) {
  const unsigned blocks = (unsigned)batch * (unsigned)p.hkv;
  if (blocks == 0) return cudaSuccess;
  if (g == 1) project_kernel<128, 1><<<blocks, 128, 0, s>>>(p);
  else if (g == 2) project_kernel<128, 2><<<blocks, 128, 0, s>>>(p);
  else project_kernel<128, 4><<<blocks, 128, 0, s>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace cbk
}  // namespace kvq
