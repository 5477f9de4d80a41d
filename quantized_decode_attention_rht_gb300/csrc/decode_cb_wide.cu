// Fused codebook decode: the 16-warp instances of the tensor-core path (plain codes, head_dim
// 128, 2 or 4 query heads per kv head) that large caches use.  Kernels in decode_cb.cuh.
#include "decode_cb.cuh"

namespace kvq {
namespace cbk {
namespace {

template <int G, int KB>
cudaError_t wide_vb(const CbParams& p, int vb, int sms, cudaStream_t s) {
  switch (vb) {
    case 2: return launch_path<PathM<128, G, KB, 2, kModePlain, true>>(p, sms, s);
    case 3: return launch_path<PathM<128, G, KB, 3, kModePlain, true>>(p, sms, s);
    default: return launch_path<PathM<128, G, KB, 4, kModePlain, true>>(p, sms, s);
  }
}

template <int G>
cudaError_t wide_kb(const CbParams& p, int kb, int vb, int sms, cudaStream_t s) {
  switch (kb) {
    case 2: return wide_vb<G, 2>(p, vb, sms, s);
    case 3: return wide_vb<G, 3>(p, vb, sms, s);
    default: return wide_vb<G, 4>(p, vb, sms, s);
  }
}

}  // namespace

cudaError_t launch_cb_wide(const CbParams& p, int g, int kb, int vb, int sms, cudaStream_t s) {
  return g == 2 ? wide_kb<2>(p, kb, vb, sms, s) : wide_kb<4>(p, kb, vb, sms, s);
}

}  // namespace cbk
}  // namespace kvq
