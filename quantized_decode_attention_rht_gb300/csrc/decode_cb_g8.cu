// Fused codebook decode: the instances for 8 query heads per kv head (plain codes, head_dim
// 128 or 256).  Each chunk of a kv head makes two items, heads 0-3 and heads 4-7, on the
// 4-head tensor-core path; every chunk of heads 0-3 is handed out before the chunks of
// heads 4-7, so the second pass over a chunk finds its pages in L2.  Kernels in decode_cb.cuh.
#include "decode_cb.cuh"

namespace kvq {
namespace cbk {
namespace {

template <int D, bool WIDE, int KB>
cudaError_t g8_vb(const CbParams& p, int vb, int sms, cudaStream_t s) {
  switch (vb) {
    case 2: return launch_path<PathM<D, 4, KB, 2, kModePlain, WIDE, true>>(p, sms, s);
    case 3: return launch_path<PathM<D, 4, KB, 3, kModePlain, WIDE, true>>(p, sms, s);
    default: return launch_path<PathM<D, 4, KB, 4, kModePlain, WIDE, true>>(p, sms, s);
  }
}

template <int D, bool WIDE>
cudaError_t g8_kb(const CbParams& p, int kb, int vb, int sms, cudaStream_t s) {
  switch (kb) {
    case 2: return g8_vb<D, WIDE, 2>(p, vb, sms, s);
    case 3: return g8_vb<D, WIDE, 3>(p, vb, sms, s);
    default: return g8_vb<D, WIDE, 4>(p, vb, sms, s);
  }
}

}  // namespace

cudaError_t launch_cb_g8(const CbParams& p, int d, bool wide, int kb, int vb, int sms, cudaStream_t s) {
  if (d == 256) return g8_kb<256, false>(p, kb, vb, sms, s);
  return wide ? g8_kb<128, true>(p, kb, vb, sms, s) : g8_kb<128, false>(p, kb, vb, sms, s);
}

}  // namespace cbk
}  // namespace kvq
