// kvq_decode_attention_noalloc: decode attention whose split-K scratch lives in a static
// device array owned by the library, for callers that cannot allocate device memory.
//
// The array is a file-scope __device__ variable of fixed size, so every GPU that loads the
// library holds it until the process exits.  Host code must not use the array's name as a
// device address (on the host it names a stand-in object): the address is fetched once per
// device with cudaGetSymbolAddress while that device is current, then handed to the
// ordinary decode entry point as its workspace.
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = KVQ_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Address of this device's scratch array; looked up on the first call made with the
// device current and remembered afterwards.
kvq_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_tier_view* tiers, int32_t num_tiers,
                                                          const uint16_t* q, int32_t batch,
                                                          int32_t num_q_heads, int32_t split_tokens,
                                                          float* out, void* stream) {
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_size(tiers, num_tiers, batch, num_q_heads, split_tokens, &need);
  if (st != KVQ_OK) return st;
  if (need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != KVQ_OK) return st;
  // The decode call itself clears the one word of scratch that must start at zero (its work
  // counter); the split-K pass writes every partial before the combine pass reads it.
  return kvq_decode_attention(tiers, num_tiers, q, batch, num_q_heads, split_tokens, out, scratch,
                              kNoAllocScratchBytes, stream);
}
