// Host-side Rademacher sign vectors of the rotation (computed once per layer at start-up).
//
// VeloxQuant-MLX page ("I Ported a Google Research Paper to Apple Silicon"), section
// "Stage 1: Random Rotation", and AdapTQ page, section "The Math Fix": every coordinate is
// multiplied by a random +1 / -1 before the Walsh-Hadamard transform.  The pages leave the
// draw open; here each sign is the lowest bit of the first output of a SplitMix64 generator
// (Steele, Lea and Flood, OOPSLA 2014) whose state starts at seed XOR key, key = layer * 2^40
// + side * 2^32 + kv head * 2^16 + coordinate: bit 0 gives +1, bit 1 gives -1.  One draw per
// sign makes every sign computable on its own, in any order.
#include "../../include/kvq.h"

namespace {

uint64_t splitmix64_first(uint64_t state) {
  uint64_t z = state + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

}  // namespace

extern "C" KVQ_API kvq_status kvq_make_signs(uint64_t seed, int32_t layer, int32_t num_kv_heads,
                                             int32_t head_dim, int8_t* k_signs, int8_t* v_signs) {
  if (!k_signs || !v_signs) return KVQ_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= (1 << 24) || num_kv_heads < 1 || num_kv_heads > (1 << 16)) return KVQ_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  int8_t* out[2] = {k_signs, v_signs};
  for (uint64_t side = 0; side < 2; ++side)
    for (int32_t h = 0; h < num_kv_heads; ++h)
      for (int32_t j = 0; j < head_dim; ++j) {
        const uint64_t key = ((uint64_t)layer << 40) + (side << 32) + ((uint64_t)h << 16) + (uint64_t)j;
        out[side][(size_t)h * head_dim + j] = (splitmix64_first(seed ^ key) & 1u) ? (int8_t)-1 : (int8_t)1;
      }
  return KVQ_OK;
}
