// Fused codebook decode: host-side dispatch and the instances for plain codebook keys (the
// kernels are in decode_cb.cuh; keys with a residual sketch are instantiated in
// decode_cb_qjl.cu).
#include "decode_cb.cuh"

namespace kvq {

constexpr size_t PS_TOKENS = 16;  // tokens per page on the codebook path

bool cb_fast_supported(int head_dim, int group, int k_fmt, int v_fmt) {
  if (group == 8)  // plain codes: the 4-head instances, two items per chunk
    return (head_dim == 128 || head_dim == 256) && v_fmt == KVQ_FMT_CODEBOOK && k_fmt == KVQ_FMT_CODEBOOK;
  return (head_dim == 128 || head_dim == 256) && (group == 1 || group == 2 || group == 4) &&
         v_fmt == KVQ_FMT_CODEBOOK &&
         (k_fmt == KVQ_FMT_CODEBOOK || k_fmt == KVQ_FMT_CODEBOOK_OUTLIER ||
          (k_fmt == KVQ_FMT_CODEBOOK_QJL && head_dim == 128));
}

cudaError_t launch_decode_cb(const DecParams& dp, int head_dim, int* counters, cudaStream_t stream,
                             bool after_split_k) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int group = dp.hq / dp.hkv;
  bool projected = false;  // every sketched tier shares the projection and the queries
  // large caches take the 16-warp tensor-core instances (measured on GB300: ragged, 1.4 GB,
  // 1118 -> 1056 us; a 138 MB cache with 2 query heads per kv head 85 -> 89 us, slower)
  size_t cb_bytes = 0;
  for (int i = 0; i < dp.num_tiers; ++i)
    if (dp.tier[i].kind == TIER_CB) cb_bytes += (size_t)dp.batch * dp.hkv * dp.tier[i].max_pages * PS_TOKENS *
                                                (dp.tier[i].k_row_bytes + dp.tier[i].v_row_bytes);
  const bool wide = cb_bytes >= ((size_t)512 << 20);  // (8 heads per kv head: the same rule)
  for (int i = 0; i < dp.num_tiers; ++i) {
    const DecTier& t = dp.tier[i];
    if (t.kind != TIER_CB) continue;
    cbk::CbParams p;
    memset(&p, 0, sizeof(p));
    p.t.k_rows = t.k_rows;
    p.t.v_rows = t.v_rows;
    p.t.k_norm = t.k_aux;
    p.t.qjl = t.k_qjl;
    p.t.outl = t.k_outl;
    p.t.v_norm = t.v_aux;
    p.t.block_table = t.block_table;
    p.t.seq_lens = t.seq_lens;
    p.t.num_pages = t.num_pages;
    p.t.max_pages = t.max_pages;
    p.t.chunk = t.chunk;
    p.t.nchunks = t.num_splits;
    p.t.split_begin = t.split_begin;
    p.q = dp.q;
    p.k_signs = dp.k_signs;
    p.k_cent = t.k_cent;
    p.v_cent = t.v_cent;
    p.ws_acc = dp.ws_acc;
    p.ws_ml = dp.ws_ml;
    p.pq = dp.ws_pq;
    p.ws_min = dp.ws_min;
    p.gate = dp.gate;
    p.track = dp.spike != nullptr && i == 0;
    p.counter = counters + i;
    p.t.err = dp.err;
    p.hq = dp.hq;
    p.hkv = dp.hkv;
    p.total_splits = dp.total_splits;
    p.total_items = dp.batch * dp.hkv * t.num_splits * (group == 8 ? 2 : 1);
    if (p.total_items == 0) continue;
    // run alongside the previous split-K grid, unless the projection (whose output this
    // launch reads) is what precedes it
    p.pdl = after_split_k ? 1 : 0;
    p.trigger = 0;
    for (int j = i + 1; j < dp.num_tiers; ++j) p.trigger |= dp.tier[j].kind == TIER_CB ? 1 : 0;
    if (t.k_fmt == KVQ_FMT_CODEBOOK_QJL && !projected) {
      if ((e = cbk::launch_project_qjl(p, group, dp.batch, stream)) != cudaSuccess) return e;
      projected = true;
      p.pdl = 0;
    }
    if (group == 8) e = cbk::launch_cb_g8(p, head_dim, wide, t.k_bits, t.v_bits, sms, stream);
    else if (t.k_fmt == KVQ_FMT_CODEBOOK_QJL) e = cbk::launch_cb_qjl(p, group, t.k_bits, t.v_bits, sms, stream);
    else if (t.k_fmt == KVQ_FMT_CODEBOOK_OUTLIER)
      e = cbk::launch_cb_outlier(p, head_dim, group, t.k_bits, t.v_bits, sms, stream);
    else if (head_dim == 128 && group >= 2 && wide)
      e = cbk::launch_cb_wide(p, group, t.k_bits, t.v_bits, sms, stream);
    else if (head_dim == 128) e = cbk::launch_g<128, cbk::kModePlain>(p, group, t.k_bits, t.v_bits, sms, stream);
    else e = cbk::launch_g<256, cbk::kModePlain>(p, group, t.k_bits, t.v_bits, sms, stream);
    if (e != cudaSuccess) return e;
    after_split_k = true;
  }
  return cudaSuccess;
}

}  // namespace kvq
