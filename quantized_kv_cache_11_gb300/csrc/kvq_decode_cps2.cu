// The uniform decode (kvq_decode_impl.cuh) as 2 CTAs of 8 warps per SM,
// for caches of many short (sequence, KV head) segments; chosen by decode_shape.
#include "kvq_decode_impl.cuh"

namespace kvq {

int decode_slots_cps2(const kvq_cache* c, int G, int* err) { return decode_slots_shape<2>(c, G, err); }

kvq_status decode_run_cps2(const kvq_cache* c, int G, const DecodeParams& p, cudaStream_t st) {
  return decode_run_shape<2>(c, G, p, st);
}

}  // namespace kvq
