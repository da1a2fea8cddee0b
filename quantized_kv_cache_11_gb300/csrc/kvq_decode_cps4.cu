// The uniform decode (kvq_decode_impl.cuh) as 4 CTAs of 4 warps per SM,
// for caches of many short (sequence, KV head) segments; chosen by decode_shape.
#include "kvq_decode_impl.cuh"

namespace kvq {

int decode_slots_cps4(const kvq_cache* c, int G, int* err) { return decode_slots_shape<4>(c, G, err); }

kvq_status decode_run_cps4(const kvq_cache* c, int G, const DecodeParams& p, cudaStream_t st) {
  return decode_run_shape<4>(c, G, p, st);
}

}  // namespace kvq
