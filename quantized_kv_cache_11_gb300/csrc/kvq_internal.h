// Host-side helpers shared by the kvq entry points (validation, sizes).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline size_t tile_bytes(const kvq_cache* c) {
  return (size_t)KVQ_GROUP * (size_t)c->head_dim * (size_t)c->bits / 8;
}

// Geometry checks (no pointer checks).  Host only, no CUDA call.
inline kvq_status validate_geometry(const kvq_cache* c) {
  if (c == nullptr) return KVQ_ERR_INVALID;
  if (c->batch < 1 || c->n_kv_heads < 1 || c->max_groups < 0) return KVQ_ERR_INVALID;
  if (c->tail_cap < KVQ_GROUP || c->tail_cap > 256 || c->tail_cap % KVQ_GROUP) return KVQ_ERR_INVALID;
  if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->bits != 2 && c->bits != 4 && c->bits != 8) return KVQ_ERR_UNSUPPORTED;
  // keep every buffer offset inside int64 and every grid dimension in range
  if ((int64_t)c->batch * c->n_kv_heads > (1 << 24)) return KVQ_ERR_UNSUPPORTED;
  if ((int64_t)c->max_groups > (1 << 26)) return KVQ_ERR_UNSUPPORTED;
  if (c->sink_cap < 0 || c->sink_cap > 256) return KVQ_ERR_INVALID;
  return KVQ_OK;
}

// Geometry plus every buffer pointer non-NULL: code, metadata and tail buffers
// 16-byte aligned, length arrays 4-byte aligned.
inline kvq_status validate_cache(const kvq_cache* c) {
  kvq_status s = validate_geometry(c);
  if (s != KVQ_OK) return s;
  const void* bufs[] = {c->k_codes, c->v_codes, c->k_meta, c->v_meta, c->k_tail, c->v_tail};
  for (const void* p : bufs)
    if (p == nullptr || !aligned(p, 16)) return KVQ_ERR_INVALID;
  const void* lens[] = {c->n_quant, c->n_tail, c->tail_head};
  for (const void* p : lens)
    if (p == nullptr || !aligned(p, 4)) return KVQ_ERR_INVALID;
  if (c->error_flags != nullptr && !aligned(c->error_flags, 4)) return KVQ_ERR_INVALID;
  if (c->sink_cap > 0) {
    if (c->k_sink == nullptr || c->v_sink == nullptr || !aligned(c->k_sink, 16) || !aligned(c->v_sink, 16))
      return KVQ_ERR_INVALID;
    if (c->n_sink == nullptr || !aligned(c->n_sink, 4)) return KVQ_ERR_INVALID;
  }
  return KVQ_OK;
}

inline kvq_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
