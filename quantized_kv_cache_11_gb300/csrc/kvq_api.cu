// kvq C ABI: sizes, status strings, version.  Host only.
#include "kvq_internal.h"

extern "C" kvq_status kvq_cache_bytes(const kvq_cache* c, size_t sizes[KVQ_NBUF]) {
  kvq_status s = kvq::validate_geometry(c);
  if (s != KVQ_OK) return s;
  if (sizes == nullptr) return KVQ_ERR_INVALID;
  const size_t bh = (size_t)c->batch * (size_t)c->n_kv_heads;
  const size_t groups = bh * (size_t)c->max_groups;
  sizes[KVQ_BUF_K_CODES] = groups * kvq::tile_bytes(c);
  sizes[KVQ_BUF_V_CODES] = groups * kvq::tile_bytes(c);
  sizes[KVQ_BUF_K_META] = groups * 2 * (size_t)c->head_dim * 2;
  sizes[KVQ_BUF_V_META] = groups * 2 * (size_t)c->head_dim * 2;
  sizes[KVQ_BUF_K_TAIL] = bh * (size_t)c->tail_cap * (size_t)c->head_dim * 2;
  sizes[KVQ_BUF_V_TAIL] = sizes[KVQ_BUF_K_TAIL];
  sizes[KVQ_BUF_LENGTHS] = (size_t)c->batch * sizeof(int32_t);
  sizes[KVQ_BUF_K_SINK] = bh * (size_t)c->sink_cap * (size_t)c->head_dim * 2;
  sizes[KVQ_BUF_V_SINK] = sizes[KVQ_BUF_K_SINK];
  return KVQ_OK;
}

extern "C" const char* kvq_status_string(int status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported geometry";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

extern "C" const char* kvq_version(void) { return "0.1.0"; }
