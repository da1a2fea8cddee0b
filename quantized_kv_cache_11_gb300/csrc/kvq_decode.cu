// C entry points of the uniform-cache decode (kernels in kvq_decode_impl.cuh).
#include "kvq_decode_impl.cuh"

namespace kvq {

inline int decode_slots(const kvq_cache* c, int G, int* err) {
#define KVQ_SLOTS(D_, B_, G_) \
  if (c->head_dim == D_ && c->bits == B_ && G == G_) return DecodeLaunch<D_, B_, G_>::slots(err);
#define KVQ_SLOTS_G(D_, B_) KVQ_SLOTS(D_, B_, 1) KVQ_SLOTS(D_, B_, 2) KVQ_SLOTS(D_, B_, 4) KVQ_SLOTS(D_, B_, 8)
  KVQ_SLOTS_G(128, 2) KVQ_SLOTS_G(128, 4) KVQ_SLOTS_G(128, 8)
  KVQ_SLOTS_G(64, 2) KVQ_SLOTS_G(64, 4) KVQ_SLOTS_G(64, 8)
#undef KVQ_SLOTS_G
#undef KVQ_SLOTS
  *err = 2;
  return 0;
}

}  // namespace kvq

extern "C" kvq_status kvq_decode_workspace_bytes(const kvq_cache* c, int32_t n_q_heads, size_t* bytes) {
  using namespace kvq;
  kvq_status s = validate_geometry(c);
  if (s != KVQ_OK) return s;
  if (bytes == nullptr) return KVQ_ERR_INVALID;
  int G = 0;
  s = validate_q_heads(c, n_q_heads, &G);
  if (s != KVQ_OK) return s;
  int err = 0;
  const int n = decode_slots(c, G, &err);
  if (err) return KVQ_ERR_CUDA;
  *bytes = decode_layout(c, G, n).total;
  return KVQ_OK;
}

extern "C" kvq_status kvq_decode_attn(const kvq_cache* c, int32_t n_q_heads, const void* q, float* out,
                                      float sm_scale, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  using namespace kvq;
  kvq_status s = validate_cache(c);
  if (s != KVQ_OK) return s;
  int G = 0;
  s = validate_q_heads(c, n_q_heads, &G);
  if (s != KVQ_OK) return s;
  if (q == nullptr || out == nullptr || workspace == nullptr) return KVQ_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(out, 16) || !aligned(workspace, 16)) return KVQ_ERR_INVALID;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID;
  int err = 0;
  const int n = decode_slots(c, G, &err);
  if (err) return KVQ_ERR_CUDA;
  const DecodeLayout L = decode_layout(c, G, n);
  if (workspace_bytes < L.total) return KVQ_ERR_INVALID;
  DecodeParams p{};
  p.k_codes = static_cast<const uint8_t*>(c->k_codes);
  p.v_codes = static_cast<const uint8_t*>(c->v_codes);
  p.k_meta = static_cast<const __half*>(c->k_meta);
  p.v_meta = static_cast<const __half*>(c->v_meta);
  p.k_tail = static_cast<const __half*>(c->k_tail);
  p.v_tail = static_cast<const __half*>(c->v_tail);
  p.n_quant = c->n_quant;
  p.n_tail = c->n_tail;
  p.tail_head = c->tail_head;
  p.k_sink = static_cast<const __half*>(c->k_sink);
  p.v_sink = static_cast<const __half*>(c->v_sink);
  p.n_sink = c->n_sink;
  p.error_flags = c->error_flags;
  p.q = static_cast<const __half*>(q);
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<int32_t*>(ws + L.counters);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.batch = c->batch;
  p.hkv = c->n_kv_heads;
  p.max_groups = c->max_groups;
  p.tail_cap = c->tail_cap;
  p.sink_cap = c->sink_cap;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->head_dim == 128) {
    if (c->bits == 2) return decode_dispatch_g<128, 2>(G, p, st);
    if (c->bits == 4) return decode_dispatch_g<128, 4>(G, p, st);
    return decode_dispatch_g<128, 8>(G, p, st);
  }
  if (c->bits == 2) return decode_dispatch_g<64, 2>(G, p, st);
  if (c->bits == 4) return decode_dispatch_g<64, 4>(G, p, st);
  return decode_dispatch_g<64, 8>(G, p, st);
}

// ---------------------------------------------------------------------------
// Decode without a caller-supplied workspace.  The split-K partials and merge
// counters live in a fixed array compiled into the library, so the call needs
// no device allocation at all.
// ---------------------------------------------------------------------------
#include <mutex>

namespace kvq {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_STATIC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device (host code cannot use
// the symbol itself: on the host it names a stand-in, not device memory).  Looked
// up once per device, with that device current.
static cudaError_t static_scratch_ptr(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

}  // namespace kvq

extern "C" kvq_status kvq_decode_attn_static(const kvq_cache* c, int32_t n_q_heads, const void* q, float* out,
                                             float sm_scale, void* stream) {
  using namespace kvq;
  kvq_status s = validate_cache(c);
  if (s != KVQ_OK) return s;
  int G = 0;
  s = validate_q_heads(c, n_q_heads, &G);
  if (s != KVQ_OK) return s;
  if (q == nullptr || out == nullptr) return KVQ_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(out, 16)) return KVQ_ERR_INVALID;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID;
  int err = 0;
  const int n = decode_slots(c, G, &err);
  if (err) return KVQ_ERR_CUDA;
  const DecodeLayout L = decode_layout(c, G, n);
  if (L.total > (size_t)KVQ_STATIC_SCRATCH_BYTES) return KVQ_ERR_CAPACITY;
  void* scratch = nullptr;
  if (static_scratch_ptr(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  // the merge counters must start at zero; a completed call leaves them zero, an
  // interrupted one might not, so clear them every time (a memset, no allocation)
  if (cudaMemsetAsync(ws + L.counters, 0, L.part - L.counters, st) != cudaSuccess) return KVQ_ERR_CUDA;
  DecodeParams p{};
  p.k_codes = static_cast<const uint8_t*>(c->k_codes);
  p.v_codes = static_cast<const uint8_t*>(c->v_codes);
  p.k_meta = static_cast<const __half*>(c->k_meta);
  p.v_meta = static_cast<const __half*>(c->v_meta);
  p.k_tail = static_cast<const __half*>(c->k_tail);
  p.v_tail = static_cast<const __half*>(c->v_tail);
  p.n_quant = c->n_quant;
  p.n_tail = c->n_tail;
  p.tail_head = c->tail_head;
  p.k_sink = static_cast<const __half*>(c->k_sink);
  p.v_sink = static_cast<const __half*>(c->v_sink);
  p.n_sink = c->n_sink;
  p.error_flags = c->error_flags;
  p.q = static_cast<const __half*>(q);
  p.out = out;
  p.counters = reinterpret_cast<int32_t*>(ws + L.counters);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.batch = c->batch;
  p.hkv = c->n_kv_heads;
  p.max_groups = c->max_groups;
  p.tail_cap = c->tail_cap;
  p.sink_cap = c->sink_cap;
  if (c->head_dim == 128) {
    if (c->bits == 2) return decode_dispatch_g<128, 2>(G, p, st);
    if (c->bits == 4) return decode_dispatch_g<128, 4>(G, p, st);
    return decode_dispatch_g<128, 8>(G, p, st);
  }
  if (c->bits == 2) return decode_dispatch_g<64, 2>(G, p, st);
  if (c->bits == 4) return decode_dispatch_g<64, 4>(G, p, st);
  return decode_dispatch_g<64, 8>(G, p, st);
}
