// C entry points of the uniform-cache decode (kernels in kvq_decode_impl.cuh).
#include "kvq_decode_impl.cuh"

#include <mutex>

namespace kvq {

inline int decode_slots(const kvq_cache* c, int G, int* err) {
  const int cps = decode_shape(c, err);
  if (*err) return 0;
  if (cps == 2) return decode_slots_cps2(c, G, err);
  if (cps == 4) return decode_slots_cps4(c, G, err);
  return decode_slots_shape<1>(c, G, err);
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

namespace kvq {

// Host-side checks shared by both uniform decode entry points; sets *G and *L
// (the workspace layout for the current device).
static kvq_status decode_prepare(const kvq_cache* c, int32_t n_q_heads, const void* q, const float* out,
                                 float sm_scale, int* G, DecodeLayout* L) {
  kvq_status s = validate_cache(c);
  if (s != KVQ_OK) return s;
  s = validate_q_heads(c, n_q_heads, G);
  if (s != KVQ_OK) return s;
  if (q == nullptr || out == nullptr) return KVQ_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(out, 16)) return KVQ_ERR_INVALID;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID;
  int err = 0;
  const int n = decode_slots(c, *G, &err);
  if (err) return KVQ_ERR_CUDA;
  *L = decode_layout(c, *G, n);
  return KVQ_OK;
}

static kvq_status decode_launch(const kvq_cache* c, int G, const DecodeParams& p, cudaStream_t st) {
  int err = 0;
  const int cps = decode_shape(c, &err);
  if (err) return KVQ_ERR_CUDA;
  if (cps == 2) return decode_run_cps2(c, G, p, st);
  if (cps == 4) return decode_run_cps4(c, G, p, st);
  return decode_run_shape<1>(c, G, p, st);
}

}  // namespace kvq

extern "C" kvq_status kvq_decode_attn(const kvq_cache* c, int32_t n_q_heads, const void* q, float* out,
                                      float sm_scale, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  using namespace kvq;
  int G = 0;
  DecodeLayout L{};
  if (workspace == nullptr || !aligned(workspace, 16)) return KVQ_ERR_INVALID;
  kvq_status s = decode_prepare(c, n_q_heads, q, out, sm_scale, &G, &L);
  if (s != KVQ_OK) return s;
  if (workspace_bytes < L.total) return KVQ_ERR_INVALID;
  const DecodeParams p = decode_params(c, q, out, sm_scale, static_cast<uint8_t*>(workspace), L);
  return decode_launch(c, G, p, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Decode without a caller-supplied workspace.  The split-K partials and merge
// counters live in a fixed array compiled into the library, so the call needs
// no device allocation at all.
// ---------------------------------------------------------------------------
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
  int G = 0;
  DecodeLayout L{};
  kvq_status s = decode_prepare(c, n_q_heads, q, out, sm_scale, &G, &L);
  if (s != KVQ_OK) return s;
  if (L.total > (size_t)KVQ_STATIC_SCRATCH_BYTES) return KVQ_ERR_CAPACITY;
  void* scratch = nullptr;
  if (static_scratch_ptr(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  // the merge counters must start at zero; a completed call leaves them zero, an
  // interrupted one might not, so clear them every time (a memset, no allocation)
  if (cudaMemsetAsync(ws + L.counters, 0, L.part - L.counters, st) != cudaSuccess) return KVQ_ERR_CUDA;
  const DecodeParams p = decode_params(c, q, out, sm_scale, ws, L);
  return decode_launch(c, G, p, st);
}
