// Helpers shared by the kvq entry points: validation and sizes on the host, and
// a byte packer for the quantizers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/kvq.h"

namespace kvq {

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

#ifdef __CUDACC__
// Four values <= 255 as the bytes of one word (a in byte 0), by byte permutes
// (three instructions, against three shifts and two ORs).
__device__ __forceinline__ uint32_t pack4_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}
#endif

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

// Launch facts of one kernel on the CURRENT device: its dynamic shared-memory
// limit raised to `smem` bytes (function attributes are per device) and the
// number of its CTAs of `threads` threads that fit on the whole GPU at once
// (SM count x CTAs per SM).  Computed once per (kernel, device) under a lock,
// so several host threads and several GPUs in one process each get their own.
// Returns 0 (and sets *err) if a CUDA query fails or no CTA fits.
inline int device_slots(const void* kernel, int threads, int smem, int* err) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = 1;
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int sms = 0, per = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem) != cudaSuccess || per < 1) {
    *err = 1;
    return 0;
  }
  cache[key] = sms * per;
  return sms * per;
}

// Raise a kernel's dynamic shared-memory limit to `smem` bytes on the current
// device, once per (kernel, device) under a lock.  Returns false if a CUDA call
// fails.
inline bool device_smem_attr(const void* kernel, int smem) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, bool> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  if (done.count(key)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
  done[key] = true;
  return true;
}

inline kvq_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
