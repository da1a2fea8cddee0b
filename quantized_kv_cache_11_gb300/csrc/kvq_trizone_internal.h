// Constants, record sizes and host-side validation of the mixed-width cache.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvq_trizone.h"
#include "kvq_internal.h"

namespace kvq {
namespace tz {

constexpr int kDim = 128;   // head_dim
constexpr int kKinds = 5;   // block kinds: value width 2, 4, 8, 16, fresh
constexpr int kKtMax = 10;  // k-tiles of three key classes over 128 channels, at most
constexpr int kSlots = 16 * kKtMax;
constexpr int kFp16TileBytes = 32 * kDim * 2;  // 32 tokens x 128 channels of fp16

// int32 fields of the index record
enum {
  H_NTOK = 0,     // [4] kept tokens per value width
  H_NFRESH = 4,   // fresh tokens
  H_NBLK = 5,     // [5] blocks per kind
  H_NCH = 10,     // [3] channels per key width
  H_KT = 13,      // [3] k-tiles per key width
  H_REC = 16,     // [5] bytes of one block of each kind
  H_OFF = 21,     // [5] byte offset of each kind's first block
  H_USED = 26,    // bytes used in the region
};

__host__ __device__ constexpr int key_code_bytes(int kt2, int kt4, int kt8) {
  return 128 * kt2 + 256 * kt4 + 512 * kt8;
}
__host__ __device__ constexpr int key_bytes(int kt2, int kt4, int kt8) {
  return key_code_bytes(kt2, kt4, kt8) + 64 * (kt2 + kt4 + kt8);
}
// value bytes of a block of value class vc (0, 1, 2 = width 2, 4, 8; 3 = fp16)
__host__ __device__ constexpr int value_bytes(int vc) {
  return vc == 3 ? kFp16TileBytes : (32 * kDim * (2 << vc) / 8 + 4 * kDim);
}
__host__ __device__ constexpr int record_bytes(int kt2, int kt4, int kt8, int vc) {
  return key_bytes(kt2, kt4, kt8) + value_bytes(vc);
}

inline int64_t region_bytes(const kvq_trizone* t) {
  const int64_t blocks = ((int64_t)t->max_old + 31) / 32 + 3;
  const int64_t fresh = ((int64_t)t->max_fresh + 31) / 32;
  const int64_t r = blocks * KVQ_TZ_MAX_BLOCK_BYTES + fresh * KVQ_TZ_FRESH_BLOCK_BYTES;
  return (r + 255) / 256 * 256;
}

inline kvq_status validate_geometry(const kvq_trizone* t) {
  if (t == nullptr) return KVQ_ERR_INVALID;
  if (t->batch < 1 || t->n_kv_heads < 1 || t->max_old < 0 || t->max_fresh < 0) return KVQ_ERR_INVALID;
  if (t->head_dim != kDim) return KVQ_ERR_UNSUPPORTED;
  if ((int64_t)t->batch * t->n_kv_heads > (1 << 20)) return KVQ_ERR_UNSUPPORTED;
  // every block offset of a region fits an int32 field of the index
  if (region_bytes(t) > ((int64_t)1 << 31) - 1) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

inline kvq_status validate_buffers(const kvq_trizone* t) {
  kvq_status s = validate_geometry(t);
  if (s != KVQ_OK) return s;
  if (t->index == nullptr || t->blocks == nullptr || !aligned(t->index, 16) || !aligned(t->blocks, 16))
    return KVQ_ERR_INVALID;
  if (t->max_old > 0 && (t->tokens == nullptr || !aligned(t->tokens, 4))) return KVQ_ERR_INVALID;
  if (t->error_flags != nullptr && !aligned(t->error_flags, 4)) return KVQ_ERR_INVALID;
  return KVQ_OK;
}

}  // namespace tz
}  // namespace kvq
