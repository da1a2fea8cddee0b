// Decode attention over a cache of pre-RoPE keys ("KV-cache quantization axes",
// ihal.it, paragraph 7 and the closing paragraph: quantize the keys before the
// rotary position embedding, rotate them after dequantization).
//
// The kernels are the uniform decode's (kvq_decode_impl.cuh) with ROPE set.  At
// 2 and 4 bits the rotated keys' products run on tensor cores: the query is
// turned back by the angle of the group's 32-position block (table row 64 + m,
// staged with the group by TMA) and each code is multiplied, exactly in fp16, by
// pieces of the cos/sin of its offset inside the block (the fp16 piece part of
// the table, in shared memory).  At 8 bits, and for the fp16 tail and sink
// chunks, a lane rotates its key pairs in fp32 and forms the dot products on
// CUDA cores, the angle of position 32 m + o from rows 64 + m and o by the
// angle-sum formulas.
#include "kvq_decode_impl.cuh"

namespace kvq {

inline int rope_blocks(const kvq_cache* c) {
  return (int)(((int64_t)c->sink_cap + (int64_t)kGroup * c->max_groups + c->tail_cap + kGroup - 1) / kGroup);
}

// table[o][i] = (cos, sin)(o theta_i) for o < 64; table[64 + m][i] = (cos, sin)(32 m theta_i).
__global__ void rope_table_kernel(float2* table, int half, int rows, double base) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)rows * half) return;
  const int row = (int)(idx / half), i = (int)(idx % half);
  const double theta = pow(base, -2.0 * i / (2.0 * half));
  const double pos = row < 64 ? (double)row : 32.0 * (double)(row - 64);
  double s, c;
  sincos(pos * theta, &s, &c);
  table[idx] = make_float2((float)c, (float)s);
}

// x rounded to nearest with at most hb significant bits (float64).
__device__ inline double round_bits(double x, int hb) {
  if (x == 0.0) return 0.0;
  int e;
  const double m = frexp(x, &e);  // x = m 2^e, 0.5 <= |m| < 1
  return ldexp(rint(ldexp(m, hb)), e - hb);
}

// The fp16 piece part (layout of kRopeTrigRow): one thread per half2 slot.
__global__ void rope_trig_kernel(uint8_t* trig, int half, double base, int hb) {
  constexpr int kSlots = kRopeTrigRows * 8 * 4 * 2 * 4;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= kSlots) return;
  const int e = idx & 3, pc = (idx >> 2) & 1, tig = (idx >> 3) & 3, kt = (idx >> 5) & 7, o = idx >> 8;
  const int i = 8 * kt + tig + 4 * (e >> 1);  // pair
  const int row = o + 8 * (e & 1);            // offset
  const double theta = pow(base, -2.0 * i / (2.0 * half));
  double sn, cs;
  sincos((double)row * theta, &sn, &cs);
  // pieces times 2^14 (exact power-of-two scaling; |hi| <= 2^14)
  const double ch = (double)__double2half(ldexp(round_bits(cs, hb), 14));
  const double sh = (double)__double2half(ldexp(round_bits(sn, hb), 14));
  const __half2 v = pc == 0 ? __halves2half2(__double2half(ch), __double2half(sh))
                            : __halves2half2(__double2half(ldexp(cs, 14) - ch), __double2half(ldexp(sn, 14) - sh));
  *reinterpret_cast<__half2*>(trig + o * kRopeTrigRow + ((kt * 4 + tig) * 2 + pc) * 16 + 4 * e) = v;
  if (idx == 0) {  // the tag in row 0's padding: which code width the pieces were cut for
    uint32_t* tag = reinterpret_cast<uint32_t*>(trig + kRopeTrigTagOffset);
    tag[0] = kRopeTrigTag;
    tag[1] = (uint32_t)(11 - hb);
  }
}

inline size_t rope_trig_offset(const kvq_cache* c) {
  return (size_t)(64 + rope_blocks(c)) * (c->head_dim / 2) * sizeof(float2);
}

}  // namespace kvq

extern "C" kvq_status kvq_rope_table_bytes(const kvq_cache* c, size_t* bytes) {
  using namespace kvq;
  kvq_status s = validate_geometry(c);
  if (s != KVQ_OK) return s;
  if (bytes == nullptr) return KVQ_ERR_INVALID;
  if (c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  *bytes = rope_trig_offset(c) + kRopeTrigBytes;
  return KVQ_OK;
}

extern "C" kvq_status kvq_rope_table(const kvq_cache* c, float base, float* table, void* stream) {
  using namespace kvq;
  kvq_status s = validate_geometry(c);
  if (s != KVQ_OK) return s;
  if (c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (table == nullptr || !aligned(table, 16) || !(base > 1.f) || !std::isfinite(base)) return KVQ_ERR_INVALID;
  const int rows = 64 + rope_blocks(c), half = c->head_dim / 2;
  const int64_t n = (int64_t)rows * half;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(reinterpret_cast<float2*>(table), half, rows,
                                                                (double)base);
  uint8_t* trig = reinterpret_cast<uint8_t*>(table) + rope_trig_offset(c);
  if (cudaMemsetAsync(trig, 0, kRopeTrigBytes, st) != cudaSuccess) return KVQ_ERR_CUDA;  // row padding
  constexpr int kSlots = kRopeTrigRows * 8 * 4 * 2 * 4;
  rope_trig_kernel<<<(kSlots + 255) / 256, 256, 0, st>>>(trig, half, (double)base, 11 - c->bits);
  return launch_status();
}

extern "C" kvq_status kvq_decode_attn_rope(const kvq_cache* c, int32_t n_q_heads, const void* q, float* out,
                                           float sm_scale, const float* table, size_t table_bytes,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  using namespace kvq;
  kvq_status s = validate_cache(c);
  if (s != KVQ_OK) return s;
  if (c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  int G = 0;
  s = validate_q_heads(c, n_q_heads, &G);
  if (s != KVQ_OK) return s;
  if (q == nullptr || out == nullptr || workspace == nullptr || table == nullptr) return KVQ_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(out, 16) || !aligned(workspace, 16) || !aligned(table, 16))
    return KVQ_ERR_INVALID;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID;
  if (table_bytes < rope_trig_offset(c) + kRopeTrigBytes) return KVQ_ERR_INVALID;
  int err = 0;
  int n = 0;
#define KVQ_RSLOTS(B_, G_) \
  if (c->bits == B_ && G == G_) n = DecodeLaunch<128, B_, G_, true>::slots(&err);
  KVQ_RSLOTS(2, 1) KVQ_RSLOTS(2, 2) KVQ_RSLOTS(2, 4) KVQ_RSLOTS(2, 8)
  KVQ_RSLOTS(4, 1) KVQ_RSLOTS(4, 2) KVQ_RSLOTS(4, 4) KVQ_RSLOTS(4, 8)
  KVQ_RSLOTS(8, 1) KVQ_RSLOTS(8, 2) KVQ_RSLOTS(8, 4) KVQ_RSLOTS(8, 8)
#undef KVQ_RSLOTS
  if (err || n == 0) return KVQ_ERR_CUDA;
  const DecodeLayout L = decode_layout(c, G, n);
  if (workspace_bytes < L.total) return KVQ_ERR_INVALID;
  DecodeParams p = decode_params(c, q, out, sm_scale, static_cast<uint8_t*>(workspace), L, table);
  p.rope_trig = reinterpret_cast<const uint8_t*>(table) + rope_trig_offset(c);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->bits == 2) return decode_dispatch_g<128, 2, true>(G, p, st);
  if (c->bits == 4) return decode_dispatch_g<128, 4, true>(G, p, st);
  return decode_dispatch_g<128, 8, true>(G, p, st);
}
