// Shared device code of the kvq library: the group quantizer, the packed tile
// layout and thin PTX wrappers.  sm_103a only.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kGroup = KVQ_GROUP;
// Online softmax: the running maximum (log2 domain) is only moved, and the
// accumulators rescaled, when a chunk's maximum exceeds it by more than this;
// the weights p~ = exp2(logit - max) then stay below 2^4 = 16 (exact after the
// final normalisation, which uses the same reference).
constexpr float kLazyRescale = 4.f;

// ---------------------------------------------------------------------------
// Group quantizer ("KV-cache quantization axes", ihal.it, paragraph 3: the
// group's range is divided into the 2^b levels of the code, one scale and one
// zero point per group).  Every fp32 operation is an explicit round-to-nearest
// intrinsic so the result is bit-identical to an IEEE fp32 evaluation.
// ---------------------------------------------------------------------------
struct GroupParams {
  __half scale_h;
  __half zero_h;
  float scale;  // fp32 value of the stored fp16 scale
  float zero;   // fp32 value of the stored fp16 zero point
  float inv;    // fp32 reciprocal of scale (round to nearest), 0 when scale is 0
};

// levels = 2^b - 1 (3, 15 or 255: exact in fp32)
__device__ __forceinline__ GroupParams group_params_levels(float mn, float mx, float levels) {
  const float rng = __fsub_rn(mx, mn);
  const float sc = __fdiv_rn(rng, levels);
  GroupParams p;
  p.scale_h = __float2half_rn(sc);
  p.zero_h = __float2half_rn(mn);  // exact: mn is an fp16 value
  p.scale = __half2float(p.scale_h);
  p.zero = __half2float(p.zero_h);
  if (p.scale == 0.f) { p.scale_h = __float2half_rn(0.f); p.scale = 0.f; }  // -0 -> +0
  if (p.zero == 0.f) { p.zero_h = __float2half_rn(0.f); p.zero = 0.f; }
  p.inv = p.scale == 0.f ? 0.f : __frcp_rn(p.scale);
  return p;
}

template <int BITS>
__device__ __forceinline__ GroupParams group_params(float mn, float mx) {
  return group_params_levels(mn, mx, (float)((1 << BITS) - 1));
}

// code = clamp(rint(fl(d / scale))), d = fl(x - zero), every op round-to-nearest.
// Fast path: y = d * fl(1/scale), the exact product inside an FMA.  With Q = d /
// scale exact, y and the rounded quotient fl(Q) each lie within 2^-24 |Q| (1 + e)
// of Q, and 0 <= Q < 2^9 here (d <= max - min and scale is that range over 2^b - 1,
// up to fp16 rounding of the scale), so |y - fl(Q)| < 2^-14: y rounds to the same
// integer as fl(Q) unless y is within 2^-14 of a half-integer.  Those rare y (window
// 2^-11, eight times the bound) take the exact IEEE division, so the code is
// bit-identical to the division.
// Rounding to an integer, ties to even: for 0 <= y < 2^22, fma(d, inv, 1.5 * 2^23)
// rounds y + 1.5 * 2^23 once to a whole number (the sum's ulp is 1), and its low
// mantissa bits are that number; fma(d, inv, -that number) is y's distance to it.
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4B400000u;
// The code clamped to [0, cmax] (cmax = 2^b - 1) from y = d * inv, and whether y
// lies in the window near a half-integer where the exact quotient must decide.
// No branch: a zero scale has inv = 0, so y = 0 and the code is 0.
__device__ __forceinline__ uint32_t quant_code_fast(float x, const GroupParams& p, uint32_t cmax, bool& near_tie) {
  const float d = __fsub_rn(x, p.zero);  // >= 0
  const float t = __fmaf_rn(d, p.inv, kRoundMagic);
  near_tie = fabsf(__fmaf_rn(d, p.inv, -__fsub_rn(t, kRoundMagic))) > 0.5f - 0x1p-11f;
  const uint32_t c = __float_as_uint(t) - kRoundMagicBits;
  return c > cmax ? cmax : c;
}

// The code from the exactly rounded quotient fl(d / scale).
__device__ __forceinline__ uint32_t quant_code_exact(float x, float scale, float zero, uint32_t cmax) {
  if (scale == 0.f) return 0u;
  const float q = __fdiv_rn(__fsub_rn(x, zero), scale);
  const uint32_t c = __float_as_uint(__fadd_rn(q, kRoundMagic)) - kRoundMagicBits;
  return c > cmax ? cmax : c;
}

// ---------------------------------------------------------------------------
// Packed tile layout (see kvq.h).  Lane L (gid = L/4, tig = L%4) owns D/2 code
// pairs; pair P lives in the lane's word P/(16/BITS), slot P%(16/BITS).
// ---------------------------------------------------------------------------
template <int D, int BITS>
struct Tile {
  static constexpr int kBytes = kGroup * D * BITS / 8;   // bytes per tile
  static constexpr int kWordsPerLane = D * BITS / 32;     // >= 4
  static constexpr int kChunksPerLane = kWordsPerLane / 4;  // 16-byte chunks
  static constexpr int kPairsPerWord = 16 / BITS;
  static_assert(kWordsPerLane % 4 == 0, "a lane owns whole 16-byte chunks");
};

// Bit position (within each 16-bit half of a word) of the codes in slot k.  For
// 2-bit codes slots 0..7 sit at 0,2,8,10,4,6,12,14: the slots of fragment
// registers 0 and 2 (one row, both k-halves) share a position after a shift
// right by 8 of the second, as do those of registers 1 and 3.
template <int BITS>
__host__ __device__ constexpr int slot_bitpos(int k) {
  return BITS == 2 ? 2 * (k & 1) + 8 * ((k >> 1) & 1) + 4 * (k >> 2) : BITS * k;
}

// (token, channel) of the FIRST code of key pair P of a lane; the second code is
// at channel + 1.
__device__ __forceinline__ void key_pair_pos(int P, int gid, int tig, int& t, int& c) {
  const int kt = P >> 3, mt = (P >> 2) & 1, i = P & 3;
  t = 16 * mt + gid + 8 * (i & 1);
  c = 16 * kt + 2 * tig + 8 * (i >> 1);
}

// (token, channel) of the FIRST code of value pair P; the second is at token + 1.
__device__ __forceinline__ void value_pair_pos(int P, int gid, int tig, int& t, int& c) {
  const int mt = P >> 3, kt = (P >> 2) & 1, i = P & 3;
  c = 16 * mt + gid + 8 * (i & 1);
  t = 16 * kt + 2 * tig + 8 * (i >> 1);
}

// Pack chunk ch (the lane's words 4ch .. 4ch + 3) of a 32 x D tile of codes held
// in shared memory (ct[t * PITCH + c]) and store it to global memory with one
// 16-byte store (a warp's 32 lanes write 512 contiguous bytes).
template <int D, int BITS, bool IS_KEY, int PITCH = D>
__device__ __forceinline__ void pack_store_chunk(const uint8_t* ct, uint8_t* dst, int lane, int ch) {
  using T = Tile<D, BITS>;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k4 = 0; k4 < 4 * T::kPairsPerWord; ++k4) {
    const int P = ch * 4 * T::kPairsPerWord + k4;
    int t, c;
    uint32_t first, second;
    if (IS_KEY) {
      key_pair_pos(P, gid, tig, t, c);  // c even: the pair is one 16-bit word
      const uint32_t pr = *reinterpret_cast<const uint16_t*>(ct + t * PITCH + c);
      first = pr & 0xFFu;
      second = pr >> 8;
    } else {
      value_pair_pos(P, gid, tig, t, c);
      first = ct[t * PITCH + c];
      second = ct[(t + 1) * PITCH + c];
    }
    const int k = k4 % T::kPairsPerWord;
    w[k4 / T::kPairsPerWord] |= (first << slot_bitpos<BITS>(k)) | (second << (16 + slot_bitpos<BITS>(k)));
  }
  *reinterpret_cast<uint4*>(dst + (size_t)(ch * 32 + lane) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Pack a whole 32 x D tile (every chunk of the lane).
template <int D, int BITS, bool IS_KEY, int PITCH = D>
__device__ __forceinline__ void pack_store_tile(const uint8_t* ct, uint8_t* dst, int lane) {
#pragma unroll
  for (int ch = 0; ch < Tile<D, BITS>::kChunksPerLane; ++ch) pack_store_chunk<D, BITS, IS_KEY, PITCH>(ct, dst, lane, ch);
}

// Metadata blocks are stored as fp16 pairs in "lane order" (see kvq.h): key
// word w = 16kt + 4tig + 2r + f holds the zero points (f = 0) or the scales
// (f = 1) of channels 16kt + 2tig + 8r and +1; pair p of a value plane holds
// tokens 16kt + 2tig + 8r (+1) of channel group j = p/16 with tig = p%16/4,
// kt = (p%4)/2, r = p%2.  The natural-order planes (nat[2][D]: scales, then
// zero points) are staged in shared memory and written out permuted.
template <int D, bool IS_KEY>
__device__ __forceinline__ void store_meta_lane_order(const __half* nat, __half* dst, int lane) {
  constexpr int PAIRS = D / 2, PER_LANE = PAIRS / 32;
  const uint16_t* n16 = reinterpret_cast<const uint16_t*>(nat);
  uint32_t* d32 = reinterpret_cast<uint32_t*>(dst);
  if (IS_KEY) {
    // word w = 16 kt + 4 tig + 2 r + f: the zero points (f = 0, nat[D + c]) or the
    // scales (f = 1, nat[c]) of channels c = 16 kt + 2 tig + 8 r and c + 1
#pragma unroll
    for (int e = 0; e < 2 * PER_LANE; ++e) {
      const int w = lane * 2 * PER_LANE + e;
      const int kt = w >> 4, tig = (w >> 2) & 3, r = (w >> 1) & 1, f = w & 1;
      const int c = 16 * kt + 2 * tig + 8 * r, base = f ? 0 : D;
      d32[w] = (uint32_t)n16[base + c] | ((uint32_t)n16[base + c + 1] << 16);
    }
    return;
  }
#pragma unroll
  for (int plane = 0; plane < 2; ++plane) {
#pragma unroll
    for (int e = 0; e < PER_LANE; ++e) {
      const int p = lane * PER_LANE + e;
      const int tig = (p % 16) / 4, w = p % 4, r = w % 2;
      const int idx = kGroup * (p / 16) + 16 * (w / 2) + 2 * tig + 8 * r;
      const uint32_t lo = n16[plane * D + idx], hi = n16[plane * D + idx + 1];
      d32[plane * PAIRS + p] = lo | (hi << 16);
    }
  }
}

// ---------------------------------------------------------------------------
// PTX wrappers.
// ---------------------------------------------------------------------------
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col); fragment layouts per
// the PTX ISA's mma.m16n8k16 tables.
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held by the warp (lane i: row i/4,
// columns 2(i%4), 2(i%4)+1, the low half first) in registers.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
// 16-byte copy that reads src_bytes (0 or 16) bytes and zero-fills the rest.
__device__ __forceinline__ void cp_async_16_zfill(void* smem, const void* gmem, int src_bytes) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_8(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
}
// Four 8x8 b16 matrices; lane i supplies the row address of row i%8 of matrix i/8.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem_row) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem_row);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* smem_row) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem_row);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---- TMA bulk copies completing on an mbarrier (shared memory, this CTA)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// L2 policy for data read once (the streamed cache): evicted first, so that it
// does not push out the small data every launch re-reads (lengths, q, partials).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// Bulk copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void tma_load_1d_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Wait for the phase with the given parity to complete, giving up after
// `max_polls` polls (each poll may suspend the thread for a short while).
// Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_polls) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < max_polls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Device-scope atomic add with acquire-release semantics: the caller's earlier
// writes (and, after a CTA barrier, those of its CTA) are visible to whoever
// acquires the new value, and writes released before the old value are visible
// to the caller.  Returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Order this thread's generic-proxy view of global memory before its later
// bulk (async-proxy) copies from global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

// 2^x with the hardware approximation (relative error about 2^-22; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

}  // namespace kvq
