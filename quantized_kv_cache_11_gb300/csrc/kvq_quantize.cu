// Prefill quantization and per-token append (with the 32-token flush) of the
// uniform cache.  One warp quantizes one 32-token tile of keys (per channel)
// and values (per token) and writes packed codes and fp16 metadata in one
// coalesced pass.
#include "kvq_common.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kPrefillWarps = 4;
// append: tile groups per block; a group of D/32 warps flushes one head's oldest
// 32 tail tokens together (the flush is on the decode step's critical path)
constexpr int kAppendGroups = 8;

struct PrefillParams {
  const __half* k;
  const __half* v;
  int64_t sb, st, sh;
  uint8_t* k_codes;
  uint8_t* v_codes;
  __half* k_meta;
  __half* v_meta;
  __half* k_tail;
  __half* v_tail;
  int32_t* n_quant;
  int32_t* n_tail;
  int32_t* tail_head;
  __half* k_sink;
  __half* v_sink;
  int32_t* n_sink;
  int32_t hkv, max_groups, tail_cap, sink_cap;
  int32_t seq_len[KVQ_MAX_BATCH];
  int32_t ntail[KVQ_MAX_BATCH];
};

// One warp quantizes one 32-token tile of keys and values whose rows it stages in
// shared memory (cp.async, VEC bytes per copy; keys first, then the values in the
// same buffer, so that twice as many warps fit an SM).  Keys: each lane owns
// D/32 channels (fp16 min/max over the 32 rows, then the codes); values: lane t
// owns token t (min/max and parameters of its D/32 groups, then the codes).  The
// codes go through a staging tile at a padded pitch (no bank conflicts) and are
// packed into the fragment layout.
template <int D>
struct StagedTile {
  static constexpr int PH = D + 8;   // halves per staged row (16-byte aligned rows)
  static constexpr int PC = D + 8;   // bytes per row of the code staging tile
  static constexpr int ROWS = kGroup * PH * 2;
  static constexpr int BYTES = ROWS + kGroup * PC + 8 * D;  // rows (keys, then values), codes, key + value meta
};

template <int D, int BITS, int VEC>
__device__ __forceinline__ void quantize_tile_staged(const __half* ksrc, const __half* vsrc, int64_t tstride,
                                                     uint8_t* kcodes_dst, __half* kmeta_dst, uint8_t* vcodes_dst,
                                                     __half* vmeta_dst, uint8_t* ws, int lane) {
  using S = StagedTile<D>;
  __half* kr = reinterpret_cast<__half*>(ws);
  __half* vr = kr;  // the value rows replace the key rows
  uint8_t* ct = ws + S::ROWS;
  __half* km = reinterpret_cast<__half*>(ws + S::ROWS + kGroup * S::PC);
  __half* vm = km + 2 * D;
  constexpr int CPR = 2 * D / VEC;  // copies per row
  auto stage = [&](__half* dst, const __half* src) {
#pragma unroll 4
    for (int e = lane; e < kGroup * CPR; e += 32) {
      const int t = e / CPR, ch = e % CPR;
      if (VEC == 16) cp_async_16(dst + t * S::PH + ch * 8, src + (int64_t)t * tstride + ch * 8);
      else cp_async_8(dst + t * S::PH + ch * 4, src + (int64_t)t * tstride + ch * 4);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
  };
  stage(kr, ksrc);  // ---- the 32 key rows
  // ---- keys: per channel over the 32 tokens; lane owns channels [c0, c0 + CPL)
  {
    constexpr int CPL = D / 32, NH = CPL / 2;  // channels, half2 pairs per lane
    const int c0 = lane * CPL;
    __half2 mn[NH], mx[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) mn[j] = mx[j] = *reinterpret_cast<const __half2*>(kr + c0 + 2 * j);
#pragma unroll 8
    for (int t = 1; t < kGroup; ++t)
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const __half2 x = *reinterpret_cast<const __half2*>(kr + t * S::PH + c0 + 2 * j);
        mn[j] = __hmin2(mn[j], x);
        mx[j] = __hmax2(mx[j], x);
      }
    GroupParams gp[CPL];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      gp[2 * j] = group_params<BITS>(__low2float(mn[j]), __low2float(mx[j]));
      gp[2 * j + 1] = group_params<BITS>(__high2float(mn[j]), __high2float(mx[j]));
    }
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      km[c0 + j] = gp[j].scale_h;
      km[D + c0 + j] = gp[j].zero_h;
    }
    constexpr uint32_t cmax = (1u << BITS) - 1u;
    // codes without a branch; bit t of `redo`: a code of token t lies near a
    // rounding tie, and the token's codes are redone with the exact quotient
    uint32_t redo = 0u;
#pragma unroll 4
    for (int t = 0; t < kGroup; ++t) {
      // the codes (each <= 255) gathered into bytes by byte permutes: three per
      // four codes, against three shifts and two ORs
      uint32_t h16[NH];  // codes of channel pair j in bytes 0 and 1
      bool near = false;
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const __half2 x = *reinterpret_cast<const __half2*>(kr + t * S::PH + c0 + 2 * j);
        bool n0, n1;
        const uint32_t a = quant_code_fast(__low2float(x), gp[2 * j], cmax, n0);
        const uint32_t b = quant_code_fast(__high2float(x), gp[2 * j + 1], cmax, n1);
        h16[j] = __byte_perm(a, b, 0x0040);
        near = near || n0 || n1;
      }
      const uint32_t w = NH == 2 ? __byte_perm(h16[0], h16[NH - 1], 0x5410) : h16[0];
      redo |= (uint32_t)near << t;
      if (CPL == 4) *reinterpret_cast<uint32_t*>(ct + t * S::PC + c0) = w;
      else *reinterpret_cast<uint16_t*>(ct + t * S::PC + c0) = (uint16_t)w;
    }
#pragma unroll 1
    while (redo != 0u) {
      const int t = __ffs(redo) - 1;
      redo &= redo - 1u;
#pragma unroll
      for (int j = 0; j < CPL; ++j)
        ct[t * S::PC + c0 + j] = (uint8_t)quant_code_exact(__half2float(kr[t * S::PH + c0 + j]), gp[j].scale,
                                                           gp[j].zero, cmax);
    }
  }
  __syncwarp();
  pack_store_tile<D, BITS, true, S::PC>(ct, kcodes_dst, lane);
  store_meta_lane_order<D, true>(km, kmeta_dst, lane);
  __syncwarp();
  stage(vr, vsrc);  // ---- the 32 value rows
  // ---- values: per token over 32-channel groups; lane t owns token t
  {
    const int t = lane;
    // rolled: the unrolled code no longer fits the instruction cache well (measured:
    // 128k prefill 215.8 -> 194.5 us)
#pragma unroll 1
    for (int j = 0; j < D / 32; ++j) {
      const uint4* row = reinterpret_cast<const uint4*>(vr + t * S::PH + 32 * j);
      uint4 x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = row[i];
      const __half2* h = reinterpret_cast<const __half2*>(x);
      __half2 mn = h[0], mx = h[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        mn = __hmin2(mn, h[i]);
        mx = __hmax2(mx, h[i]);
      }
      const GroupParams gp = group_params<BITS>(fminf(__low2float(mn), __high2float(mn)),
                                                fmaxf(__low2float(mx), __high2float(mx)));
      vm[j * kGroup + t] = gp.scale_h;
      vm[D + j * kGroup + t] = gp.zero_h;
      constexpr uint32_t cmax = (1u << BITS) - 1u;
      // bit w4 of `redo`: one of the four codes of word w4 lies near a rounding
      // tie; those words are redone with the exact quotient
      uint32_t redo = 0u;
#pragma unroll
      for (int w4 = 0; w4 < 8; ++w4) {
        bool n0, n1, n2, n3;
        const uint32_t c0 = quant_code_fast(__low2float(h[2 * w4]), gp, cmax, n0);
        const uint32_t c1 = quant_code_fast(__high2float(h[2 * w4]), gp, cmax, n1);
        const uint32_t c2 = quant_code_fast(__low2float(h[2 * w4 + 1]), gp, cmax, n2);
        const uint32_t c3 = quant_code_fast(__high2float(h[2 * w4 + 1]), gp, cmax, n3);
        redo |= (uint32_t)(n0 || n1 || n2 || n3) << w4;
        *reinterpret_cast<uint32_t*>(ct + t * S::PC + 32 * j + 4 * w4) = pack4_bytes(c0, c1, c2, c3);
      }
#pragma unroll 1
      while (redo != 0u) {
        const int w4 = __ffs(redo) - 1;
        redo &= redo - 1u;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ct[t * S::PC + 32 * j + 4 * w4 + e] =
              (uint8_t)quant_code_exact(__half2float(vr[t * S::PH + 32 * j + 4 * w4 + e]), gp.scale, gp.zero, cmax);
      }
    }
  }
  __syncwarp();
  pack_store_tile<D, BITS, false, S::PC>(ct, vcodes_dst, lane);
  store_meta_lane_order<D, false>(vm, vmeta_dst, lane);
  __syncwarp();
}

// grid (work items / warps, Hkv, B); a work item is a 32-token tile to quantize
// or a chunk of up to 32 tail tokens to copy.
template <int D, int BITS, int VEC>
__global__ void __launch_bounds__(kPrefillWarps * 32)
prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ __align__(16) uint8_t s_stage[];  // StagedTile<D>::BYTES per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int item = blockIdx.x * kPrefillWarps + warp;
  const int seq = p.seq_len[b], nt = p.ntail[b];
  const int ns = min(p.sink_cap, seq);  // sink tokens [0, ns)
  const int nq = seq - ns - nt, ng = nq / kGroup;
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
    p.n_quant[b] = nq;
    p.n_tail[b] = nt;
    p.tail_head[b] = 0;
    if (p.sink_cap > 0) p.n_sink[b] = ns;
  }
  const size_t bh = (size_t)b * p.hkv + h;
  const __half* kseq = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
  const __half* vseq = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;
  if (item < ng) {
    using T = Tile<D, BITS>;
    const size_t gi = bh * p.max_groups + item;
    quantize_tile_staged<D, BITS, VEC>(kseq + (int64_t)(ns + item * kGroup) * p.st,
                                       vseq + (int64_t)(ns + item * kGroup) * p.st,
                                       p.st, p.k_codes + gi * T::kBytes, p.k_meta + gi * 2 * D,
                                       p.v_codes + gi * T::kBytes, p.v_meta + gi * 2 * D,
                                       s_stage + warp * StagedTile<D>::BYTES, lane);
  } else {
    // fp16 row copies: tail tokens [ns + nq + 32c, ...) to ring slots 32c..
    // (ring head 0), then sink tokens [32c', ...) to sink rows 32c'..
    const int ct = (nt + kGroup - 1) / kGroup, cs = (ns + kGroup - 1) / kGroup;
    const int c = item - ng;
    if (c >= ct + cs) return;
    const bool tail = c < ct;
    const int first = tail ? 32 * c : 32 * (c - ct), count = tail ? nt : ns;
    const int src0 = tail ? ns + nq : 0;
    const int cap = tail ? p.tail_cap : p.sink_cap;
    __half* kd = tail ? p.k_tail : p.k_sink;
    __half* vd = tail ? p.v_tail : p.v_sink;
    constexpr int CPL = D / 32;
    for (int i = first; i < min(count, first + 32); ++i) {
      const int64_t src = (int64_t)(src0 + i) * p.st + lane * CPL;
      const size_t dst = (bh * cap + i) * D + lane * CPL;
      if (CPL == 4) {
        *reinterpret_cast<uint2*>(kd + dst) = *reinterpret_cast<const uint2*>(kseq + src);
        *reinterpret_cast<uint2*>(vd + dst) = *reinterpret_cast<const uint2*>(vseq + src);
      } else {
        *reinterpret_cast<uint32_t*>(kd + dst) = *reinterpret_cast<const uint32_t*>(kseq + src);
        *reinterpret_cast<uint32_t*>(vd + dst) = *reinterpret_cast<const uint32_t*>(vseq + src);
      }
    }
  }
}

// The tile of quantize_tile_staged quantized by the D/32 warps of a group
// together (wi: the warp's index in the group, bar: the group's named barrier):
// keys one channel per thread; values the 32-channel group wi, one token per
// lane; the packing split by 16-byte chunk.  The arithmetic is the same, so the
// bytes are identical.  Every staged row has been read when it returns.
template <int D, int BITS>
__device__ __forceinline__ void quantize_tile_coop(const __half* ksrc, const __half* vsrc, int64_t tstride,
                                                   uint8_t* kcodes_dst, __half* kmeta_dst, uint8_t* vcodes_dst,
                                                   __half* vmeta_dst, uint8_t* ws, int wi, int lane, int bar) {
  using S = StagedTile<D>;
  using T = Tile<D, BITS>;
  constexpr int W = D / 32, NTH = W * 32;
  constexpr uint32_t cmax = (1u << BITS) - 1u;
  __half* rows = reinterpret_cast<__half*>(ws);  // key rows, then value rows
  uint8_t* ct = ws + S::ROWS;
  __half* km = reinterpret_cast<__half*>(ws + S::ROWS + kGroup * S::PC);
  __half* vm = km + 2 * D;
  const int tid = wi * 32 + lane;
  auto sync = [&]() { asm volatile("bar.sync %0, %1;\n" ::"r"(bar), "r"(NTH) : "memory"); };
  auto stage = [&](const __half* src) {
    constexpr int CPR = 2 * D / 16;  // 16-byte copies per row
    for (int e = tid; e < kGroup * CPR; e += NTH) {
      const int t = e / CPR, ch = e % CPR;
      cp_async_16(rows + t * S::PH + ch * 8, src + (int64_t)t * tstride + ch * 8);
    }
    cp_async_commit();
    cp_async_wait<0>();
    sync();
  };
  stage(ksrc);
  {  // keys: channel tid over the 32 tokens
    const int c = tid;
    __half mn = rows[c], mx = mn;
#pragma unroll 8
    for (int t = 1; t < kGroup; ++t) {
      const __half x = rows[t * S::PH + c];
      mn = __hmin(mn, x);
      mx = __hmax(mx, x);
    }
    const GroupParams gp = group_params<BITS>(__half2float(mn), __half2float(mx));
    km[c] = gp.scale_h;
    km[D + c] = gp.zero_h;
    uint32_t redo = 0u;  // bit t: the code of token t lies near a rounding tie
#pragma unroll 8
    for (int t = 0; t < kGroup; ++t) {
      bool near;
      ct[t * S::PC + c] = (uint8_t)quant_code_fast(__half2float(rows[t * S::PH + c]), gp, cmax, near);
      redo |= (uint32_t)near << t;
    }
#pragma unroll 1
    while (redo != 0u) {
      const int t = __ffs(redo) - 1;
      redo &= redo - 1u;
      ct[t * S::PC + c] = (uint8_t)quant_code_exact(__half2float(rows[t * S::PH + c]), gp.scale, gp.zero, cmax);
    }
  }
  sync();
  for (int ch = wi; ch < T::kChunksPerLane; ch += W) pack_store_chunk<D, BITS, true, S::PC>(ct, kcodes_dst, lane, ch);
  if (wi == W - 1) store_meta_lane_order<D, true>(km, kmeta_dst, lane);
  sync();  // the rows and codes buffers are free again
  stage(vsrc);
  {  // values: group j = wi of token t = lane
    const int t = lane, j = wi;
    const uint4* row = reinterpret_cast<const uint4*>(rows + t * S::PH + 32 * j);
    uint4 x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = row[i];
    const __half2* h = reinterpret_cast<const __half2*>(x);
    __half2 mn = h[0], mx = h[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      mn = __hmin2(mn, h[i]);
      mx = __hmax2(mx, h[i]);
    }
    const GroupParams gp = group_params<BITS>(fminf(__low2float(mn), __high2float(mn)),
                                              fmaxf(__low2float(mx), __high2float(mx)));
    vm[j * kGroup + t] = gp.scale_h;
    vm[D + j * kGroup + t] = gp.zero_h;
    uint32_t redo = 0u;  // bit w4: a code of word w4 lies near a rounding tie
#pragma unroll
    for (int w4 = 0; w4 < 8; ++w4) {
      bool n0, n1, n2, n3;
      const uint32_t c0 = quant_code_fast(__low2float(h[2 * w4]), gp, cmax, n0);
      const uint32_t c1 = quant_code_fast(__high2float(h[2 * w4]), gp, cmax, n1);
      const uint32_t c2 = quant_code_fast(__low2float(h[2 * w4 + 1]), gp, cmax, n2);
      const uint32_t c3 = quant_code_fast(__high2float(h[2 * w4 + 1]), gp, cmax, n3);
      redo |= (uint32_t)(n0 || n1 || n2 || n3) << w4;
      *reinterpret_cast<uint32_t*>(ct + t * S::PC + 32 * j + 4 * w4) = pack4_bytes(c0, c1, c2, c3);
    }
#pragma unroll 1
    while (redo != 0u) {
      const int w4 = __ffs(redo) - 1;
      redo &= redo - 1u;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        ct[t * S::PC + 32 * j + 4 * w4 + e] =
            (uint8_t)quant_code_exact(__half2float(rows[t * S::PH + 32 * j + 4 * w4 + e]), gp.scale, gp.zero, cmax);
    }
  }
  sync();
  for (int ch = wi; ch < T::kChunksPerLane; ch += W) pack_store_chunk<D, BITS, false, S::PC>(ct, vcodes_dst, lane, ch);
  if (wi == W - 1) store_meta_lane_order<D, false>(vm, vmeta_dst, lane);
  sync();  // the group's buffers may be reused
}

struct AppendParams {
  const __half* k_new;
  const __half* v_new;
  uint8_t* k_codes;
  uint8_t* v_codes;
  __half* k_meta;
  __half* v_meta;
  __half* k_tail;
  __half* v_tail;
  int32_t* n_quant;
  int32_t* n_tail;
  int32_t* tail_head;
  int32_t* error_flags;
  __half* k_sink;
  __half* v_sink;
  int32_t* n_sink;
  int32_t hkv, max_groups, tail_cap, sink_cap;
};

// grid (B); each block owns one sequence so the length update is race-free.
// kAppendGroups groups of D/32 warps; group g handles heads g, g + kAppendGroups, ...
template <int D, int BITS>
__global__ void __launch_bounds__(kAppendGroups * D) append_kernel(const AppendParams p) {
  extern __shared__ __align__(16) uint8_t s_stage[];  // StagedTile<D>::BYTES per group
  constexpr int W = D / 32, NWARPS = kAppendGroups * W;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wi = warp % W;
  const int b = blockIdx.x;
  const int R = p.tail_cap;
  const int nq = p.n_quant[b], nt = p.n_tail[b], hd = p.tail_head[b];
  const int ns = p.sink_cap > 0 ? p.n_sink[b] : 0;
  if (p.sink_cap > 0 && ns < p.sink_cap) {
    // the sink window is not full: the token becomes sink row ns (nothing may
    // follow the sinks yet)
    if (ns < 0 || nq != 0 || nt != 0) {
      if (threadIdx.x == 0 && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_BAD_LENGTHS);
      return;
    }
    constexpr int CPL = D / 32;
    for (int h = warp; h < p.hkv; h += NWARPS) {
      const size_t bh = (size_t)b * p.hkv + h;
      const size_t src = bh * D + lane * CPL, dst = (bh * p.sink_cap + ns) * D + lane * CPL;
      for (int i = 0; i < CPL; ++i) {
        p.k_sink[dst + i] = p.k_new[src + i];
        p.v_sink[dst + i] = p.v_new[src + i];
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) p.n_sink[b] = ns + 1;
    return;
  }
  const bool sane = nq >= 0 && nq % kGroup == 0 && nq / kGroup <= p.max_groups && nt >= 0 &&
                    nt <= R && hd >= 0 && hd < R && hd % kGroup == 0 && ns == p.sink_cap;
  const bool flush = sane && nt == R;
  const bool fits = !flush || nq / kGroup < p.max_groups;
  if (!sane || !fits) {
    if (threadIdx.x == 0 && p.error_flags != nullptr)
      atomicOr(p.error_flags, sane ? KVQ_DEVERR_APPEND_CAPACITY : KVQ_DEVERR_BAD_LENGTHS);
    return;
  }
  const int hd2 = flush ? (hd + kGroup) % R : hd;
  const int nt2 = flush ? nt - kGroup : nt;
  const int slot = (hd2 + nt2) % R;
  constexpr int CPL = D / 32;
  for (int h = grp; h < p.hkv; h += kAppendGroups) {
    const size_t bh = (size_t)b * p.hkv + h;
    __half* kt = p.k_tail + bh * R * D;
    __half* vt = p.v_tail + bh * R * D;
    if (flush) {
      // the oldest 32 tail tokens sit in ring slots hd .. hd + 31 (hd and R are
      // multiples of 32): contiguous, 16-byte aligned rows
      using T = Tile<D, BITS>;
      const size_t gi = bh * p.max_groups + nq / kGroup;
      quantize_tile_coop<D, BITS>(kt + (size_t)hd * D, vt + (size_t)hd * D, D, p.k_codes + gi * T::kBytes,
                                  p.k_meta + gi * 2 * D, p.v_codes + gi * T::kBytes, p.v_meta + gi * 2 * D,
                                  s_stage + grp * StagedTile<D>::BYTES, wi, lane, 1 + grp);
    }
    // the new token (after a flush into slot hd, whose row the flush has read)
    if (wi != 0) continue;
    const size_t src = bh * D + lane * CPL;
    const size_t dst = (size_t)slot * D + lane * CPL;
    if (CPL == 4) {
      *reinterpret_cast<uint2*>(kt + dst) = *reinterpret_cast<const uint2*>(p.k_new + src);
      *reinterpret_cast<uint2*>(vt + dst) = *reinterpret_cast<const uint2*>(p.v_new + src);
    } else {
      *reinterpret_cast<uint32_t*>(kt + dst) = *reinterpret_cast<const uint32_t*>(p.k_new + src);
      *reinterpret_cast<uint32_t*>(vt + dst) = *reinterpret_cast<const uint32_t*>(p.v_new + src);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.n_quant[b] = nq + (flush ? kGroup : 0);
    p.n_tail[b] = nt2 + 1;
    p.tail_head[b] = hd2;
  }
}

template <template <int, int> class F, typename... A>
kvq_status dispatch_db(int d, int bits, A&&... args) {
  if (d == 128) {
    if (bits == 2) return F<128, 2>::run(args...);
    if (bits == 4) return F<128, 4>::run(args...);
    if (bits == 8) return F<128, 8>::run(args...);
  } else if (d == 64) {
    if (bits == 2) return F<64, 2>::run(args...);
    if (bits == 4) return F<64, 4>::run(args...);
    if (bits == 8) return F<64, 8>::run(args...);
  }
  return KVQ_ERR_UNSUPPORTED;
}

template <int D, int BITS>
struct PrefillLaunch {
  template <int VEC>
  static kvq_status launch(const PrefillParams& p, dim3 grid, cudaStream_t s) {
    constexpr int smem = kPrefillWarps * StagedTile<D>::BYTES;
    if (!device_smem_attr(reinterpret_cast<const void*>(prefill_kernel<D, BITS, VEC>), smem)) return KVQ_ERR_CUDA;
    prefill_kernel<D, BITS, VEC><<<grid, kPrefillWarps * 32, smem, s>>>(p);
    return launch_status();
  }
  static kvq_status run(const PrefillParams& p, int batch, int max_items, cudaStream_t s) {
    dim3 grid((max_items + kPrefillWarps - 1) / kPrefillWarps, p.hkv, batch);
    // 16-byte copies when every row start is 16-byte aligned, else 8-byte copies
    const bool a16 = ((uintptr_t)p.k % 16 == 0) && ((uintptr_t)p.v % 16 == 0) && p.sb % 8 == 0 &&
                     p.st % 8 == 0 && p.sh % 8 == 0;
    return a16 ? launch<16>(p, grid, s) : launch<8>(p, grid, s);
  }
};

template <int D, int BITS>
struct AppendLaunch {
  static kvq_status run(const AppendParams& p, int batch, cudaStream_t s) {
    constexpr int smem = kAppendGroups * StagedTile<D>::BYTES;
    if (!device_smem_attr(reinterpret_cast<const void*>(append_kernel<D, BITS>), smem)) return KVQ_ERR_CUDA;
    append_kernel<D, BITS><<<batch, kAppendGroups * D, smem, s>>>(p);
    return launch_status();
  }
};

}  // namespace kvq

extern "C" kvq_status kvq_quantize_prefill(const kvq_cache* c, const void* k, const void* v,
                                           int64_t stride_b, int64_t stride_t, int64_t stride_h,
                                           const int32_t* seq_len, const int32_t* n_tail,
                                           void* stream) {
  using namespace kvq;
  kvq_status s = validate_cache(c);
  if (s != KVQ_OK) return s;
  if (c->batch > KVQ_MAX_BATCH) return KVQ_ERR_UNSUPPORTED;
  if (k == nullptr || v == nullptr || seq_len == nullptr || n_tail == nullptr) return KVQ_ERR_INVALID;
  if (!aligned(k, 8) || !aligned(v, 8)) return KVQ_ERR_INVALID;
  if (stride_b % 4 || stride_t % 4 || stride_h % 4) return KVQ_ERR_INVALID;
  if (stride_b < 0 || stride_t < 0 || stride_h < 0) return KVQ_ERR_INVALID;
  PrefillParams p{};
  int max_items = 0;
  for (int b = 0; b < c->batch; ++b) {
    const int L = seq_len[b], nt = n_tail[b];
    const int ns = L < c->sink_cap ? L : c->sink_cap;
    if (L < 0 || nt < 0 || nt > L - ns || nt > c->tail_cap) return KVQ_ERR_INVALID;
    if ((L - ns - nt) % KVQ_GROUP) return KVQ_ERR_INVALID;
    if ((L - ns - nt) / KVQ_GROUP > c->max_groups) return KVQ_ERR_CAPACITY;
    p.seq_len[b] = L;
    p.ntail[b] = nt;
    const int items = (L - ns - nt) / KVQ_GROUP + (nt + KVQ_GROUP - 1) / KVQ_GROUP + (ns + KVQ_GROUP - 1) / KVQ_GROUP;
    max_items = items > max_items ? items : max_items;
  }
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.sb = stride_b;
  p.st = stride_t;
  p.sh = stride_h;
  p.k_codes = static_cast<uint8_t*>(c->k_codes);
  p.v_codes = static_cast<uint8_t*>(c->v_codes);
  p.k_meta = static_cast<__half*>(c->k_meta);
  p.v_meta = static_cast<__half*>(c->v_meta);
  p.k_tail = static_cast<__half*>(c->k_tail);
  p.v_tail = static_cast<__half*>(c->v_tail);
  p.n_quant = c->n_quant;
  p.n_tail = c->n_tail;
  p.tail_head = c->tail_head;
  p.k_sink = static_cast<__half*>(c->k_sink);
  p.v_sink = static_cast<__half*>(c->v_sink);
  p.n_sink = c->n_sink;
  p.hkv = c->n_kv_heads;
  p.max_groups = c->max_groups;
  p.tail_cap = c->tail_cap;
  p.sink_cap = c->sink_cap;
  if (max_items == 0) max_items = 1;  // still write the lengths
  if (c->n_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  return dispatch_db<PrefillLaunch>(c->head_dim, c->bits, p, c->batch, max_items,
                                    static_cast<cudaStream_t>(stream));
}

extern "C" kvq_status kvq_append_token(const kvq_cache* c, const void* k_new, const void* v_new,
                                       void* stream) {
  using namespace kvq;
  kvq_status s = validate_cache(c);
  if (s != KVQ_OK) return s;
  if (k_new == nullptr || v_new == nullptr || !aligned(k_new, 8) || !aligned(v_new, 8))
    return KVQ_ERR_INVALID;
  AppendParams p{};
  p.k_new = static_cast<const __half*>(k_new);
  p.v_new = static_cast<const __half*>(v_new);
  p.k_codes = static_cast<uint8_t*>(c->k_codes);
  p.v_codes = static_cast<uint8_t*>(c->v_codes);
  p.k_meta = static_cast<__half*>(c->k_meta);
  p.v_meta = static_cast<__half*>(c->v_meta);
  p.k_tail = static_cast<__half*>(c->k_tail);
  p.v_tail = static_cast<__half*>(c->v_tail);
  p.n_quant = c->n_quant;
  p.n_tail = c->n_tail;
  p.tail_head = c->tail_head;
  p.error_flags = c->error_flags;
  p.k_sink = static_cast<__half*>(c->k_sink);
  p.v_sink = static_cast<__half*>(c->v_sink);
  p.n_sink = c->n_sink;
  p.hkv = c->n_kv_heads;
  p.max_groups = c->max_groups;
  p.tail_cap = c->tail_cap;
  p.sink_cap = c->sink_cap;
  return dispatch_db<AppendLaunch>(c->head_dim, c->bits, p, c->batch,
                                   static_cast<cudaStream_t>(stream));
}
