// Build of the mixed-width ("TriZone") cache: "RDKV" summary (gist.science
// 2605.08317), sections 2.1-2.2 and "2.2 TriZone".  Two launches:
//  1. index: per (sequence, KV head) one CTA drops the width-0 tokens, orders
//     the kept old tokens by value width (stable), permutes the channels by key
//     width, and writes the index record (counts, sizes, offsets, slots);
//  2. blocks: one warp per 32-token block gathers the block's rows, quantizes
//     keys per channel (at each channel's width, over the block's tokens) and
//     values per token (at the block's width), and writes the packed record;
//     fresh blocks copy fp16 rows into fragment-ordered tiles.
// The group quantizer is the uniform cache's, bit for bit.
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_trizone_internal.h"

namespace kvq {
namespace tz {

constexpr int kIndexThreads = 1024;
constexpr int kBlockWarps = 5;
// per-warp scratch of the block kernel: 32 staged fp16 rows, codes by slot,
// key scale/zero by slot, value metadata, value reciprocal scales
constexpr int kRowsBytes = kGroup * kDim * 2;
constexpr int kCodeBytes = kGroup * kSlots;
constexpr int kWarpScratch = kRowsBytes + kCodeBytes + 4 * kSlots + 4 * kDim + 4 * kDim;

struct BuildParams {
  const __half* k;
  const __half* v;
  int64_t sb, st, sh;
  const uint8_t* v_width;
  const uint8_t* k_width;
  uint8_t* index;
  int32_t* tokens;
  uint8_t* blocks;
  int32_t* error_flags;
  int64_t region;
  int32_t hkv, max_old, max_fresh;
  int32_t t_old[KVQ_MAX_BATCH];
  int32_t n_fresh[KVQ_MAX_BATCH];
};

__device__ __forceinline__ int v_class(int w) {
  return w == 2 ? 0 : (w == 4 ? 1 : (w == 8 ? 2 : (w == 16 ? 3 : (w == 0 ? -1 : -2))));
}

// Exclusive block-wide scan of one int per thread (kIndexThreads threads).
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kIndexThreads / 32; ++w) {
    const int t = s_warp[w];
    base += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();
  total = all;
  return base + x - v;
}

// grid (Hkv, B), kIndexThreads threads.
__global__ void __launch_bounds__(kIndexThreads, 1) index_kernel(const __grid_constant__ BuildParams p) {
  __shared__ int16_t s_slots[kSlots];
  __shared__ int s_warp[kIndexThreads / 32];
  __shared__ int s_hdr[32];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const size_t seg = (size_t)b * p.hkv + h;
  const int t_old = p.t_old[b];
  const uint8_t* vw = p.v_width + seg * p.max_old;
  int32_t* toks = p.tokens + seg * p.max_old;
  bool bad = false;

  // ---- kept old tokens, grouped by value width (stable).  Each thread takes a
  // contiguous chunk (a multiple of 16 tokens), read 16 widths per load when the
  // width row is 16-byte aligned
  const int chunk = ((t_old + kIndexThreads - 1) / kIndexThreads + 15) & ~15;
  const int t0 = min(t_old, tid * chunk), t1 = min(t_old, t0 + chunk);
  const bool v16 = (reinterpret_cast<uintptr_t>(vw) & 15) == 0;
  auto each_width = [&](auto&& f) {
    int t = t0;
    if (v16)
      for (; t + 16 <= t1; t += 16) {
        const uint4 q = *reinterpret_cast<const uint4*>(vw + t);
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 16; ++k) f(t + k, (int)((w4[k >> 2] >> (8 * (k & 3))) & 0xFFu));
      }
    for (; t < t1; ++t) f(t, (int)vw[t]);
  };
  int cnt[4] = {0, 0, 0, 0};
  each_width([&](int, int w) {
    const int c = v_class(w);
    bad |= c == -2;
#pragma unroll
    for (int i = 0; i < 4; ++i) cnt[i] += c == i;
  });
  int start[4], ntok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) start[i] = block_excl_scan(cnt[i], s_warp, ntok[i]);
  int cls_first = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    start[i] += cls_first;
    cls_first += ntok[i];
  }
  each_width([&](int t, int w) {
    const int c = v_class(w);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (c == i) toks[start[i]++] = t;
  });

  // ---- channel slots by key width (2, 4, 8), each class padded to 16
  for (int i = tid; i < kSlots; i += blockDim.x) s_slots[i] = -1;
  __syncthreads();
  if (warp == 0) {
    int base = 0, nch[3], kts[3];
    for (int ci = 0; ci < 3; ++ci) {
      const int c = 2 << ci;
      int run = 0;
#pragma unroll
      for (int q = 0; q < kDim / 32; ++q) {
        const int d = 32 * q + lane;
        int w = p.k_width[seg * kDim + d];
        if (w != 2 && w != 4 && w != 8) {
          bad |= ci == 0;
          w = 8;
        }
        const unsigned m = __ballot_sync(0xffffffffu, w == c);
        if (w == c) s_slots[base + run + __popc(m & ((1u << lane) - 1u))] = (int16_t)d;
        run += __popc(m);
      }
      nch[ci] = run;
      kts[ci] = (run + 15) / 16;
      base += 16 * kts[ci];
    }
    if (lane == 0) {
      const int nf = p.n_fresh[b];
      int nblk[kKinds], rec[kKinds];
      for (int i = 0; i < 4; ++i) {
        s_hdr[H_NTOK + i] = ntok[i];
        nblk[i] = (ntok[i] + kGroup - 1) / kGroup;
        rec[i] = record_bytes(kts[0], kts[1], kts[2], i);
      }
      nblk[4] = (nf + kGroup - 1) / kGroup;
      rec[4] = KVQ_TZ_FRESH_BLOCK_BYTES;
      s_hdr[H_NFRESH] = nf;
      int off = 0;
      for (int i = 0; i < kKinds; ++i) {
        s_hdr[H_NBLK + i] = nblk[i];
        s_hdr[H_REC + i] = rec[i];
        s_hdr[H_OFF + i] = off;
        off += nblk[i] * rec[i];
      }
      for (int i = 0; i < 3; ++i) {
        s_hdr[H_NCH + i] = nch[i];
        s_hdr[H_KT + i] = kts[i];
      }
      s_hdr[H_USED] = off;
      for (int i = H_USED + 1; i < 32; ++i) s_hdr[i] = 0;
    }
  }
  if (bad && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_BAD_WIDTH);
  __syncthreads();
  // ---- index record: header, slots, zero pad
  uint32_t* dst = reinterpret_cast<uint32_t*>(p.index + seg * KVQ_TZ_INDEX_BYTES);
  for (int i = tid; i < KVQ_TZ_INDEX_BYTES / 4; i += blockDim.x) {
    uint32_t w = 0u;
    if (i < 32) w = (uint32_t)s_hdr[i];
    else if (i < 32 + kSlots / 2)
      w = (uint32_t)(uint16_t)s_slots[2 * (i - 32)] | ((uint32_t)(uint16_t)s_slots[2 * (i - 32) + 1] << 16);
    dst[i] = w;
  }
}

// Stage up to 32 fp16 rows (row t of token tok(t), t < n; zero rows after) into
// rows[32][128]: every lane issues an 8-byte asynchronous copy of 4 channels of
// every row, then waits for all of them.
template <typename TokOf>
__device__ __forceinline__ void stage_rows(__half* rows, const __half* base, int64_t st, int n, TokOf tok_of,
                                           int lane, bool replicate = false) {
  const int tok0 = tok_of(0);
#pragma unroll 8
  for (int t = 0; t < kGroup; ++t) {
    const int tok = tok_of(t);
    if (t < n) cp_async_8(rows + t * kDim + 4 * lane, base + (int64_t)tok * st + 4 * lane);
    else if (replicate && n > 0) cp_async_8(rows + t * kDim + 4 * lane, base + (int64_t)tok0 * st + 4 * lane);
    else *reinterpret_cast<uint2*>(rows + t * kDim + 4 * lane) = make_uint2(0u, 0u);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
}

__device__ __forceinline__ uint32_t h_bits(const __half* p) { return (uint32_t)__half_as_ushort(*p); }

// 16-bit value tile from staged rows: lane word P (mt = P/8, kt = P/4 % 2, i = P%4)
// = (v[t][c], v[t+1][c]) with c = 16mt + gid + 8(i%2), t = 16kt + 2tig + 8(i/2).
__device__ __forceinline__ void store_fp16_vtile(const __half* rows, uint8_t* dst, int lane) {
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll 4
  for (int ch = 0; ch < 16; ++ch) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int P = 4 * ch + i, mt = P >> 3, kt = (P >> 2) & 1;
      const int c = 16 * mt + gid + 8 * (i & 1), t = 16 * kt + 2 * tig + 8 * (i >> 1);
      w[i] = h_bits(rows + t * kDim + c) | (h_bits(rows + (t + 1) * kDim + c) << 16);
    }
    *reinterpret_cast<uint4*>(dst + (size_t)(ch * 32 + lane) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// 16-bit key tile: lane word P (kt = P/8, mt = P/4 % 2, i = P%4) = (k[t][c], k[t][c+1])
// with t = 16mt + gid + 8(i%2), c = 16kt + 2tig + 8(i/2).
__device__ __forceinline__ void store_fp16_ktile(const __half* rows, uint8_t* dst, int lane) {
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll 4
  for (int ch = 0; ch < 16; ++ch) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int P = 4 * ch + i, kt = P >> 3, mt = (P >> 2) & 1;
      const int t = 16 * mt + gid + 8 * (i & 1), c = 16 * kt + 2 * tig + 8 * (i >> 1);
      w[i] = *reinterpret_cast<const uint32_t*>(rows + t * kDim + c);
    }
    *reinterpret_cast<uint4*>(dst + (size_t)(ch * 32 + lane) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Key sub-tile of class width C: kt_c k-tiles of slots [base, base + 16 kt_c);
// lane word w at byte 4(32w + lane).
template <int C>
__device__ __forceinline__ void store_key_subtile(const uint8_t* ct, int base, int ktc, uint8_t* dst, int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  constexpr int PPW = 16 / C;  // pairs per word
  for (int kt = 0; kt < ktc; ++kt) {
    uint32_t w[C / 2];
#pragma unroll
    for (int i = 0; i < C / 2; ++i) w[i] = 0u;
#pragma unroll
    for (int P = 0; P < 8; ++P) {
      const int mt = P >> 2, i = P & 3;
      const int t = 16 * mt + gid + 8 * (i & 1), s = base + 16 * kt + 2 * tig + 8 * (i >> 1);
      const uint32_t first = ct[t * kSlots + s], second = ct[t * kSlots + s + 1];
      const int pos = slot_bitpos<C>(P % PPW);
      w[P / PPW] |= (first << pos) | (second << (16 + pos));
    }
#pragma unroll
    for (int i = 0; i < C / 2; ++i)
      *reinterpret_cast<uint32_t*>(dst + (size_t)((kt * (C / 2) + i) * 32 + lane) * 4) = w[i];
  }
}

// Per-token value quantization of the staged rows (32-channel groups) at width C:
// codes to ct[t][c] (t < n; zero after), metadata planes to vm[2][128] (natural
// order).  The 8 lanes of a group reduce min/max with shuffles; the group's
// parameters are computed once, by lane t % 8 of the group, and read back from
// shared memory (vm, vinv).
template <int C>
__device__ __forceinline__ void quantize_values(const __half* rows, int n, uint8_t* ct, __half* vm, float* vinv,
                                                int lane) {
  const int c0 = 4 * lane, j = lane / 8;
  constexpr uint32_t cmax = (1u << C) - 1u;
  // min/max of group j of every token: reduced over the group's 8 lanes; lane
  // t % 8 keeps token t's.  Eight tokens per pass, the kept pair shifted into
  // rmn / rmx (after the four passes slot 3 - k holds token lane % 8 + 8k), so
  // the pass loop stays rolled without indexing registers
  float rmn[4] = {0.f, 0.f, 0.f, 0.f}, rmx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int t8 = 0; t8 < kGroup; t8 += 8) {
    float kmn = 0.f, kmx = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint2 raw = *reinterpret_cast<const uint2*>(rows + (t8 + u) * kDim + c0);
      const __half2 lo = u32_as_h2(raw.x), hi = u32_as_h2(raw.y);
      const __half2 m2 = __hmin2(lo, hi), x2 = __hmax2(lo, hi);
      float mn = fminf(__low2float(m2), __high2float(m2));
      float mx = fmaxf(__low2float(x2), __high2float(x2));
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      }
      if ((lane & 7) == u) {
        kmn = mn;
        kmx = mx;
      }
    }
#pragma unroll
    for (int k = 3; k > 0; --k) {
      rmn[k] = rmn[k - 1];
      rmx[k] = rmx[k - 1];
    }
    rmn[0] = kmn;
    rmx[0] = kmx;
  }
  // the parameters of tokens lane % 8 + 8k of group j, every lane busy
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = (lane & 7) + 8 * k;
    GroupParams g = group_params<C>(rmn[3 - k], rmx[3 - k]);
    if (t >= n) {
      g.scale_h = __float2half_rn(0.f);
      g.zero_h = __float2half_rn(0.f);
      g.inv = 0.f;
    }
    vm[j * kGroup + t] = g.scale_h;
    vm[kDim + j * kGroup + t] = g.zero_h;
    vinv[j * kGroup + t] = g.inv;
  }
  __syncwarp();
  // the codes without a branch; bit t of `redo`: one of the lane's four codes of
  // token t lies near a rounding tie, and those four are redone with the exact
  // quotient afterwards
  uint32_t redo = 0u;
#pragma unroll 2
  for (int t = 0; t < kGroup; ++t) {
    const uint2 raw = *reinterpret_cast<const uint2*>(rows + t * kDim + c0);
    const __half2 lo = u32_as_h2(raw.x), hi = u32_as_h2(raw.y);
    GroupParams g;
    g.scale = __half2float(vm[j * kGroup + t]);
    g.zero = __half2float(vm[kDim + j * kGroup + t]);
    g.inv = vinv[j * kGroup + t];
    bool n0, n1, n2, n3;
    const uint32_t q0 = quant_code_fast(__low2float(lo), g, cmax, n0);
    const uint32_t q1 = quant_code_fast(__high2float(lo), g, cmax, n1);
    const uint32_t q2 = quant_code_fast(__low2float(hi), g, cmax, n2);
    const uint32_t q3 = quant_code_fast(__high2float(hi), g, cmax, n3);
    redo |= (uint32_t)((n0 || n1 || n2 || n3) && t < n) << t;
    *reinterpret_cast<uint32_t*>(ct + t * kDim + c0) = t < n ? pack4_bytes(q0, q1, q2, q3) : 0u;
  }
#pragma unroll 1
  while (redo != 0u) {
    const int t = __ffs(redo) - 1;
    redo &= redo - 1u;
    const uint2 raw = *reinterpret_cast<const uint2*>(rows + t * kDim + c0);
    const __half2 lo = u32_as_h2(raw.x), hi = u32_as_h2(raw.y);
    const float sc = __half2float(vm[j * kGroup + t]), ze = __half2float(vm[kDim + j * kGroup + t]);
    *reinterpret_cast<uint32_t*>(ct + t * kDim + c0) =
        pack4_bytes(quant_code_exact(__low2float(lo), sc, ze, cmax), quant_code_exact(__high2float(lo), sc, ze, cmax),
                    quant_code_exact(__low2float(hi), sc, ze, cmax), quant_code_exact(__high2float(hi), sc, ze, cmax));
  }
  __syncwarp();
}

// The lane's 4 key channels d0..d0+3 over the block's n tokens, each at its own
// width: fp16 min/max on half2, then the parameters and the codes (to ct at the
// channels' slots).  The rows past n hold copies of row 0 (stage_rows with
// replicate), so the min/max over all 32 rows is that over the n tokens; their
// codes are stored as 0.
__device__ __forceinline__ void key_channels(const __half* rows, int n, int d0, const uint8_t* slot_of,
                                             const uint8_t* kw, uint8_t* ct, __half* ksc, __half* kze) {
  __half2 mn0 = *reinterpret_cast<const __half2*>(rows + d0), mn1 = *reinterpret_cast<const __half2*>(rows + d0 + 2);
  __half2 mx0 = mn0, mx1 = mn1;
#pragma unroll 8
  for (int t = 1; t < kGroup; ++t) {
    const uint2 raw = *reinterpret_cast<const uint2*>(rows + t * kDim + d0);
    const __half2 a = u32_as_h2(raw.x), b = u32_as_h2(raw.y);
    mn0 = __hmin2(mn0, a); mx0 = __hmax2(mx0, a);
    mn1 = __hmin2(mn1, b); mx1 = __hmax2(mx1, b);
  }
  const float mns[4] = {__low2float(mn0), __high2float(mn0), __low2float(mn1), __high2float(mn1)};
  const float mxs[4] = {__low2float(mx0), __high2float(mx0), __low2float(mx1), __high2float(mx1)};
  GroupParams g[4];
  uint32_t cmax[4];
  int slot[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    cmax[i] = (1u << kw[d0 + i]) - 1u;
    g[i] = group_params_levels(mns[i], mxs[i], (float)cmax[i]);
    slot[i] = slot_of[d0 + i];
    ksc[slot[i]] = g[i].scale_h;
    kze[slot[i]] = g[i].zero_h;
  }
  // the codes without a branch; bit t of `redo`: one of the lane's four codes of
  // token t lies near a rounding tie (those four are redone with the exact
  // quotient afterwards)
  uint32_t redo = 0u;
#pragma unroll 2
  for (int t = 0; t < kGroup; ++t) {
    const uint2 raw = *reinterpret_cast<const uint2*>(rows + t * kDim + d0);
    const float x[4] = {__low2float(u32_as_h2(raw.x)), __high2float(u32_as_h2(raw.x)), __low2float(u32_as_h2(raw.y)),
                        __high2float(u32_as_h2(raw.y))};
    bool near = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      bool ni;
      const uint32_t c = quant_code_fast(x[i], g[i], cmax[i], ni);
      near = near || ni;
      ct[t * kSlots + slot[i]] = t < n ? (uint8_t)c : (uint8_t)0;
    }
    redo |= (uint32_t)(near && t < n) << t;
  }
#pragma unroll 1
  while (redo != 0u) {
    const int t = __ffs(redo) - 1;
    redo &= redo - 1u;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      ct[t * kSlots + slot[i]] =
          (uint8_t)quant_code_exact(__half2float(rows[t * kDim + d0 + i]), g[i].scale, g[i].zero, cmax[i]);
  }
}

// grid (ceil(items / kBlockWarps), Hkv, B); one warp per block record.
__global__ void __launch_bounds__(kBlockWarps * 32) block_kernel(const __grid_constant__ BuildParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_hdr[32];
  __shared__ uint8_t s_slot_of[kDim];
  __shared__ uint8_t s_kw[kDim];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const size_t seg = (size_t)b * p.hkv + h;
  const uint8_t* idx = p.index + seg * KVQ_TZ_INDEX_BYTES;
  if (threadIdx.x < 32) s_hdr[threadIdx.x] = reinterpret_cast<const int32_t*>(idx)[threadIdx.x];
  for (int s = threadIdx.x; s < kSlots; s += blockDim.x) {
    const int d = reinterpret_cast<const int16_t*>(idx + 128)[s];
    if (d >= 0 && d < kDim) s_slot_of[d] = (uint8_t)s;
  }
  for (int d = threadIdx.x; d < kDim; d += blockDim.x) {
    const int w = p.k_width[seg * kDim + d];
    s_kw[d] = (uint8_t)((w == 2 || w == 4) ? w : 8);
  }
  __syncthreads();
  uint8_t* ws = smem + warp * kWarpScratch;
  __half* rows = reinterpret_cast<__half*>(ws);
  uint8_t* ct = ws + kRowsBytes;
  __half* ksc = reinterpret_cast<__half*>(ws + kRowsBytes + kCodeBytes);
  __half* kze = ksc + kSlots;
  __half* vm = kze + kSlots;
  float* vinv = reinterpret_cast<float*>(vm + 2 * kDim);

  int j = blockIdx.x * kBlockWarps + warp, kind = 0;
  while (kind < kKinds && j >= s_hdr[H_NBLK + kind]) j -= s_hdr[H_NBLK + kind++];
  if (kind == kKinds) return;
  uint8_t* dst = p.blocks + seg * p.region + s_hdr[H_OFF + kind] + (size_t)j * s_hdr[H_REC + kind];
  const __half* kseq = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
  const __half* vseq = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;

  if (kind == 4) {  // fresh block: fp16 key tile, fp16 value tile
    const int n = min(kGroup, s_hdr[H_NFRESH] - kGroup * j);
    const int first = p.t_old[b] + kGroup * j;
    auto tok = [&](int t) { return first + t; };
    stage_rows(rows, kseq, p.st, n, tok, lane);
    store_fp16_ktile(rows, dst, lane);
    __syncwarp();
    stage_rows(rows, vseq, p.st, n, tok, lane);
    store_fp16_vtile(rows, dst + kGroup * kDim * 2, lane);
    return;
  }
  int first = kGroup * j;
  for (int i = 0; i < kind; ++i) first += s_hdr[H_NTOK + i];
  const int n = min(kGroup, s_hdr[H_NTOK + kind] - kGroup * j);
  const int my_tok = lane < n ? p.tokens[seg * p.max_old + first + lane] : 0;
  auto tok = [&](int t) { return __shfl_sync(0xffffffffu, my_tok, t); };

  // ---- keys: per channel over the block's n tokens, at the channel's width
  for (int i = lane; i < kCodeBytes / 16; i += 32) reinterpret_cast<uint4*>(ct)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = lane; i < kSlots; i += 32) {
    ksc[i] = __float2half_rn(0.f);
    kze[i] = __float2half_rn(0.f);
  }
  stage_rows(rows, kseq, p.st, n, tok, lane, true);
  key_channels(rows, n, 4 * lane, s_slot_of, s_kw, ct, ksc, kze);
  __syncwarp();
  const int kt2 = s_hdr[H_KT], kt4 = s_hdr[H_KT + 1], kt8 = s_hdr[H_KT + 2], KT = kt2 + kt4 + kt8;
  store_key_subtile<2>(ct, 0, kt2, dst, lane);
  store_key_subtile<4>(ct, 16 * kt2, kt4, dst + 128 * kt2, lane);
  store_key_subtile<8>(ct, 16 * (kt2 + kt4), kt8, dst + 128 * kt2 + 256 * kt4, lane);
  uint8_t* kmeta = dst + key_code_bytes(kt2, kt4, kt8);
  // pair 16kt + 4tig + 2r + f: the zero points (f = 0) or scales (f = 1) of
  // slots 16kt + 2tig + 8r and +1
  for (int pr = lane; pr < 16 * KT; pr += 32) {
    const int kt = pr >> 4, tg = (pr >> 2) & 3, r = (pr >> 1) & 1;
    const int s = 16 * kt + 2 * tg + 8 * r;
    const __half* src = (pr & 1) ? ksc : kze;
    reinterpret_cast<uint32_t*>(kmeta)[pr] =
        (uint32_t)__half_as_ushort(src[s]) | ((uint32_t)__half_as_ushort(src[s + 1]) << 16);
  }
  __syncwarp();
  // ---- values: per token over 32-channel groups at the block's width, or fp16
  uint8_t* vdst = kmeta + 64 * KT;
  stage_rows(rows, vseq, p.st, n, tok, lane);
  if (kind == 3) {
    store_fp16_vtile(rows, vdst, lane);
    return;
  }
  if (kind == 0) {
    quantize_values<2>(rows, n, ct, vm, vinv, lane);
    pack_store_tile<kDim, 2, false>(ct, vdst, lane);
    store_meta_lane_order<kDim, false>(vm, reinterpret_cast<__half*>(vdst + Tile<kDim, 2>::kBytes), lane);
  } else if (kind == 1) {
    quantize_values<4>(rows, n, ct, vm, vinv, lane);
    pack_store_tile<kDim, 4, false>(ct, vdst, lane);
    store_meta_lane_order<kDim, false>(vm, reinterpret_cast<__half*>(vdst + Tile<kDim, 4>::kBytes), lane);
  } else {
    quantize_values<8>(rows, n, ct, vm, vinv, lane);
    pack_store_tile<kDim, 8, false>(ct, vdst, lane);
    store_meta_lane_order<kDim, false>(vm, reinterpret_cast<__half*>(vdst + Tile<kDim, 8>::kBytes), lane);
  }
}

}  // namespace tz
}  // namespace kvq

extern "C" kvq_status kvq_trizone_bytes(const kvq_trizone* tz, size_t sizes[KVQ_TZ_NBUF]) {
  using namespace kvq::tz;
  kvq_status s = validate_geometry(tz);
  if (s != KVQ_OK) return s;
  if (sizes == nullptr) return KVQ_ERR_INVALID;
  const size_t segs = (size_t)tz->batch * tz->n_kv_heads;
  sizes[KVQ_TZ_BUF_INDEX] = segs * KVQ_TZ_INDEX_BYTES;
  sizes[KVQ_TZ_BUF_TOKENS] = segs * (size_t)tz->max_old * 4;
  sizes[KVQ_TZ_BUF_BLOCKS] = segs * (size_t)region_bytes(tz);
  return KVQ_OK;
}

extern "C" kvq_status kvq_trizone_build(const kvq_trizone* tz, const void* k, const void* v, int64_t stride_b,
                                        int64_t stride_t, int64_t stride_h, const uint8_t* v_width,
                                        const uint8_t* k_width, const int32_t* t_old, const int32_t* n_fresh,
                                        void* stream) {
  using namespace kvq;
  using namespace kvq::tz;
  kvq_status s = validate_buffers(tz);
  if (s != KVQ_OK) return s;
  if (tz->batch > KVQ_MAX_BATCH) return KVQ_ERR_UNSUPPORTED;
  if (k == nullptr || v == nullptr || v_width == nullptr || k_width == nullptr || t_old == nullptr ||
      n_fresh == nullptr)
    return KVQ_ERR_INVALID;
  if (!aligned(k, 8) || !aligned(v, 8)) return KVQ_ERR_INVALID;
  if (stride_b < 0 || stride_t < 0 || stride_h < 0 || stride_b % 4 || stride_t % 4 || stride_h % 4)
    return KVQ_ERR_INVALID;
  BuildParams p{};
  int max_items = 0;
  for (int b = 0; b < tz->batch; ++b) {
    if (t_old[b] < 0 || n_fresh[b] < 0) return KVQ_ERR_INVALID;
    if (t_old[b] > tz->max_old || n_fresh[b] > tz->max_fresh) return KVQ_ERR_CAPACITY;
    p.t_old[b] = t_old[b];
    p.n_fresh[b] = n_fresh[b];
    const int items = (t_old[b] + kGroup - 1) / kGroup + 3 + (n_fresh[b] + kGroup - 1) / kGroup;
    max_items = items > max_items ? items : max_items;
  }
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.sb = stride_b;
  p.st = stride_t;
  p.sh = stride_h;
  p.v_width = v_width;
  p.k_width = k_width;
  p.index = static_cast<uint8_t*>(tz->index);
  p.tokens = tz->tokens;
  p.blocks = static_cast<uint8_t*>(tz->blocks);
  p.error_flags = tz->error_flags;
  p.region = region_bytes(tz);
  p.hkv = tz->n_kv_heads;
  p.max_old = tz->max_old;
  p.max_fresh = tz->max_fresh;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  index_kernel<<<dim3(tz->n_kv_heads, tz->batch), kIndexThreads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  constexpr int smem = kBlockWarps * kWarpScratch;
  if (!device_smem_attr(reinterpret_cast<const void*>(block_kernel), smem)) return KVQ_ERR_CUDA;
  const int gx = (max_items + kBlockWarps - 1) / kBlockWarps;
  block_kernel<<<dim3(gx, tz->n_kv_heads, tz->batch), kBlockWarps * 32, smem, st>>>(p);
  return launch_status();
}
