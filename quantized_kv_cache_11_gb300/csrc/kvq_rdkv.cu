// RDKV bit allocation ("RDKV" summary, gist.science 2605.08317, sections 2.1
// and 2.2): the distortion weights of the prompt's tokens and channels, and the
// Lagrangian choice of a V width per old token and a K width per channel that
// the mixed-width cache is built with.
//
// How:
// * Token weights (the dense part): two passes over the causal score matrix of
//   every (sequence, query head) on tensor cores (mma.m16n8k16, fp16 in, fp32
//   accumulate).  Pass 1: per query row the log-sum-exp (base 2) of its scores,
//   one CTA per 64 query rows, key tiles staged by cp.async, double buffered.
//   Pass 2: per key the column sum of the normalised probabilities over every
//   later query of the group's heads: a CTA holds 64 keys as A fragments and
//   streams the query tiles (S^T = K Q^T), so each key's sum stays in the
//   registers of one quad of lanes; no atomics, the summation order is fixed.
// * Costs and allocation: one warp per token for the value variance; per
//   (sequence, KV head) one CTA runs the binary search over the bit pattern of
//   the float32 multiplier, each step a block-wide count of the chosen bits.
// * Channel statistics: chunks of 256 positions per CTA, one thread per
//   channel, partial sums combined in a fixed order in float64 (Chan's pairwise
//   variance update).
#include <cmath>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq_rdkv.h"

namespace kvq {
namespace rdkv {

constexpr int kD = 128;
constexpr int kBlk = 64;               // query / key positions per tile
constexpr int kPitch = 2 * kD + 16;    // bytes per staged row: conflict-free ldmatrix rows
constexpr int kTile = kBlk * kPitch;   // bytes per staged tile
constexpr int kChunk = 256;            // positions per channel-statistics chunk
constexpr int kFields = 5;             // q^2 sum, kept count, k sum, k^2 sum, k squared deviations
constexpr uint32_t kLamMax = 0x7F7FFFFFu;

inline int nchunks(int t) { return (t + kChunk - 1) / kChunk; }
// Row stride of the log-sum-exp array: a multiple of 64 floats, so every 64-row
// tile of it starts on a 16-byte boundary (it is staged with 16-byte copies).
inline int lse_stride(int t) { return (t + kBlk - 1) / kBlk * kBlk; }

struct Layout {
  size_t lse, wt, wc, part, total;
};
inline Layout layout(const kvq_rdkv* r) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t seg = (size_t)r->batch * r->n_kv_heads;
  L.lse = take((size_t)r->batch * r->n_q_heads * lse_stride(r->max_tokens) * 4);
  L.wt = take(seg * r->max_tokens * 4);
  L.wc = take(seg * kD * 4);
  L.part = take(seg * nchunks(r->max_tokens) * kFields * kD * 4);
  L.total = off;
  return L;
}

struct AttnParams {
  const __half* q;
  const __half* k;
  int64_t q_sb, q_st, q_sh, k_sb, k_st, k_sh;
  float scale_log2;
  int32_t Hq, Hkv, G, T;  // T: row capacity (stride of w)
  int32_t Tl;             // stride of lse (T rounded up to 64)
  float* lse;             // [B][Hq][Tl]: log2 of sum_t exp2(scale_log2 * s), per query row
  float* w;               // [B][Hkv][T]
  int32_t n[KVQ_MAX_BATCH];
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 64 rows x 128 fp16 (rows first .. first+63 of a strided matrix) into a staged
// tile by a CTA of 128 threads: thread i copies 16-byte chunk i % 16 of rows
// i / 16 + 8 k; rows >= n are zero-filled.
__device__ __forceinline__ void stage_tile(uint8_t* dst, const __half* base, int64_t row_stride, int first, int n) {
  const int ch = threadIdx.x & 15, j0 = threadIdx.x >> 4;
  const __half* src = base + (int64_t)(first + j0) * row_stride + ch * 8;
  const int64_t step = 8 * row_stride;
  uint8_t* d = dst + j0 * kPitch + ch * 16;
#pragma unroll
  for (int k = 0; k < kBlk / 8; ++k) {
    const bool ok = first + j0 + 8 * k < n;
    cp_async_16_zfill(d + 8 * k * kPitch, ok ? src : base, ok ? 16 : 0);
    src += step;
  }
}

// A fragments (rows row0 + gid and row0 + gid + 8, all 8 k-tiles) of a strided
// fp16 matrix; rows >= n read as zero.
__device__ __forceinline__ void load_a(uint32_t (&a)[8][4], const __half* base, int64_t row_stride, int row0, int n,
                                       int gid, int tig) {
  const int r0 = row0 + gid, r1 = r0 + 8;
  const bool ok0 = r0 < n, ok1 = r1 < n;
  const __half* p0 = base + (int64_t)(ok0 ? r0 : 0) * row_stride;
  const __half* p1 = base + (int64_t)(ok1 ? r1 : 0) * row_stride;
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
    const int c = 16 * kt + 2 * tig;
    a[kt][0] = ok0 ? *reinterpret_cast<const uint32_t*>(p0 + c) : 0u;
    a[kt][1] = ok1 ? *reinterpret_cast<const uint32_t*>(p1 + c) : 0u;
    a[kt][2] = ok0 ? *reinterpret_cast<const uint32_t*>(p0 + c + 8) : 0u;
    a[kt][3] = ok1 ? *reinterpret_cast<const uint32_t*>(p1 + c + 8) : 0u;
  }
}

// s[nt] = A (16 rows) x B^T for the 64 rows of a staged tile (B fragments by
// ldmatrix: matrix lane/8 covers tile rows 8nt + lane%8, columns 32kp + 8(lane/8)).
__device__ __forceinline__ void tile_scores(float (&s)[8][4], const uint32_t (&a)[8][4], const uint8_t* tile,
                                            int lane) {
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
#pragma unroll
  for (int kp = 0; kp < 4; ++kp)
#pragma unroll
    for (int nt = 0; nt < 8; nt += 2) {  // two n-tiles at a time: no back-to-back MMAs on one accumulator
      uint32_t b[4], c[4];
      ldmatrix_x4(b, tile + (8 * nt + (lane & 7)) * kPitch + (32 * kp + 8 * (lane >> 3)) * 2);
      ldmatrix_x4(c, tile + (8 * nt + 8 + (lane & 7)) * kPitch + (32 * kp + 8 * (lane >> 3)) * 2);
      mma_16816(s[nt], a[2 * kp], b[0], b[1]);
      mma_16816(s[nt + 1], a[2 * kp], c[0], c[1]);
      mma_16816(s[nt], a[2 * kp + 1], b[2], b[3]);
      mma_16816(s[nt + 1], a[2 * kp + 1], c[2], c[3]);
    }
}

// Row maxima of the raw scores of rows tau[0], tau[1] (this lane's 16 columns;
// with EDGE, keys t > tau or t >= n are set to -inf first).
template <bool EDGE>
__device__ __forceinline__ void row_max(float (&s)[8][4], float (&mx)[2], const int (&tau)[2], int t0, int n,
                                        int tig) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float v = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (EDGE) {
          const int t = t0 + 8 * nt + 2 * tig + c;
          if (t > tau[r] || t >= n) s[nt][2 * r + c] = -INFINITY;
        }
        v = fmaxf(v, s[nt][2 * r + c]);
      }
    mx[r] = v;
  }
}

// Column sums of exp2(scale * s - lse[tau]) into acc[r] for keys tk[r] (with
// EDGE, queries tau < tk or tau >= n contribute 0).
template <bool EDGE>
__device__ __forceinline__ void col_sums(const float (&s)[8][4], float (&acc)[2], const float* lse, float scale,
                                         const int (&tk)[2], int q0, int n, int tig) {
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float2 ls = *reinterpret_cast<const float2*>(lse + 8 * nt + 2 * tig);
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float e = fast_exp2(fmaf(s[nt][2 * r + c], scale, -(c ? ls.y : ls.x)));
        if (EDGE) {
          const int tau = q0 + 8 * nt + 2 * tig + c;
          if (tau < tk[r] || tau >= n) e = 0.f;
        }
        acc[r] += e;
      }
  }
}

// Pass 1: lse[b][hq][tau] for the 64 query rows of one CTA (4 warps x 16 rows).
// Heavy (late) query blocks are scheduled first.
__global__ void __launch_bounds__(128) rowstats_kernel(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.z, hq = blockIdx.y, h = hq / p.G;
  const int n = p.n[b];
  const int nqb = (p.T + kBlk - 1) / kBlk;
  const int qb = nqb - 1 - (int)blockIdx.x;
  if (qb * kBlk >= n) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const __half* kb_base = p.k + (int64_t)b * p.k_sb + (int64_t)h * p.k_sh;
  const __half* q_base = p.q + (int64_t)b * p.q_sb + (int64_t)hq * p.q_sh;
  stage_tile(smem, kb_base, p.k_st, 0, n);
  cp_async_commit();
  const int row0 = qb * kBlk + 16 * warp;
  uint32_t a[8][4];
  load_a(a, q_base, p.q_st, row0, n, gid, tig);
  const int tau[2] = {row0 + gid, row0 + gid + 8};
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  for (int kb = 0; kb <= qb; ++kb) {
    if (kb < qb) stage_tile(smem + ((kb + 1) & 1) * kTile, kb_base, p.k_st, (kb + 1) * kBlk, n);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    float s[8][4];
    tile_scores(s, a, smem + (kb & 1) * kTile, lane);
    float mx[2];
    if (kb == qb || (kb + 1) * kBlk > n) row_max<true>(s, mx, tau, kb * kBlk, n, tig);
    else row_max<false>(s, mx, tau, kb * kBlk, n, tig);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float v = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      const float mnew = fmaxf(m[r], v * p.scale_log2);  // the scale is positive
      if (mnew != -INFINITY) {
        const float alpha = m[r] == -INFINITY ? 0.f : fast_exp2(m[r] - mnew);
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) sum += fast_exp2(fmaf(s[nt][2 * r + c], p.scale_log2, -mnew));
        l[r] = l[r] * alpha + sum;
        m[r] = mnew;
      }
    }
    __syncthreads();  // the buffer read above is restaged next iteration
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float lt = l[r];
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    if (tig == 0 && tau[r] < n) p.lse[((size_t)b * p.Hq + hq) * p.Tl + tau[r]] = m[r] + log2f(lt);
  }
}

// Pass 2: w[b][h][t] for the 64 keys of one CTA (4 warps x 16 keys): sum over the
// group's heads and the queries tau >= t of exp2(scale_log2 * s - lse[tau]).
__global__ void __launch_bounds__(128) colsum_kernel(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* s_lse = reinterpret_cast<float*>(smem + 2 * kTile);  // [2][64]
  const int b = blockIdx.z, h = blockIdx.y, kb = blockIdx.x;
  const int n = p.n[b];
  if (kb * kBlk >= n) return;
  const int nqb = (n + kBlk - 1) / kBlk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const __half* k_base = p.k + (int64_t)b * p.k_sb + (int64_t)h * p.k_sh;
  const int row0 = kb * kBlk + 16 * warp;
  const int tk[2] = {row0 + gid, row0 + gid + 8};
  const int per_head = nqb - kb;  // query tiles per head
  const int steps = p.G * per_head;
  auto stage = [&](int step, int buf) {
    const int g = step / per_head, qb = kb + step % per_head;
    const int hq = h * p.G + g;
    stage_tile(smem + buf * kTile, p.q + (int64_t)b * p.q_sb + (int64_t)hq * p.q_sh, p.q_st, qb * kBlk, n);
    const float* lse = p.lse + ((size_t)b * p.Hq + hq) * p.Tl + qb * kBlk;
    if (threadIdx.x < 16) {
      const int t0 = qb * kBlk + 4 * threadIdx.x;
      const bool ok = t0 + 4 <= n;  // a partial chunk is read element by element below
      cp_async_16_zfill(s_lse + buf * kBlk + 4 * threadIdx.x, lse + (ok ? 4 * threadIdx.x : 0), ok ? 16 : 0);
    }
  };
  stage(0, 0);
  cp_async_commit();
  uint32_t a[8][4];
  load_a(a, k_base, p.k_st, row0, n, gid, tig);
  float acc[2] = {0.f, 0.f};
  for (int step = 0; step < steps; ++step) {
    if (step + 1 < steps) stage(step + 1, (step + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int buf = step & 1;
    const int qb = kb + step % per_head;
    if ((qb + 1) * kBlk > n && threadIdx.x < kBlk) {
      // the last tile: fetch the lse of the valid rows of a partial 4-row chunk
      const int t = qb * kBlk + threadIdx.x;
      const int hq = h * p.G + step / per_head;
      if (t < n && (t & ~3) + 4 > n) s_lse[buf * kBlk + threadIdx.x] = p.lse[((size_t)b * p.Hq + hq) * p.Tl + t];
    }
    __syncthreads();
    float s[8][4];
    tile_scores(s, a, smem + buf * kTile, lane);
    if (qb == kb || (qb + 1) * kBlk > n) col_sums<true>(s, acc, s_lse + buf * kBlk, p.scale_log2, tk, qb * kBlk, n, tig);
    else col_sums<false>(s, acc, s_lse + buf * kBlk, p.scale_log2, tk, qb * kBlk, n, tig);
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float v = acc[r];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    if (tig == 0 && tk[r] < n) p.w[((size_t)b * p.Hkv + h) * p.T + tk[r]] = v;
  }
}

// ----------------------------------------------------------------- allocation
struct CostParams {
  const __half* v;
  int64_t sb, st, sh;
  const float* w;  // [B][Hkv][T]
  int32_t T, Hkv;
  float* W;        // [B][Hkv][wstride]
  int32_t wstride;
  int32_t t_old[KVQ_MAX_BATCH];
};

// W_t = w[t] * population variance of v[t, :] (fp32), one warp per token.
__global__ void __launch_bounds__(256) token_cost_kernel(const CostParams p) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= p.t_old[b]) return;
  const __half* row = p.v + (int64_t)b * p.sb + (int64_t)t * p.st + (int64_t)h * p.sh + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(row);
  const float2 x01 = __half22float2(u32_as_h2(raw.x)), x23 = __half22float2(u32_as_h2(raw.y));
  float s = (x01.x + x01.y) + (x23.x + x23.y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s * (1.f / kD);
  const float d0 = x01.x - mean, d1 = x01.y - mean, d2 = x23.x - mean, d3 = x23.y - mean;
  float q = (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  if (lane == 0) {
    const size_t seg = (size_t)b * p.Hkv + h;
    p.W[seg * p.wstride + t] = __fmul_rn(p.w[seg * p.T + t], q * (1.f / kD));
  }
}

struct AllocParams {
  const float* W;   // [B][Hkv][wstride]
  int32_t wstride;
  uint8_t* out;     // [B][Hkv][ostride]
  int32_t ostride;
  int32_t Hkv;
  int32_t n[KVQ_MAX_BATCH];       // units per segment of sequence b
  int32_t budget[KVQ_MAX_BATCH];  // bits per segment of sequence b
};

// Width of least cost fl32(fl32(W 2^-b) + fl32(lam b)), ties to the smaller width.
template <bool VALUE>
__device__ __forceinline__ int choose(float W, float lam) {
  constexpr int NW = VALUE ? 5 : 3;
  constexpr int widths[5] = {VALUE ? 0 : 2, VALUE ? 2 : 4, VALUE ? 4 : 8, 8, 16};
  int best_b = widths[0];
  float best = __fadd_rn(__fmul_rn(W, __int_as_float((127 - widths[0]) << 23)), __fmul_rn(lam, (float)widths[0]));
#pragma unroll
  for (int i = 1; i < NW; ++i) {
    const float c = __fadd_rn(__fmul_rn(W, __int_as_float((127 - widths[i]) << 23)), __fmul_rn(lam, (float)widths[i]));
    if (c < best) { best = c; best_b = widths[i]; }
  }
  return best_b;
}

__device__ __forceinline__ long long block_sum(long long v, long long* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // s_red is free
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  long long t = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += s_red[i];
  return t;
}

// One CTA per (sequence, KV head): binary search over the multiplier's bits.
template <bool VALUE>
__global__ void __launch_bounds__(1024) alloc_kernel(const AllocParams p) {
  __shared__ long long s_red[32];
  const int b = blockIdx.y, h = blockIdx.x;
  const int n = p.n[b];
  const long long budget = p.budget[b];
  const size_t seg = (size_t)b * p.Hkv + h;
  const float* W = p.W + seg * p.wstride;
  auto total = [&](uint32_t bits) {
    const float lam = __uint_as_float(bits);
    long long c = 0;
    for (int u = threadIdx.x; u < n; u += blockDim.x) c += choose<VALUE>(W[u], lam);
    return block_sum(c, s_red);
  };
  uint32_t lo = 0, hi = kLamMax;
  if (total(hi) <= budget) {
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      if (total(mid) <= budget) hi = mid;
      else lo = mid + 1;
    }
  } else {
    lo = kLamMax;
  }
  const float lam = __uint_as_float(lo);
  for (int u = threadIdx.x; u < n; u += blockDim.x) p.out[seg * p.ostride + u] = (uint8_t)choose<VALUE>(W[u], lam);
}

struct ChanParams {
  const __half* q;
  const __half* k;
  int64_t q_sb, q_st, q_sh, k_sb, k_st, k_sh;
  const uint8_t* v_width;  // [B][Hkv][vw_stride]
  int32_t vw_stride;
  int32_t Hkv, G, nch;     // nch: chunk stride of the partials
  float* part;             // [B][Hkv][nch][kFields][D]
  float* Wc;               // [B][Hkv][D]
  int32_t n[KVQ_MAX_BATCH];
  int32_t t_old[KVQ_MAX_BATCH];
};

// Partial sums of one chunk of positions, one thread per channel.
__global__ void __launch_bounds__(kD) channel_partial_kernel(const ChanParams p) {
  const int b = blockIdx.z, h = blockIdx.y, ck = blockIdx.x, d = threadIdx.x;
  const int n = p.n[b], told = p.t_old[b];
  const int t0 = ck * kChunk;
  if (t0 >= n) return;
  const int t1 = min(n, t0 + kChunk), k1 = min(told, t0 + kChunk);
  float q2 = 0.f;
  for (int t = t0; t < t1; ++t)
    for (int g = 0; g < p.G; ++g) {
      const float x = __half2float(p.q[(int64_t)b * p.q_sb + (int64_t)t * p.q_st + (int64_t)(h * p.G + g) * p.q_sh + d]);
      q2 = fmaf(x, x, q2);
    }
  const size_t seg = (size_t)b * p.Hkv + h;
  const uint8_t* vw = p.v_width + seg * p.vw_stride;
  const __half* kc = p.k + (int64_t)b * p.k_sb + (int64_t)h * p.k_sh + d;
  float cnt = 0.f, ks = 0.f, ksq = 0.f;
  for (int t = t0; t < k1; ++t)
    if (vw[t] != 0) {
      const float x = __half2float(kc[(int64_t)t * p.k_st]);
      cnt += 1.f;
      ks += x;
      ksq = fmaf(x, x, ksq);
    }
  const float mean = cnt > 0.f ? ks / cnt : 0.f;
  float m2 = 0.f;
  for (int t = t0; t < k1; ++t)
    if (vw[t] != 0) {
      const float dx = __half2float(kc[(int64_t)t * p.k_st]) - mean;
      m2 = fmaf(dx, dx, m2);
    }
  float* o = p.part + ((seg * p.nch + ck) * kFields) * kD + d;
  o[0 * kD] = q2;
  o[1 * kD] = cnt;
  o[2 * kD] = ks;
  o[3 * kD] = ksq;
  o[4 * kD] = m2;
}

// W_c per channel from the chunk partials, combined in order in float64.
__global__ void __launch_bounds__(kD) channel_cost_kernel(const ChanParams p) {
  const int b = blockIdx.y, h = blockIdx.x, d = threadIdx.x;
  const int nck = (p.n[b] + kChunk - 1) / kChunk;
  const size_t seg = (size_t)b * p.Hkv + h;
  double q2 = 0.0, ksq = 0.0, cnt = 0.0, mean = 0.0, m2 = 0.0;
  for (int ck = 0; ck < nck; ++ck) {
    const float* o = p.part + ((seg * p.nch + ck) * kFields) * kD + d;
    q2 += o[0 * kD];
    ksq += o[3 * kD];
    const double nb = o[1 * kD];
    if (nb > 0.0) {
      const double mb = (double)o[2 * kD] / nb;
      const double tot = cnt + nb;
      const double delta = mb - mean;
      mean += delta * nb / tot;
      m2 += (double)o[4 * kD] + delta * delta * cnt * nb / tot;
      cnt = tot;
    }
  }
  const double wc = sqrt(q2) * sqrt(ksq) / sqrt((double)kD);
  const double var = cnt > 0.0 ? m2 / cnt : 0.0;
  p.Wc[seg * kD + d] = (float)(wc * var);
}

inline bool strides_ok(int64_t sb, int64_t st, int64_t sh) {
  return sb >= 0 && st >= 0 && sh >= 0 && sb % 8 == 0 && st % 8 == 0 && sh % 8 == 0;
}

inline kvq_status validate(const kvq_rdkv* r) {
  if (r == nullptr) return KVQ_ERR_INVALID;
  if (r->batch < 1 || r->n_kv_heads < 1 || r->n_q_heads < 1 || r->max_tokens < 0) return KVQ_ERR_INVALID;
  if (r->batch > KVQ_MAX_BATCH || r->max_tokens > KVQ_RDKV_MAX_TOKENS) return KVQ_ERR_UNSUPPORTED;
  if (r->head_dim != kD) return KVQ_ERR_UNSUPPORTED;
  if (r->n_q_heads % r->n_kv_heads) return KVQ_ERR_INVALID;
  const int G = r->n_q_heads / r->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVQ_ERR_UNSUPPORTED;
  if (r->n_q_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

}  // namespace rdkv
}  // namespace kvq

using namespace kvq;
using namespace kvq::rdkv;

extern "C" kvq_status kvq_rdkv_workspace_bytes(const kvq_rdkv* r, size_t* bytes) {
  const kvq_status s = validate(r);
  if (s != KVQ_OK) return s;
  if (bytes == nullptr) return KVQ_ERR_INVALID;
  *bytes = layout(r).total;
  return KVQ_OK;
}

extern "C" kvq_status kvq_rdkv_token_weights(const kvq_rdkv* r, const void* q, int64_t q_sb, int64_t q_st,
                                             int64_t q_sh, const void* k, int64_t k_sb, int64_t k_st, int64_t k_sh,
                                             const int32_t* n_tokens, float sm_scale, float* w, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  kvq_status s = validate(r);
  if (s != KVQ_OK) return s;
  if (q == nullptr || k == nullptr || n_tokens == nullptr || w == nullptr || workspace == nullptr)
    return KVQ_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(w, 4) || !aligned(workspace, 256)) return KVQ_ERR_INVALID;
  if (!strides_ok(q_sb, q_st, q_sh) || !strides_ok(k_sb, k_st, k_sh)) return KVQ_ERR_INVALID;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID;
  const Layout L = layout(r);
  if (workspace_bytes < L.total) return KVQ_ERR_INVALID;
  AttnParams p{};
  int nmax = 0;
  for (int b = 0; b < r->batch; ++b) {
    if (n_tokens[b] < 0) return KVQ_ERR_INVALID;
    if (n_tokens[b] > r->max_tokens) return KVQ_ERR_CAPACITY;
    p.n[b] = n_tokens[b];
    nmax = n_tokens[b] > nmax ? n_tokens[b] : nmax;
  }
  if (nmax == 0) return KVQ_OK;
  p.q = static_cast<const __half*>(q);
  p.k = static_cast<const __half*>(k);
  p.q_sb = q_sb; p.q_st = q_st; p.q_sh = q_sh;
  p.k_sb = k_sb; p.k_st = k_st; p.k_sh = k_sh;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.Hq = r->n_q_heads;
  p.Hkv = r->n_kv_heads;
  p.G = r->n_q_heads / r->n_kv_heads;
  p.T = r->max_tokens;
  p.Tl = lse_stride(r->max_tokens);
  p.lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.lse);
  p.w = w;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nqb = (r->max_tokens + kBlk - 1) / kBlk;
  const int smem1 = 2 * kTile, smem2 = 2 * kTile + 2 * kBlk * 4;
  if (cudaFuncSetAttribute(rowstats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1) != cudaSuccess ||
      cudaFuncSetAttribute(colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2) != cudaSuccess)
    return KVQ_ERR_CUDA;
  rowstats_kernel<<<dim3(nqb, r->n_q_heads, r->batch), 128, smem1, st>>>(p);
  colsum_kernel<<<dim3(nqb, r->n_kv_heads, r->batch), 128, smem2, st>>>(p);
  return launch_status();
}

extern "C" kvq_status kvq_rdkv_allocate(const kvq_rdkv* r, const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                                        const void* k, const void* v, int64_t k_sb, int64_t k_st, int64_t k_sh,
                                        const int32_t* n_tokens, const int32_t* t_old, const float* w,
                                        float v_avg_bits, float k_avg_bits, uint8_t* v_width, int32_t max_old,
                                        uint8_t* k_width, float* W_t, float* W_c, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  kvq_status s = validate(r);
  if (s != KVQ_OK) return s;
  if (q == nullptr || k == nullptr || v == nullptr || n_tokens == nullptr || t_old == nullptr || w == nullptr ||
      v_width == nullptr || k_width == nullptr || workspace == nullptr)
    return KVQ_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(w, 4) || !aligned(workspace, 256) ||
      (W_t != nullptr && !aligned(W_t, 4)) || (W_c != nullptr && !aligned(W_c, 4)))
    return KVQ_ERR_INVALID;
  if (!strides_ok(q_sb, q_st, q_sh) || !strides_ok(k_sb, k_st, k_sh)) return KVQ_ERR_INVALID;
  if (!(v_avg_bits >= 0.f) || !(k_avg_bits >= 0.f) || !std::isfinite(v_avg_bits) || !std::isfinite(k_avg_bits))
    return KVQ_ERR_INVALID;
  if (max_old < 0) return KVQ_ERR_INVALID;
  const Layout L = layout(r);
  if (workspace_bytes < L.total) return KVQ_ERR_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int Hkv = r->n_kv_heads, G = r->n_q_heads / r->n_kv_heads;
  CostParams cp{};
  AllocParams av{}, ak{};
  ChanParams ch{};
  int max_t_old = 0;
  for (int b = 0; b < r->batch; ++b) {
    if (n_tokens[b] < 0 || t_old[b] < 0 || t_old[b] > n_tokens[b]) return KVQ_ERR_INVALID;
    if (n_tokens[b] > r->max_tokens || t_old[b] > max_old) return KVQ_ERR_CAPACITY;
    const double vb = std::floor((double)v_avg_bits * (double)t_old[b]);
    const double kbits = std::floor((double)k_avg_bits * (double)kD);
    cp.t_old[b] = t_old[b];
    av.n[b] = t_old[b];
    av.budget[b] = vb > 2147483647.0 ? 2147483647 : (int32_t)vb;
    ak.n[b] = kD;
    ak.budget[b] = kbits > 2147483647.0 ? 2147483647 : (int32_t)kbits;
    ch.n[b] = n_tokens[b];
    ch.t_old[b] = t_old[b];
    max_t_old = t_old[b] > max_t_old ? t_old[b] : max_t_old;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // phase 2: token costs, V widths
  cp.v = static_cast<const __half*>(v);
  cp.sb = k_sb; cp.st = k_st; cp.sh = k_sh;
  cp.w = w;
  cp.T = r->max_tokens;
  cp.Hkv = Hkv;
  cp.W = W_t != nullptr ? W_t : reinterpret_cast<float*>(ws + L.wt);
  cp.wstride = W_t != nullptr ? max_old : r->max_tokens;
  if (max_t_old > 0) token_cost_kernel<<<dim3((max_t_old + 7) / 8, Hkv, r->batch), 256, 0, st>>>(cp);
  av.W = cp.W;
  av.wstride = cp.wstride;
  av.out = v_width;
  av.ostride = max_old;
  av.Hkv = Hkv;
  alloc_kernel<true><<<dim3(Hkv, r->batch), 1024, 0, st>>>(av);
  // phase 3: channel statistics over the kept old tokens, K widths
  ch.q = static_cast<const __half*>(q);
  ch.k = static_cast<const __half*>(k);
  ch.q_sb = q_sb; ch.q_st = q_st; ch.q_sh = q_sh;
  ch.k_sb = k_sb; ch.k_st = k_st; ch.k_sh = k_sh;
  ch.v_width = v_width;
  ch.vw_stride = max_old;
  ch.Hkv = Hkv;
  ch.G = G;
  ch.nch = nchunks(r->max_tokens);
  ch.part = reinterpret_cast<float*>(ws + L.part);
  ch.Wc = W_c != nullptr ? W_c : reinterpret_cast<float*>(ws + L.wc);
  if (r->max_tokens > 0)
    channel_partial_kernel<<<dim3(nchunks(r->max_tokens), Hkv, r->batch), kD, 0, st>>>(ch);
  channel_cost_kernel<<<dim3(Hkv, r->batch), kD, 0, st>>>(ch);
  ak.W = ch.Wc;
  ak.wstride = kD;
  ak.out = k_width;
  ak.ostride = kD;
  ak.Hkv = Hkv;
  alloc_kernel<false><<<dim3(Hkv, r->batch), 1024, 0, st>>>(ak);
  return launch_status();
}
