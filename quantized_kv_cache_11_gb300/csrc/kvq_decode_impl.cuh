// Fused-dequant split-K decode attention over the uniform packed cache: the
// kernel templates, shared by the entry points of kvq_decode.cu and
// kvq_decode_rope.cu.
//
// What it computes ("KV-cache quantization axes", ihal.it, paragraphs 2 and 5;
// VQKV summary, section 2 "decoding phase"): for every sequence b and query head
// hq (KV head h = hq / G), out = softmax(sm_scale * q . K_hat^T) . V_hat over the
// quantized tokens (K_hat = zero + scale * code, dequantized inside the
// products, never written out) and the fp16 tail tokens.
//
// How:
// * Work partition (stream-K): the work items of every (sequence, KV head) --
//   its quantized 32-token groups, then its fp16 tail chunks (each weighted as
//   kTailWeight items) -- are laid end to end, and the list is cut into equal
//   contiguous ranges, one per resident CTA, so ragged batches stay balanced.
//   Inside a CTA each warp streams its own sub-range of groups through a private
//   multi-stage cp.async ring in shared memory.
// * Per 32-token group (one warp, the whole GQA group of G query heads):
//   Q.K^T on tensor cores (mma.m16n8k16, fp16 in, fp32 accumulate).  The A
//   operand is the codes themselves: one mask per register leaves a code pair
//   in the low mantissa bits of two fp16 halves with a zero exponent, which
//   read as the subnormals c * 2^(p-24) (p = the codes' bit position; the
//   tensor cores take fp16 subnormals exactly).  p depends only on the
//   fragment row, so the power of two leaves the fp32 results per row.
//   B = q * scale, split into two fp16 halves (hi = fp16(q*s), lo = q*s - hi,
//   exact), in separate columns, so the per-channel scale is applied to q once
//   per group.  The zero points enter through one more small MMA (rows = zero
//   points).  Online softmax in fp32; P.V likewise with B = p * scale per
//   32-channel value group, split into hi and lo fp16 columns (exact: the
//   columns of the other heads' lo halves are otherwise empty), the value zero
//   points and the softmax denominator (a row of ones) from one small MMA.
// * Splits are merged by log-sum-exp; the last CTA to finish a (sequence, KV
//   head) merges and writes the output, then resets its counter.  No spin-wait.
#pragma once

#include <cmath>

#include "kvq_common.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kTailWeight = 3;  // a 32-token fp16 tail chunk counts as this many groups
// Polls of an mbarrier before a wait gives up (each poll may suspend the thread
// briefly): far longer than any copy takes, short enough to end a stuck kernel.
constexpr uint32_t kMaxPolls = 1u << 22;

// ROPE: the keys are stored before the rotary position embedding and rotated to
// their positions after dequantization (the K side then runs on CUDA cores).
// CPS: CTAs per SM (1, 2 or 4; the 2- and 4-bit decode without RoPE only).
// Several smaller CTAs per SM suit caches of many short (sequence, KV head)
// segments: each CTA then holds about one segment piece, and the pieces' set-up
// and merges overlap on the SM instead of running one after another.
// Pre-RoPE decode at 2 and 4 bits: the part of the kvq_rope_table table that
// holds the cos/sin of the offsets o within a 32-token block as fp16 pieces
// times 2^14 (hi: at most 11 - b significant bits, so that a b-bit code times it
// is exact in fp16; lo: the fp16 of the rest), in the order the tensor-core K
// side loads them.  Row o (< 56) holds, for k-tile kt, lane column tig and piece (hi, lo),
// 16 bytes: half2 (cos, sin) at (o, pair 8kt+tig), (o+8, that pair), (o, pair
// 8kt+tig+4), (o+8, that pair): the mma A quad of token rows o, o+8.  Rows are
// padded by 16 bytes (conflict-free 16-byte loads across a warp's 8 rows).
constexpr int kRopeTrigRows = 56;
constexpr int kRopeTrigRow = 8 * 4 * 2 * 16 + 16;
constexpr int kRopeTrigBytes = kRopeTrigRows * kRopeTrigRow;
// row 0's padding: a tag and the code width the pieces were cut for
constexpr int kRopeTrigTagOffset = 8 * 4 * 2 * 16;
constexpr uint32_t kRopeTrigTag = 0x5251564Bu;

template <int D, int BITS, int G, bool ROPE = false, int CPS = 1>
struct DecodeCfg {
  using T = Tile<D, BITS>;
  static constexpr int TB = T::kBytes;
  static constexpr int KMETA = 4 * D;  // [2][D] halves
  static constexpr int VMETA = 4 * D;  // [2][D/32][32] halves
  static constexpr int BASE = ROPE ? D / 2 * 8 : 0;  // cos/sin of the group's first position block
  // groups per stage: two consecutive groups of a segment are staged and decoded
  // together at 2 bits (one wait, one set of copies and one softmax maximum per
  // 64 tokens)
  static constexpr int GPI = (BITS == 2 && !ROPE) ? 2 : 1;
  // stage layout: the key codes of its GPI groups, their value codes, their key
  // metadata, their value metadata (each array as consecutive groups, as in the
  // cache, so that one bulk copy per array fills it), then (ROPE) the cos/sin row
  static constexpr int STAGE1 = 2 * TB + KMETA + VMETA + BASE;  // bytes of one group
  static constexpr int STAGE = GPI * (2 * TB + KMETA + VMETA) + BASE;
  static constexpr int OFF_VC = GPI * TB, OFF_KM = 2 * GPI * TB, OFF_VM = 2 * GPI * TB + GPI * KMETA,
                       OFF_BASE = GPI * (2 * TB + KMETA + VMETA);
  static constexpr int NT = (2 * G + 7) / 8;  // 8-column n-tiles: column 2g = hi, 2g+1 = lo
  static constexpr int KT = D / 16;
  static constexpr int NWL = T::kWordsPerLane;
  static constexpr int PPW = T::kPairsPerWord;
  // 16 warps per SM for 2- and 4-bit codes, as one CTA (fewer split-K partials
  // per segment) or as CPS CTAs of 16 / CPS warps (12 warps with ROPE: its stage
  // ring, offset piece table and fp32 q must fit)
  static_assert(CPS == 1 || (!ROPE && BITS != 8), "several CTAs per SM only without RoPE, at 2 and 4 bits");
  static constexpr int WARPS = BITS == 8 ? 4 : (ROPE ? 12 : 16 / CPS);
  static constexpr int NSTAGE = BITS == 8 || (ROPE && BITS == 2) ? 3 : 2;
  // ROPE at 2 and 4 bits: the rotated keys' products on tensor cores (pieces of
  // the offsets' cos/sin in shared memory); at 8 bits on CUDA cores
  static constexpr bool RTC = ROPE && BITS != 8;
  // q pairs held in registers (one n-tile) instead of re-read from shared memory
  static constexpr bool QREG = false;
  static constexpr int MIN_CTAS = CPS;
  static constexpr int PSTRIDE = D + 4;  // floats per head in a partial: m, l, pad, pad, o[D]
  static constexpr int RING = WARPS * NSTAGE * STAGE;
  static constexpr int PSROW = 48;                   // halves per head row of the p~ exchange
  static constexpr int PS = WARPS * G * PSROW * 2;   // p~ exchange, bytes
  static constexpr int ZERO = 4 * D;                 // zero row for lanes without a metadata row
  static constexpr int PREFIX = ((KVQ_MAX_BATCH + 1) * 4 + 15) / 16 * 16;
  static constexpr int QS = NT * 4 * (D / 2) * 4;     // q pairs of the segment's heads, lane order
  static constexpr int MBAR = (WARPS * NSTAGE + 1) * 8;  // one mbarrier per stage + the merge's
  // cos/sin of the offsets 0..63 within a block: fp16 pieces (RTC) or fp32
  static constexpr int INTRA = ROPE ? (RTC ? kRopeTrigBytes : 64 * (D / 2) * 8) : 0;
  static constexpr int QF = ROPE ? NT * 4 * D * 4 : 0;         // fp32 q of the segment's heads
  static constexpr int SMEM = RING + PS + ZERO + PREFIX + QS + INTRA + QF + MBAR;
  static_assert(SMEM <= 232448, "fits the shared memory of one CTA");
  // the final merge keeps its weights ([partials][G] + G floats) in the ring:
  // up to RING / (4 G) - 1 partials per segment (checked at launch)
  static constexpr int MAX_PARTS = RING / (4 * G) - 1;
  static_assert(WARPS * G * PSTRIDE * 4 <= RING, "warp partials reuse the stage ring");
  static_assert(NSTAGE * STAGE >= G * PSTRIDE * 4, "a warp's partial fits its ring slice");
  static_assert(PS % 16 == 0 && RING % 16 == 0 && ZERO % 16 == 0 && PREFIX % 16 == 0 &&
                    QS % 16 == 0 && INTRA % 16 == 0 && QF % 16 == 0 && STAGE % 16 == 0,
                "aligned shared regions (the mbarriers need 8 bytes, the copies 16)");
  static_assert(NSTAGE * STAGE >= kGroup * (2 * D + 16), "a staged tail chunk fits a warp's ring");
};

struct DecodeParams {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const __half* k_meta;
  const __half* v_meta;
  const __half* k_tail;
  const __half* v_tail;
  const int32_t* n_quant;
  const int32_t* n_tail;
  const int32_t* tail_head;
  const __half* k_sink;
  const __half* v_sink;
  const int32_t* n_sink;
  int32_t* error_flags;
  const __half* q;
  const float2* rope;  // ROPE: the table of kvq_rope_table (rows 0..63 offsets, 64 + m position blocks)
  const uint8_t* rope_trig;  // ROPE at 2 and 4 bits: its fp16 piece part (kRopeTrigBytes)
  float* out;
  int32_t* counters;
  float* part;
  float scale_log2;
  int32_t batch, hkv, max_groups, tail_cap, sink_cap;
  int32_t n_stream;
};

// Lengths as the decode sees them; an inconsistent sequence counts as empty.
struct SeqLen {
  int nq, nt, th, ns;
};
__device__ __forceinline__ SeqLen read_lengths(const DecodeParams& p, int b, bool report) {
  SeqLen s{p.n_quant[b], p.n_tail[b], p.tail_head[b], p.sink_cap > 0 ? p.n_sink[b] : 0};
  const bool ok = s.nq >= 0 && s.nq % kGroup == 0 && s.nq / kGroup <= p.max_groups && s.nt >= 0 &&
                  s.nt <= p.tail_cap && s.th >= 0 && s.th < p.tail_cap && s.th % kGroup == 0 && s.ns >= 0 &&
                  s.ns <= p.sink_cap && (s.ns == p.sink_cap || (s.nq == 0 && s.nt == 0));
  if (!ok) {
    if (report && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_BAD_LENGTHS);
    s = SeqLen{0, 0, 0, 0};
  }
  return s;
}

// Work items of one (sequence, KV head): its groups, kTailWeight per fp16 chunk
// (tail chunks, then sink chunks), and at least one (an empty sequence still
// needs its zero output written).
__device__ __forceinline__ int seq_items(const SeqLen& s) {
  const int n = s.nq / kGroup + kTailWeight * ((s.nt + kGroup - 1) / kGroup + (s.ns + kGroup - 1) / kGroup);
  return n > 0 ? n : 1;
}

// s_pref[b] = work items of the sequences before b (per KV head).
__device__ inline void build_prefix(const DecodeParams& p, int* s_pref) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int run = 0;
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int b = b0 + lane;
    int v = (b < p.batch) ? seq_items(read_lengths(p, b, blockIdx.x == 0)) : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += a;
    }
    if (b < p.batch) s_pref[b + 1] = run + v;
    run += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) s_pref[0] = 0;
}

// The stream-K CTA that owns global item x (CTA c owns [c*T/N, (c+1)*T/N)).
__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t total, int64_t n) {
  return ((x + 1) * n - 1) / total;
}

template <int D, int BITS, int G, bool ROPE = false, int CPS = 1>
struct Decoder {
  using C = DecodeCfg<D, BITS, G, ROPE, CPS>;
  static constexpr int NT = C::NT, KT = C::KT;
  // Bit position p of the codes that unpack8 puts in register 4 mt + i (row half
  // rh = i & 1 of an mma A fragment; never dependent on the k-half i >> 1): the
  // register holds the fp16 subnormals c * 2^(p - 24).  unit = 2^(24 - p).
  // p is at least 2: measured on GB300, a tensor-core dot product over such
  // subnormal operands keeps about 17 + p significant bits (relative error near
  // 2^-(17 + p) of the summed magnitudes; fp32-like from p = 6 on), so codes at
  // p = 0 would lose 7 bits against the fp32 accumulation.
  static __host__ __device__ constexpr int pos(int mt, int rh) {
    return 2 + (BITS == 2 ? 4 * mt + 2 * rh : (BITS == 4 ? 4 * rh : 0));
  }
  static __host__ __device__ constexpr float unit(int mt, int rh) { return (float)(1 << (24 - pos(mt, rh))); }
  static constexpr uint32_t kSixteenth = 0x2C002C00u;  // half2(1/16, 1/16)
  static constexpr uint32_t kOnes = 0x3C003C00u;  // half2(1, 1)

  // Per-warp running state of the online softmax for the G heads.
  float m[NT];
  float o[KT][NT][4];  // P.V accumulators: rows = channels, columns (head, hi|lo)
  float zc[NT][4];     // value-constant MMA: zero points, scale sums, row 12 = sum p~
  const uint32_t* qs;      // q pairs of column 8nt+gid (head 4nt + gid/2) in shared memory
  uint4 qr[C::QREG ? KT / 2 : 1];  // QREG: the same pairs in registers, k-tiles (kt, kt + 1) per entry
  uint32_t nhl;            // half2(-hl): 0 for the hi column, -1 for the lo column
  uint32_t ones_a;         // the ones row (row 12) of the value-constant MMA: lanes gid 4
  int lane, gid, tig, hl;
  const float* qf;         // ROPE: fp32 q [4 NT heads][D] in shared memory
  const float2* intra;     // ROPE: cos/sin(o theta_i) [64 offsets o][D/2] (fp32)
  const uint8_t* trig;     // RTC: the fp16 pieces of the offsets' cos/sin in shared memory

  // q_smem: the segment's q pairs in lane order ([4 NT heads][D/2] words)
  __device__ __forceinline__ void init(const uint32_t* q_smem) {
    lane = threadIdx.x & 31;
    gid = lane >> 2;
    tig = lane & 3;
    hl = gid & 1;
    nhl = hl ? 0xBC00BC00u : 0u;
    ones_a = gid == 4 ? kOnes : 0u;
    qs = q_smem + (gid >> 1) * (D / 2) + 4 * tig;
    if constexpr (C::QREG) {
#pragma unroll
      for (int k2 = 0; k2 < KT / 2; ++k2) qr[k2] = *reinterpret_cast<const uint4*>(qs + 16 * k2);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) zc[nt][i] = 0.f;
#pragma unroll
      for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[kt][nt][i] = 0.f;
    }
  }
  // K-side logits with the keys rotated to their positions (adjacent channel
  // pairs (2i, 2i+1) turned by pos * theta_i) in fp32 on CUDA cores.
  // keys(kt, h, k) gives the fp32 keys at channels c = 16kt + 2tig + 8h, c + 1 of
  // this lane's token rows 16(m/2) + gid + 8(m%2), m < 4; the chunk's token j sits
  // at position 32 m0 + roff + j, base = cos/sin(32 m0 theta_i) [D/2].
  template <class Keys>
  __device__ __forceinline__ void rope_logits(Keys keys, const float2* base, int roff, float scale_log2,
                                              float (&lg)[NT][2][2]) const {
    constexpr int GP = 4 * NT;
    float acc[4][GP];
#pragma unroll
    for (int m2 = 0; m2 < 4; ++m2)
#pragma unroll
      for (int g = 0; g < GP; ++g) acc[m2][g] = 0.f;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = 8 * kt + tig + 4 * h;
        const float2 bb = base[i];
        float2 qv[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) qv[g] = *reinterpret_cast<const float2*>(qf + g * D + 2 * i);
        float2 k[4];
        keys(kt, h, k);
#pragma unroll
        for (int m2 = 0; m2 < 4; ++m2) {
          const int tau = 16 * (m2 >> 1) + gid + 8 * (m2 & 1);
          const float2 in = intra[(roff + tau) * (D / 2) + i];
          const float cs = bb.x * in.x - bb.y * in.y, sn = bb.y * in.x + bb.x * in.y;
          const float k0 = k[m2].x * cs - k[m2].y * sn, k1 = k[m2].x * sn + k[m2].y * cs;
#pragma unroll
          for (int g = 0; g < GP; ++g) acc[m2][g] = fmaf(k0, qv[g].x, fmaf(k1, qv[g].y, acc[m2][g]));
        }
      }
#pragma unroll
    for (int m2 = 0; m2 < 4; ++m2)
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        acc[m2][g] += __shfl_xor_sync(0xffffffffu, acc[m2][g], 1);
        acc[m2][g] += __shfl_xor_sync(0xffffffffu, acc[m2][g], 2);
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          // this lane's head 4nt + tig
          float v = acc[2 * mt + r][0];
#pragma unroll
          for (int g = 1; g < GP; ++g) v = (g == 4 * nt + tig) ? acc[2 * mt + r][g] : v;
          lg[nt][mt][r] = v * scale_log2;
        }
  }

  // B registers of pairs i0 (r0) and i1 = i0 + 4 (r1) from the fp32 pair (v0, v1)
  // of this lane's own pair (i0 in the hi column's lane, i1 in the lo column's):
  // the hi column takes fp16(v), the lo column fp16(v - fp16(v)); each lane keeps
  // the piece of its own column and passes the other to its partner (lane ^ 4,
  // the other column of the same head).  hlf = 0 (hi) or 1 (lo).
  __device__ __forceinline__ void exchange(float v0, float v1, float hlf, uint32_t& r0, uint32_t& r1) const {
    const __half2 h = __floats2half2_rn(v0, v1);
    const float2 hf = __half22float2(h);
    const uint32_t mine = h2_as_u32(__floats2half2_rn(fmaf(-hlf, hf.x, v0), fmaf(-hlf, hf.y, v1)));
    const uint32_t send = h2_as_u32(__floats2half2_rn(fmaf(hlf - 1.f, hf.x, v0), fmaf(hlf - 1.f, hf.y, v1)));
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 4);
    r0 = hl ? recv : mine;
    r1 = hl ? mine : recv;
  }

  // K-side logits of one pre-RoPE group on tensor cores (RTC).  The group's
  // tokens sit at positions 32 m + o, o = roff + row; with beta_i = 32 m theta_i
  // and alpha_i = o theta_i, the rotated key pair (R(alpha + beta) k).q equals
  // (R(alpha) k).q~ with q~ = R(-beta) q, that is
  //   cos(alpha) (k0 q~0 + k1 q~1) + sin(alpha) (k0 q~1 - k1 q~0),  k = s c + z.
  // Codes: registers c 2^(p - 24) times the hi and lo pieces (times 2^14) of cos
  // and sin(alpha) from the piece table (hi products exact: the hi piece has at
  // most 11 - BITS bits), against B = (s0 q~0, s1 q~1) and (s0 q~1, -s1 q~0);
  // zero points: the pieces themselves as the A quad, against (z.q~, z x q~).  B
  // values in hi/lo columns as elsewhere.  kw: the lane's code words; km: the
  // group's key metadata (lane order); base: cos/sin(beta_i) [D/2].
  __device__ __forceinline__ void rope_tc_logits(const uint32_t* kw, const uint32_t* km, const float2* base,
                                                 int roff, float scale_log2, float (&lg)[NT][2][2]) const {
    float acc[2][NT][4], zac[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][nt][i] = zac[mt][nt][i] = 0.f;
    const float hlf = hl ? 1.f : 0.f;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      // this lane's own pair: 8kt + tig in the hi column's lane, + 4 in the lo one's
      const int ip = 8 * kt + tig + 4 * hl;
      // (zero, scale) of channels 2 ip, 2 ip + 1 (the lane-order metadata quad holds
      // those of pair 8kt + tig, then of pair 8kt + tig + 4)
      const uint2 mv = *reinterpret_cast<const uint2*>(km + 16 * kt + 4 * tig + 2 * hl);
      const float2 zz = __half22float2(u32_as_h2(mv.x)), ss = __half22float2(u32_as_h2(mv.y));
      const float2 bb = base[ip];
      uint32_t bc[NT][2], bs[NT][2], bz[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // head 4nt + gid/2 (heads past G have q = 0 in shared memory)
        const float2 qa = *reinterpret_cast<const float2*>(qf + (4 * nt + (gid >> 1)) * D + 2 * ip);
        const float t0 = fmaf(bb.x, qa.x, bb.y * qa.y), t1 = fmaf(bb.x, qa.y, -bb.y * qa.x);
        exchange(ss.x * t0, ss.y * t1, hlf, bc[nt][0], bc[nt][1]);
        exchange(ss.x * t1, -ss.y * t0, hlf, bs[nt][0], bs[nt][1]);
        exchange(fmaf(zz.x, t0, zz.y * t1), fmaf(zz.x, t1, -zz.y * t0), hlf, bz[nt][0], bz[nt][1]);
      }
      // the codes as in the plain decode, fp16 subnormals c 2^(p - 24); the pieces
      // are stored times 2^14, so the products c t 2^(p - 10) are normal fp16 and
      // exact (except for |c t| < 2^-4, where the subnormal grid of 2^-24 bounds
      // the absolute error by 2^-25 in those units)
      uint32_t a[8];
      unpack8(kw, 8 * kt, a);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint8_t* row = trig + (roff + 16 * mt + gid) * kRopeTrigRow + (kt * 4 + tig) * 32;
        const uint4 th = *reinterpret_cast<const uint4*>(row);
        const uint4 tl = *reinterpret_cast<const uint4*>(row + 16);
        const uint32_t x[4] = {a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3]};
        const uint32_t thv[4] = {th.x, th.y, th.z, th.w}, tlv[4] = {tl.x, tl.y, tl.z, tl.w};
        uint32_t ach[4], acl[4], ash[4], asl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 xe = u32_as_h2(x[e]), h = u32_as_h2(thv[e]), l = u32_as_h2(tlv[e]);
          ach[e] = h2_as_u32(__hmul2(xe, __low2half2(h)));
          ash[e] = h2_as_u32(__hmul2(xe, __high2half2(h)));
          acl[e] = h2_as_u32(__hmul2(xe, __low2half2(l)));
          asl[e] = h2_as_u32(__hmul2(xe, __high2half2(l)));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816(acc[mt][nt], ach, bc[nt][0], bc[nt][1]);
          mma_16816(acc[mt][nt], acl, bc[nt][0], bc[nt][1]);
          mma_16816(acc[mt][nt], ash, bs[nt][0], bs[nt][1]);
          mma_16816(acc[mt][nt], asl, bs[nt][0], bs[nt][1]);
          mma_16816(zac[mt][nt], thv, bz[nt][0], bz[nt][1]);
          mma_16816(zac[mt][nt], tlv, bz[nt][0], bz[nt][1]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          lg[nt][mt][r] = scale_log2 * fmaf(acc[mt][nt][2 * r] + acc[mt][nt][2 * r + 1],
                                            (float)(1 << 10) / (float)(1 << pos(mt, r)),
                                            (zac[mt][nt][2 * r] + zac[mt][nt][2 * r + 1]) * 0x1p-14f);
  }

  // q pairs (kt, r) and (kt + 1, r) of this lane's column in n-tile nt (kt even)
  __device__ __forceinline__ uint4 qpairs(int nt, int kt) const {
    if constexpr (C::QREG) return qr[kt / 2];
    return *reinterpret_cast<const uint4*>(qs + nt * 4 * (D / 2) + 8 * kt);
  }

  // Operands of pairs P0 .. P0+7 of the lane's words (P0 a multiple of 8): one
  // mask per register, on the word shifted left by 2 or right by 6, leaves each
  // code pair in the mantissa bits [p, p+b) of the two halves, exponent 0.  Bit
  // positions by register: 2 bits 2,4,2,4 | 6,8,6,8; 4 bits 2,6,2,6; 8 bits 2
  // (see pos()).
  static __device__ __forceinline__ void unpack8(const uint32_t* w, int P0, uint32_t (&a)[8]) {
    if (BITS == 2) {
      const uint32_t w0 = w[P0 / 8], x = w0 << 2, y = w0 >> 6;
      a[0] = x & 0x000C000Cu;  a[1] = x & 0x00300030u;  a[2] = y & 0x000C000Cu;  a[3] = y & 0x00300030u;
      a[4] = x & 0x00C000C0u;  a[5] = x & 0x03000300u;  a[6] = y & 0x00C000C0u;  a[7] = y & 0x03000300u;
    } else if (BITS == 4) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = w[P0 / 4 + h], x = w0 << 2, y = w0 >> 6;
        a[4 * h + 0] = x & 0x003C003Cu;
        a[4 * h + 1] = x & 0x03C003C0u;
        a[4 * h + 2] = y & 0x003C003Cu;
        a[4 * h + 3] = y & 0x03C003C0u;
      }
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t x = w[P0 / 2 + h];
        a[2 * h + 0] = (x << 2) & 0x03FC03FCu;
        a[2 * h + 1] = (x >> 6) & 0x03FC03FCu;
      }
    }
  }

  // hi column: fp16(x*y); lo column: x*y - fp16(x*y) (exact: x*y has <= 22 bits).
  __device__ __forceinline__ uint32_t split_mul(uint32_t a, uint32_t b) const {
    const __half2 x = u32_as_h2(a), y = u32_as_h2(b);
    const __half2 hi = __hmul2_rn(x, y);
    return h2_as_u32(__hfma2(x, y, __hmul2_rn(hi, u32_as_h2(nhl))));
  }

  // Move the running maximum of every head to max(m, mloc) and rescale the
  // accumulators to it (called only when some head's chunk maximum passed its
  // running maximum by more than kLazyRescale).
  __device__ __forceinline__ void rescale(const float (&mloc)[NT]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float mnew = fmaxf(m[nt], mloc[nt]);
      const float alpha = (mnew == m[nt]) ? 1.f : fast_exp2(m[nt] - mnew);
      m[nt] = mnew;
#pragma unroll
      for (int i = 0; i < 4; ++i) zc[nt][i] *= alpha;
#pragma unroll
      for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[kt][nt][i] *= alpha;
    }
  }

  // Online softmax over one 32-token chunk.  lg[nt][mt][r]: log2-domain logits of
  // token 16mt + gid + 8r for head 4nt + tig.  Writes p~ (fp16) to ps[g][t].
  __device__ __forceinline__ void softmax(float (&lg)[NT][2][2], __half* ps) {
    bool need = false;
    float mloc[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float mx = fmaxf(fmaxf(lg[nt][0][0], lg[nt][0][1]), fmaxf(lg[nt][1][0], lg[nt][1][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      mloc[nt] = mx;
      need |= mx > m[nt] + kLazyRescale;
    }
    if (__any_sync(0xffffffffu, need)) rescale(mloc);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = 4 * nt + tig;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const __half2 ph = __floats2half2_rn(fast_exp2(lg[nt][mt][0] - m[nt]),
                                             fast_exp2(lg[nt][mt][1] - m[nt]));
        if (g < G) {
          ps[g * C::PSROW + 16 * mt + gid] = __low2half(ph);
          ps[g * C::PSROW + 16 * mt + gid + 8] = __high2half(ph);
        }
      }
    }
    __syncwarp();
  }

  // p~ pairs for the V-side B fragments: column 8nt+gid (head 4nt + gid/2), tokens
  // 16kt + 2tig + 8r and +1.  with_lo: the lo columns (odd gid) hold p~ too (the
  // quantized groups split p~ * scale into hi and lo columns); otherwise zero
  // (the fp16 chunks multiply p~ itself, exact in one column).
  __device__ __forceinline__ void load_pp(const __half* ps, uint32_t (&pp)[NT][2][2], bool with_lo) const {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = 4 * nt + (gid >> 1);
#pragma unroll
      for (int kt = 0; kt < 2; ++kt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          pp[nt][kt][r] = (g < G && (with_lo || !hl))
                              ? *reinterpret_cast<const uint32_t*>(ps + g * C::PSROW + 16 * kt + 2 * tig + 8 * r)
                              : 0u;
    }
  }

  // Online softmax over one 32-token chunk, straight into the P.V B fragments
  // (both columns of a head hold p~, as load_pp(.., true) gives): the p~ pairs of a
  // lane's C-layout rows are transposed in registers (movmatrix), as for two-group
  // stages, instead of a round trip through shared memory.
  __device__ __forceinline__ void softmax_pp(const float (&lg)[NT][2][2], uint32_t (&pp)[NT][2][2]) {
    bool need = false;
    float mloc[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float mx = fmaxf(fmaxf(lg[nt][0][0], lg[nt][0][1]), fmaxf(lg[nt][1][0], lg[nt][1][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      mloc[nt] = mx;
      need |= mx > m[nt] + kLazyRescale;
    }
    if (__any_sync(0xffffffffu, need)) rescale(mloc);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float pf = fast_exp2(lg[nt][mt][r] - m[nt]);
          if (G % 4 != 0 && 4 * nt + tig >= G) pf = 0.f;
          pp[nt][mt][r] = movmatrix_trans(h2_as_u32(__floats2half2_rn(pf, pf)));
        }
  }

  // P.V of one staged group (value codes vc, value metadata vm) with the B
  // fragments pp of its p~ (column 8nt+gid, tokens 16kt + 2tig + 8r, +1), into o
  // and zc.  At 2 bits the codes of tokens 16..31 sit 4 bits above those of
  // tokens 0..15 of the same row (pos(1, r) = pos(0, r) + 4): their p~ is divided
  // by 16 (exactly, a power of two) so that both k-tiles share a unit.
  __device__ __forceinline__ void pv_group(const uint8_t* vc, const uint8_t* vm8, const uint32_t (&pp)[NT][2][2],
                                           const uint32_t* zrow) {
    uint32_t pv[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        pv[nt][0][r] = pp[nt][0][r];
        pv[nt][1][r] = BITS == 2 ? h2_as_u32(__hmul2(u32_as_h2(pp[nt][1][r]), u32_as_h2(kSixteenth))) : pp[nt][1][r];
      }
    const uint4* v4 = reinterpret_cast<const uint4*>(vc);
    uint32_t vw[C::NWL];
#pragma unroll
    for (int ch = 0; ch < C::NWL / 4; ++ch) {
      const uint4 v = v4[ch * 32 + lane];
      vw[4 * ch] = v.x; vw[4 * ch + 1] = v.y; vw[4 * ch + 2] = v.z; vw[4 * ch + 3] = v.w;
    }
    // value metadata, lane order: pair (j, kt, r) of this lane at 16j + 4tig + 2kt + r
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(vm8);
    const uint32_t* vsl = vm + 4 * tig;          // scale pairs
    const uint32_t* vzl = vm + D / 2 + 4 * tig;  // zero pairs
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const uint4 sv = *reinterpret_cast<const uint4*>(vsl + 16 * j);
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        const uint32_t vs0 = kt ? sv.z : sv.x, vs1 = kt ? sv.w : sv.y;
        uint32_t b[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          b[nt][0] = split_mul(pv[nt][kt][0], vs0);
          b[nt][1] = split_mul(pv[nt][kt][1], vs1);
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const int mt = 2 * j + mi;
          uint32_t a8[8];
          unpack8(vw, mt * 8, a8);  // pairs of (mt, kt = 0) then (mt, kt = 1)
          const uint32_t a[4] = {a8[4 * kt], a8[4 * kt + 1], a8[4 * kt + 2], a8[4 * kt + 3]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a, b[nt][0], b[nt][1]);
        }
      }
    }
    // constant-MMA rows (tokens 16kt + 2tig (+8r)): 0..D/32-1 = zero points of group
    // j; 12 = ones (the softmax denominator); B = p~ as rounded
    const uint4 v0 = *reinterpret_cast<const uint4*>(gid < D / 32 ? vzl + 16 * gid : zrow);
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      const uint32_t ac[4] = {kt ? v0.z : v0.x, ones_a, kt ? v0.w : v0.y, ones_a};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(zc[nt], ac, pp[nt][kt][0], pp[nt][kt][1]);
    }
  }

  // One quantized 32-token group staged in shared memory: key codes kc, value
  // codes vc, key metadata km8, value metadata vm8 (and, ROPE, the cos/sin row
  // base of its position block).  zrow: a zero row of at least D/2 words in
  // shared memory.  roff (ROPE): the group's first position modulo 32.
  __device__ __forceinline__ void quant_group(const uint8_t* kc, const uint8_t* vc, const uint8_t* km8,
                                              const uint8_t* vm8, const uint8_t* base, __half* ps,
                                              const uint32_t* zrow, float scale_log2, int roff = 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(kc);
    uint32_t kw[C::NWL];
#pragma unroll
    for (int ch = 0; ch < C::NWL / 4; ++ch) {
      const uint4 v = s4[ch * 32 + lane];
      kw[4 * ch] = v.x; kw[4 * ch + 1] = v.y; kw[4 * ch + 2] = v.z; kw[4 * ch + 3] = v.w;
    }
    // key metadata, lane order: word 16kt + 4tig + 2r + f = the zero points (f = 0) or
    // scales (f = 1) of channels 16kt + 2tig + 8r and +1
    const uint32_t* km = reinterpret_cast<const uint32_t*>(km8);
    float lg[NT][2][2];
    if constexpr (C::RTC) {
      rope_tc_logits(kw, km, reinterpret_cast<const float2*>(base), roff, scale_log2, lg);
    } else if constexpr (ROPE) {
      // the codes dequantized in fp32: pair P = 8kt + 4mt + (r + 2h) of word P / PPW
      auto keys = [&](int kt, int h, float2 (&k)[4]) {
        const int w = 16 * kt + 4 * tig + 2 * h;
        const float2 zp = __half22float2(u32_as_h2(km[w])), sc = __half22float2(u32_as_h2(km[w + 1]));
#pragma unroll
        for (int m2 = 0; m2 < 4; ++m2) {
          const int P = 8 * kt + 4 * (m2 >> 1) + (m2 & 1) + 2 * h;
          const uint32_t word = kw[P / C::PPW];
          const int bp = slot_bitpos<BITS>(P % C::PPW);
          constexpr uint32_t kMask = (1u << BITS) - 1u;
          const float x0 = __uint_as_float(0x4B000000u | ((word >> bp) & kMask)) - 8388608.f;
          const float x1 = __uint_as_float(0x4B000000u | ((word >> (16 + bp)) & kMask)) - 8388608.f;
          k[m2] = make_float2(fmaf(sc.x, x0, zp.x), fmaf(sc.y, x1, zp.y));
        }
      };
      rope_logits(keys, reinterpret_cast<const float2*>(base), roff, scale_log2, lg);
    } else {
      // one 16-byte load per k-tile, (zero r0, scale r0, zero r1, scale r1), is the
      // constant product's A quad: rows gid hold the zero points (every row alike,
      // so each lane's own column sum is q.z), rows gid + 8 the scales or zeros,
      // whose products are not read
      const uint32_t* kmt = km + 4 * tig;
      constexpr int CH = 2;  // two independent accumulation chains over kt (shorter MMA dependency)
      float sacc[CH][2][NT][4];
      float cacc[CH][NT][4];
  #pragma unroll
      for (int ch = 0; ch < CH; ++ch)
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
        for (int i = 0; i < 4; ++i) { sacc[ch][0][nt][i] = 0.f; sacc[ch][1][nt][i] = 0.f; cacc[ch][nt][i] = 0.f; }
  #pragma unroll
      for (int kt2 = 0; kt2 < KT; kt2 += 2) {
        const int ch = (kt2 / 2) % CH;
        uint4 qv[NT];
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt) qv[nt] = qpairs(nt, kt2);
        // (measured: at 2 and 4 bits both k-tiles' loads up front and the whole quad
        // as the operand run fastest (4-bit 128k step 35.5 -> 35.0 us once p~ no
        // longer went through shared memory); at 8 bits, with 4 warps per CTA and
        // more registers per code word, a load per k-tile with the scale rows zeroed)
        constexpr bool kHoist = BITS != 8;
        uint4 mvp[2];
        if (kHoist) {
          mvp[0] = *reinterpret_cast<const uint4*>(kmt + 16 * kt2);
          mvp[1] = *reinterpret_cast<const uint4*>(kmt + 16 * kt2 + 16);
        }
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kt = kt2 + h;
          const uint4 mv = kHoist ? mvp[h] : *reinterpret_cast<const uint4*>(kmt + 16 * kt);
          const uint32_t sp0 = mv.y, sp1 = mv.w;
          uint32_t a[8];
          unpack8(kw, kt * 8, a);  // pairs of (kt, mt = 0) then (kt, mt = 1)
          const uint32_t a0[4] = {a[0], a[1], a[2], a[3]};
          const uint32_t a1[4] = {a[4], a[5], a[6], a[7]};
          const uint32_t ac[4] = {mv.x, kHoist ? mv.y : 0u, mv.z, kHoist ? mv.w : 0u};
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint32_t q0 = h ? qv[nt].z : qv[nt].x, q1 = h ? qv[nt].w : qv[nt].y;
            const uint32_t b0 = split_mul(q0, sp0);
            const uint32_t b1 = split_mul(q1, sp1);
            mma_16816(sacc[ch][0][nt], a0, b0, b1);
            mma_16816(sacc[ch][1][nt], a1, b0, b1);
            mma_16816(cacc[ch][nt], ac, q0, q1);
          }
        }
      }
  #pragma unroll
      for (int c2 = 1; c2 < CH; ++c2)
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
          for (int i = 0; i < 4; ++i) {
            sacc[0][0][nt][i] += sacc[c2][0][nt][i];
            sacc[0][1][nt][i] += sacc[c2][1][nt][i];
            cacc[0][nt][i] += cacc[c2][nt][i];
          }
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // sum_d q z of head 4nt+tig, plus the code products brought to unit scale
        // (token row 16mt + gid + 8r holds codes at bit position pos(mt, r))
        const float zq = cacc[0][nt][0] * scale_log2;
  #pragma unroll
        for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
          for (int r = 0; r < 2; ++r)
            lg[nt][mt][r] = fmaf(sacc[0][mt][nt][2 * r] + sacc[0][mt][nt][2 * r + 1], scale_log2 * unit(mt, r), zq);
      }
    }
    uint32_t pp[NT][2][2];
    softmax_pp(lg, pp);
    pv_group(vc, vm8, pp, zrow);
    __syncwarp();
  }

  // Two consecutive quantized groups staged together (stage layout of DecodeCfg:
  // GPI = 2), decoded as one 64-token chunk: one softmax maximum, each group's
  // zero-point product from its own 16-byte metadata load as it stands, and the
  // p~ of both turned into P.V operands in registers (movmatrix), without a
  // shared-memory round trip.
  __device__ __forceinline__ void quant_pair(const uint8_t* stage, const uint32_t* zrow, float scale_log2) {
    static_assert(C::GPI == 2 && !ROPE, "two-group stages");
    float lg[2][NT][2][2];
    {
      float sacc[2][2][NT][4];  // [group][mt]
      float cacc[2][NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sacc[0][0][nt][i] = sacc[0][1][nt][i] = sacc[1][0][nt][i] = sacc[1][1][nt][i] = 0.f;
          cacc[0][nt][i] = cacc[1][nt][i] = 0.f;
        }
      // the key side of each group in turn (fewer live registers than both at
      // once); the zero-point product of both groups runs with the second
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const uint4* k4 = reinterpret_cast<const uint4*>(stage + x * C::TB);
        const uint32_t* kmt = reinterpret_cast<const uint32_t*>(stage + C::OFF_KM + x * C::KMETA) + 4 * tig;
        const uint32_t* kmo = reinterpret_cast<const uint32_t*>(stage + C::OFF_KM) + 4 * tig;  // first group's
#pragma unroll
        for (int kt4 = 0; kt4 < KT; kt4 += 4) {
          // the lane's code words of k-tiles kt4 .. kt4 + 3 (one word per k-tile at 2 bits)
          const uint4 v = k4[(kt4 / 4) * 32 + lane];
          const uint32_t kw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int kt = kt4 + kk;
            const uint4 mv = *reinterpret_cast<const uint4*>(kmt + 16 * kt);
            uint32_t a[8];
            unpack8(kw, kk * 8, a);
            const uint32_t a0[4] = {a[0], a[1], a[2], a[3]};
            const uint32_t a1[4] = {a[4], a[5], a[6], a[7]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 qv = qpairs(nt, kt & ~1);
              const uint32_t q0 = (kt & 1) ? qv.z : qv.x, q1 = (kt & 1) ? qv.w : qv.y;
              const uint32_t b0 = split_mul(q0, mv.y);
              const uint32_t b1 = split_mul(q1, mv.w);
              mma_16816(sacc[x][0][nt], a0, b0, b1);
              mma_16816(sacc[x][1][nt], a1, b0, b1);
              const uint32_t ac[4] = {mv.x, mv.y, mv.z, mv.w};
              mma_16816(cacc[x][nt], ac, q0, q1);
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const float zq = cacc[x][nt][0] * scale_log2;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
              lg[x][nt][mt][r] =
                  fmaf(sacc[x][mt][nt][2 * r] + sacc[x][mt][nt][2 * r + 1], scale_log2 * unit(mt, r), zq);
        }
    }
    // online softmax over the 64 tokens
    bool need = false;
    float mloc[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float mx = -INFINITY;
#pragma unroll
      for (int x = 0; x < 2; ++x)
        mx = fmaxf(mx, fmaxf(fmaxf(lg[x][nt][0][0], lg[x][nt][0][1]), fmaxf(lg[x][nt][1][0], lg[x][nt][1][1])));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      mloc[nt] = mx;
      need |= mx > m[nt] + kLazyRescale;
    }
    if (__any_sync(0xffffffffu, need)) rescale(mloc);
    // p~ to the P.V B fragments: lane (gid, tig) holds p~ of head 4nt + tig at
    // tokens 16mt + gid + 8r, i.e. the pair of columns (2tig, 2tig + 1) = (p~, p~)
    // of row gid of the 8 x 8 matrices [tokens 16mt + 8r + (0..7)] x [columns];
    // transposed in registers, lane (gid, tig) holds column gid (head gid/2's p~,
    // the hi column for even gid, the lo column for odd) at tokens 2tig, 2tig + 1:
    // the B fragment of P.V.
    uint32_t pp[2][NT][2][2];
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float pf = fast_exp2(lg[x][nt][mt][r] - m[nt]);
            if (G % 4 != 0 && 4 * nt + tig >= G) pf = 0.f;
            pp[x][nt][mt][r] = movmatrix_trans(h2_as_u32(__floats2half2_rn(pf, pf)));
          }
#pragma unroll
    for (int x = 0; x < 2; ++x)
      pv_group(stage + C::OFF_VC + x * C::TB, stage + C::OFF_VM + x * C::VMETA, pp[x], zrow);
    __syncwarp();
  }

  // One chunk of up to 32 fp16 tail tokens.  The rows are staged through the
  // warp's (idle) stage ring: keys first, then values, each as 32 rows of D
  // halves at a padded pitch (conflict-free fragment loads), missing tokens
  // zero-filled.  Fragments come from ldmatrix (keys) and ldmatrix.trans
  // (values, the transposed operand of P.V).
  static constexpr int kPitch = 2 * D + 16;  // bytes per staged row
  __device__ __forceinline__ void stage_rows(uint8_t* buf, const __half* base, int first, int count,
                                             int th, int R) const {
    constexpr int CPR = 2 * D / 16;  // 16-byte chunks per row
#pragma unroll 4
    for (int e = lane; e < kGroup * CPR; e += 32) {
      const int t = e / CPR, ch = e % CPR;
      const bool ok = t < count;
      const __half* src = base + (size_t)(ok ? (th + first + t) % R : 0) * D + ch * 8;
      cp_async_16_zfill(buf + t * kPitch + ch * 16, src, ok ? 16 : 0);
    }
    cp_async_commit();
  }
  // rope_base, roff (ROPE): cos/sin of the chunk's position block, its first
  // position modulo 32.
  __device__ __forceinline__ void tail_chunk(uint8_t* buf, const __half* kt_base, const __half* vt_base,
                                             int first, int count, int th, int R, __half* ps,
                                             float scale_log2, const float2* rope_base = nullptr, int roff = 0) {
    stage_rows(buf, kt_base, first, count, th, R);
    cp_async_wait<0>();
    __syncwarp();
    float lg[NT][2][2];
    if constexpr (ROPE) {
      auto keys = [&](int kt, int h, float2 (&k)[4]) {
#pragma unroll
        for (int m2 = 0; m2 < 4; ++m2) {
          const int row = 16 * (m2 >> 1) + gid + 8 * (m2 & 1), c = 16 * kt + 2 * tig + 8 * h;
          k[m2] = __half22float2(*reinterpret_cast<const __half2*>(buf + row * kPitch + c * 2));
        }
      };
      rope_logits(keys, rope_base, roff, scale_log2, lg);
      __syncwarp();
      stage_rows(buf, vt_base, first, count, th, R);  // overlaps the softmax below
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r)
            if (16 * mt + gid + 8 * r >= count) lg[nt][mt][r] = -INFINITY;
    } else {
    float sacc[2][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) { sacc[0][nt][i] = 0.f; sacc[1][nt][i] = 0.f; }
    // lane's ldmatrix row: matrix lane/8 -> (+8 rows if bit 0, +8 columns if bit 1)
    const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lcol = 8 * (lane >> 4);
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      uint32_t a[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
        ldmatrix_x4(a[mt], buf + (16 * mt + lrow) * kPitch + (16 * kt + lcol) * 2);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 qv = qpairs(nt, kt & ~1);
        const uint32_t q0 = (kt & 1) ? qv.z : qv.x, q1 = (kt & 1) ? qv.w : qv.y;
        mma_16816(sacc[0][nt], a[0], q0, q1);
        mma_16816(sacc[1][nt], a[1], q0, q1);
      }
    }
    __syncwarp();
    stage_rows(buf, vt_base, first, count, th, R);  // overlaps the softmax below
    // B = q in both columns of a head: use one of them
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          lg[nt][mt][r] = (16 * mt + gid + 8 * r) < count ? sacc[mt][nt][2 * r] * scale_log2 : -INFINITY;
    }
    softmax(lg, ps);
    uint32_t pp[NT][2][2];
    load_pp(ps, pp, false);
    cp_async_wait<0>();
    __syncwarp();
    // value rows: A[d][t] = v[t][d]; matrix lane/8 -> (+8 channels if bit 0, +8 tokens if bit 1)
    const int vtok = (lane & 7) + 8 * (lane >> 4), vch = 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        uint32_t a[4];
        ldmatrix_x4_trans(a, buf + (16 * kt + vtok) * kPitch + (16 * mt + vch) * 2);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a, pp[nt][kt][0], pp[nt][kt][1]);
      }
      const uint32_t ac[4] = {0u, ones_a, 0u, ones_a};  // denominator row only
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(zc[nt], ac, pp[nt][kt][0], pp[nt][kt][1]);
    }
    __syncwarp();
  }

  // After the last quantized group of a segment, before any fp16 chunk: bring
  // the code products in o to unit scale (output rows gid / gid + 8 hold the
  // codes of row half 0 / 1).
  __device__ __forceinline__ void quant_done() {
#pragma unroll
    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][nt][i] *= unit(0, i >> 1);
  }

  // Write this warp's partial (m, l, unnormalised o) for its G heads: o is the sum
  // of its hi and lo columns; row j of zc (hi column) holds sum p~ z of value
  // group j, row 12 the sum of p~.
  __device__ __forceinline__ void write_partial(float* dst) const {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = 4 * nt + tig;
      const float lt = __shfl_sync(0xffffffffu, zc[nt][2], 16 + tig);  // row 12: lanes gid 4
      float zs[D / 32];
#pragma unroll
      for (int j = 0; j < D / 32; ++j) zs[j] = __shfl_sync(0xffffffffu, zc[nt][0], 4 * j + tig);
      if (g < G) {
        float* d = dst + g * C::PSTRIDE;
        if (gid == 0) { d[0] = m[nt]; d[1] = lt; }
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          d[4 + 16 * mt + gid] = (o[mt][nt][0] + o[mt][nt][1]) + zs[mt / 2];
          d[4 + 16 * mt + gid + 8] = (o[mt][nt][2] + o[mt][nt][3]) + zs[mt / 2];
        }
      }
    }
  }
};

// Log-sum-exp merge of a segment's nparts consecutive partials into the
// normalised output [G][D], by the whole CTA.  The partials come from other CTAs
// (visible after the acquire of the split-K counter) and are read from L2 with
// ordinary loads: one warp per head finds the maximum over the non-empty partials
// and their weights (s_w [nparts][G] in shared memory, then the G sums of weights
// times denominators), then every thread sums its output elements.
template <int D, int BITS, int G, bool ROPE, int CPS, int PF>
__device__ void final_merge_pf(const float* parts, int nparts, float* out, float* s_w) {
  using C = DecodeCfg<D, BITS, G, ROPE, CPS>;
  constexpr int PS = C::PSTRIDE;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  float* s_l = s_w + (size_t)nparts * G;
  // the o values of this thread's first output element from the first PF
  // partials, loaded before the (m, l) round below so both round trips overlap
  const int e0 = tid < G * D ? tid : 0;
  float v0[PF];
#pragma unroll
  for (int k = 0; k < PF; ++k)
    v0[k] = k < nparts ? __ldcg(parts + (size_t)(k * G + e0 / D) * PS + 4 + e0 % D) : 0.f;
  for (int g = warp; g < G; g += nthreads / 32) {
    // (m, l) of partials lane, lane + 32, ...: the first 32 held in registers
    float m0 = -INFINITY, l0 = 0.f;
    if (lane < nparts) {
      m0 = __ldcg(parts + (size_t)(lane * G + g) * PS);
      l0 = __ldcg(parts + (size_t)(lane * G + g) * PS + 1);
    }
    float mx = l0 > 0.f ? m0 : -INFINITY;
    for (int i = lane + 32; i < nparts; i += 32)
      if (__ldcg(parts + (size_t)(i * G + g) * PS + 1) > 0.f) mx = fmaxf(mx, __ldcg(parts + (size_t)(i * G + g) * PS));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float lsum = 0.f;
    if (lane < nparts) {
      const float w = l0 > 0.f ? fast_exp2(m0 - mx) : 0.f;
      s_w[lane * G + g] = w;
      lsum = w * l0;
    }
    for (int i = lane + 32; i < nparts; i += 32) {
      const float li = __ldcg(parts + (size_t)(i * G + g) * PS + 1);
      const float w = li > 0.f ? fast_exp2(__ldcg(parts + (size_t)(i * G + g) * PS) - mx) : 0.f;
      s_w[i * G + g] = w;
      lsum = fmaf(w, li, lsum);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (lane == 0) s_l[g] = lsum;
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += nthreads) {
    const int g = e / D, d = e % D;
    // up to 32 independent loads in flight per round (one L2 round trip each);
    // the first round of the first element was loaded up front
    float osum = 0.f;
    int i0 = 0;
    if (e == tid) {
#pragma unroll
      for (int k = 0; k < PF; ++k)
        if (k < nparts) osum = fmaf(s_w[k * G + g], v0[k], osum);
      i0 = PF;
    }
    for (int i = i0; i < nparts; i += 32) {
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k)
        v[k] = i + k < nparts ? __ldcg(parts + (size_t)((i + k) * G + g) * PS + 4 + d) : 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (i + k < nparts) osum = fmaf(s_w[(i + k) * G + g], v[k], osum);
    }
    const float l = s_l[g];
    out[e] = l > 0.f ? osum / l : 0.f;
  }
}

// Prefetch width: 32 partials with one CTA per SM (few segments, many partials
// each), 8 with several (many short segments of a few partials each; measured:
// 32 there cost 0.4 us on the Llama-2-13B step, and saves 0.5 us on the 128k one).
template <int D, int BITS, int G, bool ROPE, int CPS>
__device__ void final_merge(const float* parts, int nparts, float* out, float* s_w) {
  final_merge_pf<D, BITS, G, ROPE, CPS, CPS == 1 ? 32 : 8>(parts, nparts, out, s_w);
}

template <int D, int BITS, int G, bool ROPE = false, int CPS = 1>
__global__ void __launch_bounds__(DecodeCfg<D, BITS, G, ROPE, CPS>::WARPS * 32,
                                  DecodeCfg<D, BITS, G, ROPE, CPS>::MIN_CTAS)
decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<D, BITS, G, ROPE, CPS>;
  constexpr int NTILES = C::NT;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last;
  uint8_t* ring = smem;
  __half* ps_all = reinterpret_cast<__half*>(smem + C::RING);
  uint32_t* zrow = reinterpret_cast<uint32_t*>(smem + C::RING + C::PS);
  int* s_pref = reinterpret_cast<int*>(smem + C::RING + C::PS + C::ZERO);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* q_smem = reinterpret_cast<uint32_t*>(smem + C::RING + C::PS + C::ZERO + C::PREFIX);
  float2* intra_s = reinterpret_cast<float2*>(smem + C::RING + C::PS + C::ZERO + C::PREFIX + C::QS);
  float* qf_s = reinterpret_cast<float*>(smem + C::RING + C::PS + C::ZERO + C::PREFIX + C::QS + C::INTRA);
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + C::RING + C::PS + C::ZERO + C::PREFIX + C::QS +
                                                   C::INTRA + C::QF);
  uint64_t* bars = bars_all + warp * C::NSTAGE;
  uint64_t* merge_bar = bars_all + C::WARPS * C::NSTAGE;
  __half* ps = ps_all + warp * G * C::PSROW;
  uint8_t* wring = ring + warp * C::NSTAGE * C::STAGE;

  // the lengths first (warp 0: their loads are the kernel's first memory round
  // trip), the shared-memory set-up of the other warps meanwhile
  build_prefix(p, s_pref);
  for (int i = threadIdx.x; i < C::ZERO / 4; i += blockDim.x) zrow[i] = 0u;
  if (lane == 0) {
    for (int st = 0; st < C::NSTAGE; ++st) mbar_init(bars + st, 1);
    if (warp == 0) mbar_init(merge_bar, 1);
    mbar_fence_init();
  }
  uint32_t parity = 0;  // bit st: parity of the next phase of stage st's mbarrier
  uint32_t merge_parity = 0;
  bool failed = false;  // a bounded wait gave up: stop using staged data
  __syncthreads();
  if constexpr (ROPE) {
    // the cos/sin of the offsets 0..63 of every pair, once per CTA (the merge
    // barrier's first phase; waited for before any thread may leave)
    if (threadIdx.x == 0) {
      fence_proxy_async();
      mbar_arrive_expect_tx(merge_bar, C::INTRA);
      tma_load_1d(intra_s, C::RTC ? static_cast<const void*>(p.rope_trig) : static_cast<const void*>(p.rope),
                  C::INTRA, merge_bar);
    }
    if (!mbar_wait(merge_bar, 0, kMaxPolls)) failed = true;
    merge_parity = 1;
    if constexpr (C::RTC) {
      const uint32_t* tag = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(intra_s) +
                                                              kRopeTrigTagOffset);
      if (!failed && threadIdx.x == 0 && (tag[0] != kRopeTrigTag || tag[1] != (uint32_t)BITS) &&
          p.error_flags != nullptr)
        atomicOr(p.error_flags, KVQ_DEVERR_BAD_TABLE);
    }
  }
  const int64_t total = (int64_t)p.hkv * s_pref[p.batch];
  const int64_t nstream = total < p.n_stream ? total : p.n_stream;
  const int64_t c = blockIdx.x;
  if (c >= nstream) return;
  const int R = p.tail_cap;
  const int64_t r0 = c * total / nstream, r1 = (c + 1) * total / nstream;
  for (int64_t x = r0; x < r1;) {
    // segment containing x: the largest b with hkv * pref[b] <= x
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)p.hkv * s_pref[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int items = s_pref[b + 1] - s_pref[b];
    const int64_t seg_first = (int64_t)p.hkv * s_pref[b];
    const int h = (int)((x - seg_first) / items);
    const int i0 = (int)((x - seg_first) % items);
    const int64_t xe = min(r1, x + (items - i0));
    const int n = (int)(xe - x);
    const int seg = b * p.hkv + h;
    const SeqLen L = read_lengths(p, b, false);
    const int ng = L.nq / kGroup;
    // this warp's contiguous share of items [i0, i0 + n)
    const int per = (n + C::WARPS - 1) / C::WARPS;
    const int ia = i0 + min(n, warp * per), ie = i0 + min(n, (warp + 1) * per);
    Decoder<D, BITS, G, ROPE, CPS> dec;
    {
      const int ga = ia, cnt = failed ? 0 : max(0, min(ie, ng) - ia);
      const size_t g0 = (size_t)seg * p.max_groups + ga;
      const int nst = (cnt + C::GPI - 1) / C::GPI;  // stages of up to GPI consecutive groups
      // one lane issues four bulk copies per stage (codes, values, key and value
      // metadata of its groups, each contiguous in the cache), completing on the
      // stage's mbarrier
      auto issue = [&](int si, int slotn) {
        if (lane == 0) {
          const int gi = si * C::GPI, n_in = min(C::GPI, cnt - gi);
          const size_t g = g0 + gi;
          uint8_t* dst = wring + slotn * C::STAGE;
          fence_proxy_async();
          mbar_arrive_expect_tx(bars + slotn, n_in * C::STAGE1);
          const uint64_t pol = l2_evict_first_policy();
          tma_load_1d_hint(dst, p.k_codes + g * C::TB, n_in * C::TB, bars + slotn, pol);
          tma_load_1d_hint(dst + C::OFF_VC, p.v_codes + g * C::TB, n_in * C::TB, bars + slotn, pol);
          tma_load_1d_hint(dst + C::OFF_KM, reinterpret_cast<const uint8_t*>(p.k_meta) + g * C::KMETA,
                           n_in * C::KMETA, bars + slotn, pol);
          tma_load_1d_hint(dst + C::OFF_VM, reinterpret_cast<const uint8_t*>(p.v_meta) + g * C::VMETA,
                           n_in * C::VMETA, bars + slotn, pol);
          if constexpr (ROPE)  // cos/sin of the group's position block: 32 (group + sinks / 32)
            tma_load_1d(dst + C::OFF_BASE, p.rope + (size_t)(64 + ga + gi + (L.ns >> 5)) * (D / 2), C::BASE,
                        bars + slotn);
        }
      };
      // start the first copies, then stage this segment's q (lane order) while they fly
      int issued = 0, waited = 0;
#pragma unroll
      for (int st = 0; st < C::NSTAGE - 1; ++st)
        if (st < nst) { issue(st, st); ++issued; }
      {
        const __half* qh = p.q + ((size_t)b * p.hkv + h) * G * D;
        for (int e = threadIdx.x; e < NTILES * 4 * (D / 2); e += blockDim.x) {
          const int g = e / (D / 2), pr = e % (D / 2);
          const int kt = 2 * (pr / 16) + (pr % 4) / 2, tg = (pr % 16) / 4, r = pr % 2;
          const int c = 16 * kt + 2 * tg + 8 * r;
          q_smem[e] = g < G ? *reinterpret_cast<const uint32_t*>(qh + g * D + c) : 0u;
        }
        if constexpr (ROPE)
          for (int e = threadIdx.x; e < NTILES * 4 * D; e += blockDim.x)
            qf_s[e] = e / D < G ? __half2float(qh[e]) : 0.f;
      }
      __syncthreads();
      dec.init(q_smem);
      dec.qf = qf_s;
      // RTC: the fp16 pieces in shared memory; the fp32 rows (tail and sink
      // chunks) read from the table in global memory
      dec.intra = C::RTC ? p.rope : intra_s;
      dec.trig = reinterpret_cast<const uint8_t*>(intra_s);
      for (int i = 0; i < nst; ++i) {
        if (i + C::NSTAGE - 1 < nst) { issue(i + C::NSTAGE - 1, (i + C::NSTAGE - 1) % C::NSTAGE); ++issued; }
        const int slotn = i % C::NSTAGE;
        const bool ok = mbar_wait(bars + slotn, (parity >> slotn) & 1u, kMaxPolls);
        parity ^= 1u << slotn;
        ++waited;
        if (!ok) { failed = true; break; }
        const uint8_t* st = wring + slotn * C::STAGE;
        if constexpr (C::GPI == 2) {
          if (cnt - i * C::GPI >= 2) {
            dec.quant_pair(st, zrow, p.scale_log2);
            continue;
          }
        }
        dec.quant_group(st, st + C::OFF_VC, st + C::OFF_KM, st + C::OFF_VM, st + C::OFF_BASE, ps, zrow,
                        p.scale_log2, L.ns & 31);
      }
      // after a timeout, wait (bounded) for this warp's copies still in flight
      for (; waited < issued; ++waited) {
        const int slotn = waited % C::NSTAGE;
        mbar_wait(bars + slotn, (parity >> slotn) & 1u, kMaxPolls);
        parity ^= 1u << slotn;
      }
      __syncwarp();
      dec.quant_done();
    }
    if (failed && lane == 0 && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_TIMEOUT);
    // fp16 chunks (tail, then sinks) whose first weighted item falls in this warp's range
    const int ctail = (L.nt + kGroup - 1) / kGroup;
    for (int t = max(ia, ng); t < (failed ? 0 : ie); ++t) {
      const int u = t - ng;
      if (u % kTailWeight != 0) continue;
      const int ci = u / kTailWeight;
      if (ci < ctail) {
        const int first = ci * kGroup;
        const int t0 = L.ns + L.nq + first;  // position of the chunk's first token
        dec.tail_chunk(wring, p.k_tail + (size_t)seg * R * D, p.v_tail + (size_t)seg * R * D, first,
                       min(kGroup, L.nt - first), L.th, R, ps, p.scale_log2,
                       ROPE ? p.rope + (size_t)(64 + (t0 >> 5)) * (D / 2) : nullptr, t0 & 31);
      } else {
        const int first = (ci - ctail) * kGroup;
        if (first >= L.ns) continue;
        const int S = p.sink_cap;
        dec.tail_chunk(wring, p.k_sink + (size_t)seg * S * D, p.v_sink + (size_t)seg * S * D, first,
                       min(kGroup, L.ns - first), 0, S, ps, p.scale_log2,
                       ROPE ? p.rope + (size_t)(64 + (first >> 5)) * (D / 2) : nullptr, first & 31);
      }
    }
    // warp partial into the warp's (now idle) ring slice, then the CTA merge
    dec.write_partial(reinterpret_cast<float*>(wring));
    __syncthreads();
    // the CTA merge: each warp takes chunks of 32 output elements (one head each);
    // lanes w < WARPS load warp w's (m, l) of that head, the weights are formed in
    // registers and broadcast by shuffles (no shared-memory round trip, one barrier)
    float* slot = p.part + (size_t)(c + seg) * G * C::PSTRIDE;
    static_assert(C::WARPS <= 32 && D % 32 == 0, "a warp's lanes hold the warps' weights");
    for (int ch = warp; ch < G * D / 32; ch += C::WARPS) {
      const int g = ch * 32 / D, d = ch * 32 % D + lane;
      float mw = -INFINITY, lw = 0.f;
      if (lane < C::WARPS) {
        const float* src = reinterpret_cast<const float*>(ring + lane * C::NSTAGE * C::STAGE) + g * C::PSTRIDE;
        mw = src[0];
        lw = src[1];
      }
      float mx = mw;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float wt = (lane < C::WARPS && mx != -INFINITY) ? fast_exp2(mw - mx) : 0.f;
      float lsum = wt * lw;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      float osum = 0.f;
#pragma unroll
      for (int w = 0; w < C::WARPS; ++w)
        osum = fmaf(__shfl_sync(0xffffffffu, wt, w),
                    reinterpret_cast<const float*>(ring + w * C::NSTAGE * C::STAGE)[g * C::PSTRIDE + 4 + d], osum);
      slot[g * C::PSTRIDE + 4 + d] = osum;
      if (d == 0) {
        slot[g * C::PSTRIDE] = mx;
        slot[g * C::PSTRIDE + 1] = lsum;
      }
    }
    __syncthreads();
    const int64_t c0 = cta_of(seg_first + (int64_t)h * items, total, nstream);
    const int nparts = (int)(cta_of(seg_first + (int64_t)(h + 1) * items - 1, total, nstream) - c0 + 1);
    // one acquire-release add publishes the CTA's partial (the barrier above
    // orders every thread's writes before it) and, for the last arrival, makes
    // the other CTAs' partials visible (the barrier below passes that on)
    if (threadIdx.x == 0) s_last = atomic_add_acq_rel(&p.counters[seg], 1) == nparts - 1;
    __syncthreads();
    if (s_last) {
      // the stage ring (idle here) holds the merge weights
      final_merge<D, BITS, G, ROPE, CPS>(p.part + (size_t)(c0 + seg) * G * C::PSTRIDE, nparts,
                                    p.out + ((size_t)b * p.hkv * G + (size_t)h * G) * D,
                                    reinterpret_cast<float*>(ring));
      if (threadIdx.x == 0) p.counters[seg] = 0;
    }
    __syncthreads();
    x = xe;
  }
}

struct DecodeLayout {
  size_t counters, part, total;
};

inline DecodeLayout decode_layout(const kvq_cache* c, int G, int n_stream) {
  DecodeLayout L;
  const size_t seg = (size_t)c->batch * c->n_kv_heads;
  const size_t pstride = (size_t)(c->head_dim + 4) * 4 * G;
  L.counters = 0;
  L.part = ((seg * 4 + 255) / 256) * 256;
  // CTA c writes its partial of segment s to slot c + s (distinct for every pair)
  L.total = L.part + ((size_t)n_stream + seg) * pstride;
  return L;
}

template <int D, int BITS, int G, bool ROPE = false, int CPS = 1>
struct DecodeLaunch {
  // resident CTAs on the whole current GPU (one wave), computed once per device
  static int slots(int* err) {
    using C = DecodeCfg<D, BITS, G, ROPE, CPS>;
    return device_slots(reinterpret_cast<const void*>(decode_kernel<D, BITS, G, ROPE, CPS>), C::WARPS * 32,
                        C::SMEM, err);
  }
  static kvq_status run(DecodeParams p, cudaStream_t s) {
    using C = DecodeCfg<D, BITS, G, ROPE, CPS>;
    int err = 0;
    const int n = slots(&err);
    if (err) return KVQ_ERR_CUDA;
    // a segment's partials come from at most n CTAs (+ one spare slot)
    if (n + 1 > C::MAX_PARTS) return KVQ_ERR_UNSUPPORTED;
    p.n_stream = n;
    decode_kernel<D, BITS, G, ROPE, CPS><<<n, C::WARPS * 32, C::SMEM, s>>>(p);
    return launch_status();
  }
};

template <int D, int BITS, bool ROPE = false, int CPS = 1>
kvq_status decode_dispatch_g(int G, const DecodeParams& p, cudaStream_t s) {
  switch (G) {
    case 1: return DecodeLaunch<D, BITS, 1, ROPE, CPS>::run(p, s);
    case 2: return DecodeLaunch<D, BITS, 2, ROPE, CPS>::run(p, s);
    case 4: return DecodeLaunch<D, BITS, 4, ROPE, CPS>::run(p, s);
    case 8: return DecodeLaunch<D, BITS, 8, ROPE, CPS>::run(p, s);
    default: return KVQ_ERR_UNSUPPORTED;
  }
}

// The uniform decode (no RoPE) of one CTA shape: resident CTAs and launch, by
// head_dim, bits and G.  Instantiated for CPS 1 in kvq_decode.cu and for CPS 2
// and 4 in their own translation units.
template <int CPS>
int decode_slots_shape(const kvq_cache* c, int G, int* err) {
#define KVQ_SLOTS(D_, B_, G_) \
  if (c->head_dim == D_ && c->bits == B_ && G == G_) return DecodeLaunch<D_, B_, G_, false, CPS>::slots(err);
#define KVQ_SLOTS_G(D_, B_) KVQ_SLOTS(D_, B_, 1) KVQ_SLOTS(D_, B_, 2) KVQ_SLOTS(D_, B_, 4) KVQ_SLOTS(D_, B_, 8)
  KVQ_SLOTS_G(128, 2) KVQ_SLOTS_G(128, 4) KVQ_SLOTS_G(64, 2) KVQ_SLOTS_G(64, 4)
  if constexpr (CPS == 1) { KVQ_SLOTS_G(128, 8) KVQ_SLOTS_G(64, 8) }
#undef KVQ_SLOTS_G
#undef KVQ_SLOTS
  *err = 2;
  return 0;
}

template <int CPS>
kvq_status decode_run_shape(const kvq_cache* c, int G, const DecodeParams& p, cudaStream_t st) {
  if (c->head_dim == 128) {
    if (c->bits == 2) return decode_dispatch_g<128, 2, false, CPS>(G, p, st);
    if (c->bits == 4) return decode_dispatch_g<128, 4, false, CPS>(G, p, st);
    if constexpr (CPS == 1) return decode_dispatch_g<128, 8, false, 1>(G, p, st);
    return KVQ_ERR_UNSUPPORTED;
  }
  if (c->bits == 2) return decode_dispatch_g<64, 2, false, CPS>(G, p, st);
  if (c->bits == 4) return decode_dispatch_g<64, 4, false, CPS>(G, p, st);
  if constexpr (CPS == 1) return decode_dispatch_g<64, 8, false, 1>(G, p, st);
  return KVQ_ERR_UNSUPPORTED;
}

// Defined in the CPS 2 and CPS 4 translation units.
int decode_slots_cps2(const kvq_cache* c, int G, int* err);
int decode_slots_cps4(const kvq_cache* c, int G, int* err);
kvq_status decode_run_cps2(const kvq_cache* c, int G, const DecodeParams& p, cudaStream_t st);
kvq_status decode_run_cps4(const kvq_cache* c, int G, const DecodeParams& p, cudaStream_t st);

// CTAs per SM for a uniform decode without RoPE: the smallest of 1, 2, 4 whose
// grid (one wave) has at least one CTA per (sequence, KV head) segment, so that a
// CTA rarely spans two segments; 1 at 8 bits.
inline int decode_shape(const kvq_cache* c, int* err) {
  if (c->bits == 8) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess) {
    *err = 1;
    return 1;
  }
  const int64_t seg = (int64_t)c->batch * c->n_kv_heads;
  if (seg <= sms) return 1;
  if (seg <= 2 * (int64_t)sms) return 2;
  return 4;
}

// The kernel parameters of one decode call: the cache's buffers and lengths, q
// and out, and the workspace (counters and partials at the offsets of L, from
// the base ws).  Shared by every decode entry point.
inline DecodeParams decode_params(const kvq_cache* c, const void* q, float* out, float sm_scale, uint8_t* ws,
                                  const DecodeLayout& L, const float* rope_table = nullptr) {
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
  p.rope = reinterpret_cast<const float2*>(rope_table);
  p.out = out;
  p.counters = reinterpret_cast<int32_t*>(ws + L.counters);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.batch = c->batch;
  p.hkv = c->n_kv_heads;
  p.max_groups = c->max_groups;
  p.tail_cap = c->tail_cap;
  p.sink_cap = c->sink_cap;
  return p;
}

inline kvq_status validate_q_heads(const kvq_cache* c, int32_t n_q_heads, int* G) {
  if (c->batch > KVQ_MAX_BATCH) return KVQ_ERR_UNSUPPORTED;
  if (n_q_heads < c->n_kv_heads || n_q_heads % c->n_kv_heads) return KVQ_ERR_INVALID;
  const int g = n_q_heads / c->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return KVQ_ERR_UNSUPPORTED;
  *G = g;
  return KVQ_OK;
}

}  // namespace kvq
