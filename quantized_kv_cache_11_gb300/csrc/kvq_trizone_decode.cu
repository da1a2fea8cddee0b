// Fused-dequant split-K decode attention over the mixed-width ("TriZone")
// cache: "RDKV" summary (gist.science 2605.08317), section "2.2 TriZone": one
// kernel reads zone A (keys per channel at 2/4/8 bits, values per token at
// 2/4/8 bits) with the dequantization inside the tensor-core products, zone B
// (fp16 values) and zone C (fp16 fresh tokens), so the cache is never expanded.
//
// How:
// * Work partition: every block of every (sequence, KV head) weighs a few units
//   by kind (the decode of a block costs about the same for every value width:
//   the arithmetic, not the record's bytes, sets its time; a key k-tile more
//   costs a few units more).  When each segment's share of the resident CTAs
//   rounds to a whole number within 15%, every segment gets that many CTAs of
//   its own, each an equal range of its units;
//   otherwise (stream-K) the units of all segments are laid end to end and cut
//   into equal ranges, one per resident CTA.  A CTA owns the blocks whose first
//   unit falls in its range.
// * Inside a CTA the warps deal the CTA's blocks of the current segment round
//   robin (blocks are stored by kind, so every warp gets a similar mix of sizes,
//   and the assignment -- hence the summation order -- is the same on every
//   call), and each warp streams its blocks with one bulk copy (TMA) per record
//   into a private byte ring, several copies in flight, completion on mbarriers
//   with bounded waits.
// * Per block (one warp, the GQA group's G heads): Q.K^T runs over the three key
//   classes with the codes turned into fp16 operands by one mask per register
//   (the code pair left in the low mantissa bits, exponent 0: the exact
//   subnormals c * 2^(p-24), p the bit position, which depends only on the
//   fragment row and the class), B = q * scale split into fp16 hi + lo, one
//   accumulator per class brought to unit scale per row, and the zero points
//   through one constant product per k-tile; masked tokens of a partial block
//   get -inf.  Online softmax (exp2 domain).  P.V by value class: codes with
//   B = p~ * scale split into hi and lo fp16 columns (exact), the accumulator
//   rescaled by a power of two when the value width changes, and one constant
//   product (zero points, the ones row = the denominator); or fp16 tiles whose
//   words are the A fragments as stored.
// * Splits merge by log-sum-exp; the last CTA of a segment writes the output
//   and resets the segment's counter.  No spin-wait on other CTAs.
#include <cmath>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_trizone_internal.h"

namespace kvq {
namespace tz {

constexpr uint32_t kMaxPolls = 1u << 22;
// Bit position of the codes that unpack8<BITS> puts in register 4 mt + i (row
// half rh = i & 1; the same for both k-halves): the register holds the fp16
// subnormals c * 2^(p - 24), so unit = 2^(24 - p) brings a product to unit scale.
// p >= 2: a tensor-core dot product over subnormal operands at position p keeps
// about 17 + p significant bits (measured on GB300), so p = 0 is avoided.
__host__ __device__ constexpr int code_pos(int bits, int mt, int rh) {
  return 2 + (bits == 2 ? 4 * mt + 2 * rh : (bits == 4 ? 4 * rh : 0));
}
__host__ __device__ constexpr float code_unit(int bits, int mt, int rh) {
  return (float)(1 << (24 - code_pos(bits, mt, rh)));
}
// Unit of the P.V accumulator rows of half rh while a warp decodes blocks of value
// kind k (widths 2, 4, 8: the codes' unit, with the 2-bit tokens 16..31 brought
// to the unit of tokens 0..15; 16 and fresh: 1).
__device__ __forceinline__ float value_unit(int k, int rh) {
  return k == 0 ? code_unit(2, 0, rh) : (k == 1 ? code_unit(4, 0, rh) : (k == 2 ? code_unit(8, 0, rh) : 1.f));
}

template <int G>
struct Cfg {
  static constexpr int NT = (2 * G + 7) / 8;  // 8-column n-tiles: column 2g = hi, 2g+1 = lo of head g
  static constexpr int WARPS = 6;
  static constexpr int MIN_CTAS = NT == 1 ? 2 : 1;
  static constexpr int RING = 16384;  // bytes of a warp's byte ring (>= the largest record)
  static constexpr int NBAR = 4;      // copies in flight per warp, at most
  static constexpr int PSTRIDE = kDim + 4;
  static constexpr int QPH = 88;  // words per head of the slot-ordered q (10 k-tiles x 8, + 8 pad)
  static constexpr int RINGS = WARPS * RING;
  static constexpr int PS = WARPS * G * 96;  // the final merge's weights, [MERGE_BATCH][G] floats
  static constexpr int ZERO = 4 * kDim;
  static constexpr int PREFIX = ((KVQ_TZ_MAX_SEGMENTS + 1) * 8 + 15) / 16 * 16;
  static constexpr int QP = 4 * NT * QPH * 4;
  static constexpr int QN = NT * 4 * (kDim / 2) * 4;
  static constexpr int HDR = 128 + 2 * kSlots;
  static constexpr int FIFO = WARPS * NBAR * 8;
  static constexpr int MBAR = (WARPS * NBAR + 1) * 8;
  static constexpr int SMEM = RINGS + PS + ZERO + PREFIX + QP + QN + HDR + FIFO + MBAR;
  static constexpr int MERGE_BATCH =
      RINGS / (G * PSTRIDE * 4) < PS / (4 * G) ? RINGS / (G * PSTRIDE * 4) : PS / (4 * G);
  static_assert(RING >= KVQ_TZ_FRESH_BLOCK_BYTES && RING >= KVQ_TZ_MAX_BLOCK_BYTES, "a record fits a ring");
  static_assert(RING >= G * PSTRIDE * 4, "a warp partial fits its ring");
  static_assert(MERGE_BATCH >= 1, "a merge batch holds one partial");
  static_assert(RINGS % 16 == 0 && PS % 16 == 0 && PREFIX % 16 == 0 && QP % 16 == 0 && QN % 16 == 0 &&
                    HDR % 16 == 0 && FIFO % 16 == 0,
                "aligned shared regions");
};

struct Params {
  const uint8_t* index;
  const uint8_t* blocks;
  int64_t region;
  int32_t* error_flags;
  const __half* q;
  float* out;
  int32_t* counters;
  float* part;
  float scale_log2;
  int32_t n_seg;
  int32_t n_stream;
};

__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t total, int64_t n) {
  return ((x + 1) * n - 1) / total;
}

// Segment-aligned partition: segment s gets c_s = max(1, round(n * w_s / W))
// CTAs of its own (rounded down instead when the rounded shares do not fit in
// n), each an equal share of its units, when no segment's share is more than
// this many percent of the mean W / n (and the c_s fit in n).  A CTA
// whose range spans two segments (the stream-K cut) pays a second set-up and a
// second merge, and, as the last arrival of the next segment, its final merge:
// measured on 32 segments of 65,536 tokens over 304 CTAs that was ~8 us at the
// end of a ~58 us launch, against 5.6% more work per CTA when aligned.
constexpr int kAlignSlack = 115;
constexpr int kHdrVecBytes = 112;  // header bytes the plan stages (words 0..27)

// Work units of one block of each kind (value width 2, 4, 8, 16, fresh) with
// 9 key k-tiles: measured decode time per block, in steps of about a hundredth;
// each key k-tile more or fewer adds or takes kKtUnits to a quantized block
// (measured: segments of 10 k-tiles took 7% longer than those of 9).
__constant__ int c_kind_units[kKinds] = {100, 100, 110, 120, 120};
constexpr int kKtUnits = 7;

__device__ __forceinline__ int kind_units(int k, const int32_t* hd) {
  int kt = hd[H_KT] + hd[H_KT + 1] + hd[H_KT + 2];
  kt = kt < 0 ? 0 : (kt > kKtMax ? kKtMax : kt);  // clamped: the index is checked later
  return k < 4 ? c_kind_units[k] + kKtUnits * (kt - 9) : c_kind_units[k];
}

// Work units of a segment as the partition sees it: its blocks by kind (block
// counts clamped so that a corrupt index cannot overflow the prefix), at least 1.
__device__ __forceinline__ int64_t seg_weight(const Params& p, int s) {
  const int32_t* hd = reinterpret_cast<const int32_t*>(p.index + (size_t)s * KVQ_TZ_INDEX_BYTES);
  int64_t w = 0;
#pragma unroll
  for (int k = 0; k < kKinds; ++k) {
    const int n = hd[H_NBLK + k];
    w += (int64_t)(n < 0 ? 0 : (n > (1 << 24) ? (1 << 24) : n)) * kind_units(k, hd);
  }
  return w > 0 ? w : 1;
}

// The index record is what the build wrote: every field consistent.
__device__ __forceinline__ bool header_ok(const int* hd, int64_t region) {
  const int kt2 = hd[H_KT], kt4 = hd[H_KT + 1], kt8 = hd[H_KT + 2];
  bool ok = kt2 >= 0 && kt4 >= 0 && kt8 >= 0 && kt2 + kt4 + kt8 <= kKtMax;
  int64_t off = 0;
  for (int k = 0; k < kKinds && ok; ++k) {
    const int n = hd[H_NBLK + k];
    const int cnt = k < 4 ? hd[H_NTOK + k] : hd[H_NFRESH];
    const int rec = k < 4 ? record_bytes(kt2, kt4, kt8, k) : KVQ_TZ_FRESH_BLOCK_BYTES;
    ok = cnt >= 0 && n <= (1 << 24) && n == (cnt + kGroup - 1) / kGroup && hd[H_REC + k] == rec &&
         hd[H_OFF + k] == off;
    off += (int64_t)n * rec;
  }
  return ok && hd[H_USED] == off && off <= region;
}

template <int G>
struct Decoder {
  using C = Cfg<G>;
  static constexpr int NT = C::NT;
  static constexpr uint32_t kOnes = 0x3C003C00u;
  static constexpr uint32_t kSixteenth = 0x2C002C00u;  // half2(1/16, 1/16)
  float m[NT];
  float o[8][NT][4];    // P.V: rows = channels (8 tiles of 16), columns (head, hi|lo); lo stays 0
  float zc[NT][4];      // value-constant products: rows j = sum p~ z of group j, 12 = sum p~
  const uint32_t* qp;   // slot-ordered q pairs of this lane's column
  const uint32_t* qn;   // natural-order q pairs of this lane's column
  uint32_t nhl, ones_a;
  int lane, gid, tig;
  int ukind;            // o holds value_unit(ukind, rh) times the true sums

  __device__ __forceinline__ void init(const uint32_t* qp_smem, const uint32_t* qn_smem) {
    lane = threadIdx.x & 31;
    gid = lane >> 2;
    tig = lane & 3;
    nhl = (gid & 1) ? 0xBC00BC00u : 0u;
    ones_a = gid == 4 ? kOnes : 0u;
    ukind = 3;
    qp = qp_smem + (gid >> 1) * C::QPH + 2 * tig;
    qn = qn_smem + (gid >> 1) * (kDim / 2) + 4 * tig;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) zc[nt][i] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
    }
  }

  // hi column: fp16(x*y); lo column: x*y - fp16(x*y) (exact)
  __device__ __forceinline__ uint32_t split_mul(uint32_t a, uint32_t b) const {
    const __half2 x = u32_as_h2(a), y = u32_as_h2(b);
    const __half2 hi = __hmul2_rn(x, y);
    return h2_as_u32(__hfma2(x, y, __hmul2_rn(hi, u32_as_h2(nhl))));
  }

  // Operands of the 8 pairs in w[0 .. BITS/2): one mask per register, on the
  // word shifted left by 2 or right by 6, leaves a code pair in mantissa bits
  // [p, p + BITS) of the two halves, exponent 0.
  template <int BITS>
  static __device__ __forceinline__ void unpack8(const uint32_t* w, uint32_t (&a)[8]) {
    if (BITS == 2) {
      const uint32_t w0 = w[0], x = w0 << 2, y = w0 >> 6;
      a[0] = x & 0x000C000Cu;  a[1] = x & 0x00300030u;  a[2] = y & 0x000C000Cu;  a[3] = y & 0x00300030u;
      a[4] = x & 0x00C000C0u;  a[5] = x & 0x03000300u;  a[6] = y & 0x00C000C0u;  a[7] = y & 0x03000300u;
    } else if (BITS == 4) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = w[h], x = w0 << 2, y = w0 >> 6;
        a[4 * h + 0] = x & 0x003C003Cu;
        a[4 * h + 1] = x & 0x03C003C0u;
        a[4 * h + 2] = y & 0x003C003Cu;
        a[4 * h + 3] = y & 0x03C003C0u;
      }
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t x = w[h];
        a[2 * h + 0] = (x << 2) & 0x03FC03FCu;
        a[2 * h + 1] = (x >> 6) & 0x03FC03FCu;
      }
    }
  }

  // One k-tile of key class BITS: codes of sub-tile word row j, global k-tile kt.
  template <int BITS>
  __device__ __forceinline__ void key_tile(const uint32_t* sub, int j, int kt, const uint32_t* kmt,
                                           float (&s0)[NT][4], float (&s1)[NT][4], float (&cc)[NT][4]) const {
    uint32_t w[BITS / 2];
#pragma unroll
    for (int i = 0; i < BITS / 2; ++i) w[i] = sub[(j * (BITS / 2) + i) * 32 + lane];
    uint32_t a[8];
    unpack8<BITS>(w, a);
    // (zero r0, scale r0, zero r1, scale r1) of the lane's slots in k-tile kt: the
    // constant product's A quad as it stands (rows gid: the zero points, every row
    // alike; rows gid + 8: scales, whose products are not read)
    const uint4 mv = *reinterpret_cast<const uint4*>(kmt + 16 * kt);
    const uint32_t a0[4] = {a[0], a[1], a[2], a[3]};
    const uint32_t a1[4] = {a[4], a[5], a[6], a[7]};
    const uint32_t ac[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint2 qv = *reinterpret_cast<const uint2*>(qp + nt * 4 * C::QPH + 8 * kt);
      const uint32_t b0 = split_mul(qv.x, mv.y), b1 = split_mul(qv.y, mv.w);
      mma_16816(s0[nt], a0, b0, b1);
      mma_16816(s1[nt], a1, b0, b1);
      mma_16816(cc[nt], ac, qv.x, qv.y);
    }
  }

  // All k-tiles of one key class into the accumulators (rows of m-tiles 0 and 1).
  template <int BITS>
  __device__ __forceinline__ void key_class(const uint32_t* sub, int ktc, int& kt, const uint32_t* kmt,
                                            float (&sacc)[2][NT][4], float (&cc)[NT][4]) const {
#pragma unroll 4
    for (int j = 0; j < ktc; ++j, ++kt) key_tile<BITS>(sub, j, kt, kmt, sacc[0], sacc[1], cc);
  }

  // Rescale o from the unit of value kind ukind to that of kind k (powers of two).
  __device__ __forceinline__ void set_units(int k) {
    if (k == ukind) return;  // warp-uniform
    const float r0 = value_unit(ukind, 0) / value_unit(k, 0), r1 = value_unit(ukind, 1) / value_unit(k, 1);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[mt][nt][0] *= r0; o[mt][nt][1] *= r0; o[mt][nt][2] *= r1; o[mt][nt][3] *= r1;
      }
    ukind = k;
  }

  // Online softmax over one 32-token block, straight into the P.V B fragments of
  // column 8nt + gid (head 4nt + gid/2): the p~ pairs of a lane's C-layout rows are
  // transposed in registers (movmatrix).  with_lo: the lo columns (odd gid) hold p~
  // too (code blocks split p~ * scale into hi and lo columns); otherwise zero (fp16
  // values multiply p~ itself, exact in one column).
  __device__ __forceinline__ void softmax_pp(const float (&lg)[NT][2][2], uint32_t (&pp)[NT][2][2], bool with_lo) {
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
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float mnew = fmaxf(m[nt], mloc[nt]);
        const float alpha = (mnew == m[nt]) ? 1.f : fast_exp2(m[nt] - mnew);
        m[nt] = mnew;
#pragma unroll
        for (int i = 0; i < 4; ++i) zc[nt][i] *= alpha;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[mt][nt][i] *= alpha;
      }
    }
    const bool zero_lo = !with_lo && (gid & 1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float pf = fast_exp2(lg[nt][mt][r] - m[nt]);
          if (G % 4 != 0 && 4 * nt + tig >= G) pf = 0.f;
          const uint32_t t = movmatrix_trans(h2_as_u32(__floats2half2_rn(pf, pf)));
          pp[nt][mt][r] = zero_lo ? 0u : t;
        }
  }

  // P.V over a value tile of codes (class VC: width 2 << VC) and its metadata.
  template <int VC>
  __device__ __forceinline__ void pv_codes(const uint8_t* vt, const uint32_t (&pp)[NT][2][2], const uint32_t* zrow) {
    constexpr int BITS = 2 << VC;
    constexpr int TB = Tile<kDim, BITS>::kBytes;
    constexpr int NWL = Tile<kDim, BITS>::kWordsPerLane;
    const uint4* s4 = reinterpret_cast<const uint4*>(vt);
    uint32_t vw[NWL];
#pragma unroll
    for (int ch = 0; ch < NWL / 4; ++ch) {
      const uint4 v = s4[ch * 32 + lane];
      vw[4 * ch] = v.x; vw[4 * ch + 1] = v.y; vw[4 * ch + 2] = v.z; vw[4 * ch + 3] = v.w;
    }
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(vt + TB);
    const uint32_t* vsl = vm + 4 * tig;             // scale pairs
    const uint32_t* vzl = vm + kDim / 2 + 4 * tig;  // zero-point pairs
    // 2-bit codes of tokens 16..31 sit 4 bits above those of tokens 0..15 of the
    // same row: their p~ is divided by 16 (exactly) for a common unit
    uint32_t pv[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        pv[nt][0][r] = pp[nt][0][r];
        pv[nt][1][r] = BITS == 2 ? h2_as_u32(__hmul2(u32_as_h2(pp[nt][1][r]), u32_as_h2(kSixteenth))) : pp[nt][1][r];
      }
#pragma unroll
    for (int j = 0; j < kDim / 32; ++j) {
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
          unpack8<BITS>(vw + mt * (BITS / 2), a8);  // pairs of (mt, kt = 0) then (mt, kt = 1)
          const uint32_t a[4] = {a8[4 * kt], a8[4 * kt + 1], a8[4 * kt + 2], a8[4 * kt + 3]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a, b[nt][0], b[nt][1]);
        }
      }
    }
    // constant rows (tokens 16kt + 2tig (+8r)): 0..3 zero points of group j, 12 ones
    const uint4 v0 = *reinterpret_cast<const uint4*>(gid < 4 ? vzl + 16 * gid : zrow);
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      const uint32_t ac[4] = {kt ? v0.z : v0.x, ones_a, kt ? v0.w : v0.y, ones_a};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(zc[nt], ac, pp[nt][kt][0], pp[nt][kt][1]);
    }
  }

  // P.V over a 16-bit value tile (the words are the A fragments).
  __device__ __forceinline__ void pv_fp16(const uint8_t* vt, const uint32_t (&pp)[NT][2][2]) {
    const uint4* s4 = reinterpret_cast<const uint4*>(vt);
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint4 v = s4[(2 * mt + kt) * 32 + lane];
        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a, pp[nt][kt][0], pp[nt][kt][1]);
      }
      const uint32_t ac[4] = {0u, ones_a, 0u, ones_a};  // the denominator row only
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(zc[nt], ac, pp[nt][kt][0], pp[nt][kt][1]);
    }
  }

  // A block of zone A/B: keys quantized in three classes, values by kind.
  __device__ __forceinline__ void quant_block(const uint8_t* rec, int kind, int nvalid, const int* hd,
                                              const uint32_t* zrow, float scale_log2) {
    const int kt2 = hd[H_KT], kt4 = hd[H_KT + 1], kt8 = hd[H_KT + 2], KT = kt2 + kt4 + kt8;
    const uint32_t* st = reinterpret_cast<const uint32_t*>(rec);
    const uint32_t* kmt = st + key_code_bytes(kt2, kt4, kt8) / 4 + 4 * tig;
    set_units(kind);
    // one accumulator set, reused by the three key classes: each class is folded
    // into the logits at its own unit before the next one starts
    float sacc[2][NT][4];  // [mt]
    float cc[NT][4];
    float lg[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) cc[nt][i] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) lg[nt][mt][r] = 0.f;
    auto fold = [&](int c) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r)
            lg[nt][mt][r] = fmaf(sacc[mt][nt][2 * r] + sacc[mt][nt][2 * r + 1], code_unit(2 << c, mt, r),
                                 lg[nt][mt][r]);
    };
    auto zero = [&]() {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) { sacc[0][nt][i] = 0.f; sacc[1][nt][i] = 0.f; }
    };
    int kt = 0;
    zero();
    key_class<2>(st, kt2, kt, kmt, sacc, cc);
    fold(0);
    zero();
    key_class<4>(st + 32 * kt2, kt4, kt, kmt, sacc, cc);
    fold(1);
    zero();
    key_class<8>(st + 32 * kt2 + 64 * kt4, kt8, kt, kmt, sacc, cc);
    fold(2);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float zq = cc[nt][0];  // q.z (every constant row holds the zero points)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          lg[nt][mt][r] = (16 * mt + gid + 8 * r) < nvalid ? (lg[nt][mt][r] + zq) * scale_log2 : -INFINITY;
    }
    uint32_t pp[NT][2][2];
    softmax_pp(lg, pp, kind < 3);
    const uint8_t* vt = rec + key_bytes(kt2, kt4, kt8);
    if (kind == 0) pv_codes<0>(vt, pp, zrow);
    else if (kind == 1) pv_codes<1>(vt, pp, zrow);
    else if (kind == 2) pv_codes<2>(vt, pp, zrow);
    else pv_fp16(vt, pp);
    __syncwarp();
  }

  // A fresh block (zone C): fp16 key tile in natural channel order, fp16 values.
  __device__ __forceinline__ void fresh_block(const uint8_t* rec, int nvalid, float scale_log2) {
    set_units(3);  // fp16 values: unit 1, as zone B
    const uint4* s4 = reinterpret_cast<const uint4*>(rec);
    float sacc[2][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) { sacc[0][nt][i] = 0.f; sacc[1][nt][i] = 0.f; }
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      uint32_t a[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint4 v = s4[(2 * kt + mt) * 32 + lane];
        a[mt][0] = v.x; a[mt][1] = v.y; a[mt][2] = v.z; a[mt][3] = v.w;
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 qv = *reinterpret_cast<const uint4*>(qn + nt * 4 * (kDim / 2) + 8 * (kt & ~1));
        const uint32_t q0 = (kt & 1) ? qv.z : qv.x, q1 = (kt & 1) ? qv.w : qv.y;
        mma_16816(sacc[0][nt], a[0], q0, q1);
        mma_16816(sacc[1][nt], a[1], q0, q1);
      }
    }
    float lg[NT][2][2];  // B = q in both columns of a head: use one
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          lg[nt][mt][r] = (16 * mt + gid + 8 * r) < nvalid ? sacc[mt][nt][2 * r] * scale_log2 : -INFINITY;
    uint32_t pp[NT][2][2];
    softmax_pp(lg, pp, false);
    pv_fp16(rec + kFp16TileBytes, pp);
    __syncwarp();
  }

  // This warp's partial (m, l, unnormalised o) for its G heads; o is brought to
  // unit scale first.
  __device__ __forceinline__ void write_partial(float* dst) {
    set_units(3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = 4 * nt + tig;
      const float lt = __shfl_sync(0xffffffffu, zc[nt][2], 16 + tig);  // row 12
      float zs[kDim / 32];
#pragma unroll
      for (int j = 0; j < kDim / 32; ++j) zs[j] = __shfl_sync(0xffffffffu, zc[nt][0], 4 * j + tig);  // row j
      if (g < G) {
        float* d = dst + g * C::PSTRIDE;
        if (gid == 0) { d[0] = m[nt]; d[1] = lt; }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          d[4 + 16 * mt + gid] = (o[mt][nt][0] + o[mt][nt][1]) + zs[mt / 2];
          d[4 + 16 * mt + gid + 8] = (o[mt][nt][2] + o[mt][nt][3]) + zs[mt / 2];
        }
      }
    }
  }
};

// Log-sum-exp merge of a segment's nparts consecutive partials into the
// normalised output [G][D]; the partials are bulk-copied MERGE_BATCH at a time
// into the (idle) rings.  Returns false if a bounded wait gave up.
template <int G>
__device__ bool final_merge(const float* parts, int nparts, float* out, uint8_t* ring, float* s_w, uint64_t* bar,
                            uint32_t& parity, float* s_M, float* s_L, float* s_scale) {
  using C = Cfg<G>;
  constexpr int PS = C::PSTRIDE;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int PER = (G * kDim + C::WARPS * 32 - 1) / (C::WARPS * 32);
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  if (tid < G) { s_M[tid] = -INFINITY; s_L[tid] = 0.f; }
  bool ok = true;
  const float* stage = reinterpret_cast<const float*>(ring);
  for (int first = 0; first < nparts; first += C::MERGE_BATCH) {
    const int nb = min(C::MERGE_BATCH, nparts - first);
    __syncthreads();
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)(nb * G * PS * 4);
      fence_proxy_async_global();  // the partials were written by other CTAs' ordinary stores
      fence_proxy_async();
      mbar_arrive_expect_tx(bar, bytes);
      tma_load_1d(ring, parts + (size_t)first * G * PS, bytes, bar);
    }
    ok = mbar_wait(bar, parity, kMaxPolls) && ok;
    parity ^= 1u;
    for (int g = warp; g < G; g += nthreads / 32) {
      float mx = -INFINITY;
      for (int i = lane; i < nb; i += 32) mx = fmaxf(mx, stage[(i * G + g) * PS]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mold = s_M[g], mnew = fmaxf(mold, mx);
      const float sc = (mnew == -INFINITY || mold == mnew) ? 1.f : fast_exp2(mold - mnew);
      float lsum = 0.f;
      for (int i = lane; i < nb; i += 32) {
        const float mi = stage[(i * G + g) * PS];
        const float w = mnew == -INFINITY ? 0.f : fast_exp2(mi - mnew);
        s_w[i * G + g] = w;
        lsum += w * stage[(i * G + g) * PS + 1];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      __syncwarp();
      if (lane == 0) { s_M[g] = mnew; s_L[g] = s_L[g] * sc + lsum; s_scale[g] = sc; }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = tid + k * nthreads;
      if (e < G * kDim) {
        const int g = e / kDim, d = e % kDim;
        float o = acc[k] * s_scale[g];
        for (int i = 0; i < nb; ++i) o += s_w[i * G + g] * stage[(i * G + g) * PS + 4 + d];
        acc[k] = o;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int e = tid + k * nthreads;
    if (e < G * kDim) {
      const float l = s_L[e / kDim];
      out[e] = l > 0.f ? acc[k] / l : 0.f;
    }
  }
  return ok;
}

template <int G>
__global__ void __launch_bounds__(Cfg<G>::WARPS * 32, Cfg<G>::MIN_CTAS) decode_kernel(const Params p) {
  using C = Cfg<G>;
  constexpr int NT = C::NT;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last, s_total;
  __shared__ int s_aligned, s_aseg, s_aj, s_acs, s_ac0;  // the segment-aligned plan
  __shared__ int s_hpre;  // the first 112 header bytes of the CTA's segment already staged
  __shared__ int s_lo[kKinds], s_cum[kKinds + 1];
  __shared__ float s_M[G], s_L[G], s_scale[G];
  uint8_t* rings = smem;
  float* s_wts = reinterpret_cast<float*>(smem + C::RINGS);  // the final merge's weights
  uint32_t* zrow = reinterpret_cast<uint32_t*>(smem + C::RINGS + C::PS);
  int64_t* s_pref = reinterpret_cast<int64_t*>(smem + C::RINGS + C::PS + C::ZERO);
  uint32_t* qp_smem = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(s_pref) + C::PREFIX);
  uint32_t* qn_smem = qp_smem + C::QP / 4;
  int* s_hdr = reinterpret_cast<int*>(qn_smem + C::QN / 4);
  const int16_t* s_slots = reinterpret_cast<const int16_t*>(s_hdr + 32);
  int* fifo_all = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(s_hdr) + C::HDR);
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(fifo_all) + C::FIFO);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = bars_all + warp * C::NBAR;
  uint64_t* merge_bar = bars_all + C::WARPS * C::NBAR;
  int* fifo = fifo_all + warp * C::NBAR * 2;  // per entry: ring offset, kind << 24 | block
  uint8_t* ring = rings + warp * C::RING;

  for (int i = tid; i < C::ZERO / 4; i += blockDim.x) zrow[i] = 0u;
  if (lane == 0) {
    for (int i = 0; i < C::NBAR; ++i) mbar_init(bars + i, 1);
    if (warp == 0) mbar_init(merge_bar, 1);
    mbar_fence_init();
  }
  // weighted prefix over the segments
  if (warp == 0) {
    // at most 32 segments: lane s also loads the first 112 bytes of segment s's
    // index record (every field the partition and the copies use), kept for the
    // segment-aligned plan, which then needs no second round trip for them
    constexpr int kHdrVec = kHdrVecBytes / 16;
    const bool few = p.n_seg <= 32;
    uint4 hw[kHdrVec];
    if (few && lane < p.n_seg) {
      const uint4* src = reinterpret_cast<const uint4*>(p.index + (size_t)lane * KVQ_TZ_INDEX_BYTES);
#pragma unroll
      for (int i = 0; i < kHdrVec; ++i) hw[i] = src[i];
    }
    int64_t run = 0;
    for (int s0 = 0; s0 < p.n_seg; s0 += 32) {
      const int s = s0 + lane;
      int64_t v = s < p.n_seg ? seg_weight(p, s) : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int64_t a = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += a;
      }
      if (s < p.n_seg) s_pref[s + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_pref[0] = 0;
    __syncwarp();
    // the segment-aligned plan (kAlignSlack): c_s per segment, rounded to the
    // nearest when those fit the slots (the heavier segments take the spare CTAs),
    // else rounded down; an inclusive scan of them gives this CTA's segment, its
    // index among the c_s and the segment's first CTA
    const int64_t ns = run < p.n_stream ? run : p.n_stream;
    bool mine = false;  // this lane's segment is the CTA's
    int64_t nround = 0;
    for (int s0 = 0; s0 < p.n_seg; s0 += 32) {
      const int s = s0 + lane;
      int64_t cs = 0;
      if (s < p.n_seg) {
        cs = (2 * ns * (s_pref[s + 1] - s_pref[s]) + run) / (2 * run);
        if (cs < 1) cs = 1;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
      nround += cs;
    }
    const bool nearest = nround <= ns;
    bool fits = true;
    int64_t cbase = 0;
    if (lane == 0) s_aseg = -1;
    __syncwarp();
    for (int s0 = 0; s0 < p.n_seg; s0 += 32) {
      const int s = s0 + lane;
      int64_t cs = 0;
      if (s < p.n_seg) {
        const int64_t ws = s_pref[s + 1] - s_pref[s];
        cs = nearest ? (2 * ns * ws + run) / (2 * run) : ns * ws / run;
        if (cs < 1) cs = 1;
        if (ws * ns * 100 > (int64_t)kAlignSlack * run * cs) fits = false;
      }
      int64_t v = cs;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int64_t a = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += a;
      }
      const int64_t first = cbase + v - cs;
      if (cs > 0 && (int64_t)blockIdx.x >= first && (int64_t)blockIdx.x < first + cs) {
        mine = true;
        s_aseg = s;
        s_aj = (int)(blockIdx.x - first);
        s_acs = (int)cs;
        s_ac0 = (int)first;
      }
      cbase += __shfl_sync(0xffffffffu, v, 31);
    }
    fits = __all_sync(0xffffffffu, fits) && cbase <= ns;
    if (lane == 0) s_aligned = fits ? 1 : 0;
    if (fits && few && mine) {
#pragma unroll
      for (int i = 0; i < kHdrVec; ++i) reinterpret_cast<uint4*>(s_hdr)[i] = hw[i];
    }
    if (lane == 0) s_hpre = fits && few ? 1 : 0;
  }
  __syncthreads();
  const int64_t total = s_pref[p.n_seg];
  const int64_t nstream = total < p.n_stream ? total : p.n_stream;
  const int64_t c = blockIdx.x;
  const bool aligned = s_aligned != 0;
  int64_t r0, r1;
  int s = 0;
  if (aligned) {
    if (s_aseg < 0) return;  // past the last segment's CTAs
    s = s_aseg;
    const int64_t S0 = s_pref[s], W0 = s_pref[s + 1] - S0;
    r0 = S0 + W0 * s_aj / s_acs;
    r1 = S0 + W0 * (s_aj + 1) / s_acs;
  } else {
    if (c >= nstream) return;
    r0 = c * total / nstream;
    r1 = (c + 1) * total / nstream;
    int lo = 0, hi = p.n_seg - 1;  // the last segment whose first unit is <= r0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pref[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    s = lo;
  }
  uint32_t issued = 0, done = 0;  // this warp's copies, over the whole kernel (mbarrier phases)
  uint32_t merge_parity = 0;
  bool failed = false;
  for (; s < p.n_seg && s_pref[s] < r1; ++s) {
    const int64_t S = s_pref[s], W = s_pref[s + 1] - S;
    const int64_t a = r0 > S ? r0 - S : 0, e = (r1 - S) < W ? r1 - S : W;
    // ---- segment header (with the slots) and q in natural channel order, in the
    // pair order of the fragments; with the header's first 112 bytes staged by
    // the plan, warp 0 cuts this CTA's blocks while the other warps load the rest
    const bool pre = s_hpre != 0;
    {
      const uint8_t* idx = p.index + (size_t)s * KVQ_TZ_INDEX_BYTES;
      const int lt = pre ? tid - 32 : tid, nth = pre ? (int)blockDim.x - 32 : (int)blockDim.x;
      if (lt >= 0) {
        const int w0 = pre ? kHdrVecBytes / 4 : 0;
        for (int w = w0 + lt; w < (128 + 2 * kSlots) / 4; w += nth)
          reinterpret_cast<uint32_t*>(s_hdr)[w] = reinterpret_cast<const uint32_t*>(idx)[w];
        const __half* qh = p.q + (size_t)s * G * kDim;
        for (int i = lt; i < NT * 4 * (kDim / 2); i += nth) {
          const int g = i / (kDim / 2), pr = i % (kDim / 2);
          const int kt = 2 * (pr / 16) + (pr % 4) / 2, tg = (pr % 16) / 4, r = pr % 2;
          const int ch = 16 * kt + 2 * tg + 8 * r;
          qn_smem[i] = g < G ? *reinterpret_cast<const uint32_t*>(qh + g * kDim + ch) : 0u;
        }
      }
    }
    if (!pre) __syncthreads();
    if (tid == 0) {
      const bool ok = header_ok(s_hdr, p.region);
      if (!ok && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_BAD_LENGTHS);
      int64_t cw = 0;
      int cum = 0;
      for (int k = 0; k < kKinds; ++k) {
        const int n = ok ? s_hdr[H_NBLK + k] : 0;
        const int wg = kind_units(k, s_hdr);
        const int64_t lo64 = a <= cw ? 0 : (a - cw + wg - 1) / wg;
        const int lo = (int)(lo64 < n ? lo64 : n);
        const int64_t hi64 = e <= cw ? 0 : (e - cw + wg - 1) / wg;
        const int hi = (int)(hi64 < n ? hi64 : n);
        s_lo[k] = lo;
        s_cum[k] = cum;
        cum += hi > lo ? hi - lo : 0;
        cw += (int64_t)n * wg;
      }
      s_cum[kKinds] = cum;
      s_total = cum;
    }
    __syncthreads();
    Decoder<G> dec;
    // ---- this warp's blocks (round robin), streamed through the ring
    {
      const int ntot = failed ? 0 : s_total;
      int wr = 0, pend = -1, taken = 0;
      bool exhausted = ntot == 0;
      auto fill = [&]() {
        while (!exhausted && issued - done < (uint32_t)C::NBAR) {
          if (pend < 0) {
            pend = warp + C::WARPS * taken++;
            if (pend >= ntot) { exhausted = true; break; }
          }
          int k = 0;
          while (k < kKinds - 1 && pend >= s_cum[k + 1]) ++k;
          const int blk = s_lo[k] + (pend - s_cum[k]);
          const int size = s_hdr[H_REC + k];
          int off;
          if (issued == done) {
            off = 0;
          } else {
            const int h0 = fifo[(done % C::NBAR) * 2];
            if (wr > h0) {
              if (C::RING - wr >= size) off = wr;
              else if (h0 >= size) off = 0;
              else break;
            } else {
              if (h0 - wr >= size) off = wr;
              else break;
            }
          }
          const int slot = issued % C::NBAR;
          __syncwarp();
          if (lane == 0) {
            fifo[slot * 2] = off;
            fifo[slot * 2 + 1] = (k << 24) | blk;
            fence_proxy_async();
            mbar_arrive_expect_tx(bars + slot, (uint32_t)size);
            tma_load_1d_hint(ring + off, p.blocks + (size_t)s * p.region + s_hdr[H_OFF + k] + (size_t)blk * size,
                             (uint32_t)size, bars + slot, l2_evict_first_policy());
          }
          __syncwarp();
          wr = off + size;
          ++issued;
          pend = -1;
        }
      };
      fill();
      // q in slot order, gathered from the staged natural copy (channel c sits in
      // pair 16 (kt / 2) + 4 tg + 2 (kt % 2) + r, c = 16 kt + 2 tg + 8 r + (c & 1)),
      // while the first copies fly
      {
        const __half* qn_h = reinterpret_cast<const __half*>(qn_smem);
        auto q_at = [&](int g, int ch) -> uint32_t {
          const int kt = ch >> 4, w16 = ch & 15, r = w16 >> 3, tg = (w16 & 7) >> 1;
          const int pr = 16 * (kt >> 1) + 4 * tg + 2 * (kt & 1) + r;
          return (uint32_t)__half_as_ushort(qn_h[2 * (g * (kDim / 2) + pr) + (ch & 1)]);
        };
        for (int i = tid; i < 4 * NT * C::QPH; i += blockDim.x) {
          const int g = i / C::QPH, w = i % C::QPH;
          uint32_t val = 0u;
          if (g < G && w < 8 * kKtMax) {
            const int kt = w >> 3, tg = (w >> 1) & 3, r = w & 1;
            const int sl = 16 * kt + 2 * tg + 8 * r;
            const int c0 = s_slots[sl], c1 = s_slots[sl + 1];
            const uint32_t lo16 = c0 >= 0 && c0 < kDim ? q_at(g, c0) : 0u;
            const uint32_t hi16 = c1 >= 0 && c1 < kDim ? q_at(g, c1) : 0u;
            val = lo16 | (hi16 << 16);
          }
          qp_smem[i] = val;
        }
      }
      __syncthreads();
      dec.init(qp_smem, qn_smem);
      while (done < issued) {
        const int slot = done % C::NBAR;
        if (!mbar_wait(bars + slot, (done / C::NBAR) & 1u, kMaxPolls)) { failed = true; break; }
        const int off = fifo[slot * 2], kb = fifo[slot * 2 + 1];
        const int k = kb >> 24, blk = kb & 0xFFFFFF;
        const int cnt = k < 4 ? s_hdr[H_NTOK + k] : s_hdr[H_NFRESH];
        const int nvalid = min(kGroup, cnt - kGroup * blk);
        if (k < 4) dec.quant_block(ring + off, k, nvalid, s_hdr, zrow, p.scale_log2);
        else dec.fresh_block(ring + off, nvalid, p.scale_log2);
        ++done;
        fill();
      }
      // after a timeout: wait (bounded) for this warp's copies still in flight
      for (; done < issued; ++done) mbar_wait(bars + done % C::NBAR, (done / C::NBAR) & 1u, kMaxPolls);
      __syncwarp();
    }
    if (failed && lane == 0 && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_TIMEOUT);
    // ---- warp partial into the warp's (idle) ring, CTA merge, last-CTA merge
    dec.write_partial(reinterpret_cast<float*>(ring));
    __syncthreads();
    float* slotp = p.part + (size_t)(c + s) * G * C::PSTRIDE;
    for (int e2 = tid; e2 < G * kDim; e2 += blockDim.x) {
      const int g = e2 / kDim, d = e2 % kDim;
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::WARPS; ++w)
        mx = fmaxf(mx, reinterpret_cast<const float*>(rings + w * C::RING)[g * C::PSTRIDE]);
      float lsum = 0.f, osum = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) {
          const float* src = reinterpret_cast<const float*>(rings + w * C::RING) + g * C::PSTRIDE;
          const float wt = fast_exp2(src[0] - mx);
          lsum += wt * src[1];
          osum += wt * src[4 + d];
        }
      }
      slotp[g * C::PSTRIDE + 4 + d] = osum;
      if (d == 0) { slotp[g * C::PSTRIDE] = mx; slotp[g * C::PSTRIDE + 1] = lsum; }
    }
    __syncthreads();
    const int64_t c0 = aligned ? s_ac0 : cta_of(S, total, nstream);
    const int nparts = aligned ? s_acs : (int)(cta_of(S + W - 1, total, nstream) - c0 + 1);
    // one acquire-release add publishes the CTA's partial (the barrier above
    // orders every thread's writes before it) and, for the last arrival, makes
    // the other CTAs' partials visible (the barrier below passes that on)
    if (tid == 0) s_last = atomic_add_acq_rel(&p.counters[s], 1) == nparts - 1;
    __syncthreads();
    if (s_last) {
      const bool ok = final_merge<G>(p.part + (size_t)(c0 + s) * G * C::PSTRIDE, nparts, p.out + (size_t)s * G * kDim,
                                     rings, s_wts, merge_bar, merge_parity, s_M, s_L,
                                     s_scale);
      if (!ok && tid == 0 && p.error_flags != nullptr) atomicOr(p.error_flags, KVQ_DEVERR_TIMEOUT);
      if (tid == 0) p.counters[s] = 0;
    }
    __syncthreads();
  }
}

struct Layout {
  size_t counters, part, total;
};

inline Layout layout(const kvq_trizone* t, int G, int n_stream) {
  Layout L;
  const size_t seg = (size_t)t->batch * t->n_kv_heads;
  L.counters = 0;
  L.part = ((seg * 4 + 255) / 256) * 256;
  L.total = L.part + ((size_t)n_stream + seg) * (size_t)(kDim + 4) * 4 * G;
  return L;
}

template <int G>
struct Launch {
  // resident CTAs on the whole current GPU, computed once per device
  static int slots(int* err) {
    using C = Cfg<G>;
    return device_slots(reinterpret_cast<const void*>(decode_kernel<G>), C::WARPS * 32, C::SMEM, err);
  }
  static kvq_status run(Params p, cudaStream_t st) {
    int err = 0;
    const int n = slots(&err);
    if (err) return KVQ_ERR_CUDA;
    p.n_stream = n;
    decode_kernel<G><<<n, Cfg<G>::WARPS * 32, Cfg<G>::SMEM, st>>>(p);
    return launch_status();
  }
};

inline int decode_slots(int G, int* err) {
  switch (G) {
    case 1: return Launch<1>::slots(err);
    case 2: return Launch<2>::slots(err);
    case 4: return Launch<4>::slots(err);
    case 8: return Launch<8>::slots(err);
    default: *err = 2; return 0;
  }
}

inline kvq_status validate_q_heads(const kvq_trizone* t, int32_t n_q_heads, int* G) {
  if ((int64_t)t->batch * t->n_kv_heads > KVQ_TZ_MAX_SEGMENTS) return KVQ_ERR_UNSUPPORTED;
  if (n_q_heads < t->n_kv_heads || n_q_heads % t->n_kv_heads) return KVQ_ERR_INVALID;
  const int g = n_q_heads / t->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return KVQ_ERR_UNSUPPORTED;
  *G = g;
  return KVQ_OK;
}

}  // namespace tz
}  // namespace kvq

extern "C" kvq_status kvq_trizone_decode_workspace_bytes(const kvq_trizone* t, int32_t n_q_heads, size_t* bytes) {
  using namespace kvq::tz;
  kvq_status s = validate_geometry(t);
  if (s != KVQ_OK) return s;
  if (bytes == nullptr) return KVQ_ERR_INVALID;
  int G = 0;
  s = validate_q_heads(t, n_q_heads, &G);
  if (s != KVQ_OK) return s;
  int err = 0;
  const int n = decode_slots(G, &err);
  if (err) return KVQ_ERR_CUDA;
  *bytes = layout(t, G, n).total;
  return KVQ_OK;
}

extern "C" kvq_status kvq_trizone_decode_attn(const kvq_trizone* t, int32_t n_q_heads, const void* q, float* out,
                                              float sm_scale, void* workspace, size_t workspace_bytes,
                                              void* stream) {
  using namespace kvq;
  using namespace kvq::tz;
  kvq_status s = validate_buffers(t);
  if (s != KVQ_OK) return s;
  int G = 0;
  s = validate_q_heads(t, n_q_heads, &G);
  if (s != KVQ_OK) return s;
  if (q == nullptr || out == nullptr || workspace == nullptr) return KVQ_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(out, 16) || !aligned(workspace, 16)) return KVQ_ERR_INVALID;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID;
  int err = 0;
  const int n = decode_slots(G, &err);
  if (err) return KVQ_ERR_CUDA;
  const Layout L = layout(t, G, n);
  if (workspace_bytes < L.total) return KVQ_ERR_INVALID;
  Params p{};
  p.index = static_cast<const uint8_t*>(t->index);
  p.blocks = static_cast<const uint8_t*>(t->blocks);
  p.region = region_bytes(t);
  p.error_flags = t->error_flags;
  p.q = static_cast<const __half*>(q);
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<int32_t*>(ws + L.counters);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.n_seg = t->batch * t->n_kv_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (G) {
    case 1: return Launch<1>::run(p, st);
    case 2: return Launch<2>::run(p, st);
    case 4: return Launch<4>::run(p, st);
    default: return Launch<8>::run(p, st);
  }
}
