/*
 * kvq_trizone.h -- C ABI of the mixed-width ("TriZone") cache of the GB300
 * (sm_103a) low-bit KV-cache library.  Conventions (device pointers owned by
 * the caller, no allocation, no stream synchronisation, host-side validation
 * before any launch, device-side error bits, no abort) are those of kvq.h.
 *
 * What it stores ("RDKV" summary, gist.science 2605.08317, sections 2.1-2.2 and
 * "2.2 TriZone"): for every (sequence, KV head)
 *   - every old token t has a value width v_width[t] in {0, 2, 4, 8, 16}: 0 drops
 *     the token (its key too), 16 keeps its value row in fp16 (zone B), 2/4/8
 *     quantize the value row per token over 32-channel groups (zone A, values);
 *   - every channel d has a key width k_width[d] in {2, 4, 8}: the keys of all
 *     kept old tokens are quantized per channel over 32-token blocks at that
 *     channel's width (zone A, keys);
 *   - the newest ("fresh") tokens stay fp16 (zone C).
 * Kept old tokens are grouped by value width (widths ascending, original order
 * inside a width) and each width is cut into 32-token blocks, the last one
 * partial; a partial block's key groups take their min/max over its tokens only.
 * Attention is invariant under this reordering (the softmax sums over tokens),
 * so decode never needs the original order; it is kept in `tokens` for callers.
 * The quantizer is the one of kvq.h, bit for bit.
 *
 * Layout (the library's own; all little-endian).  Channels are permuted by key
 * width: the 2-bit channels in ascending order, then the 4-bit, then the 8-bit,
 * each class padded to whole 16-channel k-tiles with pad slots (code 0, scale 0,
 * zero 0); kt2, kt4, kt8 are the k-tiles per class, KT their sum (<= 10).
 * One block (32 tokens of one value width) is one contiguous record:
 *   key codes: per class c in (2, 4, 8) with kt_c > 0, a sub-tile of
 *     32 tokens x 16 kt_c slots: lane L (gid = L/4, tig = L%4) owns the pairs
 *     (kt < kt_c, mt < 2, i < 4) in that order: token 16mt + gid + 8(i%2), class
 *     slots 16kt + 2tig + 8(i/2) and +1; pair P goes to lane word P/(16/c), slot
 *     P%(16/c) at the bit positions of kvq.h; lane word w at byte 4(32w + L) of
 *     the sub-tile (64 kt_c c bytes);
 *   key metadata: 16 KT fp16 pairs; pair 16kt + 4tig + 2r + f (kt over all
 *     classes' k-tiles in order) holds the zero points (f = 0) or the scales
 *     (f = 1) of slots 16kt + 2tig + 8r and +1;
 *   values of width 2/4/8: the value tile of kvq.h at that width (1024, 2048 or
 *     4096 bytes) and its metadata block (512 bytes);
 *   values of width 16: a 16-bit value tile (8192 bytes): the value pair order of
 *     kvq.h with one pair (fp16 of tokens t and t + 1 of one channel) per word;
 *   tokens past a partial block's count are zero in every field.
 * A fresh block (up to 32 fresh tokens, 16384 bytes) is the fp16 keys as a
 * 16-bit key tile (the key pair order of kvq.h in natural channel order, one
 * pair per word) followed by the fp16 values as a 16-bit value tile.
 * A (sequence, KV head) region holds its blocks by kind -- value width 2, 4, 8,
 * 16, then fresh -- every block of one kind the same size.
 * Index record of a (sequence, KV head), KVQ_TZ_INDEX_BYTES bytes: int32
 *   [0:4] kept tokens per value width (2, 4, 8, 16)  [4] fresh tokens
 *   [5:9] blocks per value width  [9] fresh blocks
 *   [10:13] channels per key width (2, 4, 8)  [13:16] k-tiles per key width
 *   [16:21] bytes of one block of each kind  [21:26] byte offset of each kind's
 *   first block in the region  [26] bytes used  [27:32] 0
 * followed by int16 [160] permuted channel slots (channel, or -1 for a pad or
 * past the last k-tile) and 64 zero bytes.
 */
#ifndef KVQ_TRIZONE_H_
#define KVQ_TRIZONE_H_

#include "kvq.h"

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_DEVERR_BAD_WIDTH 8 /* a width outside {0,2,4,8,16} / {2,4,8}: token dropped / channel at 8 bits */

#define KVQ_TZ_INDEX_BYTES 512
#define KVQ_TZ_MAX_BLOCK_BYTES 13312   /* largest block record (value width 16, KT = 10) */
#define KVQ_TZ_FRESH_BLOCK_BYTES 16384 /* fp16 key tile + fp16 value tile */
#define KVQ_TZ_MAX_SEGMENTS 1024       /* batch * n_kv_heads limit of the decode */

/*
 * Mixed-width cache.
 *   batch, n_kv_heads   B, Hkv
 *   head_dim            D, 128 only
 *   max_old             capacity in old tokens per (sequence, KV head)
 *   max_fresh           capacity in fresh tokens per (sequence, KV head)
 * Buffers (device; sizes from kvq_trizone_bytes; 256-byte aligned):
 *   index   uint8 [B][Hkv][KVQ_TZ_INDEX_BYTES]     index records
 *   tokens  int32 [B][Hkv][max_old]  original position of every kept old token,
 *           in stored (block) order
 *   blocks  uint8 [B][Hkv][region]   block records (region = sizes[KVQ_TZ_BUF_BLOCKS] / (B Hkv))
 *   error_flags int32 [1] or NULL: device error bits (KVQ_DEVERR_*)
 */
typedef struct kvq_trizone {
  int32_t batch;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t max_old;
  int32_t max_fresh;
  void* index;
  int32_t* tokens;
  void* blocks;
  int32_t* error_flags;
} kvq_trizone;

enum { KVQ_TZ_BUF_INDEX = 0, KVQ_TZ_BUF_TOKENS, KVQ_TZ_BUF_BLOCKS, KVQ_TZ_NBUF };

/*
 * kvq_trizone_bytes -- byte size of every buffer (host only; pointers unread).
 * The block region of a (sequence, KV head) is sized for the worst case:
 * (ceil(max_old/32) + 3) records of KVQ_TZ_MAX_BLOCK_BYTES plus
 * ceil(max_fresh/32) fresh blocks, rounded up to 256 bytes.
 */
kvq_status kvq_trizone_bytes(const kvq_trizone* tz, size_t sizes[KVQ_TZ_NBUF]);

/*
 * kvq_trizone_build -- compress prompt keys/values into the mixed-width cache
 * ("RDKV" summary, "2.2 TriZone": drop width-0 tokens, group the kept ones by
 * value width, quantize values per token and keys per channel at the assigned
 * widths, keep the fresh tokens in fp16).
 *   k, v      fp16 device [s][t][h][d] with element strides stride_b, stride_t,
 *             stride_h (multiples of 4), d contiguous, 8-byte aligned
 *   v_width   uint8 device [B][Hkv][max_old]; entries t >= t_old[s] are not read
 *   k_width   uint8 device [B][Hkv][128]
 *   t_old     HOST int32 [B]: tokens [0, t_old) of sequence s are old (<= max_old)
 *   n_fresh   HOST int32 [B]: tokens [t_old, t_old + n_fresh) are fresh (<= max_fresh)
 * Rewrites the index, tokens and blocks of every (sequence, KV head).  A width
 * outside the allowed set sets KVQ_DEVERR_BAD_WIDTH (the token is dropped; the
 * channel is taken at 8 bits).  batch <= KVQ_MAX_BATCH.
 */
kvq_status kvq_trizone_build(const kvq_trizone* tz, const void* k, const void* v,
                             int64_t stride_b, int64_t stride_t, int64_t stride_h,
                             const uint8_t* v_width, const uint8_t* k_width,
                             const int32_t* t_old, const int32_t* n_fresh, void* stream);

/*
 * kvq_trizone_decode_workspace_bytes -- scratch size for kvq_trizone_decode_attn
 * (depends on the GPU's SM count: query it on the device that will decode).
 *   n_q_heads  Hq, a multiple of Hkv with Hq/Hkv in {1, 2, 4, 8}
 */
kvq_status kvq_trizone_decode_workspace_bytes(const kvq_trizone* tz, int32_t n_q_heads,
                                              size_t* bytes);

/*
 * kvq_trizone_decode_attn -- single-query decode attention over the mixed-width
 * cache ("RDKV" summary, "2.2 TriZone": one kernel reads zone A with the
 * dequantization fused into the products, zone B and zone C in fp16).
 *   q, out, sm_scale   as kvq_decode_attn (out fp32, 16-byte aligned): softmax
 *             over the kept old tokens and the fresh tokens of each sequence
 *   workspace as kvq_decode_attn: zero-filled before first use, left zero-filled
 * batch * n_kv_heads <= KVQ_TZ_MAX_SEGMENTS.  Preconditions: |q[d]| * scale < 65504
 * for every key group, value scales < 4094 (as kvq_decode_attn).
 */
kvq_status kvq_trizone_decode_attn(const kvq_trizone* tz, int32_t n_q_heads, const void* q,
                                   float* out, float sm_scale, void* workspace,
                                   size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_TRIZONE_H_ */
