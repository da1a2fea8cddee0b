/*
 * kvq.h -- C ABI of the GB300 (sm_103a) low-bit KV-cache library.
 *
 * What it computes
 * ----------------
 * Asymmetric uniform integer quantization of a transformer KV cache, with the
 * grouping axes of "KV-cache quantization axes" (ihal.it, paragraphs 1 and 3-6):
 *   - keys per channel: one group = one channel over 32 consecutive tokens;
 *   - values per token: one group = 32 consecutive channels of one token;
 *   - b in {2, 4, 8} bits per code, fp16 scale and zero point per group;
 *   - the newest tokens that do not yet fill a key group stay in an fp16 tail
 *     (same article, paragraph 8: a full-precision window of recent tokens,
 *     quantized in groups once enough have arrived);
 * and single-query decode attention that reads the packed cache with the
 * dequantization fused into the Q.K^T and P.V products (VQKV summary,
 * gist.science 2603.16435, section 2 "decoding phase": the full-precision
 * sequence is never rebuilt; RDKV summary, gist.science 2605.08317, section
 * "2.2 TriZone": dequantization fused into the attention kernel), so the cache
 * is never expanded in device memory.
 *
 * Quantizer (per group x[0..n-1], fp16 inputs, every fp32 op rounded to
 * nearest even):
 *   scale = fp16( fp32(max - min) / (2^b - 1) ),  zero = fp16(min),  -0 -> +0
 *   code  = clamp( rint_half_even( (fp32(x) - fp32(zero)) / fp32(scale) ), 0, 2^b - 1 )
 *           (code = 0 when scale == 0)
 *   x_hat = zero + scale * code
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Every buffer pointer is a DEVICE pointer owned by the caller, unless a
 *   parameter says "host".  The library allocates nothing and never
 *   synchronises the stream; all work is enqueued on the given stream.
 * - Global state: per device, the library caches each kernel's launch facts
 *   (shared-memory limit, resident CTAs; computed once under a lock), and
 *   kvq_decode_attn_static uses one fixed scratch array compiled into the
 *   library.  Every entry point except kvq_decode_attn_static is re-entrant;
 *   calls of kvq_decode_attn_static that overlap on one GPU share that array
 *   and race (see its comment).
 * - Argument errors are detected on the host BEFORE any launch and return
 *   KVQ_ERR_INVALID / KVQ_ERR_UNSUPPORTED / KVQ_ERR_CAPACITY with no side
 *   effect.  A failed launch returns KVQ_ERR_CUDA.  Errors that only the device
 *   can see (an append past capacity, inconsistent device lengths) set bits in
 *   *error_flags (if non-NULL) and the offending sequence is left unchanged.
 * - No entry point aborts or throws across the ABI.
 * - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID = -1,     /* bad pointer, alignment, size or length */
  KVQ_ERR_UNSUPPORTED = -2, /* geometry outside what is compiled */
  KVQ_ERR_CAPACITY = -3,    /* lengths exceed the cache's capacity */
  KVQ_ERR_CUDA = -4         /* a CUDA launch failed */
} kvq_status;

/* Bits OR-ed into *error_flags by device code. */
#define KVQ_DEVERR_APPEND_CAPACITY 1 /* append needed a flush but the quantized region was full */
#define KVQ_DEVERR_BAD_LENGTHS 2     /* decode saw n_tail > tail_cap or n_quant beyond capacity */
#define KVQ_DEVERR_TIMEOUT 4         /* a bounded wait for staged data gave up; output invalid */
#define KVQ_DEVERR_BAD_TABLE 16      /* pre-RoPE decode: the table was built for another cache; output invalid */

#define KVQ_GROUP 32
#define KVQ_MAX_BATCH 512 /* sequences per prefill call */

/*
 * Uniform cache: one bit width for the whole cache.
 *
 * Geometry
 *   batch        B sequences (rows) of the cache
 *   n_kv_heads   Hkv
 *   head_dim     D in {64, 128}
 *   bits         b in {2, 4, 8}
 *   max_groups   capacity of the quantized region per sequence, in 32-token groups
 *   tail_cap     R, capacity of the fp16 tail in tokens: a multiple of 32, 32..256
 *
 * Buffers (device; sizes from kvq_cache_bytes; code, metadata and tail buffers
 * 16-byte aligned, the int32 arrays 4-byte aligned).  For sequence
 * s, KV head h, group g (tile = 32 tokens, TB = 32 * D * b / 8 bytes):
 *   k_codes   uint8 [B][Hkv][max_groups][TB]   packed key codes of group g
 *   v_codes   uint8 [B][Hkv][max_groups][TB]   packed value codes of tokens 32g..32g+31
 *   k_meta    fp16  [B][Hkv][max_groups][2D]     zero points and scales of key group g,
 *                                                interleaved (below)
 *   v_meta    fp16  [B][Hkv][max_groups][2][D]   scale plane, zero plane of the value
 *                                                groups of tokens 32g..32g+31
 *   k_tail    fp16  [B][Hkv][R][D]   ring of fp16 keys; logical tail token i sits
 *   v_tail    fp16  [B][Hkv][R][D]   at slot (tail_head[s] + i) mod R
 *   n_quant   int32 [B]  tokens in the quantized region (multiple of 32)
 *   n_tail    int32 [B]  tokens in the tail, 0..R
 *   tail_head int32 [B]  ring slot of the oldest tail token (multiple of 32)
 *   error_flags int32 [1] or NULL: device error bits (KVQ_DEVERR_*)
 *   sink_cap  S, attention-sink window (same article, paragraph 9: high-precision
 *             windows for the recent tokens and for the attention sinks): the
 *             first min(S, length) tokens of a sequence stay fp16 and the
 *             quantized groups start after them; 0..256, 0 = no window (the sink
 *             pointers may then be NULL)
 *   k_sink    fp16  [B][Hkv][S][D]   sink token i of a sequence at row i
 *   v_sink    fp16  [B][Hkv][S][D]
 *   n_sink    int32 [B]  sink tokens held, 0..S
 * The n_quant / n_tail / tail_head / n_sink arrays are written by
 * kvq_quantize_prefill and kvq_append_token and read by kvq_decode_attn, all on
 * the device, so a decode loop needs no host synchronisation.
 *
 * Packed tile layout.  A tile's codes are split among 32 "lanes" (gid = lane/4,
 * tig = lane%4), each owning D/2 pairs of codes in this order:
 *   keys:   for kt < D/16, mt < 2, i < 4: token t = 16mt + gid + 8(i%2),
 *           channel c = 16kt + 2tig + 8(i/2); pair = (code[t][c], code[t][c+1])
 *   values: for mt < D/16, kt < 2, i < 4: channel c = 16mt + gid + 8(i%2),
 *           token t = 16kt + 2tig + 8(i/2); pair = (code[t][c], code[t+1][c])
 * Pair P of a lane goes to the lane's 32-bit word P/(16/b), slot k = P%(16/b): the
 * first code at bits [p, p+b), the second at bits [16+p, 16+p+b), where p is
 * 0,2,8,10,4,6,12,14 for k = 0..7 at b = 2 and p = b*k at b = 4, 8.  The lane's
 * word w is stored little-endian at byte ((w/4)*32 + lane)*16 + (w%4)*4 of the
 * tile.  (The pairs are the operand fragments of a 16x8x16 tensor-core product:
 * a warp turns each word into fp16 operands with one mask per pair, the codes
 * read as fp16 subnormals, and the two k-halves of a fragment row always share
 * a bit position.)
 *
 * Metadata is stored as fp16 pairs (32-bit words) in lane order:
 *   key group, D words, word 16kt + 4tig + 2r + f (tig<4, kt<D/16, r<2, f<2):
 *       (x[c], x[c+1]) for channel c = 16kt + 2tig + 8r, x the zero points
 *       (f = 0) or the scales (f = 1), so one 16-byte load gives a lane the
 *       zero points and scales of its channels of k-tile kt
 *   value groups, a scale plane then a zero plane of D/2 words each, word
 *       16j + 4tig + 2kt + r (tig<4, j<D/32, kt<2, r<2):
 *       (x[j][t], x[j][t+1]) for channel group j, token t = 16kt + 2tig + 8r
 */
typedef struct kvq_cache {
  int32_t batch;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t bits;
  int32_t max_groups;
  int32_t tail_cap;
  void* k_codes;
  void* v_codes;
  void* k_meta;
  void* v_meta;
  void* k_tail;
  void* v_tail;
  int32_t* n_quant;
  int32_t* n_tail;
  int32_t* tail_head;
  int32_t* error_flags;
  int32_t sink_cap;
  void* k_sink;
  void* v_sink;
  int32_t* n_sink;
} kvq_cache;

/* Index of each buffer in the sizes[] array of kvq_cache_bytes. */
enum {
  KVQ_BUF_K_CODES = 0,
  KVQ_BUF_V_CODES,
  KVQ_BUF_K_META,
  KVQ_BUF_V_META,
  KVQ_BUF_K_TAIL,
  KVQ_BUF_V_TAIL,
  KVQ_BUF_LENGTHS, /* one int32 [B] array (n_quant, n_tail, tail_head and n_sink each need one) */
  KVQ_BUF_K_SINK,
  KVQ_BUF_V_SINK,
  KVQ_NBUF
};

/*
 * kvq_cache_bytes -- byte size of every buffer of a uniform cache.
 *   cache  host pointer; only the geometry fields are read (pointers may be NULL).
 *   sizes  host array of KVQ_NBUF entries, written on success.
 * Returns KVQ_ERR_INVALID / KVQ_ERR_UNSUPPORTED for a bad geometry.  Host only.
 */
kvq_status kvq_cache_bytes(const kvq_cache* cache, size_t sizes[KVQ_NBUF]);

/*
 * kvq_quantize_prefill -- compress prompt keys/values into the cache
 * (VQKV summary, section 2 "prefilling phase": the prompt's K/V are compressed
 * to integer codes and the originals are no longer needed; ihal.it article,
 * paragraphs 4-6 and 8 for the axes and the fp16 tail).
 *
 *   k, v      fp16 device tensors indexed [s][t][h][d] with element strides
 *             stride_b, stride_t, stride_h and d contiguous (stride 1); the same
 *             strides serve k and v.  Strides must be multiples of 4 elements
 *             and k, v 8-byte aligned.
 *   seq_len   HOST int32 [batch]: tokens of sequence s (0 allowed)
 *   n_tail    HOST int32 [batch]: how many of the newest tokens stay fp16;
 *             seq_len[s] - min(S, seq_len[s]) - n_tail[s] must be a multiple of
 *             32 and >= 0, n_tail[s] <= R.
 * Tokens [0, min(S, seq_len)) are copied to the sink rows, tokens
 * [min(S, seq_len), seq_len - n_tail) are quantized (keys per channel over
 * 32-token spans, values per token over 32-channel spans) and tokens
 * [seq_len - n_tail, seq_len) are copied to tail slots 0.. (tail_head = 0).
 * Sets n_quant / n_tail / tail_head / n_sink on the device.  batch <=
 * KVQ_MAX_BATCH.  KVQ_ERR_CAPACITY if a quantized region exceeds max_groups.
 */
kvq_status kvq_quantize_prefill(const kvq_cache* cache, const void* k, const void* v,
                                int64_t stride_b, int64_t stride_t, int64_t stride_h,
                                const int32_t* seq_len, const int32_t* n_tail,
                                void* stream);

/*
 * kvq_append_token -- add one decoded token per sequence
 * (ihal.it article, paragraph 8: the newest tokens are kept in full precision
 * and quantized in groups once enough of them have arrived).
 *
 *   k_new, v_new  fp16 device [batch][Hkv][D], contiguous, 8-byte aligned.
 * For every sequence: while it holds fewer than S sink tokens, the new token
 * becomes sink row n_sink (n_sink += 1).  Otherwise, if its tail holds R tokens
 * the oldest 32 are first quantized as key group n_quant/32 and value rows
 * n_quant..n_quant+31 (n_quant += 32, tail_head advances by 32); then the new
 * token is written to the tail.  If that flush would pass max_groups, the
 * sequence is left unchanged and KVQ_DEVERR_APPEND_CAPACITY is set in
 * *error_flags.
 */
kvq_status kvq_append_token(const kvq_cache* cache, const void* k_new, const void* v_new,
                            void* stream);

/*
 * kvq_decode_workspace_bytes -- scratch size needed by kvq_decode_attn.
 *   n_q_heads  Hq, a multiple of Hkv with Hq/Hkv in {1, 2, 4, 8}
 *   bytes      host pointer, written on success
 * The size depends on the geometry and on the GPU's SM count (it holds one
 * partial result per resident CTA), so query it on the device that will run
 * the decode (the current device).
 */
kvq_status kvq_decode_workspace_bytes(const kvq_cache* cache, int32_t n_q_heads, size_t* bytes);

/*
 * kvq_decode_attn -- single-query decode attention over the packed cache
 * (ihal.it article, paragraphs 2 and 5: every decode step reads the whole
 * cache, and the output is the softmax-weighted sum of value vectors;
 * VQKV summary, section 2: K/V rebuilt on demand inside the attention kernel).
 *
 *   q         fp16 device [batch][Hq][D], contiguous; query head hq reads KV
 *             head hq / (Hq/Hkv)
 *   out       fp32 device [batch][Hq][D], 16-byte aligned:
 *             softmax(sm_scale * q.K_hat^T) . V_hat over the n_sink fp16
 *             sink tokens, the n_quant quantized tokens and the n_tail fp16 tail
 *             tokens of each sequence (all zeros for an empty sequence)
 *   sm_scale  softmax scale, typically 1/sqrt(D)
 *   workspace device scratch of kvq_decode_workspace_bytes bytes, 16-byte
 *             aligned, ZERO-FILLED before its first use; every call leaves it
 *             zero-filled again, so it can be reused across calls on one stream
 *             (concurrent calls need separate workspaces).
 * Split-K over the sequence: the quantized groups of all sequences and heads
 * are cut into equal ranges on the device from the device-resident lengths
 * (ragged batches stay balanced), and the splits are merged by log-sum-exp.
 * batch <= KVQ_MAX_BATCH.  Preconditions (fp16 operand range of the fused
 * products): |q[d]| * scale_k(g, d) < 65504 for every key group, and
 * scale_v(t, j) < 4094 for every value group (the softmax weights are kept
 * below 16 between rescales).
 */
kvq_status kvq_decode_attn(const kvq_cache* cache, int32_t n_q_heads, const void* q,
                           float* out, float sm_scale, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Size of the fixed scratch array behind kvq_decode_attn_static (4 MiB). */
#define KVQ_STATIC_SCRATCH_BYTES (4u << 20)

/*
 * kvq_decode_attn_static -- kvq_decode_attn without a workspace argument, for
 * callers that cannot allocate device memory: an engine whose allocator has
 * already reserved all device memory for its own pool, a host program that
 * reaches the GPU only through this C ABI and has no device allocator, or a
 * decode loop that must not call cudaMalloc because that call can synchronize
 * the whole device.  There is no counterpart in the pages: this is an interface
 * convenience, and it computes exactly what kvq_decode_attn computes.
 *
 * The split-K partials and merge counters live in one array of
 * KVQ_STATIC_SCRATCH_BYTES compiled into the library; every GPU that loads the
 * library keeps it until the process exits.  Nothing is allocated: the call
 * clears the counters with a memset on `stream` and launches the decode.
 *   Arguments, layout and results are those of kvq_decode_attn.
 *   Returns KVQ_ERR_CAPACITY when the geometry needs more scratch than the
 *   array holds (the need is the kvq_decode_workspace_bytes value), before any
 *   work is enqueued.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls on a device share the one array and it keeps the last
 * call's contents: calls that can overlap on the GPU (different streams, or
 * different host threads without ordering) race and corrupt each other's
 * results, so issue them in order on one stream.
 */
kvq_status kvq_decode_attn_static(const kvq_cache* cache, int32_t n_q_heads, const void* q,
                                  float* out, float sm_scale, void* stream);

/*
 * Pre-RoPE keys ("KV-cache quantization axes", ihal.it, paragraph 7 and the
 * closing paragraph: the keys are quantized before the rotary position
 * embedding and rotated after dequantization, so the outlier channels that make
 * per-channel groups work are not spread over their neighbours).  The cache is
 * filled as usual (kvq_quantize_prefill / kvq_append_token) with keys taken
 * BEFORE the rotation; the decode then rotates every key (sinks, quantized
 * groups, tail) to its position: the adjacent channel pair (2i, 2i+1) of the
 * token at position t (its index in the sequence: sinks first, then the
 * quantized tokens, then the tail, oldest first) turns by t * base^(-2i/D):
 * (k0, k1) -> (k0 cos - k1 sin, k0 sin + k1 cos).  The query is passed already
 * rotated to its own position, as for kvq_decode_attn.  head_dim 128 only.
 *
 * kvq_rope_table_bytes -- bytes of the cos/sin table of a cache geometry: 64 +
 *   ceil((sink_cap + 32 max_groups + tail_cap) / 32) rows of D/2 float2, then
 *   58,240 bytes of fp16 pieces (56 rows of 1,040 bytes).
 * kvq_rope_table -- fills that table on `stream` (float64 angles and sin/cos):
 *   row o < 64 holds float32 (cos, sin)(o theta_i), row 64 + m holds float32
 *   (cos, sin)(32 m theta_i), theta_i = base^(-2i/D); the piece part holds
 *   2^14 cos/sin(o theta_i), o < 64, split into an fp16 hi piece of at most
 *   11 - bits significant bits and the fp16 of the rest, in the order the
 *   decode loads them (it depends on the cache's bits).  base > 1.  Build it
 *   once per (geometry, bits, base); table 16-byte aligned, device memory,
 *   caller-owned.
 * kvq_decode_attn_rope -- kvq_decode_attn over a cache of pre-RoPE keys, with
 *   the table of kvq_rope_table for this cache.  The rotation depends on the
 *   token, so Q.K^T is no longer one matrix product.  At 2 and 4 bits the query
 *   is turned back by the angle of each 32-position block and every code is
 *   multiplied, exactly in fp16, by the hi and lo pieces of the cos and sin of
 *   its offset inside the block before the tensor-core products; at 8 bits the
 *   keys are rotated in float32 on CUDA cores.  P.V and the merge are those of
 *   kvq_decode_attn.  table_bytes: the size of the table buffer, at least
 *   kvq_rope_table_bytes for this cache (else KVQ_ERR_INVALID, before any
 *   launch); a table built for a cache of another width (or geometry) sets
 *   KVQ_DEVERR_BAD_TABLE in error_flags and the output is invalid.
 *   workspace: at least kvq_decode_workspace_bytes bytes, zero-filled before
 *   first use, left zero-filled.  Errors as kvq_decode_attn.
 */
kvq_status kvq_rope_table_bytes(const kvq_cache* cache, size_t* bytes);
kvq_status kvq_rope_table(const kvq_cache* cache, float base, float* table, void* stream);
kvq_status kvq_decode_attn_rope(const kvq_cache* cache, int32_t n_q_heads, const void* q, float* out,
                                float sm_scale, const float* table, size_t table_bytes, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * kvq_selftest_bounded_wait -- checks, on the current device, the bounded wait
 * that the kernels use for staged data.  One CTA of two warps waits on a
 * shared-memory mbarrier that expects one arrival, polling at most max_polls
 * times.  With arrive != 0 a thread arrives first and the wait completes; with
 * arrive == 0 nothing arrives, the wait gives up, KVQ_DEVERR_TIMEOUT is OR-ed
 * into *error_flags (device int32) and the kernel returns normally (no copy is
 * in flight, the context stays usable).  There is no counterpart in the pages:
 * it is a diagnostic of the library's own failure path.  KVQ_ERR_INVALID for a
 * NULL or misaligned error_flags or max_polls == 0.
 */
kvq_status kvq_selftest_bounded_wait(int32_t* error_flags, uint32_t max_polls, int32_t arrive, void* stream);

/* Human-readable name of a status code.  Never NULL. */
const char* kvq_status_string(int status);

/* Library version, e.g. "0.1.0". */
const char* kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
