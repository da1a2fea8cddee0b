/*
 * kvq_rdkv.h -- C ABI of the RDKV bit allocation of the GB300 (sm_103a) low-bit
 * KV-cache library: the widths that kvq_trizone_build takes.  Conventions
 * (device pointers owned by the caller, no allocation, no stream
 * synchronisation, host-side validation before any launch) are those of kvq.h.
 *
 * What it computes ("RDKV" summary, gist.science 2605.08317, sections 2.1 and
 * 2.2), per (sequence b, KV head h) of a prompt of T = n_tokens[b] positions:
 *   token weight   w[t] = sum over the G query heads of the group and over the
 *                  query positions tau >= t of the causal attention
 *                  softmax_{t' <= tau}(sm_scale * q[tau] . k[t'])[t]
 *                  (section 2.1: total attention a token receives);
 *   token cost     W_t = w[t] * var(v[t, :])         (population variance over
 *                  the D channels), for the old tokens t < t_old;
 *   V widths       per old token, from {0, 2, 4, 8, 16} (0 = evicted, 16 =
 *                  fp16), minimising sum W_t 2^-b_t subject to
 *                  sum b_t <= floor(v_avg_bits * t_old)  (phase 2);
 *   channel cost   W_c = ||Q[:, c]|| ||K[:, c]|| / sqrt(D) * var(K[:, c]), Q over
 *                  all T positions and the G heads, K and its variance over the
 *                  kept old tokens (v width != 0)  (section 2.1, phase 3);
 *   K widths       per channel, from {2, 4, 8}, minimising sum W_c 2^-b_c
 *                  subject to sum b_c <= floor(k_avg_bits * D).
 * Both allocations are Lagrangian (section 2.2): with cost(b) =
 * fl32(fl32(W 2^-b) + fl32(lam b)), every unit takes the width of least cost
 * (ties to the smaller width) for the smallest float32 lam >= 0, found by a
 * binary search over its bit pattern, whose choices fit the budget; if none
 * does, lam is the largest finite float32.  Given the same W the widths are
 * exact and deterministic.
 */
#ifndef KVQ_RDKV_H_
#define KVQ_RDKV_H_

#include "kvq.h"

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_RDKV_MAX_TOKENS (1 << 20)

/*
 * Geometry.
 *   batch       B (<= KVQ_MAX_BATCH)
 *   n_q_heads   Hq, a multiple of n_kv_heads with Hq/Hkv in {1, 2, 4, 8}
 *   n_kv_heads  Hkv
 *   head_dim    D, 128 only
 *   max_tokens  row capacity of the weight arrays (>= every n_tokens[b], <= KVQ_RDKV_MAX_TOKENS)
 */
typedef struct kvq_rdkv {
  int32_t batch;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t max_tokens;
} kvq_rdkv;

/* kvq_rdkv_workspace_bytes -- scratch bytes of both calls (host only). */
kvq_status kvq_rdkv_workspace_bytes(const kvq_rdkv* r, size_t* bytes);

/*
 * kvq_rdkv_token_weights -- phase 1, V side: w[b][h][t] for every t < n_tokens[b]
 * (two tensor-core passes over the causal score matrix: per query row the
 * log-sum-exp, then per key the column sum of the normalised probabilities).
 *   q         fp16 device [s][tau][hq][d], element strides q_sb, q_st, q_sh
 *   k         fp16 device [s][t][h][d], element strides k_sb, k_st, k_sh
 *             (strides multiples of 8, bases 16-byte aligned, d contiguous)
 *   n_tokens  HOST int32 [B]: prompt positions of each sequence (0..max_tokens)
 *   sm_scale  softmax scale (e.g. 1/sqrt(D))
 *   w         fp32 device [B][Hkv][max_tokens]; entries t >= n_tokens[b] untouched
 *   workspace at least kvq_rdkv_workspace_bytes bytes, 256-byte aligned
 */
kvq_status kvq_rdkv_token_weights(const kvq_rdkv* r, const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                                  const void* k, int64_t k_sb, int64_t k_st, int64_t k_sh,
                                  const int32_t* n_tokens, float sm_scale, float* w, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * kvq_rdkv_allocate -- phases 2 and 3: V widths of the old tokens, then K widths
 * of the channels over the kept old tokens.
 *   q, k      as kvq_rdkv_token_weights; v fp16 device with the strides of k
 *   n_tokens  HOST int32 [B]: prompt positions (the rows of Q)
 *   t_old     HOST int32 [B]: tokens [0, t_old) are old (t_old <= n_tokens, <= max_old)
 *   w         the token weights of kvq_rdkv_token_weights
 *   v_avg_bits, k_avg_bits  budgets in bits per unit (>= 0, finite)
 *   v_width   uint8 device [B][Hkv][max_old]: entries t < t_old[b] written
 *   k_width   uint8 device [B][Hkv][D]
 *   W_t       fp32 device [B][Hkv][max_old] or NULL: the token costs used
 *   W_c       fp32 device [B][Hkv][D] or NULL: the channel costs used
 *   workspace as kvq_rdkv_token_weights (the same buffer may be passed to both)
 * The outputs are laid out as kvq_trizone_build reads them.
 */
kvq_status kvq_rdkv_allocate(const kvq_rdkv* r, const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                             const void* k, const void* v, int64_t k_sb, int64_t k_st, int64_t k_sh,
                             const int32_t* n_tokens, const int32_t* t_old, const float* w, float v_avg_bits,
                             float k_avg_bits, uint8_t* v_width, int32_t max_old, uint8_t* k_width, float* W_t,
                             float* W_c, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_RDKV_H_ */
