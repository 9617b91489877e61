/*
 * qk_norm_rope.h -- C ABI of the fused in-place QK-norm + RoPE step
 * (libmoe_gb300.so; status codes and stream type from moe_gb300.h).
 *
 * NVIDIA technical blog "How NVIDIA extreme hardware-software co-design
 * delivered a large inference boost for Sarvam AI's sovereign models",
 * Table 1 row "QK Norm + RoPE" (414 -> 54 us per layer on H100) and the
 * paragraph on fused positional embedding: query-key normalisation and the
 * rotary position embedding in one in-place kernel, one pass over q and k
 * instead of two reads and writes.  The Sarvam summary (peacm.com
 * news/791474, section 3.1) outlines the kernel as taking q, k and a
 * precomputed frequency table.
 *
 * For every token t and head h of q (gamma = gamma_q) and of k (gamma_k),
 * with x = the head's D values and (c_i, s_i) = cos_sin[positions[t]][i]:
 *   y_i  = x_i / sqrt(mean_j(x_j^2) + eps) * gamma_i              (RMSNorm)
 *   out_i       = y_i c_i - y_{i+D/2} s_i      for i < D/2        (RoPE,
 *   out_{i+D/2} = y_{i+D/2} c_i + y_i s_i                          rotate half)
 * computed in fp32 and written back in place, rounded to bf16 (nearest even).
 */
#ifndef QK_NORM_ROPE_H
#define QK_NORM_ROPE_H

#include "moe_gb300.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t T;            /* tokens, >= 0 (0 is a no-op)                          */
  int32_t n_q_heads;    /* query heads, >= 1                                    */
  int32_t n_kv_heads;   /* key heads, >= 1 (grouped-query attention: fewer);
                           (n_q_heads + n_kv_heads) * head_dim * 2 <= 200 KB     */
  int32_t head_dim;     /* D: 64, 128 or 256                                    */
  int32_t n_pos;        /* rows of the frequency table, >= 1                    */
  float eps;            /* RMSNorm epsilon, > 0 and finite                      */
} moe_qk_rope_config_t;

/*
 * q          [T][n_q_heads][D] bf16, normalised and rotated in place
 * k          [T][n_kv_heads][D] bf16, likewise
 * gamma_q/_k [D] float per-channel weights
 * cos_sin    [n_pos][D/2][2] float: (cos, sin) of each position and frequency
 * positions  [T] int32: the table row of each token; a position outside
 *            [0, n_pos) leaves that token's heads unchanged and records
 *            MOE_ERR_DEVICE_BOUNDS in the device status word
 * All pointers are device pointers owned by the caller, 16-byte aligned
 * (MOE_ERR_INVALID_ARG otherwise); the call is asynchronous on `stream`,
 * allocates nothing and uses no workspace.
 */
moe_status_t moe_qk_norm_rope(const moe_qk_rope_config_t* cfg, void* q, void* k, const float* gamma_q,
                              const float* gamma_k, const float* cos_sin, const int32_t* positions,
                              moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QK_NORM_ROPE_H */
