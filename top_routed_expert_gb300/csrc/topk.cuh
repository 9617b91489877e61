// Warp-level top-k with renormalised softmax gates for one token, shared by
// the CUDA-core and the tensor-core routers.  Sarvam summary (peacm.com
// news/791474) section 3.1: the router selects the top-k in place with warp-
// level reductions and writes the expert assignment and scores directly.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving 32-bit key of a finite logit (larger logit -> larger key;
// -0 is folded onto +0 so the two tie).  Non-finite logits map to 0, below
// every finite key (the smallest finite key, of -FLT_MAX, is 0x00800000).
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (!isfinite(v)) return 0u;
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// `logits` holds the E logits of one token (shared memory, bias already
// added).  k rounds each select the untaken expert with the largest logit,
// the lowest expert index among equal logits, to give ids[0..k); gates are
// exp(L_j - L_0) / sum_i exp(L_i - L_0).  A round is one warp max-reduction
// of the lanes' best keys and one min-reduction of the expert indices that
// hold it.  Non-finite logits are never selected; a token with any of them
// records MOE_ERR_DEVICE_NONFINITE (and if fewer than k logits are finite,
// its remaining slots take expert 0 with logit 0).
// EPL = experts per lane (expert e sits in lane e % 32, slot e / 32;
// E <= 32 * EPL).  Must be called by a full warp.
template <int EPL>
__device__ __forceinline__ void warp_topk_token(const float* logits, int E, int k, int lane, int32_t* ids_out,
                                                float* gates_out, unsigned* status) {
  float v[EPL];
  uint32_t key[EPL];
  bool nonfinite = false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? logits[e] : 0.f;
    key[i] = (e < E) ? logit_key(v[i]) : 0u;
    nonfinite |= (e < E) && !isfinite(v[i]);
  }
  float sel_v0 = 0.f, sum = 0.f;
  float my_z = 0.f;        // lane j keeps slot j's unnormalised gate
  int my_e = 0;
  bool bad = __any_sync(0xffffffffu, nonfinite);
  for (int j = 0; j < k; ++j) {
    // this lane's best: largest key, first slot (lowest index) among equals
    uint32_t bk = 0u;
    int bi = 0;
    float bvl = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const bool better = key[i] > bk;
      bk = better ? key[i] : bk;
      bi = better ? i : bi;
      bvl = better ? v[i] : bvl;
    }
    const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t prop = (bk == wk && wk != 0u) ? static_cast<uint32_t>(lane + 32 * bi) : 0xffffffffu;
    const uint32_t we = __reduce_min_sync(0xffffffffu, prop);
    const bool none = wk == 0u;         // no finite logit left
    const int be = none ? 0 : static_cast<int>(we);
    const float sv = __shfl_sync(0xffffffffu, bvl, be & 31);
    const float bv = none ? 0.f : sv;
    bad |= none;
#pragma unroll
    for (int i = 0; i < EPL; ++i) key[i] = (!none && lane + 32 * i == be) ? 0u : key[i];
    if (j == 0) sel_v0 = bv;
    const float z = expf(bv - sel_v0);
    sum += z;
    if (lane == j) { my_z = z; my_e = be; }
  }
  if (bad && lane == 0) set_status(status, MOE_ERR_DEVICE_NONFINITE);
  if (lane < k) {
    ids_out[lane] = my_e;
    gates_out[lane] = my_z / sum;
  }
}

}  // namespace moe
