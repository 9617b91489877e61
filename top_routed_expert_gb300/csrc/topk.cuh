// Warp-level top-k with renormalised softmax gates for one token, shared by
// the CUDA-core and the tensor-core routers.  Sarvam summary (peacm.com
// news/791474) section 3.1: the router selects the top-k in place with warp-
// level reductions and writes the expert assignment and scores directly.
#pragma once

#include "common.cuh"

namespace moe {

// `logits` holds the E logits of one token (shared memory, bias already
// added).  k rounds of a warp arg-max keyed on (logit descending, expert index
// ascending) pick ids[0..k); gates are exp(L_j - L_0) / sum_i exp(L_i - L_0).
// A token with fewer than k finite logits records MOE_ERR_DEVICE_NONFINITE.
// EPL = experts per lane (E <= 32 * EPL).  Must be called by a full warp.
template <int EPL>
__device__ __forceinline__ void warp_topk_token(const float* logits, int E, int k, int lane, int32_t* ids_out,
                                                float* gates_out, unsigned* status) {
  float v[EPL];
  bool taken[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? logits[e] : 0.f;
    taken[i] = (e >= E);
  }
  float sel_v0 = 0.f, sum = 0.f;
  float my_z = 0.f;        // lane j keeps slot j's unnormalised gate
  int my_e = 0;
  bool bad = false;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (v[i] > bv || (v[i] == bv && e < be))) { bv = v[i]; be = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if (be == 0x7fffffff || !isfinite(bv)) { bad = true; be = 0; bv = 0.f; }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i == be) taken[i] = true;
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
