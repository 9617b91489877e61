// Deterministic combine: y[t] = shared[t] + sum_j out_perm[row_of[t*k+j]],
// the routed terms added in fp32 in slot order j = 0..k-1 (a gather, no
// atomics), so the result is bitwise reproducible.  The expert outputs are
// read as fp32 (default) or as bf16 with MOE_FLAG_BF16_EXPERT_OUT.  Sarvam summary (peacm.com
// news/791474) section 2.1: the shared expert handles common features and the
// routed experts specific ones; their outputs are summed per token.
#include "common.cuh"

namespace moe {

__device__ __forceinline__ float4 load4(const float* p, size_t i) { return reinterpret_cast<const float4*>(p)[i]; }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p, size_t i) {
  const uint2 q = reinterpret_cast<const uint2*>(p)[i];
  return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u), __uint_as_float(q.y << 16),
                     __uint_as_float(q.y & 0xffff0000u));
}

template <typename IT, bool OUT_BF16>
__global__ void __launch_bounds__(256)
combine_kernel(const IT* __restrict__ out_perm, const int32_t* __restrict__ row_of,
               const IT* __restrict__ shared, void* __restrict__ y, int T, int d, int k, int P,
               unsigned* status) {
  pdl_enter();
  const int d4 = d / 4;
  const size_t total = static_cast<size_t>(T) * d4;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / d4);
    const int c = static_cast<int>(i % d4);
    float4 acc = load4(shared + static_cast<size_t>(t) * d, c);
    for (int j = 0; j < k; ++j) {
      const int r = row_of[static_cast<size_t>(t) * k + j];
      if (r < 0 || r >= P) { set_status(status, MOE_ERR_DEVICE_BOUNDS); continue; }
      const float4 v = load4(out_perm + static_cast<size_t>(r) * d, c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (OUT_BF16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + static_cast<size_t>(t) * d)[c] = packed;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(y) + static_cast<size_t>(t) * d)[c] = acc;
    }
  }
}

cudaError_t launch_combine(const void* out_perm, const int32_t* row_of, const void* shared, void* y, bool in_bf16,
                           bool y_bf16, int T, int d, int k, unsigned* status, int num_sms,
                           cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const size_t total = static_cast<size_t>(T) * (d / 4);
  const int blocks = static_cast<int>(std::min<size_t>(ceil_div(static_cast<int>(std::min<size_t>(total, 1u << 30)), 256),
                                                        static_cast<size_t>(num_sms) * 8));
  count_launches(1);
  using BF = __nv_bfloat16;
  if (in_bf16) {
    const BF* o = static_cast<const BF*>(out_perm);
    const BF* sh = static_cast<const BF*>(shared);
    if (y_bf16) return launch_pdl(combine_kernel<BF, true>, blocks, 256, 0, stream, o, row_of, sh, y, T, d, k, T * k, status);
    return launch_pdl(combine_kernel<BF, false>, blocks, 256, 0, stream, o, row_of, sh, y, T, d, k, T * k, status);
  } else {
    const float* o = static_cast<const float*>(out_perm);
    const float* sh = static_cast<const float*>(shared);
    if (y_bf16)
      return launch_pdl(combine_kernel<float, true>, blocks, 256, 0, stream, o, row_of, sh, y, T, d, k, T * k, status);
    return launch_pdl(combine_kernel<float, false>, blocks, 256, 0, stream, o, row_of, sh, y, T, d, k, T * k, status);
  }
}

}  // namespace moe
