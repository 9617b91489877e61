// Deterministic combine: y[t] = shared[t] + sum_j out_perm[row_of[t*k+j]],
// the routed terms added in slot order j = 0..k-1 (a gather, no atomics), so
// the result is bitwise reproducible.  Sarvam summary (peacm.com
// news/791474) section 2.1: the shared expert handles common features and the
// routed experts specific ones; their outputs are summed per token.
#include "common.cuh"

namespace moe {

template <bool OUT_BF16>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ out_perm, const int32_t* __restrict__ row_of,
               const float* __restrict__ shared, void* __restrict__ y, int T, int d, int k, int P,
               unsigned* status) {
  const int d4 = d / 4;
  const size_t total = static_cast<size_t>(T) * d4;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / d4);
    const int c = static_cast<int>(i % d4);
    float4 acc = reinterpret_cast<const float4*>(shared + static_cast<size_t>(t) * d)[c];
    for (int j = 0; j < k; ++j) {
      const int r = row_of[static_cast<size_t>(t) * k + j];
      if (r < 0 || r >= P) { set_status(status, MOE_ERR_DEVICE_BOUNDS); continue; }
      const float4 v = reinterpret_cast<const float4*>(out_perm + static_cast<size_t>(r) * d)[c];
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

cudaError_t launch_combine(const float* out_perm, const int32_t* row_of, const float* shared, void* y,
                           bool y_bf16, int T, int d, int k, unsigned* status, int num_sms,
                           cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const size_t total = static_cast<size_t>(T) * (d / 4);
  const int blocks = static_cast<int>(std::min<size_t>(ceil_div(static_cast<int>(std::min<size_t>(total, 1u << 30)), 256),
                                                        static_cast<size_t>(num_sms) * 8));
  count_launches(1);
  if (y_bf16)
    combine_kernel<true><<<blocks, 256, 0, stream>>>(out_perm, row_of, shared, y, T, d, k, T * k, status);
  else
    combine_kernel<false><<<blocks, 256, 0, stream>>>(out_perm, row_of, shared, y, T, d, k, T * k, status);
  return cudaGetLastError();
}

}  // namespace moe
