// Fused in-place QK-norm + RoPE (include/qk_norm_rope.h).  Sarvam blog,
// Table 1 row "QK Norm + RoPE" and the fused positional-embedding paragraph:
// one pass over q and k, normalisation and rotation together.
//
// Memory-bound: every element is read once and written once.  One block
// per token: its threads copy the token's q rows and k rows (two contiguous
// runs) into shared memory with cp.async (16 bytes per copy, none of it held
// in registers, so a resident block keeps its whole token in flight), load
// the four (cos, sin) pairs of the token's position that each thread needs
// (one 32-byte read) and the gammas while the copies land, then each thread
// computes on the 4 elements i..i+3 of a row's first half and their
// rotate-half partners i+D/2..i+D/2+3 (so each rotation pair sits in one
// thread and needs no exchange) and stores the result straight back.  D/8
// threads cover a row (its sum of squares is a shuffle reduction over
// them).  Sum of squares, the root and the rotation are fp32; the result is
// rounded to bf16 (nearest even) and stored in place.
#include "common.cuh"
#include "../../include/qk_norm_rope.h"

namespace moe {

moe_status_t current_device(unsigned** status, int* num_sms);

namespace {

constexpr int kQrThreads = 128;

__device__ __forceinline__ void unpack4(const uint2& v, float* x) {
  x[0] = __uint_as_float(v.x << 16);
  x[1] = __uint_as_float(v.x & 0xffff0000u);
  x[2] = __uint_as_float(v.y << 16);
  x[3] = __uint_as_float(v.y & 0xffff0000u);
}

__device__ __forceinline__ uint2 pack4(const float* x) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// Block t = token t; its rows h < Hq are query heads, the others key heads.
template <int D>
__global__ void __launch_bounds__(kQrThreads)
qk_norm_rope_kernel(uint16_t* __restrict__ q, uint16_t* __restrict__ k, const float* __restrict__ gq,
                    const float* __restrict__ gk, const float2* __restrict__ cos_sin,
                    const int32_t* __restrict__ positions, int T, int Hq, int Hkv, int n_pos, float eps,
                    unsigned* status) {
  constexpr int TPR = D / 8;                    // threads per row
  constexpr int GROUPS = kQrThreads / TPR;      // rows computed at a time
  constexpr int HALF = D / 2;
  extern __shared__ __align__(16) uint16_t srow[];   // [Hq + Hkv][D]
  pdl_enter();
  const int t = blockIdx.x;
  const int H = Hq + Hkv;
  uint16_t* qt = q + static_cast<size_t>(t) * Hq * D;
  uint16_t* kt = k + static_cast<size_t>(t) * Hkv * D;
  // 1. stage the token's rows
  const int nq = Hq * D / 8, nall = H * D / 8;
  for (int c = threadIdx.x; c < nall; c += kQrThreads) {
    const uint16_t* src = c < nq ? qt + c * 8 : kt + (c - nq) * 8;
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(srow + c * 8));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  // meanwhile: position, table entries and gammas of this thread's elements
  const int lr = threadIdx.x % TPR, grp = threadIdx.x / TPR;
  const int i0 = lr * 4;
  const int p = positions[t];
  const bool ok = p >= 0 && p < n_pos;
  const float4* tp = reinterpret_cast<const float4*>(cos_sin + static_cast<size_t>(ok ? p : 0) * HALF + i0);
  const float4 c01 = tp[0], c23 = tp[1];
  const float cs[4][2] = {{c01.x, c01.y}, {c01.z, c01.w}, {c23.x, c23.y}, {c23.z, c23.w}};
  const float4 gq_lo = *reinterpret_cast<const float4*>(gq + i0), gq_hi = *reinterpret_cast<const float4*>(gq + HALF + i0);
  const float4 gk_lo = *reinterpret_cast<const float4*>(gk + i0), gk_hi = *reinterpret_cast<const float4*>(gk + HALF + i0);
  if (!ok) {   // uniform over the block: leave the token's heads as they are
    if (threadIdx.x == 0) set_status(status, MOE_ERR_DEVICE_BOUNDS);
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  // 2. normalise, rotate, store (every warp runs the same number of passes;
  // rows past H compute on zeros, since the shuffles need every lane)
  for (int h0 = 0; h0 < H; h0 += GROUPS) {
    const int h = h0 + grp;
    const bool live = h < H;
    float a[4], b[4];
    unpack4(live ? *reinterpret_cast<const uint2*>(srow + h * D + i0) : make_uint2(0, 0), a);
    unpack4(live ? *reinterpret_cast<const uint2*>(srow + h * D + HALF + i0) : make_uint2(0, 0), b);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) ss = fmaf(b[i], b[i], fmaf(a[i], a[i], ss));
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rstd = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);
    const bool isq = h < Hq;
    const float glo[4] = {isq ? gq_lo.x : gk_lo.x, isq ? gq_lo.y : gk_lo.y, isq ? gq_lo.z : gk_lo.z, isq ? gq_lo.w : gk_lo.w};
    const float ghi[4] = {isq ? gq_hi.x : gk_hi.x, isq ? gq_hi.y : gk_hi.y, isq ? gq_hi.z : gk_hi.z, isq ? gq_hi.w : gk_hi.w};
    float ol[4], oh[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float ya = a[i] * rstd * glo[i];
      const float yb = b[i] * rstd * ghi[i];
      ol[i] = ya * cs[i][0] - yb * cs[i][1];
      oh[i] = yb * cs[i][0] + ya * cs[i][1];
    }
    if (live) {
      uint16_t* dst = isq ? qt + h * D : kt + (h - Hq) * D;
      *reinterpret_cast<uint2*>(dst + i0) = pack4(ol);
      *reinterpret_cast<uint2*>(dst + HALF + i0) = pack4(oh);
    }
  }
}

template <int D>
cudaError_t launch(const moe_qk_rope_config_t& c, void* q, void* k, const float* gq, const float* gk,
                   const float* cs, const int32_t* pos, unsigned* status, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  const size_t smem = static_cast<size_t>(c.n_q_heads + c.n_kv_heads) * D * 2;
  if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t err = ensure_kernel_attrs(reinterpret_cast<const void*>(qk_norm_rope_kernel<D>), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  count_launches(1);
  return launch_pdl(qk_norm_rope_kernel<D>, c.T, kQrThreads, smem, stream, static_cast<uint16_t*>(q),
                    static_cast<uint16_t*>(k), gq, gk, reinterpret_cast<const float2*>(cs), pos, c.T, c.n_q_heads,
                    c.n_kv_heads, c.n_pos, c.eps, status);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_qk_norm_rope(const moe_qk_rope_config_t* cfg, void* q, void* k, const float* gamma_q,
                                         const float* gamma_k, const float* cos_sin, const int32_t* positions,
                                         moe_stream_t stream) {
  using namespace moe;
  if (!cfg || cfg->T < 0 || cfg->n_q_heads < 1 || cfg->n_kv_heads < 1 || cfg->n_pos < 1 ||
      !(cfg->eps > 0.f) || !(cfg->eps < 1e30f))
    return MOE_ERR_INVALID_ARG;
  if (cfg->head_dim != 64 && cfg->head_dim != 128 && cfg->head_dim != 256) return MOE_ERR_INVALID_ARG;
  // a token's q and k rows are staged in shared memory (at most 200 KB)
  if (static_cast<long long>(cfg->n_q_heads + cfg->n_kv_heads) * cfg->head_dim * 2 > 200 * 1024)
    return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!q || !k || !gamma_q || !gamma_k || !cos_sin || !positions) return MOE_ERR_INVALID_ARG;
  if (!al16(q) || !al16(k) || !al16(gamma_q) || !al16(gamma_k) || !al16(cos_sin) || !al16(positions))
    return MOE_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int sms = 0;
  moe_status_t st = current_device(&status, &sms);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  switch (cfg->head_dim) {
    case 64: err = launch<64>(*cfg, q, k, gamma_q, gamma_k, cos_sin, positions, status, sms, s); break;
    case 128: err = launch<128>(*cfg, q, k, gamma_q, gamma_k, cos_sin, positions, status, sms, s); break;
    default: err = launch<256>(*cfg, q, k, gamma_q, gamma_k, cos_sin, positions, status, sms, s); break;
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
