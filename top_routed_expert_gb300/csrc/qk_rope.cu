// Fused in-place QK-norm + RoPE (include/qk_norm_rope.h).  Sarvam blog,
// Table 1 row "QK Norm + RoPE" and the fused positional-embedding paragraph:
// one pass over q and k, normalisation and rotation together.
//
// Memory-bound: every element is read once and written once.  One warp owns
// one (token, head) row of D = 32 * EPL elements, a lane EPL consecutive
// elements (one vector load); the rotate-half partner of element i < D/2 is
// element i + D/2, which sits in lane (lane ^ 16).  Each warp takes ROWS
// consecutive rows per step and issues all their loads before any
// arithmetic, so that enough bytes are in flight to keep HBM busy.  The
// token's row of the (cos, sin) table is read through L1/L2 (it is shared
// by all heads of the token).  Sum of squares, the root and the rotation are
// fp32; the result is rounded to bf16 (nearest even) and stored in place.
#include "common.cuh"
#include "../../include/qk_norm_rope.h"

namespace moe {

moe_status_t current_device(unsigned** status, int* num_sms);

namespace {

constexpr int kQrThreads = 256;
constexpr int kQrRows = 4;   // rows per warp and step

template <int EPL> struct Vec;
template <> struct Vec<2> { using T = uint32_t; };
template <> struct Vec<4> { using T = uint2; };
template <> struct Vec<8> { using T = uint4; };

template <int EPL>
__device__ __forceinline__ void unpack(const typename Vec<EPL>::T& v, float (&x)[EPL]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < EPL / 2; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int EPL>
__device__ __forceinline__ typename Vec<EPL>::T pack(const float (&x)[EPL]) {
  typename Vec<EPL>::T v;
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < EPL / 2; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return v;
}

template <int EPL>
__global__ void __launch_bounds__(kQrThreads)
qk_norm_rope_kernel(uint16_t* __restrict__ q, uint16_t* __restrict__ k, const float* __restrict__ gq,
                    const float* __restrict__ gk, const float2* __restrict__ cos_sin,
                    const int32_t* __restrict__ positions, int T, int Hq, int Hkv, int n_pos, float eps,
                    unsigned* status) {
  pdl_enter();
  constexpr int D = 32 * EPL;
  constexpr int HALF = D / 2;
  using V = typename Vec<EPL>::T;
  const int lane = threadIdx.x & 31;
  const int H = Hq + Hkv;
  const long long rows = static_cast<long long>(T) * H;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kQrThreads / 32);
  const int e0 = lane * EPL;                  // first element of this lane
  const int j0 = e0 % HALF;                   // its frequency index
  const bool lo_half = e0 < HALF;
  float gqv[EPL], gkv[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    gqv[i] = gq[e0 + i];
    gkv[i] = gk[e0 + i];
  }
  for (long long r0 = (blockIdx.x * (kQrThreads / 32) + (threadIdx.x >> 5)) * static_cast<long long>(kQrRows);
       r0 < rows; r0 += nwarps * kQrRows) {
    V v[kQrRows];
    uint16_t* ptr[kQrRows];
    int pos[kQrRows];
#pragma unroll
    for (int u = 0; u < kQrRows; ++u) {
      const long long r = r0 + u;
      ptr[u] = nullptr;
      pos[u] = -1;
      if (r < rows) {
        const int t = static_cast<int>(r / H), h = static_cast<int>(r % H);
        ptr[u] = h < Hq ? q + (static_cast<size_t>(t) * Hq + h) * D : k + (static_cast<size_t>(t) * Hkv + (h - Hq)) * D;
        pos[u] = positions[t];
        v[u] = *reinterpret_cast<const V*>(ptr[u] + e0);
      }
    }
#pragma unroll
    for (int u = 0; u < kQrRows; ++u) {
      if (ptr[u] == nullptr) continue;          // uniform across the warp
      const long long r = r0 + u;
      const bool isq = static_cast<int>(r % H) < Hq;
      if (pos[u] < 0 || pos[u] >= n_pos) {      // uniform across the warp: leave the row as it is
        if (lane == 0) set_status(status, MOE_ERR_DEVICE_BOUNDS);
        continue;
      }
      float x[EPL];
      unpack<EPL>(v[u], x);
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float rstd = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);
      float y[EPL], o[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) y[i] = x[i] * rstd * (isq ? gqv[i] : gkv[i]);
      const float2* cs = cos_sin + static_cast<size_t>(pos[u]) * HALF + j0;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const float other = __shfl_xor_sync(0xffffffffu, y[i], 16);   // the rotate-half partner
        const float2 c = cs[i];
        o[i] = lo_half ? y[i] * c.x - other * c.y : y[i] * c.x + other * c.y;
      }
      *reinterpret_cast<V*>(ptr[u] + e0) = pack<EPL>(o);
    }
  }
}

template <int EPL>
cudaError_t launch(const moe_qk_rope_config_t& c, void* q, void* k, const float* gq, const float* gk,
                   const float* cs, const int32_t* pos, unsigned* status, int num_sms, cudaStream_t stream) {
  const long long rows = static_cast<long long>(c.T) * (c.n_q_heads + c.n_kv_heads);
  const long long steps = (rows + kQrRows - 1) / kQrRows;           // warp-steps of work
  const long long blocks = (steps + kQrThreads / 32 - 1) / (kQrThreads / 32);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(blocks, 8LL * num_sms)));
  count_launches(1);
  return launch_pdl(qk_norm_rope_kernel<EPL>, grid, kQrThreads, 0, stream, static_cast<uint16_t*>(q),
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
  if (static_cast<long long>(cfg->T) * (cfg->n_q_heads + cfg->n_kv_heads) > (1LL << 40)) return MOE_ERR_INVALID_ARG;
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
    case 64: err = launch<2>(*cfg, q, k, gamma_q, gamma_k, cos_sin, positions, status, sms, s); break;
    case 128: err = launch<4>(*cfg, q, k, gamma_q, gamma_k, cos_sin, positions, status, sms, s); break;
    default: err = launch<8>(*cfg, q, k, gamma_q, gamma_k, cos_sin, positions, status, sms, s); break;
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
