// Tensor-core router for large token batches: logits on tcgen05 with fp32-
// grade accuracy, then the same warp top-k and renormalised gates as the
// CUDA-core router, all in one kernel (Sarvam blog, Table 1 row "Router
// logits and TopK" and the "MoE routing" paragraph: logits and selection fused
// in one kernel; Sarvam summary section 3.1).
//
// W_r is fp32 and x is bf16.  W_r is split exactly into three bf16 terms,
// w = hi + mid + lo (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid):
// 3 x 8 significant bits cover fp32's 24), so the three bf16 MMAs of each
// k-block sum to x . w with every product exact and fp32 accumulation -- the
// same logits as the fp32 CUDA-core path up to summation order.
//  * split kernel: W_r -> three bf16 planes [3][128][d] in the workspace.
//  * router kernel: the 128 (padded) experts fill the MMA's M lanes, 64 tokens
//    are the N columns; TMA feeds 3 weight tiles + 1 token tile per stage;
//    one thread issues tcgen05.mma kind::f16; four epilogue warps move the
//    [128 x 64] accumulator out of TMEM into shared memory (adding the bias)
//    and each picks the top-k of 16 tokens.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {

using namespace ptx;

constexpr int kRtThreads = 192;
constexpr int kRtTok = 64;                  // tokens per CTA = MMA N
constexpr int kRtBK = 64;                   // bf16 elements (128 bytes) per k-block
constexpr int kRtStages = 3;
constexpr int kRtRows = 128;                // expert rows per plane (E <= 128)
constexpr uint32_t kRtATile = kRtRows * 128;        // 16 KB per term
constexpr uint32_t kRtBTile = kRtTok * 128;         // 8 KB
constexpr uint32_t kRtStage = 3 * kRtATile + kRtBTile;
constexpr int kRtLPitch = kRtRows + 1;              // logits row pitch in shared memory (floats)
constexpr uint64_t kRtWaitNs = 2000000000ull;
constexpr uint64_t kRtDrainNs = 200000000ull;

struct __align__(16) RtCtrl {
  uint64_t full[kRtStages];
  uint64_t empty[kRtStages];
  uint64_t tfull;
  uint64_t drain;
  uint64_t ep_sync;
  uint32_t tmem_base;
  int abort;
};

// Instruction descriptor of a dense kind::f16 MMA with bf16 A and B, fp32 D,
// both K-major: D format [4,6) = 1, A format [7,10) = 1 (bf16), B format
// [10,13) = 1, N >> 3 in [17,23), M >> 4 in [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// W_r [E][d] fp32 -> planes [3][128][d] bf16 (rows >= E are zero).
__global__ void router_split_kernel(const float* __restrict__ wr, int E, int d, __nv_bfloat16* __restrict__ w3) {
  pdl_enter();
  const size_t plane = static_cast<size_t>(kRtRows) * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < plane;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int e = static_cast<int>(i / d);
    const float w = (e < E) ? wr[i] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    w3[i] = hi;
    w3[plane + i] = mid;
    w3[2 * plane + i] = __float2bfloat16_rn(r2);
  }
}

__global__ void __launch_bounds__(kRtThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                 const float* __restrict__ bias, int T, int d, int E, int k, int32_t* __restrict__ ids,
                 float* __restrict__ gates, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RtCtrl* c = reinterpret_cast<RtCtrl*>(smem + kRtStages * kRtStage);
  float* L = reinterpret_cast<float*>(smem);          // [kRtTok][kRtLPitch], reuses the stages
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtTok;
  const int nkb = d / kRtBK;
  volatile int* abort = &c->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(smem_u32(&c->full[s]), 1);
      mbar_init(smem_u32(&c->empty[s]), 1);
    }
    mbar_init(smem_u32(&c->tfull), 1);
    mbar_init(smem_u32(&c->drain), 1);
    mbar_init(smem_u32(&c->ep_sync), 128);
    c->abort = 0;
    fence_barrier_init();
  }
  pdl_enter();   // from here on the kernel reads what earlier kernels wrote
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), kRtTok);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mapW);
      tma_prefetch_desc(&mapX);
      int st = 0;
      uint32_t ph = 0, pending = 0, last_par = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(smem_u32(&c->empty[st]), ph ^ 1u, abort, kRtWaitNs)) break;
        const uint32_t full = smem_u32(&c->full[st]);
        mbar_arrive_expect_tx(full, kRtStage);
        const uint32_t sA = smem_u32(smem + st * kRtStage);
        for (int term = 0; term < 3; ++term) tma_load_2d(sA + term * kRtATile, &mapW, kb * kRtBK, term * kRtRows, full);
        tma_load_2d(sA + 3 * kRtATile, &mapX, kb * kRtBK, t0, full);
        pending |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (ph << st);
        if (++st == kRtStages) {
          st = 0;
          ph ^= 1u;
        }
      }
      int no_abort = 0;
      for (int s = 0; s < kRtStages; ++s)
        if (pending & (1u << s)) mbar_wait(smem_u32(&c->full[s]), (last_par >> s) & 1u, &no_abort, kRtDrainNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kRtRows, kRtTok);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(smem_u32(&c->full[st]), ph, abort, kRtWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = smem_u32(smem + st * kRtStage);
        const uint64_t db = desc_sw128(sA + 3 * kRtATile);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
          const uint64_t da = desc_sw128(sA + term * kRtATile);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // 4 x K=16 bf16 per 128-byte k-block
            mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, (kb | term | kk) != 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&c->empty[st]));
        if (++st == kRtStages) {
          st = 0;
          ph ^= 1u;
        }
      }
      if (ok) mma_commit(smem_u32(&c->tfull));
      mma_commit(smem_u32(&c->drain));
      int no_abort = 0;
      mbar_wait(smem_u32(&c->drain), 0, &no_abort, kRtDrainNs);
    }
  } else {
    // epilogue: TMEM [128 experts x 64 tokens] -> shared logits [token][expert]
    const int sub = warp & 3;
    const int e = sub * 32 + lane;
    const int et = threadIdx.x - 64;
    bool ok = mbar_wait(smem_u32(&c->tfull), 0, abort, kRtWaitNs);
    if (ok) {
      tc_fence_after();
      const float b = (bias && e < E) ? bias[e] : 0.f;
      const uint32_t base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
#pragma unroll
      for (int c0 = 0; c0 < kRtTok; c0 += 16) {
        float v[16];
        tmem_ld16(base + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) L[(c0 + j) * kRtLPitch + e] = v[j] + b;
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&c->ep_sync));
      ok = mbar_wait(smem_u32(&c->ep_sync), 0, abort, kRtWaitNs);
    }
    if (ok) {
      for (int r = et >> 5; r < kRtTok; r += 4) {
        const int t = t0 + r;
        if (t >= T) break;
        warp_topk_token<kRtRows / 32>(L + r * kRtLPitch, E, k, lane, ids + static_cast<size_t>(t) * k,
                                      gates + static_cast<size_t>(t) * k, status);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kRtTok);
  if (threadIdx.x == 0 && c->abort) set_status(status, MOE_ERR_DEVICE_TIMEOUT);
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn rt_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 matrix [rows][cols], box 64 elements (128 bytes) x box_rows, 128-byte swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = rt_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kRtBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The tensor-core router serves bf16 activations, up to 128 experts, and
// batches large enough to fill the SMs with 64-token tiles.
bool router_tc_supported(int T, int d, int E, bool x_bf16) {
  return x_bf16 && E <= kRtRows && d % kRtBK == 0 && T >= 1024 && rt_encode_fn() != nullptr;
}

size_t router_tc_ws_bytes(int d) { return align_up(3 * static_cast<size_t>(kRtRows) * d * 2, 256); }

cudaError_t launch_router_tc(const void* x, const float* wr, const float* bias, int T, int d, int E, int k,
                             int32_t* ids, float* w, void* ws, unsigned* status, int num_sms, cudaStream_t stream) {
  __nv_bfloat16* w3 = static_cast<__nv_bfloat16*>(ws);
  const int split_blocks = std::min(ceil_div(kRtRows * d, 256), 8 * num_sms);
  count_launches(1);
  cudaError_t err = launch_pdl(router_split_kernel, split_blocks, 256, 0, stream, wr, E, d, w3);
  if (err != cudaSuccess) return err;
  CUtensorMap mW, mX;
  if (!make_bf16_map(&mW, w3, 3 * static_cast<uint64_t>(kRtRows), d, kRtRows) ||
      !make_bf16_map(&mX, x, static_cast<uint64_t>(T), d, kRtTok))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + kRtStages * static_cast<size_t>(kRtStage) + sizeof(RtCtrl);
  static_assert(kRtStages * kRtStage >= static_cast<uint32_t>(kRtTok * kRtLPitch * 4),
                "the logits tile reuses the pipeline stages");
  err = ensure_kernel_attrs(reinterpret_cast<const void*>(router_tc_kernel), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  count_launches(1);
  return launch_pdl(router_tc_kernel, ceil_div(T, kRtTok), kRtThreads, smem, stream, mW, mX, bias, T, d, E, k, ids, w,
                    status);
}

}  // namespace moe
