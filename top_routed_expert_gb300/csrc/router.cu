// Fused router: logits, top-k selection and renormalised softmax gates in one
// launch, written straight to ids / weights with no logits round trip through
// global memory.
//
// Sarvam blog (NVIDIA, "How NVIDIA extreme hardware-software co-design
// delivered a large inference boost for Sarvam AI's sovereign models"),
// Table 1 row "Router logits and TopK" and the "MoE routing" paragraph after
// it: logit computation and selection fused into a single kernel; the router
// weights are small and replicated.  Sarvam summary (peacm.com news/791474)
// section 3.1: the kernel computes the logits in parallel, selects the top-k
// in place and writes the expert assignment directly, with warp-level
// reductions.
//
// GB300 design: a CTA owns TOK tokens and all E experts for a slice of the
// hidden dimension; the S CTAs of a thread-block cluster split the hidden
// dimension.  Each token has an owner rank; every rank stores its partial
// logits of that token into the owner's shared memory (distributed shared
// memory stores, no remote loads), and after one cluster barrier the owner
// sums them in rank order (deterministic), adds the bias and runs the warp
// top-k (redux-based arg-max rounds, one warp per token).
//
// Inside a CTA of 256 threads a thread owns one expert and keeps all TOK
// token sums in registers.  With E <= 128 the threads form two groups that
// take alternate 8-column steps of every staged chunk (two warps per SM
// sub-partition share the FMA work), and group 1 hands its sums to group 0
// through shared memory at the end.  Chunks of 64 hidden columns of W_r and
// x are staged with cp.async, double-buffered (about 36 KB a stage, so two
// CTAs fit on an SM and a 16-CTA cluster always finds room), and read back as
// float4 (W_r rows padded by 4 floats so a warp's 32 row reads spread over
// all banks; x reads are broadcasts).  Logits stay fp32 from bf16/fp32
// inputs.
#include <cooperative_groups.h>

#include "common.cuh"
#include "topk.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRouterThreads = 256;
constexpr int kRouterKC = 64;             // hidden-dim chunk per pipeline stage
constexpr int kRouterWPitch = kRouterKC + 4;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename XT>
struct XStage {          // x chunk row pitch in elements (16-byte aligned rows)
  static constexpr int kPitch = kRouterKC + 16 / static_cast<int>(sizeof(XT));
};

// eight consecutive x values as floats
__device__ __forceinline__ void x8_to_float(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void x8_to_float(const uint16_t* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <typename XT, int TOK, int EMAX>
struct RouterSmem {
  static constexpr int KG = kRouterThreads / EMAX;   // column groups (2 for E <= 128, else 1)
  static constexpr size_t kWStage = static_cast<size_t>(EMAX) * kRouterWPitch * sizeof(float);   // bytes
  static constexpr size_t kXStage = (static_cast<size_t>(TOK) * XStage<XT>::kPitch * sizeof(XT) + 15) / 16 * 16;
  static constexpr size_t kStage = kWStage + kXStage;
  // after the two staging buffers: the receive buffer [S][ceil(TOK/S)][EMAX]
  // (S * ceil(TOK/S) <= TOK + 16 rows) and one summed row per warp
  static constexpr size_t kRecv = static_cast<size_t>(TOK + 16) * EMAX * sizeof(float);
  static constexpr size_t kRows = (kRouterThreads / 32) * static_cast<size_t>(EMAX) * sizeof(float);
  static constexpr size_t kTotal = 2 * kStage + kRecv + kRows;
  static_assert(static_cast<size_t>(TOK) * EMAX * sizeof(float) <= 2 * kStage, "group hand-off exceeds staging");
};

// TOK tokens per CTA, EMAX = 128 or 256 experts per CTA (E <= EMAX).
template <typename XT, int TOK, int EMAX>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(const XT* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
              int T, int d, int E, int k, int kslice, int32_t* __restrict__ ids, float* __restrict__ gates,
              unsigned* status) {
  using L = RouterSmem<XT, TOK, EMAX>;
  constexpr int KG = L::KG;
  constexpr int XP = XStage<XT>::kPitch;
  extern __shared__ __align__(16) uint8_t smem_u8[];
  // [2 stages: W_r chunk EMAX x (KC+4) floats | x chunk TOK x XP]
  // [recv: partial logits pushed here by every rank] [one summed row per warp]
  float* recv = reinterpret_cast<float*>(smem_u8 + 2 * L::kStage);
  float* rows = recv + (TOK + 16) * EMAX;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned S = cluster.num_blocks();
  const unsigned rank = cluster.block_rank();
  const int tile = blockIdx.x / S;
  const int t0 = tile * TOK;
  const int tid = threadIdx.x;
  const int e_own = tid % EMAX;     // this thread's expert
  const int grp = tid / EMAX;       // its column group
  const int kbeg = min(d, static_cast<int>(rank) * kslice);
  const int kend = min(d, kbeg + kslice);
  const int nchunks = (kend - kbeg) / kRouterKC;

  pdl_enter();
  // distributed shared memory may only be touched once every CTA of the
  // cluster runs: arrive now, wait before the first remote store
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  auto wstage = [&](int buf) { return reinterpret_cast<float*>(smem_u8 + buf * L::kStage); };
  auto xstage = [&](int buf) { return reinterpret_cast<XT*>(smem_u8 + buf * L::kStage + L::kWStage); };

  auto stage_chunk = [&](int c, int buf) {
    const int k0 = kbeg + c * kRouterKC;
    float* wdst = wstage(buf);
    for (int i = tid; i < EMAX * (kRouterKC / 4); i += kRouterThreads) {
      const int r = i / (kRouterKC / 4), c4 = (i % (kRouterKC / 4)) * 4;
      float* dst = wdst + r * kRouterWPitch + c4;
      if (r < E) cp_async16(dst, wr + static_cast<size_t>(r) * d + k0 + c4);
      else *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    XT* xdst = xstage(buf);
    constexpr int EPC = 16 / static_cast<int>(sizeof(XT));   // elements per 16-byte piece
    for (int i = tid; i < TOK * (kRouterKC / EPC); i += kRouterThreads) {
      const int r = i / (kRouterKC / EPC), c = (i % (kRouterKC / EPC)) * EPC;
      XT* dst = xdst + r * XP + c;
      if (t0 + r < T) cp_async16(dst, x + static_cast<size_t>(t0 + r) * d + k0 + c);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  };

  float acc[TOK];
#pragma unroll
  for (int b = 0; b < TOK; ++b) acc[b] = 0.f;

  if (nchunks > 0) stage_chunk(0, 0);
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) stage_chunk(c + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const float* wrow = wstage(buf) + e_own * kRouterWPitch;
    const XT* xb = xstage(buf);
#pragma unroll 2
    for (int kk = grp * 8; kk < kRouterKC; kk += 8 * KG) {
      const float4 wa = *reinterpret_cast<const float4*>(wrow + kk);
      const float4 wb = *reinterpret_cast<const float4*>(wrow + kk + 4);
      const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int b = 0; b < TOK; ++b) {
        float xv[8];
        x8_to_float(xb + b * XP + kk, xv);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[b] = fmaf(xv[q], w[q], acc[b]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // column group 1 hands its sums to group 0 through the (now idle) staging
  // buffers; group 0 adds them in a fixed order
  if (KG == 2) {
    float* hand = reinterpret_cast<float*>(smem_u8);
    if (grp == 1) {
#pragma unroll
      for (int b = 0; b < TOK; ++b) hand[b * EMAX + e_own] = acc[b];
    }
    __syncthreads();
    if (grp == 0) {
#pragma unroll
      for (int b = 0; b < TOK; ++b) acc[b] += hand[b * EMAX + e_own];
    }
  }

  // Push: token b is owned by rank b % S (local slot b / S); every rank
  // stores its partial logits of b into the owner's receive buffer at
  // [my rank][slot][expert] through distributed shared memory.  The receive
  // buffer is never used for staging, so no rank can overwrite live data.
  const int slots = (TOK + static_cast<int>(S) - 1) / static_cast<int>(S);
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (grp == 0) {
#pragma unroll
    for (int b = 0; b < TOK; ++b) {
      const unsigned owner = static_cast<unsigned>(b) % S;
      float* dst = cluster.map_shared_rank(recv, owner) + (rank * slots + b / static_cast<int>(S)) * EMAX;
      dst[e_own] = acc[b];
    }
  }
  cluster.sync();   // every partial row has arrived at its owner
  // One warp per owned token: sum the S partial rows in rank order
  // (deterministic), add the bias, select.
  constexpr int kWarps = kRouterThreads / 32;
  const int warp = tid >> 5, lane = tid & 31;
  float* lrow = rows + warp * EMAX;
  for (int sl = warp; sl < slots; sl += kWarps) {
    const int b = sl * static_cast<int>(S) + static_cast<int>(rank);
    const int t = t0 + b;
    if (b >= TOK || t >= T) break;
    for (int e = lane; e < EMAX; e += 32) {
      float v = 0.f;
      for (unsigned q = 0; q < S; ++q) v += recv[(q * slots + sl) * EMAX + e];
      if (e < E && bias) v += bias[e];
      lrow[e] = v;
    }
    __syncwarp();
    warp_topk_token<EMAX / 32>(lrow, E, k, lane, ids + static_cast<size_t>(t) * k, gates + static_cast<size_t>(t) * k,
                               status);
    __syncwarp();
  }
}

template <typename XT, int TOK, int EMAX>
static cudaError_t launch_router_t(const void* x, const float* wr, const float* bias, int T, int d, int E, int k,
                                   int S, int32_t* ids, float* w, unsigned* status, cudaStream_t stream) {
  using L = RouterSmem<XT, TOK, EMAX>;
  const int tiles = ceil_div(T, TOK);
  // hidden-dim slice per cluster rank, a multiple of the staging chunk
  const int kslice = ceil_div(ceil_div(d, S), kRouterKC) * kRouterKC;
  constexpr size_t smem = L::kTotal;
  static_assert(smem <= 227 * 1024, "router staging exceeds shared memory");
  cudaError_t err = ensure_kernel_attrs(reinterpret_cast<const void*>(router_kernel<XT, TOK, EMAX>),
                                        static_cast<int>(smem), S > 8);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * S);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, router_kernel<XT, TOK, EMAX>, static_cast<const XT*>(x), wr, bias, T, d, E, k,
                            kslice, ids, w, status);
}

// Chooses tokens-per-CTA and the cluster split so that small T still spreads
// over the SMs: S ranks split d (up to 16, a non-portable cluster size the
// GPU supports), each rank at least two staging chunks.
cudaError_t launch_router(const void* x, bool x_bf16, const float* wr, const float* bias, int T, int d, int E,
                          int k, int32_t* ids, float* w, unsigned* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const bool big = T >= 1024;
  const int TOK = big ? 32 : 8;
  const int tiles = ceil_div(T, TOK);
  int S = 1;
  while (S < 16 && tiles * S < num_sms && d / (2 * S) >= 2 * kRouterKC) S *= 2;
  const bool e128 = E <= 128;
#define MOE_ROUTER_CASE(XT, TOKC, EM) \
  return launch_router_t<XT, TOKC, EM>(x, wr, bias, T, d, E, k, S, ids, w, status, stream)
  if (x_bf16) {
    if (big) { if (e128) MOE_ROUTER_CASE(uint16_t, 32, 128); else MOE_ROUTER_CASE(uint16_t, 32, 256); }
    else     { if (e128) MOE_ROUTER_CASE(uint16_t, 8, 128); else MOE_ROUTER_CASE(uint16_t, 8, 256); }
  } else {
    if (big) { if (e128) MOE_ROUTER_CASE(float, 32, 128); else MOE_ROUTER_CASE(float, 32, 256); }
    else     { if (e128) MOE_ROUTER_CASE(float, 8, 128); else MOE_ROUTER_CASE(float, 8, 256); }
  }
#undef MOE_ROUTER_CASE
}

}  // namespace moe
