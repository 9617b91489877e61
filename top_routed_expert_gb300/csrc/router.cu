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
// dimension and the cluster's rank-0 CTA sums their partial logits out of
// distributed shared memory in rank order (deterministic), adds the bias and
// runs a warp-per-token register top-k (k rounds of a warp arg-max keyed on
// (logit desc, index asc)).  Logits stay fp32 from bf16/fp32 inputs.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRouterThreads = 128;
constexpr int kRouterKC = 32;          // hidden-dim chunk staged in shared memory

// TT tokens per thread (TOK = 8*TT per CTA), EPT experts per thread (E <= 16*EPT).
template <typename XT, int TT, int EPT>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(const XT* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
              int T, int d, int E, int k, int kslice, int32_t* __restrict__ ids, float* __restrict__ gates,
              unsigned* status) {
  constexpr int TOK = 8 * TT;
  constexpr int EMAX = 16 * EPT;
  // Dynamic shared memory, two phases:
  //   main loop : wsm [EMAX][KC+1] | xs [TOK][KC+1]
  //   reduction : lp  [TOK][EMAX] aliases wsm (this CTA's partial logits,
  //               read by rank 0) | ls [TOK][EMAX+1] after xs (rank 0 sums)
  extern __shared__ float smem_f[];
  float (*wsm)[kRouterKC + 1] = reinterpret_cast<float (*)[kRouterKC + 1]>(smem_f);
  float (*xs)[kRouterKC + 1] = reinterpret_cast<float (*)[kRouterKC + 1]>(smem_f + EMAX * (kRouterKC + 1));
  float (*lp)[EMAX] = reinterpret_cast<float (*)[EMAX]>(smem_f);
  float (*ls)[EMAX + 1] =
      reinterpret_cast<float (*)[EMAX + 1]>(smem_f + EMAX * (kRouterKC + 1) + TOK * (kRouterKC + 1));

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned S = cluster.num_blocks();
  const unsigned rank = cluster.block_rank();
  const int tile = blockIdx.x / S;
  const int t0 = tile * TOK;
  const int tid = threadIdx.x;
  const int tg = tid >> 4;       // token group: tokens tg*TT .. +TT-1
  const int eg = tid & 15;       // experts eg + 16*i
  const int kbeg = rank * kslice;
  const int kend = min(d, kbeg + kslice);

  float acc[TT][EPT];
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int b = 0; b < EPT; ++b) acc[a][b] = 0.f;

  for (int k0 = kbeg; k0 < kend; k0 += kRouterKC) {
    // stage x[t0..t0+TOK)[k0..k0+KC) and W_r[0..E)[k0..k0+KC) as fp32
    for (int i = tid; i < TOK * kRouterKC; i += kRouterThreads) {
      const int r = i / kRouterKC, c = i % kRouterKC;
      const int t = t0 + r;
      xs[r][c] = (t < T) ? x_to_float<XT>(x[static_cast<size_t>(t) * d + k0 + c]) : 0.f;
    }
    for (int i = tid; i < EMAX * (kRouterKC / 4); i += kRouterThreads) {
      const int r = i / (kRouterKC / 4), c4 = (i % (kRouterKC / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < E) v = *reinterpret_cast<const float4*>(wr + static_cast<size_t>(r) * d + k0 + c4);
      wsm[r][c4 + 0] = v.x; wsm[r][c4 + 1] = v.y; wsm[r][c4 + 2] = v.z; wsm[r][c4 + 3] = v.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRouterKC; ++kk) {
      float xv[TT], wv[EPT];
#pragma unroll
      for (int a = 0; a < TT; ++a) xv[a] = xs[tg * TT + a][kk];
#pragma unroll
      for (int b = 0; b < EPT; ++b) wv[b] = wsm[eg + 16 * b][kk];
#pragma unroll
      for (int a = 0; a < TT; ++a)
#pragma unroll
        for (int b = 0; b < EPT; ++b) acc[a][b] = fmaf(xv[a], wv[b], acc[a][b]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int b = 0; b < EPT; ++b) lp[tg * TT + a][eg + 16 * b] = acc[a][b];

  cluster.sync();   // all partial logits of the cluster are in shared memory
  if (rank == 0) {
    for (int i = tid; i < TOK * EMAX; i += kRouterThreads) {
      const int r = i / EMAX, e = i % EMAX;
      float s = 0.f;
      for (unsigned q = 0; q < S; ++q) {
        const float* remote = cluster.map_shared_rank(&lp[0][0], q);
        s += remote[i];
      }
      if (e < E && bias) s += bias[e];
      ls[r][e] = s;
    }
  }
  cluster.sync();   // peers may exit only after rank 0 has read their partials
  if (rank != 0) return;

  // Top-k: one warp per token.
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int EPL = EMAX / 32 > 0 ? EMAX / 32 : 1;   // experts per lane
  for (int r = warp; r < TOK; r += kRouterThreads / 32) {
    const int t = t0 + r;
    if (t >= T) break;
    float v[EPL];
    bool taken[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? ls[r][e] : 0.f;
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
      ids[static_cast<size_t>(t) * k + lane] = my_e;
      gates[static_cast<size_t>(t) * k + lane] = my_z / sum;
    }
  }
}

template <int TT, int EPT>
constexpr size_t router_smem_bytes() {
  return sizeof(float) * (static_cast<size_t>(16 * EPT) * (kRouterKC + 1) + 8 * TT * (kRouterKC + 1) +
                          8 * TT * (16 * EPT + 1));
}

template <typename XT, int TT, int EPT>
static cudaError_t launch_router_t(const void* x, const float* wr, const float* bias, int T, int d, int E,
                                   int k, int S, int32_t* ids, float* w, unsigned* status,
                                   cudaStream_t stream) {
  constexpr int TOK = 8 * TT;
  const int tiles = ceil_div(T, TOK);
  // hidden-dim slice per cluster rank, a multiple of the staging chunk
  const int kslice = ceil_div(ceil_div(d, S), kRouterKC) * kRouterKC;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * S);
  cfg.blockDim = dim3(kRouterThreads);
  constexpr size_t smem = router_smem_bytes<TT, EPT>();
  static_assert(sizeof(float) * 16 * EPT * (kRouterKC + 1) >= sizeof(float) * 8 * TT * 16 * EPT,
                "partial logits must fit in the weight staging area they alias");
  cudaError_t err = cudaFuncSetAttribute(router_kernel<XT, TT, EPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, router_kernel<XT, TT, EPT>, static_cast<const XT*>(x), wr, bias, T, d, E,
                            k, kslice, ids, w, status);
}

// Chooses tokens-per-CTA and the cluster split so that small T still spreads
// over the SMs: S ranks split d, up to 8 (the portable cluster size).
cudaError_t launch_router(const void* x, bool x_bf16, const float* wr, const float* bias, int T, int d, int E,
                          int k, int32_t* ids, float* w, unsigned* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const bool big = T >= 1024;
  const int TOK = big ? 32 : 8;
  const int tiles = ceil_div(T, TOK);
  int S = 1;
  while (S < 8 && tiles * S < 2 * num_sms && d / (2 * S) >= kRouterKC * 2) S *= 2;
  const bool e128 = E <= 128;
#define MOE_ROUTER_CASE(XT, TT, EPT) return launch_router_t<XT, TT, EPT>(x, wr, bias, T, d, E, k, S, ids, w, status, stream)
  if (x_bf16) {
    if (big) { if (e128) MOE_ROUTER_CASE(uint16_t, 4, 8); else MOE_ROUTER_CASE(uint16_t, 4, 16); }
    else     { if (e128) MOE_ROUTER_CASE(uint16_t, 1, 8); else MOE_ROUTER_CASE(uint16_t, 1, 16); }
  } else {
    if (big) { if (e128) MOE_ROUTER_CASE(float, 4, 8); else MOE_ROUTER_CASE(float, 4, 16); }
    else     { if (e128) MOE_ROUTER_CASE(float, 1, 8); else MOE_ROUTER_CASE(float, 1, 16); }
  }
#undef MOE_ROUTER_CASE
}

}  // namespace moe
