// Token permutation into per-expert groups: the grouping that feeds the
// grouped expert GEMMs (Sarvam blog, H100 baseline section: expert
// parallelism "uses grouped GEMM kernels"; Table 1 row "Routed expert
// compute").
//
// A stable counting sort of the T*k pairs p = t*k+j keyed by expert:
//   1. hist    : each CTA counts the experts of its chunk of pairs.
//   2. scan    : one CTA turns the per-chunk counts into expert offsets and a
//                per-(chunk, expert) base position.
//   3. scatter : each CTA walks its chunk in pair order and places every pair
//                at base + (pairs of the same expert before it in the chunk),
//                found with a warp match and a per-warp count table.
// Deterministic and stable: within an expert the pairs come out in ascending
// p, hence ascending token.  Ids outside [0, E) are skipped and recorded in
// the device status word; their row_of entry is set to -1.
#include <mutex>

#include "common.cuh"

namespace moe {

constexpr int kPermThreads = 256;
constexpr int kPermChunk = 2048;          // pairs per CTA
constexpr int kPermMaxE = 256;

__global__ void __launch_bounds__(kPermThreads)
permute_hist_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ blk_counts,
                    unsigned* status) {
  pdl_enter();
  __shared__ int hist[kPermMaxE];
  for (int e = threadIdx.x; e < E; e += kPermThreads) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kPermChunk;
  const int end = min(P, base + kPermChunk);
  for (int p = base + threadIdx.x; p < end; p += kPermThreads) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else set_status(status, MOE_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPermThreads) blk_counts[blockIdx.x * E + e] = hist[e];
}

// One CTA of kPermThreads >= E threads.
__global__ void __launch_bounds__(kPermThreads)
permute_scan_kernel(const int32_t* __restrict__ blk_counts, int nblk, int E, int P,
                    int32_t* __restrict__ offsets, int32_t* __restrict__ blk_base) {
  pdl_enter();
  __shared__ int tot[kPermMaxE];
  __shared__ int off[kPermMaxE + 1];
  const int e = threadIdx.x;
  if (e < E) {
    int s = 0;
    for (int b = 0; b < nblk; ++b) s += blk_counts[b * E + e];
    tot[e] = s;
  }
  __syncthreads();
  if (e == 0) {
    int acc = 0;
    for (int i = 0; i < E; ++i) { off[i] = acc; acc += tot[i]; }
    off[E] = acc;
  }
  __syncthreads();
  if (e < E) {
    offsets[e] = off[e];
    int run = off[e];
    for (int b = 0; b < nblk; ++b) {
      blk_base[b * E + e] = run;
      run += blk_counts[b * E + e];
    }
  }
  if (e == 0) offsets[E] = off[E];
}

__global__ void __launch_bounds__(kPermThreads)
permute_scatter_kernel(const int32_t* __restrict__ ids, int P, int E, const int32_t* __restrict__ blk_base,
                       int32_t* __restrict__ sorted_pair, int32_t* __restrict__ row_of) {
  pdl_enter();
  constexpr int W = kPermThreads / 32;
  __shared__ int run[kPermMaxE];        // next free position per expert for this CTA
  __shared__ int wcnt[W][kPermMaxE];    // pairs per (warp, expert) in the current sub-chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += kPermThreads) run[e] = blk_base[blockIdx.x * E + e];
  const int base = blockIdx.x * kPermChunk;
  const int end = min(P, base + kPermChunk);
  for (int c0 = base; c0 < end; c0 += kPermThreads) {
    for (int i = tid; i < W * E; i += kPermThreads) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int p = c0 + tid;
    int e = -1;
    if (p < end) {
      e = ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const unsigned lt = (1u << lane) - 1u;
    const int rank_in_warp = __popc(same & lt);
    if (e >= 0 && rank_in_warp == 0) wcnt[warp][e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
      int pos = run[e] + rank_in_warp;
      for (int w2 = 0; w2 < warp; ++w2) pos += wcnt[w2][e];
      sorted_pair[pos] = p;
      row_of[p] = pos;
    } else if (p < end) {
      row_of[p] = -1;   // an out-of-range id: the combine skips (and reports) this slot
    }
    __syncthreads();
    for (int i = tid; i < E; i += kPermThreads) {
      int s = 0;
      for (int w2 = 0; w2 < W; ++w2) s += wcnt[w2][i];
      run[i] += s;
    }
    __syncthreads();
  }
}

// Whole permutation in one CTA when all pairs fit in one chunk (decode-sized
// batches): histogram, scan and stable scatter without extra launches.
__global__ void __launch_bounds__(kPermThreads)
permute_small_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ sorted_pair, int32_t* __restrict__ row_of, unsigned* status) {
  pdl_enter();
  constexpr int W = kPermThreads / 32;
  __shared__ int run[kPermMaxE + 1];
  __shared__ int wcnt[W][kPermMaxE];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += kPermThreads) run[e] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += kPermThreads) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&run[e], 1);
    else set_status(status, MOE_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      const int c = run[e];
      run[e] = acc;
      offsets[e] = acc;
      acc += c;
    }
    offsets[E] = acc;
  }
  __syncthreads();
  for (int c0 = 0; c0 < P; c0 += kPermThreads) {
    for (int i = tid; i < W * E; i += kPermThreads) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int p = c0 + tid;
    int e = -1;
    if (p < P) {
      e = ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank_in_warp == 0) wcnt[warp][e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
      int pos = run[e] + rank_in_warp;
      for (int w2 = 0; w2 < warp; ++w2) pos += wcnt[w2][e];
      sorted_pair[pos] = p;
      row_of[p] = pos;
    } else if (p < P) {
      row_of[p] = -1;   // an out-of-range id: the combine skips (and reports) this slot
    }
    __syncthreads();
    for (int i = tid; i < E; i += kPermThreads) {
      int s = 0;
      for (int w2 = 0; w2 < W; ++w2) s += wcnt[w2][i];
      run[i] += s;
    }
    __syncthreads();
  }
}

size_t permute_ws_bytes(int P, int E) {
  const int nblk = ceil_div(P, kPermChunk);
  return 2 * align_up(sizeof(int32_t) * static_cast<size_t>(nblk) * E, 256);
}

cudaError_t launch_permute(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                           int32_t* row_of, void* ws, unsigned* status, cudaStream_t stream) {
  const int nblk = ceil_div(P, kPermChunk);
  int32_t* blk_counts = static_cast<int32_t*>(ws);
  int32_t* blk_base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) +
                                                 align_up(sizeof(int32_t) * static_cast<size_t>(nblk) * E, 256));
  if (P == 0) {
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream);
  }
  if (nblk == 1) {
    count_launches(1);
    return launch_pdl(permute_small_kernel, 1, kPermThreads, 0, stream, ids, P, E, offsets, sorted_pair, row_of,
                      status);
  }
  count_launches(3);
  cudaError_t err = launch_pdl(permute_hist_kernel, nblk, kPermThreads, 0, stream, ids, P, E, blk_counts, status);
  if (err == cudaSuccess)
    err = launch_pdl(permute_scan_kernel, 1, kPermThreads, 0, stream, blk_counts, nblk, E, P, offsets, blk_base);
  if (err == cudaSuccess)
    err = launch_pdl(permute_scatter_kernel, nblk, kPermThreads, 0, stream, ids, P, E, blk_base, sorted_pair,
                     row_of);
  return err;
}

// ---------------------------------------------------------------------------
// Allocation-free entry point (moe_permute_noalloc): the per-chunk counts and
// bases live in a fixed array compiled into the library instead of a caller
// workspace.  Sized for MOE_NOALLOC_MAX_PAIRS pairs and kPermMaxE experts:
// two halves of (65536 / 2048 chunks) x 256 experts int32 = 64 KiB.
constexpr int kNoAllocChunks = MOE_NOALLOC_MAX_PAIRS / kPermChunk;
constexpr size_t kNoAllocHalfInts = static_cast<size_t>(kNoAllocChunks) * kPermMaxE;
static __device__ __align__(256) int32_t g_permute_scratch[2 * kNoAllocHalfInts];

static std::mutex g_scratch_mu;
static void* g_scratch_addr[64] = {};

// Device address of g_permute_scratch on the current device, looked up once
// per device with that device current.
static cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

moe_status_t current_device(unsigned** status, int* num_sms);

}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_ids,
                                            int32_t* expert_offsets, int32_t* sorted_pair, int32_t* row_of,
                                            moe_stream_t stream) {
  using namespace moe;
  if (moe_workspace_bytes(cfg) == 0) return MOE_ERR_INVALID_ARG;   // full configuration check
  const long long P = static_cast<long long>(cfg->T) * cfg->top_k;
  if (P > MOE_NOALLOC_MAX_PAIRS) return MOE_ERR_UNSUPPORTED;
  if (!expert_offsets) return MOE_ERR_INVALID_ARG;
  if (P > 0 && (!topk_ids || !sorted_pair || !row_of)) return MOE_ERR_INVALID_ARG;
  // the two halves must be laid out exactly as launch_permute expects
  static_assert(kNoAllocHalfInts * sizeof(int32_t) % 256 == 0, "scratch halves must stay 256-byte aligned");
  if (permute_ws_bytes(static_cast<int>(P), cfg->n_experts) > sizeof(g_permute_scratch)) return MOE_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  int sms = 0;
  moe_status_t st = current_device(&status, &sms);
  if (st != MOE_OK) return st;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_permute(topk_ids, static_cast<int>(P), cfg->n_experts, expert_offsets, sorted_pair, row_of, scratch,
                        status, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
