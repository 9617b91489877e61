// Shared device helpers of the MoE layer kernels (sm_103a).
#pragma once

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <set>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/moe_gb300.h"

namespace moe {

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization, so it may be scheduled while the
// previous kernel in the stream is still finishing.  Each kernel therefore
// calls pdl_wait() before it touches global memory that earlier work writes
// or reads (it returns once the previous kernel has completed and its writes
// are visible), and then pdl_launch_dependents() to let the next kernel be
// scheduled early.  A kernel launched without the attribute returns from
// pdl_wait() at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

// Launch with programmatic stream serialization (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}


constexpr int kMaxExperts = 256;

// Which part of the expert FFN one set of launches computes: the routed
// experts (activation rows [0, P)), the shared expert (rows [P, P+T)), or
// both; and the most CTAs its persistent GEMMs may use (the rest of the GPU
// stays free for work running beside them on another stream).
struct FfnPart {
  bool routed = true, shared = true;
  int grid_cap = 1 << 30;
  int row_begin(int P) const { return routed ? 0 : P; }
  int row_end(int P, int T) const { return shared ? P + T : P; }
};
constexpr int kMaxGroups = kMaxExperts + 1;   // routed experts + the shared expert

// Host-side count of kernel launches (moe_launch_count); defined in api.cu.
void count_launches(int n);

// Raises a kernel's dynamic shared-memory limit to at least smem_bytes (and,
// optionally, allows non-portable cluster sizes).  The limit is one value per
// (kernel, device), so it is only ever raised -- lowering it would break a
// later launch that needs more -- and the attribute call is made only when the
// limit actually grows: setting function attributes on every launch costs far
// more than the launch.
inline cudaError_t ensure_kernel_attrs(const void* kernel, int smem_bytes, bool nonportable_cluster = false) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> smem_limit;
  static std::set<std::pair<const void*, int>> nonportable;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const auto key = std::make_pair(kernel, dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = smem_limit.find(key);
  if (it == smem_limit.end() || it->second < smem_bytes) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (err != cudaSuccess) return err;
    smem_limit[key] = smem_bytes;
  }
  if (nonportable_cluster && !nonportable.count(key)) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    nonportable.insert(key);
  }
  return cudaSuccess;
}

// Device status word: kernels record the first fault they see with
// atomicCAS(0 -> code) and carry on with the fault contained (skip the bad
// access, return from a wait).  The host reads and clears it.
__device__ __forceinline__ void set_status(unsigned* status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Activation element -> float (x is fp32 or bf16).
template <typename XT> __device__ __forceinline__ float x_to_float(XT v);
template <> __device__ __forceinline__ float x_to_float<float>(float v) { return v; }
template <> __device__ __forceinline__ float x_to_float<uint16_t>(uint16_t v) { return bf16_bits_to_float(v); }

// FP8 E4M3 code -> float, through the hardware conversion.
__device__ __forceinline__ float e4m3_to_float(uint8_t code) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  return __half2float(__half(h));
}

// E2M1 code (low 4 bits) -> float.  Magnitudes by code 0..7 are the format's
// eight values 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign.
__device__ __forceinline__ float e2m1_to_float(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  float mag = (e == 0) ? 0.5f * static_cast<float>(m)
                       : (1.0f + 0.5f * static_cast<float>(m)) * static_cast<float>(1u << (e - 1));
  return (code & 8u) ? -mag : mag;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

// Expert-output element store: fp32 (default) or bf16 (MOE_FLAG_BF16_EXPERT_OUT).
__device__ __forceinline__ void store_out(void* base, size_t idx, float v, bool out_bf16) {
  if (out_bf16) static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  else static_cast<float*>(base)[idx] = v;
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Device-side group table: routed experts 0..E-1 plus the shared expert as
// group E.  rows(g) = routed count or T; tiles(g) = ceil(rows/TM).
// Fills tile_start[0..E+1] (exclusive prefix of tiles) in shared memory with
// one block-wide pass.
__device__ __forceinline__ void build_tile_table(const int32_t* __restrict__ offsets, int E, int T, int TM,
                                                 int* s_tile_start, int* s_scratch) {
  const int G = E + 1;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int rows = (g < E) ? (offsets[g + 1] - offsets[g]) : T;
    s_scratch[g] = (max(rows, 0) + TM - 1) / TM;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int g = 0; g < G; ++g) { s_tile_start[g] = acc; acc += s_scratch[g]; }
    s_tile_start[G] = acc;
  }
  __syncthreads();
}

// Largest g with tile_start[g] <= i (tile_start non-decreasing, G+1 entries).
__device__ __forceinline__ int find_group(const int* s_tile_start, int G, int i) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s_tile_start[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace moe
