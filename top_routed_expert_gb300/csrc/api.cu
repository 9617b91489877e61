// Host side of the C ABI declared in include/moe_gb300.h: argument
// validation, workspace planning and launch sequencing on the caller's
// stream.  No call synchronises the host or allocates device memory.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moe {
// launchers (one per translation unit)
cudaError_t launch_router(const void* x, bool x_bf16, const float* wr, const float* bias, int T, int d, int E,
                          int k, int32_t* ids, float* w, unsigned* status, int num_sms, cudaStream_t stream);
bool router_tc_supported(int T, int d, int E, bool x_bf16);
size_t router_tc_ws_bytes(int d);
cudaError_t launch_router_tc(const void* x, const float* wr, const float* bias, int T, int d, int E, int k,
                             int32_t* ids, float* w, void* ws, unsigned* status, int num_sms, cudaStream_t stream);
size_t permute_ws_bytes(int P, int E);
cudaError_t launch_permute(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                           int32_t* row_of, void* ws, unsigned* status, cudaStream_t stream);
size_t ffn_simt_ws_bytes(int T, int k, int f, int fs);
cudaError_t launch_ffn_simt(const void* x, bool x_bf16, int w_dtype, const float* topk_w, const int32_t* offsets,
                            const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                            bool out_bf16, int T, int d, int E, int k, int f, int fs, void* ws, unsigned* status,
                            cudaStream_t stream);
bool ffn_tc_supported(const moe_config_t& c);
size_t ffn_tc_ws_bytes(const moe_config_t& c);
cudaError_t launch_ffn_tc(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                          const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                          void* ws, unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream);
bool ffn_fp4_supported(const moe_config_t& c);
size_t ffn_fp4_ws_bytes(const moe_config_t& c);
cudaError_t launch_ffn_fp4(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                           const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                           void* ws, unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream);
bool ffn_nvf4_supported(const moe_config_t& c);
bool ffn_nvf4_preferred(const moe_config_t& c);
size_t ffn_nvf4_ws_bytes(const moe_config_t& c);
cudaError_t launch_ffn_nvf4(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                            const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                            void* ws, unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream);
cudaError_t launch_combine(const void* out_perm, const int32_t* row_of, const void* shared, void* y, bool in_bf16,
                           bool y_bf16, int T, int d, int k, unsigned* status, int num_sms, cudaStream_t stream);
}  // namespace moe

// Per-device status word (see moe_get_device_status).
__device__ unsigned g_moe_status;

// Where moe_get_device_status puts the value it takes out of the status
// word: one slot per call (a host counter picks it), so that readers on
// different host threads never share a slot unless 64 reads overlap.
constexpr int kStatusSlots = 64;
__device__ unsigned g_moe_status_slots[kStatusSlots];

// Reads and clears the status word in one atomic step, after all earlier
// work of the stream, and leaves the value in *slot.
__global__ void status_take_kernel(unsigned* status, unsigned* slot) { *slot = atomicExch(status, 0u); }

namespace moe {
static std::atomic<uint64_t> g_launches{0};
static std::atomic<uint32_t> g_status_reads{0};
void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
}  // namespace moe

namespace {

using namespace moe;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  bool arch_ok = false;
  int num_sms = 0;
  unsigned* status = nullptr;
  unsigned* status_slots = nullptr;
  // the layer's second stream (the shared expert beside the routing) and its
  // fork / join events; created with the device's first call
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_side_mu[kMaxDevices];   // one fork / join sequence at a time per device

// Looks up (once per device) the SM count, the architecture and the status
// word address of the current device.
moe_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    di.arch_ok = (major == 10 && minor == 3);
    di.num_sms = sms;
    if (di.arch_ok) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_moe_status) != cudaSuccess) return MOE_ERR_CUDA;
      di.status = static_cast<unsigned*>(p);
      if (cudaGetSymbolAddress(&p, g_moe_status_slots) != cudaSuccess) return MOE_ERR_CUDA;
      di.status_slots = static_cast<unsigned*>(p);
      if (cudaStreamCreateWithFlags(&di.side, cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&di.fork, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&di.join, cudaEventDisableTiming) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    di.ready = true;
  }
  *out = di;
  return di.arch_ok ? MOE_OK : MOE_ERR_ARCH;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status_t validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model <= 0 || c->d_model % 128 != 0 || c->d_model > 16384) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->n_experts > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->d_ff <= 0 || c->d_ff % 64 != 0 || c->d_ff_shared <= 0 || c->d_ff_shared % 64 != 0)
    return MOE_ERR_INVALID_ARG;
  if (c->d_ff > 65536 || c->d_ff_shared > 65536) return MOE_ERR_INVALID_ARG;
  if (c->x_dtype != MOE_F32 && c->x_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->w_dtype != MOE_F32 && c->w_dtype != MOE_E4M3 && c->w_dtype != MOE_NVFP4) return MOE_ERR_INVALID_ARG;
  if (c->y_dtype != MOE_F32 && c->y_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(c->T) * c->top_k > (int64_t(1) << 30)) return MOE_ERR_INVALID_ARG;
  if ((c->flags & ~(MOE_FLAG_SIMT_FFN | MOE_FLAG_SIMT_ROUTER | MOE_FLAG_BF16_EXPERT_OUT | MOE_FLAG_ACT_E4M3 |
                    MOE_FLAG_ACT_NVFP4 | MOE_FLAG_NVFP4_F16 | MOE_FLAG_NO_OVERLAP | MOE_FLAG_INJECT_TIMEOUT)) != 0)
    return MOE_ERR_INVALID_ARG;
  // NVFP4 activations exist only on the block-scaled FP4 path
  auto nvf4_width = [](int w) { return w % 256 == 0 && w <= 4096; };
  if ((c->flags & MOE_FLAG_ACT_NVFP4) &&
      (c->w_dtype != MOE_NVFP4 || c->x_dtype != MOE_BF16 || (c->flags & (MOE_FLAG_SIMT_FFN | MOE_FLAG_NVFP4_F16)) ||
       !nvf4_width(c->d_model) || !nvf4_width(c->d_ff) || !nvf4_width(c->d_ff_shared)))
    return MOE_ERR_INVALID_ARG;
  // 8-bit activations exist only on the tensor-core FP8 path
  if ((c->flags & MOE_FLAG_ACT_E4M3) &&
      (c->w_dtype != MOE_E4M3 || c->x_dtype != MOE_BF16 || (c->flags & MOE_FLAG_SIMT_FFN) || c->d_ff % 128 != 0 ||
       c->d_ff_shared % 128 != 0))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool use_tc(const moe_config_t& c) {
  return !(c.flags & MOE_FLAG_SIMT_FFN) && ffn_tc_supported(c);
}

bool use_fp4(const moe_config_t& c) {
  return !(c.flags & MOE_FLAG_SIMT_FFN) && ffn_fp4_supported(c);
}

// The block-scaled FP4 path, for configurations it supports: always with
// NVFP4 activations, and for the exact contract when the batch is
// decode-sized (the weight pointers are checked separately: its tensor maps
// need 16-byte aligned block-scale arrays).
bool use_nvf4(const moe_config_t& c) {
  return !(c.flags & (MOE_FLAG_SIMT_FFN | MOE_FLAG_NVFP4_F16)) && ffn_nvf4_supported(c) &&
         ((c.flags & MOE_FLAG_ACT_NVFP4) || ffn_nvf4_preferred(c));
}

bool use_tc_router(const moe_config_t& c) {
  return !(c.flags & MOE_FLAG_SIMT_ROUTER) && router_tc_supported(c.T, c.d_model, c.n_experts, c.x_dtype == MOE_BF16);
}

size_t ffn_ws_bytes(const moe_config_t& c) {
  size_t s = ffn_simt_ws_bytes(c.T, c.top_k, c.d_ff, c.d_ff_shared);
  if (use_tc(c)) s = std::max(s, ffn_tc_ws_bytes(c));
  if (use_fp4(c)) s = std::max(s, ffn_fp4_ws_bytes(c));
  if (use_nvf4(c)) s = std::max(s, ffn_nvf4_ws_bytes(c));
  return s;
}

// Workspace layout of moe_layer_forward.  The routing scratch (tensor-core
// router planes, permutation counts) and the expert-FFN scratch are
// separate, so that the shared expert can run beside the routing on a
// second stream.
struct FwdPlan {
  size_t ids, w, offsets, sorted_pair, row_of, out_perm, shared_out, route_scratch, scratch, total;
};

FwdPlan plan_forward(const moe_config_t& c) {
  const size_t P = static_cast<size_t>(c.T) * c.top_k;
  FwdPlan p;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += align_up(bytes, 256); return at; };
  p.ids = take(sizeof(int32_t) * P);
  p.w = take(sizeof(float) * P);
  p.offsets = take(sizeof(int32_t) * (c.n_experts + 1));
  p.sorted_pair = take(sizeof(int32_t) * P);
  p.row_of = take(sizeof(int32_t) * P);
  const size_t esz = (c.flags & MOE_FLAG_BF16_EXPERT_OUT) ? 2 : 4;   // expert-output element size
  p.out_perm = take(esz * P * c.d_model);
  p.shared_out = take(esz * static_cast<size_t>(c.T) * c.d_model);
  size_t route = permute_ws_bytes(static_cast<int>(P), c.n_experts);
  if (use_tc_router(c)) route = std::max(route, router_tc_ws_bytes(c.d_model));
  p.route_scratch = take(route);
  p.scratch = take(ffn_ws_bytes(c));
  p.total = o;
  return p;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool weights_ok(const moe_config_t& c, const moe_weights_t* w) {
  if (!w || !w->w13 || !w->w2 || !w->s13 || !w->s2) return false;
  const void* q[4] = {w->w13, w->w2, w->s13, w->s2};
  for (const void* p : q)
    if (!aligned(p, 16)) return false;
  if (c.w_dtype == MOE_E4M3 || c.w_dtype == MOE_NVFP4) {
    const void* s[4] = {w->w13_scale, w->w2_scale, w->s13_scale, w->s2_scale};
    const size_t a = (c.w_dtype == MOE_NVFP4) ? 8 : 4;   // NVFP4 scales are fetched 8 bytes at a time
    for (const void* p : s)
      if (!p || !aligned(p, a)) return false;
  }
  if (c.w_dtype == MOE_NVFP4) {
    if (!w->w13_gscale || !w->w2_gscale || !w->s13_gscale || !w->s2_gscale) return false;
  }
  return true;
}

// Which FFN kernels a validated configuration runs; kSimt cannot be split.
enum FfnPath { kFp8Tc, kNvf4, kFp4F16, kSimt, kUnsupported };

FfnPath ffn_path(const moe_config_t& c, const moe_weights_t* w) {
  if (use_tc(c)) return kFp8Tc;
  if (c.flags & MOE_FLAG_ACT_E4M3) return kUnsupported;   // no tensor-map encoder in this driver
  const bool scales16 = aligned(w->w13_scale, 16) && aligned(w->w2_scale, 16) && aligned(w->s13_scale, 16) &&
                        aligned(w->s2_scale, 16);
  if (use_nvf4(c) && scales16) return kNvf4;
  if (c.flags & MOE_FLAG_ACT_NVFP4) return kUnsupported;
  if (use_fp4(c)) return kFp4F16;
  return kSimt;
}

// The expert FFN (routed experts, shared expert, or both: `part`) on the
// kernels the configuration selects.  Arguments are already validated.
moe_status_t run_expert_ffn(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                            const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                            void* ws, const DeviceInfo& di, const FfnPart& part, cudaStream_t s) {
  switch (ffn_path(c, w)) {
    case kFp8Tc:
      return cuda_status(launch_ffn_tc(c, x, topk_w, offsets, sorted_pair, w, out_perm, shared_out, ws, di.status,
                                       di.num_sms, part, s));
    case kNvf4:
      return cuda_status(launch_ffn_nvf4(c, x, topk_w, offsets, sorted_pair, w, out_perm, shared_out, ws, di.status,
                                         di.num_sms, part, s));
    case kFp4F16:
      return cuda_status(launch_ffn_fp4(c, x, topk_w, offsets, sorted_pair, w, out_perm, shared_out, ws, di.status,
                                        di.num_sms, part, s));
    case kSimt:
      if (!part.routed || !part.shared) return MOE_ERR_UNSUPPORTED;
      return cuda_status(launch_ffn_simt(x, c.x_dtype == MOE_BF16, c.w_dtype, topk_w, offsets, sorted_pair, w,
                                         out_perm, shared_out, (c.flags & MOE_FLAG_BF16_EXPERT_OUT) != 0, c.T,
                                         c.d_model, c.n_experts, c.top_k, c.d_ff, c.d_ff_shared, ws, di.status, s));
    default:
      break;
  }
  const bool scales16 = aligned(w->w13_scale, 16) && aligned(w->w2_scale, 16) && aligned(w->s13_scale, 16) &&
                        aligned(w->s2_scale, 16);
  return (c.flags & MOE_FLAG_ACT_NVFP4) && !scales16 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
}

// Whether moe_layer_forward runs the shared expert beside the routing: for
// decode-sized batches (at most 16 routed rows per expert on average), where
// the layer streams weights and the routing leaves most SMs idle (the
// CUDA-core router of a decode batch holds 64 SMs), so the shared expert's
// FFN fits into that time on up to half the GPU and the routed experts still
// get every SM.  Larger batches are bound by the MMAs, which occupy every SM
// with one CTA each; there the shared expert stays in the routed launches
// (a split of the SMs between the two measured slower: T = 8192 FP8,
// 2.15 ms against 1.73 ms).
bool overlap_shared_expert(const moe_config_t& c) {
  return !(c.flags & MOE_FLAG_NO_OVERLAP) && static_cast<double>(c.T) * c.top_k <= 16.0 * c.n_experts;
}

// L2 warm-up of the routed gate/up weights that the GEMM's first wave reads.
// A decode batch routes to nearly every expert, and the grouped GEMM's tile
// list starts at expert 0, so its first wave streams the start of w13; the
// routing in front of it moves almost nothing through HBM.  Prefetching that
// start into L2 on the side stream while the router runs turns those reads
// into L2 hits.  Each thread issues bulk prefetches of 64 KB pieces.  128 MB
// measured best on the 8-GB decode layer (0.2857 -> 0.2844 ms per step, three
// interleaved runs each; 48 and 96 MB were within noise of none).
#ifndef MOE_L2_PREFETCH_MB
#define MOE_L2_PREFETCH_MB 128
#endif

__global__ void l2_prefetch_kernel(const char* base, size_t bytes) {
  constexpr size_t kPiece = 64 * 1024;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x * kPiece;
  for (size_t off = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kPiece; off < bytes;
       off += stride) {
    const uint32_t n = static_cast<uint32_t>(bytes - off < kPiece ? bytes - off : kPiece);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(base + off)), "r"(n)
                 : "memory");
  }
}

// Bytes of routed gate/up weights to warm (a multiple of 16, at most w13).
size_t l2_prefetch_bytes(const moe_config_t& c) {
  const size_t w13 = static_cast<size_t>(c.n_experts) * 2 * c.d_ff * c.d_model / (c.w_dtype == MOE_NVFP4 ? 2 : 1);
  const size_t want = static_cast<size_t>(MOE_L2_PREFETCH_MB) << 20;
  return (want < w13 ? want : w13) & ~static_cast<size_t>(15);
}

}  // namespace

namespace moe {
// Status word address and SM count of the current device (set up on first use).
moe_status_t current_device(unsigned** status, int* num_sms) {
  DeviceInfo di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  *status = di.status;
  *num_sms = di.num_sms;
  return MOE_OK;
}
}  // namespace moe

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_str(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
    case MOE_ERR_ARCH: return "MOE_ERR_ARCH";
    case MOE_ERR_DEVICE_NONFINITE: return "MOE_ERR_DEVICE_NONFINITE";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_workspace_bytes(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  return plan_forward(*cfg).total;
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const float* w_router, const float* expert_bias,
                       int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) ||
      (expert_bias && !aligned(expert_bias, 4)))
    return MOE_ERR_INVALID_ARG;
  if (ws && !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  if (use_tc_router(*cfg) && ws && ws_bytes >= router_tc_ws_bytes(cfg->d_model))
    return cuda_status(launch_router_tc(x, w_router, expert_bias, cfg->T, cfg->d_model, cfg->n_experts, cfg->top_k,
                                        topk_ids, topk_w, ws, di.status, di.num_sms,
                                        static_cast<cudaStream_t>(stream)));
  return cuda_status(launch_router(x, cfg->x_dtype == MOE_BF16, w_router, expert_bias, cfg->T, cfg->d_model,
                                   cfg->n_experts, cfg->top_k, topk_ids, topk_w, di.status, di.num_sms,
                                   static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, int32_t* expert_offsets,
                         int32_t* sorted_pair, int32_t* row_of, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!expert_offsets) return MOE_ERR_INVALID_ARG;
  const int P = cfg->T * cfg->top_k;
  if (P > 0 && (!topk_ids || !sorted_pair || !row_of)) return MOE_ERR_INVALID_ARG;
  const size_t need = permute_ws_bytes(P, cfg->n_experts);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return cuda_status(launch_permute(topk_ids, P, cfg->n_experts, expert_offsets, sorted_pair, row_of, ws,
                                    di.status, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x, const float* topk_w,
                            const int32_t* expert_offsets, const int32_t* sorted_pair, const moe_weights_t* weights,
                            void* out_perm, void* shared_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !topk_w || !expert_offsets || !sorted_pair || !out_perm || !shared_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out_perm, 16) || !aligned(shared_out, 16)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(*cfg, weights)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < ffn_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return run_expert_ffn(*cfg, x, topk_w, expert_offsets, sorted_pair, weights, out_perm, shared_out, ws, di,
                        FfnPart(), static_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* out_perm, const int32_t* row_of,
                         const void* shared_out, void* y, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!out_perm || !row_of || !shared_out || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(out_perm, 16) || !aligned(shared_out, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return cuda_status(launch_combine(out_perm, row_of, shared_out, y, (cfg->flags & MOE_FLAG_BF16_EXPERT_OUT) != 0,
                                    cfg->y_dtype == MOE_BF16, cfg->T,
                                    cfg->d_model, cfg->top_k, di.status, di.num_sms,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const float* w_router,
                               const float* expert_bias, const moe_weights_t* weights, void* y,
                               int32_t* topk_ids_opt, float* topk_w_opt, int32_t* expert_offsets_opt, void* ws,
                               size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) {
    if (expert_offsets_opt) {
      DeviceInfo di;
      if ((st = device_info(&di)) != MOE_OK) return st;
      return cuda_status(cudaMemsetAsync(expert_offsets_opt, 0, sizeof(int32_t) * (cfg->n_experts + 1),
                                         static_cast<cudaStream_t>(stream)));
    }
    return MOE_OK;
  }
  if (!x || !w_router || !y) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(*cfg, weights)) return MOE_ERR_INVALID_ARG;
  const FwdPlan p = plan_forward(*cfg);
  if (!ws || ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  char* base = static_cast<char*>(ws);
  int32_t* ids = reinterpret_cast<int32_t*>(base + p.ids);
  float* w = reinterpret_cast<float*>(base + p.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + p.offsets);
  int32_t* sorted_pair = reinterpret_cast<int32_t*>(base + p.sorted_pair);
  int32_t* row_of = reinterpret_cast<int32_t*>(base + p.row_of);
  void* out_perm = base + p.out_perm;
  void* shared_out = base + p.shared_out;
  void* rscratch = base + p.route_scratch;
  const size_t rscratch_bytes = p.scratch - p.route_scratch;
  void* scratch = base + p.scratch;
  const size_t scratch_bytes = p.total - p.scratch;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const FfnPath path = ffn_path(*cfg, weights);
  if (!overlap_shared_expert(*cfg) || path == kSimt || path == kUnsupported || !di.side) {
    if ((st = moe_route(cfg, x, w_router, expert_bias, ids, w, rscratch, rscratch_bytes, stream)) != MOE_OK) return st;
    if ((st = moe_permute(cfg, ids, offsets, sorted_pair, row_of, rscratch, rscratch_bytes, stream)) != MOE_OK)
      return st;
    if ((st = moe_expert_ffn(cfg, x, w, offsets, sorted_pair, weights, out_perm, shared_out, scratch, scratch_bytes,
                             stream)) != MOE_OK)
      return st;
  } else {
    // The shared expert needs no routing result (Sarvam blog, "hiding
    // latency by overlap": the shared expert runs on a second CUDA stream
    // while the router logits and top-k are computed).  Fork the library's
    // side stream off `stream`, run the shared expert there on at most half
    // the SMs while route -> permute run on `stream`, then the routed experts
    // on every SM, and join before the combine.  The two parts touch
    // disjoint rows of the FFN scratch; the routing has scratch of its own.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_side_mu[dev]);
    FfnPart shared_part, routed_part;
    shared_part.routed = false;
    shared_part.grid_cap = std::max(1, di.num_sms / 2);
    routed_part.shared = false;
    if (cudaEventRecord(di.fork, s) != cudaSuccess || cudaStreamWaitEvent(di.side, di.fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    const size_t warm = (path == kSimt) ? 0 : l2_prefetch_bytes(*cfg);
    if (warm) {
      count_launches(1);
      l2_prefetch_kernel<<<16, 128, 0, di.side>>>(static_cast<const char*>(weights->w13), warm);
      st = cuda_status(cudaGetLastError());
    }
    if (st == MOE_OK)
      st = run_expert_ffn(*cfg, x, w, offsets, sorted_pair, weights, out_perm, shared_out, scratch, di, shared_part,
                          di.side);
    // the join is recorded and awaited on every path, so a capture stays whole
    const bool joined = cudaEventRecord(di.join, di.side) == cudaSuccess;
    if (st == MOE_OK) st = moe_route(cfg, x, w_router, expert_bias, ids, w, rscratch, rscratch_bytes, stream);
    if (st == MOE_OK) st = moe_permute(cfg, ids, offsets, sorted_pair, row_of, rscratch, rscratch_bytes, stream);
    if (st == MOE_OK)
      st = run_expert_ffn(*cfg, x, w, offsets, sorted_pair, weights, out_perm, shared_out, scratch, di, routed_part,
                          s);
    if (!joined || cudaStreamWaitEvent(s, di.join, 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (st != MOE_OK) return st;
  }
  if ((st = moe_combine(cfg, out_perm, row_of, shared_out, y, stream)) != MOE_OK) return st;
  const size_t P = static_cast<size_t>(cfg->T) * cfg->top_k;
  if (topk_ids_opt &&
      cudaMemcpyAsync(topk_ids_opt, ids, sizeof(int32_t) * P, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (topk_w_opt && cudaMemcpyAsync(topk_w_opt, w, sizeof(float) * P, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (expert_offsets_opt &&
      cudaMemcpyAsync(expert_offsets_opt, offsets, sizeof(int32_t) * (cfg->n_experts + 1),
                      cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

uint64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_get_device_status(moe_stream_t stream) {
  DeviceInfo di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* slot = di.status_slots + g_status_reads.fetch_add(1, std::memory_order_relaxed) % kStatusSlots;
  count_launches(1);
  status_take_kernel<<<1, 1, 0, s>>>(di.status, slot);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, slot, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(v);
}

}  // extern "C"
