/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) MoE FFN layer forward pass.
 *
 * The layer (NVIDIA technical blog "How NVIDIA extreme hardware-software
 * co-design delivered a large inference boost for Sarvam AI's sovereign
 * models", section "Scaling multilingual sovereign AI with MoE" and Table 1):
 * 128 routed experts with top-k routing (k = 6 for the 30B shape, 8 for the
 * 100B shape), SwiGLU expert FFNs on FP8 or NVFP4 weights, one always-on
 * shared expert, and a per-token weighted combine.
 *
 *   logits  L[t,e] = x[t,:] . W_r[e,:] (+ b[e])
 *   ids[t]  = the k experts of largest L[t,e]; equal logits -> lower index first
 *   w[t,j]  = softmax over all experts, restricted to ids[t], renormalised
 *           = exp(L[t,ids_j] - L[t,ids_0]) / sum_i exp(L[t,ids_i] - L[t,ids_0])
 *   FFN_e(v) = W2_e ( silu(Wg_e v) * (Wu_e v) ),  W13_e = [Wg_e ; Wu_e]
 *   y[t]    = FFN_shared(x[t]) + sum_j w[t,j] FFN_{ids[t,j]}(x[t])
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees or retains them, never copies weights, and allocates no
 *    device memory.  Scratch memory comes from the caller's workspace
 *    (`ws`, at least moe_workspace_bytes(cfg) bytes, 256-byte aligned).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and performs no host synchronisation.  The kernels are
 *    launched with programmatic dependent launch: each waits for the work
 *    before it in the stream, and lets the next kernel be scheduled early.
 *    A kernel the caller launches next with programmatic stream
 *    serialization must therefore wait (cudaGridDependencySynchronize)
 *    before reading this call's outputs; ordinary launches, copies and
 *    events are ordered as usual.
 *  - Argument, shape, alignment and workspace errors are detected on the host
 *    before anything is launched and returned synchronously.  Launch failures
 *    return MOE_ERR_CUDA.  Faults detected on the device (an index out of
 *    range, a bounded wait that ran out, a non-finite logit row) are recorded
 *    in a per-device status word and returned by moe_get_device_status().
 *    Nothing traps, aborts or throws across this boundary.
 *  - Layouts are row-major with the last index contiguous.  Pair p = t*k + j
 *    names slot j of token t.
 *  - The device must be compute capability 10.3 (GB300); otherwise every
 *    launching call returns MOE_ERR_ARCH.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2   /* 2: NVFP4 block-scaled path and flags, shared-expert overlap, moe_qk_norm_rope */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,      /* null / misaligned pointer, bad shape        */
  MOE_ERR_UNSUPPORTED = 2,      /* valid but not implemented combination       */
  MOE_ERR_WORKSPACE = 3,        /* ws NULL or smaller than moe_workspace_bytes */
  MOE_ERR_CUDA = 4,             /* a CUDA runtime / launch error               */
  MOE_ERR_DEVICE_TIMEOUT = 5,   /* a bounded device-side wait ran out          */
  MOE_ERR_DEVICE_BOUNDS = 6,    /* an index read on the device was out of range */
  MOE_ERR_ARCH = 7,             /* current device is not sm_103                */
  MOE_ERR_DEVICE_NONFINITE = 8  /* a router row held a non-finite logit        */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2, MOE_NVFP4 = 3 } moe_dtype_t;

/* Flags (moe_config_t.flags). */
#define MOE_FLAG_SIMT_FFN 0x1u     /* run the expert FFN on the CUDA-core kernels */
#define MOE_FLAG_SIMT_ROUTER 0x2u  /* run the router on the CUDA-core kernel       */
#define MOE_FLAG_BF16_EXPERT_OUT 0x4u  /* out_perm / shared_out in bf16 (default fp32) */
/* 8-bit activations (opt-in, lossy).  By default the FP8 expert GEMMs feed each
 * activation row (x, and H after SwiGLU) to the tensor cores as two E4M3 terms
 * under a per-row power-of-two scale, which reproduces bf16 activations
 * exactly; with this flag only the first term is kept: the row is scaled by
 * s = the smallest power of two with amax <= 448 s, rounded to E4M3 (nearest,
 * ties to even) and H is rounded to bf16 before that.  The MMAs then do half
 * the work.  Error against exact activations is about 5e-2 relative L2 (the
 * E4M3 rounding of every activation), so this is a different numerical
 * contract from the default.  Valid only with E4M3 weights, bf16 x, widths
 * that are multiples of 128 and without MOE_FLAG_SIMT_FFN.  The pages fix the
 * weight formats only; this is the 8-bit-activation reading of their FP8
 * compute. */
#define MOE_FLAG_ACT_E4M3 0x8u
/* NVFP4 activations (opt-in, lossy; W4A4).  By default NVFP4 weights of a
 * decode-sized batch run on the block-scaled FP4 tensor-core MMA with every
 * activation row (x, and H after SwiGLU) written as a sum of four NVFP4 rows
 * found on the residual, which stays within about 5e-5 relative L2 of the
 * bf16 activations.  With
 * this flag only the first term is kept: each row is scaled by
 * g = the smallest power of two with amax <= 6 * 448 * g, every 16
 * consecutive elements get the smallest E4M3 scale s with
 * max|v| <= 6 g s, and each element becomes g s e2m1(v / (g s)) (nearest,
 * ties to even); H is rounded to bf16 before that.  The MMAs then do a
 * quarter of the work, at about 0.1 relative L2 from exact activations.
 * Valid only with NVFP4 weights, bf16 x, widths that are multiples of 256 and
 * at most 4096, and without MOE_FLAG_SIMT_FFN / MOE_FLAG_NVFP4_F16.  This is
 * the FP4-activation reading of the pages' NVFP4 compute. */
#define MOE_FLAG_ACT_NVFP4 0x10u
/* Run NVFP4 weights on the f16 tensor-core path instead (weights rebuilt
 * exactly in f16 in shared memory, kind::f16 MMAs); the path that also
 * serves NVFP4 widths the block-scaled path does not take. */
#define MOE_FLAG_NVFP4_F16 0x20u
/* moe_layer_forward runs the shared expert of a decode-sized batch on a
 * second stream beside the routing by default (see moe_layer_forward); with
 * this flag it runs in the same launches as the routed experts, after the
 * routing, on `stream` only.  The results are the same bit for bit. */
#define MOE_FLAG_NO_OVERLAP 0x40u
/* Test hook for the failure path: in the tensor-core expert GEMM, CTA 0
 * withholds one "accumulator ready" signal and every bounded wait shortens to
 * 20 ms, so the epilogue's wait runs out; the kernel drains its copies and
 * MMAs, frees tensor memory and returns, and moe_get_device_status() reports
 * MOE_ERR_DEVICE_TIMEOUT.  The outputs of that call are not valid. */
#define MOE_FLAG_INJECT_TIMEOUT 0x100u

typedef struct {
  int32_t T;            /* tokens, >= 0 (0 is a no-op)                          */
  int32_t d_model;      /* hidden size d: multiple of 128, <= 16384             */
  int32_t n_experts;    /* E: 1..256 (larger: MOE_ERR_INVALID_ARG, every call)  */
  int32_t top_k;        /* k: 1..min(E,16)                                      */
  int32_t d_ff;         /* routed expert width f: multiple of 64                */
  int32_t d_ff_shared;  /* shared expert width f_s: multiple of 64              */
  int32_t x_dtype;      /* MOE_F32 or MOE_BF16                                  */
  int32_t w_dtype;      /* MOE_F32, MOE_E4M3 or MOE_NVFP4 (expert + shared)     */
  int32_t y_dtype;      /* MOE_F32 or MOE_BF16                                  */
  uint32_t flags;       /* MOE_FLAG_*                                           */
} moe_config_t;

/*
 * Expert weights in their stored formats (device pointers).
 *   w13 : [E][2f][d]   rows 0..f-1 = gate (Wg), rows f..2f-1 = up (Wu)
 *   w2  : [E][d][f]    down projection
 *   s13 : [2f_s][d], s2 : [d][f_s]   shared expert, same formats
 * Per format:
 *   MOE_F32  : float values; *_scale and *_gscale unused (NULL).
 *   MOE_E4M3 : uint8 FP8 E4M3 codes; *_scale = float per output row
 *              (w13_scale [E][2f], w2_scale [E][d], s13_scale [2f_s],
 *              s2_scale [d]); value = e4m3(code) * scale[row].
 *   MOE_NVFP4: uint8, two E2M1 codes per byte along the K (last) axis, element
 *              2i in the low nibble (w13 [E][2f][d/2] ...); *_scale = uint8
 *              E4M3 codes, one per 16 consecutive K elements
 *              (w13_scale [E][2f][d/16] ...); *_gscale = float per expert
 *              ([E] for w13/w2, one float for s13/s2);
 *              value = e2m1(code) * e4m3(block scale) * gscale.
 * Alignment: w13 / w2 / s13 / s2 16 bytes; E4M3 row scales 4 bytes; NVFP4
 * block-scale arrays 8 bytes (a misaligned pointer is MOE_ERR_INVALID_ARG).
 * NVFP4 batches of at most 16 routed rows per expert on average (decode)
 * run on the block-scaled FP4 MMA when the block-scale arrays are 16-byte
 * aligned and the widths are multiples of 256, at most 4096; other NVFP4
 * batches run on the f16 path (see MOE_FLAG_NVFP4_F16).  With
 * MOE_FLAG_ACT_NVFP4 every batch runs on the block-scaled MMA, and
 * misaligned block-scale arrays are MOE_ERR_INVALID_ARG.
 * Source of the formats: the Sarvam summary page (peacm.com news/791474,
 * section 2.1, FP8 expert weights) and the Sarvam blog's Blackwell section
 * (NVFP4 weights).
 */
typedef struct {
  const void* w13; const void* w13_scale; const float* w13_gscale;
  const void* w2;  const void* w2_scale;  const float* w2_gscale;
  const void* s13; const void* s13_scale; const float* s13_gscale;
  const void* s2;  const void* s2_scale;  const float* s2_gscale;
} moe_weights_t;

typedef void* moe_stream_t;   /* a cudaStream_t */

/* ABI version of the loaded library (MOE_ABI_VERSION at build time). */
int moe_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char* moe_status_str(moe_status_t s);

/*
 * Workspace bytes that moe_permute, moe_expert_ffn and moe_layer_forward
 * need for this configuration (the maximum of the three).  Returns 0 for an
 * invalid configuration.  The workspace holds no state between calls.
 */
size_t moe_workspace_bytes(const moe_config_t* cfg);

/*
 * Fused router: logits, softmax restricted to the top k, top-k selection.
 * Sarvam blog, Table 1 row "Router logits and TopK" and the "MoE routing"
 * paragraph (one fused kernel for logit computation and selection); Sarvam
 * summary section 3.1 (the kernel writes expert indices and scores
 * directly); InferX page section 3.3 (int32 indices, fp32 weights).
 *   x           [T][d] (cfg->x_dtype)
 *   w_router    [E][d] float
 *   expert_bias [E] float added to the logits before selection, or NULL
 *   topk_ids    [T][k] int32 out: experts in descending logit order, ties to
 *               the lower index
 *   topk_w      [T][k] float out: renormalised gates (sum to one per token)
 *   ws, ws_bytes optional workspace.  With at least moe_workspace_bytes(cfg)
 *               bytes, batches of >= 1024 bf16 tokens with E <= 128 run the
 *               logits on the tensor cores (W_r split exactly into three bf16
 *               terms held in the workspace); otherwise (or with ws NULL) the
 *               CUDA-core router runs.  Both give fp32-accurate logits.
 * A token whose logits include a non-finite value (from a non-finite input)
 * is routed among its finite logits only and raises
 * MOE_ERR_DEVICE_NONFINITE in the device status word.
 */
moe_status_t moe_route(const moe_config_t* cfg, const void* x, const float* w_router,
                       const float* expert_bias, int32_t* topk_ids, float* topk_w,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Permutation of the T*k (token, slot) pairs into per-expert groups, the
 * token grouping that feeds the grouped expert GEMM (Sarvam blog, section on
 * the H100 baseline: expert parallelism "uses grouped GEMM kernels").
 *   topk_ids       [T][k] int32 in: values in [0, E); an out-of-range id is
 *                  skipped and recorded as MOE_ERR_DEVICE_BOUNDS
 *   expert_offsets [E+1] int32 out: exclusive prefix sum of per-expert counts
 *   sorted_pair    [T*k] int32 out: pairs p = t*k+j ordered by (expert, p)
 *   row_of         [T*k] int32 out: inverse of sorted_pair
 */
moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_ids,
                         int32_t* expert_offsets, int32_t* sorted_pair, int32_t* row_of,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute for callers that cannot allocate device memory: same
 * arguments and results as moe_permute, minus the workspace.  This entry
 * point has no counterpart in the pages; it exists for integrations where
 * device memory belongs to someone else -- a serving engine whose caching
 * allocator or fixed budget must account for every byte, or a latency-
 * critical loop in which a cudaMalloc (which can synchronise the device) is
 * not allowed -- so the caller has no way to obtain a workspace to pass in.
 *
 * Its scratch is one 64 KiB array compiled into the library
 * (MOE_NOALLOC_MAX_PAIRS = 65536 pairs x 256 experts of per-chunk counts and
 * bases); every GPU that loads the library holds it until the process exits.
 *   - Limit: T*k <= MOE_NOALLOC_MAX_PAIRS, else MOE_ERR_UNSUPPORTED is
 *     returned before anything is launched.  E is limited to 256 as in
 *     every entry point (a larger E is MOE_ERR_INVALID_ARG).
 *   - The first call on a device looks up the array's device address on
 *     that device (a runtime query, no allocation); make that first call
 *     before any stream capture is begun.
 *   - All calls share the one array and it keeps the last call's contents;
 *     every call overwrites all of the scratch it reads, so nothing needs to
 *     be cleared between calls.  Calls whose kernels overlap on the GPU (for
 *     example on two streams at once) race on the array: serialise them.
 *   - No cudaMalloc, cudaFree or other allocating routine is ever called.
 */
#define MOE_NOALLOC_MAX_PAIRS 65536
moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_ids, int32_t* expert_offsets,
                                 int32_t* sorted_pair, int32_t* row_of, moe_stream_t stream);

/*
 * Routed experts (grouped SwiGLU GEMMs) and the shared expert.
 * Sarvam blog, Table 1 rows "Routed expert compute" and "Shared expert
 * compute"; section "Scaling multilingual sovereign AI with MoE" (shared
 * expert design).
 *   x              [T][d] (cfg->x_dtype)
 *   topk_w         [T][k] float gates (from moe_route)
 *   expert_offsets [E+1], sorted_pair [T*k] (from moe_permute)
 *   out_perm       [T*k][d] out: row r = topk_w[p] * FFN_e(x[t]) for
 *                  p = sorted_pair[r] = t*k+j routed to expert e
 *   shared_out     [T][d] out: FFN_shared(x[t])
 * out_perm and shared_out are fp32, or bf16 with MOE_FLAG_BF16_EXPERT_OUT
 * (half the bytes; each expert output is then rounded once to bf16, which
 * costs about 1e-3 relative L2 error in y, single elements up to about
 * 2.5e-2 rms(y); all sums stay fp32).
 */
moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x, const float* topk_w,
                            const int32_t* expert_offsets, const int32_t* sorted_pair,
                            const moe_weights_t* weights, void* out_perm, void* shared_out,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Deterministic combine: y[t] = shared_out[t] + sum_{j=0..k-1} out_perm[row_of[t*k+j]],
 * added in slot order j (Sarvam summary section 2.1: shared plus routed
 * experts).  out_perm / shared_out as written by moe_expert_ffn (fp32, or
 * bf16 with MOE_FLAG_BF16_EXPERT_OUT); the sum is taken in fp32.  y is [T][d]
 * in cfg->y_dtype.  Uses no workspace.
 */
moe_status_t moe_combine(const moe_config_t* cfg, const void* out_perm, const int32_t* row_of,
                         const void* shared_out, void* y, moe_stream_t stream);

/*
 * The whole layer: route -> permute -> expert FFN (+ shared) -> combine, with
 * no host synchronisation.  The shared expert needs no routing result, so
 * for decode-sized batches (at most 16 routed rows per expert on average) it
 * runs beside the routing (Sarvam blog, Table 1 row "Shared expert compute"
 * and the paragraph on hiding latency by overlap): the call forks a stream
 * of the library's own (created with the device's first call) off `stream`,
 * runs the shared expert there on at most half the SMs while the routing
 * runs on `stream`, then the routed experts on `stream`, and makes `stream`
 * wait for the fork before the combine.  Larger batches keep the shared
 * expert in the routed launches.  To the caller this is one call on `stream`: the
 * results are ready when `stream` reaches them, and the call records into a
 * CUDA graph captured on `stream` as a fork and a join.  Calls on one device
 * share that second stream, so their shared-expert parts run one after
 * another.  MOE_FLAG_NO_OVERLAP (and the CUDA-core FFN) keep everything on
 * `stream`.  topk_ids_opt / topk_w_opt / expert_offsets_opt, when not NULL,
 * receive copies of the routing results.
 */
moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const float* w_router,
                               const float* expert_bias, const moe_weights_t* weights, void* y,
                               int32_t* topk_ids_opt, float* topk_w_opt,
                               int32_t* expert_offsets_opt, void* ws, size_t ws_bytes,
                               moe_stream_t stream);

/*
 * Number of kernels this library has launched in this process so far
 * (diagnostics: lets a caller count the launches of a timed region).
 */
uint64_t moe_launch_count(void);

/*
 * Reads and clears the current device's status word in one atomic step,
 * ordered after all work already queued on `stream`, then synchronises
 * `stream` and returns what the word held: MOE_OK, MOE_ERR_DEVICE_TIMEOUT,
 * MOE_ERR_DEVICE_BOUNDS, MOE_ERR_DEVICE_NONFINITE (the first fault recorded
 * since the last read), or MOE_ERR_CUDA if the read or the synchronisation
 * failed.  The word is per DEVICE, not per stream: a fault recorded by this
 * library's kernels on any stream of the device is reported to the next
 * reader, whichever stream it passes, and reported once.  Work still running
 * on other streams may record a fault after the read; that fault is kept for
 * the next read.
 */
moe_status_t moe_get_device_status(moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
