// Grouped SwiGLU expert FFN on the tensor cores for NVFP4 expert weights
// (Sarvam blog, Blackwell section: the model quantised to NVFP4; Table 1 rows
// "Routed expert compute" / "Shared expert compute").
//
// NVFP4 element = e2m1 code x E4M3 block scale (16 elements along K) x fp32
// global scale.  e2m1 x E4M3 has at most 2 + 4 significant bits and lies in
// [2^-10, 2688], so it is exact in f16.  Converter warps therefore rebuild the
// weight tile exactly in f16 in shared memory (cvt.rn.f16x2.e2m1x2, then one
// f16x2 multiply by the block scale), and the MMA is tcgen05 kind::f16 with
// f16 activations: each activation row is stored as v / s with s a power of
// two chosen so that the row's largest magnitude lands at 2^14 -- for a bf16
// input this is exact except for elements below amax * 2^-28.  The global
// weight scale and the row scale (times the gate weight in the down
// projection) are applied in the epilogue.
//
// Large token tiles (128 or more) interleave the two gate/up projections in
// one weight tile (IL): its 128 rows are, per 32-row TMEM sub-partition, 16
// gate rows and the 16 up rows of the same features (64 features per tile),
// so one accumulator holds both, two of them fit TMEM at 256 tokens, and an
// epilogue lane pairs gate with up through one exchange with the lane 16
// away.  Smaller tiles keep a gate tile and an up tile of 128 features each
// (two accumulators), which measured faster at decode.
//
// Warp roles (480 threads): warp 0 issues the TMA loads of the activation
// tiles into a ring of their own (up to 8 slots, so that the small decode
// tiles are fetched well ahead of the MMA), warp 1 owns TMEM and issues the
// MMAs, warps 2-5 are the epilogue,
// warps 6-13 convert weights and warp 14 streams the raw weights.  The raw
// stream runs well ahead of the MMA: every 128-element k-block of every
// weight row (64 bytes of packed codes, a TMA box of 128 rows stored with the
// 64-byte swizzle, and 8 bytes of block scales, fetched by the 32 lanes with
// cp.async and signalled through cp.async.mbarrier.arrive) lands in a ring of
// up to 16 slots, so that about 100 KB of weights per SM are in flight -- what
// a decode-sized batch needs to keep HBM busy.  Converter threads turn a slot
// into two 64-element f16 stages (one row, or half a row, per thread),
// fence the async proxy and release the slot.  Every wait is bounded
// (timeout -> status word).
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kF4Threads = 480;
constexpr int kF4Epi = 128;                 // warps 2-5
constexpr int kF4ConvWarps = 8;             // warps 6-13
constexpr int kF4BK = 64;                   // K elements per f16 stage (128 bytes of f16)
constexpr int kF4RK = 128;                  // K elements per raw slot (two f16 stages)
constexpr int kF4BM = 128;                  // weight rows per tile
constexpr uint32_t kF4ATile = kF4BM * 128;  // 16 KB f16 tile
constexpr uint32_t kF4RawCodes = kF4BM * (kF4RK / 2);    // 8 KB of packed codes per weight tile
constexpr uint32_t kF4RawScales = kF4BM * (kF4RK / 16);  // 1 KB of block scales per weight tile
constexpr int kF4MaxStages = 5;
constexpr int kF4MaxB = 8;
constexpr int kF4MaxRaw = 16;
constexpr uint64_t kF4WaitNs = 2000000000ull;
constexpr uint64_t kF4DrainNs = 200000000ull;
constexpr unsigned kF4IdleSleepNs = 128;    // poll interval of the waits that are off the critical path
constexpr int kF4SmemBudget = 214 * 1024;

struct F4Args {
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const float* topk_w;
  const uint8_t* wsc;         // routed block scales [E][rows][K/16]
  const float* wg;            // routed global scales [E]
  const uint8_t* ssc;         // shared block scales
  const float* sg;            // shared global scale (one float)
  const float* b_scale;       // per-row activation scale [P+T]
  __nv_bfloat16* h;           // gemm1 out [(P+T)][fmax]
  void* out_perm;             // gemm2 out [P][d] bf16 or fp32
  void* shared_out;           // gemm2 out [T][d]
  bool out_bf16;
  int T, k, E, P, d, f, fs, fmax;
  int routed_on, shared_on;   // which groups this launch computes (FfnPart)
  int TN, stages, bslots, raw_slots, acc_bufs, tmem_cols;
  unsigned* status;
};

struct __align__(16) F4Ctrl {
  uint64_t aready[kF4MaxStages];   // weight tiles converted (one arrival per converter warp)
  uint64_t empty[kF4MaxStages];    // weight stage free again (MMA commit)
  uint64_t bfull[kF4MaxB];         // activation tile landed (TMA tx count)
  uint64_t bempty[kF4MaxB];        // activation slot free again (MMA commit)
  uint64_t rfull[kF4MaxRaw];       // raw slot landed (TMA tx count + 32 cp.async arrivals)
  uint64_t rempty[kF4MaxRaw];      // raw slot converted (one arrival per converter warp)
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t ep_sync;
  uint32_t tmem_base;
  int abort;
  float coef[2][2 * kF4BM];        // per token row (TN <= 256), by tile parity
  GroupTable gt;
};

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// The barrier receives one arrival once all of this thread's earlier
// cp.async copies have landed (its expected count includes that arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Four e2m1 pairs (one 32-bit word of packed codes, element 2i in the low
// nibble of byte i) times an f16x2 block scale -> four f16x2 words.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t packed, uint32_t scale2, uint32_t (&out)[4]) {
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " .reg .b32 h0, h1, h2, h3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 h0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 h1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 h2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 h3, b3;\n"
      " mul.rn.f16x2 %0, h0, %5;\n"
      " mul.rn.f16x2 %1, h1, %5;\n"
      " mul.rn.f16x2 %2, h2, %5;\n"
      " mul.rn.f16x2 %3, h3, %5;\n"
      "}\n"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(packed), "r"(scale2));
}

// E4M3 block-scale byte -> the same f16 value in both halves.
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(byte | (byte << 8)), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  // D fp32 [4,6) = 1; A, B f16 (format 0); K-major; N >> 3 at 17; M >> 4 at 24
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
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

// Walks this CTA's k-block sequence (tiles blockIdx.x, +gridDim.x, ...; K/64
// k-blocks each) -- the same order for the producers, MMA and converters.
struct KbCursor {
  int i, kb, nkb;
  Tile t;
  bool valid;
};

template <int MODE>
__device__ __forceinline__ int tile_k(const F4Args& a, bool shr) {
  return MODE == 1 ? a.d : (shr ? a.fs : a.f);
}

template <int MODE>
__device__ __forceinline__ void cursor_begin(KbCursor& cu, const GroupTable& gt, int G, int total, const F4Args& a) {
  cu.i = blockIdx.x;
  cu.kb = 0;
  cu.valid = cu.i < total;
  if (cu.valid) {
    cu.t = decode_tile(gt, G, cu.i, a.TN);
    cu.nkb = tile_k<MODE>(a, cu.t.g == a.E) / kF4BK;
  }
}

template <int MODE>
__device__ __forceinline__ void cursor_next(KbCursor& cu, const GroupTable& gt, int G, int total, const F4Args& a) {
  if (!cu.valid) return;
  if (++cu.kb < cu.nkb) return;
  cu.kb = 0;
  cu.i += gridDim.x;
  cu.valid = cu.i < total;
  if (cu.valid) {
    cu.t = decode_tile(gt, G, cu.i, a.TN);
    cu.nkb = tile_k<MODE>(a, cu.t.g == a.E) / kF4BK;
  }
}

// First row (within its tensor map: routed or shared weights) of this tile's
// weights, and its K: gate/up -- the tile's gate rows (a_idx = 0) or its up
// rows (a_idx = 1), 64 of each when interleaved, else 128; down -- its 128 rows.
template <int MODE, bool IL>
__device__ __forceinline__ int weight_row(const F4Args& a, const Tile& t, int a_idx, int* K) {
  const bool shr = t.g == a.E;
  if (MODE == 1) {
    const int width = shr ? a.fs : a.f;
    *K = a.d;
    return (shr ? 0 : t.g * 2 * a.f) + (a_idx ? width : 0) + t.wt * (IL ? kF4BM / 2 : kF4BM);
  }
  *K = shr ? a.fs : a.f;
  return (shr ? 0 : t.g * a.d) + t.wt * kF4BM;
}

template <int MODE, bool IL>
__global__ void __launch_bounds__(kF4Threads, 1)
ffn_fp4_kernel(const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapA,
               const __grid_constant__ CUtensorMap mapAs, F4Args a) {
  constexpr bool GU_IL = IL && MODE == 1;
  constexpr int NA = (MODE == 1 && !GU_IL) ? 2 : 1;   // weight tiles per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = a.TN;                                   // one f16 column per token
  const uint32_t b_bytes = static_cast<uint32_t>(N) * 128;
  constexpr uint32_t stage_bytes = NA * kF4ATile;
  const uint32_t b_slot = (b_bytes + 1023u) & ~1023u;
  constexpr uint32_t raw_slot = NA * (kF4RawCodes + kF4RawScales);   // a multiple of 1024
  uint8_t* bring = smem + a.stages * stage_bytes;       // [bslots][N rows x 128 bytes]
  uint8_t* raw = bring + a.bslots * b_slot;             // [slots][NA codes | NA scales]
  F4Ctrl* c = reinterpret_cast<F4Ctrl*>(raw + a.raw_slots * raw_slot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.E + 1;
  volatile int* abort = &c->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&c->aready[s]), kF4ConvWarps);
      mbar_init(smem_u32(&c->empty[s]), 1);
    }
    for (int s = 0; s < a.bslots; ++s) {
      mbar_init(smem_u32(&c->bfull[s]), 1);
      mbar_init(smem_u32(&c->bempty[s]), 1);
    }
    for (int s = 0; s < a.raw_slots; ++s) {
      mbar_init(smem_u32(&c->rfull[s]), 33);
      mbar_init(smem_u32(&c->rempty[s]), kF4ConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c->tfull[b]), 1);
      mbar_init(smem_u32(&c->tempty[b]), kF4Epi);
    }
    mbar_init(smem_u32(&c->drain), 1);
    mbar_init(smem_u32(&c->ep_sync), kF4Epi);
    c->abort = 0;
    fence_barrier_init();
  }
  pdl_enter();   // from here on the kernel reads what earlier kernels wrote
  if (MODE == 1) {   // 64 features per tile when interleaved, else 128
    constexpr int WT = GU_IL ? kF4BM / 2 : kF4BM;
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN,
                      a.routed_on ? a.f / WT : 0, a.shared_on ? a.fs / WT : 0, a.status);
  } else {
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN,
                      a.routed_on ? a.d / kF4BM : 0, a.shared_on ? a.d / kF4BM : 0, a.status);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int total = c->gt.tile_start[G];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (activations)
      tma_prefetch_desc(&mapB);
      int st = 0;
      uint32_t ph = 0, pending = 0, last_par = 0;
      KbCursor cu;
      cursor_begin<MODE>(cu, c->gt, G, total, a);
      for (; cu.valid && !*abort; cursor_next<MODE>(cu, c->gt, G, total, a)) {
        if (!mbar_wait_sleep(smem_u32(&c->bempty[st]), ph ^ 1u, abort, kF4WaitNs, kF4IdleSleepNs)) break;
        const uint32_t full = smem_u32(&c->bfull[st]);
        mbar_arrive_expect_tx(full, b_bytes);
        tma_load_2d(smem_u32(bring + st * b_slot), &mapB, cu.kb * kF4BK, cu.t.row0, full);
        pending |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (ph << st);
        if (++st == a.bslots) {
          st = 0;
          ph ^= 1u;
        }
      }
      int no_abort = 0;
      for (int s = 0; s < a.bslots; ++s)
        if (pending & (1u << s)) mbar_wait(smem_u32(&c->bfull[s]), (last_par >> s) & 1u, &no_abort, kF4DrainNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_f16(kF4BM, N);
      int st = 0, bs = 0, ab = 0;
      uint32_t ph = 0, bph = 0, aph = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const int nkb = tile_k<MODE>(a, t.g == a.E) / kF4BK;
        if (!mbar_wait(smem_u32(&c->tempty[ab]), aph ^ 1u, abort, kF4WaitNs)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + static_cast<uint32_t>(ab * NA * N);
        const uint32_t d1 = d0 + static_cast<uint32_t>(N);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&c->bfull[bs]), bph, abort, kF4WaitNs) ||
              !mbar_wait(smem_u32(&c->aready[st]), ph, abort, kF4WaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + st * stage_bytes);
          const uint64_t da0 = desc_sw128(sA);
          const uint64_t da1 = desc_sw128(sA + kF4ATile);
          const uint64_t db = desc_sw128(smem_u32(bring + bs * b_slot));
#pragma unroll
          for (int kk = 0; kk < kF4BK / 16; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            mma_f16(d0, da0 + 2 * kk, db + 2 * kk, idesc, accum);
            if (NA == 2) mma_f16(d1, da1 + 2 * kk, db + 2 * kk, idesc, accum);
          }
          mma_commit(smem_u32(&c->empty[st]));
          mma_commit(smem_u32(&c->bempty[bs]));
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
          }
          if (++bs == a.bslots) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&c->tfull[ab]));
        if (++ab == a.acc_bufs) {
          ab = 0;
          aph ^= 1u;
        }
      }
      mma_commit(smem_u32(&c->drain));
      int no_abort = 0;
      mbar_wait(smem_u32(&c->drain), 0, &no_abort, kF4DrainNs);
    }
  } else if (warp < 6) {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int sub = warp & 3;
    const int n = sub * 32 + lane;
    const int et = threadIdx.x - 64;                 // 0..127
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    int ab = 0, cb_par = 0;
    uint32_t aph = 0, eph = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      const Tile t = decode_tile(c->gt, G, i, a.TN);
      const bool shr = t.g == a.E;
      for (int j = et; j < a.TN; j += kF4Epi) {
        float cf = 0.f;
        if (j < t.nrows) {
          const int row = t.row0 + j;
          cf = a.b_scale[row] * (shr ? a.sg[0] : a.wg[t.g]);
          if (MODE == 2 && !shr) {
            const int p = a.sorted_pair[row];
            if (p >= 0 && p < a.P) {
              cf *= a.topk_w[p];
            } else {
              cf = 0.f;
              set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
            }
          }
        }
        c->coef[cb_par][j] = cf;
      }
      mbar_arrive(smem_u32(&c->ep_sync));
      if (!mbar_wait_sleep(smem_u32(&c->ep_sync), eph, abort, kF4WaitNs, kF4IdleSleepNs)) break;
      eph ^= 1u;
      const float* coef = c->coef[cb_par];
      cb_par ^= 1;
      if (!mbar_wait_sleep(smem_u32(&c->tfull[ab]), aph, abort, kF4WaitNs, kF4IdleSleepNs)) break;
      tc_fence_after();
      const int col = t.wt * kF4BM + n;
      if constexpr (MODE == 1 && !GU_IL) {
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * 2 * N);
        for (int c0 = 0; c0 < N; c0 += 16) {       // 16 tokens per chunk
          float gv[16], uv[16];
          tmem_ld16x2(cb + c0, cb + N + c0, gv, uv);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c0 + jj;
            if (j < t.nrows) {
              const float cf = coef[j];
              a.h[static_cast<size_t>(t.row0 + j) * a.fmax + col] =
                  __float2bfloat16_rn(silu(gv[jj] * cf) * (uv[jj] * cf));
            }
          }
        }
      } else if constexpr (MODE == 1) {
        // lanes 0-15 hold gate, lanes 16-31 up, of features fb .. fb+15; per
        // 32-column chunk lane l < 16 finishes tokens c0 .. c0+15 and lane
        // l + 16 tokens c0+16 .. c0+31 after one exchange
        const bool upper = lane >= 16;
        const int fcol = t.wt * (kF4BM / 2) + sub * 16 + (lane & 15);
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * N);
        for (int c0 = 0; c0 < N; c0 += 32) {
          float v0[16], v1[16];
          tmem_ld16x2(cb + c0, cb + c0 + 16, v0, v1);
          float gg[16], uu[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float send = upper ? v0[j] : v1[j];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            gg[j] = upper ? recv : v0[j];
            uu[j] = upper ? v1[j] : recv;
          }
          const int jb = c0 + (upper ? 16 : 0);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = jb + j;
            if (tok < t.nrows) {
              const float cf = coef[tok];
              a.h[static_cast<size_t>(t.row0 + tok) * a.fmax + fcol] =
                  __float2bfloat16_rn(silu(gg[j] * cf) * (uu[j] * cf));
            }
          }
        }
      } else {
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * N);
        void* outp = shr ? a.shared_out : a.out_perm;
        const size_t out0 = static_cast<size_t>(shr ? t.row0 - a.P : t.row0) * a.d + col;
        for (int c0 = 0; c0 < N; c0 += 32) {       // 32 tokens per chunk
          float d0[16], d1[16];
          tmem_ld16x2(cb + c0, cb + c0 + 16, d0, d1);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = c0 + jj;
            if (j < t.nrows) {
              const float v = jj < 16 ? d0[jj] : d1[jj - 16];
              store_out(outp, out0 + static_cast<size_t>(j) * a.d, v * coef[j], a.out_bf16);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&c->tempty[ab]));
      if (++ab == a.acc_bufs) {
        ab = 0;
        aph ^= 1u;
      }
    }
  } else if (warp < 6 + kF4ConvWarps) {
    // -------------------------------------------------- weight converters (warps 6..13)
    // two weight tiles (gate and up, not interleaved): thread -> one row of
    // one tile; one tile: two threads per row, four 16-byte f16 chunks each
    const int ct = threadIdx.x - 192;                 // 0..255
    const int r = ct & (kF4BM - 1);
    const int ai = (NA == 2) ? (ct >> 7) : 0;
    constexpr int kChunks = (NA == 2) ? 8 : 4;        // f16 chunks (8 elements) per thread and stage
    const int c_lo = (NA == 2) ? 0 : 4 * (ct >> 7);
    const int sw = (r >> 1) & 3;                      // 64-byte swizzle of the raw code rows
    KbCursor conv;
    cursor_begin<MODE>(conv, c->gt, G, total, a);
    int st = 0, rs = 0;
    uint32_t ph = 0, rph = 0;
    for (; conv.valid && !*abort; cursor_next<MODE>(conv, c->gt, G, total, a)) {
      const int half = conv.kb & 1;                   // which 64 of the slot's 128 K elements
      if (half == 0 && !mbar_wait(smem_u32(&c->rfull[rs]), rph, abort, kF4WaitNs)) break;
      if (!mbar_wait(smem_u32(&c->empty[st]), ph ^ 1u, abort, kF4WaitNs)) break;
      const uint8_t* slot = raw + rs * raw_slot;
      const uint8_t* codes = slot + ai * kF4RawCodes + r * (kF4RK / 2);
      const uint32_t scw = *reinterpret_cast<const uint32_t*>(slot + NA * kF4RawCodes + ai * kF4RawScales +
                                                              r * (kF4RK / 16) + half * 4);
      // gate/up: raw rows 0-63 are gate features, 64-127 up features; tile row
      // 32 q + i holds gate feature 16 q + i (i < 16), 32 q + 16 + i up
      // feature 16 q + i (r and its tile row agree mod 16, so the swizzle is
      // the same)
      const int rd = GU_IL ? ((r & 63) >> 4) * 32 + (r >> 6) * 16 + (r & 15) : r;
      uint8_t* dst_row = smem + st * stage_bytes + ai * kF4ATile + rd * 128;
#pragma unroll
      for (int q = 0; q < kChunks / 4; ++q) {
        const int lc = 2 * half + (c_lo >> 2) + q;    // logical 16-byte chunk of the 64-byte code row
        const uint4 w4 = *reinterpret_cast<const uint4*>(codes + ((lc ^ sw) << 4));
        const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ch = c_lo + 4 * q + i;            // f16 chunk (8 elements) within the stage row
          const uint32_t s2 = e4m3_to_f16x2_bcast((scw >> (8 * (ch >> 1))) & 0xffu);
          uint32_t hv[4];
          e2m1x8_to_f16(words[i], s2, hv);
          *reinterpret_cast<uint4*>(dst_row + ((ch ^ (r & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->aready[st]));
      if (++st == a.stages) {
        st = 0;
        ph ^= 1u;
      }
      if (half == 1) {
        if (lane == 0) mbar_arrive(smem_u32(&c->rempty[rs]));
        if (++rs == a.raw_slots) {
          rs = 0;
          rph ^= 1u;
        }
      }
    }
  } else {
    // -------------------------------------------------- raw weight stream (warp 14)
    if (lane == 0) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapAs);
    }
    KbCursor cu;
    cursor_begin<MODE>(cu, c->gt, G, total, a);
    int rs = 0;
    uint32_t rph = 0, pending = 0, last_par = 0;
    for (; cu.valid && !*abort; cursor_next<MODE>(cu, c->gt, G, total, a)) {
      if (cu.kb & 1) continue;                        // one slot per two f16 stages
      // warp-uniform decision: either every lane fills the slot or none does
      const bool free_slot = mbar_wait_sleep(smem_u32(&c->rempty[rs]), rph ^ 1u, abort, kF4WaitNs, kF4IdleSleepNs);
      if (!__all_sync(0xffffffffu, free_slot)) break;
      const bool shr = cu.t.g == a.E;
      const uint32_t slot = smem_u32(raw + rs * raw_slot);
      const uint32_t bar = smem_u32(&c->rfull[rs]);
      const int rb = cu.kb >> 1;                      // raw block within the row
      if constexpr (GU_IL) {
        // two boxes of 64 rows (gate, then up) fill the slot's 128 raw rows
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, kF4RawCodes);
          for (int p2 = 0; p2 < 2; ++p2) {
            int K;
            const int row = weight_row<MODE, IL>(a, cu.t, p2, &K);
            tma_load_2d(slot + p2 * (kF4BM / 2) * (kF4RK / 2), shr ? &mapAs : &mapA, rb * (kF4RK / 2), row, bar);
          }
        }
#pragma unroll
        for (int j = 0; j < kF4BM / 32; ++j) {
          const int rr = lane + 32 * j;
          int K;
          const int row = weight_row<MODE, IL>(a, cu.t, rr / (kF4BM / 2), &K) + rr % (kF4BM / 2);
          const uint8_t* sc = (shr ? a.ssc : a.wsc) + static_cast<size_t>(row) * (K / 16) + rb * (kF4RK / 16);
          cp_async8(slot + kF4RawCodes + rr * (kF4RK / 16), sc);
        }
      } else {
        // one box of 128 rows per weight tile
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, NA * kF4RawCodes);
          for (int t2 = 0; t2 < NA; ++t2) {
            int K;
            const int row = weight_row<MODE, IL>(a, cu.t, t2, &K);
            tma_load_2d(slot + t2 * kF4RawCodes, shr ? &mapAs : &mapA, rb * (kF4RK / 2), row, bar);
          }
        }
        for (int t2 = 0; t2 < NA; ++t2) {
          int K;
          const int row = weight_row<MODE, IL>(a, cu.t, t2, &K);
          const uint8_t* sc = (shr ? a.ssc : a.wsc) + static_cast<size_t>(row) * (K / 16) + rb * (kF4RK / 16);
#pragma unroll
          for (int j = 0; j < kF4BM / 32; ++j) {
            const int rr = lane + 32 * j;
            cp_async8(slot + NA * kF4RawCodes + t2 * kF4RawScales + rr * (kF4RK / 16),
                      sc + static_cast<size_t>(rr) * (K / 16));
          }
        }
      }
      cp_async_arrive_noinc(bar);
      pending |= 1u << rs;
      last_par = (last_par & ~(1u << rs)) | (rph << rs);
      if (++rs == a.raw_slots) {
        rs = 0;
        rph ^= 1u;
      }
    }
    int no_abort = 0;
    for (int s = 0; s < a.raw_slots; ++s)
      if (pending & (1u << s)) mbar_wait(smem_u32(&c->rfull[s]), (last_par >> s) & 1u, &no_abort, kF4DrainNs);
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
  if (threadIdx.x == 0 && c->abort) set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
}

// Row scaler: f16 copy of an activation row divided by s = 2^(e-14), where
// amax = m 2^e (m in [0.5,1)), so the row's largest magnitude is m 2^14.
// One warp per row of the (P+T)-row space, rows [row_begin, row_end);
// GATHER_X takes row r < P from x[sorted_pair[r]/k] and row P+t from x[t],
// else row r of H (width f for routed rows, f_s for shared rows).
template <bool GATHER_X, bool IN_REGS>
__global__ void __launch_bounds__(256)
scale16_rows_kernel(const uint16_t* __restrict__ src, const int32_t* __restrict__ sorted_pair, int P, int T, int k,
                    int width_r, int width_s, int src_stride, __half* __restrict__ dst, int dst_stride,
                    float* __restrict__ scale, int row_begin, int row_end, unsigned* status) {
  pdl_enter();
  const int row = row_begin + blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= row_end) return;
  __half* drow = dst + static_cast<size_t>(row) * dst_stride;
  const uint16_t* s;
  int width;
  if (GATHER_X) {
    int t = row - P;
    width = width_r;
    if (row < P) {
      const int p = sorted_pair[row];
      t = (p >= 0 && p < P) ? p / k : -1;
    }
    if (t < 0) {
      if (lane == 0) set_status(status, MOE_ERR_DEVICE_BOUNDS);
      for (int c = lane * 8; c < width; c += 256) *reinterpret_cast<uint4*>(drow + c) = make_uint4(0, 0, 0, 0);
      if (lane == 0) scale[row] = 1.f;
      return;
    }
    s = src + static_cast<size_t>(t) * src_stride;
  } else {
    s = src + static_cast<size_t>(row) * src_stride;
    width = row < P ? width_r : width_s;
  }
  // Rows up to kRegChunks * 256 elements are read once into registers; longer
  // rows take a second pass from L2.
  constexpr int kRegChunks = 16;
  uint4 reg[IN_REGS ? kRegChunks : 1];
  const bool in_regs = IN_REGS && width <= kRegChunks * 256;
  float amax = 0.f;
  auto absmax8 = [&](const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
    }
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < (IN_REGS ? kRegChunks : 1); ++i) {
      const int c = lane * 8 + i * 256;
      reg[i] = (c < width) ? *reinterpret_cast<const uint4*>(s + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < (IN_REGS ? kRegChunks : 1); ++i) absmax8(reg[i]);
  } else {
#pragma unroll 4
    for (int c = lane * 8; c < width; c += 256) absmax8(*reinterpret_cast<const uint4*>(s + c));   // 4 loads in flight
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float sc = 1.f;
  if (amax > 0.f && isfinite(amax)) {
    int e;
    frexpf(amax, &e);
    sc = ldexpf(1.0f, e - 14);
  }
  const float inv = 1.0f / sc;   // exact: a power of two
  auto emit = [&](int c, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xffff0000u) * inv);
      o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(drow + c) = make_uint4(o[0], o[1], o[2], o[3]);
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < (IN_REGS ? kRegChunks : 1); ++i) {
      const int c = lane * 8 + i * 256;
      if (c < width) emit(c, reg[i]);
    }
  } else {
#pragma unroll 4
    for (int c = lane * 8; c < width; c += 256) emit(c, *reinterpret_cast<const uint4*>(s + c));
  }
  if (lane == 0) scale[row] = sc;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn f4_encode_fn() {
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

// f16 matrix [rows][cols] (pitch `pitch` elements), box 64 elements x box_rows, 128-byte swizzle.
bool make_f16_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch, uint32_t box_rows) {
  EncodeTiledFn fn = f4_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kF4BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed e2m1 codes [rows][K/2] bytes: box of 64 bytes (128 elements) x 128
// rows, stored with the 64-byte swizzle.
bool make_code_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
  EncodeTiledFn fn = f4_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {K / 2, rows};
  cuuint64_t strides[1] = {K / 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kF4RK / 2), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct F4Plan {
  size_t xh, sx, h, hh, sh, total;
  int TN;
};

F4Plan f4_plan(const moe_config_t& c) {
  const size_t P = static_cast<size_t>(c.T) * c.top_k, R = P + c.T;
  const size_t fmax = std::max(c.d_ff, c.d_ff_shared);
  F4Plan p;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o += align_up(b, 1024); return at; };
  p.xh = take(2 * R * c.d_model);
  p.sx = take(4 * R);
  p.h = take(2 * R * fmax);
  p.hh = take(2 * R * fmax);
  p.sh = take(4 * R);
  p.total = o;
  const double avg = static_cast<double>(P) / c.n_experts;
  // 256-token tiles once the groups are that large: an f16 MMA of N = 128
  // costs nearly as long as one of N = 256 (about 105 against 135 cycles),
  // and each converted weight row then serves twice the tokens (the gate/up
  // accumulators, 2 x 256 columns, fill TMEM and run single-buffered)
  p.TN = avg <= 12 ? 16 : avg <= 24 ? 32 : avg <= 48 ? 64 : avg <= 192 ? 128 : 256;
  return p;
}

template <int MODE, bool IL>
cudaError_t launch_f4_gemm(const CUtensorMap& mB, const CUtensorMap& mA, const CUtensorMap& mAs, F4Args a,
                           int wtiles_routed, int wtiles_shared, int grid_cap, cudaStream_t stream) {
  constexpr int NA = (MODE == 1 && !IL) ? 2 : 1;   // weight tiles per stage
  const int N = a.TN;
  const int stage_bytes = NA * kF4ATile;
  const int b_slot = static_cast<int>(align_up(static_cast<size_t>(N) * 128, 1024));
  const int raw_slot = NA * (kF4RawCodes + kF4RawScales);
  // three f16 weight stages; activation slots for about 32 KB (at least 3,
  // at most 8); the rest of the budget goes to the raw ring, which hides HBM
  // latency
  // (256-token gate/up tiles: two 32 KB activation slots, so that three raw
  // slots still fit).  Tiles of 128 tokens or more keep five f16 weight
  // stages (converters and MMA then wait on each other less), smaller ones
  // three and more raw slots
  a.stages = N >= 128 ? 5 : 3;
  a.bslots = std::max(3, std::min(kF4MaxB, 32768 / b_slot));
  auto raw_fit = [&] { return (kF4SmemBudget - a.stages * stage_bytes - a.bslots * b_slot) / raw_slot; };
  while (raw_fit() < 3 && a.bslots > 2) --a.bslots;
  a.raw_slots = std::min(kF4MaxRaw, raw_fit());
  if (a.raw_slots < 2) return cudaErrorInvalidConfiguration;
  const int per_acc = NA * N;
  a.acc_bufs = (2 * per_acc <= 512) ? 2 : 1;
  // epilogue loads: 32 columns at c0 (c0 < N, steps of 32), or, two gate/up
  // accumulators, 16 columns at c0 and at N + c0
  const int last = (a.acc_bufs - 1) * per_acc;
  const int reach = (NA == 2) ? last + N + (N + 15) / 16 * 16 : last + (N + 31) / 32 * 32;
  int cols = 32;
  while (cols < reach) cols *= 2;
  if (cols > 512) return cudaErrorInvalidConfiguration;
  a.tmem_cols = cols;
  size_t smem = 1024 + static_cast<size_t>(a.stages) * stage_bytes + static_cast<size_t>(a.bslots) * b_slot +
                static_cast<size_t>(a.raw_slots) * raw_slot + sizeof(F4Ctrl);
  smem = std::max<size_t>(smem, 120 * 1024);   // one CTA per SM: TMEM is never contended
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t err =
      ensure_kernel_attrs(reinterpret_cast<const void*>(ffn_fp4_kernel<MODE, IL>), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const long long tiles_ub = (a.routed_on ? static_cast<long long>(wtiles_routed) * (a.P / a.TN + a.E) : 0) +
                             (a.shared_on ? static_cast<long long>(wtiles_shared) * ((a.T + a.TN - 1) / a.TN) : 0);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(grid_cap, tiles_ub)));
  count_launches(1);
  return launch_pdl(ffn_fp4_kernel<MODE, IL>, grid, kF4Threads, smem, stream, mB, mA, mAs, a);
}

}  // namespace

bool ffn_fp4_supported(const moe_config_t& c) {
  return c.w_dtype == MOE_NVFP4 && c.x_dtype == MOE_BF16 && c.d_ff % 128 == 0 && c.d_ff_shared % 128 == 0 &&
         c.d_model % 128 == 0 && f4_encode_fn() != nullptr;
}

size_t ffn_fp4_ws_bytes(const moe_config_t& c) { return f4_plan(c).total; }

cudaError_t launch_ffn_fp4(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                           const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                           void* ws, unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream) {
  const int T = c.T, k = c.top_k, E = c.n_experts, d = c.d_model, f = c.d_ff, fs = c.d_ff_shared;
  if (T == 0) return cudaSuccess;
  const int P = T * k, R = P + T;
  const int fmax = std::max(f, fs);
  const F4Plan pl = f4_plan(c);
  char* base = static_cast<char*>(ws);
  __half* xh = reinterpret_cast<__half*>(base + pl.xh);
  float* sx = reinterpret_cast<float*>(base + pl.sx);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(base + pl.h);
  __half* hh = reinterpret_cast<__half*>(base + pl.hh);
  float* sh = reinterpret_cast<float*>(base + pl.sh);

  const int r0 = part.row_begin(P), r1 = part.row_end(P, T);
  const int qblocks = ceil_div(r1 - r0, 8);
  const bool regs = R <= 4096;   // see the FP8 path: registers for few rows, two passes for many
  const int cap = std::min(num_sms, part.grid_cap);
  count_launches(1);
  cudaError_t err = launch_pdl(regs ? scale16_rows_kernel<true, true> : scale16_rows_kernel<true, false>, qblocks, 256,
                               0, stream, static_cast<const uint16_t*>(x), sorted_pair, P, T, k, d, d, d, xh, d, sx,
                               r0, r1, status);
  if (err != cudaSuccess) return err;

  F4Args a = {};
  a.offsets = offsets; a.sorted_pair = sorted_pair; a.topk_w = topk_w;
  a.h = h; a.out_perm = out_perm; a.shared_out = shared_out;
  a.out_bf16 = (c.flags & MOE_FLAG_BF16_EXPERT_OUT) != 0;
  a.T = T; a.k = k; a.E = E; a.P = P; a.d = d; a.f = f; a.fs = fs; a.fmax = fmax;
  a.routed_on = part.routed; a.shared_on = part.shared;
  // token tile: from the average routed group, or, for the shared expert
  // alone, from T
  a.TN = part.routed ? pl.TN : (T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128);
  a.status = status;

  CUtensorMap mB, mA, mAs;
  // gemm1: gate / up; token tiles of 128 or more interleave gate and up
  const bool il = a.TN >= 128;
  const uint32_t abox = il ? kF4BM / 2 : kF4BM;
  if (!make_f16_map(&mB, xh, R, d, d, a.TN) ||
      !make_code_map(&mA, w->w13, static_cast<uint64_t>(E) * 2 * f, d, abox) ||
      !make_code_map(&mAs, w->s13, 2 * static_cast<uint64_t>(fs), d, abox))
    return cudaErrorInvalidValue;
  a.wsc = static_cast<const uint8_t*>(w->w13_scale); a.wg = w->w13_gscale;
  a.ssc = static_cast<const uint8_t*>(w->s13_scale); a.sg = w->s13_gscale;
  a.b_scale = sx;
  err = il ? launch_f4_gemm<1, true>(mB, mA, mAs, a, f / abox, fs / abox, cap, stream)
           : launch_f4_gemm<1, false>(mB, mA, mAs, a, f / abox, fs / abox, cap, stream);
  if (err != cudaSuccess) return err;

  count_launches(1);
  err = launch_pdl(regs ? scale16_rows_kernel<false, true> : scale16_rows_kernel<false, false>, qblocks, 256, 0,
                   stream, reinterpret_cast<const uint16_t*>(h), static_cast<const int32_t*>(nullptr), P, T, k, f, fs,
                   fmax, hh, fmax, sh, r0, r1, status);
  if (err != cudaSuccess) return err;

  // gemm2: down projection, gate weight, outputs
  if (!make_f16_map(&mB, hh, R, fmax, fmax, a.TN) ||
      !make_code_map(&mA, w->w2, static_cast<uint64_t>(E) * d, f, kF4BM) ||
      !make_code_map(&mAs, w->s2, static_cast<uint64_t>(d), fs, kF4BM))
    return cudaErrorInvalidValue;
  a.wsc = static_cast<const uint8_t*>(w->w2_scale); a.wg = w->w2_gscale;
  a.ssc = static_cast<const uint8_t*>(w->s2_scale); a.sg = w->s2_gscale;
  a.b_scale = sh;
  return launch_f4_gemm<2, false>(mB, mA, mAs, a, d / kF4BM, d / kF4BM, cap, stream);
}

}  // namespace moe
