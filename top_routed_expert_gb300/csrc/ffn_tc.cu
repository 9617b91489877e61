// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA-fed shared memory) for FP8 E4M3 expert weights.
// Sarvam blog, Table 1 rows "Routed expert compute" / "Shared expert
// compute"; Sarvam summary section 2.1 (FP8 expert weights, one byte per
// parameter); H100 baseline section (grouped GEMM kernels over the experts).
//
// Design (GB300-first, not the pages' H100 kernels):
//  * swap-AB: the weight rows fill the MMA's M = 128 lanes (A operand, read
//    straight from HBM by TMA as raw E4M3 codes), the routed tokens of a
//    group are the N columns (B operand).  Decode groups hold ~3 tokens, so
//    the tile stays full and the kernel streams weights at HBM speed.
//  * activations enter the FP8 MMA as two E4M3 terms with a per-row power-
//    of-two scale s:  v = s * (hi + lo/16).  For a bf16 input this split is
//    exact apart from elements below 2^-6 s (absolute error < 2^-14 s), so
//    the product equals the bf16-activation product; hi and lo are adjacent
//    N columns and the epilogue adds them.  Per-channel weight scales and the
//    row scale are applied in the epilogue.
//  * MOE_FLAG_ACT_E4M3 (opt-in, lossy): one E4M3 term per activation with
//    the same per-row power-of-two scale, so N is the token count and the MMAs
//    issue the layer's FLOPs once (TERMS = 1 below).
//  * gemm1 (gate+up, two accumulators) -> silu(g)*u -> H (bf16);
//    H is re-split into two E4M3 terms per row; gemm2 (down) applies the gate
//    weight and writes out_perm (routed) / shared_out (shared expert).
//  * the shared expert is group E of the same launches (rows = all tokens).
//  * persistent CTAs walk a device-built tile list (group, weight tile,
//    token tile) -- no host read-back of the expert counts.
//  * warp roles: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
//    warps 2-9 = epilogue (two per TMEM sub-partition).
//  * every mbarrier wait is bounded; on expiry the kernel records
//    MOE_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and
//    returns.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace moe {

using namespace ptx;

constexpr int kTcThreads = 320;          // producer, MMA, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kBK = 128;                // K bytes (= FP8 elements) per pipeline stage
constexpr int kBM = 128;                // weight rows per tile = MMA M
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: no legitimate wait comes close
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s
constexpr uint32_t kABytes = kBM * kBK;            // 16 KB per weight tile

// Tuning knobs (compile-time): largest token tile of the gate/up and of the
// down GEMM, and the L2 promotion of the TMA loads.
#ifndef MOE_TC_TN1_CAP
#define MOE_TC_TN1_CAP 64
#endif
#ifndef MOE_TC_TN2_CAP
#define MOE_TC_TN2_CAP 128
#endif
#ifndef MOE_TC_L2_PROMOTION
#define MOE_TC_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif

struct TcArgs {
  const int32_t* offsets;      // [E+1]
  const int32_t* sorted_pair;  // [P]
  const float* topk_w;         // [P]
  const float* a_scale;        // routed per-output-row weight scales: w13_scale [E][2f] | w2_scale [E][d]
  const float* as_scale;       // shared: s13_scale [2fs] | s2_scale [d]
  const float* b_scale;        // per-row activation scale [P+T]
  __nv_bfloat16* h;            // gemm1 out: H [(P+T)][fmax]
  void* out_perm;              // gemm2 out: [P][d] bf16 or fp32
  void* shared_out;            // gemm2 out: [T][d]
  bool out_bf16;
  int T, k, E, P, d, f, fs, fmax;
  int routed_on, shared_on;    // which groups this launch computes (FfnPart)
  int TN;                      // token rows per tile; MMA N = TERMS*TN
  int stages, acc_bufs, tmem_cols;
  uint64_t wait_ns;            // limit of every bounded wait
  int inject_drop;             // test hook: CTA 0 withholds its first "accumulator ready"
  unsigned* status;
};

struct __align__(16) TcCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t ep_sync;            // the eight epilogue warps meet here once per tile
  uint32_t tmem_base;
  int abort;
  float coef[2][2 * kBM];      // per-row epilogue coefficient (TN <= 256), double-buffered by tile parity
  GroupTable gt;
};

// TERMS = activation terms per token row: 2 (exact split, default) or 1
// (MOE_FLAG_ACT_E4M3).  The B operand holds TERMS adjacent rows per token.
template <int MODE, int TERMS>
__global__ void __launch_bounds__(kTcThreads, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapAS,
              const __grid_constant__ CUtensorMap mapB, TcArgs a) {
  constexpr int NA = (MODE == 1) ? 2 : 1;   // weight tiles per stage (gate + up, or down)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = TERMS * a.TN;
  const uint32_t b_bytes = static_cast<uint32_t>(N) * kBK;
  const uint32_t stage_bytes = NA * kABytes + ((b_bytes + 1023u) & ~1023u);
  TcCtrl* c = reinterpret_cast<TcCtrl*>(smem + a.stages * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.E + 1;
  volatile int* abort = &c->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&c->full[s]), 1);
      mbar_init(smem_u32(&c->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c->tfull[b]), 1);
      mbar_init(smem_u32(&c->tempty[b]), kEpiThreads);
    }
    mbar_init(smem_u32(&c->drain), 1);
    mbar_init(smem_u32(&c->ep_sync), kEpiThreads);
    c->abort = 0;
    fence_barrier_init();
  }
  // everything above overlaps the previous kernel's tail; from here on the
  // kernel reads what earlier kernels wrote
  pdl_enter();
  // device-side tile list: group g = expert (g < E) or the shared expert (g = E)
  if (MODE == 1)
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN, a.routed_on ? a.f / kBM : 0,
                      a.shared_on ? a.fs / kBM : 0, a.status);
  else
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN, a.routed_on ? a.d / kBM : 0,
                      a.shared_on ? a.d / kBM : 0, a.status);
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), a.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapAS);
    tma_prefetch_desc(&mapB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int total = c->gt.tile_start[G];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int st = 0;
      uint32_t ph = 0, pending = 0, last_par = 0;
      for (int i = blockIdx.x; i < total && !*abort; i += gridDim.x) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const bool shr = t.g == a.E;
        const CUtensorMap* mA = shr ? &mapAS : &mapA;
        int arow0, arow1 = 0, K;
        if (MODE == 1) {
          const int width = shr ? a.fs : a.f;
          const int base = shr ? 0 : t.g * 2 * a.f;
          arow0 = base + t.wt * kBM;
          arow1 = base + width + t.wt * kBM;
          K = a.d;
        } else {
          arow0 = (shr ? 0 : t.g * a.d) + t.wt * kBM;
          K = shr ? a.fs : a.f;
        }
        const int brow = TERMS * t.row0;
        for (int kb = 0; kb < K / kBK; ++kb) {
          if (!mbar_wait(smem_u32(&c->empty[st]), ph ^ 1u, abort, a.wait_ns)) break;
          const uint32_t full = smem_u32(&c->full[st]);
          mbar_arrive_expect_tx(full, NA * kABytes + b_bytes);
          const uint32_t sA = smem_u32(smem + st * stage_bytes);
          tma_load_2d(sA, mA, kb * kBK, arow0, full);
          if (MODE == 1) tma_load_2d(sA + kABytes, mA, kb * kBK, arow1, full);
          tma_load_2d(sA + NA * kABytes, &mapB, kb * kBK, brow, full);
          pending |= 1u << st;
          last_par = (last_par & ~(1u << st)) | (ph << st);
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // every issued copy must land before the CTA may exit
      int no_abort = 0;
      for (int s = 0; s < a.stages; ++s)
        if (pending & (1u << s)) mbar_wait(smem_u32(&c->full[s]), (last_par >> s) & 1u, &no_abort, kDrainLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_f8_e4m3(kBM, N);
      int st = 0, ab = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const bool shr = t.g == a.E;
        const int K = (MODE == 1) ? a.d : (shr ? a.fs : a.f);
        if (!mbar_wait(smem_u32(&c->tempty[ab]), aph ^ 1u, abort, a.wait_ns)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + static_cast<uint32_t>(ab * NA * N);
        const uint32_t d1 = d0 + static_cast<uint32_t>(N);
        for (int kb = 0; kb < K / kBK; ++kb) {
          if (!mbar_wait(smem_u32(&c->full[st]), ph, abort, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + st * stage_bytes);
          const uint64_t da0 = desc_sw128(sA);
          const uint64_t da1 = desc_sw128(sA + kABytes);
          const uint64_t db = desc_sw128(sA + NA * kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            mma_f8f6f4(d0, da0 + 2 * kk, db + 2 * kk, idesc, accum);
            if (MODE == 1) mma_f8f6f4(d1, da1 + 2 * kk, db + 2 * kk, idesc, accum);
          }
          mma_commit(smem_u32(&c->empty[st]));
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (!(a.inject_drop && blockIdx.x == 0 && i == static_cast<int>(blockIdx.x)))
          mma_commit(smem_u32(&c->tfull[ab]));
        if (++ab == a.acc_bufs) {
          ab = 0;
          aph ^= 1u;
        }
      }
      // no MMA may still be running when TMEM is released
      mma_commit(smem_u32(&c->drain));
      int no_abort = 0;
      mbar_wait(smem_u32(&c->drain), 0, &no_abort, kDrainLimitNs);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..9)
    // Two warps per TMEM sub-partition (warp % 4 selects the 32 lanes a warp
    // may read); the pair of warps splits the tile's column chunks.
    const int sub = warp & 3;
    const int half = (warp - 2) >> 2;               // 0 or 1
    const int n = sub * 32 + lane;                  // weight row within the tile
    const int et = threadIdx.x - 64;                // 0..255 across the epilogue warps
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    int ab = 0, cb_par = 0;
    uint32_t aph = 0, eph = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      const Tile t = decode_tile(c->gt, G, i, a.TN);
      const bool shr = t.g == a.E;
      // Per-row coefficients of this tile, loaded while the MMAs run: the
      // row's activation scale, times the gate weight of its (token, slot)
      // pair in the down projection.
      if (et < a.TN) {
        float cf = 0.f;
        if (et < t.nrows) {
          const int row = t.row0 + et;
          cf = a.b_scale[row];
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
        c->coef[cb_par][et] = cf;
      }
      // all coefficients written (bounded wait: a warp that gave up cannot
      // leave the others blocked)
      mbar_arrive(smem_u32(&c->ep_sync));
      if (!mbar_wait(smem_u32(&c->ep_sync), eph, abort, a.wait_ns)) break;
      eph ^= 1u;
      const float* coef = c->coef[cb_par];
      cb_par ^= 1;
      if (!mbar_wait(smem_u32(&c->tfull[ab]), aph, abort, a.wait_ns)) break;
      tc_fence_after();
      const int col = t.wt * kBM + n;
      if (MODE == 1) {
        const int width = shr ? a.fs : a.f;
        const float sg = shr ? a.as_scale[col] : a.a_scale[static_cast<size_t>(t.g) * 2 * a.f + col];
        const float su = shr ? a.as_scale[width + col] : a.a_scale[static_cast<size_t>(t.g) * 2 * a.f + a.f + col];
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * 2 * N);
        // chunks of 32 columns = 32 / TERMS token rows; N is a multiple of
        // 16 and a 32-wide load past N stays inside the allocation
        constexpr int TPC = 32 / TERMS;
        for (int c0 = 32 * half; c0 < N; c0 += 64) {
          float gv[32], uv[32], cf[TPC];
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) cf[jj] = coef[c0 / TERMS + jj];
          tmem_ld32x2(cb + c0, cb + N + c0, gv, uv);
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) {
            const int j = c0 / TERMS + jj;
            if (j < t.nrows) {
              const int row = t.row0 + j;
              const float gd = TERMS == 2 ? gv[2 * jj] + gv[2 * jj + 1] * 0.0625f : gv[jj];
              const float ud = TERMS == 2 ? uv[2 * jj] + uv[2 * jj + 1] * 0.0625f : uv[jj];
              const float g = gd * cf[jj] * sg;
              const float u = ud * cf[jj] * su;
              a.h[static_cast<size_t>(row) * a.fmax + col] = __float2bfloat16_rn(silu(g) * u);
            }
          }
        }
      } else {
        const float sw = shr ? a.as_scale[col] : a.a_scale[static_cast<size_t>(t.g) * a.d + col];
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * N);
        void* outp = shr ? a.shared_out : a.out_perm;
        const size_t out0 = static_cast<size_t>(shr ? t.row0 - a.P : t.row0) * a.d + col;
        // chunks of 64 columns = 64 / TERMS token rows
        constexpr int TPC = 64 / TERMS;
        for (int c0 = 64 * half; c0 < N; c0 += 128) {
          float d0[32], d1[32];
          float cf[TERMS == 2 ? TPC : 1];   // two terms: this chunk's coefficients in registers
          if (TERMS == 2) {
#pragma unroll
            for (int jj = 0; jj < TPC; ++jj) cf[jj] = coef[c0 / TERMS + jj];
          }
          tmem_ld32x2(cb + c0, cb + c0 + 32, d0, d1);
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) {
            const int j = c0 / TERMS + jj;
            if (j < t.nrows) {
              float dsum;
              if (TERMS == 2) {
                const float* dv = jj < 16 ? d0 : d1;
                const int q = 2 * (jj & 15);
                dsum = dv[q] + dv[q + 1] * 0.0625f;
              } else {
                dsum = jj < 32 ? d0[jj] : d1[jj - 32];
              }
              const float cfj = TERMS == 2 ? cf[TERMS == 2 ? jj : 0] : coef[j];
              store_out(outp, out0 + static_cast<size_t>(j) * a.d, dsum * cfj * sw, a.out_bf16);
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
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
  if (threadIdx.x == 0 && c->abort) set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Row quantiser: v = s * (hi + lo/16), s = the smallest power of two with
// amax <= 448 s (1 for an all-zero row), hi and lo E4M3 (round to nearest
// even, saturating).  With two_terms false only hi is written: the single-
// term 8-bit activation of MOE_FLAG_ACT_E4M3.  One warp per row of the
// (P+T)-row activation space, rows [row_begin, row_end).  GATHER_X: row
// r < P takes x[sorted_pair[r]/k], row P+t takes x[t] (width d); otherwise
// row r of H (width f for routed rows, f_s for shared rows).  Output
// q[2r] = hi codes, q[2r+1] = lo codes.
template <bool GATHER_X, bool IN_REGS>
__global__ void __launch_bounds__(256)
quant2_rows_kernel(const uint16_t* __restrict__ src, const int32_t* __restrict__ sorted_pair, int P, int T, int k,
                   int width_r, int width_s, int src_stride, uint8_t* __restrict__ q, int q_stride,
                   float* __restrict__ scale, bool two_terms, int row_begin, int row_end, unsigned* status) {
  pdl_enter();
  const int row = row_begin + blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= row_end) return;
  const uint16_t* s;
  int width;
  uint8_t* qh = q + static_cast<size_t>(2 * row) * q_stride;
  uint8_t* ql = qh + q_stride;
  if (GATHER_X) {
    int t = row - P;
    width = width_r;
    if (row < P) {
      const int p = sorted_pair[row];
      t = (p >= 0 && p < P) ? p / k : -1;
    }
    if (t < 0) {
      if (lane == 0) set_status(status, MOE_ERR_DEVICE_BOUNDS);
      for (int c = lane * 8; c < width; c += 256) {
        *reinterpret_cast<uint2*>(qh + c) = make_uint2(0, 0);
        if (two_terms) *reinterpret_cast<uint2*>(ql + c) = make_uint2(0, 0);
      }
      if (lane == 0) scale[row] = 1.f;
      return;
    }
    s = src + static_cast<size_t>(t) * src_stride;
  } else {
    s = src + static_cast<size_t>(row) * src_stride;
    width = row < P ? width_r : width_s;
  }
  // Rows up to kRegChunks * 256 elements are read once into registers (all
  // loads in flight together); longer rows take a second pass from L2.
  constexpr int kRegChunks = 16;
  uint4 reg[IN_REGS ? kRegChunks : 1];
  const bool in_regs = IN_REGS && width <= kRegChunks * 256;
  float amax = 0.f;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < (IN_REGS ? kRegChunks : 1); ++i) {
      const int c = lane * 8 + i * 256;
      reg[i] = (c < width) ? *reinterpret_cast<const uint4*>(s + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < (IN_REGS ? kRegChunks : 1); ++i) {
      const uint32_t w[4] = {reg[i].x, reg[i].y, reg[i].z, reg[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
      }
    }
  } else {
#pragma unroll 4
    for (int c = lane * 8; c < width; c += 256) {   // four loads in flight per lane
      const uint4 v = *reinterpret_cast<const uint4*>(s + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  // amax = m 2^e with m in [0.5, 1): 448 * 2^(e-9) = 0.875 * 2^e is the
  // smallest candidate (448 * 2^(e-10) < 2^(e-1) <= amax); both comparisons
  // are exact in fp32
  float sc = 1.f;
  if (amax > 0.f && isfinite(amax)) {
    int e;
    frexpf(amax, &e);
    sc = ldexpf(1.0f, max(e - 9, -126));
    if (amax > 448.0f * sc) sc *= 2.0f;
  }
  const float inv = 1.0f / sc;   // exact: sc is a power of two
  auto emit = [&](int c, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t hi[2] = {0, 0}, lo[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f2 = make_float2(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xffff0000u) * inv);
      const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(f2, __NV_SATFINITE, __NV_E4M3);
      const __half2_raw back = __nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3);
      const float2 bf = __half22float2(__half2(back));
      const float2 r2 = make_float2((f2.x - bf.x) * 16.0f, (f2.y - bf.y) * 16.0f);
      const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(r2, __NV_SATFINITE, __NV_E4M3);
      hi[i >> 1] |= static_cast<uint32_t>(h2) << (16 * (i & 1));
      lo[i >> 1] |= static_cast<uint32_t>(l2) << (16 * (i & 1));
    }
    *reinterpret_cast<uint2*>(qh + c) = make_uint2(hi[0], hi[1]);
    if (two_terms) *reinterpret_cast<uint2*>(ql + c) = make_uint2(lo[0], lo[1]);
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

// ---------------------------------------------------------------------------
// Host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// 2-D byte matrix [rows][cols] (row pitch = pitch bytes, default cols), box 128
// bytes x box_rows, 128-byte swizzle; rows past the end read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint64_t pitch = 0) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch ? pitch : cols};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, MOE_TC_L2_PROMOTION,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
  size_t xq, sx, h, hq, sh, total;
  int TN;
};

TcPlan plan(const moe_config_t& c) {
  const size_t P = static_cast<size_t>(c.T) * c.top_k, R = P + c.T;
  const size_t fmax = std::max(c.d_ff, c.d_ff_shared);
  TcPlan p;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o += align_up(b, 1024); return at; };
  p.xq = take(2 * R * c.d_model);
  p.sx = take(4 * R);
  p.h = take(2 * R * fmax);
  p.hq = take(2 * R * fmax);
  p.sh = take(4 * R);
  p.total = o;
  const double avg = static_cast<double>(P) / c.n_experts;
  p.TN = avg <= 6 ? 8 : avg <= 12 ? 16 : avg <= 24 ? 32 : avg <= 48 ? 64 : 128;
  return p;
}

template <int MODE, int TERMS>
cudaError_t launch_gemm(const CUtensorMap& mA, const CUtensorMap& mAS, const CUtensorMap& mB, TcArgs a,
                        int wtiles_routed, int wtiles_shared, int grid_cap, cudaStream_t stream) {
  constexpr int NA = (MODE == 1) ? 2 : 1;
  const int N = TERMS * a.TN;
  const int stage_bytes = NA * kABytes + align_up(static_cast<size_t>(N) * kBK, 1024);
  // as many stages as fit next to the control block in 227 KB
  a.stages = std::min(kMaxStages, static_cast<int>((227 * 1024 - 1024 - sizeof(TcCtrl)) / stage_bytes));
  const int per_acc = NA * N;
  a.acc_bufs = (2 * per_acc <= 512) ? 2 : 1;
  // The epilogue reads 32 columns per load (gemm1: gate and up from column c0
  // and N + c0, c0 < N in steps of 32; gemm2: 64 from c0, c0 < N in steps of
  // 64), so the allocation covers the last buffer plus that overhang.
  const int last = (a.acc_bufs - 1) * per_acc;
  const int reach = (MODE == 1) ? last + N + (N + 31) / 32 * 32 : last + (N + 63) / 64 * 64;
  int cols = 32;
  while (cols < reach) cols *= 2;
  if (cols > 512) return cudaErrorInvalidConfiguration;
  a.tmem_cols = cols;
  size_t smem = 1024 + static_cast<size_t>(a.stages) * stage_bytes + sizeof(TcCtrl);
  smem = std::max<size_t>(smem, 120 * 1024);   // one CTA per SM: TMEM is never contended
  cudaError_t err =
      ensure_kernel_attrs(reinterpret_cast<const void*>(ffn_tc_kernel<MODE, TERMS>), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const long long tiles_ub = (a.routed_on ? static_cast<long long>(wtiles_routed) * (a.P / a.TN + a.E) : 0) +
                             (a.shared_on ? static_cast<long long>(wtiles_shared) * ((a.T + a.TN - 1) / a.TN) : 0);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(grid_cap, tiles_ub)));
  count_launches(1);
  return launch_pdl(ffn_tc_kernel<MODE, TERMS>, grid, kTcThreads, smem, stream, mA, mAS, mB, a);
}

}  // namespace

bool ffn_tc_supported(const moe_config_t& c) {
  return c.w_dtype == MOE_E4M3 && c.x_dtype == MOE_BF16 && c.d_ff % 128 == 0 && c.d_ff_shared % 128 == 0 &&
         c.d_model % 128 == 0 && encode_fn() != nullptr;
}

size_t ffn_tc_ws_bytes(const moe_config_t& c) { return plan(c).total; }

cudaError_t launch_ffn_tc(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                          const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                          void* ws, unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream) {
  const int T = c.T, k = c.top_k, E = c.n_experts, d = c.d_model, f = c.d_ff, fs = c.d_ff_shared;
  if (T == 0) return cudaSuccess;
  const int P = T * k, R = P + T;
  const int fmax = std::max(f, fs);
  const TcPlan pl = plan(c);
  // activation terms per row: 2 (exact), or 1 with MOE_FLAG_ACT_E4M3 (the
  // MMA's N is then the token count, at least 16)
  const bool one_term = (c.flags & MOE_FLAG_ACT_E4M3) != 0;
  // token tile: from the average routed group, or, for the shared expert
  // alone, from T (one group of T rows: the fewest tiles, so each weight tile
  // is read as few times as possible)
  const int tn = part.routed ? pl.TN : (T <= 8 ? 8 : T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128);
  const int tn1 = one_term ? std::max(16, std::min(tn, 128)) : std::min(tn, MOE_TC_TN1_CAP);
  // one term, down GEMM: 256-token tiles once groups are that large (N = 256
  // halves the operand bytes per MAC of a 128 x 128 tile; K = f is short, so
  // the feed, not the MMA, bounds the smaller tile)
  const bool big = part.routed ? static_cast<double>(P) / E > 96 : T > 96;
  const int tn2 = one_term ? (big ? 256 : std::max(16, std::min(tn, 128))) : std::min(tn, MOE_TC_TN2_CAP);
  char* base = static_cast<char*>(ws);
  uint8_t* xq = reinterpret_cast<uint8_t*>(base + pl.xq);
  float* sx = reinterpret_cast<float*>(base + pl.sx);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(base + pl.h);
  uint8_t* hq = reinterpret_cast<uint8_t*>(base + pl.hq);
  float* sh = reinterpret_cast<float*>(base + pl.sh);

  // few rows (decode): keep each row in registers (one read, all loads in
  // flight); many rows: a lean two-pass kernel keeps more warps resident
  const int r0 = part.row_begin(P), r1 = part.row_end(P, T);
  const int qblocks = ceil_div(r1 - r0, 8);
  const bool regs = R <= 4096;
  const int cap = std::min(num_sms, part.grid_cap);
  count_launches(1);
  cudaError_t err = launch_pdl(regs ? quant2_rows_kernel<true, true> : quant2_rows_kernel<true, false>, qblocks, 256, 0,
                               stream, static_cast<const uint16_t*>(x), sorted_pair, P, T, k, d, d, d, xq, d, sx,
                               !one_term, r0, r1, status);
  if (err != cudaSuccess) return err;

  CUtensorMap mA, mAS, mB;
  TcArgs a = {};
  a.offsets = offsets; a.sorted_pair = sorted_pair; a.topk_w = topk_w;
  a.h = h; a.out_perm = out_perm; a.shared_out = shared_out;
  a.out_bf16 = (c.flags & MOE_FLAG_BF16_EXPERT_OUT) != 0;
  a.T = T; a.k = k; a.E = E; a.P = P; a.d = d; a.f = f; a.fs = fs; a.fmax = fmax;
  a.routed_on = part.routed; a.shared_on = part.shared;
  a.TN = pl.TN; a.status = status;
  const bool inject = (c.flags & MOE_FLAG_INJECT_TIMEOUT) != 0;
  a.wait_ns = inject ? 20000000ull : kWaitLimitNs;
  a.inject_drop = inject ? 1 : 0;

  // gemm1: gate/up (B: both term rows of each activation row, or the hi rows only)
  const bool mb_ok = one_term ? make_map(&mB, xq, static_cast<uint64_t>(R), d, tn1, 2 * static_cast<uint64_t>(d))
                              : make_map(&mB, xq, static_cast<uint64_t>(2) * R, d, 2 * tn1);
  if (!make_map(&mA, w->w13, static_cast<uint64_t>(E) * 2 * f, d, kBM) ||
      !make_map(&mAS, w->s13, static_cast<uint64_t>(2) * fs, d, kBM) || !mb_ok)
    return cudaErrorInvalidValue;
  a.a_scale = static_cast<const float*>(w->w13_scale);
  a.as_scale = static_cast<const float*>(w->s13_scale);
  a.b_scale = sx;
  a.TN = tn1;   // two buffers of (gate, up) x TERMS*TN columns fit TMEM at TERMS*TN <= 128
  err = one_term ? launch_gemm<1, 1>(mA, mAS, mB, a, f / kBM, fs / kBM, cap, stream)
                 : launch_gemm<1, 2>(mA, mAS, mB, a, f / kBM, fs / kBM, cap, stream);
  if (err != cudaSuccess) return err;

  count_launches(1);
  err = launch_pdl(regs ? quant2_rows_kernel<false, true> : quant2_rows_kernel<false, false>, qblocks, 256, 0, stream,
                   reinterpret_cast<const uint16_t*>(h), static_cast<const int32_t*>(nullptr), P, T, k, f, fs, fmax,
                   hq, fmax, sh, !one_term, r0, r1, status);
  if (err != cudaSuccess) return err;

  // gemm2: down projection, gate weight, outputs
  const bool mb2_ok = one_term
                          ? make_map(&mB, hq, static_cast<uint64_t>(R), fmax, tn2, 2 * static_cast<uint64_t>(fmax))
                          : make_map(&mB, hq, static_cast<uint64_t>(2) * R, fmax, 2 * tn2);
  if (!make_map(&mA, w->w2, static_cast<uint64_t>(E) * d, f, kBM) ||
      !make_map(&mAS, w->s2, static_cast<uint64_t>(d), fs, kBM) || !mb2_ok)
    return cudaErrorInvalidValue;
  a.a_scale = static_cast<const float*>(w->w2_scale);
  a.as_scale = static_cast<const float*>(w->s2_scale);
  a.b_scale = sh;
  a.TN = tn2;
  return one_term ? launch_gemm<2, 1>(mA, mAS, mB, a, d / kBM, d / kBM, cap, stream)
                  : launch_gemm<2, 2>(mA, mAS, mB, a, d / kBM, d / kBM, cap, stream);
}

}  // namespace moe
