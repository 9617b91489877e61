// Grouped SwiGLU expert FFN for NVFP4 expert weights on the block-scaled
// FP4 tensor-core MMA (tcgen05.mma kind::mxf4nvf4, 16-element blocks with
// E4M3 block scales).  Sarvam blog, Blackwell section (NVFP4 weights via
// Model Optimizer; FP4 compute); Table 1 rows "Routed expert compute" /
// "Shared expert compute".
//
// The stored weights go from HBM to the tensor core untouched: TMA lands the
// packed e2m1 codes (128-byte swizzle) and the E4M3 block scales in shared
// memory, four scale-writer warps move the block scales into tensor memory
// and the MMA consumes both.  Nothing converts weight elements, so shared
// memory carries half a byte per weight element instead of the four bytes of
// an f16 rebuild -- what lets the decode batch stream weights at HBM speed.
//
// The MMA needs FP4 on both sides.  Each activation row v (x, or H after
// SwiGLU) is therefore written as a sum of TERMS NVFP4 rows, v = sum_t a_t,
// each a_t = g_t * s_tb * e2m1 (a power-of-two row scale g_t, an E4M3 scale
// s_tb per 16 elements, e2m1 codes), found greedily on the residual
// r_0 = v, r_{t+1} = r_t - a_t.  Each term takes about a tenth of the
// remaining error: four terms leave about 5e-5 relative L2 of the row, well
// under the bf16 rounding of H (about 1e-3), so the default layer keeps the
// exact-activation contract.  With MOE_FLAG_ACT_NVFP4 a single term is kept
// (W4A4, lossy).  The terms of one token are TERMS adjacent B rows, i.e.
// adjacent MMA N columns; the epilogue adds them with their row scales.
//
// Tensor-memory layout of the block scales, as the MMA reads them (one
// K = 64 step reads 4 bytes of scales per operand row; byte j scales the j-th
// 16-element block of the step): the scales of A row m are taken from lane
// m at column (A-scale address) + m / 32; those of B row n from lane n % 32
// of the quadrant of the A row being computed, at column (B-scale address)
// + n / 32.  So B's scales are written into all four quadrants, and each K
// step kk gets its own 4-column group: A at base + 16 a + 4 kk (weight tile
// a), B at base + 32 + 4 kk.
//
// Warp roles (704 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 2-17 epilogue (four per TMEM quadrant, splitting the column
// chunks: with fewer, a large batch's epilogue -- one term per token, an
// output store per element -- kept the MMA waiting for free accumulators a
// third of the time), warps 18-21 block-scale writers (one per quadrant).  Persistent CTAs walk the device-built tile
// list of tc_sched.cuh; every wait is bounded (timeout -> status word).
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kN4EpiWarps = 16;               // warps 2-17
constexpr int kN4Epi = 32 * kN4EpiWarps;
constexpr int kN4Threads = 64 + kN4Epi + 128;
constexpr int kN4BK = 128;                    // bytes of packed codes per row and stage (256 K elements)
constexpr int kN4BM = 128;                    // weight rows per tile = MMA M
constexpr uint32_t kN4ACodes = kN4BM * kN4BK;     // 16 KB of codes per weight tile and stage
constexpr uint32_t kN4Sf = 128 * 16;              // 2 KB of block scales per operand and stage (128 rows)
constexpr int kN4MaxStages = 8;
constexpr int kN4SfCols = 48;                 // TMEM columns of scales per stage: SFA 2 x 16, SFB 16
constexpr uint64_t kN4WaitNs = 2000000000ull;
constexpr uint64_t kN4DrainNs = 200000000ull;
constexpr int kN4SmemBudget = 220 * 1024;
constexpr int kN4MaxWidth = 4096;             // widest activation row the term quantiser holds in registers

struct N4Args {
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const float* topk_w;
  const float* wg;             // routed global weight scales [E]
  const float* sg;             // shared global weight scale (one float)
  const float* b_scale;        // per activation term row scale g [(P+T) * TERMS]
  __nv_bfloat16* h;            // gemm1 out: H [(P+T)][fmax]
  void* out_perm;              // gemm2 out: [P][d]
  void* shared_out;            // gemm2 out: [T][d]
  bool out_bf16;
  int T, k, E, P, d, f, fs, fmax;
  int routed_on, shared_on;    // which groups this launch computes (FfnPart)
  int TN;                      // token rows per tile; MMA N = TERMS * TN
  int stages, acc_bufs, tmem_cols, sf_col0;
  unsigned* status;
};

struct __align__(16) N4Ctrl {
  uint64_t full[kN4MaxStages];     // TMA landed (codes + scales)
  uint64_t sfready[kN4MaxStages];  // scales written to TMEM (one arrival per scale-writer warp)
  uint64_t empty[kN4MaxStages];    // stage consumed (MMA commit)
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t ep_sync;
  uint32_t tmem_base;
  int abort;
  float coef[2][kN4BM];            // per B row (token, term) epilogue coefficient, by tile parity
  GroupTable gt;
};

__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int M, int N) {
  // block-scaled MMA: A and B E2M1 (format 1 at [7,10) and [10,13)), K-major,
  // N >> 3 at [17,23), scale type UE4M3 (bit 23 = 0), M >> 4 at [24,29),
  // scale-factor ids 0; D is fp32
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

template <int MODE, int TERMS>
__global__ void __launch_bounds__(kN4Threads, 1)
ffn_nvf4_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapAS,
                const __grid_constant__ CUtensorMap mapSA, const __grid_constant__ CUtensorMap mapSAS,
                const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapSB, N4Args a) {
  constexpr int NA = (MODE == 1) ? 2 : 1;   // weight tiles per stage (gate + up, or down)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = TERMS * a.TN;
  const uint32_t b_bytes = static_cast<uint32_t>(N) * kN4BK;
  const uint32_t b_slot = (b_bytes + 1023u) & ~1023u;
  // stage: [NA code tiles][B codes][NA weight-scale tiles][B scales]
  const uint32_t stage_bytes = NA * kN4ACodes + b_slot + (NA + 1) * kN4Sf;
  N4Ctrl* c = reinterpret_cast<N4Ctrl*>(smem + a.stages * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.E + 1;
  volatile int* abort = &c->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&c->full[s]), 1);
      mbar_init(smem_u32(&c->sfready[s]), 4);
      mbar_init(smem_u32(&c->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c->tfull[b]), 1);
      mbar_init(smem_u32(&c->tempty[b]), kN4Epi);
    }
    mbar_init(smem_u32(&c->drain), 1);
    mbar_init(smem_u32(&c->ep_sync), kN4Epi);
    c->abort = 0;
    fence_barrier_init();
  }
  pdl_enter();   // from here on the kernel reads what earlier kernels wrote
  if (MODE == 1)
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN,
                      a.routed_on ? a.f / kN4BM : 0, a.shared_on ? a.fs / kN4BM : 0, a.status);
  else
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN,
                      a.routed_on ? a.d / kN4BM : 0, a.shared_on ? a.d / kN4BM : 0, a.status);
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), a.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapAS);
    tma_prefetch_desc(&mapSA);
    tma_prefetch_desc(&mapSAS);
    tma_prefetch_desc(&mapB);
    tma_prefetch_desc(&mapSB);
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
      const uint32_t tx = NA * (kN4ACodes + static_cast<uint32_t>(kN4BM) * 16) + b_bytes + static_cast<uint32_t>(N) * 16;
      for (int i = blockIdx.x; i < total && !*abort; i += gridDim.x) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const bool shr = t.g == a.E;
        const CUtensorMap* mA = shr ? &mapAS : &mapA;
        const CUtensorMap* mS = shr ? &mapSAS : &mapSA;
        int arow0, arow1 = 0, K;
        if (MODE == 1) {
          const int width = shr ? a.fs : a.f;
          const int base = shr ? 0 : t.g * 2 * a.f;
          arow0 = base + t.wt * kN4BM;
          arow1 = base + width + t.wt * kN4BM;
          K = a.d;
        } else {
          arow0 = (shr ? 0 : t.g * a.d) + t.wt * kN4BM;
          K = shr ? a.fs : a.f;
        }
        const int brow = TERMS * t.row0;
        for (int kb = 0; kb < K / (2 * kN4BK); ++kb) {
          if (!mbar_wait(smem_u32(&c->empty[st]), ph ^ 1u, abort, kN4WaitNs)) break;
          const uint32_t full = smem_u32(&c->full[st]);
          mbar_arrive_expect_tx(full, tx);
          const uint32_t s0 = smem_u32(smem + st * stage_bytes);
          const uint32_t sB = s0 + NA * kN4ACodes;
          const uint32_t sSA = sB + b_slot;
          const uint32_t sSB = sSA + NA * kN4Sf;
          tma_load_2d(s0, mA, kb * kN4BK, arow0, full);
          tma_load_2d(sSA, mS, kb * 16, arow0, full);
          if (MODE == 1) {
            tma_load_2d(s0 + kN4ACodes, mA, kb * kN4BK, arow1, full);
            tma_load_2d(sSA + kN4Sf, mS, kb * 16, arow1, full);
          }
          tma_load_2d(sB, &mapB, kb * kN4BK, brow, full);
          tma_load_2d(sSB, &mapSB, kb * 16, brow, full);
          pending |= 1u << st;
          last_par = (last_par & ~(1u << st)) | (ph << st);
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      int no_abort = 0;
      for (int s = 0; s < a.stages; ++s)
        if (pending & (1u << s)) mbar_wait(smem_u32(&c->full[s]), (last_par >> s) & 1u, &no_abort, kN4DrainNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_mxf4nvf4(kN4BM, N);
      int st = 0, ab = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const bool shr = t.g == a.E;
        const int K = (MODE == 1) ? a.d : (shr ? a.fs : a.f);
        if (!mbar_wait(smem_u32(&c->tempty[ab]), aph ^ 1u, abort, kN4WaitNs)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + static_cast<uint32_t>(ab * NA * N);
        const uint32_t d1 = d0 + static_cast<uint32_t>(N);
        for (int kb = 0; kb < K / (2 * kN4BK); ++kb) {
          if (!mbar_wait(smem_u32(&c->full[st]), ph, abort, kN4WaitNs) ||
              !mbar_wait(smem_u32(&c->sfready[st]), ph, abort, kN4WaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s0 = smem_u32(smem + st * stage_bytes);
          const uint64_t da0 = desc_sw128(s0);
          const uint64_t da1 = desc_sw128(s0 + kN4ACodes);
          const uint64_t db = desc_sw128(s0 + NA * kN4ACodes);
          const uint32_t sf = tmem + static_cast<uint32_t>(a.sf_col0 + st * kN4SfCols);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            mma_nvf4(d0, da0 + 2 * kk, db + 2 * kk, idesc, sf + 4 * kk, sf + 32 + 4 * kk, accum);
            if (MODE == 1) mma_nvf4(d1, da1 + 2 * kk, db + 2 * kk, idesc, sf + 16 + 4 * kk, sf + 32 + 4 * kk, accum);
          }
          mma_commit(smem_u32(&c->empty[st]));
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
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
      mbar_wait(smem_u32(&c->drain), 0, &no_abort, kN4DrainNs);
    }
  } else if (warp >= 2 + kN4EpiWarps) {
    // -------------------------------------------------- block-scale writers (warps 18..21)
    // Warp w writes the lanes of TMEM quadrant q = w % 4.  Column map of a
    // stage's 48 scale columns: weight tile a (0 = gate / down, 1 = up) at
    // 16 a + 4 kk + q for weight row m = 32 q + lane; activations at
    // 32 + 4 kk + g for activation row n = 32 g + lane (every group g the
    // tile's N reaches), written in every quadrant.  kk = K step of the
    // stage.
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int groups = (N + 31) / 32;
    int st = 0;
    uint32_t ph = 0;
    for (int i = blockIdx.x; i < total && !*abort; i += gridDim.x) {
      const Tile t = decode_tile(c->gt, G, i, a.TN);
      const bool shr = t.g == a.E;
      const int K = (MODE == 1) ? a.d : (shr ? a.fs : a.f);
      bool ok = true;
      for (int kb = 0; kb < K / (2 * kN4BK); ++kb) {
        if (!mbar_wait(smem_u32(&c->full[st]), ph, abort, kN4WaitNs)) {
          ok = false;
          break;
        }
        const uint8_t* s0 = smem + st * stage_bytes;
        const uint8_t* sSA = s0 + NA * kN4ACodes + b_slot;
        const uint8_t* sSB = sSA + NA * kN4Sf;
        const uint32_t sf = tmem + lane_off + static_cast<uint32_t>(a.sf_col0 + st * kN4SfCols);
#pragma unroll
        for (int t2 = 0; t2 < NA; ++t2) {
          const uint4 w = *reinterpret_cast<const uint4*>(sSA + t2 * kN4Sf + (q * 32 + lane) * 16);
          tmem_st1(sf + 16 * t2 + 0 + q, w.x);
          tmem_st1(sf + 16 * t2 + 4 + q, w.y);
          tmem_st1(sf + 16 * t2 + 8 + q, w.z);
          tmem_st1(sf + 16 * t2 + 12 + q, w.w);
        }
        for (int g = 0; g < groups; ++g) {
          const uint4 w = *reinterpret_cast<const uint4*>(sSB + (g * 32 + lane) * 16);
          tmem_st1(sf + 32 + 0 + g, w.x);
          tmem_st1(sf + 32 + 4 + g, w.y);
          tmem_st1(sf + 32 + 8 + g, w.z);
          tmem_st1(sf + 32 + 12 + g, w.w);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c->sfready[st]));
        if (++st == a.stages) {
          st = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..17)
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;               // 0..3: splits the column chunks
    constexpr int kParts = kN4EpiWarps / 4;
    const int n = sub * 32 + lane;                  // weight row within the tile
    const int et = threadIdx.x - 64;                // 0..255
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    int ab = 0, cb_par = 0;
    uint32_t aph = 0, eph = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      const Tile t = decode_tile(c->gt, G, i, a.TN);
      const bool shr = t.g == a.E;
      // per B row (token j, term tt): the term's row scale, times the
      // weights' global scale, times the gate weight in the down projection
      if (et < N) {
        float cf = 0.f;
        const int j = et / TERMS;
        if (j < t.nrows) {
          const int row = t.row0 + j;
          cf = a.b_scale[static_cast<size_t>(row) * TERMS + (et % TERMS)] * (shr ? a.sg[0] : a.wg[t.g]);
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
      mbar_arrive(smem_u32(&c->ep_sync));
      if (!mbar_wait(smem_u32(&c->ep_sync), eph, abort, kN4WaitNs)) break;
      eph ^= 1u;
      const float* coef = c->coef[cb_par];
      cb_par ^= 1;
      if (!mbar_wait(smem_u32(&c->tfull[ab]), aph, abort, kN4WaitNs)) break;
      tc_fence_after();
      const int col = t.wt * kN4BM + n;
      if (MODE == 1) {
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * 2 * N);
        constexpr int TPC = 16 / TERMS;             // tokens per 16-column chunk
        for (int c0 = 16 * part; c0 < N; c0 += 16 * kParts) {
          float gv[16], uv[16];
          tmem_ld16x2(cb + c0, cb + N + c0, gv, uv);
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) {
            const int j = c0 / TERMS + jj;
            if (j < t.nrows) {
              float g = 0.f, u = 0.f;
#pragma unroll
              for (int tt = 0; tt < TERMS; ++tt) {
                const float cf = coef[c0 + jj * TERMS + tt];
                g += gv[jj * TERMS + tt] * cf;
                u += uv[jj * TERMS + tt] * cf;
              }
              a.h[static_cast<size_t>(t.row0 + j) * a.fmax + col] = __float2bfloat16_rn(silu(g) * u);
            }
          }
        }
      } else {
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * N);
        void* outp = shr ? a.shared_out : a.out_perm;
        const size_t out0 = static_cast<size_t>(shr ? t.row0 - a.P : t.row0) * a.d + col;
        constexpr int TPC = 32 / TERMS;             // tokens per 32-column chunk
        for (int c0 = 32 * part; c0 < N; c0 += 32 * kParts) {
          float d0[16], d1[16];
          tmem_ld16x2(cb + c0, cb + c0 + 16, d0, d1);
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) {
            const int j = c0 / TERMS + jj;
            if (j < t.nrows) {
              float v = 0.f;
#pragma unroll
              for (int tt = 0; tt < TERMS; ++tt) {
                const int q = jj * TERMS + tt;
                v += (q < 16 ? d0[q] : d1[q - 16]) * coef[c0 + q];
              }
              store_out(outp, out0 + static_cast<size_t>(j) * a.d, v, a.out_bf16);
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
// NVFP4 term quantiser: row v (bf16) -> TERMS NVFP4 rows a_t with
// v ~ sum_t a_t, found on the residual.  For each term: the row scale g is
// the smallest power of two (>= 2^-126) with max|r| <= 6 * 448 * g; each 16
// elements get the smallest E4M3 scale s with max|r_block| <= 6 g s (1.0 for
// an all-zero block; every comparison exact in fp32); each element the
// nearest e2m1 code of r / (g s), ties to even; then r -= g s e2m1.  With
// one term (the opt-in W4A4 mode, checked against an exact restatement) the
// quotient is an IEEE division; with several terms the later terms absorb
// any rounding of the quotient, so a reciprocal product serves.
// One CTA of kN4QThreads threads per row of the (P+T)-row activation space;
// a thread holds 8 consecutive elements of every kN4QThreads*8-element chunk
// (a 16-element block spans a thread pair); rows row_begin + blockIdx.x.
// GATHER_X: row r < P takes
// x[sorted_pair[r]/k], row P+t takes x[t] (width d); otherwise row r of H
// (width f for routed rows, f_s for shared rows).  Outputs, row r term t at
// row r*TERMS + t: packed codes (element 2i in the low nibble), block-scale
// codes, and the row scale g.

constexpr int kN4QThreads = 128;
constexpr int kN4QChunk = kN4QThreads * 8;   // elements per chunk

__device__ __forceinline__ float e4m3_code_value(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  return __half2float(__half(h));
}

// The smallest positive E4M3 code whose value s satisfies bam <= six_g * s.
__device__ __forceinline__ uint32_t block_scale_code(float bam, float six_g) {
  if (!(bam > 0.f)) return 0x38u;   // all-zero block: scale 1
  const float tgt = bam / six_g;
  uint32_t code = static_cast<uint32_t>(__nv_cvt_float_to_fp8(tgt, __NV_SATFINITE, __NV_E4M3)) & 0x7Fu;
  code = max(code, 1u);
  code = min(code, 0x7Eu);
  if (six_g * e4m3_code_value(code) < bam) code = min(code + 1u, 0x7Eu);
  else if (code > 1u && six_g * e4m3_code_value(code - 1u) >= bam) code -= 1u;
  return code;
}

// The smallest power of two g >= 2^-126 with amax <= 2688 g (1 without a
// positive finite amax).
__device__ __forceinline__ float nvfp4_row_scale_dev(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 1.f;
  int e;
  frexpf(amax, &e);                                  // amax = m 2^e, m in [0.5, 1)
  float g = ldexpf(1.0f, max(e - 12, -126));         // 2688 * 2^(e-12) = 0.65625 * 2^e
  if (amax > 2688.0f * g) g *= 2.0f;
  return g;
}

template <bool GATHER_X, int TERMS>
__global__ void __launch_bounds__(kN4QThreads)
nvf4_terms_kernel(const uint16_t* __restrict__ src, const int32_t* __restrict__ sorted_pair, int P, int T, int k,
                  int width_r, int width_s, int src_stride, uint8_t* __restrict__ codes, int code_stride,
                  uint8_t* __restrict__ scales, int scale_stride, float* __restrict__ gsc, int row_begin,
                  unsigned* status) {
  pdl_enter();
  constexpr int kChunks = kN4MaxWidth / kN4QChunk;
  constexpr int kWarps = kN4QThreads / 32;
  __shared__ float red[TERMS][kWarps];
  const int row = row_begin + blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (row >= P + T) return;
  const uint16_t* s;
  int width;
  if (GATHER_X) {
    int t = row - P;
    width = width_r;
    if (row < P) {
      const int p = sorted_pair[row];
      t = (p >= 0 && p < P) ? p / k : -1;
    }
    if (t < 0) {   // a bad pair: zero terms (the GEMM's epilogue reports the pair)
      if (tid == 0) set_status(status, MOE_ERR_DEVICE_BOUNDS);
      for (int tt = 0; tt < TERMS; ++tt) {
        const size_t r2 = static_cast<size_t>(row) * TERMS + tt;
        for (int cc = tid * 4; cc < width / 2; cc += 4 * kN4QThreads)
          *reinterpret_cast<uint32_t*>(codes + r2 * code_stride + cc) = 0u;
        for (int cc = tid; cc < width / 16; cc += kN4QThreads) scales[r2 * scale_stride + cc] = 0x38u;
        if (tid == 0) gsc[r2] = 0.f;
      }
      return;
    }
    s = src + static_cast<size_t>(t) * src_stride;
  } else {
    s = src + static_cast<size_t>(row) * src_stride;
    width = row < P ? width_r : width_s;
  }
  // widths are multiples of 256, so a thread pair (one 16-element block) is
  // either wholly inside the row or wholly past it
  float r[kChunks][8];
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int e0 = i * kN4QChunk + tid * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (e0 < width) v = *reinterpret_cast<const uint4*>(s + e0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      r[i][2 * q] = __uint_as_float(w[q] << 16);
      r[i][2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
  }
#pragma unroll 1
  for (int tt = 0; tt < TERMS; ++tt) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kChunks; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(r[i][e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[tt][warp] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) amax = fmaxf(amax, red[tt][w]);
    const float g = nvfp4_row_scale_dev(amax);
    const float six_g = 6.0f * g;
    const size_t r2 = static_cast<size_t>(row) * TERMS + tt;
    uint8_t* crow = codes + r2 * code_stride;
    uint8_t* srow = scales + r2 * scale_stride;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int e0 = i * kN4QChunk + tid * 8;
      if (i * kN4QChunk < width) {               // uniform over the warp pair
        float bam = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) bam = fmaxf(bam, fabsf(r[i][e]));
        bam = fmaxf(bam, __shfl_xor_sync(0xffffffffu, bam, 1));
        const uint32_t sc = block_scale_code(bam, six_g);
        const float sv = e4m3_code_value(sc) * g;     // exact: 4 significant bits times a power of two
        const float inv = 1.0f / sv;
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float q0 = TERMS == 1 ? __fdiv_rn(r[i][e], sv) : r[i][e] * inv;
          const float q1 = TERMS == 1 ? __fdiv_rn(r[i][e + 1], sv) : r[i][e + 1] * inv;
          uint16_t b;
          // the first source lands in the high nibble: element e+1 high, element e low
          asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}\n"
              : "=h"(b) : "f"(q1), "f"(q0));
          uint32_t h2;
          asm("{\n .reg .b8 t;\n cvt.u8.u16 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(h2) : "h"(b));
          const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          r[i][e] -= back.x * sv;
          r[i][e + 1] -= back.y * sv;
          packed |= static_cast<uint32_t>(b & 0xffu) << (4 * e);
        }
        if (e0 < width) {
          *reinterpret_cast<uint32_t*>(crow + e0 / 2) = packed;
          if ((tid & 1) == 0) srow[e0 / 16] = static_cast<uint8_t>(sc);
        }
      }
    }
    if (tid == 0) gsc[r2] = g;
  }
}

// ---------------------------------------------------------------------------
// Host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn n4_encode_fn() {
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

// Byte matrix [rows][cols] (row pitch = cols), box of box_cols bytes x
// box_rows; 128-byte swizzle for the 128-byte code boxes, none for the
// 16-byte scale boxes; rows past the end read as zero.
bool make_byte_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows) {
  EncodeTiledFn fn = n4_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct N4Plan {
  size_t xq, xs, xg, h, hq, hs, hg, total;
  int terms, TN;
};

N4Plan n4_plan(const moe_config_t& c) {
  const size_t P = static_cast<size_t>(c.T) * c.top_k, R = P + c.T;
  const size_t fmax = std::max(c.d_ff, c.d_ff_shared);
  N4Plan p;
  p.terms = (c.flags & MOE_FLAG_ACT_NVFP4) ? 1 : 4;
  const size_t tr = R * p.terms;
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o += align_up(b, 1024); return at; };
  p.xq = take(tr * c.d_model / 2);
  p.xs = take(tr * c.d_model / 16);
  p.xg = take(4 * tr);
  p.h = take(2 * R * fmax);
  p.hq = take(tr * fmax / 2);
  p.hs = take(tr * fmax / 16);
  p.hg = take(4 * tr);
  p.total = o;
  // token rows per tile: N = terms * TN must be a multiple of 16 and at most 128
  const double avg = static_cast<double>(P) / c.n_experts;
  // (four terms: a tile about twice the average group, so that most groups
  // of a decode batch fit one tile and each weight tile is read once)
  if (p.terms == 4) p.TN = avg <= 2 ? 4 : avg <= 5 ? 8 : avg <= 16 ? 16 : 32;   // 32: only when forced (larger batches)
  else p.TN = avg <= 16 ? 16 : avg <= 32 ? 32 : avg <= 64 ? 64 : 128;
  return p;
}

template <int MODE, int TERMS>
cudaError_t launch_n4_gemm(const CUtensorMap& mA, const CUtensorMap& mAS, const CUtensorMap& mSA,
                           const CUtensorMap& mSAS, const CUtensorMap& mB, const CUtensorMap& mSB, N4Args a,
                           int wtiles_routed, int wtiles_shared, int grid_cap, cudaStream_t stream) {
  constexpr int NA = (MODE == 1) ? 2 : 1;
  const int N = TERMS * a.TN;
  if (N % 16 != 0 || N < 16 || N > 128) return cudaErrorInvalidConfiguration;
  const int b_slot = static_cast<int>(align_up(static_cast<size_t>(N) * kN4BK, 1024));
  const int stage_bytes = NA * kN4ACodes + b_slot + (NA + 1) * kN4Sf;
  a.stages = std::min(kN4MaxStages, kN4SmemBudget / stage_bytes);
  // TMEM: accumulators (double-buffered when they fit), then kN4SfCols scale
  // columns per stage.  The epilogue's loads (gemm1: 16 columns at c0 and at
  // N + c0; gemm2: 32 from c0) stay within the rounded reach below, after
  // which the scale region starts.
  const int per_acc = NA * N;
  auto sf_start = [&](int bufs) {
    const int acc_end = bufs * per_acc;
    const int reach = (MODE == 1) ? (bufs - 1) * per_acc + N + (N + 31) / 32 * 32
                                  : (bufs - 1) * per_acc + (N + 63) / 64 * 64;
    return static_cast<int>(align_up(static_cast<size_t>(std::max(acc_end, reach)), 32));
  };
  a.acc_bufs = (sf_start(2) + a.stages * kN4SfCols <= 512) ? 2 : 1;
  a.sf_col0 = sf_start(a.acc_bufs);
  a.stages = std::min(a.stages, (512 - a.sf_col0) / kN4SfCols);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  int cols = 32;
  while (cols < a.sf_col0 + a.stages * kN4SfCols) cols *= 2;
  if (cols > 512) return cudaErrorInvalidConfiguration;
  a.tmem_cols = cols;
  size_t smem = 1024 + static_cast<size_t>(a.stages) * stage_bytes + sizeof(N4Ctrl);
  smem = std::max<size_t>(smem, 120 * 1024);   // one CTA per SM: TMEM is never contended
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t err = ensure_kernel_attrs(reinterpret_cast<const void*>(ffn_nvf4_kernel<MODE, TERMS>),
                                        static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const long long tiles_ub = (a.routed_on ? static_cast<long long>(wtiles_routed) * (a.P / a.TN + a.E) : 0) +
                             (a.shared_on ? static_cast<long long>(wtiles_shared) * ((a.T + a.TN - 1) / a.TN) : 0);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(grid_cap, tiles_ub)));
  count_launches(1);
  return launch_pdl(ffn_nvf4_kernel<MODE, TERMS>, grid, kN4Threads, smem, stream, mA, mAS, mSA, mSAS, mB, mSB, a);
}

template <int TERMS>
cudaError_t run_nvf4(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                     const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out, void* ws,
                     unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream) {
  const int T = c.T, k = c.top_k, E = c.n_experts, d = c.d_model, f = c.d_ff, fs = c.d_ff_shared;
  const int P = T * k, R = P + T;
  const int fmax = std::max(f, fs);
  const N4Plan pl = n4_plan(c);
  char* base = static_cast<char*>(ws);
  uint8_t* xq = reinterpret_cast<uint8_t*>(base + pl.xq);
  uint8_t* xs = reinterpret_cast<uint8_t*>(base + pl.xs);
  float* xg = reinterpret_cast<float*>(base + pl.xg);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(base + pl.h);
  uint8_t* hq = reinterpret_cast<uint8_t*>(base + pl.hq);
  uint8_t* hs = reinterpret_cast<uint8_t*>(base + pl.hs);
  float* hg = reinterpret_cast<float*>(base + pl.hg);
  const uint64_t TR = static_cast<uint64_t>(R) * TERMS;

  const int r0 = part.row_begin(P), r1 = part.row_end(P, T);
  const int cap = std::min(num_sms, part.grid_cap);
  count_launches(1);
  cudaError_t err = launch_pdl(nvf4_terms_kernel<true, TERMS>, r1 - r0, kN4QThreads, 0, stream,
                               static_cast<const uint16_t*>(x), sorted_pair, P, T, k, d, d, d, xq, d / 2, xs, d / 16,
                               xg, r0, status);
  if (err != cudaSuccess) return err;

  N4Args a = {};
  a.offsets = offsets; a.sorted_pair = sorted_pair; a.topk_w = topk_w;
  a.h = h; a.out_perm = out_perm; a.shared_out = shared_out;
  a.out_bf16 = (c.flags & MOE_FLAG_BF16_EXPERT_OUT) != 0;
  a.T = T; a.k = k; a.E = E; a.P = P; a.d = d; a.f = f; a.fs = fs; a.fmax = fmax;
  a.routed_on = part.routed; a.shared_on = part.shared;
  // token tile: from the average routed group, or, for the shared expert
  // alone, from T (N = TERMS * TN <= 128)
  const int tn_cap = 128 / TERMS;
  const int tn_sh = T <= 4 ? 4 : T <= 8 ? 8 : T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128;
  a.TN = part.routed ? pl.TN : std::max(16 / TERMS, std::min(tn_sh, tn_cap));
  a.status = status;

  CUtensorMap mA, mAS, mSA, mSAS, mB, mSB;
  // gemm1: gate / up
  if (!make_byte_map(&mA, w->w13, static_cast<uint64_t>(E) * 2 * f, d / 2, kN4BK, kN4BM) ||
      !make_byte_map(&mAS, w->s13, static_cast<uint64_t>(2) * fs, d / 2, kN4BK, kN4BM) ||
      !make_byte_map(&mSA, w->w13_scale, static_cast<uint64_t>(E) * 2 * f, d / 16, 16, kN4BM) ||
      !make_byte_map(&mSAS, w->s13_scale, static_cast<uint64_t>(2) * fs, d / 16, 16, kN4BM) ||
      !make_byte_map(&mB, xq, TR, d / 2, kN4BK, TERMS * a.TN) ||
      !make_byte_map(&mSB, xs, TR, d / 16, 16, TERMS * a.TN))
    return cudaErrorInvalidValue;
  a.wg = w->w13_gscale; a.sg = w->s13_gscale;
  a.b_scale = xg;
  err = launch_n4_gemm<1, TERMS>(mA, mAS, mSA, mSAS, mB, mSB, a, f / kN4BM, fs / kN4BM, cap, stream);
  if (err != cudaSuccess) return err;

  count_launches(1);
  err = launch_pdl(nvf4_terms_kernel<false, TERMS>, r1 - r0, kN4QThreads, 0, stream,
                   reinterpret_cast<const uint16_t*>(h), static_cast<const int32_t*>(nullptr), P, T, k, f, fs, fmax, hq,
                   fmax / 2, hs, fmax / 16, hg, r0, status);
  if (err != cudaSuccess) return err;

  // gemm2: down projection, gate weight, outputs
  if (!make_byte_map(&mA, w->w2, static_cast<uint64_t>(E) * d, f / 2, kN4BK, kN4BM) ||
      !make_byte_map(&mAS, w->s2, static_cast<uint64_t>(d), fs / 2, kN4BK, kN4BM) ||
      !make_byte_map(&mSA, w->w2_scale, static_cast<uint64_t>(E) * d, f / 16, 16, kN4BM) ||
      !make_byte_map(&mSAS, w->s2_scale, static_cast<uint64_t>(d), fs / 16, 16, kN4BM) ||
      !make_byte_map(&mB, hq, TR, fmax / 2, kN4BK, TERMS * a.TN) ||
      !make_byte_map(&mSB, hs, TR, fmax / 16, 16, TERMS * a.TN))
    return cudaErrorInvalidValue;
  a.wg = w->w2_gscale; a.sg = w->s2_gscale;
  a.b_scale = hg;
  return launch_n4_gemm<2, TERMS>(mA, mAS, mSA, mSAS, mB, mSB, a, d / kN4BM, d / kN4BM, cap, stream);
}

}  // namespace

// The block-scaled path takes NVFP4 weights with bf16 x when every width is
// a multiple of 256 (so a row's block scales are a multiple of 16 bytes, as
// TMA requires) and fits the term quantiser's registers.
bool ffn_nvf4_supported(const moe_config_t& c) {
  auto ok = [](int w) { return w % 256 == 0 && w <= kN4MaxWidth; };
  return c.w_dtype == MOE_NVFP4 && c.x_dtype == MOE_BF16 && ok(c.d_model) && ok(c.d_ff) && ok(c.d_ff_shared) &&
         n4_encode_fn() != nullptr;
}

// Whether the exact (four-term) contract should take the block-scaled path:
// yes while the routed groups are small (up to 16 rows per expert on
// average, the decode regime, where the layer streams weights and the four
// terms cost nothing); large batches are bound by the MMAs, which issue four
// times the layer's FLOPs at N = 128 and are fed slower than the f16 path's.
bool ffn_nvf4_preferred(const moe_config_t& c) {
  return static_cast<double>(c.T) * c.top_k <= 16.0 * c.n_experts;
}

size_t ffn_nvf4_ws_bytes(const moe_config_t& c) { return n4_plan(c).total; }

cudaError_t launch_ffn_nvf4(const moe_config_t& c, const void* x, const float* topk_w, const int32_t* offsets,
                            const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                            void* ws, unsigned* status, int num_sms, const FfnPart& part, cudaStream_t stream) {
  if (c.T == 0) return cudaSuccess;
  if (c.flags & MOE_FLAG_ACT_NVFP4)
    return run_nvf4<1>(c, x, topk_w, offsets, sorted_pair, w, out_perm, shared_out, ws, status, num_sms, part, stream);
  return run_nvf4<4>(c, x, topk_w, offsets, sorted_pair, w, out_perm, shared_out, ws, status, num_sms, part, stream);
}

}  // namespace moe
