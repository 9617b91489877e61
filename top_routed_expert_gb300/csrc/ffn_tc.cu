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
//  * large batches run on CTA pairs (clusters of two, cta_group::2): one
//    MMA covers M = 256 weight rows, each CTA staging its 128 rows and half
//    of the token rows, so each SM reads half the B operand per MAC that a
//    lone 128-row tile needs; the even CTA issues the MMAs of both.  There
//    the two activation terms share one accumulator: the hi and lo MMAs are
//    block-scaled FP8 MMAs (kind::mxf8f6f4) whose B scales are 2^0 and 2^-4,
//    both exact, so each token takes one accumulator column instead of two
//    and a token tile holds twice the tokens for the same TMEM.
//  * every mbarrier wait is bounded; on expiry the kernel records
//    MOE_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and
//    returns.
#include <cuda.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace moe {

using namespace ptx;

// Warps: producer, MMA issuer, then the epilogue warps -- 8, or 16 for the
// CTA-pair down projection, whose epilogue (one fp32 store per output
// element) is the slowest part of a tile and needs more stores in flight.
template <int MODE, int CG>
__host__ __device__ constexpr int tc_epi_warps() { return (MODE == 2 && CG == 2) ? 16 : 8; }
template <int MODE, int CG>
__host__ __device__ constexpr int tc_threads() { return 64 + 32 * tc_epi_warps<MODE, CG>(); }
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
  int sf_col;                  // merged terms: first of the 24 TMEM columns of block scales
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

// MMA N of a tile of `rows` token rows (TERMS B rows each) under the
// launch's full width N: the rows rounded up to 16 (the MMA's N granule),
// at most N.
template <int TERMS>
__device__ __forceinline__ int tile_n_t(int rows, int N) {
  return min(N, (TERMS * rows + 15) & ~15);
}

// TERMS = activation terms per token row: 2 (exact split, default) or 1
// (MOE_FLAG_ACT_E4M3).  The B operand holds TERMS adjacent rows per token.
// CG = CTAs per MMA: 1, or 2 for a CTA pair (launched as clusters of two)
// whose weight tiles are 256 rows: CTA rank r of the pair stages rows
// [128 r, 128 r + 128) of the tile and B rows [r N/2, (r+1) N/2), its TMA
// copies complete on the even CTA's "full" barriers, the even CTA issues the
// MMAs and its commits arrive on the barriers of both CTAs, and both
// epilogues release an accumulator on the even CTA's "tempty" barrier.
// MERGED (pairs with two terms): mapB views the hi rows and mapBL the lo
// rows of the quantised activations (TN / 2 rows per CTA each); the MMA N is
// the token count and the stage holds the CTA's hi tile, then its lo tile.
template <int MODE, int TERMS, int CG>
__global__ void __launch_bounds__(tc_threads<MODE, CG>(), 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapAS,
              const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapBL, TcArgs a) {
  constexpr bool PAIR = CG == 2;
  constexpr bool MERGED = PAIR && TERMS == 2;
  // merged gate/up: one 128-row A tile holds 64 features of gate and of up,
  // interleaved by 16 rows, so one accumulator carries both
  constexpr bool GU_IL = MERGED && MODE == 1;
  constexpr int NA = (MODE == 1 && !GU_IL) ? 2 : 1;   // weight tiles per stage (gate + up, or one)
  constexpr int kEpiThreads = 32 * tc_epi_warps<MODE, CG>();
  constexpr int kParts = tc_epi_warps<MODE, CG>() / 4;   // epilogue warps per TMEM sub-partition
  constexpr int ET = MERGED ? 1 : TERMS;    // accumulator columns per token
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = ET * a.TN;                  // MMA N (the launch's widest)
  const int brows = MERGED ? a.TN : N / CG;   // B rows staged by this CTA per stage
  const uint32_t b_bytes = static_cast<uint32_t>(brows) * kBK;
  const uint32_t lo_off = static_cast<uint32_t>(a.TN / 2) * kBK;   // merged: the lo tile after the hi tile
  const uint32_t stage_bytes = NA * kABytes + ((b_bytes + 1023u) & ~1023u);
  TcCtrl* c = reinterpret_cast<TcCtrl*>(smem + a.stages * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.E + 1;
  volatile int* abort = &c->abort;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // CTA within the pair
  // per-tile MMA N on the pair path (its large-batch tiles are often
  // ragged); the one-CTA path keeps the launch's N, which measured faster at
  // decode, where a tile's rows fill one 16-column granule anyway
  auto tile_n = [](int rows, int n) { return PAIR ? tile_n_t<ET>(rows, n) : n; };
  const bool leader = rank == 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);   // worker index
  const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&c->full[s]), 1);
      mbar_init(smem_u32(&c->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c->tfull[b]), 1);
      mbar_init(smem_u32(&c->tempty[b]), CG * kEpiThreads);
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
  // (weight tiles of CG * 128 rows; interleaved gate/up: 128 features per pair)
  constexpr int WT = GU_IL ? kBM : CG * kBM;
  if (MODE == 1)
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN, a.routed_on ? a.f / WT : 0,
                      a.shared_on ? a.fs / WT : 0, a.status);
  else
    build_group_table(c->gt, a.routed_on ? a.offsets : nullptr, a.E, a.P, a.T, a.TN, a.routed_on ? a.d / WT : 0,
                      a.shared_on ? a.d / WT : 0, a.status);
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(&c->tmem_base), a.tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&c->tmem_base), a.tmem_cols);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapAS);
    tma_prefetch_desc(&mapB);
    if (MERGED) tma_prefetch_desc(&mapBL);
  }
  tc_fence_before();
  // a pair: both CTAs' barriers are initialised and TMEM allocated before
  // either CTA touches the other's
  if constexpr (PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int total = c->gt.tile_start[G];
  if constexpr (MERGED) {
    // block scales (UE8M0) in every lane of both CTAs: A 2^0 (4 columns),
    // B 2^0 for the hi MMAs (8 columns), B 2^-4 for the lo MMAs (8 columns);
    // the sub-partition of warp w is w % 4
    if (warp >= 2 && warp < 6) {
      const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t sf = tmem + lo + static_cast<uint32_t>(a.sf_col);
      tmem_st_fill4(sf, 0x7F7F7F7Fu);
      tmem_st_fill8(sf + 8, 0x7F7F7F7Fu);
      tmem_st_fill8(sf + 16, 0x7B7B7B7Bu);
      tmem_st_wait();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
  }

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int st = 0;
      uint32_t ph = 0, pending = 0, last_par = 0;
      for (int i = unit; i < total && !*abort; i += units) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const bool shr = t.g == a.E;
        const CUtensorMap* mA = shr ? &mapAS : &mapA;
        const int rt = CG * t.wt + static_cast<int>(rank);   // this CTA's 128-row weight tile
        int arow0, arow1 = 0, K;
        if (MODE == 1) {
          const int width = shr ? a.fs : a.f;
          const int base = shr ? 0 : t.g * 2 * a.f;
          arow0 = base + rt * kBM;
          arow1 = base + width + rt * kBM;
          K = a.d;
        } else {
          arow0 = (shr ? 0 : t.g * a.d) + rt * kBM;
          K = shr ? a.fs : a.f;
        }
        // the pair splits the tile's MMA N (its rows, rounded up to 16) evenly
        const int brow = (MERGED ? 1 : TERMS) * t.row0 + static_cast<int>(rank) * (tile_n(t.nrows, N) / CG);
        for (int kb = 0; kb < K / kBK; ++kb) {
          if (!mbar_wait(smem_u32(&c->empty[st]), ph ^ 1u, abort, a.wait_ns)) break;
          const uint32_t full = smem_u32(&c->full[st]);
          const uint32_t sA = smem_u32(smem + st * stage_bytes);
          if constexpr (PAIR) {
            // the even CTA's barrier counts the bytes of both CTAs
            if (leader) mbar_arrive_expect_tx(full, CG * (NA * kABytes + b_bytes));
            const uint32_t fullc = mapa_shared(full, 0);
            if constexpr (GU_IL) {
              // sub-partition q (tile rows 32q..32q+31): 16 gate rows, then
              // the 16 up rows of the same features (boxes of 16 rows)
              const int width = shr ? a.fs : a.f;
              const int frow = (shr ? 0 : t.g * 2 * a.f) + t.wt * kBM + static_cast<int>(rank) * 64;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                tma_load_2d_pair(sA + (32 * q) * kBK, mA, kb * kBK, frow + 16 * q, fullc);
                tma_load_2d_pair(sA + (32 * q + 16) * kBK, mA, kb * kBK, frow + width + 16 * q, fullc);
              }
            } else {
              tma_load_2d_pair(sA, mA, kb * kBK, arow0, fullc);
              if (MODE == 1) tma_load_2d_pair(sA + kABytes, mA, kb * kBK, arow1, fullc);
            }
            tma_load_2d_pair(sA + NA * kABytes, &mapB, kb * kBK, brow, fullc);
            if (MERGED) tma_load_2d_pair(sA + NA * kABytes + lo_off, &mapBL, kb * kBK, brow, fullc);
          } else {
            mbar_arrive_expect_tx(full, NA * kABytes + b_bytes);
            tma_load_2d(sA, mA, kb * kBK, arow0, full);
            if (MODE == 1) tma_load_2d(sA + kABytes, mA, kb * kBK, arow1, full);
            tma_load_2d(sA + NA * kABytes, &mapB, kb * kBK, brow, full);
          }
          pending |= 1u << st;
          last_par = (last_par & ~(1u << st)) | (ph << st);
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // every issued copy must land before the CTA may exit
      if constexpr (PAIR) {
        // A pair's copies complete on the even CTA's barriers.  Without an
        // abort the MMAs consumed every one of them (so they have landed);
        // after an abort, give copies still in flight 2 ms to land.
        if (*abort) {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
        }
      } else {
        int no_abort = 0;
        for (int s = 0; s < a.stages; ++s)
          if (pending & (1u << s)) mbar_wait(smem_u32(&c->full[s]), (last_par >> s) & 1u, &no_abort, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer
      int st = 0, ab = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int i = unit; i < total && ok; i += units) {
        const Tile t = decode_tile(c->gt, G, i, a.TN);
        const bool shr = t.g == a.E;
        const int K = (MODE == 1) ? a.d : (shr ? a.fs : a.f);
        // MMA N of this tile: its rows (x terms) rounded up to 16, so a ragged
        // last tile of a group costs no MMA work beyond that
        const uint32_t idesc = MERGED ? idesc_mxf8_ue8m0(CG * kBM, tile_n(t.nrows, N))
                                      : idesc_f8_e4m3(CG * kBM, tile_n(t.nrows, N));
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
          const uint64_t dbl = desc_sw128(sA + NA * kABytes + lo_off);
          const uint32_t sfa = tmem + static_cast<uint32_t>(a.sf_col);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (MERGED) {
              mma_mxf8_pair(d0, da0 + 2 * kk, db + 2 * kk, idesc, accum, sfa, sfa + 8);
              mma_mxf8_pair(d0, da0 + 2 * kk, dbl + 2 * kk, idesc, 1u, sfa, sfa + 16);
              if (MODE == 1 && !GU_IL) {
                mma_mxf8_pair(d1, da1 + 2 * kk, db + 2 * kk, idesc, accum, sfa, sfa + 8);
                mma_mxf8_pair(d1, da1 + 2 * kk, dbl + 2 * kk, idesc, 1u, sfa, sfa + 16);
              }
            } else if constexpr (PAIR) {
              mma_f8f6f4_pair(d0, da0 + 2 * kk, db + 2 * kk, idesc, accum);
              if (MODE == 1) mma_f8f6f4_pair(d1, da1 + 2 * kk, db + 2 * kk, idesc, accum);
            } else {
              mma_f8f6f4(d0, da0 + 2 * kk, db + 2 * kk, idesc, accum);
              if (MODE == 1) mma_f8f6f4(d1, da1 + 2 * kk, db + 2 * kk, idesc, accum);
            }
          }
          if constexpr (PAIR)
            mma_commit_pair(smem_u32(&c->empty[st]), 3);
          else
            mma_commit(smem_u32(&c->empty[st]));
          if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (!(a.inject_drop && unit == 0 && i == unit)) {
          if constexpr (PAIR)
            mma_commit_pair(smem_u32(&c->tfull[ab]), 3);
          else
            mma_commit(smem_u32(&c->tfull[ab]));
        }
        if (++ab == a.acc_bufs) {
          ab = 0;
          aph ^= 1u;
        }
      }
      // no MMA may still be running when TMEM is released
      if constexpr (PAIR)
        mma_commit_pair(smem_u32(&c->drain), 3);
      else
        mma_commit(smem_u32(&c->drain));
      int no_abort = 0;
      mbar_wait(smem_u32(&c->drain), 0, &no_abort, kDrainLimitNs);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..9)
    // Two warps per TMEM sub-partition (warp % 4 selects the 32 lanes a warp
    // may read); the pair of warps splits the tile's column chunks.
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;               // 0 .. kParts-1: splits the column chunks
    const int n = sub * 32 + lane;                  // weight row within the tile
    const int et = threadIdx.x - 64;                // 0..255 across the epilogue warps
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    int ab = 0, cb_par = 0;
    uint32_t aph = 0, eph = 0;
    for (int i = unit; i < total; i += units) {
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
      const int col = (CG * t.wt + static_cast<int>(rank)) * kBM + n;
      if constexpr (GU_IL) {
        // lanes 0-15 of the sub-partition hold gate, lanes 16-31 up, of the
        // same 16 features; lane l < 16 finishes tokens c0..c0+15 of a chunk
        // and lane l + 16 tokens c0+16..c0+31, after one exchange
        const bool upper = lane >= 16;
        const int fcol = t.wt * kBM + static_cast<int>(rank) * 64 + sub * 16 + (lane & 15);
        const int width = shr ? a.fs : a.f;
        const float sg = shr ? a.as_scale[fcol] : a.a_scale[static_cast<size_t>(t.g) * 2 * a.f + fcol];
        const float su =
            shr ? a.as_scale[width + fcol] : a.a_scale[static_cast<size_t>(t.g) * 2 * a.f + a.f + fcol];
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * N);
        const int nt = tile_n(t.nrows, N);
        for (int c0 = 32 * part; c0 < nt; c0 += 32 * kParts) {
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
              const float cfj = coef[tok];
              const float g = gg[j] * cfj * sg;
              const float u = uu[j] * cfj * su;
              a.h[static_cast<size_t>(t.row0 + tok) * a.fmax + fcol] = __float2bfloat16_rn(silu(g) * u);
            }
          }
        }
      } else if (MODE == 1) {
        const int width = shr ? a.fs : a.f;
        const float sg = shr ? a.as_scale[col] : a.a_scale[static_cast<size_t>(t.g) * 2 * a.f + col];
        const float su = shr ? a.as_scale[width + col] : a.a_scale[static_cast<size_t>(t.g) * 2 * a.f + a.f + col];
        const uint32_t cb = tmem + lane_off + static_cast<uint32_t>(ab * 2 * N);
        // chunks of 32 columns = 32 / ET token rows; N is a multiple of
        // 16 and a 32-wide load past N stays inside the allocation
        constexpr int TPC = 32 / ET;
        const int nt = tile_n(t.nrows, N);
        for (int c0 = 32 * part; c0 < nt; c0 += 32 * kParts) {
          float gv[32], uv[32], cf[TPC];
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) cf[jj] = coef[c0 / ET + jj];
          tmem_ld32x2(cb + c0, cb + N + c0, gv, uv);
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) {
            const int j = c0 / ET + jj;
            if (j < t.nrows) {
              const int row = t.row0 + j;
              const float gd = ET == 2 ? gv[2 * jj] + gv[2 * jj + 1] * 0.0625f : gv[jj];
              const float ud = ET == 2 ? uv[2 * jj] + uv[2 * jj + 1] * 0.0625f : uv[jj];
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
        // chunks of 64 columns = 64 / ET token rows
        constexpr int TPC = 64 / ET;
        const int nt = tile_n(t.nrows, N);
        if constexpr (ET == 1) {
          // one column per token: chunk c0 holds tokens c0..c0+63 (c0 < nt
          // implies c0 < nrows); the output pointer steps one row per token
          for (int c0 = 64 * part; c0 < nt; c0 += 64 * kParts) {
            float d0[32], d1[32];
            tmem_ld32x2(cb + c0, cb + c0 + 32, d0, d1);
            const int jn = min(64, t.nrows - c0);
            const size_t first = out0 + static_cast<size_t>(c0) * a.d;
            if (a.out_bf16) {
              __nv_bfloat16* p = static_cast<__nv_bfloat16*>(outp) + first;
#pragma unroll
              for (int jj = 0; jj < 64; ++jj, p += a.d)
                if (jj < jn) *p = __float2bfloat16_rn((jj < 32 ? d0[jj] : d1[jj - 32]) * coef[c0 + jj] * sw);
            } else {
              float* p = static_cast<float*>(outp) + first;
#pragma unroll
              for (int jj = 0; jj < 64; ++jj, p += a.d)
                if (jj < jn) *p = (jj < 32 ? d0[jj] : d1[jj - 32]) * coef[c0 + jj] * sw;
            }
          }
        } else
        for (int c0 = 64 * part; c0 < nt; c0 += 64 * kParts) {
          float d0[32], d1[32];
          float cf[ET == 2 ? TPC : 1];   // two terms: this chunk's coefficients in registers
          if (ET == 2) {
#pragma unroll
            for (int jj = 0; jj < TPC; ++jj) cf[jj] = coef[c0 / ET + jj];
          }
          tmem_ld32x2(cb + c0, cb + c0 + 32, d0, d1);
#pragma unroll
          for (int jj = 0; jj < TPC; ++jj) {
            const int j = c0 / ET + jj;
            if (j < t.nrows) {
              float dsum;
              if (ET == 2) {
                const float* dv = jj < 16 ? d0 : d1;
                const int q = 2 * (jj & 15);
                dsum = dv[q] + dv[q + 1] * 0.0625f;
              } else {
                dsum = jj < 32 ? d0[jj] : d1[jj - 32];
              }
              const float cfj = ET == 2 ? cf[ET == 2 ? jj : 0] : coef[j];
              store_out(outp, out0 + static_cast<size_t>(j) * a.d, dsum * cfj * sw, a.out_bf16);
            }
          }
        }
      }
      tc_fence_before();
      if constexpr (PAIR)
        mbar_arrive_cluster(mapa_shared(smem_u32(&c->tempty[ab]), 0));
      else
        mbar_arrive(smem_u32(&c->tempty[ab]));
      if (++ab == a.acc_bufs) {
        ab = 0;
        aph ^= 1u;
      }
    }
  }

  tc_fence_before();
  // a pair: neither CTA frees TMEM or exits while the pair's MMAs, copies or
  // arrivals may still reach it
  if constexpr (PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, a.tmem_cols);
    else
      tmem_dealloc(tmem, a.tmem_cols);
  }
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

// Most clusters of two CTAs of `kernel` (with `smem` bytes each) that the
// GPU holds at once, cached per (kernel, smem, device).
int max_pairs(const void* kernel, size_t smem, int threads) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, size_t, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple(kernel, smem, dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
  cache[key] = n;
  return n;
}

// wtiles_* = weight tiles per group, of CG * 128 rows.
template <int MODE, int TERMS, int CG>
cudaError_t launch_gemm(const CUtensorMap& mA, const CUtensorMap& mAS, const CUtensorMap& mB, const CUtensorMap& mBL,
                        TcArgs a, int wtiles_routed, int wtiles_shared, int grid_cap, cudaStream_t stream) {
  constexpr bool MERGED = CG == 2 && TERMS == 2;
  constexpr int NA = (MODE == 1 && !MERGED) ? 2 : 1;   // merged gate/up: one interleaved A tile
  const int N = (MERGED ? 1 : TERMS) * a.TN;
  const int brows = MERGED ? a.TN : N / CG;
  const int stage_bytes = NA * kABytes + align_up(static_cast<size_t>(brows) * kBK, 1024);
  // as many stages as fit next to the control block in 227 KB
  a.stages = std::min(kMaxStages, static_cast<int>((227 * 1024 - 1024 - sizeof(TcCtrl)) / stage_bytes));
  const int per_acc = NA * N;
  a.acc_bufs = (2 * per_acc <= 512) ? 2 : 1;
  // The epilogue reads 32 columns per load (gemm1: gate and up from column c0
  // and N + c0, c0 < N in steps of 32, or one interleaved accumulator; gemm2:
  // 64 from c0, c0 < N in steps of 64), so the allocation covers the last
  // buffer plus that overhang.
  const int last = (a.acc_bufs - 1) * per_acc;
  const int reach = (MODE == 1) ? last + (NA == 2 ? N : 0) + (N + 31) / 32 * 32 : last + (N + 63) / 64 * 64;
  int cols = 32;
  a.sf_col = 0;
  if (MERGED) {
    // 24 columns of block scales after the accumulators (the epilogue's
    // overhanging loads may read them; they read past no allocation)
    a.sf_col = align_up(static_cast<size_t>(a.acc_bufs * per_acc), 8);
    cols = 512;
    if (a.sf_col + 24 > 512 || reach > 512) return cudaErrorInvalidConfiguration;
  }
  while (cols < reach) cols *= 2;
  if (cols > 512) return cudaErrorInvalidConfiguration;
  a.tmem_cols = cols;
  size_t smem = 1024 + static_cast<size_t>(a.stages) * stage_bytes + sizeof(TcCtrl);
  smem = std::max<size_t>(smem, 120 * 1024);   // one CTA per SM: TMEM is never contended
  const void* kfn = reinterpret_cast<const void*>(ffn_tc_kernel<MODE, TERMS, CG>);
  cudaError_t err = ensure_kernel_attrs(kfn, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const long long tiles_ub = (a.routed_on ? static_cast<long long>(wtiles_routed) * (a.P / a.TN + a.E) : 0) +
                             (a.shared_on ? static_cast<long long>(wtiles_shared) * ((a.T + a.TN - 1) / a.TN) : 0);
  if (CG == 1) {
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(grid_cap, tiles_ub)));
    count_launches(1);
    return launch_pdl(ffn_tc_kernel<MODE, TERMS, CG>, grid, tc_threads<MODE, CG>(), smem, stream, mA, mAS, mB, mBL,
                      a);
  }
  // pairs: no more clusters than the GPU holds at once (each walks its share
  // of the tile list in turn)
  const int resident = max_pairs(kfn, smem, tc_threads<MODE, CG>());
  if (resident < 1) return cudaErrorInvalidConfiguration;
  const int pairs = static_cast<int>(
      std::max<long long>(1, std::min<long long>(std::min(resident, std::max(1, grid_cap / 2)), tiles_ub)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(tc_threads<MODE, CG>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, ffn_tc_kernel<MODE, TERMS, CG>, mA, mAS, mB, mBL, a);
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
  int tn1 = one_term ? std::max(16, std::min(tn, 128)) : std::min(tn, MOE_TC_TN1_CAP);
  // one term, down GEMM: 256-token tiles once groups are that large (N = 256
  // halves the operand bytes per MAC of a 128 x 128 tile; K = f is short, so
  // the feed, not the MMA, bounds the smaller tile)
  const bool big = part.routed ? static_cast<double>(P) / E > 96 : T > 96;
  int tn2 = one_term ? (big ? 256 : std::max(16, std::min(tn, 128))) : std::min(tn, MOE_TC_TN2_CAP);
  // CTA pairs (M = 256) for large batches, where the MMAs rather than the
  // weight stream bound the GEMMs: average routed groups above 48 rows and
  // widths that split into 256-row tiles.  With two terms the pair merges
  // them into one accumulator and gate/up interleaves gate and up rows in
  // one A tile: token tiles of 224 for both GEMMs (two accumulator buffers
  // of 224 columns and the block scales fill TMEM), so each MMA has N = 224
  // (an FP8 MMA with N <= 128 costs nearly as long as one with N = 224).
  const bool inject = (c.flags & MOE_FLAG_INJECT_TIMEOUT) != 0;
  const bool pair = P > 48 * E && f % 256 == 0 && fs % 256 == 0 && d % 256 == 0 && !inject &&
                    (one_term ? tn1 >= 128 && tn2 >= 128 : true);
  const bool merged = pair && !one_term;
  if (merged) {
    tn1 = 224;
    tn2 = 224;
  }
  const int cg = pair ? 2 : 1;
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

  CUtensorMap mA, mAS, mB, mBL;
  TcArgs a = {};
  a.offsets = offsets; a.sorted_pair = sorted_pair; a.topk_w = topk_w;
  a.h = h; a.out_perm = out_perm; a.shared_out = shared_out;
  a.out_bf16 = (c.flags & MOE_FLAG_BF16_EXPERT_OUT) != 0;
  a.T = T; a.k = k; a.E = E; a.P = P; a.d = d; a.f = f; a.fs = fs; a.fmax = fmax;
  a.routed_on = part.routed; a.shared_on = part.shared;
  a.TN = pl.TN; a.status = status;
  a.wait_ns = inject ? 20000000ull : kWaitLimitNs;
  a.inject_drop = inject ? 1 : 0;

  // gemm1: gate/up (B: both term rows of each activation row; the hi rows
  // only; or, merged, the hi rows and the lo rows as two views)
  bool mb_ok;
  if (merged)
    mb_ok = make_map(&mB, xq, static_cast<uint64_t>(R), d, tn1 / 2, 2 * static_cast<uint64_t>(d)) &&
            make_map(&mBL, xq + d, static_cast<uint64_t>(R), d, tn1 / 2, 2 * static_cast<uint64_t>(d));
  else
    mb_ok = one_term ? make_map(&mB, xq, static_cast<uint64_t>(R), d, tn1 / cg, 2 * static_cast<uint64_t>(d))
                     : make_map(&mB, xq, static_cast<uint64_t>(2) * R, d, 2 * tn1 / cg);
  if (!merged) mBL = mB;
  // (merged: gate and up rows are fetched in boxes of 16 rows, interleaved)
  const uint32_t abox = merged ? 16 : kBM;
  if (!make_map(&mA, w->w13, static_cast<uint64_t>(E) * 2 * f, d, abox) ||
      !make_map(&mAS, w->s13, static_cast<uint64_t>(2) * fs, d, abox) || !mb_ok)
    return cudaErrorInvalidValue;
  a.a_scale = static_cast<const float*>(w->w13_scale);
  a.as_scale = static_cast<const float*>(w->s13_scale);
  a.b_scale = sx;
  a.TN = tn1;   // two buffers of (gate, up) x (columns per token) x TN fit TMEM
  // weight tiles per group: of cg * 128 rows, or, merged gate/up, of 128
  // features (64 of gate and up per CTA)
  const int wt_f = merged ? f / kBM : f / (cg * kBM), wt_fs = merged ? fs / kBM : fs / (cg * kBM);
  const int wt_d = d / (cg * kBM);
  if (pair)
    err = one_term ? launch_gemm<1, 1, 2>(mA, mAS, mB, mBL, a, wt_f, wt_fs, cap, stream)
                   : launch_gemm<1, 2, 2>(mA, mAS, mB, mBL, a, wt_f, wt_fs, cap, stream);
  else
    err = one_term ? launch_gemm<1, 1, 1>(mA, mAS, mB, mBL, a, wt_f, wt_fs, cap, stream)
                   : launch_gemm<1, 2, 1>(mA, mAS, mB, mBL, a, wt_f, wt_fs, cap, stream);
  if (err != cudaSuccess) return err;

  count_launches(1);
  err = launch_pdl(regs ? quant2_rows_kernel<false, true> : quant2_rows_kernel<false, false>, qblocks, 256, 0, stream,
                   reinterpret_cast<const uint16_t*>(h), static_cast<const int32_t*>(nullptr), P, T, k, f, fs, fmax,
                   hq, fmax, sh, !one_term, r0, r1, status);
  if (err != cudaSuccess) return err;

  // gemm2: down projection, gate weight, outputs
  bool mb2_ok;
  if (merged)
    mb2_ok = make_map(&mB, hq, static_cast<uint64_t>(R), fmax, tn2 / 2, 2 * static_cast<uint64_t>(fmax)) &&
             make_map(&mBL, hq + fmax, static_cast<uint64_t>(R), fmax, tn2 / 2, 2 * static_cast<uint64_t>(fmax));
  else
    mb2_ok = one_term ? make_map(&mB, hq, static_cast<uint64_t>(R), fmax, tn2 / cg, 2 * static_cast<uint64_t>(fmax))
                      : make_map(&mB, hq, static_cast<uint64_t>(2) * R, fmax, 2 * tn2 / cg);
  if (!merged) mBL = mB;
  if (!make_map(&mA, w->w2, static_cast<uint64_t>(E) * d, f, kBM) ||
      !make_map(&mAS, w->s2, static_cast<uint64_t>(d), fs, kBM) || !mb2_ok)
    return cudaErrorInvalidValue;
  a.a_scale = static_cast<const float*>(w->w2_scale);
  a.as_scale = static_cast<const float*>(w->s2_scale);
  a.b_scale = sh;
  a.TN = tn2;
  if (pair)
    return one_term ? launch_gemm<2, 1, 2>(mA, mAS, mB, mBL, a, wt_d, wt_d, cap, stream)
                    : launch_gemm<2, 2, 2>(mA, mAS, mB, mBL, a, wt_d, wt_d, cap, stream);
  return one_term ? launch_gemm<2, 1, 1>(mA, mAS, mB, mBL, a, wt_d, wt_d, cap, stream)
                  : launch_gemm<2, 2, 1>(mA, mAS, mB, mBL, a, wt_d, wt_d, cap, stream);
}

}  // namespace moe
