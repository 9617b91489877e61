// Grouped SwiGLU expert FFN on CUDA cores: the general path for every weight
// format (fp32, FP8 E4M3 per-channel, NVFP4) and the reference against which
// the tensor-core path is developed.  Sarvam blog, Table 1 rows "Routed
// expert compute" and "Shared expert compute"; section "Scaling multilingual
// sovereign AI with MoE" (routed top-k experts plus one shared expert).
//
// Groups 0..E-1 are the routed experts (rows = their pairs in sorted order),
// group E is the shared expert (rows = all T tokens, gate weight 1).  The
// tile list over (group, 32-row tile) is rebuilt on the device from the
// expert offsets, so nothing is read back to the host.
//   ffn1: H[row, n] = silu(x . Wg[n]) * (x . Wu[n])      (fp32 H in workspace)
//   ffn2: out[row, n] = gate(row) * (H[row] . W2[n])
// Weights are dequantised to fp32 while they are staged in shared memory.
#include "common.cuh"

namespace moe {

enum WFmt { kWF32 = 0, kWE4M3 = 1, kWNVFP4 = 2 };

constexpr int kSimtThreads = 256;
constexpr int kTM = 32;    // rows per tile
constexpr int kTN = 64;    // output columns per tile
constexpr int kKC = 32;    // K chunk

struct MatRef {              // one [rows][K] weight matrix in its stored format
  const void* q;
  const void* scale;         // e4m3: float per row; nvfp4: u8 e4m3 per 16 K
  float gscale;              // nvfp4 global scale
};

// Stage rows [r0, r0+64) x K [k0, k0+32) of a matrix, dequantised, into ws.
template <int FMT>
__device__ __forceinline__ void stage_weights(const MatRef& m, int K, int r0, int k0, float (*ws)[kKC + 1]) {
  const int row = threadIdx.x >> 2;          // 0..63
  const int seg = (threadIdx.x & 3) * 8;     // 8 consecutive K elements
  const size_t gr = static_cast<size_t>(r0 + row);
  float v[8];
  if (FMT == kWF32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(m.q) + gr * K + k0 + seg);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else if (FMT == kWE4M3) {
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(m.q) + gr * K + k0 + seg);
    const float s = static_cast<const float*>(m.scale)[gr];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = e4m3_to_float((raw.x >> (8 * i)) & 0xff) * s;
      v[4 + i] = e4m3_to_float((raw.y >> (8 * i)) & 0xff) * s;
    }
  } else {
    const uint32_t raw =
        *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(m.q) + gr * (K / 2) + (k0 + seg) / 2);
    const uint8_t bs = static_cast<const uint8_t*>(m.scale)[gr * (K / 16) + (k0 + seg) / 16];
    const float s = e4m3_to_float(bs) * m.gscale;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = e2m1_to_float((raw >> (4 * i)) & 0xf) * s;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) ws[row][seg + i] = v[i];
}

__device__ __forceinline__ MatRef expert_mat(const void* q, const void* scale, const float* gscale, int fmt,
                                             int e, int rows, int K) {
  MatRef m;
  const size_t n = static_cast<size_t>(rows) * K;
  if (fmt == kWF32) {
    m.q = static_cast<const float*>(q) + e * n;
    m.scale = nullptr;
    m.gscale = 1.f;
  } else if (fmt == kWE4M3) {
    m.q = static_cast<const uint8_t*>(q) + e * n;
    m.scale = static_cast<const float*>(scale) + static_cast<size_t>(e) * rows;
    m.gscale = 1.f;
  } else {
    m.q = static_cast<const uint8_t*>(q) + e * (n / 2);
    m.scale = static_cast<const uint8_t*>(scale) + e * (n / 16);
    m.gscale = gscale[e];
  }
  return m;
}

struct FfnArgs {
  const void* x;              // [T][d] f32 or bf16
  const float* topk_w;        // [T*k]
  const int32_t* offsets;     // [E+1]
  const int32_t* sorted_pair; // [P]
  moe_weights_t w;
  float* h;                   // [P][f]   routed SwiGLU activations
  float* hs;                  // [T][fs]  shared-expert activations
  void* out_perm;             // [P][d] bf16 or fp32
  void* shared_out;           // [T][d]
  bool out_bf16;
  int T, d, E, k, f, fs;
  unsigned* status;
};

// Resolves this CTA's (group, first row, rows) from the device tile table.
struct TileInfo { int g, row0, rows, base; };

__device__ __forceinline__ bool tile_of_block(const FfnArgs& a, int* s_tile_start, int* s_scratch, TileInfo* ti) {
  build_tile_table(a.offsets, a.E, a.T, kTM, s_tile_start, s_scratch);
  const int G = a.E + 1;
  const int i = blockIdx.x;
  if (i >= s_tile_start[G]) return false;
  const int g = find_group(s_tile_start, G, i);
  const int m = i - s_tile_start[g];
  int base = 0, rows = a.T;
  if (g < a.E) {
    base = a.offsets[g];
    rows = a.offsets[g + 1] - base;
    const int P = a.T * a.k;
    if (base < 0 || rows < 0 || base + rows > P) {
      if (threadIdx.x == 0) set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
      return false;
    }
  }
  ti->g = g;
  ti->row0 = m * kTM;
  ti->rows = min(kTM, rows - m * kTM);
  ti->base = base;
  return true;
}

template <int FMT, typename XT>
__global__ void __launch_bounds__(kSimtThreads) ffn1_simt_kernel(FfnArgs a) {
  __shared__ int s_tile_start[kMaxGroups + 1];
  __shared__ int s_scratch[kMaxGroups];
  __shared__ int s_tok[kTM];
  __shared__ float xs[kTM][kKC + 1];
  __shared__ float wg[kTN][kKC + 1];
  __shared__ float wu[kTN][kKC + 1];
  TileInfo ti;
  if (!tile_of_block(a, s_tile_start, s_scratch, &ti)) return;
  const bool shared_grp = ti.g == a.E;
  const int width = shared_grp ? a.fs : a.f;
  const int n0 = blockIdx.y * kTN;
  if (n0 >= width) return;
  const int P = a.T * a.k;
  if (threadIdx.x < kTM) {
    int t = -1;
    if (threadIdx.x < ti.rows) {
      const int r = ti.row0 + threadIdx.x;
      if (shared_grp) {
        t = r;
      } else {
        const int p = a.sorted_pair[ti.base + r];
        if (p >= 0 && p < P) t = p / a.k;
        else set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
      }
    }
    s_tok[threadIdx.x] = t;
  }
  MatRef W = shared_grp ? expert_mat(a.w.s13, a.w.s13_scale, a.w.s13_gscale, FMT, 0, 2 * a.fs, a.d)
                        : expert_mat(a.w.w13, a.w.w13_scale, a.w.w13_gscale, FMT, ti.g, 2 * a.f, a.d);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float ag[2][4] = {}, au[2][4] = {};
  const XT* x = static_cast<const XT*>(a.x);
  __syncthreads();
  for (int k0 = 0; k0 < a.d; k0 += kKC) {
    {  // x tile: 32 rows x 32 K, 4 elements per thread
      const int r = threadIdx.x >> 3, c = (threadIdx.x & 7) * 4;
      const int t = s_tok[r];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        xs[r][c + i] = (t >= 0) ? x_to_float<XT>(x[static_cast<size_t>(t) * a.d + k0 + c + i]) : 0.f;
    }
    stage_weights<FMT>(W, a.d, n0, k0, wg);
    stage_weights<FMT>(W, a.d, width + n0, k0, wu);
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      const float x0 = xs[ty][kk], x1 = xs[ty + 16][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float g = wg[tx + 16 * j][kk], u = wu[tx + 16 * j][kk];
        ag[0][j] = fmaf(x0, g, ag[0][j]);
        ag[1][j] = fmaf(x1, g, ag[1][j]);
        au[0][j] = fmaf(x0, u, au[0][j]);
        au[1][j] = fmaf(x1, u, au[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty + 16 * i;
    if (r >= ti.rows) continue;
    float* hrow = shared_grp ? a.hs + static_cast<size_t>(ti.row0 + r) * a.fs
                             : a.h + static_cast<size_t>(ti.base + ti.row0 + r) * a.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) hrow[n0 + tx + 16 * j] = silu(ag[i][j]) * au[i][j];
  }
}

template <int FMT>
__global__ void __launch_bounds__(kSimtThreads) ffn2_simt_kernel(FfnArgs a) {
  __shared__ int s_tile_start[kMaxGroups + 1];
  __shared__ int s_scratch[kMaxGroups];
  __shared__ float s_gate[kTM];
  __shared__ float hsm[kTM][kKC + 1];
  __shared__ float w2s[kTN][kKC + 1];
  TileInfo ti;
  if (!tile_of_block(a, s_tile_start, s_scratch, &ti)) return;
  const bool shared_grp = ti.g == a.E;
  const int K = shared_grp ? a.fs : a.f;
  const int n0 = blockIdx.y * kTN;
  const int P = a.T * a.k;
  if (threadIdx.x < kTM) {
    float gw = 0.f;
    if (threadIdx.x < ti.rows) {
      if (shared_grp) {
        gw = 1.f;
      } else {
        const int p = a.sorted_pair[ti.base + ti.row0 + threadIdx.x];
        if (p >= 0 && p < P) gw = a.topk_w[p];
      }
    }
    s_gate[threadIdx.x] = gw;
  }
  MatRef W = shared_grp ? expert_mat(a.w.s2, a.w.s2_scale, a.w.s2_gscale, FMT, 0, a.d, a.fs)
                        : expert_mat(a.w.w2, a.w.w2_scale, a.w.w2_gscale, FMT, ti.g, a.d, a.f);
  const float* hbase = shared_grp ? a.hs + static_cast<size_t>(ti.row0) * a.fs
                                  : a.h + static_cast<size_t>(ti.base + ti.row0) * a.f;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[2][4] = {};
  for (int k0 = 0; k0 < K; k0 += kKC) {
    {
      const int r = threadIdx.x >> 3, c = (threadIdx.x & 7) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < ti.rows) v = *reinterpret_cast<const float4*>(hbase + static_cast<size_t>(r) * K + k0 + c);
      hsm[r][c] = v.x; hsm[r][c + 1] = v.y; hsm[r][c + 2] = v.z; hsm[r][c + 3] = v.w;
    }
    stage_weights<FMT>(W, K, n0, k0, w2s);
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      const float h0 = hsm[ty][kk], h1 = hsm[ty + 16][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = w2s[tx + 16 * j][kk];
        acc[0][j] = fmaf(h0, w, acc[0][j]);
        acc[1][j] = fmaf(h1, w, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty + 16 * i;
    if (r >= ti.rows) continue;
    void* outp = shared_grp ? a.shared_out : a.out_perm;
    const size_t orow = static_cast<size_t>(shared_grp ? ti.row0 + r : ti.base + ti.row0 + r) * a.d;
    const float gw = s_gate[r];
#pragma unroll
    for (int j = 0; j < 4; ++j) store_out(outp, orow + n0 + tx + 16 * j, acc[i][j] * gw, a.out_bf16);
  }
}

size_t ffn_simt_ws_bytes(int T, int k, int f, int fs) {
  const size_t P = static_cast<size_t>(T) * k;
  return align_up(sizeof(float) * P * f, 256) + align_up(sizeof(float) * static_cast<size_t>(T) * fs, 256);
}

cudaError_t launch_ffn_simt(const void* x, bool x_bf16, int w_dtype, const float* topk_w, const int32_t* offsets,
                            const int32_t* sorted_pair, const moe_weights_t* w, void* out_perm, void* shared_out,
                            bool out_bf16, int T, int d, int E, int k, int f, int fs, void* ws, unsigned* status,
                            cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  FfnArgs a;
  a.x = x; a.topk_w = topk_w; a.offsets = offsets; a.sorted_pair = sorted_pair; a.w = *w;
  const size_t P = static_cast<size_t>(T) * k;
  a.h = static_cast<float*>(ws);
  a.hs = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(sizeof(float) * P * f, 256));
  a.out_perm = out_perm; a.shared_out = shared_out; a.out_bf16 = out_bf16;
  a.T = T; a.d = d; a.E = E; a.k = k; a.f = f; a.fs = fs; a.status = status;
  // upper bound of (group, 32-row) tiles: sum_e ceil(c_e/32) <= P/32 + E, plus the shared group
  const int tiles = static_cast<int>(P / kTM) + E + ceil_div(T, kTM) + 1;
  const dim3 g1(tiles, ceil_div(std::max(f, fs), kTN));
  const dim3 g2(tiles, ceil_div(d, kTN));
  const int fmt = (w_dtype == MOE_F32) ? kWF32 : (w_dtype == MOE_E4M3) ? kWE4M3 : kWNVFP4;
  count_launches(2);
#define MOE_FFN1(F, XT) ffn1_simt_kernel<F, XT><<<g1, kSimtThreads, 0, stream>>>(a)
  if (fmt == kWF32) { if (x_bf16) MOE_FFN1(kWF32, uint16_t); else MOE_FFN1(kWF32, float); }
  else if (fmt == kWE4M3) { if (x_bf16) MOE_FFN1(kWE4M3, uint16_t); else MOE_FFN1(kWE4M3, float); }
  else { if (x_bf16) MOE_FFN1(kWNVFP4, uint16_t); else MOE_FFN1(kWNVFP4, float); }
#undef MOE_FFN1
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (fmt == kWF32) ffn2_simt_kernel<kWF32><<<g2, kSimtThreads, 0, stream>>>(a);
  else if (fmt == kWE4M3) ffn2_simt_kernel<kWE4M3><<<g2, kSimtThreads, 0, stream>>>(a);
  else ffn2_simt_kernel<kWNVFP4><<<g2, kSimtThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
