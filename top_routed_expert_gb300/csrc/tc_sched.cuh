// Device-side tile list shared by the tensor-core grouped GEMMs: groups are
// the routed experts (g < E, rows = their pairs in expert-sorted order) and
// the shared expert (g = E, rows = all T tokens); a tile is (group, weight
// tile, token tile), numbered group-major, then weight tile, then token tile,
// so that CTAs working at the same time share weight tiles and token slabs
// in L2.  Built per CTA from the expert offsets -- no host read-back.
#pragma once

#include "common.cuh"

namespace moe {

struct GroupTable {
  int tile_start[kMaxGroups + 1];
  int row_base[kMaxGroups];    // first row of the group in the (P+T)-row activation space
  int rows[kMaxGroups];
  int mtiles[kMaxGroups];
};

struct Tile {
  int g, wt, row0, nrows;
};

__device__ __forceinline__ Tile decode_tile(const GroupTable& gt, int G, int i, int TN) {
  Tile t;
  t.g = find_group(gt.tile_start, G, i);
  const int local = i - gt.tile_start[t.g];
  const int mt_n = gt.mtiles[t.g];
  t.wt = local / mt_n;
  const int mt = local - t.wt * mt_n;
  t.row0 = gt.row_base[t.g] + mt * TN;
  t.nrows = min(TN, gt.rows[t.g] - mt * TN);
  return t;
}


// Fills the table for E routed groups plus the shared group; wtiles_routed /
// wtiles_shared weight tiles per group (0 leaves that part out), token tiles
// of TN rows.  Offsets that are not monotone or leave [0, P] make that group
// empty and record MOE_ERR_DEVICE_BOUNDS; offsets == nullptr (a launch of the
// shared part alone, which may run while the offsets are being written)
// makes every routed group empty without reading them.  Called by every
// thread of the block (it contains __syncthreads): one thread per group
// fills the group's entries, then warp 0
// turns the per-group tile counts into their exclusive prefix sum with warp
// shuffles.  Returns after the table is visible to the whole block.
__device__ __forceinline__ void build_group_table(GroupTable& gt, const int32_t* offsets, int E, int P, int T, int TN,
                                                  int wtiles_routed, int wtiles_shared, unsigned* status) {
  const int G = E + 1;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int base, rows;
    if (g < E && offsets == nullptr) {
      base = 0;
      rows = 0;
    } else if (g < E) {
      base = offsets[g];
      rows = offsets[g + 1] - base;
      if (base < 0 || rows < 0 || base + rows > P) {
        set_status(status, MOE_ERR_DEVICE_BOUNDS);
        base = 0;
        rows = 0;
      }
    } else {
      base = P;
      rows = T;
    }
    const int mt = (rows + TN - 1) / TN;
    gt.row_base[g] = base;
    gt.rows[g] = rows;
    gt.mtiles[g] = mt;
    gt.tile_start[g] = mt * ((g < E) ? wtiles_routed : wtiles_shared);   // tile count, scanned below
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int c0 = 0; c0 < G; c0 += 32) {
      const int g = c0 + lane;
      const int cnt = (g < G) ? gt.tile_start[g] : 0;
      int v = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
      }
      if (g < G) gt.tile_start[g] = carry + v - cnt;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) gt.tile_start[G] = carry;
  }
  __syncthreads();
}

}  // namespace moe
