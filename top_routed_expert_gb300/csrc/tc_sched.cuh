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
// wtiles_shared weight tiles per group, token tiles of TN rows.  Offsets that
// are not monotone or leave [0, P] make that group empty and record
// MOE_ERR_DEVICE_BOUNDS.  Returns the number of tiles.  One thread.
__device__ __forceinline__ int build_group_table(GroupTable& gt, const int32_t* offsets, int E, int P, int T, int TN,
                                                 int wtiles_routed, int wtiles_shared, unsigned* status) {
  int acc = 0;
  for (int g = 0; g <= E; ++g) {
    int base, rows;
    if (g < E) {
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
    const int wt = (g < E) ? wtiles_routed : wtiles_shared;
    const int mt = (rows + TN - 1) / TN;
    gt.tile_start[g] = acc;
    gt.row_base[g] = base;
    gt.rows[g] = rows;
    gt.mtiles[g] = mt;
    acc += mt * wt;
  }
  gt.tile_start[E + 1] = acc;
  return acc;
}

}  // namespace moe
