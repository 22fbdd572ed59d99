// Host-only check of the batched path's tile geometry (moe_kernels.cu),
// compiled and run by tests/test_plan_host.py: for every hidden and inter
// size the ABI accepts, gate/up tiles hold whole row pairs, every row of a
// tile is covered by the warps' lane streams (the mapping of tile_tokens), a
// row has at most four 32-group chunks, and a tile's shared memory fits the
// per-block opt-in limit.  Prints "ok <shapes>" and exits 0, or names the first
// violation and exits 1.
#include <cstdio>

#include "../include/moe.h"
#include "../bit_expert_matvec_moe_b300/csrc/moe_kernels.cu"

namespace {

// rows covered by tile_tokens' lanes for rows of ng groups: warp w takes chunk
// w % chunks and rows (w / chunks) * rpp + lane / lpr + k * nstreams * rpp
bool covers(int ng, int rows) {
  const moe::RowMap m = moe::make_rowmap(ng);
  const int nstreams = moe::kWsWarps / m.chunks;
  if (nstreams < 1) return false;
  for (int r = 0; r < rows; ++r) {
    bool hit = false;
    for (int s = 0; s < nstreams && !hit; ++s)
      for (int j = 0; j < m.rpp && !hit; ++j)
        for (int k = 0; k < moe::kMaxRowsPerLane && !hit; ++k) hit = s * m.rpp + j + k * nstreams * m.rpp == r;
    if (!hit) return false;
  }
  return true;
}

}  // namespace

int main() {
  const size_t optin = 232448;
  int n = 0;
  for (int H = 64; H <= MOE_MAX_HIDDEN; H += 64) {
    for (int I = 64; I <= MOE_MAX_INTER; I += 64) {
      const int gt = moe::gu_tile_rows(H), dt = moe::dn_tile_rows(I);
      const int ngh = H / 64, ngi = I / 64;
      if (gt < 2 || gt % 2 || dt < 1) {
        std::printf("H=%d I=%d: tile rows %d / %d\n", H, I, gt, dt);
        return 1;
      }
      if (!covers(ngh, gt) || !covers(ngi, dt)) {
        std::printf("H=%d I=%d: tile rows not covered by the lane streams\n", H, I);
        return 1;
      }
      if ((ngh + 31) / 32 > 4 || (ngi + 31) / 32 > 4) {
        std::printf("H=%d I=%d: more than four row chunks\n", H, I);
        return 1;
      }
      const size_t sg = moe::tile_smem(gt, moe::make_fmt(4, H, I).gu_row, moe::make_fmt(2, H, I).gu_row, ngh);
      const size_t sd = moe::tile_smem(dt, moe::make_fmt(4, H, I).d_row, moe::make_fmt(2, H, I).d_row, ngi);
      if (sg > optin || sd > optin) {
        std::printf("H=%d I=%d: tile shared memory %zu / %zu\n", H, I, sg, sd);
        return 1;
      }
      ++n;
    }
  }
  std::printf("ok %d\n", n);
  return 0;
}
