// CTA -> output-tile mapping shared by the SGEMM kernels.
#pragma once

namespace sgemm {

// Map a linear CTA index to (tile_m, tile_n), walking GROUP_M tile rows at a
// time so that CTAs resident together share slabs of A and B in L2.
template <int GROUP_M>
__device__ __forceinline__ void grouped_tile(int pid, int tiles_m, int tiles_n, int &tm, int &tn) {
    const int per_group = GROUP_M * tiles_n;
    const int group = pid / per_group;
    const int first_m = group * GROUP_M;
    const int rows = min(tiles_m - first_m, GROUP_M);
    const int in_group = pid - group * per_group;
    tm = first_m + in_group % rows;
    tn = in_group / rows;
}

}  // namespace sgemm
