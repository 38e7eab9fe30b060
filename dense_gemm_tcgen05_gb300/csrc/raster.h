// raster.h -- grouped tile rasteriser shared by the persistent kernels and the
// host (which exports it for tests).
//
// Work index t in [0, tiles_m * tiles_n) is mapped to an output tile so that
// consecutive indices -- the tiles resident on the GPU at the same time -- stay
// inside a band of `group` tile rows and walk down that band before moving one
// tile column to the right.  Concurrent tiles then share a few row panels of
// one operand and a few column panels of the other, which keeps them in L2.
// When group does not divide tiles_m the last band is short.
// ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4", "Step 6: Block
// Scheduling for Cache Reuse": blocks are assigned tiles in groups of rows,
// GroupSize = 8, with a short last group.)
#pragma once

#include <cstdint>

namespace gb300 {

// With `snake` set, odd bands walk the tile columns from right to left, so a
// band starts on the column panels the previous band ended on.
__host__ __device__ inline void raster_tile(int64_t t, int64_t tiles_m, int64_t tiles_n,
                                            int64_t group, int64_t* tm, int64_t* tn,
                                            bool snake = false) {
    const int64_t per_band = group * tiles_n;      // tiles in one full band
    const int64_t band = t / per_band;
    const int64_t first_row = band * group;
    const int64_t rows_left = tiles_m - first_row;
    const int64_t band_rows = rows_left < group ? rows_left : group;
    const int64_t local = t - band * per_band;      // position inside the band
    *tm = first_row + local % band_rows;
    const int64_t col = local / band_rows;
    *tn = (snake && (band & 1)) ? tiles_n - 1 - col : col;
}

}  // namespace gb300
