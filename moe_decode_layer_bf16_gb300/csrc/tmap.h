// Host side of the TMA tensor maps shared by the expert kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once; null if unavailable.
EncodeTiledFn encode_fn();

// 2-D map over a dense uint8 array [rows][cols] (cols bytes a row, a multiple
// of 16) with a {box_cols, box_rows} box and the 128-byte swizzle; rows past
// the end read as zeros.
bool tmap_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows);

}  // namespace moe
