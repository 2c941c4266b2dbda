// tmap.cuh -- host helpers shared by the tensor-core launchers (defined in chunk_tc.cu).
#pragma once

#include <cuda.h>

namespace osdn {
// Tensor map over [rows][H][inner] 16-bit elements (rows = B*T tokens), box (64, 1, 64),
// 128-byte swizzle: one 64-token x 64-element tile of one head per copy.
bool make_row_tmap(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int inner, int H, long long rows);
// Multiprocessor count of the current device (cached).
int device_sm_count();
}  // namespace osdn
