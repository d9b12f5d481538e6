// Host-side helpers: TMA tensor maps for [rows, heads, 128] bf16 tensors and
// device properties, shared by the bf16 kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace treeattn {

// A 3-D map over a token-major [n, heads, 128] bf16 tensor whose box is
// 64 head-dim elements x 1 head x box_rows tokens, 128-byte swizzled. Loading
// the two halves (d = 0 and d = 64) of one (head, 128-token) tile gives the
// K-major operand layout the tcgen05 shared-memory descriptors expect; a box
// of 8 tokens is one 1024-byte swizzle atom of that layout. Rows outside
// [0, n) load as zeros. Returns false if the driver rejects the map.
bool make_tile_map(CUtensorMap* map, const void* base, int n, int heads, int box_rows = 128);

// Tensor maps of one [n, heads, 128] bf16 tensor with boxes of 8 << k rows
// (k = 0..4), for loading gathered key tiles.
struct GatherMaps {
  CUtensorMap box[5];
};

// The five maps of a gathered K or V tensor: boxes of 8, 16, 32, 64 and 128 rows.
bool make_gather_maps(GatherMaps* maps, const void* base, int n, int heads);

int sm_count();

}  // namespace treeattn
