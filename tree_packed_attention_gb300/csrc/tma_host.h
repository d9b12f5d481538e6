// Host-side helpers: TMA tensor maps for [rows, heads, 128] bf16 tensors and
// device properties, shared by the bf16 kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace treeattn {

// A 3-D map over a token-major [n, heads, 128] bf16 tensor whose box is
// 64 head-dim elements x 1 head x 128 tokens, 128-byte swizzled. Loading
// the two halves (d = 0 and d = 64) of one (head, 128-token) tile gives the
// K-major operand layout the tcgen05 shared-memory descriptors expect.
// Returns false if the driver rejects the map.
bool make_tile_map(CUtensorMap* map, const void* base, int n, int heads);

int sm_count();

}  // namespace treeattn
