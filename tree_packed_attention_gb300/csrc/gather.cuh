// Loading a gathered key tile (K or V) with TMA, shared by the q-stationary
// kernels.
//
// A gathered tile holds up to 16 atoms of 8 consecutive key rows; atom a's
// first row is given per tile (negative: the atom loads as zeros). Runs of
// atoms whose rows follow on from each other load as power-of-two boxes of
// 1, 2, 4, 8 or 16 atoms (8 to 128 rows), each landing at the place a single
// 128-row box would give those rows: the 128-byte swizzle is the same within
// every 1024-byte atom, so the tile's layout is the one the tcgen05
// descriptors read.
#pragma once

#include <cuda.h>

#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace treeattn {
namespace dev {

// Producer warp (warp-collective). Lane l holds the first row of atom l % 16
// (`arow`); lanes 0-15 issue the boxes of the first 64 columns, lanes 16-31
// those of the second. A run of n atoms from atom s is cut into boxes by the
// set bits of n, largest first: bit k gives 2^k atoms from atom
// s + (n >> (k + 1) << (k + 1)).
__device__ __forceinline__ void load_gathered(uint8_t* dst, const GatherMaps& maps, uint64_t* bar,
                                              int head, int arow, int lane) {
  constexpr uint32_t kHalf = 128 * 64 * 2;
  const int a = lane & 15, half = lane >> 4;
  const int prev = __shfl_sync(0xffffffffu, arow, (lane & 16) | ((a + 15) & 15));
  const bool start = a == 0 || arow < 0 || prev < 0 || arow != prev + 8;
  const uint32_t starts = __ballot_sync(0xffffffffu, start) & 0xffffu;
  const uint32_t upto = (2u << a) - 1u;  // bits 0..a
  const int s = 31 - __clz(starts & upto);
  const uint32_t above = starts & ~upto;
  const int e = above ? __ffs(above) - 1 : 16;
  const int n = e - s, d = a - s;
#pragma unroll
  for (int k = 4; k >= 0; --k) {
    if (((n >> k) & 1) && d == ((n >> (k + 1)) << (k + 1)))
      tma_load_3d(dst + half * kHalf + a * 1024, &maps.box[k], bar, half * 64, head, arow);
  }
}

}  // namespace dev
}  // namespace treeattn
