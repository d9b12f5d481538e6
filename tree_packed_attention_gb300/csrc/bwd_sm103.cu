// Backward tree attention, bf16 in / fp32 accumulate, on the sm_103a tensor
// cores, as two kernels with no atomics and no fp32 accumulator in HBM:
//
//  1. dQ kernel (Q-stationary; one 128-row q-tile of one q head per work
//     item, walking the plan's non-empty k-tiles of that q-tile):
//        Delta_i = dO_i . O_i,  P = exp2(S*scale*log2e - lse_i*log2e),
//        dP = dO V^T,  dS = P (dP - Delta),  dQ += dS K,  dq = scale * dQ.
//     It also writes Delta and lse*log2(e) into padded [hq, Tq*128] rows of
//     the workspace for kernel 2.
//  2. dK/dV kernel (KV-stationary; one 128-key tile of one kv head per item,
//     walking every q head of the group and every q-tile that sees the key
//     tile -- one contiguous range [kt_qlo, kt_qhi), because the rows that
//     see key j are exactly [j, key_end[j])):
//        S^T = K Q^T, P^T, dP^T = V dO^T, dS^T = P^T (dP^T - Delta),
//        dV += P^T dO,  dK += dS^T Q,  dk = scale * dK.
//
// ("Tree Training", arXiv 2511.00413, §3.2 "Attention Mask" and App. A.1 for
// the mask; the derivatives are the standard softmax-attention ones.)
// Recomputing S and dP in both kernels costs two extra 128^3 products per
// tile pair (7 instead of 5) but removes the dQ reduction traffic, which on
// this GPU throttled a single-kernel design to a fifth of the tensor rate.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "kernels.h"
#include "gather.cuh"
#include "sched.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace treeattn {
namespace {

using namespace dev;

constexpr uint32_t kTileBytes = 128 * 128 * 2;
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr float kLog2e = 1.4426950408889634f;

// (a wait that gives up records the line it was called from)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status, int line = __builtin_LINE()) {
  const bool ok = mbar_wait(bar, parity, abort, status, kSiteBwd + line);
  return __all_sync(0xffffffffu, ok);
}

// D = A B^T, A and B both K-major 128 x 128 tiles (K = 128).
// The GEMM helpers are warp-collective: one elected lane issues each MMA.
__device__ __forceinline__ void mma_kk(uint32_t d, uint32_t a, uint32_t b, uint32_t acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
  const uint64_t ad = sdesc_sw128(a, 16, 1024), bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss_warp(d, sdesc_advance(ad, off), sdesc_advance(bd, off), idesc, (acc || kk > 0) ? 1u : 0u);
  }
}


// D = A B^T, A from TMEM split in two halves: K elements 0-63 in columns 0-31
// and K elements 64-127 in columns 64-95 (each written by one warpgroup over
// columns it had already read), B MN-major in smem.
__device__ __forceinline__ void mma_tn_split(uint32_t d, uint32_t a_tmem, uint32_t b, uint32_t acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
  const uint64_t bd = sdesc_sw128(b, kHalfBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_warp(d, a_tmem + kk * 8 + (kk >= 4 ? 32 : 0), sdesc_advance(bd, kk * 2048), idesc,
                (acc || kk > 0) ? 1u : 0u);
}

// Write 32 consecutive fp32 values of one 128-wide row, times `mul`, as fp32 or
// bf16; with 32-byte stores when the destination allows (`v8`).
__device__ __forceinline__ void store_row(void* dst_base, size_t off, int c, const uint32_t (&v)[32],
                                          float mul, int out_f32, int v8) {
  if (out_f32) {
    float* dst = static_cast<float*>(dst_base) + off + c * 32;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(v[8 * u + e]) * mul);
      if (v8) {
        st_global_v8(dst + 8 * u, w);
      } else {
        reinterpret_cast<uint4*>(dst + 8 * u)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst + 8 * u)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(dst_base) + off + c * 32;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        w[e] = pack_bf16x2(__uint_as_float(v[16 * u + 2 * e]) * mul,
                           __uint_as_float(v[16 * u + 2 * e + 1]) * mul);
      if (v8) {
        st_global_v8(dst + 16 * u, w);
      } else {
        reinterpret_cast<uint4*>(dst + 16 * u)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst + 16 * u)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }
}

// 32 bytes to global memory: one 32-byte store if the destination is 32-byte
// aligned (v8), else two 16-byte stores.
__device__ __forceinline__ void store32(void* dst, const uint32_t (&w)[8], int v8) {
  if (v8) {
    st_global_v8(dst, w);
  } else {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// ============================================================== dQ kernel
// 384 threads: warp 0 TMA producer, warp 1 MMA issuer + TMEM owner, warps 4-11
// one q row per thread, two warpgroups splitting the keys of each tile.
// TMEM: S_a | S_b | dP | dQ (128 columns each); dS is written as bf16 into the
// S buffer it came from and read by the dQ MMA from TMEM.
constexpr int kDqThreads = 384;
// K_t is read by S_t and, a step later, by dQ_t; S_{t+2} is issued right after
// dQ_t, so K needs a third stage for its load to overlap a whole step. The
// same ring carries each item's O tile (for Delta) ahead of its K tiles.
constexpr int kDqKStages = 3;
// Launched at 168 registers a thread; warps 0-3 drop to 72 and the softmax
// warpgroups rise to 216 (128 x 72 + 256 x 216 = 384 x 168).
constexpr uint32_t kDqRegsCtl = 72, kDqRegsSoftmax = 216;
static_assert(128 * kDqRegsCtl + 256 * kDqRegsSoftmax <= 384 * 168, "register split");
constexpr int kDqVStages = 2;
constexpr uint32_t kDqOffQ = 0;
constexpr uint32_t kDqOffDO = kTileBytes;
constexpr uint32_t kDqOffK = 2 * kTileBytes;
constexpr uint32_t kDqOffV = kDqOffK + kDqKStages * kTileBytes;
constexpr uint32_t kDqOffKe = kDqOffV + kDqVStages * kTileBytes;  // per K stage: 128 key_end
// Delta of the tile's 128 rows, two buffers (items alternate)
constexpr uint32_t kDqOffDelta = kDqOffKe + kDqKStages * 512;
// mbarriers, then the item ring, then the TMEM base and the abort flag
constexpr uint32_t kDqOffBar = kDqOffDelta + 2 * 512;
constexpr uint32_t kDqNumBars = 3 + 2 * kDqKStages + 2 * kDqVStages + 2 + 5 + 4 + 1 + 1;
constexpr uint32_t kDqOffRing = kDqOffBar + kDqNumBars * 8;
constexpr uint32_t kDqOffMisc = kDqOffRing + sizeof(ItemRing);
constexpr uint32_t kDqSmem = kDqOffMisc + 16;
static_assert(kDqSmem <= 232448, "shared memory budget");

struct DqParams {
  const int32_t* gq_ptr;     // q-tile -> its gathered key tiles
  const int32_t* gt_kind;    // per tile: 0 empty, 1 partial, 2 full
  const int32_t* gt_atom;    // per tile: first key row of each 8-column atom (-8: zeros)
  const int32_t* gt_bidx;    // per tile: row of its key bounds, -1 if not PARTIAL
  const int32_t* gt_bounds;  // per bounds row: key_end of each column
  const int32_t* order;
  const __nv_bfloat16* o;
  const float* lse;
  float* lse2;   // out: [hq, Npad], -lse * log2(e)
  float* delta;  // out: [hq, Npad], -Delta
  void* dq;
  int* status;
  SchedSlot* sched;
  int N, Npad, hq, group, n_items, out_f32;
  int out_v8;  // dq is 32-byte aligned
  int has_gateway;
  float scale, scale_log2;
};


__global__ void __launch_bounds__(kDqThreads, 1)
    tree_attn_bwd_dq_sm103(const __grid_constant__ CUtensorMap map_q,
                           const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_v,
                           const __grid_constant__ CUtensorMap map_do,
                           const __grid_constant__ CUtensorMap map_o,
                           const __grid_constant__ GatherMaps gmap_k,
                           const __grid_constant__ GatherMaps gmap_v,
                           const __grid_constant__ GatherMaps gmap_pk,
                           const __grid_constant__ GatherMaps gmap_pv, const DqParams p) {
  // All shared state sits in the dynamic block (no static shared memory), so
  // the block starts 1024-aligned as the 128B-swizzled tiles need.
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicExch(p.status, 9);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDqOffBar);
  uint64_t& bar_q_full = bars[0];
  uint64_t& bar_q_empty = bars[1];
  uint64_t& bar_final = bars[2];
  uint64_t (&bar_k_full)[kDqKStages] = *reinterpret_cast<uint64_t(*)[kDqKStages]>(bars + 3);
  uint64_t (&bar_k_empty)[kDqKStages] =
      *reinterpret_cast<uint64_t(*)[kDqKStages]>(bars + 3 + kDqKStages);
  uint64_t (&bar_v_full)[kDqVStages] =
      *reinterpret_cast<uint64_t(*)[kDqVStages]>(bars + 3 + 2 * kDqKStages);
  uint64_t (&bar_v_empty)[kDqVStages] =
      *reinterpret_cast<uint64_t(*)[kDqVStages]>(bars + 3 + 2 * kDqKStages + kDqVStages);
  // one per S buffer: a buffer is refilled only after its dS was consumed, so
  // each barrier is at most one phase ahead
  uint64_t (&bar_s_full)[2] =
      *reinterpret_cast<uint64_t(*)[2]>(bars + 3 + 2 * kDqKStages + 2 * kDqVStages);
  uint64_t* tail = bars + 5 + 2 * kDqKStages + 2 * kDqVStages;
  uint64_t& bar_dp_full = tail[0];
  // one per S buffer, like bar_s_full: the dS of tile t sits in buffer t % 2,
  // and with the S buffers doubled a warp can finish tile t+1 before another
  // has stored its dS of tile t, so one shared barrier could complete tile t's
  // phase with a tile t+1 arrival and let the dQ product read a dS that is not
  // there yet. Buffer b's next dS needs S_{t+2}, which waits for this phase.
  uint64_t& bar_ds_full0 = tail[1];
  uint64_t& bar_ds_full1 = tail[10];
  uint64_t& bar_dq_full = tail[2];
  uint64_t& bar_dq_free = tail[3];
  uint64_t& bar_dp_read = tail[4];  // the softmax warps hold dP_t in registers
  // per row quarter: both warps of the quarter wrote their half of its Delta
  uint64_t* bar_delta = tail + 5;
  uint64_t& bar_o_read = tail[9];  // the softmax warps read the item's O tile
  ItemRing& ring = *reinterpret_cast<ItemRing*>(smem + kDqOffRing);
  uint32_t& tmem_base_s = *reinterpret_cast<uint32_t*>(smem + kDqOffMisc);
  int& abort_s = *reinterpret_cast<int*>(smem + kDqOffMisc + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort = &abort_s;
  if (threadIdx.x == 0) {
    item_ring_init(&ring, 9);  // consumers: the MMA warp and the 8 softmax warps
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_final, 1);
    for (int s = 0; s < kDqKStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
    }
    for (int s = 0; s < kDqVStages; ++s) {
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_v_empty[s], 1);
    }
    mbar_init(&bar_s_full[0], 1);
    mbar_init(&bar_s_full[1], 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_ds_full0, 256);
    mbar_init(&bar_ds_full1, 256);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_free, 256);
    mbar_init(&bar_dp_read, 256);
    for (int qq = 0; qq < 4; ++qq) mbar_init(&bar_delta[qq], 2);
    mbar_init(&bar_o_read, 8);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_do);
    tma_prefetch_desc(&map_o);
    for (int b = 0; b < 5; ++b) {
      tma_prefetch_desc(&gmap_k.box[b]);
      tma_prefetch_desc(&gmap_v.box[b]);
      if (p.has_gateway) {
        tma_prefetch_desc(&gmap_pk.box[b]);
        tma_prefetch_desc(&gmap_pv.box[b]);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tS = tmem, tDP = tmem + 256, tDQ = tmem + 384;  // S_a at 0, S_b at 128

  if (warp == 0) {
    regs_dec<kDqRegsCtl>();
    // ------------------------------------------------------------ producer
    // kv counts tiles (the V ring); kk counts entries of the K ring, which
    // carries each item's O tile (read once, for Delta) ahead of its K tiles.
    uint32_t kv = 0, kk = 0, qn = 0, pub = 0;
    auto k_slot_free = [&](uint32_t e) {
      return e < kDqKStages ||
             warp_wait(&bar_k_empty[e % kDqKStages], ((e / kDqKStages) & 1) ^ 1, abort, p.status);
    };
    // The next item is taken once every load of this one is issued (taking
    // it earlier can leave two long items on one CTA).
    // Items are published with their header (q-tile, tile range) so the
    // other roles need no global loads to start one.
    int nqt = 0, nbeg = 0, nend = 0;
    auto take = [&]() {
      const int id = item_fetch(p.sched, p.n_items);
      if (id >= 0) {
        nqt = __ldg(p.order + id / p.hq);
        nbeg = __ldg(p.gq_ptr + nqt);
        nend = __ldg(p.gq_ptr + nqt + 1);
      }
      return id;
    };
    int cur = take();
    bool ok = item_put(&ring, pub, cur, abort, p.status, nqt, nbeg, nend);
    while (ok && cur >= 0) {
      const int qt = nqt, h = cur % p.hq, kvh = h / p.group, beg = nbeg, end = nend;
      if (qn > 0 && !(ok = warp_wait(&bar_q_empty, (qn - 1) & 1, abort, p.status))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_q_full, 2 * kTileBytes);
        tma_load_3d(smem + kDqOffQ, &map_q, &bar_q_full, 0, h, qt * 128);
        tma_load_3d(smem + kDqOffQ + kHalfBytes, &map_q, &bar_q_full, 64, h, qt * 128);
        tma_load_3d(smem + kDqOffDO, &map_do, &bar_q_full, 0, h, qt * 128);
        tma_load_3d(smem + kDqOffDO + kHalfBytes, &map_do, &bar_q_full, 64, h, qt * 128);
      }
      __syncwarp();
      ++qn;
      if (!(ok = k_slot_free(kk))) break;
      if (lane == 0) {
        const uint32_t so = kk % kDqKStages;
        uint8_t* dst = smem + kDqOffK + so * kTileBytes;
        mbar_arrive_expect_tx(&bar_k_full[so], kTileBytes);
        tma_load_3d(dst, &map_o, &bar_k_full[so], 0, h, qt * 128);
        tma_load_3d(dst + kHalfBytes, &map_o, &bar_k_full[so], 64, h, qt * 128);
      }
      __syncwarp();
      ++kk;
      // this lane's atom and the bounds row of the next tile, one tile ahead
      int arow_next = 0, bidx_next = -1, kind_next = 0;
      if (beg < end) {
        arow_next = ldg_pinned(p.gt_atom + 16 * beg + (lane & 15));
        bidx_next = ldg_pinned(p.gt_bidx + beg);
        kind_next = ldg_pinned(p.gt_kind + beg);
      }
      for (int t = beg; t < end; ++t, ++kv, ++kk) {
        const int arow = arow_next, bidx = bidx_next;
        const bool gw = (kind_next >> 4) & 1;  // gateway keys: the past K/V tensors
        if (t + 1 < end) {
          arow_next = ldg_pinned(p.gt_atom + 16 * (t + 1) + (lane & 15));
          bidx_next = ldg_pinned(p.gt_bidx + t + 1);
          kind_next = ldg_pinned(p.gt_kind + t + 1);
        }
        const uint32_t sk = kk % kDqKStages;
        if (!(ok = k_slot_free(kk))) break;
        uint8_t* kdst = smem + kDqOffK + sk * kTileBytes;
        if (lane == 0) {
          // a PARTIAL tile's 128 key bounds travel with it
          mbar_arrive_expect_tx(&bar_k_full[sk], kTileBytes + (bidx >= 0 ? 512u : 0u));
          if (bidx >= 0)
            bulk_load(smem + kDqOffKe + sk * 512, p.gt_bounds + static_cast<size_t>(bidx) * 128, 512,
                      &bar_k_full[sk]);
        }
        __syncwarp();
        load_gathered(kdst, gw ? gmap_pk : gmap_k, &bar_k_full[sk], kvh, arow, lane);
        __syncwarp();
        const uint32_t sv = kv % kDqVStages, pv = (kv / kDqVStages) & 1;
        if (kv >= kDqVStages && !(ok = warp_wait(&bar_v_empty[sv], pv ^ 1, abort, p.status))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar_v_full[sv], kTileBytes);
        __syncwarp();
        load_gathered(smem + kDqOffV + sv * kTileBytes, gw ? gmap_pv : gmap_v, &bar_v_full[sv], kvh, arow,
                      lane);
        __syncwarp();
      }
      if (!ok) break;
      cur = take();
      if (!(ok = item_put(&ring, pub, cur, abort, p.status, nqt, nbeg, nend))) break;
      if (cur >= 0 && lane == 0) {  // its Q and dO into L2 while this item finishes
        const int nh = cur % p.hq;
        tma_prefetch_l2_3d(&map_q, 0, nh, nqt * 128);
        tma_prefetch_l2_3d(&map_q, 64, nh, nqt * 128);
        tma_prefetch_l2_3d(&map_do, 0, nh, nqt * 128);
        tma_prefetch_l2_3d(&map_do, 64, nh, nqt * 128);
        tma_prefetch_l2_3d(&map_o, 0, nh, nqt * 128);
        tma_prefetch_l2_3d(&map_o, 64, nh, nqt * 128);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      if (qn > 0) mbar_drain(&bar_q_full, (qn - 1) & 1);
      for (uint32_t i = kk >= kDqKStages ? kk - kDqKStages : 0; i <= kk; ++i)
        mbar_drain(&bar_k_full[i % kDqKStages], (i / kDqKStages) & 1);
      for (uint32_t i = kv >= kDqVStages ? kv - kDqVStages : 0; i <= kv; ++i)
        mbar_drain(&bar_v_full[i % kDqVStages], (i / kDqVStages) & 1);
    }
  } else if (warp == 1) {
    regs_dec<kDqRegsCtl>();
    // ---------------------------------------------------------- MMA issuer
    // Per item: S_0, dP_0, [O read] release of the O entry, S_1; then per
    // tile t: [dP_t read] dP_{t+1}; [dS_t] dQ += dS_t K_t, S_{t+2} (into the S
    // buffer dQ_t just read).
    const uint32_t aQ = smem_u32(smem + kDqOffQ), aDO = smem_u32(smem + kDqOffDO);
    const uint32_t aK = smem_u32(smem + kDqOffK), aV = smem_u32(smem + kDqOffV);
    uint32_t kv = 0, kk = 0, qn = 0, n = 0, got = 0;
    uint32_t dsu0 = 0, dsu1 = 0;  // dS phases consumed per S buffer
    bool ok = true;
    int hdr[3];
    for (int cur; (ok = item_get(&ring, got, cur, abort, p.status, hdr)) && cur >= 0;) {
      const int T = hdr[2] - hdr[1];
      if (!(ok = warp_wait(&bar_q_full, qn & 1, abort, p.status))) break;
      ++qn;
      auto k_stage = [&](uint32_t i) { return aK + (i % kDqKStages) * kTileBytes; };
      auto v_stage = [&](uint32_t i) { return aV + (i % kDqVStages) * kTileBytes; };
      auto wait_k = [&](uint32_t i) {
        return warp_wait(&bar_k_full[i % kDqKStages], (i / kDqKStages) & 1, abort, p.status);
      };
      auto wait_v = [&](uint32_t i) {
        return warp_wait(&bar_v_full[i % kDqVStages], (i / kDqVStages) & 1, abort, p.status);
      };
      // K ring: the item's O tile at entry eo, its K tiles from eo + 1. The
      // O entry is waited for like a K tile so this warp keeps step with
      // every phase of the ring.
      const uint32_t eo = kk;
      if (!(ok = wait_k(eo))) break;
      if (!(ok = wait_k(eo + 1))) break;
      tc_fence_after_sync();
      mma_kk(tS, aQ, k_stage(eo + 1), 0);  // S_0
      mma_commit_warp(&bar_s_full[0]);
      if (!(ok = wait_v(kv))) break;
      tc_fence_after_sync();
      mma_kk(tDP, aDO, v_stage(kv), 0);  // dP_0
      mma_commit_warp(&bar_dp_full);
      mma_commit_warp(&bar_v_empty[kv % kDqVStages]);
      // the O entry's slot is free once every softmax warp has read it
      if (!(ok = warp_wait(&bar_o_read, (qn - 1) & 1, abort, p.status))) break;
      if (lane == 0) mbar_arrive(&bar_k_empty[eo % kDqKStages]);
      __syncwarp();
      if (T > 1) {
        if (!(ok = wait_k(eo + 2))) break;
        tc_fence_after_sync();
        mma_kk(tS + 128, aQ, k_stage(eo + 2), 0);  // S_1
        mma_commit_warp(&bar_s_full[1]);
      }
      for (int t = 0; t < T && ok; ++t, ++n) {
        const uint32_t i = kv + t, ik = eo + 1 + t;  // V ring, K ring
        // dP_{t+1} as soon as the softmax warps hold dP_t, ahead of dQ_t
        if (t + 1 < T) {
          if (!(ok = warp_wait(&bar_dp_read, n & 1, abort, p.status))) break;
          if (!(ok = wait_v(i + 1))) break;
          tc_fence_after_sync();
          mma_kk(tDP, aDO, v_stage(i + 1), 0);
          mma_commit_warp(&bar_dp_full);
          mma_commit_warp(&bar_v_empty[(i + 1) % kDqVStages]);
          // dP_{T-1} is the item's last reader of Q and dO (S_{T-1} came
          // before it, and Delta read dO before the first dP was released):
          // the next item's Q and dO load during the last step.
          if (t + 2 == T) mma_commit_warp(&bar_q_empty);
        }
        {
          const bool odd = (t & 1) != 0;
          if (!(ok = warp_wait(odd ? &bar_ds_full1 : &bar_ds_full0, (odd ? dsu1 : dsu0) & 1, abort,
                               p.status)))
            break;
          dsu1 += odd ? 1u : 0u;
          dsu0 += odd ? 0u : 1u;
        }
        if (t == 0 && qn > 1 && !(ok = warp_wait(&bar_dq_free, (qn - 2) & 1, abort, p.status)))
          break;
        tc_fence_after_sync();
        mma_tn_split(tDQ, tS + (t & 1) * 128, k_stage(ik), t > 0);  // dQ += dS_t K_t
        mma_commit_warp(&bar_k_empty[ik % kDqKStages]);
        if (t + 1 == T) mma_commit_warp(&bar_dq_full);
        if (T == 1) mma_commit_warp(&bar_q_empty);  // the softmax warps read dO for Delta
                                                    // before the first dS arrives
        if (t + 2 < T) {
          if (!(ok = wait_k(ik + 2))) break;
          tc_fence_after_sync();
          mma_kk(tS + (t & 1) * 128, aQ, k_stage(ik + 2), 0);  // S_{t+2}
          mma_commit_warp(&bar_s_full[t & 1]);
        }
      }
      kv += T;
      kk += T + 1;
    }
    mma_commit_warp(&bar_final);
    mbar_drain(&bar_final, 0);
  } else if (warp < 4) {
    regs_dec<kDqRegsCtl>();  // warps 2-3: idle
  } else {
    regs_inc<kDqRegsSoftmax>();
    // ---- two warpgroups split each tile's 128 keys: warps 4-7 take keys
    // 0-63, warps 8-11 keys 64-127; one q row per thread (TMEM lane = row).
    // Each half writes its dS (bf16) over the first 32 columns of its own S
    // columns, so the halves never touch each other's unread data.
    const int half = (warp - 4) / 4;
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = half * 64;
    const float sl2 = p.scale_log2;
    uint32_t n = 0, kk = 0, qn = 0, su0 = 0, su1 = 0;  // kk: K ring entries (O, then K tiles)
    bool ok = true;
    // The next item's q-tile and tile range are read one item ahead, and each
    // tile's kind and k-tile one tile ahead, so no global load latency sits
    // between two passes over S. A tile's key bounds come with its K stage.
    int hdr[3] = {0, 0, 0};  // the next item's q-tile and tile range, from the ring
    int nt_kind = 0, nt_arow = 0, nt_at = -1;  // nt_arow: first key of atom lane % 16
    auto fetch_tile = [&](int t) {
      nt_kind = ldg_pinned(p.gt_kind + t) & 19;  // kind, and 16 for gateway keys
      nt_arow = ldg_pinned(p.gt_atom + 16 * t + (lane & 15));
      nt_at = t;
    };
    // The next item's number is read once this item's tiles are done (the
    // producer publishes it when this item's loads are issued); its header
    // loads overlap the wait for the last dQ product.
    uint32_t got = 0;
    int cur = -1;
    ok = item_get(&ring, got, cur, abort, p.status, hdr);
    // The thread's lse is loaded as soon as the item is known (right after
    // the previous item's last tile), so its latency passes during the
    // previous epilogue.
    float lse_pre = INFINITY;
    auto load_lse = [&](int item) {
      const int ii = hdr[0] * 128 + r;
      lse_pre = ii < p.N ? __ldg(p.lse + static_cast<size_t>(item % p.hq) * p.N + ii) : INFINITY;
    };
    if (ok && cur >= 0) load_lse(cur);
    auto next_item = [&](int& nxt) -> bool {
      if (!item_get(&ring, got, nxt, abort, p.status, hdr)) return false;
      if (nxt >= 0) load_lse(nxt);
      return true;
    };
    while (ok && cur >= 0) {
      const int qt = hdr[0], h = cur % p.hq, beg = hdr[1], end = hdr[2];
      int nxt = -1;
      const int i = qt * 128 + r;
      if (!(ok = warp_wait(&bar_q_full, qn & 1, abort, p.status))) break;
      // the item's O tile, in the K ring ahead of its K tiles
      if (!(ok = warp_wait(&bar_k_full[kk % kDqKStages], (kk / kDqKStages) & 1, abort, p.status)))
        break;
      // Delta = dO . O of this thread's row. The two warps of a row quarter
      // split its 32 rows, 16 each (warps 4-7 the first 16). Each lane forms
      // its part of the warp's 16 dot products (lane l: dims 4l..4l+3 of O
      // and dO, both 128B-swizzled tiles in smem; rows past N count zero); a
      // transposing reduction leaves row 2m's sum in lanes 2m and 2m+1; the
      // two warps of the quarter swap halves through smem.
      // both kept negated (they are addends below), and stored so for dK/dV
      float ndelta = 0.f, nlse2 = -INFINITY;
      {
        float part[16];
        const int r0 = qt * 128 + quarter * 32 + half * 16;
        const uint32_t lane_byte = (lane >> 4) * kHalfBytes + (lane & 1) * 8;
        const uint8_t* dbase = smem + kDqOffDO + lane_byte;
        const uint8_t* obase = smem + kDqOffK + (kk % kDqKStages) * kTileBytes + lane_byte;
        const int chunk = (lane >> 1) & 7;
        const int nvalid = min(16, p.N - r0);
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          const int rt = quarter * 32 + half * 16 + rr;  // row within the tile
          const uint32_t off = rt * 128 + ((chunk ^ (rt & 7)) * 16);
          const uint2 dv = *reinterpret_cast<const uint2*>(dbase + off);
          const uint2 ov = *reinterpret_cast<const uint2*>(obase + off);
          const float2 o01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov.x));
          const float2 o23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov.y));
          const float2 d01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dv.x));
          const float2 d23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dv.y));
          const float acc = fmaf(o01.x, d01.x, fmaf(o01.y, d01.y, fmaf(o23.x, d23.x, o23.y * d23.y)));
          part[rr] = rr < nvalid ? acc : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_o_read);  // the O entry's slot may be refilled
        ++kk;
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const int k = 16 >> st;  // lanes with bit k keep the upper half of the rows
          const bool up = (lane & k) != 0;
#pragma unroll
          for (int j = 0; j < (8 >> st); ++j) {
            const float send = up ? part[j] : part[j + (8 >> st)];
            const float keep = up ? part[j + (8 >> st)] : part[j];
            part[j] = keep + __shfl_xor_sync(0xffffffffu, send, k);
          }
        }
        part[0] += __shfl_xor_sync(0xffffffffu, part[0], 1);
        float* sd = reinterpret_cast<float*>(smem + kDqOffDelta + (qn & 1) * 512) + quarter * 32;
        if ((lane & 1) == 0) sd[half * 16 + (lane >> 1)] = part[0];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_delta[quarter]);
        if (!(ok = warp_wait(&bar_delta[quarter], qn & 1, abort, p.status))) break;
        ndelta = -sd[lane];
        nlse2 = -(lse_pre * kLog2e);
      }
      if (half == 0) {
        p.delta[static_cast<size_t>(h) * p.Npad + i] = ndelta;
        p.lse2[static_cast<size_t>(h) * p.Npad + i] = nlse2;
      }
      ++qn;
      if (nt_at != beg) fetch_tile(beg);
      for (int t = beg; t < end; ++t, ++n, ++kk) {
        const int kd = nt_kind & 3, tile_arow = nt_arow;
        const bool tile_gw = (nt_kind >> 4) & 1;  // gateway keys precede every row
        if (t + 1 < end) fetch_tile(t + 1);
        // What this warp's 32 rows x 64 keys of the tile hold: 1 every pair
        // visible (no mask), 0 a mix (mask per element; the key <= i half only
        // where some key may follow a row), 2 no visible pair (P = dS = 0: no
        // exponentials, no dP read).
        int mode = kd == 2 ? 1 : 0;
        bool diag = false;
        const int* ke = nullptr;
        int arow[8];  // first key of each atom of this half (column c: arow[c/8] + c%8)
        if (kd == 1) {  // PARTIAL: the tile's key bounds arrived with its K stage
          // (the stage is refilled only after this tile's dQ product, which
          // waits for every softmax thread's dS)
          if (!(ok = warp_wait(&bar_k_full[kk % kDqKStages], (kk / kDqKStages) & 1, abort, p.status)))
            break;
          ke = reinterpret_cast<const int*>(smem + kDqOffKe + (kk % kDqKStages) * 512) + col0;
          int mn = min(ke[lane], ke[lane + 32]), mx = max(ke[lane], ke[lane + 32]);
          // this half's atoms are lanes 8*half .. 8*half+7 of the atom word
          const bool mine = (lane & 15) >> 3 == half;
          int amax = mine ? tile_arow : -8;
          int amin = mine && tile_arow >= 0 ? tile_arow : 0x7fffffff;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            amin = min(amin, __shfl_xor_sync(0xffffffffu, amin, o));
          }
#pragma unroll
          for (int a = 0; a < 8; ++a) arow[a] = __shfl_sync(0xffffffffu, tile_arow, half * 8 + a);
          const int r0 = qt * 128 + quarter * 32;
          // rows [r0, r0+32) see key j iff j <= row < key_end[j]; gateway
          // keys come before every row, so only the key_end bound applies
          diag = !tile_gw && amax + 7 > r0;
          mode = (mx <= r0 || (!tile_gw && amin > r0 + 31)) ? 2 : (!diag && mn > r0 + 31) ? 1 : 0;
        }
        const int sb = (t - beg) & 1;
        const uint32_t tSb = tS + lane_off + sb * 128 + col0;
        if (!(ok = warp_wait(&bar_s_full[sb], (sb ? su1 : su0) & 1, abort, p.status))) break;
        su1 += sb ? 1u : 0u;
        su0 += sb ? 0u : 1u;
        tc_fence_after_sync();
        float pv[64];
        if (mode != 2) {
          uint32_t rr[64];
          tmem_ld64(tSb, rr);  // this half of the S row, one wait
          const float2 sc2 = make_float2(sl2, sl2), nl2 = make_float2(nlse2, nlse2);
#pragma unroll
          for (int jj = 0; jj < 64; jj += 2) {
            const float2 x = fma2(make_float2(__uint_as_float(rr[jj]), __uint_as_float(rr[jj + 1])), sc2, nl2);
            pv[jj] = ex2_approx(x.x);
            pv[jj + 1] = ex2_approx(x.y);
          }
        }
        if (mode == 0 && diag) {
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const int4 b = reinterpret_cast<const int4*>(ke)[c4];
            const int j = arow[c4 >> 1] + 4 * (c4 & 1);  // key of this half's column 4*c4
            if (!(j + 0 <= i && i < b.x)) pv[4 * c4 + 0] = 0.f;
            if (!(j + 1 <= i && i < b.y)) pv[4 * c4 + 1] = 0.f;
            if (!(j + 2 <= i && i < b.z)) pv[4 * c4 + 2] = 0.f;
            if (!(j + 3 <= i && i < b.w)) pv[4 * c4 + 3] = 0.f;
          }
        } else if (mode == 0) {  // every key of this half precedes every row of this warp
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const int4 b = reinterpret_cast<const int4*>(ke)[c4];
            if (!(i < b.x)) pv[4 * c4 + 0] = 0.f;
            if (!(i < b.y)) pv[4 * c4 + 1] = 0.f;
            if (!(i < b.z)) pv[4 * c4 + 2] = 0.f;
            if (!(i < b.w)) pv[4 * c4 + 3] = 0.f;
          }
        }
        if (!(ok = warp_wait(&bar_dp_full, n & 1, abort, p.status))) break;
        tc_fence_after_sync();
        if (mode == 2) {
          mbar_arrive(&bar_dp_read);  // nothing to read
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pk[jj] = 0u;
          tmem_st16(tSb, pk);
          tmem_st16(tSb + 16, pk);
        } else {
          uint32_t rr[64];
          tmem_ld64(tDP + lane_off + col0, rr);  // this half of the dP row, one wait
          tc_fence_before_sync();
          mbar_arrive(&bar_dp_read);  // the dP buffer may take dP_{t+1}
          const float2 nd2 = make_float2(ndelta, ndelta);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int col = c * 32 + 2 * jj;
              const float2 y = mul2(make_float2(pv[col], pv[col + 1]),
                                    add2(make_float2(__uint_as_float(rr[col]), __uint_as_float(rr[col + 1])),
                                         nd2));
              pk[jj] = pack_bf16x2(y.x, y.y);
            }
            tmem_st16(tSb + c * 16, pk);  // dS over the first 32 columns of this half
          }
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(sb ? &bar_ds_full1 : &bar_ds_full0);
      }
      if (!ok) break;
      if (!(ok = next_item(nxt))) break;
      // epilogue: dq = scale * dQ, this half's 64 columns. Once they are in
      // registers the accumulator is free for the next item; chunks are then
      // exchanged within lane groups (exchange_chunks) so each store
      // instruction writes whole 128- or 256-byte pieces of rows.
      if (!(ok = warp_wait(&bar_dq_full, (qn - 1) & 1, abort, p.status))) break;
      tc_fence_after_sync();
      {
        uint32_t v[64];
        tmem_ld64(tDQ + lane_off + col0, v);
        tc_fence_before_sync();
        mbar_arrive(&bar_dq_free);
        const int rq = qt * 128 + quarter * 32;  // the warp's first row
        if (!p.out_f32) {  // 4 chunks of 16 bf16 columns, groups of 4 lanes
          uint32_t pk[4][8];
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[c][e] = pack_bf16x2(__uint_as_float(v[16 * c + 2 * e]) * p.scale,
                                     __uint_as_float(v[16 * c + 2 * e + 1]) * p.scale);
          exchange_chunks<4>(pk, lane);
          const int i0 = rq + (lane & ~3), pos = lane & 3;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (i0 + k >= p.N) continue;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dq) +
                                 (static_cast<size_t>(i0 + k) * p.hq + h) * 128 + col0 + 16 * pos;
            store32(dst, pk[k], p.out_v8);
          }
        } else {  // 8 chunks of 8 fp32 columns, groups of 8 lanes
          uint32_t pk[8][8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[c][e] = __float_as_uint(__uint_as_float(v[8 * c + e]) * p.scale);
          exchange_chunks<8>(pk, lane);
          const int i0 = rq + (lane & ~7), pos = lane & 7;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (i0 + k >= p.N) continue;
            float* dst = static_cast<float*>(p.dq) + (static_cast<size_t>(i0 + k) * p.hq + h) * 128 + col0 + 8 * pos;
            store32(dst, pk[k], p.out_v8);
          }
        }
      }
      if (nxt >= 0) fetch_tile(hdr[1]);  // the next item's first tile
      cur = nxt;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) sched_finish(p.sched);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ dK/dV kernel
// 384 threads: warp 0 TMA producer, warp 1 MMA issuer + TMEM owner, warps
// 4-11 one key row per thread, two warpgroups splitting the q columns (at the
// end of an item they store the dV and dK rows). TMEM: S^T | dP^T, then dS^T
// and P^T over it | dV | dK. Both products that need P^T and dS^T read them
// from TMEM, so no operand is written to shared memory.
// Q_n is read by S^T_n and, a step later, by dK_n, so Q is staged three deep;
// dO_n (with the step's lse and Delta) is released after dV_n, two deep.
constexpr int kKvThreads = 384;
constexpr uint32_t kKvRegsCtl = 72, kKvRegsSoftmax = 216;  // 128 x 72 + 256 x 216 = 384 x 168
static_assert(128 * kKvRegsCtl + 256 * kKvRegsSoftmax <= 384 * 168, "register split");
constexpr int kKvQStages = 3;
constexpr int kKvDoStages = 2;
constexpr uint32_t kKvOffK = 0;
constexpr uint32_t kKvOffV = kKvOffK + kTileBytes;
constexpr uint32_t kKvOffQ = kKvOffV + kTileBytes;
constexpr uint32_t kKvOffDO = kKvOffQ + kKvQStages * kTileBytes;
constexpr uint32_t kKvOffLse = kKvOffDO + kKvDoStages * kTileBytes;  // per dO stage: 128 fp32
constexpr uint32_t kKvOffDelta = kKvOffLse + kKvDoStages * 512;     // per dO stage: 128 fp32
constexpr uint32_t kKvOffBar = kKvOffDelta + kKvDoStages * 512;
constexpr uint32_t kKvNumBars = 20;
constexpr uint32_t kKvOffRing = kKvOffBar + kKvNumBars * 8 + 16;
constexpr uint32_t kKvSmem = kKvOffRing + sizeof(ItemRing);
static_assert(kKvSmem <= 232448, "shared memory budget");

struct KvParams {
  const int32_t* key_end;
  const int32_t* kt_qlo;
  const int32_t* kt_qhi;
  const int32_t* order;
  const int32_t* gw_kend;  // gateway keys: N if visible, else 0 (partition plans)
  const int32_t* gw_kt;    // gateway key tiles with a visible key
  float* past_dk;          // gateway gradients, accumulated in fp32
  float* past_dv;
  int n_gw, past_len, Tq;
  const float* lse2;   // [hq, Npad], -lse * log2(e) (from the dQ phase)
  const float* delta;  // [hq, Npad], -Delta
  void* dk;
  void* dv;
  int* status;
  SchedSlot* sched;
  int N, Npad, hq, hkv, group, n_items, out_f32;
  int out_v8;  // dk and dv are 32-byte aligned
  float scale, scale_log2;
};

struct KvItem {
  int kt, kvh, qlo, nq, steps, gw;  // gw: a tile of gateway keys (seen by every row)
};

// Items: the gateway key tiles first (they walk every q-tile), then the
// partition's own key tiles in the plan's order.
__device__ __forceinline__ KvItem decode_kv(const KvParams& p, int it) {
  KvItem x;
  const int u = it / p.hkv;
  x.kvh = it % p.hkv;
  if (u < p.n_gw) {
    x.gw = 1;
    x.kt = p.gw_kt[u];
    x.qlo = 0;
    x.nq = p.Tq;
  } else {
    x.gw = 0;
    x.kt = p.order[u - p.n_gw];
    x.qlo = p.kt_qlo[x.kt];
    x.nq = p.kt_qhi[x.kt] - x.qlo;
  }
  x.steps = x.nq * p.group;
  return x;
}

// Add 32 consecutive fp32 values of one 128-wide row, times `mul`, into dst.
__device__ __forceinline__ void accumulate_row(float* dst_base, size_t off, int c,
                                               const uint32_t (&v)[32], float mul) {
  float4* dst = reinterpret_cast<float4*>(dst_base + off + c * 32);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    float4 a = dst[u];
    a.x += __uint_as_float(v[4 * u + 0]) * mul;
    a.y += __uint_as_float(v[4 * u + 1]) * mul;
    a.z += __uint_as_float(v[4 * u + 2]) * mul;
    a.w += __uint_as_float(v[4 * u + 3]) * mul;
    dst[u] = a;
  }
}

__global__ void __launch_bounds__(kKvThreads, 1)
    tree_attn_bwd_dkdv_sm103(const __grid_constant__ CUtensorMap map_q,
                             const __grid_constant__ CUtensorMap map_k,
                             const __grid_constant__ CUtensorMap map_v,
                             const __grid_constant__ CUtensorMap map_do,
                             const __grid_constant__ CUtensorMap map_pk,
                             const __grid_constant__ CUtensorMap map_pv, const KvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (smem_u32(smem) & 1023u) {  // the layout needs a 1024-aligned base
    if (threadIdx.x == 0) atomicExch(p.status, 9);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kKvOffBar);
  uint64_t* bar_kv_full = bars + 0;
  uint64_t* bar_kv_empty = bars + 1;
  uint64_t* bar_q_full = bars + 2;    // [kKvQStages]
  uint64_t* bar_q_empty = bars + 5;   // [kKvQStages]
  uint64_t* bar_do_full = bars + 8;   // [kKvDoStages]
  uint64_t* bar_do_empty = bars + 10; // [kKvDoStages]
  uint64_t* bar_s_full = bars + 12;
  uint64_t* bar_dp_full = bars + 13;
  uint64_t* bar_ds_full = bars + 14;
  uint64_t* bar_dkdv_full = bars + 15;
  uint64_t* bar_dkdv_free = bars + 16;
  uint64_t* bar_final = bars + 17;
  uint64_t* bar_s_read = bars + 18;  // the softmax warps hold S^T_n in registers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kKvNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + kKvNumBars) + 1;
  ItemRing* ring = reinterpret_cast<ItemRing*>(smem + kKvOffRing);

  if (threadIdx.x == 0) {
    item_ring_init(ring, 9);  // consumers: the MMA warp and the 8 softmax warps
    mbar_init(bar_kv_full, 1);
    mbar_init(bar_kv_empty, 1);
    for (int s = 0; s < kKvQStages; ++s) {
      mbar_init(bar_q_full + s, 1);
      mbar_init(bar_q_empty + s, 1);
    }
    for (int s = 0; s < kKvDoStages; ++s) {
      mbar_init(bar_do_full + s, 1);
      mbar_init(bar_do_empty + s, 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_ds_full, 256);
    mbar_init(bar_dkdv_full, 1);
    mbar_init(bar_dkdv_free, 256);
    mbar_init(bar_final, 1);
    mbar_init(bar_s_read, 256);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_do);
    if (p.n_gw > 0) {
      tma_prefetch_desc(&map_pk);
      tma_prefetch_desc(&map_pv);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tA = tmem, tB = tmem + 128, tC = tmem + 256, tD = tmem + 384;

  if (warp == 0) {
    regs_dec<kKvRegsCtl>();
    // ------------------------------------------------------------ producer
    uint32_t n = 0, items = 0, pub = 0;
    // The next item is taken once every load of this one is issued: items
    // differ in length by two orders of magnitude, and taking one early can
    // leave two long ones on one CTA while the others finish.
    int cur = item_fetch(p.sched, p.n_items);
    bool ok = item_put(ring, pub, cur, abort, p.status);
    while (ok && cur >= 0) {
      const KvItem x = decode_kv(p, cur);
      if (items > 0 && !(ok = warp_wait(bar_kv_empty, (items - 1) & 1, abort, p.status))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_kv_full, 2 * kTileBytes);
        const int row0 = x.kt * 128;
        const CUtensorMap* mk = x.gw ? &map_pk : &map_k;
        const CUtensorMap* mv = x.gw ? &map_pv : &map_v;
        tma_load_3d(smem + kKvOffK, mk, bar_kv_full, 0, x.kvh, row0);
        tma_load_3d(smem + kKvOffK + kHalfBytes, mk, bar_kv_full, 64, x.kvh, row0);
        tma_load_3d(smem + kKvOffV, mv, bar_kv_full, 0, x.kvh, row0);
        tma_load_3d(smem + kKvOffV + kHalfBytes, mv, bar_kv_full, 64, x.kvh, row0);
      }
      __syncwarp();
      for (int j = 0; j < x.steps; ++j, ++n) {
        // q-tile major, the group's heads inner: the CTAs that share a key
        // prefix walk the same q-tiles a fixed distance apart, so the Q and dO
        // tiles they all read stay in L2 between them
        const int qt = x.qlo + j / p.group;
        const int h = x.kvh * p.group + j % p.group;
        const uint32_t sq = n % kKvQStages, pq = (n / kKvQStages) & 1;
        if (n >= kKvQStages && !(ok = warp_wait(bar_q_empty + sq, pq ^ 1, abort, p.status))) break;
        if (lane == 0) {
          uint8_t* q = smem + kKvOffQ + sq * kTileBytes;
          mbar_arrive_expect_tx(bar_q_full + sq, kTileBytes);
          tma_load_3d(q, &map_q, bar_q_full + sq, 0, h, qt * 128);
          tma_load_3d(q + kHalfBytes, &map_q, bar_q_full + sq, 64, h, qt * 128);
        }
        __syncwarp();
        const uint32_t sd = n % kKvDoStages, pd = (n / kKvDoStages) & 1;
        if (n >= kKvDoStages && !(ok = warp_wait(bar_do_empty + sd, pd ^ 1, abort, p.status))) break;
        if (lane == 0) {
          uint64_t* b = bar_do_full + sd;
          uint8_t* d = smem + kKvOffDO + sd * kTileBytes;
          mbar_arrive_expect_tx(b, kTileBytes + 1024);
          tma_load_3d(d, &map_do, b, 0, h, qt * 128);
          tma_load_3d(d + kHalfBytes, &map_do, b, 64, h, qt * 128);
          const size_t off = static_cast<size_t>(h) * p.Npad + qt * 128;
          bulk_load(smem + kKvOffLse + sd * 512, p.lse2 + off, 512, b);
          bulk_load(smem + kKvOffDelta + sd * 512, p.delta + off, 512, b);
        }
        __syncwarp();
      }
      if (!ok) break;
      ++items;
      cur = item_fetch(p.sched, p.n_items);
      if (!(ok = item_put(ring, pub, cur, abort, p.status))) break;
      if (cur >= 0 && lane == 0) {  // its K and V into L2 while this item finishes
        const KvItem y = decode_kv(p, cur);
        const CUtensorMap* mk = y.gw ? &map_pk : &map_k;
        const CUtensorMap* mv = y.gw ? &map_pv : &map_v;
        tma_prefetch_l2_3d(mk, 0, y.kvh, y.kt * 128);
        tma_prefetch_l2_3d(mk, 64, y.kvh, y.kt * 128);
        tma_prefetch_l2_3d(mv, 0, y.kvh, y.kt * 128);
        tma_prefetch_l2_3d(mv, 64, y.kvh, y.kt * 128);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      if (items > 0) mbar_drain(bar_kv_full, (items - 1) & 1);
      for (uint32_t i = n >= kKvQStages ? n - kKvQStages : 0; i <= n; ++i) {
        mbar_drain(bar_q_full + i % kKvQStages, (i / kKvQStages) & 1);
        mbar_drain(bar_do_full + i % kKvDoStages, (i / kKvDoStages) & 1);
      }
    }
  } else if (warp == 1) {
    regs_dec<kKvRegsCtl>();
    // ---------------------------------------------------------- MMA issuer
    // Per step n (S^T_n and dP^T_n already issued):
    //   [S^T_n read] S^T_{n+1};  [dS_n] dV += P^T_n dO_n, dK += dS^T_n Q_n, dP^T_{n+1}
    // P^T_n and dS^T_n both sit in the dP^T buffer, so the S^T buffer is free
    // as soon as the softmax warps have S^T_n in registers, and S^T_{n+1}
    // runs while they compute P_n and dS_n.
    const uint32_t aK = smem_u32(smem + kKvOffK), aV = smem_u32(smem + kKvOffV);
    auto q_addr = [&](uint32_t i) { return smem_u32(smem + kKvOffQ + (i % kKvQStages) * kTileBytes); };
    auto do_addr = [&](uint32_t i) { return smem_u32(smem + kKvOffDO + (i % kKvDoStages) * kTileBytes); };
    auto wait_q = [&](uint32_t i) {
      return warp_wait(bar_q_full + i % kKvQStages, (i / kKvQStages) & 1, abort, p.status);
    };
    auto wait_do = [&](uint32_t i) {
      return warp_wait(bar_do_full + i % kKvDoStages, (i / kKvDoStages) & 1, abort, p.status);
    };
    uint32_t n = 0, items = 0, got = 0;
    bool ok = true;
    for (int cur; (ok = item_get(ring, got, cur, abort, p.status)) && cur >= 0; ++items) {
      const KvItem x = decode_kv(p, cur);
      if (!(ok = warp_wait(bar_kv_full, items & 1, abort, p.status))) break;
      for (int j = 0; j < x.steps; ++j, ++n) {
        if (j == 0) {
          if (!(ok = wait_q(n))) break;
          tc_fence_after_sync();
          mma_kk(tA, aK, q_addr(n), 0);  // S^T = K Q^T
          mma_commit_warp(bar_s_full);
          if (!(ok = wait_do(n))) break;
          tc_fence_after_sync();
          mma_kk(tB, aV, do_addr(n), 0);  // dP^T = V dO^T
          mma_commit_warp(bar_dp_full);
        }
        const bool has_next = j + 1 < x.steps;
        if (has_next) {
          if (!(ok = warp_wait(bar_s_read, n & 1, abort, p.status))) break;
          if (!(ok = wait_q(n + 1))) break;
          tc_fence_after_sync();
          mma_kk(tA, aK, q_addr(n + 1), 0);  // next S^T
          mma_commit_warp(bar_s_full);
        }
        if (!(ok = warp_wait(bar_ds_full, n & 1, abort, p.status))) break;
        if (j == 0 && items > 0 &&
            !(ok = warp_wait(bar_dkdv_free, (items - 1) & 1, abort, p.status)))
          break;
        tc_fence_after_sync();
        mma_tn_split(tC, tB + 32, do_addr(n), j > 0);  // dV += P^T dO (P^T from TMEM)
        mma_commit_warp(bar_do_empty + n % kKvDoStages);
        mma_tn_split(tD, tB, q_addr(n), j > 0);  // dK += dS^T Q (dS^T from TMEM)
        mma_commit_warp(bar_q_empty + n % kKvQStages);
        if (has_next) {
          if (!(ok = wait_do(n + 1))) break;
          tc_fence_after_sync();
          mma_kk(tB, aV, do_addr(n + 1), 0);  // next dP^T (dS^T_n already read by dK)
          mma_commit_warp(bar_dp_full);
        }
      }
      if (!ok) break;
      mma_commit_warp(bar_dkdv_full);
      mma_commit_warp(bar_kv_empty);
    }
    mma_commit_warp(bar_final);
    mbar_drain(bar_final, 0);
  } else if (warp < 4) {
    regs_dec<kKvRegsCtl>();  // warps 2-3: idle
  } else {
    regs_inc<kKvRegsSoftmax>();
    // ---- two warpgroups split each step's 128 q columns: warps 4-7 take
    // columns 0-63, warps 8-11 columns 64-127; one key row per thread. Each
    // half reads its S^T columns (then releases the S^T buffer) and its dP^T
    // columns, and writes dS^T over the first 32 and P^T over the second 32
    // of its own dP^T columns. At the end of an item each half stores its 64
    // columns of dV and dK.
    const int half = (warp - 4) / 4;
    const int quarter = warp % 4;
    const int kr = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = half * 64;
    const uint32_t tSr = tA + lane_off + col0, tPr = tB + lane_off + col0;
    const float sl2 = p.scale_log2;
    uint32_t n = 0, items = 0, got = 0;
    bool ok = true;
    for (int cur; (ok = item_get(ring, got, cur, abort, p.status)) && cur >= 0; ++items) {
      const KvItem x = decode_kv(p, cur);
      // rows [jk, ke) see this key; a gateway key comes before every row and is
      // seen by all of them if visible (ke = N), by none otherwise (ke = 0)
      const int krow = x.kt * 128 + kr;
      const int jk = x.gw ? -1 : krow;
      const int ke = x.gw ? __ldg(p.gw_kend + krow) : (krow < p.N ? __ldg(p.key_end + krow) : 0);
      for (int j = 0; j < x.steps; ++j, ++n) {
        const int q0 = (x.qlo + j / p.group) * 128 + col0;  // first q column of this half
        const uint32_t sd = n % kKvDoStages, pd = (n / kKvDoStages) & 1;
        const float* nlse2 = reinterpret_cast<const float*>(smem + kKvOffLse + sd * 512) + col0;
        const float* ndlt = reinterpret_cast<const float*>(smem + kKvOffDelta + sd * 512) + col0;
        if (!(ok = warp_wait(bar_do_full + sd, pd, abort, p.status))) break;
        if (!(ok = warp_wait(bar_s_full, n & 1, abort, p.status))) break;
        tc_fence_after_sync();
        // every column of this half visible to every key of this warp: no mask
        const bool all_full = __all_sync(0xffffffffu, jk <= q0 && q0 + 64 <= ke);
        float pv[64];
        {
          uint32_t rr[64];
          tmem_ld64(tSr, rr);  // this half of the S^T row, one wait
          tc_fence_before_sync();
          mbar_arrive(bar_s_read);  // the S^T buffer may take the next S^T
          // P^T = 2^(S^T * scale * log2e - lse * log2e); the workspace holds
          // -lse * log2e, so each column pair is one packed fma
          const float2 sc2 = make_float2(sl2, sl2);
#pragma unroll
          for (int jj = 0; jj < 64; jj += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + jj);
            const float2 x01 = fma2(make_float2(__uint_as_float(rr[jj + 0]), __uint_as_float(rr[jj + 1])),
                                    sc2, make_float2(l4.x, l4.y));
            const float2 x23 = fma2(make_float2(__uint_as_float(rr[jj + 2]), __uint_as_float(rr[jj + 3])),
                                    sc2, make_float2(l4.z, l4.w));
            pv[jj + 0] = ex2_approx(x01.x);
            pv[jj + 1] = ex2_approx(x01.y);
            pv[jj + 2] = ex2_approx(x23.x);
            pv[jj + 3] = ex2_approx(x23.y);
          }
          if (!all_full) {
#pragma unroll
            for (int jj = 0; jj < 64; ++jj) {
              const int q = q0 + jj;
              if (!(jk <= q && q < ke)) pv[jj] = 0.f;
            }
          }
        }
        if (!(ok = warp_wait(bar_dp_full, n & 1, abort, p.status))) break;
        tc_fence_after_sync();
        {
          uint32_t rr[64];
          tmem_ld64(tPr, rr);  // this half of the dP^T row, one wait
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              pk[jj] = pack_bf16x2(pv[c * 32 + 2 * jj], pv[c * 32 + 2 * jj + 1]);
            tmem_st16(tPr + 32 + c * 16, pk);  // P^T over the second 32 columns of this half
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
              const int col = c * 32 + jj;
              const float4 d4 = *reinterpret_cast<const float4*>(ndlt + col);  // -Delta
              const float2 y01 = mul2(make_float2(pv[col], pv[col + 1]),
                                      add2(make_float2(__uint_as_float(rr[col]), __uint_as_float(rr[col + 1])),
                                           make_float2(d4.x, d4.y)));
              const float2 y23 = mul2(make_float2(pv[col + 2], pv[col + 3]),
                                      add2(make_float2(__uint_as_float(rr[col + 2]), __uint_as_float(rr[col + 3])),
                                           make_float2(d4.z, d4.w)));
              pk[jj / 2] = pack_bf16x2(y01.x, y01.y);
              pk[jj / 2 + 1] = pack_bf16x2(y23.x, y23.y);
            }
            tmem_st16(tPr + c * 16, pk);  // dS^T over the first 32 columns of this half
          }
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bar_ds_full);
      }
      if (!ok) break;
      // ---- this item's dV and dK (scaled) from TMEM, this half's 64 columns
      if (!(ok = warp_wait(bar_dkdv_full, items & 1, abort, p.status))) break;
      tc_fence_after_sync();
      const size_t out = (static_cast<size_t>(krow) * p.hkv + x.kvh) * 128;
      const bool keep = x.gw ? krow < p.past_len : krow < p.N;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tC + lane_off + col0 + c * 32, v);
        if (keep) {
          if (x.gw)
            accumulate_row(p.past_dv, out, half * 2 + c, v, 1.f);
          else
            store_row(p.dv, out, half * 2 + c, v, 1.f, p.out_f32, p.out_v8);
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tD + lane_off + col0 + c * 32, v);
        if (keep) {
          if (x.gw)
            accumulate_row(p.past_dk, out, half * 2 + c, v, p.scale);
          else
            store_row(p.dk, out, half * 2 + c, v, p.scale, p.out_f32, p.out_v8);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(bar_dkdv_free);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) sched_finish(p.sched);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd_bf16(const AttnBwdArgs& a) {
  const tree_plan* pl = a.plan;
  const int N = pl->N, Npad = pl->Tq * 128;
  float* lse2 = static_cast<float*>(a.workspace);
  float* delta = lse2 + static_cast<size_t>(a.hq) * Npad;

  CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map(&mq, a.q, N, a.hq) || !make_tile_map(&mk, a.k, N, a.hkv) ||
      !make_tile_map(&mv, a.v, N, a.hkv) || !make_tile_map(&mdo, a.dout, N, a.hq))
    return cudaErrorInvalidValue;
  const int sms = sm_count();

  DqParams d;
  d.gq_ptr = pl->dev.gq_ptr;
  d.gt_kind = pl->dev.gt_kind;
  d.gt_atom = pl->dev.gt_atom;
  d.gt_bidx = pl->dev.gt_bidx;
  d.gt_bounds = pl->dev.gt_bounds;
  d.order = pl->dev.fwd_order;
  d.o = static_cast<const __nv_bfloat16*>(a.o);
  d.lse = a.lse;
  d.lse2 = lse2;
  d.delta = delta;
  d.dq = a.dq;
  d.status = a.status;
  d.sched = next_sched_slot();
  d.N = N;
  d.Npad = Npad;
  d.hq = a.hq;
  d.group = a.hq / a.hkv;
  d.n_items = pl->Tq * a.hq;
  d.out_f32 = a.grad_f32 ? 1 : 0;
  d.out_v8 = (reinterpret_cast<uintptr_t>(a.dq) & 31u) == 0;
  d.has_gateway = pl->past_len > 0 ? 1 : 0;
  d.scale = a.scale;
  d.scale_log2 = a.scale * kLog2e;

  KvParams k;
  k.key_end = pl->dev.key_end;
  k.kt_qlo = pl->dev.kt_qlo;
  k.kt_qhi = pl->dev.kt_qhi;
  k.order = pl->dev.bwd_order;
  k.gw_kend = pl->dev.gw_kend;
  k.gw_kt = pl->dev.gw_kt;
  k.past_dk = a.past_dk;
  k.past_dv = a.past_dv;
  k.n_gw = static_cast<int>(pl->field[TREE_FIELD_GW_KT].size());
  k.past_len = pl->past_len;
  k.Tq = pl->Tq;
  k.lse2 = lse2;
  k.delta = delta;
  k.dk = a.dk;
  k.dv = a.dv;
  k.status = a.status;
  k.sched = next_sched_slot();
  if (!d.sched || !k.sched) return cudaErrorInvalidDevicePointer;
  k.N = N;
  k.Npad = Npad;
  k.hq = a.hq;
  k.hkv = a.hkv;
  k.group = a.hq / a.hkv;
  k.n_items = (pl->Tk + k.n_gw) * a.hkv;
  k.out_f32 = a.grad_f32 ? 1 : 0;
  k.out_v8 = ((reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 31u) == 0;
  k.scale = a.scale;
  k.scale_log2 = a.scale * kLog2e;

  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tree_attn_bwd_dq_sm103,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tree_attn_bwd_dkdv_sm103,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (a.phases & 1) {
    CUtensorMap mo;
    GatherMaps gk, gv, gpk, gpv;
    if (!make_tile_map(&mo, a.o, N, a.hq) || !make_gather_maps(&gk, a.k, N, a.hkv) ||
        !make_gather_maps(&gv, a.v, N, a.hkv))
      return cudaErrorInvalidValue;
    if (pl->past_len > 0) {
      if (!make_gather_maps(&gpk, a.past_k, pl->past_len, a.hkv) ||
          !make_gather_maps(&gpv, a.past_v, pl->past_len, a.hkv))
        return cudaErrorInvalidValue;
    } else {
      gpk = gk;
      gpv = gv;
    }
    tree_attn_bwd_dq_sm103<<<d.n_items < sms ? d.n_items : sms, kDqThreads, kDqSmem, a.stream>>>(
        mq, mk, mv, mdo, mo, gk, gv, gpk, gpv, d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!(a.phases & 2)) return cudaSuccess;
  CUtensorMap mpk = mk, mpv = mv;
  if (pl->past_len > 0 && (!make_tile_map(&mpk, a.past_k, pl->past_len, a.hkv) ||
                           !make_tile_map(&mpv, a.past_v, pl->past_len, a.hkv)))
    return cudaErrorInvalidValue;
  tree_attn_bwd_dkdv_sm103<<<k.n_items < sms ? k.n_items : sms, kKvThreads, kKvSmem, a.stream>>>(
      mq, mk, mv, mdo, mpk, mpv, k);
  return cudaGetLastError();
}

}  // namespace treeattn
