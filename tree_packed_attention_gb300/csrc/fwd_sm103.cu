// Forward tree attention, bf16 in / fp32 accumulate, on the sm_103a tensor
// cores (tcgen05.mma with TMEM accumulators, TMA-staged operands).
//
// What it computes ("Tree Training", arXiv 2511.00413, §3.2 "Attention Mask"
// and App. A.1): o_i = softmax over the keys visible to row i of scale*q_i.k_j,
// times v, and lse_i = log sum_j exp(scale*q_i.k_j). Key j is visible to row i
// iff j <= i < key_end[j]. Tiles with no visible pair are never loaded or
// multiplied (the plan lists only non-empty tiles, as the FlashMask kernel of
// App. A.1 skips masked blocks); FULL tiles skip the per-element mask.
//
// Key tiles are gathered: a work item's tiles hold the keys its rows see,
// the keys every row sees first, packed as runs of consecutive keys starting
// at multiples of 8 columns. A tile arrives as 16 TMA boxes of 8 key rows (one
// per 128B-swizzle atom, each landing where a 128-row box would put those
// rows), or as one 128-row box when its keys are consecutive. Column c holds
// key atom_row[c/8] + c%8; on a PARTIAL tile row i sees it iff
// key <= i < key_end[c] (key_end 0 for padding columns).
//
// CTA organisation (one persistent CTA per SM, 384 threads):
//   warp 0     TMA producer: the two Q tiles of a work item, then K/V tiles
//              into a 2-stage ring (128 keys x 128 dims each, 128B-swizzled);
//              a PARTIAL tile's 128 key bounds travel with its V tile.
//   warp 1     TMEM owner and MMA issuer (one thread issues tcgen05.mma).
//   warps 4-7  softmax for Q slot 0;  warps 8-11 softmax for Q slot 1.
// A work item is two 128-row Q tiles that share K/V: two q heads of one kv
// group at the same q-tile (grouped heads), or q-tiles 2p and 2p+1 of one
// head (else), walking the union of their tile lists.
//
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each. The softmax
// warps read S (one row per thread), write P = exp2(S*c - m) as bf16 over the
// first 64 columns of S, and the PV MMA reads P straight from TMEM. The MMA
// order per tile is PV_s(t) then S_s(t+1), so when S_s(t+1) is complete the
// previous PV into O_s is complete too and O_s may be rescaled in place.
// The running max is updated lazily: O and l are rescaled only when the max
// grows by more than 8 (log2 units), which keeps every P <= 2^8.
// The epilogue writes O / l as bf16 into a 16 KB staging tile per slot, 64
// columns at a time, and one thread of the slot stores it with TMA, so the
// softmax warps do not wait for the global stores.
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

constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 operand tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // its 64-column half (one TMA box)
// Shared memory (dynamic, 1024-byte aligned; no static shared variables, so
// the block starts aligned as the 128B-swizzled tiles need).
constexpr uint32_t kOffQ = 0;                                    // 2 slots
constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;               // kStages
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;         // kStages
constexpr uint32_t kStageBytes = kHalfBytes;                     // 128 rows x 64 columns bf16
constexpr uint32_t kOffStage = kOffV + kStages * kTileBytes;     // 2 slots
constexpr uint32_t kOffBounds = kOffStage + 2 * kStageBytes;     // per V stage: 128 key_end
constexpr uint32_t kOffBar = kOffBounds + kStages * 512;
constexpr uint32_t kNumBars = 3 + 4 * kStages + 6 * 2;
constexpr uint32_t kOffRing = kOffBar + kNumBars * 8;
constexpr uint32_t kOffMisc = kOffRing + sizeof(ItemRing);
constexpr uint32_t kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kRegsCtl = 72, kRegsSoftmax = 216;

struct FwdParams {
  const int32_t* list_ptr;   // item (q-tile or pair) -> its tiles in the gathered table
  const int32_t* gt_kind;    // per tile: kind of slot 0 | kind of slot 1 << 2 (pairs)
  const int32_t* gt_atom;    // per tile: first key row of each 8-column atom (-8: zeros)
  const int32_t* gt_bidx;    // per tile: row of its key bounds, -1 if not PARTIAL
  const int32_t* gt_bounds;  // per bounds row: key_end of each column
  const int32_t* order;
  float* lse;
  int* status;
  SchedSlot* sched;
  int N, hq, group, n_items, n_inner, mode, Tq;
  int has_gateway;   // the plan's tiles include gateway keys
  float scale_log2;  // softmax scale * log2(e)
};

struct Item {
  int qtile[2];
  int head[2];
  int kvh;
  int beg, end;
};

// mode 0: two heads of one kv group at one q-tile; mode 1: q-tiles 2p, 2p+1 of one head.
// hdr = {order entry (q-tile or pair), first and end of its tile list}: the
// producer reads it once and publishes it with the item number.
__device__ __forceinline__ Item decode_item(const FwdParams& p, int it, const int (&hdr)[3]) {
  Item x;
  const int inner = it % p.n_inner;
  if (p.mode == 0) {
    x.qtile[0] = x.qtile[1] = hdr[0];
    x.head[0] = 2 * inner;
    x.head[1] = 2 * inner + 1;
    x.kvh = (2 * inner) / p.group;
  } else {
    x.qtile[0] = 2 * hdr[0];
    x.qtile[1] = 2 * hdr[0] + 1;
    x.head[0] = x.head[1] = inner;
    x.kvh = inner / p.group;
  }
  x.beg = hdr[1];
  x.end = hdr[2];
  return x;
}

__device__ __forceinline__ void read_header(const FwdParams& p, int it, int (&hdr)[3]) {
  hdr[0] = __ldg(p.order + it / p.n_inner);
  hdr[1] = __ldg(p.list_ptr + hdr[0]);
  hdr[2] = __ldg(p.list_ptr + hdr[0] + 1);
}

// One tile of a slot's list as the softmax warps need it, loaded two tiles
// ahead: its kind for this slot and the first key of atom (lane % 16). A
// PARTIAL tile's key bounds come with its V stage.
struct TileInfo {
  int kind, arow, gw;  // gw: the tile holds gateway keys (past K/V, before every row)
};

__device__ __forceinline__ TileInfo load_tile(const FwdParams& p, int t, int s, int lane) {
  TileInfo x;
  const int k = ldg_pinned(p.gt_kind + t);
  x.kind = ((p.mode == 0 ? (k | (k << 2)) : k) >> (2 * s)) & 3;
  x.arow = ldg_pinned(p.gt_atom + 16 * t + (lane & 15));
  x.gw = (k >> 4) & 1;
  return x;
}


// (a wait that gives up records the line it was called from)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status, int line = __builtin_LINE()) {
  const bool ok = mbar_wait(bar, parity, abort, status, kSiteFwd + line);
  return __all_sync(0xffffffffu, ok);
}

// S = Q K^T over D = 128 (8 MMAs of K = 16); both operands K-major.
// Warp-collective: one elected lane issues.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
  const uint64_t qd = sdesc_sw128(q_addr, 16, 1024), kd = sdesc_sw128(k_addr, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss_warp(d_tmem, sdesc_advance(qd, off), sdesc_advance(kd, off), idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V: P (128 x 128 keys, bf16) from TMEM, V (keys x D) MN-major in smem.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
  const uint64_t vd = sdesc_sw128(v_addr, kHalfBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_warp(d_tmem, p_tmem + kk * 8, sdesc_advance(vd, kk * 2048), idesc,
                (accumulate || kk > 0) ? 1u : 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
    tree_attn_fwd_sm103(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ GatherMaps map_k,
                        const __grid_constant__ GatherMaps map_v,
                        const __grid_constant__ GatherMaps map_pk,
                        const __grid_constant__ GatherMaps map_pv,
                        const __grid_constant__ CUtensorMap map_o, const FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicExch(p.status, 9);
    return;
  }
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t& bar_q_full = bars[0];
  uint64_t& bar_q_empty = bars[1];
  uint64_t& bar_final = bars[2];
  uint64_t* bar_k_full = bars + 3;
  uint64_t* bar_k_empty = bar_k_full + kStages;
  uint64_t* bar_v_full = bar_k_empty + kStages;
  uint64_t* bar_v_empty = bar_v_full + kStages;
  uint64_t* bar_s_full = bar_v_empty + kStages;  // [2] per slot from here on
  uint64_t* bar_p_full = bar_s_full + 2;
  uint64_t* bar_o_full = bar_p_full + 2;
  uint64_t* bar_o_free = bar_o_full + 2;
  uint64_t* bar_stage_full = bar_o_free + 2;  // the slot's 128 threads wrote a staging half
  uint64_t* bar_stage_free = bar_stage_full + 2;  // its TMA store has read the staging tile
  ItemRing& ring = *reinterpret_cast<ItemRing*>(smem + kOffRing);
  uint32_t& tmem_base_s = *reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int& abort_s = *reinterpret_cast<int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort = &abort_s;

  if (threadIdx.x == 0) {
    item_ring_init(&ring, 9);  // consumers: the MMA warp and the 8 softmax warps
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_final, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_p_full[s], 128);
      mbar_init(&bar_o_full[s], 1);
      mbar_init(&bar_o_free[s], 128);
      mbar_init(&bar_stage_full[s], 128);
      mbar_init(&bar_stage_free[s], 1);
    }
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_o);
    for (int b = 0; b < 5; ++b) {
      tma_prefetch_desc(&map_k.box[b]);
      tma_prefetch_desc(&map_v.box[b]);
      if (p.has_gateway) {
        tma_prefetch_desc(&map_pk.box[b]);
        tma_prefetch_desc(&map_pv.box[b]);
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
  // Registers: launched with 168 a thread (384 x 168 = 64512); warps 0-3 give
  // theirs down to 72 and the two softmax warpgroups take 216:
  // 128 x 72 + 256 x 216 = 64512.
  static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * 168, "register split");

  if (warp == 0) {
    regs_dec<kRegsCtl>();
    // ------------------------------------------------------------ producer
    uint32_t kv = 0, qn = 0, pub = 0;
    // The next item is taken from the launch's counter once every load of
    // this one is issued, a couple of tiles before the CTA is free: taking it
    // earlier can leave two long items on one CTA while another sits idle.
    int hdr[3] = {0, 0, 0};
    int cur = item_fetch(p.sched, p.n_items);
    if (cur >= 0) read_header(p, cur, hdr);
    bool ok = item_put(&ring, pub, cur, abort, p.status, hdr[0], hdr[1], hdr[2]);
    while (ok && cur >= 0) {
      const Item x = decode_item(p, cur, hdr);
      if (qn > 0 && !(ok = warp_wait(&bar_q_empty, (qn - 1) & 1, abort, p.status))) break;
      if (lane == 0) {
        const uint32_t bytes = (x.qtile[1] < p.Tq ? 2u : 1u) * kTileBytes;
        mbar_arrive_expect_tx(&bar_q_full, bytes);
        for (int s = 0; s < 2; ++s) {
          if (x.qtile[s] >= p.Tq) continue;
          tma_load_3d(sQ + s * kTileBytes, &map_q, &bar_q_full, 0, x.head[s], x.qtile[s] * 128);
          tma_load_3d(sQ + s * kTileBytes + kHalfBytes, &map_q, &bar_q_full, 64, x.head[s],
                      x.qtile[s] * 128);
        }
      }
      __syncwarp();
      ++qn;
      // this lane's atom and the bounds row of the next tile, one tile ahead
      int arow_next = 0, bidx_next = -1, kind_next = 0;
      if (x.beg < x.end) {
        arow_next = ldg_pinned(p.gt_atom + 16 * x.beg + (lane & 15));
        bidx_next = ldg_pinned(p.gt_bidx + x.beg);
        kind_next = ldg_pinned(p.gt_kind + x.beg);
      }
      for (int t = x.beg; t < x.end; ++t, ++kv) {
        const int arow = arow_next, bidx = bidx_next;
        const bool gw = (kind_next >> 4) & 1;  // gateway keys: the past K/V tensors
        if (t + 1 < x.end) {
          arow_next = ldg_pinned(p.gt_atom + 16 * (t + 1) + (lane & 15));
          bidx_next = ldg_pinned(p.gt_bidx + t + 1);
          kind_next = ldg_pinned(p.gt_kind + t + 1);
        }
        const uint32_t st = kv % kStages, ph = (kv / kStages) & 1;
        if (kv >= kStages && !(ok = warp_wait(&bar_k_empty[st], ph ^ 1, abort, p.status))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar_k_full[st], kTileBytes);
        __syncwarp();
        load_gathered(sK + st * kTileBytes, gw ? map_pk : map_k, &bar_k_full[st], x.kvh, arow, lane);
        __syncwarp();
        if (kv >= kStages && !(ok = warp_wait(&bar_v_empty[st], ph ^ 1, abort, p.status))) break;
        if (lane == 0) {
          // a PARTIAL tile's key bounds travel with its V tile: the stage is
          // refilled only after the tile's PV products, which wait for P
          mbar_arrive_expect_tx(&bar_v_full[st], kTileBytes + (bidx >= 0 ? 512u : 0u));
          if (bidx >= 0)
            bulk_load(smem + kOffBounds + st * 512, p.gt_bounds + static_cast<size_t>(bidx) * 128,
                      512, &bar_v_full[st]);
        }
        __syncwarp();
        load_gathered(sV + st * kTileBytes, gw ? map_pv : map_v, &bar_v_full[st], x.kvh, arow, lane);
        __syncwarp();
      }
      if (!ok) break;
      cur = item_fetch(p.sched, p.n_items);
      if (cur >= 0) read_header(p, cur, hdr);
      if (!(ok = item_put(&ring, pub, cur, abort, p.status, hdr[0], hdr[1], hdr[2]))) break;
      if (cur >= 0 && lane == 0) {  // its Q tiles into L2 while this item finishes
        const Item y = decode_item(p, cur, hdr);
        for (int s = 0; s < 2; ++s) {
          if (y.qtile[s] >= p.Tq) continue;
          tma_prefetch_l2_3d(&map_q, 0, y.head[s], y.qtile[s] * 128);
          tma_prefetch_l2_3d(&map_q, 64, y.head[s], y.qtile[s] * 128);
        }
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {  // let copies in flight land before the CTA exits
      if (qn > 0) mbar_drain(&bar_q_full, (qn - 1) & 1);
      for (uint32_t i = kv >= kStages ? kv - kStages : 0; i <= kv; ++i) {
        mbar_drain(&bar_k_full[i % kStages], (i / kStages) & 1);
        mbar_drain(&bar_v_full[i % kStages], (i / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    regs_dec<kRegsCtl>();
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this branch; one elected lane issues each MMA.
    uint32_t kv = 0, qn = 0, got = 0;
    uint32_t pc0 = 0, pc1 = 0, oc0 = 0, oc1 = 0;  // P and O phases per slot
    const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
    bool ok = true;
    int hdr[3];
    // Kinds of a tile for both slots (0 = no rows of the slot see it). With
    // grouped heads both slots hold the same rows and every listed tile has
    // a visible pair, so nothing is loaded; else they are read two tiles ahead.
    auto kinds_ahead = [&](int t) { return p.mode == 0 ? 5 : ldg_pinned(p.gt_kind + t); };
    for (int cur; (ok = item_get(&ring, got, cur, abort, p.status, hdr)) && cur >= 0;) {
      const Item x = decode_item(p, cur, hdr);
      const int T = x.end - x.beg;
      int kd_next = kinds_ahead(x.beg);                       // tile t
      int kd_next2 = T > 1 ? kinds_ahead(x.beg + 1) : 0;      // tile t + 1
      if (!(ok = warp_wait(&bar_q_full, qn & 1, abort, p.status))) break;
      ++qn;
      bool first0 = true, first1 = true;
      {  // S(0)
        const uint32_t st = kv % kStages, ph = (kv / kStages) & 1;
        if (!(ok = warp_wait(&bar_k_full[st], ph, abort, p.status))) break;
        tc_fence_after_sync();
        if (kd_next & 3) {
          issue_qk(tmem, q_addr, k_addr + st * kTileBytes);
          mma_commit_warp(&bar_s_full[0]);
        }
        if ((kd_next >> 2) & 3) {
          issue_qk(tmem + 128, q_addr + kTileBytes, k_addr + st * kTileBytes);
          mma_commit_warp(&bar_s_full[1]);
        }
        mma_commit_warp(&bar_k_empty[st]);
        if (T == 1) mma_commit_warp(&bar_q_empty);
      }
      for (int t = 0; t < T && ok; ++t) {
        const uint32_t kvt = kv + t;
        const uint32_t st = kvt % kStages, ph = (kvt / kStages) & 1;
        const uint32_t stn = (kvt + 1) % kStages, phn = ((kvt + 1) / kStages) & 1;
        const int kd = kd_next, kdn = kd_next2;
        kd_next = kd_next2;
        kd_next2 = t + 2 < T ? kinds_ahead(x.beg + t + 2) : 0;
        const bool has_next = t + 1 < T;
        if (!(ok = warp_wait(&bar_v_full[st], ph, abort, p.status))) break;
        // slot 0: PV(t), then S(t+1); slot 1 likewise
        if (kd & 3) {
          if (!(ok = warp_wait(&bar_p_full[0], pc0 & 1, abort, p.status))) break;
          ++pc0;
          if (first0 && oc0 > 0 && !(ok = warp_wait(&bar_o_free[0], (oc0 - 1) & 1, abort, p.status)))
            break;
          tc_fence_after_sync();
          issue_pv(tmem + 256, tmem, v_addr + st * kTileBytes, !first0);
          first0 = false;
        }
        if (!has_next && x.qtile[0] < p.Tq) {  // slot 0's O is final once this PV completes
          mma_commit_warp(&bar_o_full[0]);
          ++oc0;
        }
        if (has_next) {
          if (!(ok = warp_wait(&bar_k_full[stn], phn, abort, p.status))) break;
          tc_fence_after_sync();
          if (kdn & 3) {
            issue_qk(tmem, q_addr, k_addr + stn * kTileBytes);
            mma_commit_warp(&bar_s_full[0]);
          }
        }
        if ((kd >> 2) & 3) {
          if (!(ok = warp_wait(&bar_p_full[1], pc1 & 1, abort, p.status))) break;
          ++pc1;
          if (first1 && oc1 > 0 && !(ok = warp_wait(&bar_o_free[1], (oc1 - 1) & 1, abort, p.status)))
            break;
          tc_fence_after_sync();
          issue_pv(tmem + 384, tmem + 128, v_addr + st * kTileBytes, !first1);
          first1 = false;
        }
        if (!has_next && x.qtile[1] < p.Tq) {
          mma_commit_warp(&bar_o_full[1]);
          ++oc1;
        }
        if (has_next && ((kdn >> 2) & 3)) {
          issue_qk(tmem + 128, q_addr + kTileBytes, k_addr + stn * kTileBytes);
          mma_commit_warp(&bar_s_full[1]);
        }
        mma_commit_warp(&bar_v_empty[st]);
        if (has_next) mma_commit_warp(&bar_k_empty[stn]);
        if (t + 2 == T) mma_commit_warp(&bar_q_empty);  // the item's last S MMAs were just issued
      }
      if (!ok) break;
      kv += T;
    }
    mma_commit_warp(&bar_final);  // every MMA issued by this CTA completes before TMEM is freed
    if (lane == 0) mbar_drain(&bar_final, 0);
    __syncwarp();
  } else if (warp < 4) {
    regs_dec<kRegsCtl>();  // warps 2-3: idle
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------- softmax
    const int s = (warp - 4) / 4;
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + s * 128;
    const uint32_t tO = tmem + lane_off + 256 + s * 128;
    const float sl2 = p.scale_log2;
    const bool issuer = quarter == 0 && lane == 0;  // stores the slot's staging tile
    uint8_t* stage = smem + kOffStage + s * kStageBytes;
    uint32_t sc = 0, oc = 0, halves = 0;  // S and O phases; staging halves written
    uint32_t kvs = 0;                     // tiles so far (the V ring's counter)
    bool ok = true;
    // The next item's header is read one item ahead, and the kind and atom of
    // each tile two tiles ahead, so no global load latency sits between two
    // softmax passes.
    int n_qt = 0, n_h = 0, n_beg = 0, n_end = 0;  // next item: q-tile, head, tile range
    int hdr[3];
    auto fetch_header = [&](int at) {
      const Item y = decode_item(p, at, hdr);
      n_qt = y.qtile[s];
      n_h = y.head[s];
      n_beg = y.beg;
      n_end = y.end;
    };
    // The next item's number and header are read from the ring once this
    // item's tiles are done (the producer publishes them when this item's
    // loads are issued); its first tiles' loads overlap this epilogue.
    uint32_t got = 0;
    int cur = -1;
    ok = item_get(&ring, got, cur, abort, p.status, hdr);
    if (ok && cur >= 0) fetch_header(cur);
    TileInfo nt{}, nn{};  // tiles t+1 and t+2 of the walk
    int nt_at = -1;
    while (ok && cur >= 0) {
      const int qt = n_qt, h = n_h, beg = n_beg, end = n_end;
      int nxt = -1;
      if (qt >= p.Tq) {  // this slot has no rows in the item
        kvs += end - beg;
        if ((ok = item_get(&ring, got, nxt, abort, p.status, hdr)) && nxt >= 0) fetch_header(nxt);
        cur = nxt;
        continue;
      }
      const int i = qt * 128 + r;
      float m_ref = -INFINITY, l = 0.f;
      if (nt_at != beg) {
        nt = load_tile(p, beg, s, lane);
        if (beg + 1 < end) nn = load_tile(p, beg + 1, s, lane);
      }
      for (int t = beg; t < end; ++t, ++kvs) {
        const TileInfo tl = nt;
        nt = nn;
        nt_at = t + 1;
        if (t + 2 < end) nn = load_tile(p, t + 2, s, lane);
        const int kd = tl.kind;
        if (kd == 0) continue;
        // What this warp's 32 rows of the tile hold: 1 every pair visible (no
        // mask), 0 a mix (mask per element; the key <= i half only where some
        // key may follow a row), 2 no visible pair (P = 0, no exponentials).
        int mode = kd == 2 ? 1 : 0;
        bool diag = false;
        const int* ke = nullptr;
        int arow[16];  // first key of each atom (column c holds arow[c/8] + c%8)
        int amax = 0, amin = 0;
        if (kd == 1) {
          // over the atoms that hold keys: the largest first key (keys reach
          // at most 7 past it) and the smallest
          amax = tl.arow;
          amin = tl.arow >= 0 ? tl.arow : 0x7fffffff;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            amin = min(amin, __shfl_xor_sync(0xffffffffu, amin, o));
          }
#pragma unroll
          for (int a = 0; a < 16; ++a) arow[a] = __shfl_sync(0xffffffffu, tl.arow, a);
        }
        if (!(ok = warp_wait(&bar_s_full[s], sc & 1, abort, p.status))) break;
        ++sc;
        tc_fence_after_sync();
        if (kd == 1) {
          // PARTIAL: the key bounds arrived with the tile's V stage. Waited for
          // after S: S(t) was issued once the V loads of earlier tiles landed,
          // so this stage's barrier cannot still be a phase behind tile t.
          const uint32_t st = kvs % kStages, ph = (kvs / kStages) & 1;
          if (!(ok = warp_wait(&bar_v_full[st], ph, abort, p.status))) break;
          ke = reinterpret_cast<const int*>(smem + kOffBounds + st * 512);
          const int4 kq = reinterpret_cast<const int4*>(ke)[lane];  // columns 4*lane .. +3
          int mn = min(min(kq.x, kq.y), min(kq.z, kq.w));
          int mx = max(max(kq.x, kq.y), max(kq.z, kq.w));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          }
          const int r0 = qt * 128 + quarter * 32;
          // rows [r0, r0+32) see key j iff j <= row < key_end[j]; gateway
          // keys come before every row, so only the key_end bound applies
          diag = !tl.gw && amax + 7 > r0;
          mode = (mx <= r0 || (!tl.gw && amin > r0 + 31)) ? 2 : (!diag && mn > r0 + 31) ? 1 : 0;
        }
        if (mode == 2) {  // P = 0; m and l of the row are unchanged
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pk[jj] = 0u;
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_st16(tS + c * 16, pk);
          tmem_wait_st();
          tc_fence_before_sync();
          mbar_arrive(&bar_p_full[s]);
          continue;
        }
        float sv[128];
        {
          uint32_t rr[128];
          tmem_ld128(tS, rr);  // the whole S row, one wait
#pragma unroll
          for (int jj = 0; jj < 128; ++jj) sv[jj] = __uint_as_float(rr[jj]);
        }
        if (mode == 0) {
          if (diag) {
#pragma unroll
            for (int c4 = 0; c4 < 32; ++c4) {
              const int4 b = reinterpret_cast<const int4*>(ke)[c4];
              const int j = arow[c4 >> 1] + 4 * (c4 & 1);  // key of column 4*c4
              if (!(j + 0 <= i && i < b.x)) sv[4 * c4 + 0] = -INFINITY;
              if (!(j + 1 <= i && i < b.y)) sv[4 * c4 + 1] = -INFINITY;
              if (!(j + 2 <= i && i < b.z)) sv[4 * c4 + 2] = -INFINITY;
              if (!(j + 3 <= i && i < b.w)) sv[4 * c4 + 3] = -INFINITY;
            }
          } else {  // every key of the tile precedes every row of this warp
#pragma unroll
            for (int c4 = 0; c4 < 32; ++c4) {
              const int4 b = reinterpret_cast<const int4*>(ke)[c4];
              if (!(i < b.x)) sv[4 * c4 + 0] = -INFINITY;
              if (!(i < b.y)) sv[4 * c4 + 1] = -INFINITY;
              if (!(i < b.z)) sv[4 * c4 + 2] = -INFINITY;
              if (!(i < b.w)) sv[4 * c4 + 3] = -INFINITY;
            }
          }
        }
        // row max: three-input maxima in 8 independent chains, then a tree
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = fmaxf(sv[u], sv[8 + u]);
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = max3f(m8[u], sv[c + u], sv[c + 8 + u]);
        const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                               fmaxf(m8[6], m8[7]));
        const float m_tile = mx * sl2;
        const float m_new = fmaxf(m_ref, m_tile);
        const bool rescale = (m_ref != -INFINITY) && (m_new > m_ref + kRescaleThreshold);
        const float f = rescale ? ex2_approx(m_ref - m_new) : 1.f;
        if (rescale) {
          l *= f;
          m_ref = m_new;
        } else if (m_ref == -INFINITY) {
          m_ref = m_new;  // first visible keys of this row (or still none)
        }
        const float mr = (m_ref == -INFINITY) ? 0.f : m_ref;
        // P = 2^(S * scale * log2e - m), the scaling in column pairs; the row
        // sum in two independent pair chains
        const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-mr, -mr);
        float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const float2 x = fma2(make_float2(sv[c * 32 + 2 * jj], sv[c * 32 + 2 * jj + 1]), sc2, nm2);
            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            rs2[jj & 1] = add2(rs2[jj & 1], pp);
            pk[jj] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st16(tS + c * 16, pk);
        }
        const float rs = (rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y);
        if (__any_sync(0xffffffffu, rescale)) {
          // O_s is quiescent: its last PV completed before this S did, and the
          // next PV waits for the P arrival below.
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t rr[32];
            tmem_ld32(tO + c * 32, rr);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) rr[jj] = __float_as_uint(__uint_as_float(rr[jj]) * f);
            tmem_st32(tO + c * 32, rr);
          }
        }
        l += rs;
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&bar_p_full[s]);
      }
      if (!ok) break;
      if (!(ok = item_get(&ring, got, nxt, abort, p.status, hdr))) break;
      if (nxt >= 0) {  // its header, and its first tiles' loads during this epilogue
        fetch_header(nxt);
        nt_at = n_beg;
        nt = load_tile(p, n_beg, s, lane);
        if (n_beg + 1 < n_end) nn = load_tile(p, n_beg + 1, s, lane);
      }
      // ---- epilogue: O / l as bf16 through the staging tile, 64 columns at
      // a time; the slot's first thread issues each half's TMA store (rows
      // past N are not written by it)
      if (!(ok = warp_wait(&bar_o_full[s], oc & 1, abort, p.status))) break;
      ++oc;
      tc_fence_after_sync();
      uint32_t ov[128];
      tmem_ld128(tO, ov);  // the whole O row, one wait
      tc_fence_before_sync();
      mbar_arrive(&bar_o_free[s]);  // O_s is in registers: the next item's PV may start
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float2 inv2 = make_float2(inv, inv);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf, ++halves) {
        // the store of the previous half has read the staging tile
        if (halves > 0 && !(ok = warp_wait(&bar_stage_free[s], (halves - 1) & 1, abort, p.status)))
          break;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row, 128B-swizzled
          const int col = hf * 64 + c * 8;
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 y = mul2(make_float2(__uint_as_float(ov[col + 2 * u]),
                                              __uint_as_float(ov[col + 2 * u + 1])), inv2);
            w4[u] = pack_bf16x2(y.x, y.y);
          }
          const uint4 w = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ (r & 7)) * 16)) = w;
        }
        fence_proxy_async_shared();
        mbar_arrive(&bar_stage_full[s]);
        if (issuer) {  // (a wait that gives up leaves the loop below, with the whole warp)
          ok = mbar_wait(&bar_stage_full[s], halves & 1, abort, p.status, kSiteFwd + __LINE__);
          if (ok) {
            tma_store_3d(&map_o, stage, hf * 64, h, qt * 128);
            bulk_commit_group();
            bulk_wait_group_read<0>();
            mbar_arrive(&bar_stage_free[s]);
          }
        }
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
      }
      if (!ok) break;
      if (i < p.N)
        p.lse[static_cast<size_t>(h) * p.N + i] =
            l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      cur = nxt;
    }
    if (issuer) bulk_wait_group<0>();  // every O store has landed
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

cudaError_t launch_fwd_bf16(const AttnArgs& a) {
  const tree_plan* pl = a.plan;
  CUtensorMap mq, mo;
  GatherMaps mk, mv, mpk, mpv;
  if (!make_tile_map(&mq, a.q, pl->N, a.hq) || !make_gather_maps(&mk, a.k, pl->N, a.hkv) ||
      !make_gather_maps(&mv, a.v, pl->N, a.hkv) || !make_tile_map(&mo, a.o, pl->N, a.hq))
    return cudaErrorInvalidValue;
  const bool gw = pl->past_len > 0;
  if (gw) {
    if (!make_gather_maps(&mpk, a.past_k, pl->past_len, a.hkv) ||
        !make_gather_maps(&mpv, a.past_v, pl->past_len, a.hkv))
      return cudaErrorInvalidValue;
  } else {
    mpk = mk;
    mpv = mv;
  }
  FwdParams p;
  const int G = a.hq / a.hkv;
  p.mode = (G >= 2 && G % 2 == 0) ? 0 : 1;
  p.gt_kind = pl->dev.gt_kind;
  p.gt_atom = pl->dev.gt_atom;
  p.gt_bidx = pl->dev.gt_bidx;
  p.gt_bounds = pl->dev.gt_bounds;
  if (p.mode == 0) {
    p.list_ptr = pl->dev.gq_ptr;
    p.order = pl->dev.fwd_order;
    p.n_inner = a.hq / 2;
    p.n_items = pl->Tq * p.n_inner;
  } else {
    p.list_ptr = pl->dev.gp_ptr;
    p.order = pl->dev.qp_order;
    p.n_inner = a.hq;
    p.n_items = pl->P * p.n_inner;
  }
  p.lse = a.lse;
  p.status = a.status;
  p.sched = next_sched_slot();
  if (!p.sched) return cudaErrorInvalidDevicePointer;
  p.N = pl->N;
  p.hq = a.hq;
  p.group = G;
  p.Tq = pl->Tq;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.has_gateway = gw ? 1 : 0;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tree_attn_fwd_sm103,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = p.n_items < sm_count() ? p.n_items : sm_count();
  tree_attn_fwd_sm103<<<grid, kThreads, kSmemBytes, a.stream>>>(mq, mk, mv, mpk, mpv, mo, p);
  return cudaGetLastError();
}

}  // namespace treeattn
