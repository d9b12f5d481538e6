// Backward tree attention, bf16 in / fp32 accumulate, on the sm_103a tensor
// cores. Three kernels:
//   1. preprocess: Delta_i = sum_d dO_id O_id and lse_i*log2(e) into padded
//      [hq, Tq*128] rows, and zeroing of the fp32 dQ accumulator;
//   2. main: one persistent CTA per SM; a work item is one 128-key tile of one
//      kv head ("KV-stationary"); it walks every q head of the group and every
//      q-tile that sees the key tile -- one contiguous range [kt_qlo, kt_qhi),
//      because the rows that see key j are exactly [j, key_end[j]);
//   3. finalize: dQ = scale * accumulator, converted to the gradient dtype.
//
// Per step (q-tile, q head) the main kernel computes, with S^T = K Q^T:
//   P^T  = exp2(S^T * scale*log2e - lse*log2e)  (masked to j <= i < key_end[j])
//   dP^T = V dO^T,  dS^T = P^T (dP^T - Delta)
//   dV += P^T dO,  dK += dS^T Q,  dQ^T = K^T dS^T (added to the fp32 accumulator)
// ("Tree Training", arXiv 2511.00413, §3.2 mask / App. A.1; the derivatives
// are the standard softmax-attention ones).
//
// Roles (384 threads): warp 0 TMA producer (K, V per item; Q, dO, lse, Delta
// per step into a 2-stage ring); warp 1 TMEM owner and MMA issuer; warps 4-7
// compute P^T (to TMEM, bf16) and dS^T (to shared memory, bf16, 128B-swizzled)
// with one key row per thread; warps 8-11 drain dQ^T from TMEM into the fp32
// accumulator (one head-dim row per thread, coalesced reductions) and write
// dK, dV at the end of an item.
// TMEM (512 columns): S^T/P^T | dP^T/dQ^T | dV | dK.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace treeattn {
namespace {

using namespace dev;

constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = 128 * 128 * 2;
constexpr uint32_t kHalfBytes = kTileBytes / 2;

// Dynamic shared memory layout (the base must be 1024-byte aligned).
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffQ = kOffV + kTileBytes;        // 2 stages
constexpr uint32_t kOffDO = kOffQ + 2 * kTileBytes;   // 2 stages
constexpr uint32_t kOffDS = kOffDO + 2 * kTileBytes;  // dS^T, 128 keys x 128 q
constexpr uint32_t kOffLse = kOffDS + kTileBytes;     // 2 stages x 128 fp32
constexpr uint32_t kOffDelta = kOffLse + 2 * 512;     // 2 stages x 128 fp32
constexpr uint32_t kOffBar = kOffDelta + 2 * 512;
constexpr uint32_t kNumBars = 16;
constexpr uint32_t kSmemBytes = kOffBar + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct BwdParams {
  const int32_t* key_end;
  const int32_t* kt_qlo;
  const int32_t* kt_qhi;
  const int32_t* order;
  const float* lse2;   // [hq, Npad]
  const float* delta;  // [hq, Npad]
  float* dq_acc;       // [N, hq, 128]
  void* dk;
  void* dv;
  int* status;
  int N, Npad, hq, hkv, group, n_items, grad_f32;
  float scale, scale_log2;
};

struct BwdItem {
  int kt, kvh, qlo, nq, steps;
};

__device__ __forceinline__ BwdItem decode_bwd(const BwdParams& p, int it) {
  BwdItem x;
  x.kt = p.order[it / p.hkv];
  x.kvh = it % p.hkv;
  x.qlo = p.kt_qlo[x.kt];
  x.nq = p.kt_qhi[x.kt] - x.qlo;
  x.steps = x.nq * p.group;
  return x;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  const bool ok = mbar_wait(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

// D = A B^T with A [128 x 128] K-major and B [128 x 128] K-major (K = 128).
__device__ __forceinline__ void mma_kk(uint32_t d, uint32_t a, uint32_t b, uint32_t acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss(d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc,
           (acc || kk > 0) ? 1u : 0u);
  }
}

// D = A B^T with A K-major and B MN-major (B stored K rows x N contiguous).
__device__ __forceinline__ void mma_kn(uint32_t d, uint32_t a, uint32_t b, uint32_t acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss(d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + kk * 2048, kHalfBytes, 1024), idesc,
           (acc || kk > 0) ? 1u : 0u);
  }
}

// D = A B^T with A from TMEM (bf16 pairs) and B MN-major.
__device__ __forceinline__ void mma_tn(uint32_t d, uint32_t a_tmem, uint32_t b, uint32_t acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d, a_tmem + kk * 8, sdesc_sw128(b + kk * 2048, kHalfBytes, 1024), idesc,
           (acc || kk > 0) ? 1u : 0u);
}

// D = A B^T with A MN-major (stored K rows x M contiguous) and B MN-major.
__device__ __forceinline__ void mma_nn(uint32_t d, uint32_t a, uint32_t b, uint32_t acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 1, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ss(d, sdesc_sw128(a + kk * 2048, kHalfBytes, 1024),
           sdesc_sw128(b + kk * 2048, kHalfBytes, 1024), idesc, (acc || kk > 0) ? 1u : 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
    tree_attn_bwd_sm103(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (smem_u32(smem) & 1023u) {  // the layout needs a 1024-aligned base
    if (threadIdx.x == 0) atomicExch(p.status, 9);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_kv_full = bars + 0;
  uint64_t* bar_kv_empty = bars + 1;
  uint64_t* bar_qdo_full = bars + 2;   // [2]
  uint64_t* bar_qdo_empty = bars + 4;  // [2]
  uint64_t* bar_s_full = bars + 6;
  uint64_t* bar_dp_full = bars + 7;
  uint64_t* bar_ds_full = bars + 8;
  uint64_t* bar_dq_full = bars + 9;
  uint64_t* bar_dq_free = bars + 10;
  uint64_t* bar_dkdv_full = bars + 11;
  uint64_t* bar_dkdv_free = bars + 12;
  uint64_t* bar_final = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + kNumBars) + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv_full, 1);
    mbar_init(bar_kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qdo_full + s, 1);
      mbar_init(bar_qdo_empty + s, 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_ds_full, 128);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_free, 128);
    mbar_init(bar_dkdv_full, 1);
    mbar_init(bar_dkdv_free, 128);
    mbar_init(bar_final, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_do);
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
    // ------------------------------------------------------------ producer
    uint32_t n = 0, items = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++items) {
      const BwdItem x = decode_bwd(p, it);
      if (items > 0 && !(ok = warp_wait(bar_kv_empty, (items - 1) & 1, abort, p.status))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_kv_full, 2 * kTileBytes);
        const int row0 = x.kt * 128;
        tma_load_3d(smem + kOffK, &map_k, bar_kv_full, 0, x.kvh, row0);
        tma_load_3d(smem + kOffK + kHalfBytes, &map_k, bar_kv_full, 64, x.kvh, row0);
        tma_load_3d(smem + kOffV, &map_v, bar_kv_full, 0, x.kvh, row0);
        tma_load_3d(smem + kOffV + kHalfBytes, &map_v, bar_kv_full, 64, x.kvh, row0);
      }
      __syncwarp();
      for (int j = 0; j < x.steps; ++j, ++n) {
        const int h = x.kvh * p.group + j / x.nq;
        const int qt = x.qlo + j % x.nq;
        const uint32_t st = n & 1, ph = (n >> 1) & 1;
        if (n >= 2 && !(ok = warp_wait(bar_qdo_empty + st, ph ^ 1, abort, p.status))) break;
        if (lane == 0) {
          uint64_t* b = bar_qdo_full + st;
          mbar_arrive_expect_tx(b, 2 * kTileBytes + 1024);
          uint8_t* q = smem + kOffQ + st * kTileBytes;
          uint8_t* d = smem + kOffDO + st * kTileBytes;
          tma_load_3d(q, &map_q, b, 0, h, qt * 128);
          tma_load_3d(q + kHalfBytes, &map_q, b, 64, h, qt * 128);
          tma_load_3d(d, &map_do, b, 0, h, qt * 128);
          tma_load_3d(d + kHalfBytes, &map_do, b, 64, h, qt * 128);
          const size_t off = static_cast<size_t>(h) * p.Npad + qt * 128;
          bulk_load(smem + kOffLse + st * 512, p.lse2 + off, 512, b);
          bulk_load(smem + kOffDelta + st * 512, p.delta + off, 512, b);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      if (items > 0) mbar_drain(bar_kv_full, (items - 1) & 1);
      for (uint32_t i = n >= 2 ? n - 2 : 0; i <= n; ++i) mbar_drain(bar_qdo_full + (i & 1), (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t aK = smem_u32(smem + kOffK), aV = smem_u32(smem + kOffV);
    const uint32_t aDS = smem_u32(smem + kOffDS);
    uint32_t n = 0, items = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++items) {
      const BwdItem x = decode_bwd(p, it);
      if (!(ok = warp_wait(bar_kv_full, items & 1, abort, p.status))) break;
      // Issue order per step n (S^T_n and dP^T_n already issued):
      //   dQ^T_n, dV_n, S^T_{n+1}, dK_n, [dQ^T_n drained] dP^T_{n+1}
      // so the dQ drain overlaps dV/S/dK and the next softmax overlaps dK/dP.
      for (int j = 0; j < x.steps; ++j, ++n) {
        const uint32_t st = n & 1, ph = (n >> 1) & 1;
        const uint32_t aQ = smem_u32(smem + kOffQ + st * kTileBytes);
        const uint32_t aDO = smem_u32(smem + kOffDO + st * kTileBytes);
        if (j == 0) {
          if (!(ok = warp_wait(bar_qdo_full + st, ph, abort, p.status))) break;
          tc_fence_after_sync();
          if (lane == 0) {
            mma_kk(tA, aK, aQ, 0);  // S^T = K Q^T
            mma_commit(bar_s_full);
          }
          __syncwarp();
          // dP^T overwrites the dQ^T of the previous step: wait for its drain
          if (n > 0 && !(ok = warp_wait(bar_dq_free, (n - 1) & 1, abort, p.status))) break;
          tc_fence_after_sync();
          if (lane == 0) {
            mma_kk(tB, aV, aDO, 0);  // dP^T = V dO^T
            mma_commit(bar_dp_full);
          }
          __syncwarp();
        }
        if (!(ok = warp_wait(bar_ds_full, n & 1, abort, p.status))) break;
        if (j == 0 && items > 0 &&
            !(ok = warp_wait(bar_dkdv_free, (items - 1) & 1, abort, p.status)))
          break;
        tc_fence_after_sync();
        if (lane == 0) {
          mma_nn(tB, aK, aDS, 0);      // dQ^T = K^T dS^T
          mma_commit(bar_dq_full);
          mma_tn(tC, tA, aDO, j > 0);  // dV += P^T dO
        }
        __syncwarp();
        const bool has_next = j + 1 < x.steps;
        const uint32_t stn = (n + 1) & 1, phn = ((n + 1) >> 1) & 1;
        const uint32_t aQn = smem_u32(smem + kOffQ + stn * kTileBytes);
        const uint32_t aDOn = smem_u32(smem + kOffDO + stn * kTileBytes);
        if (has_next) {
          if (!(ok = warp_wait(bar_qdo_full + stn, phn, abort, p.status))) break;
          tc_fence_after_sync();
          if (lane == 0) {
            mma_kk(tA, aK, aQn, 0);  // S^T of the next step (P^T_n already consumed by dV)
            mma_commit(bar_s_full);
          }
          __syncwarp();
        }
        if (lane == 0) {
          mma_kn(tD, aDS, aQ, j > 0);  // dK += dS^T Q
          mma_commit(bar_qdo_empty + st);
        }
        __syncwarp();
        if (has_next) {
          if (!(ok = warp_wait(bar_dq_free, n & 1, abort, p.status))) break;
          tc_fence_after_sync();
          if (lane == 0) {
            mma_kk(tB, aV, aDOn, 0);  // dP^T of the next step
            mma_commit(bar_dp_full);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(bar_dkdv_full);
        mma_commit(bar_kv_empty);
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(bar_final);
      mbar_drain(bar_final, 0);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // -------------------------------------------- P^T and dS^T, one key per thread
    const int quarter = warp % 4;
    const int kr = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tSr = tA + lane_off, tPr = tB + lane_off;
    uint8_t* ds_row = smem + kOffDS + kr * 128;
    const float sl2 = p.scale_log2;
    uint32_t n = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
      const BwdItem x = decode_bwd(p, it);
      const int jk = x.kt * 128 + kr;
      const int ke = jk < p.N ? __ldg(p.key_end + jk) : 0;  // rows [jk, ke) see this key
      for (int j = 0; j < x.steps; ++j, ++n) {
        const int q0 = (x.qlo + j % x.nq) * 128;
        const uint32_t st = n & 1, ph = (n >> 1) & 1;
        const float* lse2 = reinterpret_cast<const float*>(smem + kOffLse + st * 512);
        const float* dlt = reinterpret_cast<const float*>(smem + kOffDelta + st * 512);
        if (!(ok = warp_wait(bar_qdo_full + st, ph, abort, p.status))) break;
        if (!(ok = warp_wait(bar_s_full, n & 1, abort, p.status))) break;
        tc_fence_after_sync();
        float pv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          tmem_ld32(tSr + c * 32, rr);
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c * 32 + jj);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int q = q0 + c * 32 + jj + u;
              const bool vis = jk <= q && q < ke;
              const float e = ex2_approx(fmaf(__uint_as_float(rr[jj + u]), sl2, -lv[u]));
              pv[c * 32 + jj + u] = vis ? e : 0.f;
            }
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pk[jj] = pack_bf16x2(pv[c * 32 + 2 * jj], pv[c * 32 + 2 * jj + 1]);
          tmem_st16(tSr + c * 16, pk);  // P^T over the first 64 columns of S^T
        }
        if (!(ok = warp_wait(bar_dp_full, n & 1, abort, p.status))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          tmem_ld32(tPr + c * 32, rr);
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dlt + c * 32 + jj);
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              const float ds0 = pv[c * 32 + jj + u] * (__uint_as_float(rr[jj + u]) - dv4[u]);
              const float ds1 = pv[c * 32 + jj + u + 1] * (__uint_as_float(rr[jj + u + 1]) - dv4[u + 1]);
              pk[(jj + u) / 2] = pack_bf16x2(ds0, ds1);
            }
          }
          // dS^T row kr, q columns c*32 .. c*32+31: four 16-byte chunks, 128B-swizzled
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int chunk = (c & 1) * 4 + u;
            uint4* dst = reinterpret_cast<uint4*>(ds_row + (c >> 1) * kHalfBytes +
                                                  ((chunk ^ (kr & 7)) * 16));
            *dst = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(bar_ds_full);
      }
    }
  } else if (warp >= 8) {
    // -------------------------------- dQ^T drain and the dK/dV epilogue
    const int quarter = warp % 4;
    const int rr_lane = quarter * 32 + lane;  // head-dim index for dQ^T, key row for dK/dV
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t n = 0, items = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++items) {
      const BwdItem x = decode_bwd(p, it);
      for (int j = 0; j < x.steps; ++j, ++n) {
        const int h = x.kvh * p.group + j / x.nq;
        const int q0 = (x.qlo + j % x.nq) * 128;
        if (!(ok = warp_wait(bar_dq_full, n & 1, abort, p.status))) break;
        tc_fence_after_sync();
        float* base = p.dq_acc + static_cast<size_t>(h) * 128 + rr_lane;
        const size_t row_stride = static_cast<size_t>(p.hq) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tB + lane_off + c * 32, v);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int q = q0 + c * 32 + jj;
            if (q < p.N) atomicAdd(base + static_cast<size_t>(q) * row_stride, __uint_as_float(v[jj]));
          }
        }
        tc_fence_before_sync();
        mbar_arrive(bar_dq_free);
      }
      if (!ok) break;
      if (!(ok = warp_wait(bar_dkdv_full, items & 1, abort, p.status))) break;
      tc_fence_after_sync();
      const int jk = x.kt * 128 + rr_lane;
      const size_t out = (static_cast<size_t>(jk) * p.hkv + x.kvh) * 128;
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: dV (TMEM C), 1: dK (TMEM D, times scale)
        const uint32_t t = (which ? tD : tC) + lane_off;
        const float mul = which ? p.scale : 1.f;
        void* dst_base = which ? p.dk : p.dv;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(t + c * 32, v);
          if (jk < p.N) {
            if (p.grad_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(dst_base) + out + c * 32);
#pragma unroll
              for (int u = 0; u < 8; ++u)
                dst[u] = make_float4(__uint_as_float(v[4 * u]) * mul, __uint_as_float(v[4 * u + 1]) * mul,
                                     __uint_as_float(v[4 * u + 2]) * mul, __uint_as_float(v[4 * u + 3]) * mul);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst_base) + out + c * 32);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                dst[u] = make_uint4(
                    pack_bf16x2(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul),
                    pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul),
                    pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul),
                    pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul));
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(bar_dkdv_free);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// Delta = rowsum(dO * O) and lse*log2(e), both [hq, Npad] with padded rows
// (Delta 0, lse +inf); zero the fp32 dQ accumulator. One warp per (row, head).
__global__ void __launch_bounds__(256) bwd_pre_bf16_kernel(
    const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ o,
    const float* __restrict__ lse, float* __restrict__ delta, float* __restrict__ lse2,
    float* __restrict__ dq_acc, int N, int Npad, int hq) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // i * hq + h
  if (row >= static_cast<long long>(Npad) * hq) return;
  const int i = static_cast<int>(row / hq), h = static_cast<int>(row % hq);
  float s = 0.f;
  if (i < N) {
    const uint2 a = reinterpret_cast<const uint2*>(dout + row * 128)[lane];
    const uint2 b = reinterpret_cast<const uint2*>(o + row * 128)[lane];
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float2 fa = __bfloat1622float2(a2[u]);
      const float2 fb = __bfloat1622float2(b2[u]);
      s = fmaf(fa.x, fb.x, s);
      s = fmaf(fa.y, fb.y, s);
    }
    reinterpret_cast<float4*>(dq_acc + row * 128)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    const size_t idx = static_cast<size_t>(h) * Npad + i;
    delta[idx] = s;
    lse2[idx] = i < N ? lse[static_cast<size_t>(h) * N + i] * 1.4426950408889634f : INFINITY;
  }
}

// dq = scale * dq_acc, to bf16 or fp32. Each thread converts 4 elements.
__global__ void __launch_bounds__(256) bwd_finalize_kernel(const float* __restrict__ acc,
                                                          void* __restrict__ dq, long long n4,
                                                          float scale, int out_f32) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[i];
  if (out_f32) {
    reinterpret_cast<float4*>(dq)[i] = make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale);
  } else {
    reinterpret_cast<uint2*>(dq)[i] =
        make_uint2(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale));
  }
}

}  // namespace

cudaError_t launch_bwd_bf16(const AttnBwdArgs& a) {
  const tree_plan* pl = a.plan;
  const int N = pl->N, Npad = pl->Tq * 128;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const size_t acc_bytes = (static_cast<size_t>(N) * a.hq * 128 * 4 + 255) / 256 * 256;
  float* dq_acc = reinterpret_cast<float*>(ws);
  float* delta = reinterpret_cast<float*>(ws + acc_bytes);
  float* lse2 = delta + static_cast<size_t>(a.hq) * Npad;

  const long long rows = static_cast<long long>(Npad) * a.hq;
  bwd_pre_bf16_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.dout), static_cast<const __nv_bfloat16*>(a.o), a.lse,
      delta, lse2, dq_acc, N, Npad, a.hq);

  CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map(&mq, a.q, N, a.hq) || !make_tile_map(&mk, a.k, N, a.hkv) ||
      !make_tile_map(&mv, a.v, N, a.hkv) || !make_tile_map(&mdo, a.dout, N, a.hq))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.key_end = pl->dev.key_end;
  p.kt_qlo = pl->dev.kt_qlo;
  p.kt_qhi = pl->dev.kt_qhi;
  p.order = pl->dev.bwd_order;
  p.lse2 = lse2;
  p.delta = delta;
  p.dq_acc = dq_acc;
  p.dk = a.dk;
  p.dv = a.dv;
  p.status = a.status;
  p.N = N;
  p.Npad = Npad;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.group = a.hq / a.hkv;
  p.n_items = pl->Tk * a.hkv;
  p.grad_f32 = a.grad_f32 ? 1 : 0;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tree_attn_bwd_sm103,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = p.n_items < sm_count() ? p.n_items : sm_count();
  tree_attn_bwd_sm103<<<grid, kThreads, kSmemBytes, a.stream>>>(mq, mk, mv, mdo, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const long long n4 = static_cast<long long>(N) * a.hq * 128 / 4;
  bwd_finalize_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, a.stream>>>(
      dq_acc, a.dq, n4, a.scale, a.grad_f32 ? 1 : 0);
  return cudaGetLastError();
}


}  // namespace treeattn
