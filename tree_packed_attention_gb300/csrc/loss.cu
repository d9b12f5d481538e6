// Fused weighted next-token cross-entropy over a DFS-serialized trie
// ("Tree Training", arXiv 2511.00413, §3.1 eq. 3-5 and §3.2 "Loss Weights").
//
// On every root-to-leaf path the token after position r is predicted from the
// logits row of r: in the DFS layout that is token r + 1 when it lies in r's
// segment, else the first token of each child segment of r's segment (none
// after a leaf's last token). Prediction r -> t weighs lambda_t:
//
//   row_loss[r] = sum over r -> t of lambda_t * (logsumexp(z_r) - z_r[x_t])
//   dz_r        = grad_scale * (W_r * softmax(z_r) - sum over r -> t of lambda_t * e_{x_t}),
//   W_r         = sum over r -> t of lambda_t.
//
// One CTA per logits row (persistent over rows). Pass 1 streams the row once
// with 16-byte loads and keeps a running (max, sum of exponentials) per thread,
// merged across the CTA; the row's predictions are then collected by walking
// the children of r's segment; pass 2 streams the row again, mostly from L2
// (pass 1 loads with an evict-last policy; pass 2's loads and the dz stores
// are marked as last uses, so the dz stream does not evict the rows; two CTAs
// per SM keep about 2 x 152 rows in flight), and writes dz with the targets'
// one-hot terms folded in, so each element is rounded once and dz may
// overwrite z. The row losses are summed in a fixed order by a second kernel.
//
// Both passes form each exponent from z - max (exact near the max), so the
// softmax's relative error does not grow with the logits' magnitude; the loss
// takes (max - z_x) + ln(sum) without rounding lse itself.
//
// HBM traffic per row: V elements read (pass 1; most of pass 2 hits L2) and V written.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "tma_host.h"

namespace treeattn {
namespace {

constexpr int kCeThreads = 512;
constexpr int kCeWarps = kCeThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16 bytes of a row as floats: 8 bf16 or 4 fp32.
// pass 1: keep the row in L2 for pass 2 (evict-last policy)
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld16_keep(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
// pass 2: the row's last read, and dz, need not stay in L2
__device__ __forceinline__ uint4 ld16_last(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ static void unpack(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(f[2 * i + 1]), "f"(f[2 * i]));
    __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(p[0]); }
};
template <>
struct Vec<float> {
  static constexpr int E = 4;
  __device__ static void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float* p, const float (&f)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
  }
  __device__ static float one(const float* p) { return p[0]; }
};

// Merge two (max, sum of 2^(x*log2e - max*log2e)) pairs.
__device__ __forceinline__ void merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  s = s * ex2f((m - mn) * kLog2e) + s2 * ex2f((m2 - mn) * kLog2e);
  m = mn;
}

struct CeParams {
  const int32_t* tokens;
  const float* lam;
  const int32_t* token_seg;
  const int32_t* subtree_end;
  float* row_loss;
  int* status;
  int N, V;
  float gs;
};

template <typename T>
__global__ void __launch_bounds__(kCeThreads, 2)
    tree_ce_kernel(const T* z, T* dz, const CeParams p) {
  constexpr int E = Vec<T>::E;
  constexpr int U = 4;  // vectors in flight per thread
  __shared__ float red_m[kCeWarps], red_s[kCeWarps];
  __shared__ int tgt_x[kCeMaxTargets];
  __shared__ float tgt_w[kCeMaxTargets];
  __shared__ int s_ntgt;
  __shared__ float s_m, s_l2, s_w;  // row max, log2 of the row's sum of 2^((z - max) log2e)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V;
  const uint64_t keep = policy_evict_last();
  for (int r = blockIdx.x; r < p.N; r += gridDim.x) {
    const T* zr = z + static_cast<size_t>(r) * V;
    // ---- pass 1: running max and sum of exponentials
    float m = -INFINITY, s = 0.f;
    for (int v0 = tid * E; v0 < V; v0 += kCeThreads * E * U) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kCeThreads * E;
        if (v < V) raw[u] = ld16_keep(zr + v, keep);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kCeThreads * E;
        if (v >= V) break;
        float f[E];
        Vec<T>::unpack(raw[u], f);
        float vm = f[0];
#pragma unroll
        for (int e = 1; e < E; ++e) vm = fmaxf(vm, f[e]);
        if (vm > m) {
          s *= ex2f((m - vm) * kLog2e);
          m = vm;
        }
        // z - max first (exact near the max), so that the exponent's error
        // does not grow with the logits' magnitude
#pragma unroll
        for (int e = 0; e < E; ++e) s += ex2f((f[e] - m) * kLog2e);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      merge(m, s, m2, s2);
    }
    if (lane == 0) {
      red_m[warp] = m;
      red_s[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
      m = lane < kCeWarps ? red_m[lane] : -INFINITY;
      s = lane < kCeWarps ? red_s[lane] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        merge(m, s, m2, s2);
      }
      if (lane == 0) {
        const float ls = logf(s);  // lse = m + ls, kept apart
        // ---- the predictions made from row r (successor walk, fixed order)
        float loss = 0.f, w_sum = 0.f;
        int nt = 0;
        auto add = [&](int t) {
          const int x = p.tokens[t];
          if (x < 0) return;  // not predicted (ignored token)
          if (x >= V) {
            atomicExch(p.status, 8);
            return;
          }
          const float w = p.lam[t];
          if (w == 0.f) return;
          loss += w * ((m - Vec<T>::one(zr + x)) + ls);
          w_sum += w;
          for (int j = 0; j < nt; ++j)
            if (tgt_x[j] == x) {
              tgt_w[j] += w;
              return;
            }
          if (nt < kCeMaxTargets) {
            tgt_x[nt] = x;
            tgt_w[nt] = w;
            ++nt;
          } else {
            atomicExch(p.status, 7);  // more distinct targets than a row can hold
          }
        };
        const int seg = p.token_seg[r];
        if (r + 1 < p.N && p.token_seg[r + 1] == seg) {
          add(r + 1);
        } else {
          const int e = p.subtree_end[seg];
          for (int t = r + 1; t < e; t = p.subtree_end[p.token_seg[t]]) add(t);
        }
        p.row_loss[r] = loss;
        s_ntgt = nt;
        s_m = m;
        s_l2 = ls * kLog2e;
        s_w = w_sum;
      }
    }
    __syncthreads();
    // ---- pass 2: dz = gs * (W * softmax - one-hot terms)
    const int nt = s_ntgt;
    const float a = p.gs * s_w, mr = s_m, nl2 = -s_l2;
    T* dr = dz + static_cast<size_t>(r) * V;
    for (int v0 = tid * E; v0 < V; v0 += kCeThreads * E * U) {
      uint4 raw[U];
      if (a != 0.f) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kCeThreads * E;
          if (v < V) raw[u] = ld16_last(zr + v);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kCeThreads * E;
        if (v >= V) break;
        float f[E];
        if (a != 0.f) {
          Vec<T>::unpack(raw[u], f);
#pragma unroll
          for (int e = 0; e < E; ++e) f[e] = a * ex2f(fmaf(f[e] - mr, kLog2e, nl2));
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) f[e] = 0.f;
        }
        for (int j = 0; j < nt; ++j) {
          const int x = tgt_x[j] - v;
          if (x >= 0 && x < E) {
#pragma unroll
            for (int e = 0; e < E; ++e)
              if (e == x) f[e] -= p.gs * tgt_w[j];
          }
        }
        Vec<T>::store(dr + v, f);
      }
    }
    __syncthreads();  // the shared row state is rewritten for the next row
  }
}

// Sum of the row losses in a fixed order (fp64), one CTA.
__global__ void __launch_bounds__(1024) tree_ce_sum(const float* row_loss, int N, double* out) {
  __shared__ double part[32];
  double acc = 0.0;
  for (int i = threadIdx.x; i < N; i += blockDim.x) acc += row_loss[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    acc = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (threadIdx.x == 0) *out = acc;
  }
}

}  // namespace

cudaError_t launch_weighted_ce(const CeArgs& a) {
  CeParams p;
  p.tokens = a.tokens;
  p.lam = a.lam;
  p.token_seg = a.token_seg;
  p.subtree_end = a.subtree_end;
  p.row_loss = a.row_loss;
  p.status = a.status;
  p.N = a.N;
  p.V = a.V;
  p.gs = a.grad_scale;
  const int grid = a.N < 2 * sm_count() ? a.N : 2 * sm_count();
  if (a.f32)
    tree_ce_kernel<float><<<grid, kCeThreads, 0, a.stream>>>(static_cast<const float*>(a.logits),
                                                             static_cast<float*>(a.dlogits), p);
  else
    tree_ce_kernel<__nv_bfloat16><<<grid, kCeThreads, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.logits), static_cast<__nv_bfloat16*>(a.dlogits), p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !a.loss) return e;
  tree_ce_sum<<<1, 1024, 0, a.stream>>>(a.row_loss, a.N, a.loss);
  return cudaGetLastError();
}

}  // namespace treeattn
