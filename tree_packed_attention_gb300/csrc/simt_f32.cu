// fp32 tree attention on the CUDA cores: forward, backward preprocess, dQ and
// dK/dV. Used for fp32 inputs, where the tolerance (1e-4) rules out the
// bf16/TF32 tensor-core paths.
//
// Mask ("Tree Training" §3.2 "Attention Mask" / App. A.1), column form: row i
// sees key j iff j <= i < key_end[j] (key_end = end of the DFS subtree of j's
// segment). The forward walks the plan's non-empty k-tiles of each q-tile;
// the dK/dV kernel walks, for key j, exactly the rows [j, key_end[j]).
//
// One warp owns one row (or one key); each lane holds D/32 consecutive
// elements of the head vector; dot products are warp reductions. No atomics:
// results are deterministic.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace treeattn {
namespace {

constexpr int kWarps = 4;

template <int E>
__device__ __forceinline__ float dot_lanes(const float (&a)[E], const float* __restrict__ b) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = fmaf(a[e], b[e], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

// grid (Tq, hq), block 128: warp w owns rows qt*128 + w, +4, ...
template <int D>
__global__ void __launch_bounds__(kWarps * 32) fwd_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    float* __restrict__ o, float* __restrict__ lse, const int32_t* __restrict__ key_end,
    const int32_t* __restrict__ qt_ptr, const int32_t* __restrict__ qt_kt, int N, int hq, int hkv,
    float scale) {
  constexpr int E = D / 32;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int kvh = h / (hq / hkv);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e0 = lane * E;
  for (int r = warp; r < 128; r += kWarps) {
    const int i = qt * 128 + r;
    if (i >= N) break;
    float qi[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qi[e] = q[((size_t)i * hq + h) * D + e0 + e];
      acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int t = qt_ptr[qt]; t < qt_ptr[qt + 1]; ++t) {
      const int j0 = qt_kt[t] * 128;
      const int j1 = min(N, j0 + 128);
      for (int j = j0; j < j1; ++j) {
        if (!(j <= i && i < key_end[j])) continue;  // uniform across the warp
        const float s = scale * dot_lanes<E>(qi, k + ((size_t)j * hkv + kvh) * D + e0);
        const float m_new = fmaxf(m, s);
        const float corr = expf(m - m_new);  // 0 when m = -inf
        const float p = expf(s - m_new);
        l = l * corr + p;
        const float* vj = v + ((size_t)j * hkv + kvh) * D + e0;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vj[e], acc[e] * corr);
        m = m_new;
      }
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) o[((size_t)i * hq + h) * D + e0 + e] = acc[e] * inv;
    if (lane == 0) lse[(size_t)h * N + i] = m + logf(l);
  }
}

// delta[h][i] = sum_d dO[i,h,d] * O[i,h,d]; one warp per (row, head).
template <int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_pre_f32_kernel(const float* __restrict__ dout,
                                                                 const float* __restrict__ o,
                                                                 float* __restrict__ delta, int N,
                                                                 int hq) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long row = (long long)blockIdx.x * kWarps + warp;  // row = i * hq + h
  if (row >= (long long)N * hq) return;
  float a[E];
#pragma unroll
  for (int e = 0; e < E; ++e) a[e] = dout[row * D + lane * E + e];
  const float s = dot_lanes<E>(a, o + row * D + lane * E);
  if (lane == 0) {
    const int i = (int)(row / hq), h = (int)(row % hq);
    delta[(size_t)h * N + i] = s;
  }
}

// dq_i = scale * sum_j P_ij (dP_ij - delta_i) k_j over the visible keys of i.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dout, const float* __restrict__ lse, const float* __restrict__ delta,
    float* __restrict__ dq, const int32_t* __restrict__ key_end, const int32_t* __restrict__ qt_ptr,
    const int32_t* __restrict__ qt_kt, int N, int hq, int hkv, float scale) {
  constexpr int E = D / 32;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int kvh = h / (hq / hkv);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e0 = lane * E;
  for (int r = warp; r < 128; r += kWarps) {
    const int i = qt * 128 + r;
    if (i >= N) break;
    float qi[E], di[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qi[e] = q[((size_t)i * hq + h) * D + e0 + e];
      di[e] = dout[((size_t)i * hq + h) * D + e0 + e];
      acc[e] = 0.f;
    }
    const float lse_i = lse[(size_t)h * N + i];
    const float delta_i = delta[(size_t)h * N + i];
    for (int t = qt_ptr[qt]; t < qt_ptr[qt + 1]; ++t) {
      const int j0 = qt_kt[t] * 128;
      const int j1 = min(N, j0 + 128);
      for (int j = j0; j < j1; ++j) {
        if (!(j <= i && i < key_end[j])) continue;
        const float* kj = k + ((size_t)j * hkv + kvh) * D + e0;
        const float p = expf(scale * dot_lanes<E>(qi, kj) - lse_i);
        const float dp = dot_lanes<E>(di, v + ((size_t)j * hkv + kvh) * D + e0);
        const float ds = p * (dp - delta_i);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(ds, kj[e], acc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) dq[((size_t)i * hq + h) * D + e0 + e] = scale * acc[e];
  }
}

// dk_j, dv_j summed over the q heads of kv head kvh and over rows [j, key_end[j]).
// grid (Tk, hkv), warp w owns keys kt*128 + w, +4, ...
template <int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dout, const float* __restrict__ lse, const float* __restrict__ delta,
    float* __restrict__ dk, float* __restrict__ dv, const int32_t* __restrict__ key_end, int N,
    int hq, int hkv, float scale) {
  constexpr int E = D / 32;
  const int kt = blockIdx.x, kvh = blockIdx.y;
  const int G = hq / hkv;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e0 = lane * E;
  for (int r = warp; r < 128; r += kWarps) {
    const int j = kt * 128 + r;
    if (j >= N) break;
    float kj[E], vj[E], ak[E], av[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kj[e] = k[((size_t)j * hkv + kvh) * D + e0 + e];
      vj[e] = v[((size_t)j * hkv + kvh) * D + e0 + e];
      ak[e] = 0.f;
      av[e] = 0.f;
    }
    const int i1 = key_end[j];
    for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
      for (int i = j; i < i1; ++i) {
        const float* qi = q + ((size_t)i * hq + h) * D + e0;
        const float* di = dout + ((size_t)i * hq + h) * D + e0;
        const float p = expf(scale * dot_lanes<E>(kj, qi) - lse[(size_t)h * N + i]);
        const float dp = dot_lanes<E>(vj, di);
        const float ds = p * (dp - delta[(size_t)h * N + i]);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          av[e] = fmaf(p, di[e], av[e]);
          ak[e] = fmaf(ds, qi[e], ak[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dk[((size_t)j * hkv + kvh) * D + e0 + e] = scale * ak[e];
      dv[((size_t)j * hkv + kvh) * D + e0 + e] = av[e];
    }
  }
}

template <int D>
cudaError_t fwd_f32(const AttnArgs& a) {
  const tree_plan* p = a.plan;
  dim3 grid(p->Tq, a.hq);
  fwd_f32_kernel<D><<<grid, kWarps * 32, 0, a.stream>>>(
      static_cast<const float*>(a.q), static_cast<const float*>(a.k),
      static_cast<const float*>(a.v), static_cast<float*>(a.o), a.lse, p->dev.key_end,
      p->dev.qt_ptr, p->dev.qt_kt, p->N, a.hq, a.hkv, a.scale);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_f32(const AttnBwdArgs& a) {
  const tree_plan* p = a.plan;
  const int N = p->N;
  float* delta = static_cast<float*>(a.workspace);
  const long long rows = (long long)N * a.hq;
  if (a.phases & 1) {
    bwd_pre_f32_kernel<D><<<(unsigned)((rows + kWarps - 1) / kWarps), kWarps * 32, 0, a.stream>>>(
        static_cast<const float*>(a.dout), static_cast<const float*>(a.o), delta, N, a.hq);
    bwd_dq_f32_kernel<D><<<dim3(p->Tq, a.hq), kWarps * 32, 0, a.stream>>>(
        static_cast<const float*>(a.q), static_cast<const float*>(a.k),
        static_cast<const float*>(a.v), static_cast<const float*>(a.dout), a.lse, delta,
        static_cast<float*>(a.dq), p->dev.key_end, p->dev.qt_ptr, p->dev.qt_kt, N, a.hq, a.hkv,
        a.scale);
  }
  if (!(a.phases & 2)) return cudaGetLastError();
  bwd_dkdv_f32_kernel<D><<<dim3(p->Tk, a.hkv), kWarps * 32, 0, a.stream>>>(
      static_cast<const float*>(a.q), static_cast<const float*>(a.k),
      static_cast<const float*>(a.v), static_cast<const float*>(a.dout), a.lse, delta,
      static_cast<float*>(a.dk), static_cast<float*>(a.dv), p->dev.key_end, N, a.hq, a.hkv,
      a.scale);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_f32(int64_t n, int hq) {
  return static_cast<size_t>((n * hq * 4 + 255) / 256 * 256);
}

cudaError_t launch_fwd_f32(const AttnArgs& a) {
  return a.d == 64 ? fwd_f32<64>(a) : fwd_f32<128>(a);
}

cudaError_t launch_bwd_f32(const AttnBwdArgs& a) {
  return a.d == 64 ? bwd_f32<64>(a) : bwd_f32<128>(a);
}

}  // namespace treeattn
