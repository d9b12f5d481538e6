// Gated DeltaNet forward over a DFS-serialized trie with tree state routing
// ("Tree Training", arXiv 2511.00413, §3.2 "SSM Layers (GDN)" eq. 10 and
// App. A.2): every tree node's segment is one chunk, and a chunk starts from
// the final state of its parent chunk (a root from the initial state), never
// from the chunk before it in DFS order.
//
// Per value head h (query/key head h / G), state S [Dk = 128, Dv = 128] fp32,
// token t (log decay g_t, write strength beta_t), the gated delta rule:
//   S_t = exp(g_t) S_{t-1} + k_t (beta_t (v_t - exp(g_t) S_{t-1}^T k_t))^T
//   o_t = S_t^T q_t
// Columns of S evolve independently given the token, so a CTA owns one head of
// one trie and each thread one value column, S[:, j] (128 fp32 registers): the
// two dot products over Dk need no exchange, and every lane reads the same
// staged key and query (shared-memory broadcasts). The CTA walks the trie's
// tokens in DFS order, 32 at a time staged in shared memory as fp32; at a
// segment's first token the state is the initial state (a root), kept in
// registers (the segment right before it in DFS order is its parent), or
// reloaded from the parent's saved end state; every segment's end state is
// written out. Tries are launched longest first.
//
// Bound by the FMA pipe: about 3 Dk Dv fused multiply-adds per token and head
// (the key dot product, the state update, the query dot product), issued as
// packed fp32 pairs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace treeattn {
namespace {

constexpr int kD = 128;          // Dk = Dv
constexpr int kThreads = kD;     // one value column per thread
constexpr int kChunk = 32;       // tokens staged at a time

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// A shared-memory read the compiler must issue where it stands (keeping the
// key in registers across both loops would double the register footprint).
__device__ __forceinline__ float4 lds4(const float* p) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return r;
}

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ void put(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void put(float* p, float x) { *p = x; }

template <typename T>
__global__ void __launch_bounds__(kThreads) tree_gdn_fwd_kernel(const GdnArgs a) {
  __shared__ __align__(16) float sk[kChunk][kD];
  __shared__ __align__(16) float sq[kChunk][kD];
  __shared__ __align__(16) float sv[kChunk][kD];
  __shared__ float sa[kChunk], sb[kChunk];  // exp(g) and beta
  const int r = __ldg(a.trie_order + blockIdx.x), h = blockIdx.y;
  const int j = threadIdx.x;  // this thread's value column: S[:, j] in registers
  const int hq = h / a.group;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  T* o = static_cast<T*>(a.o);
  const size_t state_elems = static_cast<size_t>(kD) * kD;
  auto state_ptr = [&](int seg) { return a.states + (static_cast<size_t>(seg) * a.hv + h) * state_elems; };

  const int d0 = __ldg(a.trie_ptr + r), d1 = __ldg(a.trie_ptr + r + 1);
  if (d0 >= d1) return;
  const int T0 = __ldg(a.cu + r), T1 = __ldg(a.cu + r + 1);  // the trie's DFS tokens
  float2 S[kD / 2];  // S[x] = rows 2x, 2x+1 of column j
  int d = d0;
  int4 seg = a.segs[d];  // (segment id, first token, length, parent id)
  int prev = -2;         // the segment whose end state is in registers
  for (int c0 = T0; c0 < T1; c0 += kChunk) {
    const int n = min(kChunk, T1 - c0);
    // ---- stage the chunk as fp32: q and k rows of head hq, v rows of head h,
    // exp(g) and beta
    __syncthreads();
    for (int e = threadIdx.x; e < n * (kD / 8); e += kThreads) {
      const int i = e / (kD / 8), c8 = (e % (kD / 8)) * 8;
      const size_t row = (static_cast<size_t>(c0 + i) * a.hk + hq) * kD + c8;
      const size_t vrow = (static_cast<size_t>(c0 + i) * a.hv + h) * kD + c8;
      float f[8];
      load8<T>(k + row, f);
      *reinterpret_cast<float4*>(&sk[i][c8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&sk[i][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
      load8<T>(q + row, f);
      *reinterpret_cast<float4*>(&sq[i][c8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&sq[i][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
      load8<T>(v + vrow, f);
      *reinterpret_cast<float4*>(&sv[i][c8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&sv[i][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
    if (threadIdx.x < n) {
      const size_t gi = static_cast<size_t>(c0 + threadIdx.x) * a.hv + h;
      sa[threadIdx.x] = expf(__ldg(a.g + gi));
      sb[threadIdx.x] = __ldg(a.beta + gi);
    }
    __syncthreads();
    for (int i = 0; i < n; ++i) {
      const int t = c0 + i;
      if (t == seg.y) {  // a segment's first token: its initial state
        const float* src = seg.w < 0 ? (a.s0 ? a.s0 + static_cast<size_t>(h) * state_elems : nullptr)
                           : (seg.w != prev ? state_ptr(seg.w) : nullptr);
        if (src) {
          src += j;
#pragma unroll
          for (int x = 0; x < kD / 2; ++x) S[x] = make_float2(src[(2 * x) * kD], src[(2 * x + 1) * kD]);
        } else if (seg.w < 0) {
#pragma unroll
          for (int x = 0; x < kD / 2; ++x) S[x] = make_float2(0.f, 0.f);
        }
      }
      // u = S^T k (every lane reads the same k: broadcast), in packed pairs
      const float* kr = &sk[i][0];
      float2 u2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int x = 0; x < kD / 4; ++x) {
        const float4 kk = lds4(kr + 4 * x);
        u2[0] = __ffma2_rn(S[2 * x], make_float2(kk.x, kk.y), u2[0]);
        u2[1] = __ffma2_rn(S[2 * x + 1], make_float2(kk.z, kk.w), u2[1]);
      }
      const float u = (u2[0].x + u2[0].y) + (u2[1].x + u2[1].y);
      const float al = sa[i];
      const float delta = sb[i] * (sv[i][j] - al * u);
      const float2 al2 = make_float2(al, al), de2 = make_float2(delta, delta);
      // S = exp(g) S + k delta, then o = S^T q
      const float* qr = &sq[i][0];
      float2 o2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int x = 0; x < kD / 4; ++x) {
        const float4 kk = lds4(kr + 4 * x);
        S[2 * x] = __ffma2_rn(S[2 * x], al2, __fmul2_rn(make_float2(kk.x, kk.y), de2));
        S[2 * x + 1] = __ffma2_rn(S[2 * x + 1], al2, __fmul2_rn(make_float2(kk.z, kk.w), de2));
        const float4 qq = lds4(qr + 4 * x);
        o2[0] = __ffma2_rn(S[2 * x], make_float2(qq.x, qq.y), o2[0]);
        o2[1] = __ffma2_rn(S[2 * x + 1], make_float2(qq.z, qq.w), o2[1]);
      }
      put(o + (static_cast<size_t>(t) * a.hv + h) * kD + j, (o2[0].x + o2[0].y) + (o2[1].x + o2[1].y));
      if (t == seg.y + seg.z - 1) {  // the segment's last token: save its end state
        float* dst = state_ptr(seg.x) + j;
#pragma unroll
        for (int x = 0; x < kD / 2; ++x) {
          dst[(2 * x) * kD] = S[x].x;
          dst[(2 * x + 1) * kD] = S[x].y;
        }
        prev = seg.x;
        if (++d < d1) seg = a.segs[d];
      }
    }
  }
}

}  // namespace

cudaError_t launch_gdn_fwd(const GdnArgs& a) {
  const dim3 grid(a.R, a.hv);
  if (a.f32)
    tree_gdn_fwd_kernel<float><<<grid, kThreads, 0, a.stream>>>(a);
  else
    tree_gdn_fwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, a.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace treeattn
