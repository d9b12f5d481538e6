// Rotary position embedding at tree position ids.
//
// Tree Training (arXiv 2511.00413) §3.2 "Position Embedding", eq. 9: a token
// at offset j of node n takes the position sum_{ancestors n'} |T_n'| + j, the
// one it has in every standalone root-to-leaf sequence through it, so that
// RoPE gives the per-path result. The rotation is RoFormer's rotary matrix
// (Su et al. 2023): dimension pair i of a head turns by pos * theta_i,
// theta_i = base^(-2i/D). The pair is (2i, 2i+1) (RoFormer's own layout) or, with
// rotate_half, (i, i + D/2) (the split-halves layout many checkpoints use).
// The inverse rotation (angle -pos * theta_i) is the backward of the forward
// one: the rotation is orthogonal, so grad_x = R^T grad_y.
//
// The op is a streaming pass over x[N, H, D] (read once, written once), so
// HBM bandwidth bounds it: rows move in 16-byte chunks and each token's sines
// and cosines are computed once and shared by all its heads. The angle is
// formed and reduced modulo 2 pi in fp64 (positions reach 10^5 radians at
// theta_0 = 1, beyond fp32's resolution), then sincosf works on about [0, 2 pi).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "kernels.h"

namespace treeattn {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeMaxPairs = 64;  // head_dim <= 128

struct RopeParams {
  const int32_t* pos;  // [N] position ids (eq. 9)
  void* x;             // [N, H, D]
  void* x2;            // [N, H2, D] or nullptr (H2 = 0): the same tokens' second tensor
  int N, H, H2, D, rotate_half, f32;
  float sign;          // +1 forward, -1 inverse
  double theta[kRopeMaxPairs];
};

__device__ __forceinline__ void rotate(float& a, float& b, float c, float s) {
  const float ya = fmaf(a, c, -b * s);
  const float yb = fmaf(a, s, b * c);
  a = ya;
  b = yb;
}

template <typename T>
__device__ __forceinline__ float ld(const T* p);
template <>
__device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T>
__device__ __forceinline__ void st(T* p, float v);
template <>
__device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Eight consecutive elements of a row: loaded raw (one 16-byte access for
// bf16, two for fp32) so several can be in flight in few registers, then
// widened to fp32, rotated, rounded and stored back.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void widen(float (&v)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void widen(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

// The angle pos * theta_i reduced by a whole number of turns, in fp64. The
// turn count comes from a multiply by 1 / (2 pi), not a division (fp64 runs
// at a small fraction of the fp32 rate here): near a multiple of 2 pi it may
// be one off, which leaves r just outside [0, 2 pi) and the same sine and
// cosine.
__device__ __forceinline__ void angle_sincos(const RopeParams& p, int32_t pos, int i, float& s, float& c) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  const double a = static_cast<double>(pos) * p.theta[i];
  const float r = static_cast<float>(fma(-two_pi, floor(a * inv_two_pi), a));
  sincosf(r, &s, &c);
  s *= p.sign;
}

// Vector path (head_dim a multiple of 16): a block takes kRopeTokens tokens at
// a time, first fills a table of their sines and cosines in shared memory,
// then streams their rows (the heads of x, then those of x2) in 8-element
// chunks. Interleaved pairs: a chunk
// holds pairs 4q..4q+3. Split halves: a work unit is chunk q of the first
// half and chunk q of the second (pairs 8q..8q+7).
constexpr int kRopeTokens = 8;
// chunks in flight per thread: 16 bytes each for bf16, 32 for fp32
template <typename T>
constexpr int rope_unroll() { return sizeof(T) == 2 ? 4 : 2; }

template <typename T>
__global__ void __launch_bounds__(kRopeThreads, 4) tree_rope_vec_kernel(const RopeParams p) {
  __shared__ float s_sin[kRopeTokens][kRopeMaxPairs], s_cos[kRopeTokens][kRopeMaxPairs];
  const int pairs = p.D / 2;
  const int units_per_row = p.rotate_half ? p.D / 16 : p.D / 8;
  T* x = static_cast<T*>(p.x);
  T* x2 = static_cast<T*>(p.x2);
  for (int t0 = blockIdx.x * kRopeTokens; t0 < p.N; t0 += gridDim.x * kRopeTokens) {
    __syncthreads();  // the previous tokens' table is no longer read
    for (int e = threadIdx.x; e < kRopeTokens * pairs; e += kRopeThreads) {
      const int tt = e / pairs, i = e % pairs;
      float sn = 0.f, cs = 1.f;
      if (t0 + tt < p.N) angle_sincos(p, __ldg(p.pos + t0 + tt), i, sn, cs);
      s_sin[tt][i] = sn;
      s_cos[tt][i] = cs;
    }
    __syncthreads();
    // kUnroll units per thread at a time, all loads issued before any use,
    // so enough bytes are in flight to cover the memory latency
    const int tokens_here = p.N - t0 < kRopeTokens ? p.N - t0 : kRopeTokens;
    // units: those of x's rows (token-major), then those of x2's
    const int live1 = tokens_here * p.H * units_per_row;
    const int live = live1 + tokens_here * p.H2 * units_per_row;
    // unit u's chunk q, its row, and the row's token within the table
    auto locate = [&](int u, int& q, int& tt) -> T* {
      const bool second = u >= live1;
      const int uu = second ? u - live1 : u, H = second ? p.H2 : p.H;
      q = uu % units_per_row;
      const int rest = uu / units_per_row;  // row of the block's tokens, token-major
      tt = rest / H;
      return (second ? x2 : x) + (static_cast<size_t>(t0) * H + rest) * p.D;
    };
    constexpr int kUnroll = rope_unroll<T>();
    for (int u0 = threadIdx.x; u0 < live; u0 += kRopeThreads * kUnroll) {
      Raw8<T> ra[kUnroll], rb[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int u = u0 + k * kRopeThreads;
        if (u >= live) continue;
        int q, tt;
        const T* row = locate(u, q, tt);
        ra[k].load(row + 8 * q);
        if (p.rotate_half) rb[k].load(row + pairs + 8 * q);
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int u = u0 + k * kRopeThreads;
        if (u >= live) continue;
        int q, tt;
        T* row = locate(u, q, tt);
        float a[8];
        ra[k].widen(a);
        if (p.rotate_half) {
          float b[8];
          rb[k].widen(b);
#pragma unroll
          for (int j = 0; j < 8; ++j) rotate(a[j], b[j], s_cos[tt][8 * q + j], s_sin[tt][8 * q + j]);
          Raw8<T>::store(row + 8 * q, a);
          Raw8<T>::store(row + pairs + 8 * q, b);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) rotate(a[2 * j], a[2 * j + 1], s_cos[tt][4 * q + j], s_sin[tt][4 * q + j]);
          Raw8<T>::store(row + 8 * q, a);
        }
      }
    }
  }
}

// General path (any even head_dim up to 128): one thread per pair index,
// scalar accesses, the pair's sine and cosine reused for every head.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads) tree_rope_kernel(const RopeParams p) {
  const int pairs = p.D / 2;
  const int groups = kRopeThreads / pairs;  // threads sharing a pair index, each on other heads
  const int i = threadIdx.x % pairs, g = threadIdx.x / pairs;
  if (g >= groups) return;  // pairs that do not divide 256 leave a few threads idle
  T* x = static_cast<T*>(p.x);
  T* x2 = static_cast<T*>(p.x2);
  for (int t = blockIdx.x; t < p.N; t += gridDim.x) {
    float s, c;
    angle_sincos(p, __ldg(p.pos + t), i, s, c);
    for (int h = g; h < p.H + p.H2; h += groups) {
      T* e = h < p.H ? x + (static_cast<size_t>(t) * p.H + h) * p.D
                     : x2 + (static_cast<size_t>(t) * p.H2 + (h - p.H)) * p.D;
      T* ea = p.rotate_half ? e + i : e + 2 * i;
      T* eb = p.rotate_half ? e + i + pairs : e + 2 * i + 1;
      float va = ld(ea), vb = ld(eb);
      rotate(va, vb, c, s);
      st(ea, va);
      st(eb, vb);
    }
  }
}

}  // namespace

bool rope_shape_ok(int head_dim) { return head_dim >= 2 && head_dim % 2 == 0 && head_dim / 2 <= kRopeMaxPairs; }

cudaError_t launch_rope(const RopeArgs& a) {
  RopeParams p;
  p.pos = a.pos;
  p.x = a.x;
  p.x2 = a.x2;
  p.N = a.N;
  p.H = a.heads;
  p.H2 = a.x2 ? a.heads2 : 0;
  p.D = a.head_dim;
  p.rotate_half = a.rotate_half;
  p.f32 = a.f32;
  p.sign = a.inverse ? -1.f : 1.f;
  for (int i = 0; i < kRopeMaxPairs; ++i)
    p.theta[i] = i < a.head_dim / 2 ? std::pow(static_cast<double>(a.base), -2.0 * i / a.head_dim) : 0.0;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (a.head_dim % 16 == 0) {  // rows split into 16-byte (bf16) or 32-byte (fp32) chunks
    const int tiles = (a.N + kRopeTokens - 1) / kRopeTokens;
    const int blocks = tiles < sms * 8 ? tiles : sms * 8;
    if (a.f32)
      tree_rope_vec_kernel<float><<<blocks, kRopeThreads, 0, a.stream>>>(p);
    else
      tree_rope_vec_kernel<__nv_bfloat16><<<blocks, kRopeThreads, 0, a.stream>>>(p);
  } else {
    const int blocks = a.N < sms * 8 ? a.N : sms * 8;
    if (a.f32)
      tree_rope_kernel<float><<<blocks, kRopeThreads, 0, a.stream>>>(p);
    else
      tree_rope_kernel<__nv_bfloat16><<<blocks, kRopeThreads, 0, a.stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace treeattn
