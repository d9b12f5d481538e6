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
// Columns of S evolve independently given the token, and each column's two
// products over Dk split into partial sums, so a CTA owns one head of one
// unit (a chain of segments, each the only child of the one before) and each
// group of kCols adjacent lanes kCols value columns, c + (128 /
// kCols) m: the lane of part p holds rows 4 kCols x + 4p .. +3 of those
// columns (128 fp32 registers in all), and the group adds its partial
// products with log2(kCols) shuffles. Each lane reads only its share of a
// staged key or query row (shared-memory broadcasts, the shares in different
// banks), so the staged bytes read per token and head fall with kCols while
// the shuffles and per-column scalars grow; two columns a lane is the faster
// of two and four. Both products a token needs come from the state before it,
//   x1 = S_{t-1}^T k_t,  x2 = S_{t-1}^T q_t,
//   delta_t = beta_t (v_t - exp(g_t) x1),  o_t = exp(g_t) x2 + delta_t (k_t . q_t),
// so one pass over the registers updates S with token t and forms x1, x2 of
// token t + 1 in independent accumulation chains. The registers hold
// S' = S / A, A the product of the decays exp(g) since the state was last
// held in full, so the update is one fused multiply-add per element,
// S' += k (delta / A); when A would fall below 2^-40 (or one decay does) the
// token takes the plain update, S' = (A exp(g)) S' + k delta^T, and A is 1
// again. Scaled back by A, the rounding stays that of the plain recurrence.
// The CTA walks the unit's tokens in DFS order, 32 at a time staged in shared
// memory as fp32 (with k . q per token); at a segment's first token the state
// is the initial state (a root), kept in registers (its parent is the segment
// before it), or, at the unit's first segment, its parent's end state, and the
// products come from a pass of their own (likewise after a chunk's last
// token); every segment's end state is written out. The units of one level
// (its branch-point depth: the children of a segment with several children
// start new units, one level below) are one launch, longest first, so sibling
// branches run side by side once their parent's state exists.
//
// 3 Dk Dv fused multiply-adds per token and head (the state update and the
// two products), issued as packed fp32 pairs; the staged rows each lane reads
// per token (3 x 64 floats of shared memory) weigh as much.
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

// A shared-memory read the compiler must issue where it stands: left free to
// move, the loads of a pass are hoisted ahead of their uses and the kernel
// runs 3-5 % slower at the same register count.
__device__ __forceinline__ float4 lds4(const float* p) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return r;
}

__device__ __forceinline__ void put(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void put(float* p, float x) { *p = x; }

constexpr int kCols = 2;                // value columns per lane
constexpr int kPairs = kD / kCols / 2;  // row pairs per lane and column
constexpr int kStep = 4 * kCols;        // row stride between a lane's groups of 4
constexpr int kChains = 4 / kCols;      // accumulation chains per column and product

// This lane's partial products of its columns with a staged key and query
// row (its kD / kCols rows).
struct Acc {
  float2 a[kCols][2][kChains];  // [column][product: k, q][chain]
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int c = 0; c < kCols; ++c)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int z = 0; z < kChains; ++z) a[c][m][z] = make_float2(0.f, 0.f);
  }
  // rows kStep x + 4p .. +3: pairs 2x (first two rows) and 2x + 1 of each column
  __device__ __forceinline__ void add(const float2 (&S)[kCols][kPairs], int x, const float4& kk,
                                      const float4& qq) {
    const float2 k0 = make_float2(kk.x, kk.y), k1 = make_float2(kk.z, kk.w);
    const float2 q0 = make_float2(qq.x, qq.y), q1 = make_float2(qq.z, qq.w);
    const int z = x % kChains;
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      a[c][0][z] = __ffma2_rn(S[c][2 * x], k0, __ffma2_rn(S[c][2 * x + 1], k1, a[c][0][z]));
      a[c][1][z] = __ffma2_rn(S[c][2 * x], q0, __ffma2_rn(S[c][2 * x + 1], q1, a[c][1][z]));
    }
  }
  // the columns' full products: this lane's part plus the group's others
  __device__ __forceinline__ void total(float (&x1)[kCols], float (&x2)[kCols]) const {
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      float p1 = 0.f, p2 = 0.f;
#pragma unroll
      for (int z = 0; z < kChains; ++z) {
        p1 += a[c][0][z].x + a[c][0][z].y;
        p2 += a[c][1][z].x + a[c][1][z].y;
      }
#pragma unroll
      for (int m = 1; m < kCols; m <<= 1) {
        p1 += __shfl_xor_sync(0xffffffffu, p1, m);
        p2 += __shfl_xor_sync(0xffffffffu, p2, m);
      }
      x1[c] = p1;
      x2[c] = p2;
    }
  }
};

// x1, x2 of this lane's columns from the state as it stands (kr, qr: this
// lane's share of the staged rows, at column offset 4p)
__device__ __forceinline__ void products(const float2 (&S)[kCols][kPairs], const float* kr,
                                         const float* qr, float (&x1)[kCols], float (&x2)[kCols]) {
  Acc acc;
  acc.zero();
#pragma unroll
  for (int x = 0; x < kPairs / 2; ++x) acc.add(S, x, lds4(kr + kStep * x), lds4(qr + kStep * x));
  acc.total(x1, x2);
}

// The update of this lane's columns with token t's row kr: with kScaled,
// S' += k w (w = delta / A for the new A); else S' = c S' + k w (c = the old A
// times exp(g), w = delta, A then 1). With kn / qn (token t + 1's rows) also
// that token's products of S' (the caller scales them by A), in the same
// chains and order as products().
template <bool kNext, bool kScaled>
__device__ __forceinline__ void update(float2 (&S)[kCols][kPairs], const float* kr, float c,
                                       const float (&w)[kCols], const float* kn, const float* qn,
                                       float (&x1)[kCols], float (&x2)[kCols]) {
  const float2 c2 = make_float2(c, c);
  Acc acc;
  acc.zero();
#pragma unroll
  for (int x = 0; x < kPairs / 2; ++x) {
    const float4 kk = lds4(kr + kStep * x);
    const float2 k0 = make_float2(kk.x, kk.y), k1 = make_float2(kk.z, kk.w);
#pragma unroll
    for (int col = 0; col < kCols; ++col) {
      const float2 w2 = make_float2(w[col], w[col]);
      if (kScaled) {
        S[col][2 * x] = __ffma2_rn(k0, w2, S[col][2 * x]);
        S[col][2 * x + 1] = __ffma2_rn(k1, w2, S[col][2 * x + 1]);
      } else {
        S[col][2 * x] = __ffma2_rn(S[col][2 * x], c2, __fmul2_rn(k0, w2));
        S[col][2 * x + 1] = __ffma2_rn(S[col][2 * x + 1], c2, __fmul2_rn(k1, w2));
      }
    }
    if (kNext) acc.add(S, x, lds4(kn + kStep * x), lds4(qn + kStep * x));
  }
  if (kNext) acc.total(x1, x2);
}

constexpr float kMinScale = 9.094947e-13f;  // 2^-40: the smallest A the registers carry

template <typename T>
__global__ void __launch_bounds__(kThreads, 3) tree_gdn_fwd_kernel(const GdnArgs a, int unit0) {
  __shared__ __align__(16) float sk[kChunk][kD];
  __shared__ __align__(16) float sq[kChunk][kD];
  __shared__ __align__(16) float sv[kChunk][kD];
  __shared__ float sa[kChunk], sb[kChunk], skq[kChunk];  // exp(g), beta, k . q
  const int4 unit = a.units[unit0 + blockIdx.x];  // this CTA's chain of segments
  const int h = blockIdx.y;
  const int part = threadIdx.x % kCols;  // which rows of its columns this lane holds
  const int cb = threadIdx.x / kCols;    // its columns: cb + (kD / kCols) m
  const int hq = h / a.group;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  T* o = static_cast<T*>(a.o);
  const size_t state_elems = static_cast<size_t>(kD) * kD;
  auto state_ptr = [&](int seg) { return a.states + (static_cast<size_t>(seg) * a.hv + h) * state_elems; };
  // offset of (row kStep x + 4 part + 2y + e, column cb + (kD / kCols) c) in a
  // row-major [Dk, Dv] state
  auto at = [&](int x, int y, int e, int c) {
    return (kStep * x + 4 * part + 2 * y + e) * kD + cb + (kD / kCols) * c;
  };

  const int d0 = unit.x, d1 = unit.y;    // its DFS positions
  const int T0 = unit.z, T1 = unit.w;    // and tokens
  float2 S[kCols][kPairs];  // S'[c][2x + y] = rows kStep x + 4 part + 2y, +1 of column c
  float A = 1.f;            // the state is A times the registers
  int d = d0;
  int4 seg = a.segs[d];  // (segment id, first token, length, parent id)
  int prev = -2;         // the segment whose end state is in registers
  float x1[kCols], x2[kCols];  // the next token's products, when `ready`
#pragma unroll
  for (int c = 0; c < kCols; ++c) x1[c] = x2[c] = 0.f;
  bool ready = false;
  for (int c0 = T0; c0 < T1; c0 += kChunk) {
    const int n = min(kChunk, T1 - c0);
    // ---- stage the chunk as fp32: q and k rows of head hq, v rows of head h,
    // exp(g) and beta; k . q per token from the half-warp that staged its row
    __syncthreads();
    for (int base = 0; base < kChunk * (kD / 8); base += kThreads) {
      const int e = base + threadIdx.x, i = e / (kD / 8), c8 = (e % (kD / 8)) * 8;
      float dot = 0.f;
      if (i < n) {
        const size_t row = (static_cast<size_t>(c0 + i) * a.hk + hq) * kD + c8;
        const size_t vrow = (static_cast<size_t>(c0 + i) * a.hv + h) * kD + c8;
        float fk[8], fq[8], f[8];
        load8<T>(k + row, fk);
        *reinterpret_cast<float4*>(&sk[i][c8]) = make_float4(fk[0], fk[1], fk[2], fk[3]);
        *reinterpret_cast<float4*>(&sk[i][c8 + 4]) = make_float4(fk[4], fk[5], fk[6], fk[7]);
        load8<T>(q + row, fq);
        *reinterpret_cast<float4*>(&sq[i][c8]) = make_float4(fq[0], fq[1], fq[2], fq[3]);
        *reinterpret_cast<float4*>(&sq[i][c8 + 4]) = make_float4(fq[4], fq[5], fq[6], fq[7]);
        load8<T>(v + vrow, f);
        *reinterpret_cast<float4*>(&sv[i][c8]) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(&sv[i][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
#pragma unroll
        for (int u = 0; u < 8; ++u) dot = fmaf(fk[u], fq[u], dot);
      }
      // the 16 lanes of a half-warp hold one token's row
#pragma unroll
      for (int m = 8; m > 0; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
      if (i < n && (threadIdx.x & 15) == 0) skq[i] = dot;
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
#pragma unroll
          for (int c = 0; c < kCols; ++c)
#pragma unroll
            for (int x = 0; x < kPairs / 2; ++x)
#pragma unroll
              for (int y = 0; y < 2; ++y) S[c][2 * x + y] = make_float2(src[at(x, y, 0, c)], src[at(x, y, 1, c)]);
          A = 1.f;
        } else if (seg.w < 0) {
#pragma unroll
          for (int c = 0; c < kCols; ++c)
#pragma unroll
            for (int z = 0; z < kPairs; ++z) S[c][z] = make_float2(0.f, 0.f);
          A = 1.f;
        }
        ready = false;
      }
      const float* kr = &sk[i][4 * part];
      if (!ready) {  // products of the state, A S'
        products(S, kr, &sq[i][4 * part], x1, x2);
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          x1[c] *= A;
          x2[c] *= A;
        }
      }
      const float al = sa[i], be = sb[i], kq = skq[i];
      float delta[kCols];
#pragma unroll
      for (int c = 0; c < kCols; ++c) delta[c] = be * (sv[i][cb + (kD / kCols) * c] - al * x1[c]);
      // the group's lanes hold the same products: lane `part` writes column part
      float oc = 0.f;
#pragma unroll
      for (int c = 0; c < kCols; ++c)
        if (c == part) oc = fmaf(delta[c], kq, al * x2[c]);
      put(o + (static_cast<size_t>(t) * a.hv + h) * kD + cb + (kD / kCols) * part, oc);
      const bool seg_end = t == seg.y + seg.z - 1;
      const bool next = !seg_end && i + 1 < n;  // the next token is in this segment and chunk
      const float At = A * al;
      if (At >= kMinScale) {  // S' += k delta / A_t
        float w[kCols];
        const float inv = 1.f / At;
#pragma unroll
        for (int c = 0; c < kCols; ++c) w[c] = delta[c] * inv;
        if (next)
          update<true, true>(S, kr, 0.f, w, &sk[i + 1][4 * part], &sq[i + 1][4 * part], x1, x2);
        else
          update<false, true>(S, kr, 0.f, w, nullptr, nullptr, x1, x2);
        A = At;
      } else {  // S' = A_t S' + k delta, and A = 1
        if (next)
          update<true, false>(S, kr, At, delta, &sk[i + 1][4 * part], &sq[i + 1][4 * part], x1, x2);
        else
          update<false, false>(S, kr, At, delta, nullptr, nullptr, x1, x2);
        A = 1.f;
      }
      if (next) {
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          x1[c] *= A;
          x2[c] *= A;
        }
      }
      ready = next;
      if (seg_end) {  // the segment's last token: save its end state
        float* dst = state_ptr(seg.x);
#pragma unroll
        for (int c = 0; c < kCols; ++c)
#pragma unroll
          for (int x = 0; x < kPairs / 2; ++x)
#pragma unroll
            for (int y = 0; y < 2; ++y) {
              dst[at(x, y, 0, c)] = A * S[c][2 * x + y].x;
              dst[at(x, y, 1, c)] = A * S[c][2 * x + y].y;
            }
        prev = seg.x;
        if (++d < d1) seg = a.segs[d];
      }
    }
  }
}

}  // namespace

// One launch per level: a level's units start from end states that the
// launches before it wrote (stream order).
cudaError_t launch_gdn_fwd(const GdnArgs& a) {
  for (int l = 0; l < a.levels; ++l) {
    const int u0 = a.level_ptr[l], n = a.level_ptr[l + 1] - u0;
    const dim3 grid(n, a.hv);
    if (a.f32)
      tree_gdn_fwd_kernel<float><<<grid, kThreads, 0, a.stream>>>(a, u0);
    else
      tree_gdn_fwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, a.stream>>>(a, u0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace treeattn
