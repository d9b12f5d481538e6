// Tree-correct causal depthwise convolution.
//
// Tree Training (arXiv 2511.00413) App. A.3 "Tree-Correct Causal Convolution"
// (eq. 11 in §3.2): in DFS order the K-1 tokens just before a child segment
// belong to a sibling branch, so each segment takes its left context from its
// parent's last K-1 effective tokens instead (and those reach further up for
// short segments). Equivalently, token t sees its k-th predecessor on its own
// root-to-leaf path, pred_k(t), with zeros before the root:
//   y[t, c] = act(b[c] + sum_{k=0}^{K-1} w[c, K-1-k] x[pred_k(t), c])
// (weight index K-1 on the token itself, as in a causal conv1d). The host
// builds pred_k for k = 1..K-1 once per kernel size, and the inverse lists
// (which (t, k) read token u) for the backward's gather.
//
// All kernels stream rows of C channels (token-major [N, C], 8 channels per
// thread and access), so they are bound by memory bandwidth. The backward reads
// x and dy and writes dx once (one pass over each block's token range, the
// gradient at the pre-activation kept in registers), plus a gather over the
// inverse lists for the few tokens just before a branch into several
// children. It is deterministic: every dx is a sum in a fixed order, and
// dweight / dbias reduce fixed token ranges per block and then the blocks in
// order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <string>
#include <vector>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace treeattn {
namespace {

using namespace dev;

constexpr int kConvThreads = 256;
// The forward and the backward stage the rows they stream (x; x and dy) through
// shared memory with bulk copies: a block's slice of a row (its 2048 channels)
// per token, kConvBatchBytes per tensor and batch, kConvBufs batches in flight.
constexpr uint32_t kConvBatchBytes = 16 * 1024;
constexpr int kConvBufs = 3;
constexpr int kSiteConv = 40000;  // status word of a conv wait that gave up: 40000 + line
constexpr int kConvPartialBlocks = 512;  // token ranges of the backward (and its dweight / dbias sums)

// V consecutive channels of one row (V = 4 or 8: one 8- or 16-byte access
// in bf16, one or two 16-byte accesses in fp32)
template <typename T, int V>
struct Vec;
template <int V>
struct Vec<__nv_bfloat16, V> {
  static_assert(V == 2 || V == 4 || V == 8, "2, 4 or 8 channels");
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[V]) {
    uint32_t w[V / 2];
    if constexpr (V == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if constexpr (V == 2) {
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      w[0] = u.x; w[1] = u.y;
    }
#pragma unroll
    for (int j = 0; j < V / 2; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[V]) {
    uint32_t w[V / 2];
#pragma unroll
    for (int j = 0; j < V / 2; ++j) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if constexpr (V == 8)
      *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else if constexpr (V == 2)
      *reinterpret_cast<uint32_t*>(p) = w[0];
    else
      *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  }
};
template <int V>
struct Vec<float, V> {
  static_assert(V == 2 || V == 4 || V == 8, "2, 4 or 8 channels");
  static __device__ __forceinline__ void load(const float* p, float (&v)[V]) {
    if constexpr (V == 2) {
      const float2 a = *reinterpret_cast<const float2*>(p);
      v[0] = a.x;
      v[1] = a.y;
      return;
    }
#pragma unroll
    for (int h = 0; h < V / 4; ++h) {
      const float4 a = reinterpret_cast<const float4*>(p)[h];
      v[4 * h] = a.x; v[4 * h + 1] = a.y; v[4 * h + 2] = a.z; v[4 * h + 3] = a.w;
    }
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[V]) {
    if constexpr (V == 2) {
      *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
      return;
    }
#pragma unroll
    for (int h = 0; h < V / 4; ++h)
      reinterpret_cast<float4*>(p)[h] = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
  }
};

// SiLU and its derivative, from the fast exponential and division intrinsics
// (relative error near 1e-7: within the fp32 tolerance of the outputs).
__device__ __forceinline__ float sigmoid(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }
__device__ __forceinline__ float silu(float z) { return z * sigmoid(z); }
__device__ __forceinline__ float silu_grad(float z) {
  const float s = sigmoid(z);
  return s * (1.f + z * (1.f - s));
}

// Each thread owns one chunk of V channels (q) for the whole launch and keeps
// their K weights (and biases) in registers; blocks stride over tokens, and
// blockIdx.y picks the group of 256 chunks.
template <int K, int V = 8>
struct Taps {
  float w[V][K];
  __device__ __forceinline__ void load(const float* weight, int q) {
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
      for (int k = 0; k < K; ++k) w[j][k] = __ldg(weight + (V * q + j) * K + k);
  }
};

// token read by token t at distance k (k = 0 is t itself); -1 before the root
template <int K>
__device__ __forceinline__ int pred_of(const ConvArgs& a, int t, int k) {
  return k == 0 ? t : __ldg(a.pred + static_cast<size_t>(t) * (K - 1) + (k - 1));
}

// The K rows token t reads, x[pred_k(t)] for k = 0..K-1, for one chunk of V
// channels. A thread walks a contiguous token range: when t's immediate path
// predecessor is t-1 (inside a segment, or a first child right after its
// parent) the window shifts by one row; otherwise it is reloaded from the
// predecessor table (segment starts). The next token's row and predecessor
// are loaded one token ahead.
template <typename T, int K, int V = 8>
struct Window {
  float v[K][V];
  __device__ __forceinline__ void reload(const ConvArgs& a, int t, int q, const float (&xt)[V]) {
    const T* x = static_cast<const T*>(a.x);
#pragma unroll
    for (int j = 0; j < V; ++j) v[0][j] = xt[j];
#pragma unroll
    for (int k = 1; k < K; ++k) {
      const int u = pred_of<K>(a, t, k);
      if (u < 0) {
#pragma unroll
        for (int j = 0; j < V; ++j) v[k][j] = 0.f;  // before the root
      } else {
        Vec<T, V>::load(x + static_cast<size_t>(u) * a.C + V * q, v[k]);
      }
    }
  }
  __device__ __forceinline__ void shift(const float (&xt)[V]) {
#pragma unroll
    for (int k = K - 1; k > 0; --k)
#pragma unroll
      for (int j = 0; j < V; ++j) v[k][j] = v[k - 1][j];
#pragma unroll
    for (int j = 0; j < V; ++j) v[0][j] = xt[j];
  }
  // the pre-activation, channels in packed pairs
  __device__ __forceinline__ void pre(const Taps<K, V>& tp, const float (&b)[V], float (&z)[V]) const {
    float2 z2[V / 2];
#pragma unroll
    for (int jp = 0; jp < V / 2; ++jp) z2[jp] = make_float2(b[2 * jp], b[2 * jp + 1]);
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
      for (int jp = 0; jp < V / 2; ++jp)
        z2[jp] = __ffma2_rn(make_float2(tp.w[2 * jp][K - 1 - k], tp.w[2 * jp + 1][K - 1 - k]),
                            make_float2(v[k][2 * jp], v[k][2 * jp + 1]), z2[jp]);
#pragma unroll
    for (int jp = 0; jp < V / 2; ++jp) {
      z[2 * jp] = z2[jp].x;
      z[2 * jp + 1] = z2[jp].y;
    }
  }
};

// a block's contiguous token range
__device__ __forceinline__ void token_range(const ConvArgs& a, int& t0, int& t1) {
  const int per = (a.N + gridDim.x - 1) / gridDim.x;
  t0 = blockIdx.x * per;
  t1 = min(a.N, t0 + per);
}

// Bulk-copy staging of NT token-major tensors for one block: batch i (tokens
// tb .. tb+n-1) of tensor s sits at buf + (i % kConvBufs) * NT * kConvBatchBytes
// + s * kConvBatchBytes, token u of the batch at u * (row stride).
template <typename T, int NT, int V = 8>
struct Stage {
  static constexpr uint32_t kStride = kConvThreads * V * sizeof(T);  // smem bytes per token row
  // tokens per batch: as many rows as kConvBatchBytes holds, at most 8
  static constexpr int kBatch = static_cast<int>(kConvBatchBytes / kStride) < 8
                                    ? static_cast<int>(kConvBatchBytes / kStride) : 8;
  static constexpr uint32_t kBytes = kBatch * kStride;  // one tensor's batch buffer
  uint8_t* buf;
  uint64_t* bar;       // [kConvBufs]
  const T* src[NT];
  int C, g0;           // channels; the group's first channel
  uint32_t row_bytes;  // bytes of a token's slice (the group's channels)
  int t0, te;          // tokens staged: [t0, te)
  __device__ int batches() const { return (te - t0 + kBatch - 1) / kBatch; }
  // issued by one thread
  __device__ void issue(int i) const {
    const int s = i % kConvBufs, tb = t0 + i * kBatch, n = min(kBatch, te - tb);
    uint64_t* b = bar + s;
    mbar_arrive_expect_tx(b, static_cast<uint32_t>(n) * row_bytes * NT);
    for (int u = 0; u < n; ++u)
#pragma unroll
      for (int k = 0; k < NT; ++k)
        bulk_load(buf + (s * NT + k) * kBytes + u * kStride,
                  src[k] + static_cast<size_t>(tb + u) * C + g0, row_bytes, b);
  }
  __device__ const uint8_t* row(int i, int k, int u) const {
    return buf + ((i % kConvBufs) * NT + k) * kBytes + u * kStride;
  }
};

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads) conv_fwd_kernel(const ConvArgs a) {
  extern __shared__ __align__(128) uint8_t cbuf[];
  __shared__ uint64_t bar[kConvBufs];
  __shared__ int abort_s;
  const int q = blockIdx.y * kConvThreads + threadIdx.x;
  const bool valid = q < a.C / 8;
  Stage<T, 1> st;
  st.buf = cbuf;
  st.bar = bar;
  st.src[0] = static_cast<const T*>(a.x);
  st.C = a.C;
  st.g0 = blockIdx.y * kConvThreads * 8;
  st.row_bytes = static_cast<uint32_t>(min(kConvThreads * 8, a.C - st.g0) * sizeof(T));
  token_range(a, st.t0, st.te);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kConvBufs; ++i) mbar_init(&bar[i], 1);
    abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int nb = st.t0 < st.te ? st.batches() : 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kConvBufs && i < nb; ++i) st.issue(i);
  Taps<K> tp;
  float b[8];
  if (valid) {
    tp.load(a.weight, q);
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = a.bias ? __ldg(a.bias + 8 * q + j) : 0.f;
  }
  T* y = static_cast<T*>(a.y);
  Window<T, K> win;
  constexpr int B = Stage<T, 1>::kBatch;
  int i = 0;
  for (; i < nb; ++i) {
    const int tb = st.t0 + i * B, n = min(B, st.te - tb);
    int p1[B];  // the batch's immediate path predecessors
#pragma unroll
    for (int u = 0; u < B; ++u) p1[u] = u < n ? (K > 1 ? pred_of<K>(a, tb + u, 1) : tb + u - 1) : -1;
    const bool ok = mbar_wait(&bar[i % kConvBufs], (i / kConvBufs) & 1, &abort_s, a.status,
                              kSiteConv + __LINE__);
    if (!__syncthreads_and(ok)) break;
    if (valid) {
#pragma unroll
      for (int u = 0; u < B; ++u) {
        if (u >= n) break;
        const int t = tb + u;
        float xt[8];
        Vec<T, 8>::load(reinterpret_cast<const T*>(st.row(i, 0, u)) + 8 * threadIdx.x, xt);
        if (t > st.t0 && p1[u] == t - 1)
          win.shift(xt);
        else
          win.reload(a, t, q, xt);
        float z[8];
        win.pre(tp, b, z);
        if (a.act == 1) {
#pragma unroll
          for (int j = 0; j < 8; ++j) z[j] = silu(z[j]);
        }
        Vec<T, 8>::store(y + static_cast<size_t>(t) * a.C + 8 * q, z);
      }
    }
    __syncthreads();  // every thread is done with this batch's buffer
    if (threadIdx.x == 0 && i + kConvBufs < nb) st.issue(i + kConvBufs);
  }
  if (i < nb && threadIdx.x == 0)  // gave up a wait: let the copies in flight land
    for (int k = i; k < nb && k < i + kConvBufs; ++k) mbar_drain(&bar[k % kConvBufs], (k / kConvBufs) & 1);
}

// Blocks per SM of the backward's walk by registers: at 2 channels a thread
// four for up to 4 taps (64 registers, no spills), three for 5 and 6 (at most
// 85), two beyond; at 4 channels two for up to 5 taps; one otherwise. The
// launch also caps it by shared memory (fp32 rows stage twice the bytes).
constexpr int conv_bwd_blocks_per_sm(int K, int V) {
  return V == 2 ? (K <= 4 ? 4 : K <= 6 ? 3 : 2) : (V == 4 && K <= 5 ? 2 : 1);
}

// The backward in one pass over each block's token range, in DFS order:
//   g[t]  = dy[t] * act'(pre_t), from the window that the forward also walks;
//   dweight[c, K-1-k] += g[t] x[pred_k(t)] and dbias[c] += g[t] for t in the
//   range (per-block sums, reduced in block order afterwards);
//   dx[u] = sum over k of w[c, K-1-k] g[u+k] over the k for which u, u+1, ..,
//   u+k is an unbroken run of path steps (each token's path predecessor is
//   the one before it in DFS order), which is every (t, k) with pred_k(t) = u
//   unless u is listed as irregular (some reader of u lies after a jump in
//   the DFS order: a second or later child); those get dx from
//   conv_bwd_dx_irregular_kernel. The walk runs K-1 tokens past the range
//   (g only) so the range's last tokens see their readers; g never leaves
//   registers.
template <typename T, int K, int V>
__global__ void __launch_bounds__(kConvThreads, conv_bwd_blocks_per_sm(K, V))
    conv_bwd_fused_kernel(const ConvArgs a) {
  extern __shared__ __align__(128) uint8_t cbuf[];
  __shared__ uint64_t bar[kConvBufs];
  __shared__ int abort_s;
  const int q = blockIdx.y * kConvThreads + threadIdx.x;
  const bool valid = q < a.C / V;
  int t0, t1;
  token_range(a, t0, t1);
  Stage<T, 2, V> st;
  st.buf = cbuf;
  st.bar = bar;
  st.src[0] = static_cast<const T*>(a.x);
  st.src[1] = static_cast<const T*>(a.dy);
  st.C = a.C;
  st.g0 = blockIdx.y * kConvThreads * V;
  st.row_bytes = static_cast<uint32_t>(min(kConvThreads * V, a.C - st.g0) * sizeof(T));
  st.t0 = t0;
  st.te = t0 < t1 ? min(a.N, t1 + K - 1) : t0;  // K-1 tokens past the range: their g
  if (threadIdx.x == 0) {
    for (int i = 0; i < kConvBufs; ++i) mbar_init(&bar[i], 1);
    abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int nb = st.t0 < st.te ? st.batches() : 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kConvBufs && i < nb; ++i) st.issue(i);
  Taps<K, V> tp;
  float b[V];
  if (valid) {
    tp.load(a.weight, q);
#pragma unroll
    for (int j = 0; j < V; ++j) b[j] = a.bias ? __ldg(a.bias + V * q + j) : 0.f;
  }
  T* dx = static_cast<T*>(a.dx);
  float acc[K + 1][V];
#pragma unroll
  for (int k = 0; k <= K; ++k)
#pragma unroll
    for (int j = 0; j < V; ++j) acc[k][j] = 0.f;
  float gh[K][V];  // gh[k] = g of the token k steps back in DFS order
#pragma unroll
  for (int k = 0; k < K; ++k)
#pragma unroll
    for (int j = 0; j < V; ++j) gh[k][j] = 0.f;
  uint32_t cont = 0;  // bit k: the token k steps back follows its DFS predecessor on its path
  Window<T, K, V> win;
  constexpr int B = Stage<T, 2, V>::kBatch;
  const int tend = t0 < t1 ? t1 + K - 1 : t0;  // walk end, virtual tokens past N included
  const int nsteps = (tend - t0 + B - 1) / B;  // batches of the walk (the last ones may be virtual)
  int i = 0;
  bool ok = true;
  for (; i < nsteps; ++i) {
    const int tb = t0 + i * B;
    const int n = i < nb ? min(B, st.te - tb) : 0;  // real tokens of this batch
    int p1[B];
#pragma unroll
    for (int u = 0; u < B; ++u) p1[u] = u < n ? (K > 1 ? pred_of<K>(a, tb + u, 1) : tb + u - 1) : -1;
    if (i < nb) {
      ok = mbar_wait(&bar[i % kConvBufs], (i / kConvBufs) & 1, &abort_s, a.status, kSiteConv + __LINE__);
      if (!__syncthreads_and(ok)) break;
    }
    if (valid) {
#pragma unroll
      for (int u = 0; u < B; ++u) {
        const int t = tb + u;
        if (t >= tend) break;
        float g[V];
        bool step = false;
        if (u < n) {
          float xt[V];
          Vec<T, V>::load(reinterpret_cast<const T*>(st.row(i, 0, u)) + V * threadIdx.x, xt);
          Vec<T, V>::load(reinterpret_cast<const T*>(st.row(i, 1, u)) + V * threadIdx.x, g);
          step = p1[u] == t - 1;
          if (t > t0 && step)
            win.shift(xt);
          else
            win.reload(a, t, q, xt);
          if (a.act == 1) {
            float z[V];
            win.pre(tp, b, z);
#pragma unroll
            for (int j = 0; j < V; ++j) g[j] *= silu_grad(z[j]);
          }
          if (t < t1) {
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
              for (int jp = 0; jp < V / 2; ++jp) {
                const float2 r2 = __ffma2_rn(make_float2(g[2 * jp], g[2 * jp + 1]),
                                             make_float2(win.v[k][2 * jp], win.v[k][2 * jp + 1]),
                                             make_float2(acc[k][2 * jp], acc[k][2 * jp + 1]));
                acc[k][2 * jp] = r2.x;
                acc[k][2 * jp + 1] = r2.y;
              }
#pragma unroll
            for (int j = 0; j < V; ++j) acc[K][j] += g[j];
          }
        } else {  // past the last token: no readers
#pragma unroll
          for (int j = 0; j < V; ++j) g[j] = 0.f;
        }
#pragma unroll
        for (int k = K - 1; k > 0; --k)
#pragma unroll
          for (int j = 0; j < V; ++j) gh[k][j] = gh[k - 1][j];
#pragma unroll
        for (int j = 0; j < V; ++j) gh[0][j] = g[j];
        cont = (cont << 1) | (step ? 1u : 0u);
        // token u0 = t - (K-1) now has all of its run readers u0 .. t
        const int u0 = t - (K - 1);
        if (u0 >= t0 && u0 < a.N && !(__ldg(a.irr_bits + (u0 >> 5)) >> (u0 & 31) & 1u)) {
          float2 o2[V / 2];
#pragma unroll
          for (int jp = 0; jp < V / 2; ++jp)  // k = 0: u0 itself
            o2[jp] = __fmul2_rn(make_float2(tp.w[2 * jp][K - 1], tp.w[2 * jp + 1][K - 1]),
                                make_float2(gh[K - 1][2 * jp], gh[K - 1][2 * jp + 1]));
          bool run = true;
#pragma unroll
          for (int k = 1; k < K; ++k) {
            run = run && ((cont >> (K - 1 - k)) & 1u);  // u0 + k follows u0 + k - 1
            if (run) {
#pragma unroll
              for (int jp = 0; jp < V / 2; ++jp)
                o2[jp] = __ffma2_rn(make_float2(tp.w[2 * jp][K - 1 - k], tp.w[2 * jp + 1][K - 1 - k]),
                                    make_float2(gh[K - 1 - k][2 * jp], gh[K - 1 - k][2 * jp + 1]), o2[jp]);
            }
          }
          float o[V];
#pragma unroll
          for (int jp = 0; jp < V / 2; ++jp) {
            o[2 * jp] = o2[jp].x;
            o[2 * jp + 1] = o2[jp].y;
          }
          Vec<T, V>::store(dx + static_cast<size_t>(u0) * a.C + V * q, o);
        }
      }
    }
    if (i < nb) {
      __syncthreads();  // every thread is done with this batch's buffer
      if (threadIdx.x == 0 && i + kConvBufs < nb) st.issue(i + kConvBufs);
    }
  }
  if (!ok && threadIdx.x == 0)  // gave up a wait: let the copies in flight land
    for (int k = i; k < nb && k < i + kConvBufs; ++k) mbar_drain(&bar[k % kConvBufs], (k / kConvBufs) & 1);
  if (valid) {
    float* part = a.partial + static_cast<size_t>(blockIdx.x) * (K + 1) * a.C;
#pragma unroll
    for (int k = 0; k <= K; ++k)
#pragma unroll
      for (int j = 0; j < V; ++j) part[static_cast<size_t>(k) * a.C + V * q + j] = acc[k][j];
  }
}

// dx of the irregular tokens: the gather over every (t, k) with pred_k(t) = u
// in list order, g[t] recomputed from t's window and dy[t]
template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads) conv_bwd_dx_irregular_kernel(const ConvArgs a) {
  const int q = blockIdx.y * kConvThreads + threadIdx.x;
  if (q >= a.C / 8) return;
  Taps<K> tp;
  tp.load(a.weight, q);
  float b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = a.bias ? __ldg(a.bias + 8 * q + j) : 0.f;
  const T* x = static_cast<const T*>(a.x);
  const T* dy = static_cast<const T*>(a.dy);
  T* dx = static_cast<T*>(a.dx);
  for (int i = blockIdx.x; i < a.num_irr; i += gridDim.x) {
    const int u = __ldg(a.irr_list + i);
    const int e0 = __ldg(a.succ_ptr + u), e1 = __ldg(a.succ_ptr + u + 1);
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int e = e0; e < e1; ++e) {
      const int packed = __ldg(a.succ + e), t = packed >> 3, k = packed & 7;
      float g[8];
      Vec<T, 8>::load(dy + static_cast<size_t>(t) * a.C + 8 * q, g);
      if (a.act == 1) {
        float xt[8];
        Vec<T, 8>::load(x + static_cast<size_t>(t) * a.C + 8 * q, xt);
        Window<T, K> win;
        win.reload(a, t, q, xt);
        float z[8];
        win.pre(tp, b, z);
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] *= silu_grad(z[j]);
      }
#pragma unroll
      for (int kk = 0; kk < K; ++kk) {  // select tap k without indexing registers at run time
        if (kk != k) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = fmaf(tp.w[j][K - 1 - kk], g[j], o[j]);
      }
    }
    Vec<T, 8>::store(dx + static_cast<size_t>(u) * a.C + 8 * q, o);
  }
}

// dweight[c, K-1-k] and dbias[c]: the blocks' partial sums in block order
__global__ void __launch_bounds__(kConvThreads) conv_bwd_dw_reduce_kernel(const ConvArgs a, int blocks) {
  const int total = (a.K + 1) * a.C;
  for (int e = blockIdx.x * kConvThreads + threadIdx.x; e < total; e += gridDim.x * kConvThreads) {
    float s = 0.f;
    for (int b = 0; b < blocks; ++b) s += a.partial[static_cast<size_t>(b) * total + e];
    const int k = e / a.C, c = e % a.C;
    if (k < a.K)
      a.dweight[c * a.K + (a.K - 1 - k)] = s;
    else if (a.dbias)
      a.dbias[c] = s;
  }
}


}  // namespace

// pred[t][k-1] for k = 1..K-1 (-1 before the root) and the inverse lists,
// from the plan's DFS layout; uploaded into one device block owned by the plan.
tree_status_t conv_tables_build(tree_plan* p, int K, cudaStream_t stream) {
  if (p->conv.block && p->conv.K == K) {
    int cur = -1;
    if (cudaGetDevice(&cur) == cudaSuccess && cur == p->conv.device) return TREE_OK;
  }
  conv_tables_free(p);
  const int32_t N = p->N, S = p->S;
  const auto& seg = p->field[TREE_FIELD_TOKEN_SEG];
  const auto& start = p->field[TREE_FIELD_SEG_START];
  const auto& anc_ptr = p->field[TREE_FIELD_ANC_PTR];
  const auto& anc_idx = p->field[TREE_FIELD_ANC_IDX];
  std::vector<int32_t> parent(S), len(S, 0);
  for (int32_t t = 0; t < N; ++t) ++len[seg[t]];
  for (int32_t s = 0; s < S; ++s) parent[s] = anc_ptr[s + 1] > anc_ptr[s] ? anc_idx[anc_ptr[s + 1] - 1] : -1;
  const int W = K - 1;
  std::vector<int32_t> pred(static_cast<size_t>(N) * (W > 0 ? W : 1), -1);
  for (int32_t t = 0; t < N; ++t)
    for (int k = 1; k <= W; ++k) {
      int32_t u = t, m = k;  // step back m tokens along the path from u
      while (u >= 0 && m > 0) {
        const int32_t s = seg[u], off = u - start[s];
        if (m <= off) {
          u -= m;
          m = 0;
        } else {  // leave the segment: continue from the parent's last token
          m -= off + 1;
          u = parent[s] < 0 ? -1 : start[parent[s]] + len[parent[s]] - 1;
        }
      }
      pred[static_cast<size_t>(t) * W + (k - 1)] = u;
    }
  std::vector<int32_t> ptr(N + 1, 0);
  for (int32_t t = 0; t < N; ++t) {
    ++ptr[t + 1];  // k = 0: itself
    for (int k = 1; k <= W; ++k) {
      const int32_t u = pred[static_cast<size_t>(t) * W + (k - 1)];
      if (u >= 0) ++ptr[u + 1];
    }
  }
  for (int32_t u = 0; u < N; ++u) ptr[u + 1] += ptr[u];
  std::vector<int32_t> succ(ptr[N]), fill(ptr.begin(), ptr.end() - 1);
  for (int32_t t = 0; t < N; ++t) {  // entries in increasing t: a fixed order
    succ[fill[t]++] = t << 3;
    for (int k = 1; k <= W; ++k) {
      const int32_t u = pred[static_cast<size_t>(t) * W + (k - 1)];
      if (u >= 0) succ[fill[u]++] = (t << 3) | k;
    }
  }
  // Irregular tokens: some reader (t, k) of u is not u + k reached by k
  // single path steps along the DFS order (step[t]: t's path predecessor is
  // t - 1).
  std::vector<uint32_t> irr_bits((static_cast<size_t>(N) + 31) / 32, 0u);
  std::vector<int32_t> irr_list;
  {
    std::vector<uint8_t> step(N, 0);
    for (int32_t t = 1; t < N; ++t) step[t] = W > 0 && pred[static_cast<size_t>(t) * W] == t - 1;
    for (int32_t u = 0; u < N; ++u) {
      bool regular = true;
      for (int32_t e = ptr[u]; e < ptr[u + 1] && regular; ++e) {
        const int32_t t = succ[e] >> 3, k = succ[e] & 7;
        if (t != u + k) {
          regular = false;
          break;
        }
        for (int32_t j = 1; j <= k; ++j)
          if (!step[u + j]) regular = false;
      }
      if (!regular) {
        irr_bits[u >> 5] |= 1u << (u & 31);
        irr_list.push_back(u);
      }
    }
  }
  auto round256 = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t b_pred = round256(pred.size() * 4), b_ptr = round256(ptr.size() * 4),
               b_succ = round256(succ.size() * 4 + 4), b_bits = round256(irr_bits.size() * 4 + 4),
               b_irr = round256(irr_list.size() * 4 + 4);
  void* block = nullptr;
  cudaError_t e = cudaMalloc(&block, b_pred + b_ptr + b_succ + b_bits + b_irr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TREE_ERR_OOM, std::string("cudaMalloc of the conv tables: ") + cudaGetErrorString(e));
  }
  uint8_t* base = static_cast<uint8_t*>(block);
  e = cudaMemcpyAsync(base, pred.data(), pred.size() * 4, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(base + b_pred, ptr.data(), ptr.size() * 4, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess && !succ.empty())
    e = cudaMemcpyAsync(base + b_pred + b_ptr, succ.data(), succ.size() * 4, cudaMemcpyHostToDevice, stream);
  uint8_t* const p_bits = base + b_pred + b_ptr + b_succ;
  if (e == cudaSuccess && !irr_bits.empty())
    e = cudaMemcpyAsync(p_bits, irr_bits.data(), irr_bits.size() * 4, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess && !irr_list.empty())
    e = cudaMemcpyAsync(p_bits + b_bits, irr_list.data(), irr_list.size() * 4, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaFree(block);
    return fail(TREE_ERR_CUDA, std::string("conv table upload: ") + cudaGetErrorString(e));
  }
  int cur = 0;
  cudaGetDevice(&cur);
  p->conv.block = block;
  p->conv.device = cur;
  p->conv.K = K;
  p->conv.pred = reinterpret_cast<const int32_t*>(base);
  p->conv.succ_ptr = reinterpret_cast<const int32_t*>(base + b_pred);
  p->conv.succ = reinterpret_cast<const int32_t*>(base + b_pred + b_ptr);
  p->conv.irr_bits = reinterpret_cast<const uint32_t*>(p_bits);
  p->conv.irr_list = reinterpret_cast<const int32_t*>(p_bits + b_bits);
  p->conv.num_irr = static_cast<int>(irr_list.size());
  return TREE_OK;
}

void conv_tables_free(tree_plan* p) {
  if (!p->conv.block) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != p->conv.device) cudaSetDevice(p->conv.device);
  cudaFree(p->conv.block);
  if (cur >= 0 && cur != p->conv.device) cudaSetDevice(cur);
  p->conv = ConvTables{};
}

size_t conv_bwd_workspace(int N, int C, int K) {
  (void)N;
  return static_cast<size_t>(kConvPartialBlocks) * (K + 1) * C * 4 + 256;
}

// dynamic shared memory of the staged kernels, set once per instantiation
template <typename F>
cudaError_t smem_attr(F* kernel, uint32_t bytes, bool& done) {
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done = true;
  return e;
}

constexpr uint32_t kFwdSmem = kConvBufs * kConvBatchBytes;      // x
// Channels per thread in the backward's walk. Its per-thread state (the
// window, the last K gradients, the dweight / dbias sums and the taps) at 4
// channels fits two 256-thread blocks per SM up to 5 taps; beyond, 2 channels
// keep two or three blocks per SM where 4 would leave one (6 taps: 1.90 ->
// 1.66 ms on 131k tokens x 4096 channels). Up to 5 taps 4 channels are faster
// than 2 (4 taps: 1.07 against 1.29 ms), as a thread's per-token overhead
// then covers twice the channels.
constexpr int bwd_channels(int K) { return K <= 5 ? 4 : 2; }
template <typename T, int V>
constexpr uint32_t bwd_smem() {  // x and dy
  return kConvBufs * 2 * Stage<T, 2, V>::kBytes;
}

template <int K>
cudaError_t conv_fwd_k(const ConvArgs& a, dim3 grid) {
  static bool done[2] = {false, false};
  cudaError_t e;
  if (a.f32) {
    if ((e = smem_attr(conv_fwd_kernel<float, K>, kFwdSmem, done[1])) != cudaSuccess) return e;
    conv_fwd_kernel<float, K><<<grid, kConvThreads, kFwdSmem, a.stream>>>(a);
  } else {
    if ((e = smem_attr(conv_fwd_kernel<__nv_bfloat16, K>, kFwdSmem, done[0])) != cudaSuccess) return e;
    conv_fwd_kernel<__nv_bfloat16, K><<<grid, kConvThreads, kFwdSmem, a.stream>>>(a);
  }
  return cudaGetLastError();
}

// blocks: groups of 256 chunks of `chans` channels (y) times token ranges
// (x), `per_sm` blocks per SM in all (two 256-thread blocks per SM for the
// forward and the backward's walk)
dim3 conv_grid(const ConvArgs& a, int per_sm, int chans = 8) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  const int groups = (a.C / chans + kConvThreads - 1) / kConvThreads;
  int tx = sms * per_sm / groups;
  tx = tx < 1 ? 1 : (tx > a.N ? a.N : tx);
  return dim3(tx, groups);
}

// The walk over token ranges, then dx of the irregular tokens; *pblocks
// gets the token ranges (blocks along x), whose dweight / dbias partial sums
// the reduce kernel adds.
template <int K>
cudaError_t conv_bwd_k(const ConvArgs& a, dim3 grid, int* pblocks) {
  constexpr int V = bwd_channels(K);
  static bool done[2] = {false, false};
  // blocks per SM: by registers, and by shared memory (228 KB per SM, 1 KB of
  // it reserved per block)
  const uint32_t smem = a.f32 ? bwd_smem<float, V>() : bwd_smem<__nv_bfloat16, V>();
  const int by_smem = static_cast<int>(233472u / (smem + 1024u));
  const int by_regs = conv_bwd_blocks_per_sm(K, V);
  const dim3 pgrid = conv_grid(a, by_regs < by_smem ? by_regs : by_smem, V);
  *pblocks = static_cast<int>(pgrid.x) < kConvPartialBlocks ? static_cast<int>(pgrid.x) : kConvPartialBlocks;
  const dim3 pg(*pblocks, pgrid.y);
  const dim3 igrid(a.num_irr < 1024 ? (a.num_irr > 0 ? a.num_irr : 1) : 1024, grid.y);
  cudaError_t e;
  if (a.f32) {
    if ((e = smem_attr(conv_bwd_fused_kernel<float, K, V>, smem, done[1])) != cudaSuccess) return e;
    conv_bwd_fused_kernel<float, K, V><<<pg, kConvThreads, smem, a.stream>>>(a);
    if (a.num_irr > 0) conv_bwd_dx_irregular_kernel<float, K><<<igrid, kConvThreads, 0, a.stream>>>(a);
  } else {
    if ((e = smem_attr(conv_bwd_fused_kernel<__nv_bfloat16, K, V>, smem, done[0])) != cudaSuccess) return e;
    conv_bwd_fused_kernel<__nv_bfloat16, K, V><<<pg, kConvThreads, smem, a.stream>>>(a);
    if (a.num_irr > 0)
      conv_bwd_dx_irregular_kernel<__nv_bfloat16, K><<<igrid, kConvThreads, 0, a.stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_conv_fwd(const ConvArgs& a) {
  const dim3 grid = conv_grid(a, 2);
  switch (a.K) {
    case 1: return conv_fwd_k<1>(a, grid);
    case 2: return conv_fwd_k<2>(a, grid);
    case 3: return conv_fwd_k<3>(a, grid);
    case 4: return conv_fwd_k<4>(a, grid);
    case 5: return conv_fwd_k<5>(a, grid);
    case 6: return conv_fwd_k<6>(a, grid);
    case 7: return conv_fwd_k<7>(a, grid);
    case 8: return conv_fwd_k<8>(a, grid);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_conv_bwd(ConvArgs a) {
  const dim3 grid = conv_grid(a, 8);  // the irregular tokens' gather
  int pblocks = 0;
  cudaError_t e;
  switch (a.K) {
    case 1: e = conv_bwd_k<1>(a, grid, &pblocks); break;
    case 2: e = conv_bwd_k<2>(a, grid, &pblocks); break;
    case 3: e = conv_bwd_k<3>(a, grid, &pblocks); break;
    case 4: e = conv_bwd_k<4>(a, grid, &pblocks); break;
    case 5: e = conv_bwd_k<5>(a, grid, &pblocks); break;
    case 6: e = conv_bwd_k<6>(a, grid, &pblocks); break;
    case 7: e = conv_bwd_k<7>(a, grid, &pblocks); break;
    case 8: e = conv_bwd_k<8>(a, grid, &pblocks); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  const int total = (a.K + 1) * a.C;
  const int rblocks = (total + kConvThreads - 1) / kConvThreads;
  conv_bwd_dw_reduce_kernel<<<rblocks, kConvThreads, 0, a.stream>>>(a, pblocks);
  return cudaGetLastError();
}

}  // namespace treeattn
