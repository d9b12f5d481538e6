// C-ABI glue: plan upload, argument validation and dispatch to the kernels,
// the device status word.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "kernels.h"
#include "plan_internal.h"
#include "sched.cuh"

namespace treeattn {

// Set by kernels that give up a bounded wait; read and cleared by tree_status_sync.
__device__ int g_status_word = 0;

// Work counters of the persistent kernels, one slot per launch in turn; a
// launch's last CTA zeroes its slot.
__device__ SchedSlot g_sched[kSchedSlots];

SchedSlot* next_sched_slot() {
  static std::atomic<uint32_t> seq{0};
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_sched) != cudaSuccess) return nullptr;
  return static_cast<SchedSlot*>(p) + seq.fetch_add(1u) % kSchedSlots;
}

namespace {

tree_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(TREE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

int* status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct FieldSlot {
  tree_plan_field_t f;
  const int32_t** dst;
};

void free_device(tree_plan* p) {
  if (!p->dev.block) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != p->dev.device) cudaSetDevice(p->dev.device);
  cudaFree(p->dev.block);  // synchronizes the device
  if (cur >= 0 && cur != p->dev.device) cudaSetDevice(cur);
  p->dev = DevicePlan{};
}

tree_status_t check_plan_on_device(const tree_plan* p) {
  if (p->N == 0) return TREE_OK;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return fail(TREE_ERR_CUDA, "no CUDA device");
  if (!p->dev.block || p->dev.device != cur)
    return fail(TREE_ERR_NOT_ON_DEVICE, "call tree_plan_to_device on the current device first");
  return TREE_OK;
}

tree_status_t check_heads(int32_t hq, int32_t hkv, int32_t d, tree_dtype_t dtype) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0)
    return fail(TREE_ERR_INVALID_ARG, "need hq > 0, hkv > 0 and hq % hkv == 0");
  if (hq > 65535) return fail(TREE_ERR_UNSUPPORTED, "hq > 65535");
  if (dtype == TREE_DTYPE_F32) {
    if (d != 64 && d != 128) return fail(TREE_ERR_UNSUPPORTED, "fp32 path needs head_dim 64 or 128");
  } else if (dtype == TREE_DTYPE_BF16) {
    if (d != 128) return fail(TREE_ERR_UNSUPPORTED, "bf16 path needs head_dim 128");
  } else {
    return fail(TREE_ERR_INVALID_ARG, "unknown dtype");
  }
  return TREE_OK;
}

float resolve_scale(float s, int d) { return s == 0.f ? 1.f / std::sqrt(static_cast<float>(d)) : s; }

}  // namespace

// lse*log2(e) and Delta, each fp32 [hq, npad] (npad = 128 * number of q-tiles).
size_t bwd_workspace_bf16(int64_t n, int hq, int /*d*/) {
  const int64_t npad = (n + kBlockM - 1) / kBlockM * kBlockM;
  return static_cast<size_t>(2 * hq * npad * 4);
}

}  // namespace treeattn

using namespace treeattn;

extern "C" tree_status_t tree_plan_to_device(tree_plan_t* p, tree_stream_t stream) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->dev.block && p->dev.device == cur) return TREE_OK;
  free_device(p);
  if (p->N == 0) return TREE_OK;
  DevicePlan d;
  const FieldSlot slots[] = {
      {TREE_FIELD_KEY_END, &d.key_end},     {TREE_FIELD_QT_PTR, &d.qt_ptr},
      {TREE_FIELD_QT_KT, &d.qt_kt},         {TREE_FIELD_QT_KIND, &d.qt_kind},
      {TREE_FIELD_FWD_ORDER, &d.fwd_order}, {TREE_FIELD_QP_PTR, &d.qp_ptr},
      {TREE_FIELD_QP_KT, &d.qp_kt},         {TREE_FIELD_QP_KIND, &d.qp_kind},
      {TREE_FIELD_QP_ORDER, &d.qp_order},   {TREE_FIELD_KT_QLO, &d.kt_qlo},
      {TREE_FIELD_KT_QHI, &d.kt_qhi},       {TREE_FIELD_BWD_ORDER, &d.bwd_order},
      {TREE_FIELD_POS_ID, &d.pos_id},       {TREE_FIELD_GQ_PTR, &d.gq_ptr},
      {TREE_FIELD_GP_PTR, &d.gp_ptr},       {TREE_FIELD_GT_KIND, &d.gt_kind},
      {TREE_FIELD_GT_ATOM, &d.gt_atom},     {TREE_FIELD_GT_BIDX, &d.gt_bidx},
      {TREE_FIELD_GT_BOUNDS, &d.gt_bounds}, {TREE_FIELD_GW_KEND, &d.gw_kend},
      {TREE_FIELD_GW_KT, &d.gw_kt},         {TREE_FIELD_TOKEN_SEG, &d.token_seg},
      {TREE_FIELD_SUBTREE_END, &d.subtree_end}, {TREE_FIELD_CU_SEQLENS, &d.cu_seqlens},
  };
  // key_end is padded with zeros to whole 128-key tiles: the kernels copy it
  // a tile at a time, and a zero bound hides the keys past N from every row.
  auto slot_elems = [&](size_t s) {
    const size_t n = p->field[slots[s].f].size();
    if (slots[s].f != TREE_FIELD_KEY_END) return n;
    const size_t padded = static_cast<size_t>(p->Tk) * kBlockM;
    return n > padded ? n : padded;
  };
  size_t offs[sizeof(slots) / sizeof(slots[0])];
  size_t total = 0;
  for (size_t s = 0; s < sizeof(slots) / sizeof(slots[0]); ++s) {
    offs[s] = total;
    total += (slot_elems(s) * 4 + 255) / 256 * 256;
  }
  // the GDN segment table, built from the DFS layout
  std::vector<int32_t> seg_table(static_cast<size_t>(p->S) * 4);
  {
    const auto& order = p->field[TREE_FIELD_DFS_ORDER];
    const auto& start = p->field[TREE_FIELD_SEG_START];
    const auto& tseg = p->field[TREE_FIELD_TOKEN_SEG];
    const auto& ap = p->field[TREE_FIELD_ANC_PTR];
    const auto& ai = p->field[TREE_FIELD_ANC_IDX];
    std::vector<int32_t> len(static_cast<size_t>(p->S), 0);
    for (int32_t t = 0; t < p->N; ++t) ++len[tseg[t]];
    for (int32_t d = 0; d < p->S; ++d) {
      const int32_t s = order[d];
      seg_table[4 * d + 0] = s;
      seg_table[4 * d + 1] = start[s];
      seg_table[4 * d + 2] = len[s];
      seg_table[4 * d + 3] = ap[s + 1] > ap[s] ? ai[ap[s + 1] - 1] : -1;
    }
  }
  const size_t off_segs = total;
  total += (seg_table.size() * 4 + 255) / 256 * 256;
  const size_t off_units = total;
  total += (p->gdn_units.size() * 4 + 255) / 256 * 256;
  std::vector<uint8_t> host(total, 0);
  for (size_t s = 0; s < sizeof(slots) / sizeof(slots[0]); ++s) {
    const auto& v = p->field[slots[s].f];
    if (!v.empty()) std::memcpy(host.data() + offs[s], v.data(), v.size() * 4);
  }
  std::memcpy(host.data() + off_segs, seg_table.data(), seg_table.size() * 4);
  if (!p->gdn_units.empty())
    std::memcpy(host.data() + off_units, p->gdn_units.data(), p->gdn_units.size() * 4);
  void* block = nullptr;
  e = cudaMalloc(&block, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TREE_ERR_OOM, std::string("cudaMalloc of the plan: ") + cudaGetErrorString(e));
  }
  e = cudaMemcpyAsync(block, host.data(), total, cudaMemcpyHostToDevice,
                      static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaFree(block);
    return cuda_fail(e, "plan upload");
  }
  for (size_t s = 0; s < sizeof(slots) / sizeof(slots[0]); ++s)
    *slots[s].dst = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(block) + offs[s]);
  d.seg_table = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(block) + off_segs);
  d.gdn_units = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(block) + off_units);
  d.block = block;
  d.bytes = total;
  d.device = cur;
  p->dev = d;
  return TREE_OK;
}

extern "C" void tree_plan_destroy(tree_plan_t* p) {
  if (!p) return;
  free_device(p);
  conv_tables_free(p);
  delete p;
}

namespace {

tree_status_t fwd_entry(const tree_plan_t* p, const void* q, const void* k, const void* v,
                        const void* past_k, const void* past_v, void* o, float* lse, int32_t hq,
                        int32_t hkv, int32_t head_dim, tree_dtype_t dtype, float softmax_scale,
                        tree_stream_t stream, bool gateway_call) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  tree_status_t st = check_heads(hq, hkv, head_dim, dtype);
  if (st != TREE_OK) return st;
  if (!std::isfinite(softmax_scale) || softmax_scale < 0.f)
    return fail(TREE_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (p->past_len > 0 && !gateway_call)
    return fail(TREE_ERR_INVALID_ARG, "the plan has a gateway: use tree_attn_fwd_gateway");
  if (gateway_call && dtype != TREE_DTYPE_BF16)
    return fail(TREE_ERR_UNSUPPORTED, "gateway attention is bf16 only");
  if (p->N == 0) return TREE_OK;
  if (!q || !k || !v || !o || !lse) return fail(TREE_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(TREE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (p->past_len > 0) {
    if (!past_k || !past_v) return fail(TREE_ERR_INVALID_ARG, "NULL gateway key or value pointer");
    if (!aligned16(past_k) || !aligned16(past_v))
      return fail(TREE_ERR_INVALID_ARG, "gateway pointers must be 16-byte aligned");
  }
  if ((st = check_plan_on_device(p)) != TREE_OK) return st;
  int* status = status_ptr();
  if (!status) return fail(TREE_ERR_CUDA, "status word unavailable");
  AttnArgs a{p, q, k, v, o, lse, hq, hkv, head_dim, resolve_scale(softmax_scale, head_dim),
             static_cast<cudaStream_t>(stream), status};
  a.past_k = past_k;
  a.past_v = past_v;
  cudaError_t e = dtype == TREE_DTYPE_F32 ? launch_fwd_f32(a) : launch_fwd_bf16(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_attn_fwd launch");
  return TREE_OK;
}

}  // namespace

extern "C" tree_status_t tree_attn_fwd(const tree_plan_t* p, const void* q, const void* k,
                                       const void* v, void* o, float* lse, int32_t hq,
                                       int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                                       float softmax_scale, tree_stream_t stream) {
  return fwd_entry(p, q, k, v, nullptr, nullptr, o, lse, hq, hkv, head_dim, dtype, softmax_scale,
                   stream, false);
}

extern "C" tree_status_t tree_attn_fwd_gateway(const tree_plan_t* p, const void* q, const void* k,
                                               const void* v, const void* past_k,
                                               const void* past_v, void* o, float* lse, int32_t hq,
                                               int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                                               float softmax_scale, tree_stream_t stream) {
  return fwd_entry(p, q, k, v, past_k, past_v, o, lse, hq, hkv, head_dim, dtype, softmax_scale,
                   stream, true);
}

extern "C" tree_status_t tree_weighted_ce(const tree_plan_t* p, const void* logits, void* dlogits,
                                          const int32_t* tokens, const float* lambda, int32_t vocab,
                                          tree_dtype_t dtype, float grad_scale, float* row_loss,
                                          double* loss, tree_stream_t stream) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32) return fail(TREE_ERR_INVALID_ARG, "unknown dtype");
  if (vocab <= 0 || vocab % 8 != 0) return fail(TREE_ERR_INVALID_ARG, "vocab must be a positive multiple of 8");
  if (!std::isfinite(grad_scale)) return fail(TREE_ERR_INVALID_ARG, "grad_scale must be finite");
  if (p->N == 0) {
    if (loss && cudaMemsetAsync(loss, 0, sizeof(double), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return fail(TREE_ERR_CUDA, "loss clear");
    return TREE_OK;
  }
  if (!logits || !dlogits || !tokens || !lambda || !row_loss) return fail(TREE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(logits) || !aligned16(dlogits))
    return fail(TREE_ERR_INVALID_ARG, "logits and dlogits must be 16-byte aligned");
  const size_t row_bytes = static_cast<size_t>(vocab) * (dtype == TREE_DTYPE_F32 ? 4 : 2);
  const size_t bytes = row_bytes * static_cast<size_t>(p->N);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(logits), b0 = reinterpret_cast<uintptr_t>(dlogits);
  if (a0 != b0 && a0 < b0 + bytes && b0 < a0 + bytes)
    return fail(TREE_ERR_INVALID_ARG, "dlogits must be logits itself or not overlap it");
  // the distinct targets of one row are the first tokens of one segment's
  // children: bound the fan-out on the host
  {
    const auto& ap = p->field[TREE_FIELD_ANC_PTR];
    const auto& ai = p->field[TREE_FIELD_ANC_IDX];
    std::vector<int32_t> fan(static_cast<size_t>(p->S), 0);
    for (int32_t s = 0; s < p->S; ++s)
      if (ap[s + 1] > ap[s]) ++fan[ai[ap[s + 1] - 1]];
    for (int32_t s = 0; s < p->S; ++s)
      if (fan[s] > kCeMaxTargets)
        return fail(TREE_ERR_UNSUPPORTED, "a segment has more than " + std::to_string(kCeMaxTargets) +
                                              " children");
  }
  tree_status_t st = check_plan_on_device(p);
  if (st != TREE_OK) return st;
  int* status = status_ptr();
  if (!status) return fail(TREE_ERR_CUDA, "status word unavailable");
  CeArgs a;
  a.logits = logits;
  a.dlogits = dlogits;
  a.tokens = tokens;
  a.lam = lambda;
  a.token_seg = p->dev.token_seg;
  a.subtree_end = p->dev.subtree_end;
  a.row_loss = row_loss;
  a.loss = loss;
  a.status = status;
  a.N = p->N;
  a.V = vocab;
  a.f32 = dtype == TREE_DTYPE_F32 ? 1 : 0;
  a.grad_scale = grad_scale;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_weighted_ce(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_weighted_ce launch");
  return TREE_OK;
}

extern "C" tree_status_t tree_gdn_fwd(const tree_plan_t* p, const void* q, const void* k, const void* v,
                                      const float* g, const float* beta, const float* initial_state,
                                      void* o, float* segment_states, int32_t hk, int32_t hv,
                                      int32_t head_dim, tree_dtype_t dtype, tree_stream_t stream) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32) return fail(TREE_ERR_INVALID_ARG, "unknown dtype");
  if (hk <= 0 || hv <= 0 || hv % hk != 0) return fail(TREE_ERR_INVALID_ARG, "need hk > 0, hv > 0 and hv % hk == 0");
  if (hv > 65535) return fail(TREE_ERR_UNSUPPORTED, "hv > 65535");
  if (head_dim != 128) return fail(TREE_ERR_UNSUPPORTED, "GDN head_dim must be 128");
  if (p->N == 0) return TREE_OK;
  if (!q || !k || !v || !g || !beta || !o || !segment_states) return fail(TREE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(segment_states) ||
      (initial_state && !aligned16(initial_state)))
    return fail(TREE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  tree_status_t st = check_plan_on_device(p);
  if (st != TREE_OK) return st;
  GdnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.s0 = initial_state;
  a.o = o;
  a.states = segment_states;
  a.segs = reinterpret_cast<const int4*>(p->dev.seg_table);
  a.units = reinterpret_cast<const int4*>(p->dev.gdn_units);
  a.level_ptr = p->gdn_level_ptr.data();
  a.levels = static_cast<int>(p->gdn_level_ptr.size()) - 1;
  a.hk = hk;
  a.hv = hv;
  a.group = hv / hk;
  a.f32 = dtype == TREE_DTYPE_F32 ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_gdn_fwd(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_gdn_fwd launch");
  return TREE_OK;
}

namespace {

// pair: q and k in one call (x2 = k), checked like x
tree_status_t rope_entry(const tree_plan_t* p, void* x, int32_t heads, void* x2, int32_t heads2, bool pair,
                         int32_t head_dim, tree_dtype_t dtype, float base, int32_t rotate_half,
                         int32_t inverse, tree_stream_t stream) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (heads <= 0 || (pair && heads2 <= 0)) return fail(TREE_ERR_INVALID_ARG, "heads must be positive");
  if (!rope_shape_ok(head_dim))
    return fail(TREE_ERR_UNSUPPORTED, "head_dim must be even and at most 128");
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32)
    return fail(TREE_ERR_INVALID_ARG, "dtype must be TREE_DTYPE_BF16 or TREE_DTYPE_F32");
  if (!std::isfinite(base) || base <= 0.f) return fail(TREE_ERR_INVALID_ARG, "base must be finite and > 0");
  if ((rotate_half != 0 && rotate_half != 1) || (inverse != 0 && inverse != 1))
    return fail(TREE_ERR_INVALID_ARG, "rotate_half and inverse must be 0 or 1");
  if (p->N == 0) return TREE_OK;
  if (!x || (pair && !x2)) return fail(TREE_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(x) || (x2 && !aligned16(x2)))
    return fail(TREE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const size_t elem = dtype == TREE_DTYPE_F32 ? 4 : 2;
  if (static_cast<int64_t>(p->N) * heads * head_dim > (int64_t{1} << 40) ||
      (x2 && static_cast<int64_t>(p->N) * heads2 * head_dim > (int64_t{1} << 40)))
    return fail(TREE_ERR_OVERFLOW, "tensor too large");
  if (x2) {  // the two tensors must not share an element
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(x), a1 = a0 + static_cast<size_t>(p->N) * heads * head_dim * elem;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(x2), b1 = b0 + static_cast<size_t>(p->N) * heads2 * head_dim * elem;
    if (a0 < b1 && b0 < a1) return fail(TREE_ERR_INVALID_ARG, "the two tensors overlap");
  }
  tree_status_t st = check_plan_on_device(p);
  if (st != TREE_OK) return st;
  RopeArgs a{p->dev.pos_id, x, x2, p->N, heads, x2 ? heads2 : 0, head_dim, rotate_half, inverse,
             dtype == TREE_DTYPE_F32 ? 1 : 0, base, static_cast<cudaStream_t>(stream)};
  cudaError_t e = launch_rope(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_rope launch");
  return TREE_OK;
}

}  // namespace

extern "C" tree_status_t tree_rope(const tree_plan_t* p, void* x, int32_t heads, int32_t head_dim,
                                   tree_dtype_t dtype, float base, int32_t rotate_half,
                                   int32_t inverse, tree_stream_t stream) {
  return rope_entry(p, x, heads, nullptr, 0, false, head_dim, dtype, base, rotate_half, inverse, stream);
}

extern "C" tree_status_t tree_rope_qk(const tree_plan_t* p, void* q, int32_t q_heads, void* k,
                                      int32_t k_heads, int32_t head_dim, tree_dtype_t dtype,
                                      float base, int32_t rotate_half, int32_t inverse,
                                      tree_stream_t stream) {
  return rope_entry(p, q, q_heads, k, k_heads, true, head_dim, dtype, base, rotate_half, inverse, stream);
}

namespace {

tree_status_t conv_check(const tree_plan_t* p, int32_t channels, tree_dtype_t dtype, int32_t activation) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (channels <= 0 || channels % 8 != 0)
    return fail(TREE_ERR_UNSUPPORTED, "channels must be a positive multiple of 8");
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32)
    return fail(TREE_ERR_INVALID_ARG, "dtype must be TREE_DTYPE_BF16 or TREE_DTYPE_F32");
  if (activation != TREE_ACT_NONE && activation != TREE_ACT_SILU)
    return fail(TREE_ERR_INVALID_ARG, "activation must be TREE_ACT_NONE or TREE_ACT_SILU");
  if (p->N == 0) return TREE_OK;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return fail(TREE_ERR_CUDA, "no CUDA device");
  if (!p->conv.block || p->conv.device != cur)
    return fail(TREE_ERR_NOT_ON_DEVICE, "call tree_conv_prepare on the current device first");
  return TREE_OK;
}

ConvArgs conv_args(const tree_plan_t* p, const void* x, const float* weight, const float* bias,
                   int32_t channels, tree_dtype_t dtype, int32_t activation, tree_stream_t stream) {
  ConvArgs a{};
  a.pred = p->conv.pred;
  a.succ_ptr = p->conv.succ_ptr;
  a.succ = p->conv.succ;
  a.irr_bits = p->conv.irr_bits;
  a.irr_list = p->conv.irr_list;
  a.num_irr = p->conv.num_irr;
  a.x = x;
  a.weight = weight;
  a.bias = bias;
  a.N = p->N;
  a.C = channels;
  a.K = p->conv.K;
  a.act = activation;
  a.f32 = dtype == TREE_DTYPE_F32 ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status_ptr();
  return a;
}

}  // namespace

extern "C" tree_status_t tree_conv_prepare(tree_plan_t* p, int32_t kernel_size, tree_stream_t stream) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (kernel_size < 1 || kernel_size > kConvMaxK)
    return fail(TREE_ERR_UNSUPPORTED, "kernel_size must be 1 to " + std::to_string(kConvMaxK));
  if (p->N >= (1 << 28)) return fail(TREE_ERR_OVERFLOW, "too many tokens for the conv tables");
  if (p->N == 0) {  // no tables; the kernel size still sizes the weight gradient
    p->conv.K = kernel_size;
    return TREE_OK;
  }
  return conv_tables_build(p, kernel_size, static_cast<cudaStream_t>(stream));
}

extern "C" tree_status_t tree_conv_fwd(const tree_plan_t* p, const void* x, const float* weight,
                                       const float* bias, void* y, int32_t channels,
                                       tree_dtype_t dtype, int32_t activation, tree_stream_t stream) {
  tree_status_t st = conv_check(p, channels, dtype, activation);
  if (st != TREE_OK || p->N == 0) return st;
  if (!x || !weight || !y) return fail(TREE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(y)) return fail(TREE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  ConvArgs a = conv_args(p, x, weight, bias, channels, dtype, activation, stream);
  a.y = y;
  cudaError_t e = launch_conv_fwd(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_conv_fwd launch");
  return TREE_OK;
}

extern "C" size_t tree_conv_bwd_workspace_bytes(const tree_plan_t* p, int32_t channels) {
  if (!p || channels <= 0 || p->conv.K == 0) return 0;
  return conv_bwd_workspace(p->N, channels, p->conv.K);
}

extern "C" tree_status_t tree_conv_bwd(const tree_plan_t* p, const void* x, const float* weight,
                                       const float* bias, const void* dy, void* dx, float* dweight,
                                       float* dbias, int32_t channels, tree_dtype_t dtype,
                                       int32_t activation, void* workspace, size_t workspace_bytes,
                                       tree_stream_t stream) {
  tree_status_t st = conv_check(p, channels, dtype, activation);
  if (st != TREE_OK) return st;
  if (p->N == 0) {  // no tokens: dweight and dbias (overwritten, not accumulated) are zero
    if (p->conv.K == 0) return fail(TREE_ERR_NOT_ON_DEVICE, "call tree_conv_prepare first");
    if (!dweight) return fail(TREE_ERR_INVALID_ARG, "NULL pointer");
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(dweight, 0, static_cast<size_t>(channels) * p->conv.K * sizeof(float), s);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, static_cast<size_t>(channels) * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "tree_conv_bwd zero gradients");
    return TREE_OK;
  }
  if (!x || !weight || !dy || !dx || !dweight || !workspace) return fail(TREE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(workspace))
    return fail(TREE_ERR_INVALID_ARG, "x, dy, dx and workspace must be 16-byte aligned");
  if (workspace_bytes < conv_bwd_workspace(p->N, channels, p->conv.K))
    return fail(TREE_ERR_INVALID_ARG, "workspace too small");
  ConvArgs a = conv_args(p, x, weight, bias, channels, dtype, activation, stream);
  a.dy = dy;
  a.dx = dx;
  a.dweight = dweight;
  a.dbias = dbias;
  a.partial = static_cast<float*>(workspace);
  cudaError_t e = launch_conv_bwd(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_conv_bwd launch");
  return TREE_OK;
}

extern "C" size_t tree_attn_bwd_workspace_bytes(const tree_plan_t* p, int32_t hq, int32_t head_dim,
                                                tree_dtype_t dtype) {
  if (!p || hq <= 0 || head_dim <= 0) return 0;
  return dtype == TREE_DTYPE_F32 ? bwd_workspace_f32(p->N, hq)
                                 : bwd_workspace_bf16(p->N, hq, head_dim);
}

namespace {

// Shared by the whole backward and its two phases. phases: bit 0 the dQ phase
// (Delta, lse*log2e into the workspace, dQ), bit 1 the dK/dV phase.
tree_status_t bwd_entry(const tree_plan_t* p, const void* dout, const void* q, const void* k,
                        const void* v, const void* o, const float* lse, void* dq, void* dk,
                        void* dv, int32_t hq, int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                        tree_dtype_t grad_dtype, float softmax_scale, void* workspace,
                        size_t workspace_bytes, tree_stream_t stream, int phases,
                        const void* past_k = nullptr, const void* past_v = nullptr,
                        float* past_dk = nullptr, float* past_dv = nullptr,
                        bool gateway_call = false) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  tree_status_t st = check_heads(hq, hkv, head_dim, dtype);
  if (st != TREE_OK) return st;
  if (p->past_len > 0 && !gateway_call)
    return fail(TREE_ERR_INVALID_ARG, "the plan has a gateway: use tree_attn_bwd_gateway");
  if (gateway_call && dtype != TREE_DTYPE_BF16)
    return fail(TREE_ERR_UNSUPPORTED, "gateway attention is bf16 only");
  if (grad_dtype != TREE_DTYPE_F32 && grad_dtype != TREE_DTYPE_BF16)
    return fail(TREE_ERR_INVALID_ARG, "unknown grad_dtype");
  if (dtype == TREE_DTYPE_F32 && grad_dtype != TREE_DTYPE_F32)
    return fail(TREE_ERR_INVALID_ARG, "fp32 inputs need fp32 gradients");
  if (!std::isfinite(softmax_scale) || softmax_scale < 0.f)
    return fail(TREE_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (p->N == 0) return TREE_OK;
  const void* common[] = {dout, q, k, v, lse, workspace};
  const void* phase_dq[] = {o, dq};
  const void* phase_kv[] = {dk, dv};
  auto check = [](const void* const* xs, size_t n) -> tree_status_t {
    for (size_t i = 0; i < n; ++i) {
      if (!xs[i]) return fail(TREE_ERR_INVALID_ARG, "NULL tensor or workspace pointer");
      if (!aligned16(xs[i])) return fail(TREE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    }
    return TREE_OK;
  };
  if ((st = check(common, 6)) != TREE_OK) return st;
  if ((phases & 1) && (st = check(phase_dq, 2)) != TREE_OK) return st;
  if ((phases & 2) && (st = check(phase_kv, 2)) != TREE_OK) return st;
  if (p->past_len > 0) {
    const void* gws[] = {past_k, past_v, past_dk, past_dv};
    if ((st = check(gws, 4)) != TREE_OK) return st;
  }
  const size_t need = tree_attn_bwd_workspace_bytes(p, hq, head_dim, dtype);
  if (workspace_bytes < need)
    return fail(TREE_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(need) + " bytes");
  if ((st = check_plan_on_device(p)) != TREE_OK) return st;
  int* status = status_ptr();
  if (!status) return fail(TREE_ERR_CUDA, "status word unavailable");
  AttnBwdArgs a{p,  dout, q,   k,   v,        o,        lse,
                dq, dk,   dv,  hq,  hkv,      head_dim, grad_dtype == TREE_DTYPE_F32,
                resolve_scale(softmax_scale, head_dim), workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), status, phases};
  a.past_k = past_k;
  a.past_v = past_v;
  a.past_dk = past_dk;
  a.past_dv = past_dv;
  cudaError_t e = dtype == TREE_DTYPE_F32 ? launch_bwd_f32(a) : launch_bwd_bf16(a);
  if (e != cudaSuccess) return cuda_fail(e, "tree_attn_bwd launch");
  return TREE_OK;
}

}  // namespace

extern "C" tree_status_t tree_attn_bwd_gateway(const tree_plan_t* p, const void* dout,
                                               const void* q, const void* k, const void* v,
                                               const void* past_k, const void* past_v,
                                               const void* o, const float* lse, void* dq, void* dk,
                                               void* dv, float* past_dk_acc, float* past_dv_acc,
                                               int32_t hq, int32_t hkv, int32_t head_dim,
                                               tree_dtype_t dtype, tree_dtype_t grad_dtype,
                                               float softmax_scale, void* workspace,
                                               size_t workspace_bytes, tree_stream_t stream) {
  return bwd_entry(p, dout, q, k, v, o, lse, dq, dk, dv, hq, hkv, head_dim, dtype, grad_dtype,
                   softmax_scale, workspace, workspace_bytes, stream, 3, past_k, past_v,
                   past_dk_acc, past_dv_acc, true);
}

extern "C" tree_status_t tree_attn_bwd(const tree_plan_t* p, const void* dout, const void* q,
                                       const void* k, const void* v, const void* o,
                                       const float* lse, void* dq, void* dk, void* dv, int32_t hq,
                                       int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                                       tree_dtype_t grad_dtype, float softmax_scale,
                                       void* workspace, size_t workspace_bytes,
                                       tree_stream_t stream) {
  return bwd_entry(p, dout, q, k, v, o, lse, dq, dk, dv, hq, hkv, head_dim, dtype, grad_dtype,
                   softmax_scale, workspace, workspace_bytes, stream, 3);
}

extern "C" tree_status_t tree_attn_bwd_dq(const tree_plan_t* p, const void* dout, const void* q,
                                          const void* k, const void* v, const void* o,
                                          const float* lse, void* dq, int32_t hq, int32_t hkv,
                                          int32_t head_dim, tree_dtype_t dtype,
                                          tree_dtype_t grad_dtype, float softmax_scale,
                                          void* workspace, size_t workspace_bytes,
                                          tree_stream_t stream) {
  return bwd_entry(p, dout, q, k, v, o, lse, dq, nullptr, nullptr, hq, hkv, head_dim, dtype,
                   grad_dtype, softmax_scale, workspace, workspace_bytes, stream, 1);
}

extern "C" tree_status_t tree_attn_bwd_dkdv(const tree_plan_t* p, const void* dout, const void* q,
                                            const void* k, const void* v, const float* lse,
                                            void* dk, void* dv, int32_t hq, int32_t hkv,
                                            int32_t head_dim, tree_dtype_t dtype,
                                            tree_dtype_t grad_dtype, float softmax_scale,
                                            void* workspace, size_t workspace_bytes,
                                            tree_stream_t stream) {
  return bwd_entry(p, dout, q, k, v, nullptr, lse, nullptr, dk, dv, hq, hkv, head_dim, dtype,
                   grad_dtype, softmax_scale, workspace, workspace_bytes, stream, 2);
}

namespace treeattn {
namespace {

// One thread waits on an mbarrier that nothing completes, through the same
// bounded wait as every kernel of the library, so that the wait gives up after
// limit_ns, stores kSiteDiag in the status word and the kernel returns.
__global__ void diag_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_s;
  dev::mbar_init(&bar, 1);
  abort_s = 0;
  dev::fence_mbar_init();
  dev::mbar_wait(&bar, 0, &abort_s, status, dev::kSiteDiag, limit_ns);
}

}  // namespace
}  // namespace treeattn

extern "C" tree_status_t tree_diag_wait_timeout(int64_t limit_ns, tree_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000ll)
    return fail(TREE_ERR_INVALID_ARG, "limit_ns outside [1e3, 1e10]");
  int* st = status_ptr();
  if (!st) return fail(TREE_ERR_CUDA, "status word address");
  diag_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(st, static_cast<uint64_t>(limit_ns));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "diagnostic wait launch");
  set_error("");
  return TREE_OK;
}

extern "C" tree_status_t tree_status_sync(tree_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
    if (word == 9)
      return fail(TREE_ERR_CUDA, "a kernel's shared memory block was not 1024-byte aligned");
    if (word == 8)
      return fail(TREE_ERR_INVALID_ARG, "a token id was >= vocab (its prediction was skipped)");
    if (word == 7)
      return fail(TREE_ERR_UNSUPPORTED, "a logits row had more distinct targets than it can hold");
    return fail(TREE_ERR_TIMEOUT, "a kernel gave up a bounded wait (wait site " +
                                      std::to_string(word) + ")");
  }
  return TREE_OK;
}
