// Internal launcher declarations shared by the C-ABI glue and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include "plan_internal.h"

namespace treeattn {

struct SchedSlot;
// A fresh run-time scheduler counter for one kernel launch (nullptr on error).
SchedSlot* next_sched_slot();

// Rotary position embedding at tree position ids, in place (rope.cu).
struct RopeArgs {
  const int32_t* pos;  // device [N]
  void* x;             // device [N, heads, head_dim]
  void* x2;            // device [N, heads2, head_dim] or nullptr: rotated in the same pass
  int N, heads, heads2, head_dim, rotate_half, inverse, f32;
  float base;
  cudaStream_t stream;
};
bool rope_shape_ok(int head_dim);
cudaError_t launch_rope(const RopeArgs& a);

// Tree-correct causal depthwise conv (conv.cu).
constexpr int kConvMaxK = 8;
struct ConvArgs {
  const int32_t* pred;
  const int32_t* succ_ptr;
  const int32_t* succ;
  const uint32_t* irr_bits;
  const int32_t* irr_list;
  int num_irr;
  const void* x;         // [N, C]
  const float* weight;   // [C, K]
  const float* bias;     // [C] or nullptr
  void* y;               // forward output [N, C]
  const void* dy;        // backward input [N, C]
  void* dx;              // backward output [N, C]
  float* dweight;        // [C, K]
  float* dbias;          // [C] or nullptr
  float* partial;        // workspace: per token range, the sums of dweight and dbias
  int* status;           // device status word (a bounded wait that gives up)
  int N, C, K, act, f32;
  cudaStream_t stream;
};
tree_status_t conv_tables_build(tree_plan* p, int K, cudaStream_t stream);
void conv_tables_free(tree_plan* p);
size_t conv_bwd_workspace(int N, int C, int K);
cudaError_t launch_conv_fwd(const ConvArgs& a);
cudaError_t launch_conv_bwd(ConvArgs a);

// Fused weighted next-token cross-entropy over the trie (loss.cu).
constexpr int kCeMaxTargets = 1024;  // distinct target ids predicted from one row
struct CeArgs {
  const void* logits;  // [N, V]
  void* dlogits;       // [N, V] (may be logits itself)
  const int32_t* tokens;
  const float* lam;
  const int32_t* token_seg;    // plan (device)
  const int32_t* subtree_end;  // plan (device)
  float* row_loss;             // [N]
  double* loss;                // sum of row_loss, or nullptr
  int* status;
  int N, V, f32;
  float grad_scale;
  cudaStream_t stream;
};
cudaError_t launch_weighted_ce(const CeArgs& a);
// Gated DeltaNet forward with tree state routing (gdn.cu).
struct GdnArgs {
  const void* q;       // [N, hk, 128]
  const void* k;       // [N, hk, 128]
  const void* v;       // [N, hv, 128]
  const float* g;      // [N, hv] log decay
  const float* beta;   // [N, hv]
  const float* s0;     // [hv, 128, 128] or nullptr (zeros)
  void* o;             // [N, hv, 128]
  float* states;       // [S, hv, 128, 128]: each segment's end state
  const int4* segs;    // per DFS position: (segment id, first token, length, parent id)
  const int4* units;   // (first DFS position, end position, first token, end token), by level
  const int32_t* level_ptr;  // host: units of level l are level_ptr[l] .. level_ptr[l+1]
  int levels, hk, hv, group, f32;
  cudaStream_t stream;
};
cudaError_t launch_gdn_fwd(const GdnArgs& a);
struct AttnArgs {
  const tree_plan* plan;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int hq, hkv, d;
  float scale;  // softmax scale (already resolved; never 0)
  cudaStream_t stream;
  int* status;  // device status word
  const void* past_k = nullptr;  // gateway keys and values of a partition plan
  const void* past_v = nullptr;
};

struct AttnBwdArgs {
  const tree_plan* plan;
  const void* dout;
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int hq, hkv, d;
  bool grad_f32;  // gradients written as fp32 (else bf16)
  float scale;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  int* status;
  int phases;  // bit 0: Delta + dQ phase; bit 1: dK/dV phase (reads what phase 0 wrote)
  const void* past_k = nullptr;  // gateway keys and values of a partition plan
  const void* past_v = nullptr;
  float* past_dk = nullptr;      // their gradients, accumulated in fp32
  float* past_dv = nullptr;
};

// Workspace layouts.
size_t bwd_workspace_f32(int64_t n, int hq);
size_t bwd_workspace_bf16(int64_t n, int hq, int d);

// fp32 CUDA-core path (any D in {64, 128}).
cudaError_t launch_fwd_f32(const AttnArgs& a);
cudaError_t launch_bwd_f32(const AttnBwdArgs& a);

// bf16 tcgen05 path (D = 128).
cudaError_t launch_fwd_bf16(const AttnArgs& a);
cudaError_t launch_bwd_bf16(const AttnBwdArgs& a);

}  // namespace treeattn
