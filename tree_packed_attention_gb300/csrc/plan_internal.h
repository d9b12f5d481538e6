// Internal definition of the plan object shared by the host plan builder and
// the kernel launchers. Not part of the public C-ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include "treeattn.h"

namespace treeattn {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per tile

enum TileKind : int32_t { kEmpty = 0, kPartial = 1, kFull = 2 };

// Device copy of the fields the kernels read (one allocation, int32 arrays).
struct DevicePlan {
  int device = -1;
  void* block = nullptr;
  size_t bytes = 0;
  const int32_t* key_end = nullptr;    // [N]
  const int32_t* qt_ptr = nullptr;     // [Tq+1]
  const int32_t* qt_kt = nullptr;      // [nnz]
  const int32_t* qt_kind = nullptr;    // [nnz]
  const int32_t* fwd_order = nullptr;  // [Tq]
  const int32_t* qp_ptr = nullptr;     // [P+1]
  const int32_t* qp_kt = nullptr;      // [nnz_pairs]
  const int32_t* qp_kind = nullptr;    // [nnz_pairs]
  const int32_t* qp_order = nullptr;   // [P]
  const int32_t* kt_qlo = nullptr;     // [Tk]
  const int32_t* kt_qhi = nullptr;     // [Tk]
  const int32_t* bwd_order = nullptr;  // [Tk]
  const int32_t* pos_id = nullptr;     // [N]
  const int32_t* gq_ptr = nullptr;     // [Tq+1]
  const int32_t* gp_ptr = nullptr;     // [P+1]
  const int32_t* gt_kind = nullptr;    // [gathered tiles]
  const int32_t* gt_atom = nullptr;    // [gathered tiles * 16]
  const int32_t* gt_bidx = nullptr;    // [gathered tiles]
  const int32_t* gt_bounds = nullptr;  // [bounds rows * 128]
  const int32_t* gw_kend = nullptr;    // [128 * gateway key tiles]
  const int32_t* gw_kt = nullptr;      // [gateway key tiles with a visible key]
  const int32_t* token_seg = nullptr;  // [N]
  const int32_t* subtree_end = nullptr;  // [S]
  const int32_t* cu_seqlens = nullptr;   // [R+1]
  // GDN state routing: per DFS position (segment, first token, length,
  // parent or -1) as int4, and the units of the level-by-level launch (see
  // tree_plan::gdn_units) as int4
  const int32_t* seg_table = nullptr;
  const int32_t* gdn_units = nullptr;
};

// Tables of the tree-correct causal conv for one kernel size (conv.cu): the
// path predecessors of every token and their inverse lists, on one device.
struct ConvTables {
  int device = -1;
  int K = 0;
  void* block = nullptr;
  const int32_t* pred = nullptr;      // [N, K-1]: k-th path predecessor (k = 1..K-1), -1 before the root
  const int32_t* succ_ptr = nullptr;  // [N+1]
  const int32_t* succ = nullptr;      // (t << 3) | k for every (t, k) with pred_k(t) = u, t increasing
  // Tokens whose readers are not all t = u + k along an unbroken run of the DFS
  // order (the last K-1 tokens before a branch into several children): their
  // dx is gathered over the full lists by a separate pass.
  const uint32_t* irr_bits = nullptr;  // [ceil(N / 32)]
  const int32_t* irr_list = nullptr;   // [num_irr]
  int num_irr = 0;
};

}  // namespace treeattn

struct tree_plan {
  int32_t N = 0, S = 0, R = 0;
  int32_t Tq = 0, Tk = 0, P = 0;
  int64_t visible_pairs = 0;
  int32_t past_len = 0;      // gateway keys of a partition plan
  int64_t past_visible = 0;  // of which visible
  std::vector<std::pair<int32_t, int32_t>> gw_runs;  // visible gateway key runs [a, b)
  std::vector<int32_t> field[TREE_FIELD_COUNT];
  // GDN state routing, one launch per level: a unit is a maximal chain of
  // segments each the only child of the one before (consecutive in DFS
  // order), as (first DFS position, end position, first token, end token);
  // roots' units are level 0 and a unit's level is one more than its
  // parent's. Units are ordered by level, then by tokens (most first);
  // gdn_level_ptr[l] .. gdn_level_ptr[l+1] are level l's.
  std::vector<int32_t> gdn_units;
  std::vector<int32_t> gdn_level_ptr;
  treeattn::DevicePlan dev;
  treeattn::ConvTables conv;
};

namespace treeattn {
// Thread-local error message used by every C-ABI call.
void set_error(const std::string& msg);
tree_status_t fail(tree_status_t st, const std::string& msg);
}  // namespace treeattn
