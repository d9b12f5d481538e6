/*
 * treeattn.h -- C-ABI of libtreeattn: tree-packed attention on one GB300 (sm_103a).
 *
 * The method: "Tree Training: Accelerating Agentic LLMs Training via Shared
 * Prefix Reuse" (arXiv 2511.00413). A trie of token segments is laid out once
 * in depth-first order (§3.1 eq. 8). Token i attends to token j iff j <= i and
 * the segments of i and j lie on one root-to-leaf path (§3.2 "Attention
 * Mask"): its ancestors' segments in full and its own segment causally
 * (App. A.1). The result for every token equals running each root-to-leaf
 * path alone (§3.1 eq. 6). The per-token loss weight is g_t/K (§3.1 eq. 4).
 *
 * Conventions for every call:
 *  - Status: every call returns tree_status_t (TREE_OK = 0) and never aborts;
 *    on failure tree_last_error() holds a message (thread-local). All
 *    argument, shape and alignment checks run on the host before any launch.
 *  - Ownership: the caller owns every tensor and the workspace. The library
 *    owns only the plan (host arrays and the plan's device copy).
 *  - Streams: calls that take a stream enqueue work on it and return
 *    without waiting (stream-ordered). `stream` is a cudaStream_t passed as
 *    void* (NULL = the legacy default stream).
 *  - Concurrency: the attention kernels hand out their work items from a
 *    counter of a library-owned ring of 1024, one per launch in turn, which
 *    the launch's last block puts back to zero. Launches may overlap on
 *    different streams as long as fewer than 1024 are in flight at once. A
 *    launch captured in a CUDA graph keeps the counter it was given, so
 *    replays of one graph must not overlap one another (replays one after
 *    another on a stream are fine).
 *  - Tensor layout: token-major, contiguous, in DFS order. q and o are
 *    [N, hq, D]; k and v are [N, hkv, D]; lse is [hq, N] fp32, natural log.
 *    Segment s occupies tokens [seg_start[s], seg_start[s] + lengths[s]).
 *    Grouped heads: q head h reads kv head h / (hq / hkv).
 *  - Device pointers must be 16-byte aligned.
 *  - Dtypes: TREE_DTYPE_BF16 runs the tcgen05 tensor-core kernels (D = 128);
 *    TREE_DTYPE_F32 runs the fp32 CUDA-core kernels (D = 64 or 128).
 *  - Tile grid: 128 x 128 (query x key) tiles; a tile with no visible pair
 *    is never loaded or multiplied.
 */
#ifndef TREEATTN_H
#define TREEATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TREE_OK = 0,
  TREE_ERR_INVALID_ARG = 1,    /* bad pointer, size, shape, alignment or parent id */
  TREE_ERR_CYCLE = 2,          /* some segment does not reach a root */
  TREE_ERR_EMPTY_SEGMENT = 3,  /* a segment with fewer than one token */
  TREE_ERR_OVERFLOW = 4,       /* a count does not fit int32 */
  TREE_ERR_UNSUPPORTED = 5,    /* valid, but outside what the kernels handle (e.g. D) */
  TREE_ERR_CUDA = 6,           /* a CUDA runtime call failed */
  TREE_ERR_TIMEOUT = 7,        /* a kernel gave up a bounded wait (device status word) */
  TREE_ERR_OOM = 8,            /* host or device allocation failed */
  TREE_ERR_NOT_ON_DEVICE = 9   /* tree_plan_to_device has not been called */
} tree_status_t;

typedef enum { TREE_DTYPE_F32 = 0, TREE_DTYPE_BF16 = 1 } tree_dtype_t;

typedef void* tree_stream_t; /* a cudaStream_t */

typedef struct tree_plan tree_plan_t; /* opaque, library-owned */

typedef struct {
  int64_t num_tokens;     /* N = sum of segment lengths */
  int64_t num_segments;   /* S */
  int64_t num_tries;      /* R = number of roots */
  int64_t block_m;        /* query rows per tile (128) */
  int64_t block_n;        /* keys per tile (128) */
  int64_t num_q_tiles;    /* ceil(N / block_m) */
  int64_t num_k_tiles;    /* ceil(N / block_n) */
  int64_t nnz_tiles;      /* non-empty (q-tile, k-tile) tiles */
  int64_t num_pairs;      /* ceil(num_q_tiles / 2): q-tile pairs (2p, 2p+1) */
  int64_t nnz_pair_tiles; /* entries of the q-tile-pair union lists */
  int64_t num_ancestors;  /* sum over segments of the number of ancestors */
  int64_t visible_pairs;  /* sum over rows of the visible keys, diagonal included */
  int64_t num_gathered_tiles; /* entries of TREE_FIELD_GT_KIND (both unit sizes) */
  int64_t past_len;       /* gateway keys of a partition plan (0 otherwise) */
  int64_t past_visible;   /* of which visible to the partition's rows */
  int64_t gdn_levels;     /* launches of tree_gdn_fwd: 1 + the most segments with several
                             children on one root-to-leaf path (0 for an empty plan) */
} tree_plan_info_t;

/* Plan fields readable with tree_plan_get. All are int32 arrays. */
typedef enum {
  TREE_FIELD_DFS_ORDER = 0,   /* [S]   segments in DFS visit order (eq. 8; children and roots in ascending id) */
  TREE_FIELD_SEG_START = 1,   /* [S]   first DFS token of each segment (by segment id) */
  TREE_FIELD_DEPTH = 2,       /* [S]   number of ancestors (a root has 0) */
  TREE_FIELD_SUBTREE_END = 3, /* [S]   one past the last DFS token of the segment's subtree */
  TREE_FIELD_TRIE_ID = 4,     /* [S]   index of the segment's root among the roots in ascending id */
  TREE_FIELD_G = 5,           /* [S]   g_n: root-to-leaf paths through the segment (§3.1) */
  TREE_FIELD_ANC_PTR = 6,     /* [S+1] CSR offsets into ANC_IDX */
  TREE_FIELD_ANC_IDX = 7,     /* [num_ancestors] ancestors of each segment, root first, itself excluded */
  TREE_FIELD_TOKEN_SEG = 8,   /* [N]   segment of each DFS token */
  TREE_FIELD_POS_ID = 9,      /* [N]   position id of eq. 9 (offset within every path through the token) */
  TREE_FIELD_KEY_END = 10,    /* [N]   rows key_end[j] > i >= j are exactly the rows that see key j */
  TREE_FIELD_CU_SEQLENS = 11, /* [R+1] token range of each trie */
  TREE_FIELD_TRIE_PATHS = 12, /* [R]   K of each trie: its number of root-to-leaf paths */
  TREE_FIELD_QT_PTR = 13,     /* [num_q_tiles+1] CSR offsets of the forward tile lists */
  TREE_FIELD_QT_KT = 14,      /* [nnz_tiles] non-empty k-tiles of each q-tile, ascending */
  TREE_FIELD_QT_KIND = 15,    /* [nnz_tiles] 1 = PARTIAL (needs masking), 2 = FULL */
  TREE_FIELD_KT_QLO = 16,     /* [num_k_tiles] first q-tile that sees the k-tile */
  TREE_FIELD_KT_QHI = 17,     /* [num_k_tiles] one past the last; every q-tile in between sees it */
  TREE_FIELD_FWD_ORDER = 18,  /* [num_q_tiles] forward/dQ work order: q-tiles last to first */
  TREE_FIELD_BWD_ORDER = 19,  /* [num_k_tiles] dK/dV work order: k-tiles first to last */
  TREE_FIELD_QP_PTR = 20,     /* [num_pairs+1] CSR offsets of the q-tile-pair union lists */
  TREE_FIELD_QP_KT = 21,      /* [nnz_pair_tiles] union of the k-tiles of q-tiles 2p and 2p+1, ascending */
  TREE_FIELD_QP_KIND = 22,    /* [nnz_pair_tiles] kind for q-tile 2p | (kind for 2p+1) << 2; 0 = EMPTY */
  TREE_FIELD_QP_ORDER = 23,   /* [num_pairs] forward work order of pairs: last to first */
  /* Gathered key tiles: for a unit of q rows (a q-tile of 128 rows, or a
   * pair of q-tiles, 256 rows) the keys that at least one of its rows sees,
   * the keys that every one of its rows sees first, each part ascending, are
   * packed into tiles of 128 key columns. A run of consecutive keys starts at
   * a column that is a multiple of 8 (an "atom" of 8 columns), so a tile's
   * keys load as 16 atoms of 8 consecutive rows each; columns left over in a
   * run's last atom, and atoms after the unit's last run, are padding. */
  TREE_FIELD_GQ_PTR = 24,     /* [num_q_tiles+1] tiles of each q-tile (units of 128 rows) */
  TREE_FIELD_GP_PTR = 25,     /* [num_pairs+1] tiles of each q-tile pair (units of 256 rows), after
                                 the q-tiles' tiles in the same tile table */
  TREE_FIELD_GT_KIND = 26,    /* [num_gathered_tiles] kind of the first 128 rows | kind of the next
                                 128 rows << 2 (0 EMPTY, 1 PARTIAL, 2 FULL: all 128x128 pairs visible)
                                 | 16 when the tile holds gateway keys (partition plans, below) */
  TREE_FIELD_GT_ATOM = 27,    /* [num_gathered_tiles*16] first key row of each atom; -8 for an atom
                                 with no key (loaded as zeros) */
  TREE_FIELD_GT_BIDX = 28,    /* [num_gathered_tiles] row of the tile in GT_BOUNDS, -1 when no slot of
                                 the tile is PARTIAL */
  TREE_FIELD_GT_BOUNDS = 29,  /* [num_bounds*128] key_end of each column's key, 0 for padding.
                                 Column c holds key GT_ATOM[c/8] + c%8, and row i sees it iff
                                 key <= i < key_end[c]; gateway keys (kind bit 16) precede
                                 every row, so only i < key_end[c] applies to them */
  /* Partition plans only (tree_plan_build_partition), empty otherwise: */
  TREE_FIELD_GW_KEND = 30,    /* [128*ceil(past_len/128)] N for a visible gateway key, 0 for a
                                 hidden one and past past_len */
  TREE_FIELD_GW_KT = 31,      /* [gateway key tiles with a visible key] their indices (128 keys each) */
  TREE_FIELD_COUNT = 32
} tree_plan_field_t;

/*
 * Build a plan from a trie (or a forest: several roots pack several tries in
 * one row). Host only; no GPU needed.
 *   segment_parents[s]: parent segment id of s, or -1 for a root (host, int32[num_segments]).
 *   segment_lengths[s]: tokens of segment s, >= 1 (host, int32[num_segments]).
 * Parents may come after their children in id order. The inputs are copied.
 * Errors: TREE_ERR_INVALID_ARG (parent out of [-1, S) or equal to s; NULL
 * pointer with num_segments > 0; num_segments < 0), TREE_ERR_EMPTY_SEGMENT,
 * TREE_ERR_CYCLE, TREE_ERR_OVERFLOW (more than 2^31-129 tokens, or more than
 * 2^31-1 ancestor entries or tiles), TREE_ERR_OOM. num_segments == 0 gives an empty plan (N = 0).
 * Follows §3.1 (trie, g_n, K), eq. 8 (DFS layout), eq. 9 (positions), and the
 * mask of §3.2 / App. A.1 for the tile map. *out is set only on TREE_OK.
 */
tree_status_t tree_plan_build(const int32_t* segment_parents, const int32_t* segment_lengths,
                              int32_t num_segments, tree_plan_t** out);

/*
 * Plan for one partition of a partitioned trie (§3.3 "Partitioning"; App. B):
 * the partition's own segments as in tree_plan_build, plus a gateway of
 * past_len cached keys (App. B.2: the parent partition's own gateway
 * followed by its DFS tokens up to the end of the cut node). Every row of the
 * partition sees gateway key j iff past_visible[j] != 0 (App. B.3 eq. 16: the
 * parent's gateway and the cut node's ancestors within the parent are
 * visible, the parent's other subtrees are not); the partition's own keys
 * keep the tree mask (eq. 14). past_visible is a host array of past_len bytes
 * (copied). pos_offset (App. B.4 eq. 17) is added to every position id, so
 * that a root of the partition continues the positions of the path above it:
 * pass tree_partition's pos_offset of the partition, and the position ids
 * (TREE_FIELD_POS_ID, tree_rope) equal those of the same tokens in the whole
 * trie. past_len == 0 and pos_offset == 0 give the plan of tree_plan_build.
 * Errors as tree_plan_build, and past_len < 0, pos_offset < 0, or a NULL
 * past_visible with past_len > 0 -> TREE_ERR_INVALID_ARG; pos_offset plus the
 * token count above 2^31-1 -> TREE_ERR_OVERFLOW.
 */
tree_status_t tree_plan_build_partition(const int32_t* segment_parents,
                                        const int32_t* segment_lengths, int32_t num_segments,
                                        const uint8_t* past_visible, int32_t past_len,
                                        int32_t pos_offset, tree_plan_t** out);

/* Sizes of a plan (host). */
tree_status_t tree_plan_info(const tree_plan_t* plan, tree_plan_info_t* out);

/* Copy one int32 field into host memory `dst` of exactly `bytes` bytes
 * (field length x 4; TREE_ERR_INVALID_ARG otherwise). */
tree_status_t tree_plan_get(const tree_plan_t* plan, tree_plan_field_t field, void* dst, size_t bytes);

/* Number of int32 elements of a field. */
tree_status_t tree_plan_field_len(const tree_plan_t* plan, tree_plan_field_t field, int64_t* out);

/* Copy the fields the kernels read to the current CUDA device (allocated by
 * and owned by the plan; stream-ordered copy on `stream`). Calling it again
 * on the same device is a no-op; on another device it replaces the copy. */
tree_status_t tree_plan_to_device(tree_plan_t* plan, tree_stream_t stream);

/* Free the plan and its device copy (waits for the device first). NULL is a no-op. */
void tree_plan_destroy(tree_plan_t* plan);

/*
 * Forward tree attention (§3.2 mask; App. A.1 block skipping).
 *   q [N,hq,D], k,v [N,hkv,D]: device, dtype `dtype`.
 *   o [N,hq,D] (device, dtype `dtype`), lse [hq,N] (device, fp32): written.
 *   softmax_scale: logits are scale * q.k; 0 selects 1/sqrt(D); negative is invalid.
 * o_i = sum_j softmax_j(scale q_i.k_j over the keys visible to i) v_j and
 * lse_i = log sum_j exp(scale q_i.k_j). Requires hq % hkv == 0, D in {64,128}
 * for fp32 and D == 128 for bf16 (else TREE_ERR_UNSUPPORTED).
 */
tree_status_t tree_attn_fwd(const tree_plan_t* plan, const void* q, const void* k, const void* v,
                            void* o, float* lse, int32_t hq, int32_t hkv, int32_t head_dim,
                            tree_dtype_t dtype, float softmax_scale, tree_stream_t stream);

/* Workspace the backward needs, in bytes (device memory the caller provides). */
size_t tree_attn_bwd_workspace_bytes(const tree_plan_t* plan, int32_t hq, int32_t head_dim,
                                     tree_dtype_t dtype);

/*
 * Backward tree attention: the analytic gradients of the forward.
 *   dout, q, o [N,hq,D] and k, v [N,hkv,D]: device, dtype `dtype`;
 *   lse [hq,N] fp32 from tree_attn_fwd (same scale).
 *   dq [N,hq,D], dk, dv [N,hkv,D]: device, dtype `grad_dtype`, written
 *   (grad_dtype must be F32 when dtype is F32).
 *   workspace: device, >= tree_attn_bwd_workspace_bytes(...) bytes; its
 *   contents on entry do not matter.
 * With P = exp(scale S - lse), Delta_i = dO_i.O_i, dS = P (dO V^T - Delta):
 * dq = scale dS K, dk = scale dS^T Q, dv = P^T dO (dk, dv summed over the q
 * heads of a group). Every sum is taken in a fixed order: results repeat bit
 * for bit from run to run.
 * It is tree_attn_bwd_dq followed by tree_attn_bwd_dkdv on the same stream.
 */
tree_status_t tree_attn_bwd(const tree_plan_t* plan, const void* dout, const void* q, const void* k,
                            const void* v, const void* o, const float* lse, void* dq, void* dk,
                            void* dv, int32_t hq, int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                            tree_dtype_t grad_dtype, float softmax_scale, void* workspace,
                            size_t workspace_bytes, tree_stream_t stream);

/*
 * The two phases of tree_attn_bwd, for callers that schedule (or time) them
 * apart. Arguments mean what they mean for tree_attn_bwd.
 * tree_attn_bwd_dq writes Delta_i = dO_i.O_i (and, for bf16, lse_i*log2(e))
 * into the workspace, then dq. tree_attn_bwd_dkdv reads them back and writes
 * dk, dv: it must run after a tree_attn_bwd_dq with the same plan, tensors,
 * heads, dtypes, scale and workspace, ordered after it on the GPU (the same
 * stream, or an event between streams), with the workspace unchanged between.
 */
tree_status_t tree_attn_bwd_dq(const tree_plan_t* plan, const void* dout, const void* q,
                               const void* k, const void* v, const void* o, const float* lse,
                               void* dq, int32_t hq, int32_t hkv, int32_t head_dim,
                               tree_dtype_t dtype, tree_dtype_t grad_dtype, float softmax_scale,
                               void* workspace, size_t workspace_bytes, tree_stream_t stream);
tree_status_t tree_attn_bwd_dkdv(const tree_plan_t* plan, const void* dout, const void* q,
                                 const void* k, const void* v, const float* lse, void* dk, void* dv,
                                 int32_t hq, int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                                 tree_dtype_t grad_dtype, float softmax_scale, void* workspace,
                                 size_t workspace_bytes, tree_stream_t stream);

/*
 * Attention of a partition with its gateway (App. B.2 eq. 14): rows attend
 * to the visible gateway keys past_k / past_v [past_len, hkv, D] (device,
 * same dtype and layout as k and v) and to their own keys under the tree
 * mask, in one softmax. The plan must come from tree_plan_build_partition;
 * other arguments and outputs as tree_attn_fwd. bf16 only (D = 128);
 * fp32 -> TREE_ERR_UNSUPPORTED. A plan with a gateway is refused by
 * tree_attn_fwd / tree_attn_bwd (TREE_ERR_INVALID_ARG).
 */
tree_status_t tree_attn_fwd_gateway(const tree_plan_t* plan, const void* q, const void* k,
                                    const void* v, const void* past_k, const void* past_v, void* o,
                                    float* lse, int32_t hq, int32_t hkv, int32_t head_dim,
                                    tree_dtype_t dtype, float softmax_scale, tree_stream_t stream);

/*
 * Backward of tree_attn_fwd_gateway: dq, dk, dv as tree_attn_bwd (written),
 * and the gateway keys' gradients ADDED in fp32 to past_dk_acc /
 * past_dv_acc [past_len, hkv, D] (device fp32, caller-initialised): several
 * child partitions that share a cut node accumulate into the same gateway
 * gradients without bf16 rounding in between (App. B.5 eq. 18). Hidden
 * gateway keys get + 0. Workspace as tree_attn_bwd (same size). Errors as
 * tree_attn_bwd and tree_attn_fwd_gateway.
 */
tree_status_t tree_attn_bwd_gateway(const tree_plan_t* plan, const void* dout, const void* q,
                                    const void* k, const void* v, const void* past_k,
                                    const void* past_v, const void* o, const float* lse, void* dq,
                                    void* dk, void* dv, float* past_dk_acc, float* past_dv_acc,
                                    int32_t hq, int32_t hkv, int32_t head_dim, tree_dtype_t dtype,
                                    tree_dtype_t grad_dtype, float softmax_scale, void* workspace,
                                    size_t workspace_bytes, tree_stream_t stream);

/*
 * Backward for callers that cannot allocate device memory when they call it
 * (for example a runtime whose memory pool already owns the whole device, or a
 * latency-critical loop where a cudaMalloc would synchronize the device).
 * The paper has no counterpart: this is tree_attn_bwd (same arguments, same
 * results) with its scratch taken from a fixed array of
 * TREE_STATIC_SCRATCH_BYTES compiled into the library instead of from a
 * workspace argument. It calls no cudaMalloc, cudaFree or allocating routine.
 *  - Size limit: requests whose tree_attn_bwd_workspace_bytes exceeds
 *    TREE_STATIC_SCRATCH_BYTES return TREE_ERR_UNSUPPORTED with a message.
 *  - Every GPU that loads the library holds the array until the process exits.
 *  - The first call on a device looks the array's device address up (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - All calls share the one array: calls that overlap on the GPU (on
 *    different streams, or from different threads) race on it. Stale contents
 *    from an earlier call are harmless; nothing needs clearing.
 */
#define TREE_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
tree_status_t tree_attn_bwd_static_scratch(const tree_plan_t* plan, const void* dout, const void* q,
                                           const void* k, const void* v, const void* o,
                                           const float* lse, void* dq, void* dk, void* dv,
                                           int32_t hq, int32_t hkv, int32_t head_dim,
                                           tree_dtype_t dtype, tree_dtype_t grad_dtype,
                                           float softmax_scale, tree_stream_t stream);

/* Per-token loss weights g_t / K of the token's trie (§3.1 eq. 4, §3.2 "Loss
 * Weights"), each rounded once to fp32, into host memory out_host[N]. */
tree_status_t tree_weights(const tree_plan_t* plan, float* out_host);

/* Per-token weights for any path weighting (§3.1, after eq. 5: with path
 * weights w_k, token t carries lambda_t = sum of w_k over the paths k through
 * it; w_k = 1/K of the trie gives tree_weights). path_weights_host has one
 * fp64 weight per root-to-leaf path of the whole forest, TREE_FIELD_TRIE_PATHS
 * summed; paths are numbered by their leaf segments in DFS order (the order
 * the leaves' tokens appear in the layout). The sums are formed in fp64 and
 * each lambda_t is rounded once to fp32 into host memory out_host[N].
 * Errors: NULL pointers (with N > 0), num_paths different from the forest's
 * path count, or a non-finite weight -> TREE_ERR_INVALID_ARG. */
tree_status_t tree_weights_paths(const tree_plan_t* plan, const double* path_weights_host,
                                 int32_t num_paths, float* out_host);

/* One partition of the redundancy-free tree partitioning (§3.3
 * "Partitioning"; App. B). A partition is a connected piece of one trie, cut
 * only at node boundaries, processed as one DFS forward pass. */
typedef struct {
  int32_t root;       /* segment at the top of the partition */
  int32_t parent;     /* partition holding the root's parent segment; -1 at a trie root */
  int64_t tokens;     /* tokens of the partition's own segments (at most the cap) */
  int64_t pos_offset; /* App. B.4 eq. 17: position id of the root's first token */
  int64_t past_len;   /* App. B.2 gateway length: the parent's past_len plus the parent's DFS
                         tokens up to and including the cut node (the root's parent); 0 at a
                         trie root */
} tree_partition_t;

/* Partition the forest into the fewest connected pieces of at most cap_tokens
 * tokens each, cutting only between a segment and its parent (§3.3
 * "Partitioning": node-boundary cuts keep the partitions' dependency graph a
 * tree). Bottom-up, each segment keeps its children's uncut remainders and,
 * while its total exceeds the cap, cuts off the heaviest one (ties: the
 * lowest segment id) -- the greedy of Kundu and Misra (1977), optimal for the
 * number of pieces. Outputs (host memory):
 *  - part_of_segment[S]: the partition of each segment;
 *  - parts[S] (the first *num_parts used): partitions numbered by their roots
 *    in DFS order, so a parent partition precedes its children;
 *  - *peak_path_tokens: the largest sum of partition sizes along a chain of
 *    parent partitions (what the backward keeps alive at once, §3.3).
 * Errors: NULL pointers (S > 0) or cap_tokens < 1 -> TREE_ERR_INVALID_ARG; a
 * segment longer than cap_tokens -> TREE_ERR_UNSUPPORTED (no node-boundary
 * partition exists). */
tree_status_t tree_partition(const tree_plan_t* plan, int64_t cap_tokens, int32_t* part_of_segment,
                             tree_partition_t* parts, int32_t* num_parts, int64_t* peak_path_tokens);

/* Tree-correct causal depthwise convolution (App. A.3 "Tree-Correct Causal
 * Convolution"; eq. 11): each segment takes its left context from its
 * parent's last K-1 effective tokens, so every token sees the K-1 tokens
 * before it on its own root-to-leaf path (zeros before the root), as in a
 * standalone per-path forward:
 *   y[t, c] = act(bias[c] + sum_{k=0}^{K-1} weight[c, K-1-k] x[pred_k(t), c]),
 * pred_0(t) = t and pred_k(t) the k-th token before t on its path (weight
 * index K-1 on the token itself, the causal conv1d convention).
 * Tensors are token-major in the plan's DFS order: x, y, dy, dx [N, channels]
 * (bf16 or fp32 by dtype, 16-byte aligned); weight, dweight [channels, K] and
 * bias, dbias [channels] in fp32. Arithmetic is fp32; the backward is
 * deterministic. activation: TREE_ACT_NONE or TREE_ACT_SILU. */
typedef enum { TREE_ACT_NONE = 0, TREE_ACT_SILU = 1 } tree_activation_t;

/* Build and upload the path-predecessor tables for kernel size K (1 to 8) on
 * the current device; the plan keeps one kernel size at a time and frees them
 * with the plan. Preparing another size frees the previous tables (after a
 * device synchronization) and rebuilds them, so alternating sizes on one plan
 * pays a rebuild each time, and a plan must not be prepared for a different
 * size while another thread is calling tree_conv_fwd / tree_conv_bwd with it:
 * threads that need different kernel sizes build their own plans.
 * Errors: K out of range -> TREE_ERR_UNSUPPORTED. */
tree_status_t tree_conv_prepare(tree_plan_t* plan, int32_t kernel_size, tree_stream_t stream);

/* y = conv(x). bias may be NULL. Errors: channels not a positive multiple of
 * 8 -> TREE_ERR_UNSUPPORTED; NULL or misaligned pointers, a bad dtype or
 * activation -> TREE_ERR_INVALID_ARG; tables not prepared on this device ->
 * TREE_ERR_NOT_ON_DEVICE. */
tree_status_t tree_conv_fwd(const tree_plan_t* plan, const void* x, const float* weight,
                            const float* bias, void* y, int32_t channels, tree_dtype_t dtype,
                            int32_t activation, tree_stream_t stream);

/* Scratch the backward needs (fp32 dy * act'(pre) and the reduction's
 * partial sums), for the prepared kernel size. */
size_t tree_conv_bwd_workspace_bytes(const tree_plan_t* plan, int32_t channels);

/* dx, dweight (and dbias unless NULL) of the conv, overwritten (not
 * accumulated). The pre-activation is recomputed from x, weight and bias.
 * An N = 0 plan (after tree_conv_prepare, which records the kernel size)
 * zeroes dweight and dbias and launches no kernel.
 * Errors as tree_conv_fwd, and a workspace below
 * tree_conv_bwd_workspace_bytes -> TREE_ERR_INVALID_ARG. */
tree_status_t tree_conv_bwd(const tree_plan_t* plan, const void* x, const float* weight,
                            const float* bias, const void* dy, void* dx, float* dweight,
                            float* dbias, int32_t channels, tree_dtype_t dtype, int32_t activation,
                            void* workspace, size_t workspace_bytes, tree_stream_t stream);

/* Rotary position embedding at tree position ids, in place on the device
 * tensor x[N, heads, head_dim] (token-major, the plan's DFS token order,
 * contiguous, 16-byte aligned, bf16 or fp32 by dtype). Token t takes the
 * position TREE_FIELD_POS_ID[t] of §3.2 "Position Embedding" (eq. 9), the one
 * it has in every standalone root-to-leaf sequence, so the result equals
 * RoPE (RoFormer, Su et al. 2023) applied to each path on its own.
 *  - Dimension pair i turns by pos * base^(-2i/head_dim): pairs (2i, 2i+1)
 *    when rotate_half = 0, pairs (i, i + head_dim/2) when rotate_half = 1.
 *  - inverse = 1 turns by the opposite angle: the backward of the forward
 *    rotation (grad_x = R^T grad_y) and its exact inverse up to rounding.
 *  - Arithmetic in fp32 (angle reduced in fp64); bf16 results rounded once.
 * Asynchronous on `stream`; the plan must be on the current device (an N = 0
 * plan does nothing, after the scalar checks; x may then be NULL).
 * Errors: head_dim odd or above 128 -> TREE_ERR_UNSUPPORTED; heads <= 0, a bad
 * dtype, base not finite and positive, rotate_half or inverse not 0/1, NULL
 * or misaligned x -> TREE_ERR_INVALID_ARG; plan not on the device ->
 * TREE_ERR_NOT_ON_DEVICE. */
tree_status_t tree_rope(const tree_plan_t* plan, void* x, int32_t heads, int32_t head_dim,
                        tree_dtype_t dtype, float base, int32_t rotate_half, int32_t inverse,
                        tree_stream_t stream);

/* tree_rope on a layer's queries and keys in one launch: q device [N, q_heads,
 * head_dim] and k device [N, k_heads, head_dim] of the same dtype, each
 * rotated in place exactly as tree_rope would (bit for bit), with each
 * token's sines and cosines computed once for both. Errors as tree_rope, and
 * NULL k, k_heads <= 0 or q and k sharing an element -> TREE_ERR_INVALID_ARG. */
tree_status_t tree_rope_qk(const tree_plan_t* plan, void* q, int32_t q_heads, void* k,
                           int32_t k_heads, int32_t head_dim, tree_dtype_t dtype, float base,
                           int32_t rotate_half, int32_t inverse, tree_stream_t stream);

/* Fused weighted next-token cross-entropy over the trie, loss and gradient in
 * one pass ("Tree Training" §3.1 eq. 3-5: the tree loss is sum_t lambda_t *
 * l_t over unique tokens; §3.2 "Loss Weights").
 * On every root-to-leaf path the token after position r is predicted from the
 * logits row r: in the DFS layout token r + 1 when it is in r's segment, else
 * the first token of each child segment of r's segment (a leaf's last token
 * predicts nothing, a root's first token is predicted by nothing). With t
 * predicted from r:
 *   row_loss[r] = sum over r -> t of lambda[t] * (logsumexp(z_r) - z_r[tokens[t]])
 *   dlogits[r]  = grad_scale * sum over r -> t of lambda[t] * (softmax(z_r) - e_tokens[t])
 *   *loss       = sum of row_loss (fp64, fixed order)
 *  - logits, dlogits: device [N, vocab] row-major, bf16 or fp32 by dtype,
 *    16-byte aligned; dlogits may be logits itself (in place) but must not
 *    overlap it otherwise; every element of dlogits is written, each rounded
 *    once from fp32.
 *  - tokens: device int32 [N], the token ids of the DFS sequence; a negative id
 *    means the token is not predicted (an ignored position); an id >= vocab is
 *    skipped and reported by tree_status_sync (TREE_ERR_INVALID_ARG).
 *  - lambda: device fp32 [N], the weight of the prediction of each token (e.g.
 *    tree_weights: g_t / K; any sign; 0 skips it).
 *  - row_loss: device fp32 [N] out; loss: device fp64 out, or NULL.
 *  - vocab: a positive multiple of 8. Arithmetic in fp32 with hardware ex2;
 *    one CTA per row, two passes over it (the second from L2).
 * Asynchronous on `stream`; the plan must be on the current device (an N = 0
 * plan only clears *loss). Errors: NULL plan or pointer, bad dtype or vocab,
 * misaligned or partially overlapping logits/dlogits, grad_scale not finite
 * -> TREE_ERR_INVALID_ARG; a segment with more than 1024 children ->
 * TREE_ERR_UNSUPPORTED; plan not on the device -> TREE_ERR_NOT_ON_DEVICE. */
tree_status_t tree_weighted_ce(const tree_plan_t* plan, const void* logits, void* dlogits,
                               const int32_t* tokens, const float* lambda, int32_t vocab,
                               tree_dtype_t dtype, float grad_scale, float* row_loss, double* loss,
                               tree_stream_t stream);

/* Gated DeltaNet forward with tree state routing ("Tree Training" §3.2 "SSM
 * Layers (GDN)" eq. 10, App. A.2): every segment is one chunk and starts from
 * the end state of its parent segment (a root from initial_state, or zeros),
 * never from the segment before it in DFS order. Per value head h (query/key
 * head h / (hv / hk)) with state S [128, 128] (key dim x value dim), token t:
 *   S_t = exp(g_t) S_{t-1} + k_t (beta_t (v_t - exp(g_t) S_{t-1}^T k_t))^T
 *   o_t = S_t^T q_t
 * q and k are used as given (a GDN layer's L2 normalisation and query scale
 * are applied by the caller).
 *  - q, k: device [N, hk, 128]; v, o: device [N, hv, 128]; bf16 or fp32 by
 *    dtype, token-major in the plan's DFS order, contiguous, 16-byte aligned.
 *  - g (log decay), beta: device fp32 [N, hv].
 *  - initial_state: device fp32 [hv, 128, 128] or NULL (zeros).
 *  - segment_states: device fp32 [S, hv, 128, 128] out (by segment id): the
 *    state after each segment's last token (what a child partition's gateway
 *    carries, App. B.7); also the routing's own store of parent states.
 *  - Arithmetic in fp32 (CUDA cores); o rounded once to its dtype.
 *  - Launches: tree_plan_info's gdn_levels kernels in stream order, one per
 *    level of branch points (sibling branches run side by side).
 * Asynchronous on `stream`; the plan must be on the current device. Errors:
 * head_dim != 128 or hv > 65535 -> TREE_ERR_UNSUPPORTED; NULL plan or pointer,
 * bad dtype, hv % hk != 0, misaligned pointers -> TREE_ERR_INVALID_ARG; plan
 * not on the device -> TREE_ERR_NOT_ON_DEVICE. */
tree_status_t tree_gdn_fwd(const tree_plan_t* plan, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, const float* initial_state, void* o,
                           float* segment_states, int32_t hk, int32_t hv, int32_t head_dim,
                           tree_dtype_t dtype, tree_stream_t stream);

/* Wait for `stream`, then read and clear the device status word of the
 * current device: TREE_ERR_TIMEOUT if a kernel gave up a bounded wait since
 * the last check (the message names the wait: 10000 + source line in the
 * forward kernel file, 20000 + line in the backward one, 30000 + warp for
 * the work ring, 40000 + line in the conv kernel file, 50000 for
 * tree_diag_wait_timeout), TREE_ERR_INVALID_ARG if tree_weighted_ce met a
 * token id >= vocab, TREE_ERR_CUDA on a CUDA error, else TREE_OK. */
tree_status_t tree_status_sync(tree_stream_t stream);

/* Diagnostic of the failure path: launches one thread on `stream` that waits
 * on an mbarrier nothing completes, through the bounded wait every kernel of
 * the library uses, with a limit of limit_ns nanoseconds (1e3 to 1e10) of the
 * GPU's global timer instead of the kernels' 4 s. The wait gives up, stores
 * 50000 in the device status word and the kernel returns, leaving the context
 * usable: the next tree_status_sync reports TREE_ERR_TIMEOUT naming wait site
 * 50000 and clears the word. No fault, trap or hang is involved. Errors:
 * limit_ns out of range -> TREE_ERR_INVALID_ARG (nothing is launched); a
 * launch failure -> TREE_ERR_CUDA. */
tree_status_t tree_diag_wait_timeout(int64_t limit_ns, tree_stream_t stream);

/* Message for the last failing call on this thread ("" if none). */
const char* tree_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TREEATTN_H */
