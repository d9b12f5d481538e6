// Host plan builder: trie -> DFS layout, ancestors, g_n, K, position ids, the
// per-key visibility bound and the tile visibility map.
//
// "Tree Training" (arXiv 2511.00413): §3.1 (trie, g_n, K), eq. 8 (DFS
// serialization), eq. 9 (position ids), §3.2 "Attention Mask" and App. A.1
// (ancestor segments in full, own segment causal; masked blocks skipped).
//
// Column form of the mask used here (a consequence of eq. 8's pre-order):
// the rows that see key j (segment s) are exactly [j, subtree_end(s)), since
// the subtree of s is one contiguous token range in DFS order. For a k-tile
// the union of these row ranges is the single range [k0, max key_end), so
// each k-tile is seen by one contiguous run of q-tiles starting at its own
// diagonal tile.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <new>
#include <numeric>

#include "plan_internal.h"

namespace treeattn {

thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

tree_status_t fail(tree_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

namespace {

// Visible pairs between rows [ra, rb) and keys [k0, k1) that all share the
// bound E (one segment): row i sees key j iff j <= i < E.
int64_t run_pairs(int64_t k0, int64_t k1, int64_t E, int64_t ra, int64_t rb) {
  const int64_t hi = std::min(rb, E);
  if (hi <= ra || k1 <= k0) return 0;
  int64_t total = 0;
  const int64_t c = std::min(k1, ra + 1);  // keys at or before the first row see every row up to hi
  if (c > k0) total += (c - k0) * (hi - ra);
  const int64_t d0 = std::max(k0, ra + 1), d1 = std::min(k1, hi);  // key j sees rows [j, hi)
  if (d1 > d0) total += (d1 - d0) * (2 * hi - d0 - d1 + 1) / 2;
  return total;
}

// Gathered key tiles for units of U query rows (U = 128 or 256); appends to
// the tile table and writes the unit -> tile CSR into ptr.
void build_gathered(tree_plan* p, int32_t U, std::vector<int32_t>& ptr) {
  auto& F = p->field;
  const int32_t N = p->N;
  const auto& tok_seg = F[TREE_FIELD_TOKEN_SEG];
  const auto& seg_start = F[TREE_FIELD_SEG_START];
  const auto& sub_end = F[TREE_FIELD_SUBTREE_END];
  const auto& anc_ptr = F[TREE_FIELD_ANC_PTR];
  const auto& anc_idx = F[TREE_FIELD_ANC_IDX];
  const auto& key_end = F[TREE_FIELD_KEY_END];
  auto& kind = F[TREE_FIELD_GT_KIND];
  auto& atom = F[TREE_FIELD_GT_ATOM];
  auto& bidx = F[TREE_FIELD_GT_BIDX];
  auto& bounds = F[TREE_FIELD_GT_BOUNDS];
  const int32_t units = (N + U - 1) / U;
  const int32_t slots = U / kBlockM;
  ptr.assign(units + 1, static_cast<int32_t>(kind.size()));
  std::vector<int32_t> len_of(p->S);
  for (int32_t s = 0; s < p->S; ++s) len_of[s] = 0;
  for (int32_t t = 0; t < N; ++t) ++len_of[tok_seg[t]];
  using Iv = std::pair<int32_t, int32_t>;
  std::vector<Iv> iv, merged, common, rest, runs;
  struct Piece { int32_t tile, col, key, n, every; };  // n keys from key at column col of a tile
  std::vector<Piece> pieces;
  for (int32_t u = 0; u < units; ++u) {
    const int32_t r0 = u * U, r1 = std::min(N, r0 + U);
    // keys seen by some row: per spanned segment its ancestors and its own
    // prefix up to its last row in the unit
    iv.clear();
    for (int32_t r = r0; r < r1;) {
      const int32_t s = tok_seg[r];
      const int32_t se = seg_start[s] + len_of[s];
      const int32_t rb = std::min(r1, se);
      for (int32_t e = anc_ptr[s]; e < anc_ptr[s + 1]; ++e) {
        const int32_t a = anc_idx[e];
        iv.emplace_back(seg_start[a], seg_start[a] + len_of[a]);
      }
      iv.emplace_back(seg_start[s], rb);
      r = rb;
    }
    std::sort(iv.begin(), iv.end());
    merged.clear();
    for (const Iv& x : iv) {
      if (!merged.empty() && x.first <= merged.back().second)
        merged.back().second = std::max(merged.back().second, x.second);
      else
        merged.push_back(x);
    }
    // split into keys every row sees (j <= r0 and key_end[j] >= r1) and the rest
    common.clear();
    rest.clear();
    auto push = [](std::vector<Iv>& v, int32_t a, int32_t b) {
      if (b <= a) return;
      if (!v.empty() && v.back().second == a)
        v.back().second = b;
      else
        v.emplace_back(a, b);
    };
    for (const Iv& x : merged) {
      for (int32_t j = x.first; j < x.second;) {  // walk the interval by segments
        const int32_t s = tok_seg[j];
        const int32_t e = std::min(x.second, seg_start[s] + len_of[s]);
        if (sub_end[s] >= r1) {
          const int32_t c = std::min(e, r0 + 1);
          push(common, j, std::max(j, c));
          push(rest, std::max(j, c), e);
        } else {
          push(rest, j, e);
        }
        j = e;
      }
    }
    // gateway keys first: every row of the partition sees the visible ones
    // (their own tiles, flagged; atoms hold rows of the past keys)
    if (!p->gw_runs.empty()) {
      int32_t gcol = kBlockN;
      pieces.clear();
      int32_t gtiles = 0;
      for (const Iv& x : p->gw_runs) {
        int32_t k = x.first, n = x.second - x.first;
        while (n > 0) {
          if (gcol >= kBlockN) {
            ++gtiles;
            gcol = 0;
          }
          const int32_t m = std::min(n, kBlockN - gcol);
          pieces.push_back({gtiles - 1, gcol, k, m, 1});
          gcol += m;
          k += m;
          n -= m;
        }
        gcol = (gcol + 7) & ~7;
      }
      for (size_t b = 0, e = 0; b < pieces.size(); b = e) {
        const int32_t tile = pieces[b].tile;
        int32_t cols = 0;
        while (e < pieces.size() && pieces[e].tile == tile) cols += pieces[e++].n;
        int32_t kw = 16;
        bool partial = false;
        for (int32_t sl = 0; sl < slots; ++sl) {
          const int32_t ra = r0 + sl * kBlockM, rb = std::min(r1, ra + kBlockM);
          int32_t kd = kEmpty;
          if (ra < rb) kd = (cols == kBlockN && rb - ra == kBlockM) ? kFull : kPartial;
          partial = partial || kd == kPartial;
          kw |= kd << (2 * sl);
        }
        kind.push_back(kw);
        int32_t a_row[kBlockN / 8];
        for (int32_t a = 0; a < kBlockN / 8; ++a) a_row[a] = -8;
        for (size_t q = b; q < e; ++q)
          for (int32_t c = pieces[q].col; c < pieces[q].col + pieces[q].n; c += 8)
            a_row[c / 8] = pieces[q].key + (c - pieces[q].col);
        atom.insert(atom.end(), a_row, a_row + kBlockN / 8);
        if (partial) {
          bidx.push_back(static_cast<int32_t>(bounds.size() / kBlockN));
          const size_t b0 = bounds.size();
          bounds.resize(b0 + kBlockN, 0);
          for (size_t q = b; q < e; ++q)
            for (int32_t c = 0; c < pieces[q].n; ++c) bounds[b0 + pieces[q].col + c] = N;
        } else {
          bidx.push_back(-1);
        }
      }
    }
    runs.clear();
    for (const Iv& x : common) push(runs, x.first, x.second);
    // runs[0 .. n_common) hold only keys every row of the unit sees (the run
    // that joins the two lists, if any, counts as mixed)
    size_t n_common = runs.size();
    for (const Iv& x : rest) {
      if (!runs.empty() && runs.back().second == x.first && runs.size() == n_common) --n_common;
      push(runs, x.first, x.second);
    }
    // place the runs: each starts at an 8-aligned column, a tile holds 128
    pieces.clear();
    int32_t ntiles = 0, col = kBlockN;
    for (size_t ri = 0; ri < runs.size(); ++ri) {
      const Iv& x = runs[ri];
      const int32_t every = ri < n_common ? 1 : 0;
      int32_t k = x.first, n = x.second - x.first;
      while (n > 0) {
        if (col >= kBlockN) {
          ++ntiles;
          col = 0;
        }
        const int32_t m = std::min(n, kBlockN - col);
        pieces.push_back({ntiles - 1, col, k, m, every});
        col += m;
        k += m;
        n -= m;
      }
      col = (col + 7) & ~7;
    }
    for (size_t b = 0, e = 0; b < pieces.size(); b = e) {
      const int32_t tile = pieces[b].tile;
      while (e < pieces.size() && pieces[e].tile == tile) ++e;
      int32_t kw = 0;
      bool partial = false;
      for (int32_t sl = 0; sl < slots; ++sl) {
        const int32_t ra = r0 + sl * kBlockM, rb = std::min(r1, ra + kBlockM);
        int32_t kd = kEmpty;
        if (ra < rb) {
          int64_t pairs = 0;
          for (size_t q = b; q < e; ++q) {
            const Piece& pc = pieces[q];
            if (pc.every) {  // every row of the unit sees every key of the piece
              pairs += static_cast<int64_t>(pc.n) * (rb - ra);
              continue;
            }
            for (int32_t j = pc.key; j < pc.key + pc.n;) {
              const int32_t s = tok_seg[j];
              const int32_t se = std::min(pc.key + pc.n, seg_start[s] + len_of[s]);
              pairs += run_pairs(j, se, sub_end[s], ra, rb);
              j = se;
            }
          }
          if (pairs == int64_t{kBlockM} * kBlockN) kd = kFull;
          else if (pairs > 0) kd = kPartial;
        }
        partial = partial || kd == kPartial;
        kw |= kd << (2 * sl);
      }
      kind.push_back(kw);
      int32_t a_row[kBlockN / 8];
      for (int32_t a = 0; a < kBlockN / 8; ++a) a_row[a] = -8;
      for (size_t q = b; q < e; ++q)
        for (int32_t c = pieces[q].col; c < pieces[q].col + pieces[q].n; c += 8)
          a_row[c / 8] = pieces[q].key + (c - pieces[q].col);
      atom.insert(atom.end(), a_row, a_row + kBlockN / 8);
      if (partial) {
        bidx.push_back(static_cast<int32_t>(bounds.size() / kBlockN));
        const size_t b0 = bounds.size();
        bounds.resize(b0 + kBlockN, 0);
        for (size_t q = b; q < e; ++q)
          for (int32_t c = 0; c < pieces[q].n; ++c)
            bounds[b0 + pieces[q].col + c] = key_end[pieces[q].key + c];
      } else {
        bidx.push_back(-1);
      }
    }
    ptr[u + 1] = static_cast<int32_t>(kind.size());
  }
}

// The gateway of a partition plan: visible key runs and the per-key bound.
void build_gateway(tree_plan* p, const uint8_t* visible, int32_t past_len) {
  auto& F = p->field;
  p->past_len = past_len;
  p->gw_runs.clear();
  int64_t nvis = 0;
  for (int32_t j = 0; j < past_len;) {
    if (!visible[j]) {
      ++j;
      continue;
    }
    int32_t e = j;
    while (e < past_len && visible[e]) ++e;
    p->gw_runs.emplace_back(j, e);
    nvis += e - j;
    j = e;
  }
  p->past_visible = nvis;
  const int32_t tiles = (past_len + kBlockN - 1) / kBlockN;
  auto& kend = F[TREE_FIELD_GW_KEND];
  kend.assign(static_cast<size_t>(tiles) * kBlockN, 0);
  for (int32_t j = 0; j < past_len; ++j) kend[j] = visible[j] ? p->N : 0;
  auto& kt = F[TREE_FIELD_GW_KT];
  kt.clear();
  for (int32_t t = 0; t < tiles; ++t) {
    bool any = false;
    for (int32_t j = t * kBlockN; j < std::min(past_len, (t + 1) * kBlockN) && !any; ++j) any = visible[j] != 0;
    if (any) kt.push_back(t);
  }
}

// Units and levels of the GDN forward's level-by-level launch (tree_plan::
// gdn_units): a segment starts a unit unless it is the only child of its
// parent (then it follows the parent in DFS order and continues its state).
void build_gdn_units(tree_plan* p, const int32_t* parents) {
  const int32_t S = p->S;
  const auto& order = p->field[TREE_FIELD_DFS_ORDER];
  const auto& start = p->field[TREE_FIELD_SEG_START];
  std::vector<int32_t> nchild(S, 0), unit_of(S, -1), level;
  for (int32_t s = 0; s < S; ++s)
    if (parents[s] >= 0) ++nchild[parents[s]];
  std::vector<int32_t> u;  // 4 per unit, DFS order
  for (int32_t d = 0; d < S; ++d) {
    const int32_t s = order[d], par = parents[s];
    if (par >= 0 && nchild[par] == 1) {  // continues its parent's unit (at d - 1)
      const int32_t id = unit_of[par];
      unit_of[s] = id;
      u[4 * id + 1] = d + 1;
      continue;
    }
    const int32_t id = static_cast<int32_t>(level.size());
    unit_of[s] = id;
    level.push_back(par < 0 ? 0 : level[unit_of[par]] + 1);
    u.insert(u.end(), {d, d + 1, start[s], 0});
  }
  // a unit's tokens end where its last segment's own tokens end
  std::vector<int32_t> seg_len(S, 0);
  for (int32_t t : p->field[TREE_FIELD_TOKEN_SEG]) ++seg_len[t];
  const int32_t U = static_cast<int32_t>(level.size());
  for (int32_t id = 0; id < U; ++id) {
    const int32_t last = order[u[4 * id + 1] - 1];
    u[4 * id + 3] = start[last] + seg_len[last];
  }
  std::vector<int32_t> idx(U);
  for (int32_t i = 0; i < U; ++i) idx[i] = i;
  std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
    if (level[a] != level[b]) return level[a] < level[b];
    return u[4 * a + 3] - u[4 * a + 2] > u[4 * b + 3] - u[4 * b + 2];
  });
  const int32_t L = U ? 1 + *std::max_element(level.begin(), level.end()) : 0;
  p->gdn_units.resize(static_cast<size_t>(U) * 4);
  p->gdn_level_ptr.assign(static_cast<size_t>(L) + 1, 0);
  for (int32_t i = 0; i < U; ++i) {
    for (int c = 0; c < 4; ++c) p->gdn_units[4 * i + c] = u[4 * idx[i] + c];
    ++p->gdn_level_ptr[level[idx[i]] + 1];
  }
  for (int32_t l = 0; l < L; ++l) p->gdn_level_ptr[l + 1] += p->gdn_level_ptr[l];
}

tree_status_t build(const int32_t* parents, const int32_t* lengths, int32_t S, tree_plan* p,
                    const uint8_t* past_visible = nullptr, int32_t past_len = 0,
                    int32_t pos_offset = 0) {
  auto& F = p->field;
  // ---- validation
  for (int32_t s = 0; s < S; ++s) {
    if (parents[s] < -1 || parents[s] >= S || parents[s] == s)
      return fail(TREE_ERR_INVALID_ARG, "segment " + std::to_string(s) + ": parent " +
                                            std::to_string(parents[s]) + " out of range");
  }
  int64_t n_tokens = 0;
  for (int32_t s = 0; s < S; ++s) {
    if (lengths[s] < 1)
      return fail(TREE_ERR_EMPTY_SEGMENT, "segment " + std::to_string(s) + " has " +
                                              std::to_string(lengths[s]) + " tokens");
    n_tokens += lengths[s];
  }
  if (n_tokens > std::numeric_limits<int32_t>::max() - kBlockM)
    return fail(TREE_ERR_OVERFLOW, "more than 2^31-129 tokens");
  if (n_tokens + pos_offset > std::numeric_limits<int32_t>::max())
    return fail(TREE_ERR_OVERFLOW, "position ids past 2^31-1");
  const int32_t N = static_cast<int32_t>(n_tokens);

  // ---- children (ascending id) and roots (ascending id)
  std::vector<int32_t> child_ptr(S + 1, 0), child_idx(S);
  std::vector<int32_t> roots;
  for (int32_t s = 0; s < S; ++s) {
    if (parents[s] < 0)
      roots.push_back(s);
    else
      child_ptr[parents[s] + 1]++;
  }
  for (int32_t s = 0; s < S; ++s) child_ptr[s + 1] += child_ptr[s];
  {
    std::vector<int32_t> fill(child_ptr.begin(), child_ptr.end() - 1);
    for (int32_t s = 0; s < S; ++s)
      if (parents[s] >= 0) child_idx[fill[parents[s]]++] = s;
  }

  // ---- pre-order (eq. 8): a node, then each child's subtree in ascending id
  std::vector<int32_t>& order = F[TREE_FIELD_DFS_ORDER];
  order.reserve(S);
  {
    std::vector<int32_t> stack;
    for (auto it = roots.rbegin(); it != roots.rend(); ++it) stack.push_back(*it);
    while (!stack.empty()) {
      int32_t s = stack.back();
      stack.pop_back();
      order.push_back(s);
      for (int32_t e = child_ptr[s + 1] - 1; e >= child_ptr[s]; --e) stack.push_back(child_idx[e]);
    }
  }
  if (static_cast<int32_t>(order.size()) != S)
    return fail(TREE_ERR_CYCLE, "some segment does not reach a root (cycle)");

  // ---- per-segment fields
  std::vector<int32_t>& seg_start = F[TREE_FIELD_SEG_START];
  std::vector<int32_t>& depth = F[TREE_FIELD_DEPTH];
  std::vector<int32_t>& sub_end = F[TREE_FIELD_SUBTREE_END];
  std::vector<int32_t>& trie_id = F[TREE_FIELD_TRIE_ID];
  std::vector<int32_t>& g = F[TREE_FIELD_G];
  seg_start.assign(S, 0);
  depth.assign(S, 0);
  sub_end.assign(S, 0);
  trie_id.assign(S, 0);
  g.assign(S, 0);
  std::vector<int32_t> pos_base(S, 0);
  {
    int32_t off = 0, root_rank = 0;
    for (int32_t s : order) {
      seg_start[s] = off;
      off += lengths[s];
      const int32_t par = parents[s];
      if (par < 0) {
        depth[s] = 0;
        pos_base[s] = pos_offset;
        trie_id[s] = root_rank++;
      } else {  // the parent precedes its children in pre-order
        depth[s] = depth[par] + 1;
        pos_base[s] = pos_base[par] + lengths[par];
        trie_id[s] = trie_id[par];
      }
      sub_end[s] = seg_start[s] + lengths[s];
    }
  }
  for (int32_t e = S - 1; e >= 0; --e) {  // reverse pre-order: children before parents
    const int32_t s = order[e];
    if (g[s] == 0) g[s] = 1;  // a leaf carries one path
    const int32_t par = parents[s];
    if (par >= 0) {
      g[par] += g[s];
      sub_end[par] = std::max(sub_end[par], sub_end[s]);
    }
  }
  const int32_t R = static_cast<int32_t>(roots.size());
  std::vector<int32_t>& cu = F[TREE_FIELD_CU_SEQLENS];
  std::vector<int32_t>& K = F[TREE_FIELD_TRIE_PATHS];
  cu.resize(R + 1);
  K.resize(R);
  for (int32_t r = 0; r < R; ++r) {
    cu[r] = seg_start[roots[r]];
    K[r] = g[roots[r]];
  }
  cu[R] = N;

  // ---- ancestors (CSR by segment id, root first)
  std::vector<int32_t>& anc_ptr = F[TREE_FIELD_ANC_PTR];
  std::vector<int32_t>& anc_idx = F[TREE_FIELD_ANC_IDX];
  anc_ptr.assign(S + 1, 0);
  {
    int64_t total = 0;
    for (int32_t s = 0; s < S; ++s) {
      total += depth[s];
      if (total > std::numeric_limits<int32_t>::max())
        return fail(TREE_ERR_OVERFLOW, "more than 2^31-1 ancestor entries");
      anc_ptr[s + 1] = static_cast<int32_t>(total);
    }
    anc_idx.resize(static_cast<size_t>(total));
    for (int32_t s = 0; s < S; ++s) {
      int32_t w = anc_ptr[s + 1];
      for (int32_t a = parents[s]; a >= 0; a = parents[a]) anc_idx[--w] = a;
    }
  }

  // ---- per-token fields
  std::vector<int32_t>& tok_seg = F[TREE_FIELD_TOKEN_SEG];
  std::vector<int32_t>& pos_id = F[TREE_FIELD_POS_ID];
  std::vector<int32_t>& key_end = F[TREE_FIELD_KEY_END];
  tok_seg.resize(N);
  pos_id.resize(N);
  key_end.resize(N);
  int64_t visible = 0;
  for (int32_t s : order) {
    const int32_t a = seg_start[s], L = lengths[s], ke = sub_end[s];
    for (int32_t j = 0; j < L; ++j) {
      tok_seg[a + j] = s;
      pos_id[a + j] = pos_base[s] + j;
      key_end[a + j] = ke;
      visible += ke - (a + j);
    }
  }

  // ---- tile map on the 128 x 128 grid
  const int32_t Tq = (N + kBlockM - 1) / kBlockM;
  const int32_t Tk = (N + kBlockN - 1) / kBlockN;
  std::vector<int32_t>& kt_qlo = F[TREE_FIELD_KT_QLO];
  std::vector<int32_t>& kt_qhi = F[TREE_FIELD_KT_QHI];
  kt_qlo.resize(Tk);
  kt_qhi.resize(Tk);
  std::vector<int32_t> min_ke(Tk), max_ke(Tk);
  for (int32_t kt = 0; kt < Tk; ++kt) {
    const int32_t j0 = kt * kBlockN, j1 = std::min(N, j0 + kBlockN);
    int32_t lo = key_end[j0], hi = key_end[j0];
    for (int32_t j = j0 + 1; j < j1; ++j) {
      lo = std::min(lo, key_end[j]);
      hi = std::max(hi, key_end[j]);
    }
    min_ke[kt] = lo;
    max_ke[kt] = hi;
    kt_qlo[kt] = kt;                               // the diagonal tile: every key sees itself
    kt_qhi[kt] = (hi - 1) / kBlockM + 1;           // the last row that sees a key of the tile
  }
  std::vector<int32_t>& qt_ptr = F[TREE_FIELD_QT_PTR];
  std::vector<int32_t>& qt_kt = F[TREE_FIELD_QT_KT];
  std::vector<int32_t>& qt_kind = F[TREE_FIELD_QT_KIND];
  qt_ptr.assign(Tq + 1, 0);
  int64_t nnz = 0;
  for (int32_t kt = 0; kt < Tk; ++kt) {
    for (int32_t qt = kt_qlo[kt]; qt < kt_qhi[kt]; ++qt) qt_ptr[qt + 1]++;
    nnz += kt_qhi[kt] - kt_qlo[kt];
  }
  if (nnz > std::numeric_limits<int32_t>::max()) return fail(TREE_ERR_OVERFLOW, "too many tiles");
  for (int32_t qt = 0; qt < Tq; ++qt) qt_ptr[qt + 1] += qt_ptr[qt];
  qt_kt.resize(nnz);
  qt_kind.resize(nnz);
  {
    std::vector<int32_t> fill(qt_ptr.begin(), qt_ptr.end() - 1);
    for (int32_t kt = 0; kt < Tk; ++kt) {  // ascending kt -> ascending lists
      for (int32_t qt = kt_qlo[kt]; qt < kt_qhi[kt]; ++qt) {
        const int32_t r1 = (qt + 1) * kBlockM;
        // FULL: all keys precede all rows, every row below every key's bound, tile inside N
        const bool full = kt < qt && r1 <= N && min_ke[kt] >= r1;
        const int32_t e = fill[qt]++;
        qt_kt[e] = kt;
        qt_kind[e] = full ? kFull : kPartial;
      }
    }
  }

  // ---- q-tile pair union lists (q-tiles 2p and 2p+1)
  const int32_t P = (Tq + 1) / 2;
  std::vector<int32_t>& qp_ptr = F[TREE_FIELD_QP_PTR];
  std::vector<int32_t>& qp_kt = F[TREE_FIELD_QP_KT];
  std::vector<int32_t>& qp_kind = F[TREE_FIELD_QP_KIND];
  qp_ptr.assign(P + 1, 0);
  for (int32_t pr = 0; pr < P; ++pr) {
    const int32_t q0 = 2 * pr, q1 = 2 * pr + 1;
    int32_t a = qt_ptr[q0], ae = qt_ptr[q0 + 1];
    int32_t b = q1 < Tq ? qt_ptr[q1] : 0, be = q1 < Tq ? qt_ptr[q1 + 1] : 0;
    while (a < ae || b < be) {
      int32_t kt, k0 = kEmpty, k1 = kEmpty;
      if (b >= be || (a < ae && qt_kt[a] < qt_kt[b])) {
        kt = qt_kt[a];
        k0 = qt_kind[a++];
      } else if (a >= ae || qt_kt[b] < qt_kt[a]) {
        kt = qt_kt[b];
        k1 = qt_kind[b++];
      } else {
        kt = qt_kt[a];
        k0 = qt_kind[a++];
        k1 = qt_kind[b++];
      }
      qp_kt.push_back(kt);
      qp_kind.push_back(k0 | (k1 << 2));
    }
    qp_ptr[pr + 1] = static_cast<int32_t>(qp_kt.size());
  }

  // ---- work orders: DFS position. Q-tiles (and pairs) last to first: a
  // q-tile late in a trie sees at least as many keys as the ones before it
  // on its path, so heavy work starts first, and neighbouring q-tiles, which
  // share most of their k-tiles, run side by side. K-tiles first to last:
  // ancestors precede their subtrees, so the longest q-tile ranges start first.
  {
    std::vector<int32_t>& fo = F[TREE_FIELD_FWD_ORDER];
    fo.resize(Tq);
    for (int32_t t = 0; t < Tq; ++t) fo[t] = Tq - 1 - t;
    std::vector<int32_t>& po = F[TREE_FIELD_QP_ORDER];
    po.resize(P);
    for (int32_t t = 0; t < P; ++t) po[t] = P - 1 - t;
    std::vector<int32_t>& bo = F[TREE_FIELD_BWD_ORDER];
    bo.resize(Tk);
    std::iota(bo.begin(), bo.end(), 0);
  }

  p->N = N;
  p->S = S;
  p->R = R;
  p->Tq = Tq;
  p->Tk = Tk;
  p->P = P;
  p->visible_pairs = visible;

  if (past_len > 0) build_gateway(p, past_visible, past_len);
  build_gdn_units(p, parents);
  // ---- gathered key tiles: q-tiles first, then q-tile pairs, one table
  {
    const size_t est = static_cast<size_t>(nnz) * 3 / 2 + 16;  // about nnz + nnz / 2 tiles
    F[TREE_FIELD_GT_KIND].reserve(est);
    F[TREE_FIELD_GT_BIDX].reserve(est);
    F[TREE_FIELD_GT_ATOM].reserve(est * (kBlockN / 8));
  }
  build_gathered(p, kBlockM, F[TREE_FIELD_GQ_PTR]);
  build_gathered(p, 2 * kBlockM, F[TREE_FIELD_GP_PTR]);
  if (F[TREE_FIELD_GT_KIND].size() > static_cast<size_t>(std::numeric_limits<int32_t>::max() / 16))
    return fail(TREE_ERR_OVERFLOW, "too many gathered tiles");
  return TREE_OK;
}

}  // namespace
}  // namespace treeattn

using namespace treeattn;

namespace {
tree_status_t plan_entry(const int32_t* segment_parents, const int32_t* segment_lengths,
                         int32_t num_segments, const uint8_t* past_visible, int32_t past_len,
                         int32_t pos_offset, tree_plan_t** out) {
  if (!out) return fail(TREE_ERR_INVALID_ARG, "out is NULL");
  if (num_segments < 0) return fail(TREE_ERR_INVALID_ARG, "num_segments < 0");
  if (num_segments > 0 && (!segment_parents || !segment_lengths))
    return fail(TREE_ERR_INVALID_ARG, "NULL parents or lengths");
  if (past_len < 0) return fail(TREE_ERR_INVALID_ARG, "past_len < 0");
  if (past_len > 0 && !past_visible) return fail(TREE_ERR_INVALID_ARG, "NULL past_visible");
  if (pos_offset < 0) return fail(TREE_ERR_INVALID_ARG, "pos_offset < 0");
  tree_plan* p = new (std::nothrow) tree_plan();
  if (!p) return fail(TREE_ERR_OOM, "out of host memory");
  tree_status_t st;
  try {
    st = build(segment_parents, segment_lengths, num_segments, p, past_visible, past_len, pos_offset);
  } catch (const std::bad_alloc&) {
    st = fail(TREE_ERR_OOM, "out of host memory");
  }
  if (st != TREE_OK) {
    delete p;
    return st;
  }
  *out = p;
  set_error("");
  return TREE_OK;
}
}  // namespace

extern "C" tree_status_t tree_plan_build(const int32_t* segment_parents,
                                         const int32_t* segment_lengths, int32_t num_segments,
                                         tree_plan_t** out) {
  return plan_entry(segment_parents, segment_lengths, num_segments, nullptr, 0, 0, out);
}

extern "C" tree_status_t tree_plan_build_partition(const int32_t* segment_parents,
                                                   const int32_t* segment_lengths,
                                                   int32_t num_segments, const uint8_t* past_visible,
                                                   int32_t past_len, int32_t pos_offset,
                                                   tree_plan_t** out) {
  return plan_entry(segment_parents, segment_lengths, num_segments, past_visible, past_len,
                    pos_offset, out);
}

extern "C" tree_status_t tree_plan_info(const tree_plan_t* p, tree_plan_info_t* out) {
  if (!p || !out) return fail(TREE_ERR_INVALID_ARG, "NULL plan or out");
  out->num_tokens = p->N;
  out->num_segments = p->S;
  out->num_tries = p->R;
  out->block_m = kBlockM;
  out->block_n = kBlockN;
  out->num_q_tiles = p->Tq;
  out->num_k_tiles = p->Tk;
  out->nnz_tiles = static_cast<int64_t>(p->field[TREE_FIELD_QT_KT].size());
  out->num_pairs = p->P;
  out->nnz_pair_tiles = static_cast<int64_t>(p->field[TREE_FIELD_QP_KT].size());
  out->num_ancestors = static_cast<int64_t>(p->field[TREE_FIELD_ANC_IDX].size());
  out->visible_pairs = p->visible_pairs;
  out->num_gathered_tiles = static_cast<int64_t>(p->field[TREE_FIELD_GT_KIND].size());
  out->past_len = p->past_len;
  out->past_visible = p->past_visible;
  out->gdn_levels = p->gdn_level_ptr.empty() ? 0 : static_cast<int64_t>(p->gdn_level_ptr.size()) - 1;
  return TREE_OK;
}

extern "C" tree_status_t tree_plan_field_len(const tree_plan_t* p, tree_plan_field_t f,
                                             int64_t* out) {
  if (!p || !out) return fail(TREE_ERR_INVALID_ARG, "NULL plan or out");
  if (static_cast<int>(f) < 0 || f >= TREE_FIELD_COUNT)
    return fail(TREE_ERR_INVALID_ARG, "unknown field");
  *out = static_cast<int64_t>(p->field[f].size());
  return TREE_OK;
}

extern "C" tree_status_t tree_plan_get(const tree_plan_t* p, tree_plan_field_t f, void* dst,
                                       size_t bytes) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (static_cast<int>(f) < 0 || f >= TREE_FIELD_COUNT)
    return fail(TREE_ERR_INVALID_ARG, "unknown field");
  const auto& v = p->field[f];
  if (bytes != v.size() * sizeof(int32_t))
    return fail(TREE_ERR_INVALID_ARG, "field has " + std::to_string(v.size() * 4) +
                                          " bytes, got " + std::to_string(bytes));
  if (!v.empty()) {
    if (!dst) return fail(TREE_ERR_INVALID_ARG, "NULL dst");
    std::memcpy(dst, v.data(), bytes);
  }
  return TREE_OK;
}

extern "C" tree_status_t tree_weights(const tree_plan_t* p, float* out_host) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (p->N > 0 && !out_host) return fail(TREE_ERR_INVALID_ARG, "NULL out");
  const auto& seg = p->field[TREE_FIELD_TOKEN_SEG];
  const auto& g = p->field[TREE_FIELD_G];
  const auto& trie = p->field[TREE_FIELD_TRIE_ID];
  const auto& K = p->field[TREE_FIELD_TRIE_PATHS];
  for (int32_t t = 0; t < p->N; ++t) {
    const int32_t s = seg[t];
    // g and K are below 2^31; the fp64 quotient rounded to fp32 is the
    // correctly rounded fp32 quotient when both are below 2^24 (53 >= 2*24+2).
    out_host[t] = static_cast<float>(static_cast<double>(g[s]) / static_cast<double>(K[trie[s]]));
  }
  return TREE_OK;
}

extern "C" tree_status_t tree_weights_paths(const tree_plan_t* p, const double* w, int32_t num_paths,
                                           float* out_host) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  int64_t K_total = 0;
  for (int32_t k : p->field[TREE_FIELD_TRIE_PATHS]) K_total += k;
  if (num_paths != K_total)
    return fail(TREE_ERR_INVALID_ARG, "the forest has " + std::to_string(K_total) + " paths, got " +
                                          std::to_string(num_paths) + " weights");
  if (p->N == 0) return TREE_OK;
  if (!w || !out_host) return fail(TREE_ERR_INVALID_ARG, "NULL pointer");
  for (int32_t k = 0; k < num_paths; ++k)
    if (!std::isfinite(w[k])) return fail(TREE_ERR_INVALID_ARG, "non-finite path weight");
  const auto& order = p->field[TREE_FIELD_DFS_ORDER];
  const auto& start = p->field[TREE_FIELD_SEG_START];
  const auto& sub_end = p->field[TREE_FIELD_SUBTREE_END];
  const auto& anc_ptr = p->field[TREE_FIELD_ANC_PTR];
  const auto& anc_idx = p->field[TREE_FIELD_ANC_IDX];
  const auto& seg = p->field[TREE_FIELD_TOKEN_SEG];
  // A segment is a leaf when its subtree holds nothing past its own tokens;
  // leaves meet in DFS order, which numbers the paths. Each path adds its
  // weight to its leaf and to every ancestor of it.
  std::vector<int32_t> len(p->S, 0);
  for (int32_t t = 0; t < p->N; ++t) ++len[seg[t]];
  std::vector<double> lam(p->S, 0.0);
  int32_t k = 0;
  for (int32_t s : order) {
    if (sub_end[s] != start[s] + len[s]) continue;
    lam[s] += w[k];
    for (int32_t a = anc_ptr[s]; a < anc_ptr[s + 1]; ++a) lam[anc_idx[a]] += w[k];
    ++k;
  }
  for (int32_t t = 0; t < p->N; ++t) out_host[t] = static_cast<float>(lam[seg[t]]);
  return TREE_OK;
}

extern "C" tree_status_t tree_partition(const tree_plan_t* p, int64_t cap, int32_t* part_of,
                                       tree_partition_t* parts, int32_t* num_parts,
                                       int64_t* peak_path_tokens) {
  if (!p) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  if (cap < 1) return fail(TREE_ERR_INVALID_ARG, "cap_tokens must be at least 1");
  if (!num_parts || !peak_path_tokens) return fail(TREE_ERR_INVALID_ARG, "NULL output");
  *num_parts = 0;
  *peak_path_tokens = 0;
  const int32_t S = p->S;
  if (S == 0) return TREE_OK;
  if (!part_of || !parts) return fail(TREE_ERR_INVALID_ARG, "NULL output");
  const auto& order = p->field[TREE_FIELD_DFS_ORDER];
  const auto& anc_ptr = p->field[TREE_FIELD_ANC_PTR];
  const auto& anc_idx = p->field[TREE_FIELD_ANC_IDX];
  const auto& seg = p->field[TREE_FIELD_TOKEN_SEG];
  const auto& start = p->field[TREE_FIELD_SEG_START];
  const auto& pos = p->field[TREE_FIELD_POS_ID];
  std::vector<int64_t> len(S, 0);
  for (int32_t t = 0; t < p->N; ++t) ++len[seg[t]];
  std::vector<int32_t> parent(S);
  for (int32_t v = 0; v < S; ++v) parent[v] = anc_ptr[v + 1] > anc_ptr[v] ? anc_idx[anc_ptr[v + 1] - 1] : -1;
  for (int32_t v = 0; v < S; ++v)
    if (len[v] > cap)
      return fail(TREE_ERR_UNSUPPORTED, "segment " + std::to_string(v) + " has " + std::to_string(len[v]) +
                                            " tokens, above the cap of " + std::to_string(cap));
  std::vector<std::vector<int32_t>> children(S);
  for (int32_t v = 0; v < S; ++v)
    if (parent[v] >= 0) children[parent[v]].push_back(v);  // ascending id
  // bottom-up: residual[v] = tokens of v's piece below and at v (uncut part)
  std::vector<int64_t> residual(S, 0);
  std::vector<char> is_root(S, 0);
  for (int32_t e = S - 1; e >= 0; --e) {  // reverse DFS order: children first
    const int32_t v = order[e];
    int64_t total = len[v];
    for (int32_t c : children[v]) total += residual[c];
    while (total > cap) {
      int32_t best = -1;
      for (int32_t c : children[v])
        if (!is_root[c] && (best < 0 || residual[c] > residual[best])) best = c;
      is_root[best] = 1;  // len[v] <= cap, so an uncut child remains while total > cap
      total -= residual[best];
    }
    residual[v] = total;
    if (parent[v] < 0) is_root[v] = 1;
  }
  // number the partitions by their roots in DFS order; run[] counts each
  // partition's DFS tokens so far (its DFS sequence is the global one restricted)
  std::vector<int64_t> run, upto(S, 0);
  int32_t n = 0;
  for (int32_t v : order) {
    if (is_root[v]) {
      tree_partition_t& q = parts[n];
      q.root = v;
      q.parent = parent[v] < 0 ? -1 : part_of[parent[v]];
      q.tokens = 0;
      q.pos_offset = pos[start[v]];
      q.past_len = q.parent < 0 ? 0 : parts[q.parent].past_len + upto[parent[v]];
      part_of[v] = n++;
      run.push_back(0);
    } else {
      part_of[v] = part_of[parent[v]];
    }
    run[part_of[v]] += len[v];
    upto[v] = run[part_of[v]];
    parts[part_of[v]].tokens += len[v];
  }
  std::vector<int64_t> chain(n, 0);
  int64_t peak = 0;
  for (int32_t i = 0; i < n; ++i) {  // parents have smaller numbers
    chain[i] = parts[i].tokens + (parts[i].parent >= 0 ? chain[parts[i].parent] : 0);
    peak = chain[i] > peak ? chain[i] : peak;
  }
  *num_parts = n;
  *peak_path_tokens = peak;
  return TREE_OK;
}

extern "C" const char* tree_last_error(void) { return g_last_error.c_str(); }
