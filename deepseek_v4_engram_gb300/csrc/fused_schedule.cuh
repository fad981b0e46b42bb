// Order of the work items of the fused projection + gate kernel.
//
// A work item is one 256-token tile times one column tile of kv: a key tile (256 key columns of
// one stream) or a value tile (256 value columns, shared by every stream). A value tile of a token
// tile needs that tile's gates, which exist only once all of its key tiles are done, so every
// value item is placed after all the key items of its token tile. Token tiles are taken in groups
// of `group`; within a group the items go column by column (the token tiles of the group in turn),
// so the few pairs working on one column at a time share its wkv tile in L2. The value items of
// group g - 1 are spread evenly over the key items of group g from `lag` items in (with lag at
// least the group's key items, they simply follow them), so that the HBM traffic of the value
// epilogues (x of every stream in, out of every stream written) overlaps the compute of key tiles
// instead of piling up at the end. The value items of the last group come last.
//
// Pairs take items in this order from a global counter. Since every value item comes after the key
// items it waits for, and each pair finishes its items in the order it took them, the pair holding
// the smallest-index waiting value item can always be served: no wait cycle can form.
#pragma once

#include <cstdint>

namespace engram {

struct FusedSchedule {
  int32_t m_tiles;   // 256-token tiles
  int32_t group;     // token tiles per group
  int32_t groups;    // ceil(m_tiles / group)
  int32_t nk_all;    // key tiles per token tile: hc * dim / 256
  int32_t nv_all;    // value tiles per token tile: dim / 256
  int32_t lag;       // key items of a group before the previous group's value items begin
  int64_t items;     // m_tiles * (nk_all + nv_all)
};

struct FusedItem {
  int32_t value;     // 0: key tile, 1: value tile
  int32_t mt;        // token tile
  int32_t col;       // key tile in [0, nk_all) (stream = col / (dim / 256)) or value tile
};

inline FusedSchedule make_fused_schedule(int64_t m_tiles, int32_t nk_all, int32_t nv_all,
                                         int32_t pairs) {
  FusedSchedule s{};
  s.m_tiles = static_cast<int32_t>(m_tiles);
  s.nk_all = nk_all;
  s.nv_all = nv_all;
  // A group's key items span about eight waves of the resident pairs, and the previous group's
  // value items follow them: a pair holds up to about three items (being loaded, multiplied and
  // drained), so value items placed much earlier would wait for gates; measured on 4096 tokens,
  // shorter groups or value items spread among the key items were slower.
  int64_t g = (8 * int64_t(pairs) + nk_all - 1) / nk_all;
  if (g < 1) g = 1;
  if (g > m_tiles) g = m_tiles;
  s.group = static_cast<int32_t>(g);
  s.groups = static_cast<int32_t>((m_tiles + g - 1) / g);
  s.lag = static_cast<int32_t>(g * nk_all);
  s.items = m_tiles * int64_t(nk_all + nv_all);
  return s;
}

__host__ __device__ inline int64_t fused_group_tiles(const FusedSchedule& s, int64_t g) {
  return g == s.groups - 1 ? s.m_tiles - int64_t(s.groups - 1) * s.group : s.group;
}

// i-th item (0 <= i < s.items) in the order above.
__host__ __device__ inline FusedItem fused_item_at(const FusedSchedule& s, int64_t i) {
  const int64_t G = s.group;
  auto key = [&](int64_t g, int64_t ki) {
    const int64_t n = fused_group_tiles(s, g);
    return FusedItem{0, static_cast<int32_t>(g * G + ki % n), static_cast<int32_t>(ki / n)};
  };
  auto value = [&](int64_t g, int64_t vi) {
    const int64_t n = fused_group_tiles(s, g);
    return FusedItem{1, static_cast<int32_t>(g * G + vi % n), static_cast<int32_t>(vi / n)};
  };
  const int64_t k0 = int64_t(s.nk_all) * fused_group_tiles(s, 0);
  if (i < k0) return key(0, i);
  i -= k0;
  if (s.groups == 1) return value(0, i);
  // segments g = 1 .. groups - 1: key items of group g with the value items of group g - 1
  // (a full group); all but the last have the same length
  const int64_t seg = int64_t(s.nk_all + s.nv_all) * G;
  const int64_t n_full = s.groups - 2;
  int64_t g;
  if (i < n_full * seg) {
    g = 1 + i / seg;
    i -= (g - 1) * seg;
  } else {
    i -= n_full * seg;
    g = s.groups - 1;
    const int64_t last = int64_t(s.nk_all) * fused_group_tiles(s, g) + int64_t(s.nv_all) * G;
    if (i >= last) return value(g, i - last);   // the last group's value items
  }
  const int64_t K = int64_t(s.nk_all) * fused_group_tiles(s, g);
  const int64_t V = int64_t(s.nv_all) * G;
  const int64_t lead = s.lag < K ? s.lag : K;
  if (i < lead) return key(g, i);
  const int64_t r = i - lead, total = K - lead + V;
  const int64_t cv = (r + 1) * V / total;   // value items among merged positions 0 .. r
  if (cv > r * V / total) return value(g - 1, cv - 1);
  return key(g, lead + r - cv);
}

}  // namespace engram
