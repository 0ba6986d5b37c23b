// Work list of a persistent launch: each CTA of the grid runs a list of work
// items one after the other.  An item is a unit of one (batch, head): a pair of
// query tiles in the forward, a key tile in the backward; its id is
// bh * units + unit.
//
// With `table`, CTA c runs list[start[c] .. start[c+1]) in that order.  The
// host builds the table once per problem shape: heads are taken in groups
// whose operands fit in L2 together (so the CTAs working at one time share
// them), and within a group the items go longest first, each to the CTA with
// the least work so far.  Under a causal mask the units of a head differ in
// work ("Question bank -- Flash attention and efficient attention", the causal
// block-skipping item), which is what the balancing is for.
//
// Without a table (more items than fit in the kernel's parameters), CTA c runs
// items c, c + G, c + 2G, ... of the head-major order, the heaviest unit of a
// head first.
#pragma once
#include <cstdint>

namespace fa {

constexpr int WL_MAX_CTAS = 160;
constexpr int WL_MAX_ITEMS = 6144;

struct WorkList {
  int n_items;
  int table;
  uint16_t start[WL_MAX_CTAS + 1];
  uint32_t list[WL_MAX_ITEMS];
};

// Number of items of this CTA.
__device__ __forceinline__ int wl_count(const WorkList& w) {
  const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
  if (w.table) return w.start[c + 1] - w.start[c];
  return c < w.n_items ? (w.n_items - 1 - c) / G + 1 : 0;
}

// Item k of this CTA as (bh, unit).  Without a table the heaviest unit of a
// head is unit units - 1 (heaviest_last) or unit 0.
__device__ __forceinline__ void wl_item(const WorkList& w, int k, int units, bool heaviest_last, int& bh,
                                        int& unit) {
  const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
  if (w.table) {
    const int id = static_cast<int>(w.list[w.start[c] + k]);
    bh = id / units;
    unit = id % units;
  } else {
    const int i = c + k * G;
    bh = i / units;
    unit = heaviest_last ? units - 1 - i % units : i % units;
  }
}

}  // namespace fa
