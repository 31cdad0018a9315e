// Work-item walk shared by the persistent block-major kernels: CTA c takes the items c,
// c + gridDim.x, ... of a grouping (group.h) and cuts each into tiles of `ept` list entries
// (a tile row is one (query, head) of an entry).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "group.h"

namespace pisa {

struct ItemView {
  int beg, n_ent, kbase, b, kv;
  int64_t head;
};

struct ItemSource {
  GroupPlan gp;
  const int4* items;
  const int32_t* list;
  int Hkv;
};

__device__ __forceinline__ ItemView view_item(const ItemSource& src, int it) {
  const int4 item = src.items[it];
  ItemView v;
  v.beg = item.y;
  v.n_ent = item.z;
  v.kbase = src.gp.leaf_of(item.x) * 64;
  v.head = src.gp.head_of(item.x);
  v.b = static_cast<int>(v.head / src.Hkv);
  v.kv = static_cast<int>(v.head % src.Hkv);
  return v;
}

struct TileCursor {
  int it, j, n_tiles;
  ItemView v;
};

__device__ __forceinline__ bool first_tile(const ItemSource& src, int n_items, int ept, TileCursor& c) {
  c.it = blockIdx.x;
  c.j = 0;
  if (c.it >= n_items) return false;
  c.v = view_item(src, c.it);
  c.n_tiles = (c.v.n_ent + ept - 1) / ept;
  return true;
}

__device__ __forceinline__ bool next_tile(const ItemSource& src, int n_items, int ept, TileCursor& c) {
  if (++c.j < c.n_tiles) return true;
  c.it += gridDim.x;
  c.j = 0;
  if (c.it >= n_items) return false;
  c.v = view_item(src, c.it);
  c.n_tiles = (c.v.n_ent + ept - 1) / ept;
  return true;
}

// List entry (query << 6 | slot) of tile row r, -1 past the end of the item.
__device__ __forceinline__ int row_entry(const ItemSource& src, const TileCursor& c, int ept, int G, int r) {
  const int e = c.j * ept + r / G;
  return e < c.v.n_ent ? src.list[c.v.beg + e] : -1;
}

}  // namespace pisa
