// Grouping plan shared by the grouping kernels and the block-major kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "internal.h"

namespace pisa {

size_t align256(size_t x);

// Bins are (head = b*Hkv + kv, query chunk, leaf); a work item is {bin, list start, count}.
// With shift = 1 the bins are pairs of sibling leaves (2m, 2m + 1): only the even leaf of a pair
// is an entry (its odd sibling, when it is a candidate too, sits at the next slot), n0 counts
// the pairs, and an item's keys start at leaf 2m.
// With dedup = 1 (selections, whose slots need not hold both siblings) either member of a pair
// is an entry, the odd one only when its even sibling is not in the previous slot, so a row
// appears once per pair with the slot of its first selected member.
struct GroupPlan {
  int N, n0, W, cap, Nq, nch, shift, dedup;
  int wlog;   // log2(W) when W is a power of two, else -1
  int64_t heads, bins, total, max_items;
  __host__ __device__ int64_t bin(int64_t head, int i, int t) const {
    return (head * nch + i / Nq) * n0 + t;
  }
  __host__ __device__ int leaf_of(int64_t b) const { return static_cast<int>(b % n0); }
  __host__ __device__ int64_t head_of(int64_t b) const { return b / (static_cast<int64_t>(nch) * n0); }
};

// Byte offsets of the grouping buffers inside a workspace, starting at `base`.
struct GroupWs {
  size_t off, cursor, icount, list, items, end;
};

// Nq = the multiple of C nearest below `nq_target` (at least C, at most N).
GroupPlan make_group_plan(const Dims& s, int W, int64_t nq_target, int cap, int shift = 0, int dedup = 0);
GroupWs group_ws(const GroupPlan& gp, size_t base);
// Fills off/list/items of `w` from the selection-like array sel [heads, N, W] (-1 = none).
// The item count is icount[bins] on the device; at most gp.max_items.
int launch_group_items(const GroupPlan& gp, const int32_t* sel, char* ws, const GroupWs& w,
                       cudaStream_t st);

}  // namespace pisa
