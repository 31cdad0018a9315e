// Work-item walk shared by the persistent block-major kernels: each CTA takes items of a
// grouping (group.h) in a dynamic order and cuts each into tiles of `ept` list entries (a
// tile row is one (query, head) of an entry).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "group.h"

namespace pisa {

// One work item: its list entries [beg, beg + n_ent), its leaf's first key, and its KV head
// (batch b, head kv; head = b * Hkv + kv). n_ent = -1 marks the end of a sequence.
struct __align__(16) ItemView {
  int beg, n_ent, kbase, b, kv, pad;
  int64_t head;
};

struct ItemSource {
  GroupPlan gp;
  const int4* items;
  const int32_t* list;
  int Hkv;
};

// The view of an item record {bin, first list entry, entries, -}.
__device__ __forceinline__ ItemView view_of(const ItemSource& src, const int4 item) {
  ItemView v;
  v.beg = item.y;
  v.n_ent = item.z;
  v.kbase = src.gp.leaf_of(item.x) * (64 << src.gp.shift);
  v.head = src.gp.head_of(item.x);
  v.b = static_cast<int>(v.head / src.Hkv);
  v.kv = static_cast<int>(v.head % src.Hkv);
  v.pad = 0;
  return v;
}

}  // namespace pisa

// ---------------------------------------------------------------------------------------
// Dynamic item order for the persistent kernels. One scheduler thread per CTA takes items
// from a global counter (atomicAdd: a CTA that finishes early takes more, and all CTAs walk
// the grouping roughly in its order, so the Q rows of a query chunk stay in L2), reads their
// records and publishes their views through a ring in shared memory (n_ent = -1 ends the
// sequence), so that no role waits on a global load or does index arithmetic at an item
// boundary. Each consumer warp reads every position in order and frees it after its last
// look; the scheduler refills a slot once every consumer warp has freed it (the ring is
// deeper than the spread between the CTA's roles). One lead warp (the first producer warp,
// which runs ahead of the other roles) also marks each position as demanded when it reaches
// it, and the scheduler publishes position k once k - kItemAhead is demanded: a CTA holds few
// items that another CTA could have run, and the next record is fetched as soon as one is
// published, so its latency passes while the consumers work. The scheduler sleeps in
// mbarrier.try_wait (no polling: a spinning warp takes issue slots from its SM partition).
// Every wait is bounded (the launch's wait limit, one second unless the host set another) and a
// wait that gives up sets the CTA's abort flag.
// ---------------------------------------------------------------------------------------
namespace pisa {

constexpr int kItemRing = 16;
constexpr int kItemAhead = 3;

struct ItemQueue {
  ItemView view[kItemRing];
  uint64_t full[kItemRing], empty[kItemRing], demand[kItemRing];
  uint64_t limit_ns;   // bound of every wait on the queue
};

__device__ __forceinline__ uint32_t queue_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One thread, before the CTA's first barrier: full and demand slots take one arrival, empty
// slots one per consumer warp.
__device__ __forceinline__ void queue_init(ItemQueue& q, int consumer_warps, uint64_t limit_ns) {
  q.limit_ns = limit_ns;
  for (int k = 0; k < kItemRing; ++k) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(queue_addr(&q.full[k])), "r"(1));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(queue_addr(&q.empty[k])), "r"(consumer_warps));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(queue_addr(&q.demand[k])), "r"(1));
  }
}

__device__ __forceinline__ uint64_t queue_clock() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with the given parity; false (and the abort flag set) after
// limit_ns nanoseconds, or at once when the CTA has aborted.
__device__ __forceinline__ bool queue_wait(const uint64_t* bar, uint32_t parity, int* abort_flag,
                                           uint64_t limit_ns) {
  const uint32_t a = queue_addr(bar);
  uint64_t t0 = 0;
  for (int it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
    if (it == 0) t0 = queue_clock();
    else if ((it & 63) == 0 && queue_clock() - t0 > limit_ns) break;
  }
  atomicOr(abort_flag, 1);
  return false;
}

// Scheduler thread: publishes the views of the items it takes until the counter passes
// n_items (or the CTA aborts).
__device__ __forceinline__ void queue_fill(ItemQueue& q, const ItemSource& src, int32_t* counter, int n_items,
                                           int* abort_flag) {
  auto fetch = [&]() {
    const int item = atomicAdd(counter, 1);
    return item < n_items ? src.items[item] : make_int4(-1, 0, 0, 0);
  };
  int4 rec = fetch();
  for (int k = 0;; ++k) {
    const int sl = k % kItemRing;
    if (!queue_wait(&q.empty[sl], ((k / kItemRing) & 1) ^ 1, abort_flag, q.limit_ns)) return;
    const int kd = k - kItemAhead;
    if (kd >= 0 && !queue_wait(&q.demand[kd % kItemRing], (kd / kItemRing) & 1, abort_flag, q.limit_ns)) return;
    q.view[sl] = rec.x >= 0 ? view_of(src, rec) : ItemView{0, -1, 0, 0, 0, 0, 0};
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(queue_addr(&q.full[sl])) : "memory");
    if (rec.x < 0) return;
    rec = fetch();
  }
}

// The item at position k (n_ent = -1 past the end or when the CTA gave up). Any number of
// lanes may call it; they all see the same value.
__device__ __forceinline__ ItemView queue_peek(ItemQueue& q, int k, int* abort_flag) {
  const int sl = k % kItemRing;
  if (!queue_wait(&q.full[sl], (k / kItemRing) & 1, abort_flag, q.limit_ns)) return ItemView{0, -1, 0, 0, 0, 0, 0};
  return q.view[sl];
}

__device__ __forceinline__ void queue_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(queue_addr(bar)) : "memory");
}

// A position in the CTA's dynamic tile sequence: tile j of the item at queue position k.
// The cursor functions are called by whole warps. Within a warp each position is loaded once
// by the cursor that looks at it last (`release`), which then frees it; the lead warp's
// releasing cursor (`lead`) also marks it demanded. `lanes`: the calling lanes (a whole warp,
// or the one lane of a single-thread role).
struct DynCursor {
  int k, j, n_tiles;
  ItemView v;
};

__device__ __forceinline__ bool dyn_load(ItemQueue& q, int ept, int* abort_flag, DynCursor& c, bool release,
                                         bool lead, unsigned lanes) {
  c.j = 0;
  c.v = queue_peek(q, c.k, abort_flag);
  if (release) {
    __syncwarp(lanes);
    if ((threadIdx.x & 31) == __ffs(lanes) - 1) {
      queue_arrive(&q.empty[c.k % kItemRing]);
      if (lead) queue_arrive(&q.demand[c.k % kItemRing]);
    }
  }
  if (c.v.n_ent < 0) return false;
  c.n_tiles = (c.v.n_ent + ept - 1) / ept;
  return true;
}

__device__ __forceinline__ bool dyn_first(ItemQueue& q, int ept, int* abort_flag, DynCursor& c, bool release,
                                          bool lead = false, unsigned lanes = 0xffffffffu) {
  c.k = 0;
  return dyn_load(q, ept, abort_flag, c, release, lead, lanes);
}

__device__ __forceinline__ bool dyn_next(ItemQueue& q, int ept, int* abort_flag, DynCursor& c, bool release,
                                         bool lead = false, unsigned lanes = 0xffffffffu) {
  if (++c.j < c.n_tiles) return true;
  ++c.k;
  return dyn_load(q, ept, abort_flag, c, release, lead, lanes);
}

// One lane of a single-thread role: the item at position k, freed at once (its only look).
__device__ __forceinline__ ItemView queue_take(ItemQueue& q, int k, int* abort_flag) {
  const ItemView v = queue_peek(q, k, abort_flag);
  queue_arrive(&q.empty[k % kItemRing]);
  return v;
}

__device__ __forceinline__ int row_entry(const ItemSource& src, const DynCursor& c, int ept, int G, int r) {
  const int e = c.j * ept + r / G;
  return e < c.v.n_ent ? src.list[c.v.beg + e] : -1;
}

}  // namespace pisa
