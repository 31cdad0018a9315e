// Grouping of (leaf block, query) pairs for the block-major kernels.
//
// The prefill/training kernels gather the queries that use the same leaf key block into
// tiles so that block's keys are read once per tile ("Block Sparse Attention with
// Log-Linear Complexity", daily digest page, "Reference value of the work": Qtile).
// Here the pairs are counting-sorted into bins (head, query chunk, leaf): queries are cut
// into chunks of Nq consecutive tokens so that the blocks running at the same time touch
// one chunk's query rows (which then stay in L2), and every bin's list is cut into work
// items of at most `cap` pairs so no CTA gets a list thousands of tiles long (early leaves
// are visible to, and chosen by, far more queries than late ones).
#include "device.cuh"
#include "group.h"
#include "profile.h"

namespace pisa {

namespace {

// Pairs are binned per block of kGQ consecutive units (head * N + query): their bins lie in
// at most two consecutive (head, chunk) groups in every block but a rare one at a short last
// chunk, so a block counts them in a shared-memory histogram of 2 * n0 leaves and touches
// each global counter once per block instead of once per pair. A block whose range spans
// more groups (or any block when the histogram does not fit) falls back to global atomics.
constexpr int kGQ = 256;          // units per block
constexpr int kGThreads = 512;

struct BinRange {
  int64_t u0, e0, g0;   // first unit, its first pair, its (head, chunk) group
  int n;                // pairs in the block
  bool local;
};

__device__ __forceinline__ int64_t group_of(const GroupPlan& gp, int64_t unit) {
  return (unit / gp.N) * gp.nch + (unit % gp.N) / gp.Nq;
}

__device__ __forceinline__ BinRange bin_range(const GroupPlan& gp, bool local_ok) {
  const int64_t units = gp.total / gp.W;
  const int64_t u0 = blockIdx.x * static_cast<int64_t>(kGQ);
  const int64_t u1 = min(u0 + kGQ, units);
  BinRange r;
  r.u0 = u0;
  r.e0 = u0 * gp.W;
  r.n = static_cast<int>((u1 - u0) * gp.W);
  r.g0 = group_of(gp, u0);
  r.local = local_ok && group_of(gp, u1 - 1) - r.g0 <= 1;
  return r;
}

// The bin key of a selected leaf t (prev: the unit's previous slot, -1 at slot 0): t itself, or
// with pairs the pair index; -1 for no entry (none, out of range, or a pair's member that is
// not its first entry).
__device__ __forceinline__ int bin_key(const GroupPlan& gp, int t, int prev) {
  if (t < 0) return -1;
  if (gp.shift) {
    if (t & 1) {
      if (!gp.dedup || prev == t - 1) return -1;
    }
    t >>= 1;
  }
  return t < gp.n0 ? t : -1;
}
__device__ __forceinline__ int entry_key(const GroupPlan& gp, const int32_t* __restrict__ sel, int64_t e, int k) {
  const bool first = (gp.wlog >= 0 ? k & (gp.W - 1) : k % gp.W) == 0;   // slot 0 of its unit
  return bin_key(gp, sel[e], gp.dedup && !first ? sel[e - 1] : -1);
}

// Per unit of the block: its query i and its (head, chunk) group relative to r.g0, tabulated
// once so that a pair needs no division by N or Nq.
struct UnitTab {
  int i[kGQ], dg[kGQ];
};
__device__ __forceinline__ void fill_units(const GroupPlan& gp, const BinRange& r, UnitTab& tab) {
  for (int lu = threadIdx.x; lu < kGQ; lu += kGThreads) {
    const int64_t u = r.u0 + lu, h = u / gp.N;
    const int i = static_cast<int>(u - h * gp.N);
    tab.i[lu] = i;
    tab.dg[lu] = static_cast<int>(h * gp.nch + i / gp.Nq - r.g0);
  }
}

// Pair k of the block: its query i, slot and (head, chunk) group.
__device__ __forceinline__ void pair_at(const GroupPlan& gp, const BinRange& r, const UnitTab& tab, int k, int& i,
                                        int& slot, int64_t& g) {
  const int lu = gp.wlog >= 0 ? k >> gp.wlog : k / gp.W;
  slot = k - lu * gp.W;
  i = tab.i[lu];
  g = r.g0 + tab.dg[lu];
}

__global__ void __launch_bounds__(kGThreads)
gcount_kernel(GroupPlan gp, bool local_ok, const int32_t* __restrict__ sel, int32_t* __restrict__ counts) {
  extern __shared__ int32_t hist[];                 // [2 * n0]
  __shared__ UnitTab tab;
  const BinRange r = bin_range(gp, local_ok);
  fill_units(gp, r, tab);
  if (r.local)
    for (int k = threadIdx.x; k < 2 * gp.n0; k += kGThreads) hist[k] = 0;
  __syncthreads();
  for (int k = threadIdx.x; k < r.n; k += kGThreads) {
    const int t = entry_key(gp, sel, r.e0 + k, k);
    if (t < 0) continue;
    int i, slot;
    int64_t g;
    pair_at(gp, r, tab, k, i, slot, g);
    if (r.local) atomicAdd(&hist[(g - r.g0) * gp.n0 + t], 1);
    else atomicAdd(&counts[g * gp.n0 + t], 1);
  }
  if (!r.local) return;
  __syncthreads();
  for (int k = threadIdx.x; k < 2 * gp.n0; k += kGThreads) {
    const int c = hist[k];
    if (c) atomicAdd(&counts[r.g0 * gp.n0 + k], c);
  }
}

// An in-place exclusive scan and the work items in one 1024-thread block: off (n = gp.bins counts) becomes
// the exclusive scan with off[n] = the total, every bin's list is cut into items of at most
// gp.cap pairs, written in bin order to items[], and icount[n] receives the item count.
__global__ void __launch_bounds__(1024) gscan_items_kernel(GroupPlan gp, int32_t* off, int32_t* icount,
                                                           int4* __restrict__ items) {
  __shared__ int32_t warp_tot[2][32];
  const int64_t n = gp.bins;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t per = (n + 1023) / 1024;
  const int64_t s0 = min(tid * per, n), s1 = min(s0 + per, n);
  int32_t lp = 0, li = 0;                    // this thread's pairs and items
  for (int64_t k = s0; k < s1; ++k) {
    const int32_t c = off[k];
    lp += c;
    li += (c + gp.cap - 1) / gp.cap;
  }
  int32_t vp = lp, vi = li;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t yp = __shfl_up_sync(0xffffffffu, vp, o), yi = __shfl_up_sync(0xffffffffu, vi, o);
    if (lane >= o) { vp += yp; vi += yi; }
  }
  if (lane == 31) { warp_tot[0][w] = vp; warp_tot[1][w] = vi; }
  __syncthreads();
  if (w == 0) {
    int32_t tp = warp_tot[0][lane], ti = warp_tot[1][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t yp = __shfl_up_sync(0xffffffffu, tp, o), yi = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) { tp += yp; ti += yi; }
    }
    warp_tot[0][lane] = tp;
    warp_tot[1][lane] = ti;
  }
  __syncthreads();
  int32_t run = vp - lp + (w > 0 ? warp_tot[0][w - 1] : 0);
  int32_t irun = vi - li + (w > 0 ? warp_tot[1][w - 1] : 0);
  for (int64_t k = s0; k < s1; ++k) {
    const int32_t c = off[k];
    off[k] = run;
    for (int32_t q = 0; q < c; q += gp.cap)
      items[irun++] = make_int4(static_cast<int>(k), run + q, min(gp.cap, c - q), 0);
    run += c;
  }
  if (tid == 1023) {
    off[n] = run;
    icount[n] = irun;
  }
}

// Scatter: a local block ranks its pairs within each bin in shared memory, reserves each
// bin's range with one global atomic, then writes list[off + base + rank] = (i << 6) | slot.
__global__ void __launch_bounds__(kGThreads)
gscatter_kernel(GroupPlan gp, bool local_ok, const int32_t* __restrict__ sel, const int32_t* __restrict__ off,
                int32_t* __restrict__ cursor, int32_t* __restrict__ list) {
  extern __shared__ int32_t hist[];                 // [2 * n0] counts, then bases; ranks [kGQ * W]
  int32_t* rank = hist + 2 * gp.n0;
  __shared__ UnitTab tab;
  const BinRange r = bin_range(gp, local_ok);
  fill_units(gp, r, tab);
  if (r.local)
    for (int k = threadIdx.x; k < 2 * gp.n0; k += kGThreads) hist[k] = 0;
  __syncthreads();
  for (int k = threadIdx.x; k < r.n; k += kGThreads) {
    const int t = entry_key(gp, sel, r.e0 + k, k);
    if (t < 0) continue;
    int i, slot;
    int64_t g;
    pair_at(gp, r, tab, k, i, slot, g);
    if (r.local) {
      rank[k] = atomicAdd(&hist[(g - r.g0) * gp.n0 + t], 1);
    } else {
      const int64_t bin = g * gp.n0 + t;
      list[off[bin] + atomicAdd(&cursor[bin], 1)] = (i << 6) | slot;
    }
  }
  if (!r.local) return;
  __syncthreads();
  for (int k = threadIdx.x; k < 2 * gp.n0; k += kGThreads) {
    const int c = hist[k];
    if (c) {
      const int64_t bin = r.g0 * gp.n0 + k;
      hist[k] = off[bin] + atomicAdd(&cursor[bin], c);
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < r.n; k += kGThreads) {
    const int t = entry_key(gp, sel, r.e0 + k, k);
    if (t < 0) continue;
    int i, slot;
    int64_t g;
    pair_at(gp, r, tab, k, i, slot, g);
    list[hist[(g - r.g0) * gp.n0 + t] + rank[k]] = (i << 6) | slot;
  }
}

}  // namespace

GroupPlan make_group_plan(const Dims& s, int W, int64_t nq_target, int cap, int shift, int dedup) {
  GroupPlan gp{};
  gp.N = s.N;
  gp.shift = shift;
  gp.dedup = dedup;
  gp.n0 = (s.n0 + (1 << shift) - 1) >> shift;
  gp.W = W;
  gp.wlog = -1;
  for (int l = 0; l < 31; ++l)
    if (W == (1 << l)) gp.wlog = l;
  gp.cap = cap;
  int64_t nq = (nq_target / s.C) * s.C;
  if (nq < s.C) nq = s.C;
  if (nq > s.N) nq = s.N;
  gp.Nq = static_cast<int>(nq);
  gp.nch = static_cast<int>((s.N + nq - 1) / nq);
  gp.heads = static_cast<int64_t>(s.B) * s.Hkv;
  gp.bins = gp.heads * gp.nch * gp.n0;
  gp.total = gp.heads * s.N * W;
  gp.max_items = gp.total / cap + gp.bins + 1;
  return gp;
}

GroupWs group_ws(const GroupPlan& gp, size_t base) {
  GroupWs w{};
  size_t o = base;
  w.off = o;    o += align256((gp.bins + 1) * 4);
  w.cursor = o; o += align256((gp.bins + 1) * 4);
  w.icount = o; o += align256((gp.bins + 1) * 4);
  w.list = o;   o += align256(static_cast<size_t>(gp.total) * 4);
  w.items = o;  o += align256(static_cast<size_t>(gp.max_items) * 16);
  w.end = o;
  return w;
}

int launch_group_items(const GroupPlan& gp, const int32_t* sel, char* ws, const GroupWs& w,
                       cudaStream_t st) {
  int32_t* off = reinterpret_cast<int32_t*>(ws + w.off);
  int32_t* cursor = reinterpret_cast<int32_t*>(ws + w.cursor);
  int32_t* icount = reinterpret_cast<int32_t*>(ws + w.icount);
  int32_t* list = reinterpret_cast<int32_t*>(ws + w.list);
  int4* items = reinterpret_cast<int4*>(ws + w.items);
  cudaError_t e = cudaMemsetAsync(off, 0, sizeof(int32_t) * (gp.bins + 1), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(cursor, 0, sizeof(int32_t) * (gp.bins + 1), st);
  if (e != cudaSuccess) return e;
  // shared-memory binning when the histogram and the ranks fit (n0 up to ~20K leaves)
  const int64_t blocks = (gp.total / gp.W + kGQ - 1) / kGQ;
  const size_t hist_bytes = static_cast<size_t>(2) * gp.n0 * 4;
  const size_t rank_bytes = static_cast<size_t>(kGQ) * gp.W * 4;
  const bool local_ok = hist_bytes + rank_bytes <= 200 * 1024;
  const size_t sm_count = local_ok ? hist_bytes : 0, sm_scatter = local_ok ? hist_bytes + rank_bytes : 0;
  if (blocks > 0) {
    // above 48 KB per block (the dynamic part plus the kernels' static unit table) a launch
    // needs the opt-in; set on every call, since the attribute is per function and process
    const size_t dflt = 48 * 1024 - sizeof(UnitTab);
    if (sm_scatter > dflt) {
      e = cudaFuncSetAttribute(gscatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sm_scatter));
      if (e == cudaSuccess && sm_count > dflt)
        e = cudaFuncSetAttribute(gcount_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sm_count));
      if (e != cudaSuccess) return e;
    }
    {
      ProfScope ps(st, "group_count");
      gcount_kernel<<<static_cast<unsigned>(blocks), kGThreads, sm_count, st>>>(gp, local_ok, sel, off);
    }
    {
      ProfScope ps(st, "group_scan");
      gscan_items_kernel<<<1, 1024, 0, st>>>(gp, off, icount, items);
    }
    {
      ProfScope ps(st, "group_scatter");
      gscatter_kernel<<<static_cast<unsigned>(blocks), kGThreads, sm_scatter, st>>>(gp, local_ok, sel, off,
                                                                                     cursor, list);
    }
  } else {
    ProfScope ps(st, "group_scan");
    gscan_items_kernel<<<1, 1024, 0, st>>>(gp, off, icount, items);
  }
  return cudaGetLastError();
}

}  // namespace pisa
