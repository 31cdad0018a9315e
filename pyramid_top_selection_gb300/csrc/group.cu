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

__global__ void gcount_kernel(GroupPlan gp, const int32_t* __restrict__ sel, int32_t* __restrict__ counts) {
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < gp.total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = sel[e];
    if (t >= 0) {
      const int64_t unit = e / gp.W;
      const int i = static_cast<int>(unit % gp.N);
      atomicAdd(&counts[gp.bin(unit / gp.N, i, t)], 1);
    }
  }
}

// In-place exclusive scan of n counts (counts[n] receives the total), one 1024-thread block.
__global__ void __launch_bounds__(1024) gscan_kernel(int32_t* counts, int64_t n) {
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x;
  const int64_t per = (n + 1023) / 1024;
  const int64_t s0 = min(tid * per, n), s1 = min(s0 + per, n);
  int32_t local = 0;
  for (int64_t k = s0; k < s1; ++k) local += counts[k];
  const int lane = tid & 31, w = tid >> 5;
  int32_t v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) warp_tot[w] = v;
  __syncthreads();
  if (w == 0) {
    int32_t t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int32_t run = v - local + (w > 0 ? warp_tot[w - 1] : 0);
  for (int64_t k = s0; k < s1; ++k) {
    const int32_t c = counts[k];
    counts[k] = run;
    run += c;
  }
  if (tid == 1023) counts[n] = run;
}

__global__ void gscatter_kernel(GroupPlan gp, const int32_t* __restrict__ sel, const int32_t* __restrict__ off,
                                int32_t* __restrict__ cursor, int32_t* __restrict__ list) {
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < gp.total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = sel[e];
    if (t >= 0) {
      const int64_t unit = e / gp.W;
      const int slot = static_cast<int>(e - unit * gp.W);
      const int i = static_cast<int>(unit % gp.N);
      const int64_t bin = gp.bin(unit / gp.N, i, t);
      list[off[bin] + atomicAdd(&cursor[bin], 1)] = (i << 6) | slot;
    }
  }
}

__global__ void icount_kernel(GroupPlan gp, const int32_t* __restrict__ off, int32_t* __restrict__ icount) {
  for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < gp.bins;
       b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int len = off[b + 1] - off[b];
    icount[b] = (len + gp.cap - 1) / gp.cap;
  }
}

__global__ void ifill_kernel(GroupPlan gp, const int32_t* __restrict__ off, const int32_t* __restrict__ ioff,
                             int4* __restrict__ items) {
  for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < gp.bins;
       b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int beg = off[b], len = off[b + 1] - beg;
    int k = 0;
    for (int s = 0; s < len; s += gp.cap, ++k)
      items[ioff[b] + k] = make_int4(static_cast<int>(b), beg + s, min(gp.cap, len - s), 0);
  }
}

inline int grid_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  return static_cast<int>(b < 1 ? 1 : (b > 152 * 32 ? 152 * 32 : b));
}

}  // namespace

GroupPlan make_group_plan(const Dims& s, int W, int64_t nq_target, int cap) {
  GroupPlan gp{};
  gp.N = s.N;
  gp.n0 = s.n0;
  gp.W = W;
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
  {
    ProfScope ps(st, "group_count");
    gcount_kernel<<<grid_for(gp.total, 256), 256, 0, st>>>(gp, sel, off);
  }
  {
    ProfScope ps(st, "group_scan");
    gscan_kernel<<<1, 1024, 0, st>>>(off, gp.bins);
  }
  {
    ProfScope ps(st, "group_scatter");
    gscatter_kernel<<<grid_for(gp.total, 256), 256, 0, st>>>(gp, sel, off, cursor, list);
  }
  {
    ProfScope ps(st, "group_items");
    icount_kernel<<<grid_for(gp.bins, 256), 256, 0, st>>>(gp, off, icount);
    gscan_kernel<<<1, 1024, 0, st>>>(icount, gp.bins);
    ifill_kernel<<<grid_for(gp.bins, 256), 256, 0, st>>>(gp, off, icount, items);
  }
  return cudaGetLastError();
}

}  // namespace pisa
