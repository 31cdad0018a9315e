// Causal block-sparse attention over the selected leaf blocks.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference
// value of the work": attention runs only over the selected blocks and gradients pass
// only through that attention (the discrete selection takes none); the prefill kernel
// groups the queries that use the same leaf key block into tiles so the block's keys are
// read once per tile.
//
// Forward, block-major: the selected (leaf, query) pairs are grouped by (KV head, query
// chunk, leaf) and cut into work items; one CTA per item keeps the leaf block's K
// (row-major) and V (transposed) in shared memory and runs S = Q K^T and O = P V on MMAs
// for 16-row tiles of (query, head) rows. Each (row, block) yields a normalised partial
// output and its block LSE. Every query counts its finished blocks with one atomic; the
// warp that finishes a query's last block merges that query's <= K partials right away,
// while they are still in L2: lse = log sum_t exp(lse_t), o = sum_t exp(lse_t - lse) o_t,
// then discards the merged partials' L2 lines (they are dead) so they are never written
// back to HBM. Nothing waits on anything: the counter only decides who merges.
#include "device.cuh"
#include "group.h"
#include "profile.h"

namespace pisa {

namespace {

constexpr int kWarps = 4;

template <int D>
__device__ __forceinline__ void load_kv_tiles(const Dims& s, int b, int kv, int t,
                                              const __nv_bfloat16* K, const __nv_bfloat16* V,
                                              __nv_bfloat16* sK, __nv_bfloat16* sVt) {
  constexpr int KROW = D + 16, VROW = 64 + 8;
  for (int it = threadIdx.x; it < 64 * (D / 8); it += blockDim.x) {
    const int r = it / (D / 8), c = it % (D / 8);
    const int64_t j = static_cast<int64_t>(t) * 64 + r;
    uint4 kvv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (j < s.N) {
      const int64_t o = ((static_cast<int64_t>(b) * s.N + j) * s.Hkv + kv) * D + c * 8;
      kvv = ldg_u4(K + o);
      vv = ldg_u4(V + o);
    }
    *reinterpret_cast<uint4*>(&sK[r * KROW + c * 8]) = kvv;
    const __nv_bfloat16* ve = reinterpret_cast<const __nv_bfloat16*>(&vv);
#pragma unroll
    for (int e = 0; e < 8; ++e) sVt[(c * 8 + e) * VROW + r] = ve[e];
  }
}

__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Merge the nsel block partials of query i (all G heads of KV head kv) -- one warp.
template <int D, int G>
__device__ __forceinline__ void merge_query(const Dims& s, int b, int kv, int i, int nsel,
                                            __nv_bfloat16* part_o, const float* part_lse,
                                            __nv_bfloat16* O, float* lse_out, int lane) {
  constexpr int PER = D / 32;
  for (int h = 0; h < G; ++h) {
    const int64_t row = (static_cast<int64_t>(b) * s.N + i) * s.Hq + kv * G + h;
    const float* pl = part_lse + row * s.K;
    float m = neg_inf();
    for (int q = 0; q < nsel; ++q) m = fmaxf(m, __ldcg(pl + q));
    float den = 0.f, acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = 0.f;
    for (int q = 0; q < nsel; ++q) {
      const float w = m == neg_inf() ? 0.f : expf(__ldcg(pl + q) - m);
      den += w;
      const __nv_bfloat16* src = part_o + (row * s.K + q) * D + lane * PER;
      if (PER == 4) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(src));
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
        for (int u = 0; u < PER; ++u) acc[u] += w * __bfloat162float(e[u]);
      } else {
        const unsigned int v = __ldcg(reinterpret_cast<const unsigned int*>(src));
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
        for (int u = 0; u < PER; ++u) acc[u] += w * __bfloat162float(e[u]);
      }
    }
    const float r = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16* dst = O + row * D + lane * PER;
#pragma unroll
    for (int u = 0; u < PER; u += 2)
      *reinterpret_cast<uint32_t*>(dst + u) = pack_bf16(acc[u] * r, acc[u + 1] * r);
    if (lane == 0)
      lse_out[(static_cast<int64_t>(b) * s.Hq + kv * G + h) * s.N + i] = den > 0.f ? m + logf(den) : neg_inf();
    // the merged partials (whole 128-byte lines of this row only) are dead: drop them from L2
    __syncwarp();
    const int lines = nsel * D * 2 / 128;
    const char* base = reinterpret_cast<const char*>(part_o + row * s.K * D);
    if ((reinterpret_cast<uintptr_t>(base) & 127) == 0)
      for (int k = lane; k < lines; k += 32) discard_l2_line(base + k * 128);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
attn_fwd_kernel(Dims s, GroupPlan gp, const __nv_bfloat16* __restrict__ Q,
                const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                const int32_t* __restrict__ idx, const int32_t* __restrict__ list,
                const int4* __restrict__ items, const int32_t* __restrict__ n_items,
                __nv_bfloat16* part_o, float* part_lse, int32_t* __restrict__ counter,
                __nv_bfloat16* __restrict__ O, float* __restrict__ lse_out) {
  constexpr int KS = D / 16, KROW = D + 16, VROW = 64 + 8, QPT = 16 / G, ND = D / 8;
  __shared__ __align__(16) __nv_bfloat16 sK[64 * KROW];
  __shared__ __align__(16) __nv_bfloat16 sVt[D * VROW];
  if (static_cast<int>(blockIdx.x) >= *n_items) return;
  const int4 it = items[blockIdx.x];
  const int64_t bin = it.x;
  const int beg = it.y, n_ent = it.z;
  const int t = gp.leaf_of(bin);
  const int64_t head = gp.head_of(bin);
  const int b = static_cast<int>(head / s.Hkv), kv = static_cast<int>(head % s.Hkv);
  load_kv_tiles<D>(s, b, kv, t, K, V, sK, sVt);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
  const int n_mt = (n_ent + QPT - 1) / QPT;
  const int kbase = t * 64;
  const int Ksel = s.K;
  for (int mt = warp; mt < n_mt; mt += kWarps) {
    const int e0 = mt * QPT + g / G, h0 = g % G;
    const int e1 = mt * QPT + (g + 8) / G, h1 = (g + 8) % G;
    const bool ok0 = e0 < n_ent, ok1 = e1 < n_ent;
    const int pk0 = ok0 ? list[beg + e0] : 0, pk1 = ok1 ? list[beg + e1] : 0;
    const int i0 = pk0 >> 6, i1 = pk1 >> 6;
    const int64_t row0 = (static_cast<int64_t>(b) * s.N + i0) * s.Hq + kv * G + h0;
    const int64_t row1 = (static_cast<int64_t>(b) * s.N + i1) * s.Hq + kv * G + h1;
    const __nv_bfloat16* q0 = Q + row0 * D;
    const __nv_bfloat16* q1 = Q + row1 * D;
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint2 x0 = ok0 ? ldg_u2(q0 + 16 * ks + 4 * p) : make_uint2(0, 0);
      const uint2 x1 = ok1 ? ldg_u2(q1 + 16 * ks + 4 * p) : make_uint2(0, 0);
      const uint32_t a[4] = {x0.x, x1.x, x0.y, x1.y};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const uint2 bb = *reinterpret_cast<const uint2*>(&sK[(nt * 8 + g) * KROW + 16 * ks + 4 * p]);
        mma_bf16(sacc[nt], a, bb.x, bb.y);
      }
    }
    float m0 = neg_inf(), m1 = neg_inf();
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kbase + nt * 8 + 2 * p + e;
        sacc[nt][e] = key <= i0 ? s.scale * sacc[nt][e] : neg_inf();
        sacc[nt][2 + e] = key <= i1 ? s.scale * sacc[nt][2 + e] : neg_inf();
        m0 = fmaxf(m0, sacc[nt][e]);
        m1 = fmaxf(m1, sacc[nt][2 + e]);
      }
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    const float ms0 = m0 == neg_inf() ? 0.f : m0, ms1 = m1 == neg_inf() ? 0.f : m1;
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sacc[nt][e] = expf(sacc[nt][e] - ms0);
        sacc[nt][2 + e] = expf(sacc[nt][2 + e] - ms1);
        l0 += sacc[nt][e];
        l1 += sacc[nt][2 + e];
      }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // O = P V: P (bf16) in the A layout straight from the S accumulators
    float oacc[ND][4];
#pragma unroll
    for (int nd = 0; nd < ND; ++nd)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[nd][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t a[4] = {pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]),
                             pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]),
                             pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]),
                             pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3])};
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const __nv_bfloat16* vr = &sVt[(nd * 8 + g) * VROW + 16 * kk + 2 * p];
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(vr);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(vr + 8);
        mma_bf16(oacc[nd], a, b0, b1);
      }
    }
    // a block with no key visible to the row (not a valid selection) contributes nothing
    const float r0 = l0 > 0.f ? 1.f / l0 : 0.f, r1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const int slot0 = pk0 & 63, slot1 = pk1 & 63;
    __nv_bfloat16* po0 = part_o + (row0 * Ksel + slot0) * D;
    __nv_bfloat16* po1 = part_o + (row1 * Ksel + slot1) * D;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      if (ok0)
        *reinterpret_cast<uint32_t*>(po0 + nd * 8 + 2 * p) = pack_bf16(oacc[nd][0] * r0, oacc[nd][1] * r0);
      if (ok1)
        *reinterpret_cast<uint32_t*>(po1 + nd * 8 + 2 * p) = pack_bf16(oacc[nd][2] * r1, oacc[nd][3] * r1);
    }
    if (p == 0) {
      if (ok0) part_lse[row0 * Ksel + slot0] = l0 > 0.f ? ms0 + logf(l0) : neg_inf();
      if (ok1) part_lse[row1 * Ksel + slot1] = l1 > 0.f ? ms1 + logf(l1) : neg_inf();
    }
    // arrival: lane e < QPT reports entry mt*QPT + e (all its G rows are in this tile)
    __threadfence();
    __syncwarp();
    int qi = -1, nsel = 0, last = 0;
    if (lane < QPT) {
      const int e = mt * QPT + lane;
      if (e < n_ent) {
        qi = list[beg + e] >> 6;
        const int64_t unit = head * s.N + qi;
        const int32_t* id = idx + unit * Ksel;
        for (int q = 0; q < Ksel; ++q) nsel += id[q] >= 0 ? 1 : 0;
        last = atomicAdd(&counter[unit], 1) == nsel - 1;
      }
    }
    unsigned lm = __ballot_sync(0xffffffffu, last);
    if (lm) __threadfence();
    while (lm) {
      const int src = __ffs(lm) - 1;
      lm &= lm - 1;
      const int i = __shfl_sync(0xffffffffu, qi, src);
      const int ns = __shfl_sync(0xffffffffu, nsel, src);
      merge_query<D, G>(s, b, kv, i, ns, part_o, part_lse, O, lse_out, lane);
    }
  }
}

template <int D, int G>
void fwd_launch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                __nv_bfloat16* po, float* pl, int32_t* counter, void* O, float* lse, cudaStream_t st) {
  ProfScope ps(st, "attn_fwd");
  attn_fwd_kernel<D, G><<<static_cast<unsigned>(gp.max_items), kWarps * 32, 0, st>>>(
      s, gp, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
      static_cast<const __nv_bfloat16*>(V), idx, list, items, n_items, po, pl, counter,
      static_cast<__nv_bfloat16*>(O), lse);
}

template <int D>
void fwd_dispatch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                  const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                  __nv_bfloat16* po, float* pl, int32_t* counter, void* O, float* lse, cudaStream_t st) {
  switch (s.G) {
    case 1: fwd_launch<D, 1>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, counter, O, lse, st); break;
    case 2: fwd_launch<D, 2>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, counter, O, lse, st); break;
    case 4: fwd_launch<D, 4>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, counter, O, lse, st); break;
    default: fwd_launch<D, 8>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, counter, O, lse, st); break;
  }
}

// Query chunk so that one chunk's block partials take about 64 MiB (they live in L2 until
// merged); about 1024 (query, head) rows per work item.
GroupPlan fwd_plan(const Dims& s) {
  const int64_t per_query = static_cast<int64_t>(s.G) * s.K * s.d * 2;
  return make_group_plan(s, s.K, (int64_t(64) << 20) / per_query, 1024 / s.G);
}

}  // namespace

AttnFwdWs attn_fwd_ws(const Dims& s) {
  AttnFwdWs w{};
  const GroupPlan gp = fwd_plan(s);
  const size_t rows = static_cast<size_t>(s.B) * s.N * s.Hq;
  const GroupWs g = group_ws(gp, 0);
  size_t o = g.end;
  w.part_o = o;   o += align256(rows * s.K * s.d * 2);
  w.part_lse = o; o += align256(rows * s.K * 4);
  w.counter = o;  o += align256(static_cast<size_t>(s.B) * s.Hkv * s.N * 4);
  w.total = o;
  return w;
}

int launch_attn_fwd(const Dims& s, const void* Q, const void* K, const void* V,
                    const int32_t* idx, void* O, float* lse, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnFwdWs w = attn_fwd_ws(s);
  const GroupPlan gp = fwd_plan(s);
  const GroupWs g = group_ws(gp, 0);
  int err = launch_group_items(gp, idx, ws, g, st);
  if (err) return err;
  int32_t* counter = reinterpret_cast<int32_t*>(ws + w.counter);
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(int32_t) * s.B * s.Hkv * s.N, st);
  if (e != cudaSuccess) return e;
  const int32_t* list = reinterpret_cast<const int32_t*>(ws + g.list);
  const int4* items = reinterpret_cast<const int4*>(ws + g.items);
  const int32_t* n_items = reinterpret_cast<const int32_t*>(ws + g.icount) + gp.bins;
  __nv_bfloat16* po = reinterpret_cast<__nv_bfloat16*>(ws + w.part_o);
  float* pl = reinterpret_cast<float*>(ws + w.part_lse);
  if (s.d == 128) fwd_dispatch<128>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, counter, O, lse, st);
  else fwd_dispatch<64>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, counter, O, lse, st);
  return cudaGetLastError();
}

}  // namespace pisa
