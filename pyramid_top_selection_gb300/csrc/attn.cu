// Causal block-sparse attention over the selected leaf blocks.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference
// value of the work": attention runs only over the selected blocks and gradients pass
// only through that attention (the discrete selection takes none); the prefill kernel
// groups the queries that use the same leaf key block into tiles so the block's keys are
// read once per tile.
//
// Forward, block-major: the selected (leaf, query) pairs are grouped by leaf; one CTA per
// leaf block keeps the block's K (row-major) and V (transposed) in shared memory and runs
// S = Q K^T and O = P V on MMAs for 16-row tiles of (query, head) rows. Each (row, block)
// yields a normalised partial output and its block LSE; a combine kernel merges the
// <= K partials of every row: lse = log sum_t exp(lse_t), o = sum_t exp(lse_t - lse) o_t.
#include "device.cuh"
#include "profile.h"

namespace pisa {

int launch_group(const Dims& s, const int32_t* cand, int W, int32_t* counts, int32_t* cursor,
                 int32_t* list, cudaStream_t st);
size_t align256(size_t x);

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

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
attn_fwd_partial_kernel(Dims s, const __nv_bfloat16* __restrict__ Q,
                        const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                        const int32_t* __restrict__ off, const int32_t* __restrict__ list,
                        __nv_bfloat16* __restrict__ part_o, float* __restrict__ part_lse) {
  constexpr int KS = D / 16, KROW = D + 16, VROW = 64 + 8, QPT = 16 / G, ND = D / 8;
  __shared__ __align__(16) __nv_bfloat16 sK[64 * KROW];
  __shared__ __align__(16) __nv_bfloat16 sVt[D * VROW];
  const int t = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
  const int64_t head = static_cast<int64_t>(b) * s.Hkv + kv;
  const int64_t bin = head * s.n0 + t;
  const int beg = off[bin], end = off[bin + 1];
  if (beg == end) return;
  load_kv_tiles<D>(s, b, kv, t, K, V, sK, sVt);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
  const int n_ent = end - beg;
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
    const float r0 = 1.f / l0, r1 = 1.f / l1;
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
      if (ok0) part_lse[row0 * Ksel + slot0] = ms0 + logf(l0);
      if (ok1) part_lse[row1 * Ksel + slot1] = ms1 + logf(l1);
    }
  }
}

// One warp per (b, query, head) row: merges the row's <= K block partials.
template <int D>
__global__ void __launch_bounds__(256)
attn_combine_kernel(Dims s, const int32_t* __restrict__ idx, const __nv_bfloat16* __restrict__ part_o,
                    const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ O,
                    float* __restrict__ lse_out) {
  constexpr int PER = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x * 8LL + warp;     // (b*N + i)*Hq + h
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  if (row >= rows) return;
  const int h = static_cast<int>(row % s.Hq);
  const int64_t bi = row / s.Hq;
  const int i = static_cast<int>(bi % s.N), b = static_cast<int>(bi / s.N);
  const int kv = h / s.G;
  const int32_t* id = idx + ((static_cast<int64_t>(b) * s.Hkv + kv) * s.N + i) * s.K;
  const float* pl = part_lse + row * s.K;
  float m = neg_inf();
  for (int q = 0; q < s.K; ++q)
    if (id[q] >= 0) m = fmaxf(m, pl[q]);
  float den = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int q = 0; q < s.K; ++q) {
    if (id[q] < 0) continue;
    const float w = expf(pl[q] - m);
    den += w;
    const __nv_bfloat16* src = part_o + (row * s.K + q) * D + lane * PER;
    if (PER == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] += w * __bfloat162float(e[u]);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] += w * __bfloat162float(e[u]);
    }
  }
  const float r = 1.f / den;
  __nv_bfloat16* dst = O + row * D + lane * PER;
#pragma unroll
  for (int u = 0; u < PER; u += 2)
    *reinterpret_cast<uint32_t*>(dst + u) = pack_bf16(acc[u] * r, acc[u + 1] * r);
  if (lane == 0) lse_out[(static_cast<int64_t>(b) * s.Hq + h) * s.N + i] = m + logf(den);
}

template <int D, int G>
void fwd_launch(const Dims& s, const void* Q, const void* K, const void* V, const int32_t* off,
                const int32_t* list, __nv_bfloat16* po, float* pl, cudaStream_t st) {
  ProfScope ps(st, "attn_fwd_partial");
  attn_fwd_partial_kernel<D, G><<<dim3(s.n0, s.Hkv, s.B), kWarps * 32, 0, st>>>(
      s, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
      static_cast<const __nv_bfloat16*>(V), off, list, po, pl);
}

template <int D>
void fwd_dispatch(const Dims& s, const void* Q, const void* K, const void* V, const int32_t* off,
                  const int32_t* list, __nv_bfloat16* po, float* pl, cudaStream_t st) {
  switch (s.G) {
    case 1: fwd_launch<D, 1>(s, Q, K, V, off, list, po, pl, st); break;
    case 2: fwd_launch<D, 2>(s, Q, K, V, off, list, po, pl, st); break;
    case 4: fwd_launch<D, 4>(s, Q, K, V, off, list, po, pl, st); break;
    default: fwd_launch<D, 8>(s, Q, K, V, off, list, po, pl, st); break;
  }
}

}  // namespace

AttnFwdWs attn_fwd_ws(const Dims& s) {
  AttnFwdWs w{};
  const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.N;
  const size_t rows = static_cast<size_t>(s.B) * s.N * s.Hq;
  const size_t bins = static_cast<size_t>(s.B) * s.Hkv * s.n0;
  size_t o = 0;
  w.counts = o;   o += align256((bins + 1) * 4);
  w.cursor = o;   o += align256((bins + 1) * 4);
  w.list = o;     o += align256(units * s.K * 4);
  w.part_o = o;   o += align256(rows * s.K * s.d * 2);
  w.part_lse = o; o += align256(rows * s.K * 4);
  w.total = o;
  return w;
}

int launch_attn_fwd(const Dims& s, const void* Q, const void* K, const void* V,
                    const int32_t* idx, void* O, float* lse, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnFwdWs w = attn_fwd_ws(s);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + w.counts);
  int32_t* cursor = reinterpret_cast<int32_t*>(ws + w.cursor);
  int32_t* list = reinterpret_cast<int32_t*>(ws + w.list);
  __nv_bfloat16* po = reinterpret_cast<__nv_bfloat16*>(ws + w.part_o);
  float* pl = reinterpret_cast<float*>(ws + w.part_lse);
  int err = launch_group(s, idx, s.K, counts, cursor, list, st);
  if (err) return err;
  if (s.d == 128) fwd_dispatch<128>(s, Q, K, V, counts, list, po, pl, st);
  else fwd_dispatch<64>(s, Q, K, V, counts, list, po, pl, st);
  if ((err = cudaGetLastError())) return err;
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  ProfScope ps(st, "attn_combine");
  if (s.d == 128)
    attn_combine_kernel<128><<<blocks, 256, 0, st>>>(s, idx, po, pl, static_cast<__nv_bfloat16*>(O), lse);
  else
    attn_combine_kernel<64><<<blocks, 256, 0, st>>>(s, idx, po, pl, static_cast<__nv_bfloat16*>(O), lse);
  return cudaGetLastError();
}

}  // namespace pisa
