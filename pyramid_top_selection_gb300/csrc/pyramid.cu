// Key pyramid build: leaf sums over C tokens, then parents = left + right.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Method key
// points": leaf blocks of C tokens, mean pooling upward with merge factor 2, O(log N)
// levels. The kernels store SUMS (a node's mean is its sum over its token count), so a
// parent is exactly the fp32 sum of its two children, and the decode step can rebuild a
// leaf and its ancestors with the identical arithmetic.
//
// Fixed summation order (relied upon by the decode kernel for bit-exact updates):
//   leaf:   acc = 0.0f; for tokens j ascending: acc += float(k_j)     (per dimension)
//   parent: S(l,m) = S(l-1,2m) + S(l-1,2m+1), or S(l-1,2m) when 2m+1 does not exist.
// Bound: HBM. One launch reads N*Hkv*d*2 bytes of K and writes ~2*n0*Hkv*d*4 bytes.
#include "device.cuh"
#include "profile.h"

namespace pisa {

namespace {

constexpr int kLeavesPerCta = 8;   // leaves reduced by one CTA; levels 1..3 finish in-CTA
constexpr int kInCtaLevels = 3;

// Grid (ceil(n0/8), Hkv, B); block (D/8) * 8 threads: thread = (leaf, 8-dim chunk).
// SQ: sums of squared keys instead (per dimension; same order), for the PISA-2 ablation.
template <int D, bool SQ>
__global__ void __launch_bounds__(D)
build_leaves_kernel(const __nv_bfloat16* __restrict__ K, const int32_t* __restrict__ len,
                    int64_t T, int Hkv, int C, Geo geo, float* __restrict__ pyr) {
  constexpr int CH = D / 8;
  __shared__ __align__(16) float sm[2][kLeavesPerCta][D];
  const int b = blockIdx.z, kv = blockIdx.y;
  const int leaf0 = blockIdx.x * kLeavesPerCta;
  const int ll = threadIdx.x / CH, ch = threadIdx.x % CH;
  const int t = leaf0 + ll;
  const int64_t present = len ? min(static_cast<int64_t>(max(len[b], 0)), T) : T;
  const int64_t head = static_cast<int64_t>(b) * Hkv + kv;
  float* pyr_h = pyr + head * geo.nodes * D;

  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  if (t < geo.size[0]) {
    const int64_t s = static_cast<int64_t>(t) * C;
    const int64_t e_ = min(s + C, present);
    const __nv_bfloat16* base = K + (static_cast<int64_t>(b) * T * Hkv + kv) * D + ch * 8;
    const int64_t stride = static_cast<int64_t>(Hkv) * D;
    int64_t j = s;
    for (; j + 8 <= e_; j += 8) {          // eight rows in flight, added in token order
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = ldg_u4(base + (j + u) * stride);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&v[u]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __bfloat162float(h[e]);
          acc[e] += SQ ? x * x : x;
        }
      }
    }
    for (; j < e_; ++j) {
      uint4 v = ldg_u4(base + j * stride);
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = __bfloat162float(h[e]);
        acc[e] += SQ ? x * x : x;
      }
    }
    float4* out = reinterpret_cast<float4*>(pyr_h + (geo.off[0] + t) * D + ch * 8);
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) sm[0][ll][ch * 8 + e] = acc[e];
  __syncthreads();

  // Levels 1..3: node m at level l covers leaves [m<<l, (m+1)<<l), all inside this CTA.
  int cur = 0;
  for (int l = 1; l <= kInCtaLevels && l < geo.n_levels; ++l) {
    const int here = kLeavesPerCta >> l;
    for (int it = threadIdx.x; it < here * D; it += blockDim.x) {
      const int nl = it / D, k = it % D;
      const int m = (leaf0 >> l) + nl;
      float v = sm[cur][2 * nl][k];
      if (2 * m + 1 < geo.size[l - 1]) v = v + sm[cur][2 * nl + 1][k];
      sm[cur ^ 1][nl][k] = v;
      if (m < geo.size[l]) pyr_h[(geo.off[l] + m) * D + k] = v;
    }
    cur ^= 1;
    __syncthreads();
  }
}

// Upper levels by subtrees: grid (ceil(n_src / 64), heads). A CTA loads 64 nodes of level
// l_src (those of its subtree) and computes the up to kSubLevels levels above them in shared
// memory, writing every node it completes (parent = left + right, or left alone).
constexpr int kSubNodes = 64;
constexpr int kSubLevels = 6;                  // 64 nodes -> 1

template <int D>
__global__ void __launch_bounds__(256)
build_subtree_kernel(Geo geo, int l_src, float* __restrict__ pyr) {
  __shared__ __align__(16) float sa[kSubNodes * D];          // levels l_src, l_src + 2, ...
  __shared__ __align__(16) float sb[(kSubNodes / 2) * D];    // levels l_src + 1, l_src + 3, ...
  const int64_t head = blockIdx.y;
  float* pyr_h = pyr + head * geo.nodes * D;
  const int m0 = blockIdx.x * kSubNodes;
  const int here = min(kSubNodes, geo.size[l_src] - m0);
  const float4* src = reinterpret_cast<const float4*>(pyr_h + (geo.off[l_src] + m0) * D);
  for (int it = threadIdx.x; it < here * D / 4; it += blockDim.x)
    reinterpret_cast<float4*>(sa)[it] = src[it];
  __syncthreads();
  int cnt = here;                              // nodes of the current level inside the subtree
  const float* cur = sa;
  float* nxt = sb;
  for (int l = l_src + 1; l <= l_src + kSubLevels && l < geo.n_levels; ++l) {
    const int nl = (cnt + 1) / 2, first = m0 >> (l - l_src), nc = geo.size[l - 1];
    const int c0 = m0 >> (l - 1 - l_src);     // first child index at level l - 1
    for (int it = threadIdx.x; it < nl * D; it += blockDim.x) {
      const int m = it / D, k = it % D;
      float v = cur[(2 * m) * D + k];
      if (c0 + 2 * m + 1 < nc) v = v + cur[(2 * m + 1) * D + k];
      nxt[it] = v;
      if (first + m < geo.size[l]) pyr_h[(geo.off[l] + first + m) * D + k] = v;
    }
    __syncthreads();
    float* t = const_cast<float*>(cur);
    cur = nxt;
    nxt = t;
    cnt = nl;
  }
}

template <int D, bool SQ = false>
int build_impl(const Dims& s, const Geo& g, const void* K, const int32_t* len, int64_t T,
               float* pyr, cudaStream_t st) {
  dim3 grid((g.size[0] + kLeavesPerCta - 1) / kLeavesPerCta, s.Hkv, s.B);
  { ProfScope ps(st, SQ ? "build_sq_leaves" : "build_leaves");
  build_leaves_kernel<D, SQ><<<grid, (D / 8) * kLeavesPerCta, 0, st>>>(
      static_cast<const __nv_bfloat16*>(K), len, T, s.Hkv, s.C, g, pyr); }
  for (int l = kInCtaLevels; l + 1 < g.n_levels; l += kSubLevels) {
    ProfScope ps(st, "build_upper");
    const int n = g.size[l];
    build_subtree_kernel<D><<<dim3((n + kSubNodes - 1) / kSubNodes, s.B * s.Hkv), 256, 0, st>>>(g, l, pyr);
  }
  return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_build_pyramid(const Dims& s, const Geo& g, const void* K, const int32_t* len,
                         int64_t tokens_per_seq, float* pyr, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s.d == 128) return build_impl<128>(s, g, K, len, tokens_per_seq, pyr, st);
  return build_impl<64>(s, g, K, len, tokens_per_seq, pyr, st);
}

// Pyramid of per-dimension sums of squared keys (same layout and summation order), one per
// real KV head also when the selection units are query heads.
int launch_build_pyramid_sq(const Dims& s, const Geo& g, const void* K, float* sq, cudaStream_t st) {
  Dims k = s;
  k.Hkv = s.Hkv_r;
  k.G = s.Hq / s.Hkv_r;
  k.kvr = 1;
  if (s.d == 128) return build_impl<128, true>(k, g, K, nullptr, s.N, sq, st);
  return build_impl<64, true>(k, g, K, nullptr, s.N, sq, st);
}

const char* cuda_error_string(int err) {
  return cudaGetErrorString(static_cast<cudaError_t>(err));
}

}  // namespace pisa
