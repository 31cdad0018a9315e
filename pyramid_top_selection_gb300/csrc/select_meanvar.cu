// PISA-2 ablation selection: the coarse-to-fine pyramid descent with every block, leaves
// included, scored by its mean and its per-dimension variance.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Method key points":
// in the ablation PISA-1 scores blocks by the mean and PISA-2 by mean + variance; the full LSE
// works best. The pages give no formula for PISA-2; the reading taken here is the second-order
// cumulant expansion of a block's log-mean-exp with a diagonal covariance: block m at level l
// scores, for query i of a KV head with heads h,
//     sum_h [ s q_h . mu + (s^2 / 2) sum_k q_hk^2 var_k ],
// mu and var the mean and the population variance (per dimension) of the block's keys j <= i.
// The sum over the heads moves inside both dot products, so with Q1 = sum_h q_h and
// Q2 = sum_h q_h * q_h (per dimension) a block costs two d-long dots:
//     s (S / n) . Q1 + (s^2 / 2) (SQ / n - (S / n)^2) . Q2,
// S and SQ the block's key sums and squared-key sums over its n causal keys.
//
// One warp per (b, KV head, query i), lanes over dimensions (fp32 FMA; this ablation is not on
// the method's hot path and runs on the CUDA cores). The causal prefix sums of the path node
// at every level (the node holding i) are built bottom-up from the query's own-leaf keys and
// the full left siblings on its ancestor path, and kept in shared memory. The descent, the
// candidate sets, the tie rule and the output are those of the other selections; the leaf
// candidates' scores go to the top-K finish.
#include "device.cuh"
#include "profile.h"

namespace pisa {

int launch_build_pyramid_sq(const Dims& s, const Geo& g, const void* K, float* sq, cudaStream_t st);
int launch_topk(const Dims& s, int W, const int32_t* cand, const float* cscore, const float* chead,
                int32_t* idx, float* score, float* head_lse, const int32_t* status, cudaStream_t st);
size_t align256(size_t x);

namespace {

constexpr int kWarps = 4;
constexpr int kMaxCand = 64;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
meanvar_kernel(Dims s, Geo geo, const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Kt,
               const float* __restrict__ pyr, const float* __restrict__ sqp, int32_t* __restrict__ cand_out,
               float* __restrict__ cscore_out) {
  constexpr int E = D / 32;                   // dimensions per lane: lane*E .. lane*E + E - 1
  extern __shared__ __align__(16) float smv[];   // per warp: [levels][2][D] path prefix sums
  __shared__ int s_cand[kWarps][kMaxCand];
  __shared__ int s_kept[kWarps][kMaxCand / 2];
  __shared__ float s_sc[kWarps][kMaxCand];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, kv = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  if (i >= s.N) return;                       // no block-wide barriers below
  const int G = s.G, Ksel = s.K, C = s.C, L = geo.n_levels;
  const int ti = i / C;
  const int64_t head = static_cast<int64_t>(b) * s.Hkv + kv;                       // selection unit
  const int64_t head_k = static_cast<int64_t>(b) * s.Hkv_r + kv / s.kvr;           // its KV head
  const float* pyr_h = pyr + head_k * geo.nodes * D;
  const float* sq_h = sqp + head_k * geo.nodes * D;
  float* pre = smv + static_cast<size_t>(warp) * L * 2 * D;
  const int d0 = lane * E;

  // Q1 = sum_h q_h, Q2 = sum_h q_h^2 on the lane's dimensions
  float q1[E], q2[E];
#pragma unroll
  for (int e = 0; e < E; ++e) q1[e] = q2[e] = 0.f;
  for (int h = 0; h < G; ++h) {
    const __nv_bfloat16* qr = Q + ((static_cast<int64_t>(b) * s.N + i) * s.Hq + kv * G + h) * D + d0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float x = __bfloat162float(qr[e]);
      q1[e] += x;
      q2[e] += x * x;
    }
  }
  // path prefix sums: level 0 = the own leaf's keys j <= i; level l adds the full left sibling
  // of the level-(l-1) ancestor when that ancestor is a right child
  {
    float ps[E], pq[E];
#pragma unroll
    for (int e = 0; e < E; ++e) ps[e] = pq[e] = 0.f;
    for (int64_t j = static_cast<int64_t>(ti) * C; j <= i; ++j) {
      const __nv_bfloat16* kr = Kt + ((static_cast<int64_t>(b) * s.N + j) * s.Hkv_r + kv / s.kvr) * D + d0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = __bfloat162float(kr[e]);
        ps[e] += x;
        pq[e] += x * x;
      }
    }
    for (int l = 0; l < L; ++l) {
      if (l > 0 && ((ti >> (l - 1)) & 1)) {
        const int64_t node = geo.off[l - 1] + (ti >> (l - 1)) - 1;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          ps[e] += pyr_h[node * D + d0 + e];
          pq[e] += sq_h[node * D + d0 + e];
        }
      }
#pragma unroll
      for (int e = 0; e < E; ++e) {
        pre[(l * 2) * D + d0 + e] = ps[e];
        pre[(l * 2 + 1) * D + d0 + e] = pq[e];
      }
    }
  }
  __syncwarp();

  const float sc1 = s.scale, sc2 = 0.5f * s.scale * s.scale;
  // score of node c at level l (warp-wide; every lane returns the total)
  auto node_score = [&](int l, int c) {
    const int64_t span = static_cast<int64_t>(C) << l, st = c * span;
    const float* S;
    const float* SQ;
    float n;
    if (c == (ti >> l)) {            // the node holding i: its keys j <= i
      S = pre + (l * 2) * D;
      SQ = pre + (l * 2 + 1) * D;
      n = static_cast<float>(i - st + 1);
    } else {
      S = pyr_h + (geo.off[l] + c) * D;
      SQ = sq_h + (geo.off[l] + c) * D;
      n = static_cast<float>(min(st + span, static_cast<int64_t>(s.N)) - st);
    }
    const float inv = 1.f / n;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float mu = S[d0 + e] * inv;
      const float var = SQ[d0 + e] * inv - mu * mu;
      part += sc1 * mu * q1[e] + sc2 * var * q2[e];
    }
    return no_nan(warp_sum(part));
  };

  int* cand = s_cand[warp];
  int* kept = s_kept[warp];
  float* sc = s_sc[warp];
  int nkept = 1;
  if (lane == 0) kept[0] = 0;
  __syncwarp();
  const unsigned ltm = lanemask_lt();
  int nc = 1;
  if (L == 1 && lane == 0) cand[0] = 0;
  for (int lam = L - 2; lam >= 0; --lam) {
    // candidates at level lam: the visible children of the kept nodes of level lam + 1
    const int64_t span = static_cast<int64_t>(C) << lam;
    {
      const int a = lane < nkept ? kept[lane] : -1;
      const bool c0 = a >= 0;
      const bool c1 = a >= 0 && static_cast<int64_t>(2 * a + 1) * span <= i;
      const unsigned m0 = __ballot_sync(0xffffffffu, c0), m1 = __ballot_sync(0xffffffffu, c1);
      const int pos = __popc(m0 & ltm) + __popc(m1 & ltm);
      __syncwarp();
      if (c0) cand[pos] = 2 * a;
      if (c1) cand[pos + 1] = 2 * a + 1;
      nc = __popc(m0) + __popc(m1);
    }
    __syncwarp();
    if (lam == 0) break;
    if (nc <= Ksel) {
      if (lane < nc) kept[lane] = cand[lane];
      nkept = nc;
      __syncwarp();
      continue;
    }
    for (int k = 0; k < nc; ++k) {
      const float v = node_score(lam, cand[k]);
      if (lane == 0) sc[k] = v;
    }
    __syncwarp();
    for (int s2 = lane; s2 < nc; s2 += 32) {
      const float my = sc[s2];
      const int mi = cand[s2];
      int rank = 0;
      for (int o = 0; o < nc; ++o) rank += beats(sc[o], cand[o], my, mi) ? 1 : 0;
      if (rank < Ksel) kept[rank] = mi;
    }
    nkept = Ksel;
    __syncwarp();
  }
  // leaf candidates and their scores go to the top-K finish
  for (int k = 0; k < nc; ++k) {
    const float v = node_score(0, cand[k]);
    if (lane == 0) sc[k] = v;
  }
  __syncwarp();
  const int64_t u = (head * s.N + i) * (2 * Ksel);
  for (int q = lane; q < 2 * Ksel; q += 32) {
    cand_out[u + q] = q < nc ? cand[q] : -1;
    cscore_out[u + q] = q < nc ? sc[q] : neg_inf();
  }
}

struct MeanVarWs {
  size_t status, sq, cand, cscore, total;
};

MeanVarWs meanvar_ws_of(const Dims& s, const Geo& g) {
  MeanVarWs w{};
  const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.N;
  size_t o = 0;
  w.status = o; o += 256;
  w.sq = o;     o += align256(static_cast<size_t>(s.B) * s.Hkv_r * g.nodes * s.d * 4);
  w.cand = o;   o += align256(units * 2 * s.K * 4);
  w.cscore = o; o += align256(units * 2 * s.K * 4);
  w.total = o;
  return w;
}

}  // namespace

size_t meanvar_ws(const Dims& s, const Geo& g) { return meanvar_ws_of(s, g).total; }

int launch_select_meanvar(const Dims& s, const Geo& g, const void* Q, const void* K, const float* pyr,
                          int32_t* idx, float* score, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const MeanVarWs w = meanvar_ws_of(s, g);
  float* sq = reinterpret_cast<float*>(ws + w.sq);
  int32_t* cand = reinterpret_cast<int32_t*>(ws + w.cand);
  float* cscore = reinterpret_cast<float*>(ws + w.cscore);
  int err = cudaMemsetAsync(ws + w.status, 0, 256, st);     // no bounded waits here: stays 0
  if (err) return err;
  if ((err = launch_build_pyramid_sq(s, g, K, sq, st))) return err;
  const size_t smem = static_cast<size_t>(kWarps) * g.n_levels * 2 * s.d * 4;
  dim3 grid((s.N + kWarps - 1) / kWarps, s.Hkv, s.B);
  {
    ProfScope ps(st, "route_meanvar");
    if (s.d == 128) {
      cudaFuncSetAttribute(meanvar_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      meanvar_kernel<128><<<grid, kWarps * 32, smem, st>>>(s, g, static_cast<const __nv_bfloat16*>(Q),
                                                           static_cast<const __nv_bfloat16*>(K), pyr, sq, cand, cscore);
    } else {
      cudaFuncSetAttribute(meanvar_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      meanvar_kernel<64><<<grid, kWarps * 32, smem, st>>>(s, g, static_cast<const __nv_bfloat16*>(Q),
                                                          static_cast<const __nv_bfloat16*>(K), pyr, sq, cand, cscore);
    }
  }
  if ((err = cudaGetLastError())) return err;
  return launch_topk(s, 2 * s.K, cand, cscore, nullptr, idx, score, nullptr,
                     reinterpret_cast<const int32_t*>(ws + w.status), st);
}

}  // namespace pisa
