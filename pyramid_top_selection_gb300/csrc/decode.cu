// Single-kernel decode step: append, ancestor-path pyramid update, all-level selection
// and sparse attention for one new token per sequence, in ONE launch.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference
// value of the work": decoding fuses all pyramid levels in a single kernel to avoid
// repeated launches, and the cached mean pyramid is updated only on the ancestor path of
// the current token, amortised O(log N) per step.
//
// One CTA per (KV head, sequence), 8 warps. The cached pyramid holds key SUMS over the
// tokens present so far (absent tokens count as zero), so the node that holds the new
// token p already carries the causal prefix sum; its mean is the sum over its present
// token count. Arithmetic order of the update matches the pyramid build kernel exactly
// (leaf: fp32 sum of the leaf's keys in token order; parent = left + right), so the
// incrementally maintained pyramid equals one rebuilt from the cache, bit for bit.
#include "device.cuh"
#include "profile.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCand = 64;

struct DecodeSmem {
  // offsets in floats inside dynamic shared memory
  int q32, S, lh, red, dots;
  int total;
};

__host__ __device__ inline DecodeSmem decode_smem(int G, int D, int K) {
  DecodeSmem m{};
  int o = 0;
  m.q32 = o;  o += G * (D + 16);   // per head: 4 quarters of D/4 floats, each padded by 4
  m.S = o;    o += 2 * K * (64 * G + 4);   // per candidate leaf: 64 keys x G heads + 4 pad
  m.lh = o;   o += 2 * K * G;
  m.red = o;  o += kWarps * G * D;
  m.dots = o; o += kMaxCand * 2 * G;
  m.total = o;
  return m;
}

// GT: the query heads per KV head (1, 2, 4 or 8), a compile-time constant so that every
// per-head loop unrolls and the attention loop reads a key's G probabilities in one load.
template <int D, int GT>
__global__ void __launch_bounds__(kThreads, 2)   // two CTAs per SM: a batch of sequences x KV heads in one wave
decode_kernel(Dims s, Geo geo, const int32_t* __restrict__ pos, __nv_bfloat16* Kc,
              __nv_bfloat16* Vc, float* pyr, const __nv_bfloat16* __restrict__ qn,
              const __nv_bfloat16* __restrict__ kn, const __nv_bfloat16* __restrict__ vn,
              __nv_bfloat16* __restrict__ o_out, int32_t* __restrict__ idx_out,
              float* __restrict__ score_out, int32_t* __restrict__ status) {
  constexpr int KS = D / 16;
  extern __shared__ __align__(16) float sm[];
  __shared__ int s_cand[kMaxCand];
  __shared__ int s_kept[kMaxCand];
  __shared__ float s_sc[kMaxCand];
  __shared__ int s_sel[kMaxCand / 2];    // selected candidate slots, ascending leaf order
  __shared__ float s_lse[8];
  __shared__ int s_n[2];

  const int kv = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, pq = lane & 3;
  constexpr int G = GT;
  const int Ksel = s.K, C = s.C, Ncap = s.N;
  const int p = pos[b];
  if (p < 0 || p >= Ncap) {
    if (tid == 0) atomicOr(status, PISA_STATUS_POS_RANGE);
    return;
  }
  const DecodeSmem L = decode_smem(G, D, Ksel);
  float* q32 = sm + L.q32;
  float* Sb = sm + L.S;
  float* lh = sm + L.lh;
  float* red = sm + L.red;
  float* dots = sm + L.dots;

  const int64_t head = static_cast<int64_t>(b) * s.Hkv + kv;
  float* pyr_h = pyr + head * geo.nodes * D;
  auto krow = [&](int64_t j) { return Kc + ((static_cast<int64_t>(b) * Ncap + j) * s.Hkv + kv) * D; };
  auto vrow = [&](int64_t j) { return Vc + ((static_cast<int64_t>(b) * Ncap + j) * s.Hkv + kv) * D; };

  // 1. append k/v at slot p; q to shared memory
  if (tid < D / 8) {
    reinterpret_cast<uint4*>(krow(p))[tid] = ldg_u4(kn + head * D + tid * 8);
    reinterpret_cast<uint4*>(vrow(p))[tid] = ldg_u4(vn + head * D + tid * 8);
  }
  const __nv_bfloat16* qg = qn + (static_cast<int64_t>(b) * s.Hq + kv * G) * D;
  // quarters 16 bytes apart in bank terms, so the level dots' 4 quarter readers never collide
  for (int it = tid; it < G * D; it += kThreads)
    q32[(it / D) * (D + 16) + (it % D) / (D / 4) * (D / 4 + 4) + it % (D / 4)] = __bfloat162float(qg[it]);
  __syncthreads();

  // 2. leaf recompute (token order) and ancestor path (left + right)
  const int tp = p / C;
  if (tid < D) {
    float acc = 0.0f;
    for (int64_t j = static_cast<int64_t>(tp) * C; j <= p; ++j) acc += __bfloat162float(krow(j)[tid]);
    pyr_h[(geo.off[0] + tp) * D + tid] = acc;
    int m = tp;
    float v = acc;
    for (int l = 1; l < geo.n_levels; ++l) {
      const int sib = m ^ 1;
      if (sib < geo.size[l - 1]) {
        const float sv = pyr_h[(geo.off[l - 1] + sib) * D + tid];
        v = (m & 1) ? (sv + v) : (v + sv);
      }
      m >>= 1;
      pyr_h[(geo.off[l] + m) * D + tid] = v;
    }
  }
  __syncthreads();

  // 3. intermediate levels. Warp 0 drives the descent: it expands the kept nodes into
  // candidates (ballot compaction) and keeps them all while there are at most K, with no
  // CTA barrier; a level with more candidates is published for the CTA-wide dot phase (two
  // barriers), then warp 0 scores the candidates and keeps the top K by shuffle ranks.
  __shared__ int s_lam;
  const int Lv = geo.n_levels;
  int lam = Lv - 2;          // warp 0: the level whose candidates come next
  int n_kept = 1;            // warp 0: kept nodes (in s_kept) at level lam + 1
  if (tid == 0) s_kept[0] = 0;
  __syncwarp();
  while (true) {
    if (warp == 0) {
      int nc = 0;
      for (; lam >= 1; --lam) {
        const int64_t span = static_cast<int64_t>(C) << lam;
        int a = 0;
        bool c1 = false;
        if (lane < n_kept) {
          a = s_kept[lane];
          c1 = static_cast<int64_t>(2 * a + 1) * span <= p;
        }
        const unsigned m1 = __ballot_sync(0xffffffffu, c1);
        const int pos = lane + __popc(m1 & lanemask_lt());
        if (lane < n_kept) {
          s_cand[pos] = 2 * a;
          if (c1) s_cand[pos + 1] = 2 * a + 1;
        }
        nc = n_kept + __popc(m1);
        __syncwarp();
        if (nc > Ksel) break;
        if (lane < nc) s_kept[lane] = s_cand[lane];
        n_kept = nc;
        __syncwarp();
      }
      if (lane == 0) {
        s_lam = lam;
        s_n[0] = n_kept;
        s_n[1] = nc;
      }
    }
    __syncthreads();
    const int lv = s_lam;
    if (lv < 1) break;
    const int nc = s_n[1];
    const int64_t cspan = static_cast<int64_t>(C) << (lv - 1);
    {
      // child rows (candidate cs, child e) -> row 2cs+e, 64 rows per pass; thread = (row,
      // quarter of the dims): its D/4 dims of the row load at once, each head's partial dot
      // is combined over the 4 quarters (adjacent lanes) with two shuffles
      constexpr int QD = D / 4, NV = QD / 4;
      const int rq = tid >> 2, qt = tid & 3;
      for (int base = 0; base < 2 * nc; base += kThreads / 4) {
        const int row = base + rq;
        const int64_t ch = row < 2 * nc ? 2LL * s_cand[row >> 1] + (row & 1) : 0;
        const int64_t st = ch * cspan;
        const bool vis = row < 2 * nc && st <= p;
        float4 xr[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          xr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (vis) xr[u] = reinterpret_cast<const float4*>(pyr_h + (geo.off[lv - 1] + ch) * D + qt * QD)[u];
        }
        const float cnt = vis ? static_cast<float>(min(st + cspan, static_cast<int64_t>(p) + 1) - st) : 1.f;
        for (int h = 0; h < G; ++h) {
          const float4* qq = reinterpret_cast<const float4*>(q32 + h * (D + 16) + qt * (QD + 4));
          float part = 0.f;
#pragma unroll
          for (int u = 0; u < NV; ++u) {
            const float4 y = qq[u];
            part = fmaf(xr[u].x, y.x, part);
            part = fmaf(xr[u].y, y.y, part);
            part = fmaf(xr[u].z, y.z, part);
            part = fmaf(xr[u].w, y.w, part);
          }
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          if (qt == 0 && row < 2 * nc) dots[row * G + h] = vis ? s.scale * part / cnt : neg_inf();
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // scores of candidates lane and lane + 32, then each one's rank among all of them
      float sc[2];
      int ci[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u;
        sc[u] = neg_inf();
        ci[u] = 0;
        if (c < nc) {
          float tot = 0.f;
          for (int h = 0; h < G; ++h) {
            const float x0 = dots[(2 * c) * G + h], x1 = dots[(2 * c + 1) * G + h];
            if (x1 == neg_inf()) {
              tot += x0;
            } else {                                 // two-term LSE: max + log(1 + exp(-|difference|))
              tot += fmaxf(x0, x1) + __logf(1.f + __expf(-fabsf(x0 - x1)));
            }
          }
          sc[u] = no_nan(tot);
          ci[u] = s_cand[c];
        }
      }
      int rk[2] = {0, 0};
      const int nv = nc > 32 ? 2 : 1;
      for (int v = 0; v < nv; ++v)
        for (int o = 0; o < 32; ++o) {
          const float so = __shfl_sync(0xffffffffu, sc[v], o);
          const int io = __shfl_sync(0xffffffffu, ci[v], o);
          if (o + 32 * v < nc) {
            rk[0] += beats(so, io, sc[0], ci[0]) ? 1 : 0;
            rk[1] += beats(so, io, sc[1], ci[1]) ? 1 : 0;
          }
        }
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (lane + 32 * u < nc && rk[u] < Ksel) s_kept[rk[u]] = ci[u];
      n_kept = Ksel;
      --lam;
      __syncwarp();
    }
  }

  // 4. leaf candidates and exact leaf LSE (MMA: rows = keys, columns = heads)
  if (tid == 0) {
    int nc = 0;
    if (Lv == 1) {
      s_cand[nc++] = 0;
    } else {
      for (int k = 0; k < s_n[0]; ++k) {
        const int a = s_kept[k];
        s_cand[nc++] = 2 * a;
        if (static_cast<int64_t>(2 * a + 1) * C <= p) s_cand[nc++] = 2 * a + 1;
      }
    }
    s_n[1] = nc;
  }
  __syncthreads();
  const int nlc = s_n[1];
  {
    // k-step 2 kp + e of fragment lane pq takes dims 32 kp + 8 pq + 4 e .. + 3 (a dot product may
    // take its terms in any order as long as both operands agree): a lane's dims for the two
    // k-steps of a pair are 8 adjacent ones, one 16-byte load per key row
    uint32_t qb[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint2 v = g < G ? ldg_u2(qg + static_cast<int64_t>(g) * D + 32 * (ks >> 1) + 8 * pq + 4 * (ks & 1))
                            : make_uint2(0, 0);
      qb[ks][0] = v.x;
      qb[ks][1] = v.y;
    }
    for (int cs = warp; cs < nlc; cs += kWarps) {
      const int64_t t0 = static_cast<int64_t>(s_cand[cs]) * C;
      float* Sr = Sb + static_cast<int64_t>(cs) * (64 * G + 4);
#pragma unroll
      for (int mh = 0; mh < 2; ++mh) {               // two 16-key tiles per round, all loads in flight
        uint4 x[2][2][KS / 2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int rr = (2 * mh + m) * 16 + g + 8 * hr;
            const bool vr = t0 + rr <= p;
            const __nv_bfloat16* kr = krow(t0 + rr) + 8 * pq;
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) x[m][hr][kp] = vr ? ldg_u4(kr + 32 * kp) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int r0 = (2 * mh + m) * 16 + g, r1 = r0 + 8;
          const bool v0 = t0 + r0 <= p, v1 = t0 + r1 <= p;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kp = 0; kp < KS / 2; ++kp) {
            const uint4 x0 = x[m][0][kp], x1 = x[m][1][kp];
            const uint32_t a0[4] = {x0.x, x1.x, x0.y, x1.y}, a1[4] = {x0.z, x1.z, x0.w, x1.w};
            mma_bf16(acc, a0, qb[2 * kp][0], qb[2 * kp][1]);
            mma_bf16(acc, a1, qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * pq + e;
            if (h < G) {
              Sr[r0 * G + h] = v0 ? s.scale * acc[e] : neg_inf();
              Sr[r1 * G + h] = v1 ? s.scale * acc[2 + e] : neg_inf();
            }
          }
        }
      }
    }
  }
  __syncthreads();
  for (int it = tid; it < nlc * G; it += kThreads) {
    const int cs = it / G, h = it % G;
    const float* Sr = Sb + static_cast<int64_t>(cs) * (64 * G + 4);
    float mx = neg_inf();
    for (int k = 0; k < 64; ++k) mx = fmaxf(mx, Sr[k * G + h]);
    float sum = 0.f;
    for (int k = 0; k < 64; ++k) sum += expf(Sr[k * G + h] - mx);
    lh[it] = mx + logf(sum);
  }
  __syncthreads();
  if (tid < nlc) {
    float tot = 0.f;
    for (int h = 0; h < G; ++h) tot += lh[tid * G + h];
    s_sc[tid] = no_nan(tot);
  }
  __syncthreads();
  // 5. top K leaves, ascending
  if (tid < nlc) {
    const float my = s_sc[tid];
    const int mi = s_cand[tid];
    int rank = 0;
    for (int o = 0; o < nlc; ++o) rank += beats(s_sc[o], s_cand[o], my, mi) ? 1 : 0;
    s_kept[tid] = rank < Ksel ? 1 : 0;
  }
  __syncthreads();
  if (tid < nlc && s_kept[tid]) {
    int posn = 0;
    for (int o = 0; o < nlc; ++o) posn += (s_kept[o] && s_cand[o] < s_cand[tid]) ? 1 : 0;
    s_sel[posn] = tid;
    idx_out[head * Ksel + posn] = s_cand[tid];
    if (score_out) score_out[head * Ksel + posn] = s_sc[tid];
  }
  const int nsel = min(nlc, Ksel);
  if (tid >= nsel && tid < Ksel) {
    idx_out[head * Ksel + tid] = -1;
    if (score_out) score_out[head * Ksel + tid] = neg_inf();
  }
  __syncthreads();
  // 6. attention over the selected leaves, reusing the leaf logits S
  if (tid < G) {
    float mx = neg_inf();
    for (int k = 0; k < nsel; ++k) mx = fmaxf(mx, lh[s_sel[k] * G + tid]);
    float sum = 0.f;
    for (int k = 0; k < nsel; ++k) sum += expf(lh[s_sel[k] * G + tid] - mx);
    s_lse[tid] = mx + logf(sum);
  }
  __syncthreads();
  // P = exp(S - lse) of the selected leaves, in place (one pass, all threads)
  for (int it = tid; it < nsel * 64 * G; it += kThreads) {
    const int k = it / (64 * G), rem = it % (64 * G);
    float* Sr = Sb + static_cast<int64_t>(s_sel[k]) * (64 * G + 4);
    Sr[rem] = expf(Sr[rem] - s_lse[rem % G]);
  }
  __syncthreads();
  {
    // o_h = sum over the selected keys of P[key][h] v_key: the keys of all selected leaves
    // are one flat list; each warp takes kKeyBatch consecutive keys at a time with all of
    // their V rows (lane: dims lane*PER ..) in flight before any is used
    constexpr int PER = D / 32;
    constexpr int kKeyBatch = 16;
    float acc[G][PER];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[h][u] = 0.f;
    const int nkeys = nsel * 64;
    const int64_t vstride = static_cast<int64_t>(s.Hkv) * D;   // cache row stride between tokens
    // a batch (16 keys, a multiple of 16 from the start) lies inside one selected leaf: its
    // leaf, first value row and probability row are looked up once
    for (int base = warp * kKeyBatch; base < nkeys; base += kWarps * kKeyBatch) {
      const int sl = s_sel[base >> 6];
      const int64_t j0 = static_cast<int64_t>(s_cand[sl]) * C + (base & 63);
      const __nv_bfloat16* v0 = vrow(j0) + lane * PER;
      const float* P0 = Sb + static_cast<int64_t>(sl) * (64 * G + 4) + (base & 63) * G;
      uint2 x[kKeyBatch];
#pragma unroll
      for (int u = 0; u < kKeyBatch; ++u) {
        x[u] = make_uint2(0, 0);
        if (j0 + u <= p) {
          const __nv_bfloat16* vr = v0 + u * vstride;
          if (PER == 4) x[u] = *reinterpret_cast<const uint2*>(vr);
          else x[u].x = *reinterpret_cast<const uint32_t*>(vr);
        }
      }
#pragma unroll
      for (int u = 0; u < kKeyBatch; ++u) {
        const float* Pr = P0 + u * G;
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&x[u]);
        float vv[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) vv[q] = __bfloat162float(e[q]);
        float pw[G];                                  // the key's G probabilities, one load
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int h4 = 0; h4 < G / 4; ++h4) {
            const float4 t = reinterpret_cast<const float4*>(Pr)[h4];
            pw[4 * h4] = t.x;
            pw[4 * h4 + 1] = t.y;
            pw[4 * h4 + 2] = t.z;
            pw[4 * h4 + 3] = t.w;
          }
        } else if constexpr (G == 2) {
          const float2 t = *reinterpret_cast<const float2*>(Pr);
          pw[0] = t.x;
          pw[1] = t.y;
        } else {
          pw[0] = Pr[0];
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int q = 0; q < PER; ++q) acc[h][q] = fmaf(pw[h], vv[q], acc[h][q]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int u = 0; u < PER; ++u) red[(warp * G + h) * D + lane * PER + u] = acc[h][u];
  }
  __syncthreads();
  for (int it = tid; it < G * D; it += kThreads) {
    const int h = it / D, k = it % D;
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v += red[(w * G + h) * D + k];
    o_out[(static_cast<int64_t>(b) * s.Hq + kv * G + h) * D + k] = __float2bfloat16_rn(v);
  }
}

}  // namespace

int launch_decode_step(const Dims& s, int32_t Ncap, const Geo& g, const int32_t* pos, void* Kc,
                       void* Vc, float* pyr, const void* q, const void* k_new, const void* v_new,
                       void* o, int32_t* idx, float* score, int32_t* status, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Dims d = s;
  d.N = Ncap;
  const DecodeSmem L = decode_smem(s.G, s.d, s.K);
  const size_t smem = static_cast<size_t>(L.total) * sizeof(float);
  dim3 grid(s.Hkv, s.B);
  ProfScope ps(st, "decode_step");
  auto run = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    kernel<<<grid, kThreads, smem, st>>>(
        d, g, pos, static_cast<__nv_bfloat16*>(Kc), static_cast<__nv_bfloat16*>(Vc), pyr,
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
        static_cast<const __nv_bfloat16*>(v_new), static_cast<__nv_bfloat16*>(o), idx, score, status);
  };
#define PISA_DECODE_CASE(DD, GG) \
  if (s.d == DD && s.G == GG) run(decode_kernel<DD, GG>);
  PISA_DECODE_CASE(128, 1) PISA_DECODE_CASE(128, 2) PISA_DECODE_CASE(128, 4) PISA_DECODE_CASE(128, 8)
  PISA_DECODE_CASE(64, 1) PISA_DECODE_CASE(64, 2) PISA_DECODE_CASE(64, 4) PISA_DECODE_CASE(64, 8)
#undef PISA_DECODE_CASE
  return cudaGetLastError();
}

}  // namespace pisa
