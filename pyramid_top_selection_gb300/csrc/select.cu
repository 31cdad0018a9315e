// Pyramid Top-K selection (two stages) and the flat comparator.
//
// "Block Sparse Attention with Log-Linear Complexity":
//  * abstract (arxivdaily page): coarse-to-fine hierarchy of pooled keys, selection from
//    the coarsest level, LogSumExp scoring of a bounded candidate set at every level down
//    to the finest, without materialising the query-key score matrix;
//  * daily digest page, "Method key points": candidate set starts with 1 node, at most gK
//    candidates per level, keep top K, expand only kept nodes; leaves scored by exact LSE
//    over raw keys, intermediate nodes by LSE over children's mean summaries; GQA heads
//    of one KV head share the selection; prefill runs in two stages: intermediate-level
//    routing first, then queries grouped per leaf key block so the block's keys are read
//    once per tile ("Reference value of the work").
//
// Stage 1 (route_kernel): one warp per (b, KV head, query i). The candidates' children
//   are contracted against the G query heads with bf16 MMAs on a hi/lo split of the fp32
//   key sums (fp32-accurate dots), LSE per head, sum over heads, warp top-K by rank.
//   The node that contains i is causal-partial: its dot is q . (sum of keys j <= i in it),
//   built bottom-up from the query's own-leaf prefix and the full left siblings on the
//   ancestor path; a prefix pass (route_prefix_kernel) computes these for 16 (query, head)
//   rows of one leaf at a time, which share the keys and siblings they read. Output: <= 2K
//   leaf candidates per query.
// Grouping: counting sort of (leaf, query) pairs into (KV head, query chunk, leaf) bins,
//   cut into work items (group.cu).
// Stage 2 (leaf_tc.cu): a persistent warp-specialised tcgen05 kernel walks the work items;
//   each item's 64 keys arrive by TMA and every (query, head) row is scored against them.
// Finish (topk_kernel): top K of the <= 2K exact leaf scores, output ascending.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"

namespace pisa {

int launch_leaf_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const int32_t* list,
                   const int4* items, const int32_t* n_items, int W, float* pair_score, float* pair_head,
                   int32_t* status, cudaStream_t st);


namespace {

constexpr int kWarps = 4;
constexpr int kMaxCand = 64;   // 2K for K <= 32


// Dimension order of the m16n8k16 fragments (a dot product may take its terms in any order,
// as long as both operands agree): lane p's four k-slots of k-step ks hold dims kdim(ks, p) ..
// + 3, so a lane's dims for k-steps 2kp and 2kp+1 are 8 adjacent ones. The four lanes of a
// fragment row then read a whole 128-byte line of a split row (32-byte loads) and 64
// contiguous bytes of a bf16 row (16-byte loads) per pair of k-steps.
__host__ __device__ constexpr int kdim(int ks, int p) { return 32 * (ks >> 1) + 8 * p + 4 * (ks & 1); }

// fp32 [rows, D] -> hi/lo bf16 rows: per 4 dims, 16 bytes {hi0..hi3, lo0..lo3}.
__global__ void split_kernel(const float4* __restrict__ src, uint4* __restrict__ dst, int64_t n4) {
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n4;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 v = src[q];
    __nv_bfloat16 h[4], l[4];
    split_bf16(v.x, h[0], l[0]);
    split_bf16(v.y, h[1], l[1]);
    split_bf16(v.z, h[2], l[2]);
    split_bf16(v.w, h[3], l[3]);
    uint4 o;
    o.x = (uint32_t)__bfloat16_as_ushort(h[0]) | ((uint32_t)__bfloat16_as_ushort(h[1]) << 16);
    o.y = (uint32_t)__bfloat16_as_ushort(h[2]) | ((uint32_t)__bfloat16_as_ushort(h[3]) << 16);
    o.z = (uint32_t)__bfloat16_as_ushort(l[0]) | ((uint32_t)__bfloat16_as_ushort(l[1]) << 16);
    o.w = (uint32_t)__bfloat16_as_ushort(l[2]) | ((uint32_t)__bfloat16_as_ushort(l[3]) << 16);
    dst[q] = o;
  }
}

// 32-byte read-only load: one fragment lane's split chunks for k-steps 2kp and 2kp+1.
__device__ __forceinline__ void ldg_pair(const uint4* a, uint4& x, uint4& y) {
  asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w), "=r"(y.x), "=r"(y.y), "=r"(y.z), "=r"(y.w)
      : "l"(a));
}

// Two-row hi/lo MMA: rows r0 (A row g) and r1 (A row g+8) of the split pyramid (always valid
// addresses); invalid rows contribute zeros and load nothing (a lane group whose row is
// invalid issues no request, so sparse row sets cost only their valid rows).
template <int KS>
__device__ __forceinline__ void mma_split_rows(float (&acc)[4], const uint4* r0, bool v0,
                                               const uint4* r1, bool v1, int p,
                                               const uint32_t (&qb)[KS][2]) {
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int kp = 0; kp < KS / 2; ++kp) {
    uint4 x0[2] = {z, z}, x1[2] = {z, z};
    if (v0) ldg_pair(r0 + 8 * kp + 2 * p, x0[0], x0[1]);
    if (v1) ldg_pair(r1 + 8 * kp + 2 * p, x1[0], x1[1]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint4 a = x0[e], c = x1[e];
      const uint32_t ahi[4] = {a.x, c.x, a.y, c.y};
      const uint32_t alo[4] = {a.z, c.z, a.w, c.w};
      mma_bf16(acc, ahi, qb[2 * kp + e][0], qb[2 * kp + e][1]);
      mma_bf16(acc, alo, qb[2 * kp + e][0], qb[2 * kp + e][1]);
    }
  }
}

// Order-preserving unsigned image of a score (after no_nan): x < y iff ordered_bits(x) <
// ordered_bits(y); -0 and +0 map to the same value, so equal scores tie on the index.
__device__ __forceinline__ uint32_t ordered_bits(float x) {
  const uint32_t u = __float_as_uint(x + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// A node's selection key: higher score first, then lower node index (the order of beats()).
__device__ __forceinline__ uint64_t node_key(float sc, int node) {
  return (static_cast<uint64_t>(ordered_bits(sc)) << 32) | (0x7fffffffu - static_cast<uint32_t>(node));
}

// Dots of a candidate's two children with the G heads (child, head), padded to 80 bytes.
struct __align__(16) CDot {
  float v[2][8];
  float pad[4];
};

// Fan-out 4: the visible grandchildren 4a .. 4a+3 at the level below the next (node span
// `span` tokens; visible when the first token is <= i) of the kept node `a` held by each lane
// (-1: none), compacted in lane order into cand. Returns their number. A node's visible
// grandchildren are a prefix of the four, so a lane's count tells them all.
__device__ __forceinline__ int expand4(int a, int64_t span, int i, int* cand, unsigned ltm) {
  int n = 0;
  if (a >= 0)
    for (int c = 0; c < 4; ++c) n += static_cast<int64_t>(4 * a + c) * span <= i ? 1 : 0;
  int pos = 0, tot = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const unsigned m = __ballot_sync(0xffffffffu, n > c);
    pos += __popc(m & ltm);
    tot += __popc(m);
  }
  for (int c = 0; c < n; ++c) cand[pos + c] = 4 * a + c;
  return tot;
}

// Causal path prefixes for stage 1, one pass before the descent: pd[l][h] = q_h . (sum of the
// keys j <= i in the ancestor of i's leaf at level l), for the levels l < LP the descent can
// score. Level 0 is the own-leaf prefix; level l adds the left sibling of the level-(l-1)
// ancestor when that ancestor is a right child. A CTA takes 16 * NW (query, head) rows of one
// KV head, all in one leaf, so the leaf's keys (staged once in shared memory) and the siblings
// on its ancestor path serve all of them; a warp takes 16 rows. Both contractions run on
// mma.sync with the rows as A (the dimension order of kdim), the keys (exact bf16 products) or
// the split sibling rows (hi and lo: fp32-accurate) as B.
__host__ __device__ constexpr int prefix_warps(int G) { return G >= 2 ? 8 : 4; }   // <= 64 queries per CTA
constexpr int kMaxSib = 25;   // N < 2^31 tokens in leaves of C = 64: at most 26 levels, 25 siblings
constexpr int kFirstChildren = 64;   // children of the first scored level: at most 4K (K <= 16)

template <int D, int G>
__global__ void __launch_bounds__(prefix_warps(G) * 32, G >= 8 ? 4 : 3)   // CTAs per SM: registers, then shared memory
route_prefix_kernel(Dims s, Geo geo, int LP, const __nv_bfloat16* __restrict__ Q,
                    const __nv_bfloat16* __restrict__ Kt, const uint4* __restrict__ spl, float* __restrict__ pd,
                    float* __restrict__ cfirst) {
  constexpr int KS = D / 16, RQ = D / 4, QW = 16 / G, NW = prefix_warps(G), CH = D / 8;
  __shared__ __align__(16) uint4 s_key[64 * CH];                // the leaf's keys, [key][chunk ^ (key & 7)]
  __shared__ __align__(16) uint4 s_sib[kMaxSib * 2 * CH];     // split sibling rows, [level][chunk ^ (level & 7)]
  __shared__ float s_dot[NW][16][kMaxSib];                     // [row][level]: sibling dots
  __shared__ float s_p0[NW][16];                               // [row]: own-leaf prefix dots
  extern __shared__ __align__(16) uint4 s_ch[];                // first-level children (split rows), when asked
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
  const int b = blockIdx.z, kv = blockIdx.y;
  const int ic = blockIdx.x * NW * QW;                          // the CTA's first query
  const int i0 = ic + warp * QW;                                // the warp's first query
  const int ti = ic / s.C, L = geo.n_levels;
  const int kvk = kv / s.kvr;
  const int64_t head = static_cast<int64_t>(b) * s.Hkv + kv;
  const uint4* spl_h = spl + (static_cast<int64_t>(b) * s.Hkv_r + kvk) * geo.nodes * RQ;
  const int64_t j0 = static_cast<int64_t>(ti) * s.C;

  // A fragments: rows g and g + 8 (query i0 + r / G, head r % G); rows past N read row ic.
  // Issued first: their latency overlaps the staging below.
  const int qa = i0 + g / G, qb = i0 + (g + 8) / G;
  const __nv_bfloat16* rowa =
      Q + ((static_cast<int64_t>(b) * s.N + (qa < s.N ? qa : ic)) * s.Hq + kv * G + g % G) * D;
  const __nv_bfloat16* rowb =
      Q + ((static_cast<int64_t>(b) * s.N + (qb < s.N ? qb : ic)) * s.Hq + kv * G + (g + 8) % G) * D;
  uint32_t qf[KS][4];
#pragma unroll
  for (int kp = 0; kp < KS / 2; ++kp) {
    const uint4 x0 = ldg_u4(rowa + kdim(2 * kp, p)), x1 = ldg_u4(rowb + kdim(2 * kp, p));
    qf[2 * kp][0] = x0.x; qf[2 * kp][1] = x1.x; qf[2 * kp][2] = x0.y; qf[2 * kp][3] = x1.y;
    qf[2 * kp + 1][0] = x0.z; qf[2 * kp + 1][1] = x1.z; qf[2 * kp + 1][2] = x0.w; qf[2 * kp + 1][3] = x1.w;
  }

  // the first scored level (g = 2, when asked): its candidates are all visible nodes of the
  // level, the same for every query of the leaf; their children are the nch first nodes of the
  // level below
  int lam0 = 0, nch = 0;
  if (cfirst != nullptr) {
    for (int lam = L - 2; lam >= 1; --lam)
      if ((ti >> lam) + 1 > s.K) {
        lam0 = lam;
        break;
      }
    if (lam0 >= 1) nch = (ti >> (lam0 - 1)) + 1;               // <= 4K <= kFirstChildren
  }

  // staged in shared memory for all warps: the keys j0 .. (the CTA's last query), the left
  // siblings on the leaf's ancestor path (a level whose ancestor is a left child is zeros) and
  // the first-level children, 16-byte chunks swizzled by row
  {
    for (int e = threadIdx.x; e < nch * 2 * CH; e += NW * 32) {
      const int r = e / (2 * CH), c = e - r * 2 * CH;
      tc::cp_async16(tc::su32(&s_ch[r * 2 * CH + (c ^ (r & 7))]), spl_h + (geo.off[lam0 - 1] + r) * RQ + c, true);
    }
    const int nkc = min(ic + NW * QW - 1, s.N - 1) - static_cast<int>(j0) + 1;
    for (int e = threadIdx.x; e < nkc * CH; e += NW * 32) {
      const int key = e / CH, c = e - key * CH;
      tc::cp_async16(tc::su32(&s_key[key * CH + (c ^ (key & 7))]),
                     Kt + ((static_cast<int64_t>(b) * s.N + j0 + key) * s.Hkv_r + kvk) * D + c * 8, true);
    }
    for (int e = threadIdx.x; e < (L - 1) * 2 * CH; e += NW * 32) {
      const int l = e / (2 * CH), c = e - l * 2 * CH;
      const bool sv = (ti >> l) & 1;
      tc::cp_async16(tc::su32(&s_sib[l * 2 * CH + (c ^ (l & 7))]),
                     spl_h + (sv ? (geo.off[l] + (ti >> l) - 1) * RQ + c : 0), sv);
    }
    tc::cp_async_commit();
    tc::cp_async_wait<0>();
    __syncthreads();
  }
  if (i0 >= s.N) return;                   // no block-wide barriers below

  // own leaf: keys j0 .. (the warp's last query), 8 per tile (B column = key, read from shared
  // memory); a row adds the keys up to its query
  const int nk = min(i0 + QW - 1, s.N - 1) - static_cast<int>(j0) + 1;
  const int la = qa - static_cast<int>(j0), lb = qb - static_cast<int>(j0);   // key n counts iff n <= la
  float pa = 0.f, pb = 0.f;
  for (int nt = 0; nt * 8 < nk; ++nt) {
    const int n = nt * 8 + g;                 // this lane's key; n & 7 == g
    const bool kvld = n < nk;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {     // chunk 4 kp + p holds dims kdim(2 kp, p) .. + 7
      const uint4 x = kvld ? s_key[n * CH + ((4 * kp + p) ^ g)] : make_uint4(0, 0, 0, 0);
      mma_bf16(acc, qf[2 * kp], x.x, x.y);
      mma_bf16(acc, qf[2 * kp + 1], x.z, x.w);
    }
    const int c0 = nt * 8 + 2 * p;            // this lane's two keys (columns 2p, 2p + 1)
    pa += (c0 <= la ? acc[0] : 0.f) + (c0 + 1 <= la ? acc[1] : 0.f);
    pb += (c0 <= lb ? acc[2] : 0.f) + (c0 + 1 <= lb ? acc[3] : 0.f);
  }
  pa += __shfl_xor_sync(0xffffffffu, pa, 1);
  pa += __shfl_xor_sync(0xffffffffu, pa, 2);
  pb += __shfl_xor_sync(0xffffffffu, pb, 1);
  pb += __shfl_xor_sync(0xffffffffu, pb, 2);
  if (p == 0) {
    s_p0[warp][g] = pa;
    s_p0[warp][g + 8] = pb;
  }

  // left siblings on the path, 8 levels per tile (B column = level l): the node left of the
  // level-l ancestor when that ancestor is a right child, else zero
  for (int st = 0; st * 8 < L - 1; ++st) {
    const int l = st * 8 + g;                 // l & 7 == g
    const bool sv = l < L - 1;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {     // chunks 8 kp + 2p, + 1: dims kdim(2 kp, p) .. + 7
      uint4 y0 = make_uint4(0, 0, 0, 0), y1 = y0;
      if (sv) {
        y0 = s_sib[l * 2 * CH + ((8 * kp + 2 * p) ^ g)];
        y1 = s_sib[l * 2 * CH + ((8 * kp + 2 * p + 1) ^ g)];
      }
      mma_bf16(acc, qf[2 * kp], y0.x, y0.y);           // hi
      mma_bf16(acc, qf[2 * kp], y0.z, y0.w);           // lo
      mma_bf16(acc, qf[2 * kp + 1], y1.x, y1.y);
      mma_bf16(acc, qf[2 * kp + 1], y1.z, y1.w);
    }
    const int c0 = st * 8 + 2 * p;            // levels c0, c0 + 1 (none past kMaxSib - 1)
    if (c0 < kMaxSib) {
      s_dot[warp][g][c0] = acc[0];
      s_dot[warp][g + 8][c0] = acc[2];
    }
    if (c0 + 1 < kMaxSib) {
      s_dot[warp][g][c0 + 1] = acc[1];
      s_dot[warp][g + 8][c0 + 1] = acc[3];
    }
  }
  // the first scored level's child dots, into cfirst[unit][child][h] (the path child's full
  // dot too: the descent replaces it with the causal prefix); two tiles of 8 children at a
  // time, so that two independent MMA chains overlap
  for (int nt = 0; nt * 8 < nch; nt += 2) {
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int n = (nt + t) * 8 + g;       // n & 7 == g
        uint4 y0 = make_uint4(0, 0, 0, 0), y1 = y0;
        if (n < nch) {
          y0 = s_ch[n * 2 * CH + ((8 * kp + 2 * p) ^ g)];
          y1 = s_ch[n * 2 * CH + ((8 * kp + 2 * p + 1) ^ g)];
        }
        mma_bf16(acc[t], qf[2 * kp], y0.x, y0.y);
        mma_bf16(acc[t], qf[2 * kp], y0.z, y0.w);
        mma_bf16(acc[t], qf[2 * kp + 1], y1.x, y1.y);
        mma_bf16(acc[t], qf[2 * kp + 1], y1.z, y1.w);
      }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int c0 = (nt + t) * 8 + 2 * p;
      if (qa < s.N) {
        float* o = cfirst + ((head * s.N + qa) * kFirstChildren + c0) * G + g % G;
        if (c0 < nch) o[0] = acc[t][0];
        if (c0 + 1 < nch) o[G] = acc[t][1];
      }
      if (qb < s.N) {
        float* o = cfirst + ((head * s.N + qb) * kFirstChildren + c0) * G + (g + 8) % G;
        if (c0 < nch) o[0] = acc[t][2];
        if (c0 + 1 < nch) o[G] = acc[t][3];
      }
    }
  }
  __syncwarp();
  // lane r < 16: row r's prefix over the levels, written as pd[unit][l][h]
  if (lane < 16) {
    const int qi = i0 + lane / G, h = lane % G;
    if (qi < s.N) {
      float v = s_p0[warp][lane];
      float* out = pd + (head * s.N + qi) * LP * G + h;
      for (int l = 0; l < LP; ++l) {
        out[l * G] = v;
        if (l < L - 1) v += s_dot[warp][lane][l];
      }
    }
  }
}

// MC: the most candidates a level can hold (2K rounded up to 32 or 64); the smaller size lets
// more CTAs share an SM. MEAN: the PISA-1 ablation -- every block, leaves included, is scored
// by s q . (its causal key sum) / (its visible key count), summed over the G heads; the leaf
// candidates' scores go to cscore_out (same layout as cand_out) for the final top-K.
template <int D, int MC, bool MEAN>
__global__ void __launch_bounds__(kWarps * 32)
route_kernel(Dims s, Geo geo, int LP, const __nv_bfloat16* __restrict__ Q, const float* __restrict__ pd,
             const float* __restrict__ cfirst, const uint4* __restrict__ spl, int32_t* __restrict__ cand_out,
             float* __restrict__ cscore_out) {
  constexpr int KS = D / 16;
  constexpr int RQ = D / 4;     // uint4 chunks per split row
  __shared__ int s_cand[kWarps][MC];
  __shared__ int s_kept[kWarps][MC / 2];
  __shared__ float s_sc[kWarps][MC];
  __shared__ uint64_t s_key[kWarps][MC];   // node_key of every scored candidate
  __shared__ __align__(16) float s_pd[kWarps][PISA_MAX_LEVELS][8];   // [level][head]: path prefixes
  // dots of every candidate's two children (q . key sum, per head), two level buffers
  // (80-byte rows: a lane per candidate reads and writes its row with 16-byte accesses, and a
  // 20-word stride spreads 8 consecutive rows over all 32 banks)
  __shared__ CDot s_cdot[kWarps][2][MC];
  __shared__ int s_kslot[kWarps][MC / 2];   // candidate slot each kept node came from
  __shared__ int s_par[kWarps][MC];         // 2 * (kept slot of the parent) + which child

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
  const int b = blockIdx.z, kv = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  if (i >= s.N) return;                   // no block-wide barriers below
  const int G = s.G, Ksel = s.K, C = s.C, W = s.g * s.K;
  const int ti = i / C;
  const int L = geo.n_levels;
  const int64_t head = static_cast<int64_t>(b) * s.Hkv + kv;            // selection unit
  const int kvk = kv / s.kvr;                                           // its KV head
  const uint4* spl_h = spl + (static_cast<int64_t>(b) * s.Hkv_r + kvk) * geo.nodes * RQ;

  // q of the G heads as MMA B fragments (column n = head g; heads >= G are zero).
  uint32_t qb[KS][2];
  {
    const __nv_bfloat16* qrow =
        Q + ((static_cast<int64_t>(b) * s.N + i) * s.Hq + kv * G + min(g, G - 1)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint2 v = g < G ? ldg_u2(qrow + kdim(ks, p)) : make_uint2(0, 0);
      qb[ks][0] = v.x;
      qb[ks][1] = v.y;
    }
  }

  // the causal path prefix dots of the levels the descent scores, from the prefix pass
  {
    const float* src = pd + (head * s.N + i) * LP * G;
    for (int e = lane; e < LP * 8; e += 32) {
      const int l = e >> 3, h = e & 7;
      s_pd[warp][l][h] = h < G ? src[l * G + h] : 0.f;
    }
  }
  __syncwarp();

  int* cand = s_cand[warp];
  int* kept = s_kept[warp];
  float* sc = s_sc[warp];
  uint64_t* key = s_key[warp];
  int nkept = 1;
  if (lane == 0) kept[0] = 0;
  __syncwarp();

  const unsigned ltm = lanemask_lt();
  // Right-child shortcut: the key sum of a node is the sum of its children's, so once a
  // level has been scored the dot of every next candidate c is known, and for c's children
  // only the left one needs loading: q.S(2c+1) = q.S(c) - q.S(2c). The node on the query's
  // path uses its causal prefix dot instead.
  bool have_pdot = false;   // dots of the current candidates are known (previous level scored)
  bool scored = false;      // a level has been scored
  int cur = 0;              // s_cdot buffer written by the previous scored level
  int* kslot = s_kslot[warp];
  // Visited levels: L-1 (the top node), then one level down per step (g = 2) or two (g = 4,
  // the candidates being the kept nodes' visible grandchildren), down to the leaves; the last
  // step is one level when two would pass them. Intermediate levels are scored here.
  const int step = s.g == 4 ? 2 : 1;
  int lp = L - 1;
  for (int lam = lp - step; lam >= 1; lp = lam, lam -= step) {
    // candidates at level lam: visible children of the kept nodes of level lam+1 (g = 2: each
    // records its kept slot and which child, for the parent-dot shortcut), or visible
    // grandchildren of the kept nodes of level lam+2 (g = 4: both children scored directly)
    const int64_t span = static_cast<int64_t>(C) << lam;
    int nc;
    if (step == 1) {
      const int a = lane < nkept ? kept[lane] : -1;
      const bool c0 = a >= 0;
      const bool c1 = a >= 0 && static_cast<int64_t>(2 * a + 1) * span <= i;
      const unsigned m0 = __ballot_sync(0xffffffffu, c0), m1 = __ballot_sync(0xffffffffu, c1);
      const int pos = __popc(m0 & ltm) + __popc(m1 & ltm);
      __syncwarp();
      if (c0) { cand[pos] = 2 * a; s_par[warp][pos] = lane * 2 + 0; }
      if (c1) { cand[pos + 1] = 2 * a + 1; s_par[warp][pos + 1] = lane * 2 + 1; }
      nc = __popc(m0) + __popc(m1);
    } else {
      nc = expand4(lane < nkept ? kept[lane] : -1, span, i, cand, ltm);
      have_pdot = false;
    }
    __syncwarp();
    if (nc <= Ksel) {
      if (lane < nc) kept[lane] = cand[lane];
      nkept = nc;
      have_pdot = false;
      __syncwarp();
      continue;
    }
    const int64_t cspan = static_cast<int64_t>(C) << (lam - 1);
    const int pathc = ti >> (lam - 1);
    const int nxt = cur ^ 1;
    // the first scored level's child dots come from the prefix pass (g = 2); a later level
    // without parent dots (kept whole after a scored one) loads its own
    const bool pre = !scored && step == 1 && cfirst != nullptr;
    CDot* cd = s_cdot[warp][nxt];
    const CDot* pdots = s_cdot[warp][cur];
    const int64_t loff = geo.off[lam - 1];
    // 1. Child dots by MMA (lane (g, p): heads 2p, 2p+1 of A rows g and g + 8) into cd[slot]:
    //    the left child of 16 candidates per tile when the parents' dots are known, else both
    //    children of 8 candidates per tile. The path child is not loaded (its dot is the
    //    causal prefix, set below).
    if (have_pdot) {
      for (int mt = 0; mt * 16 < nc; ++mt) {
        const int csa = mt * 16 + g, csb = csa + 8;
        const int ca = csa < nc ? cand[csa] : -1, cb = csb < nc ? cand[csb] : -1;
        const bool la = ca >= 0 && 2 * ca != pathc, lb = cb >= 0 && 2 * cb != pathc;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4* ra = spl_h + (la ? (loff + 2 * ca) * RQ : 0);
        const uint4* rb = spl_h + (lb ? (loff + 2 * cb) * RQ : 0);
        mma_split_rows<KS>(acc, ra, la, rb, lb, p, qb);
        if (csa < nc) *reinterpret_cast<float2*>(&cd[csa].v[0][2 * p]) = make_float2(acc[0], acc[1]);
        if (csb < nc) *reinterpret_cast<float2*>(&cd[csb].v[0][2 * p]) = make_float2(acc[2], acc[3]);
      }
    } else if (!pre) {
      for (int mt = 0; mt * 8 < nc; ++mt) {
        const int cs = mt * 8 + g;
        const int c = cs < nc ? cand[cs] : -1;
        const bool v0 = c >= 0 && 2 * c != pathc;
        const bool v1 = c >= 0 && 2 * c + 1 != pathc && static_cast<int64_t>(2 * c + 1) * cspan <= i;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4* r0 = spl_h + (v0 ? (loff + 2 * c) * RQ : 0);
        const uint4* r1 = spl_h + (v1 ? (loff + 2 * c + 1) * RQ : 0);
        mma_split_rows<KS>(acc, r0, v0, r1, v1, p, qb);
        if (cs < nc) {
          *reinterpret_cast<float2*>(&cd[cs].v[0][2 * p]) = make_float2(acc[0], acc[1]);
          *reinterpret_cast<float2*>(&cd[cs].v[1][2 * p]) = make_float2(acc[2], acc[3]);
        }
      }
    }
    __syncwarp();
    // 2. One lane per candidate: both children's dots for every head (right = parent - left
    //    when only the left was loaded; the path child takes the causal prefix dot), written
    //    back for the next level, then the score = sum over the G heads of the LSE of the
    //    visible children's mean scores (MEAN: of the candidate's own mean).
    // Key counts: a visible child off the query's path ends before i, so it is full (cspan
    // keys); the path child holds the keys up to i. Scale factors s / count, once per level.
    const float cnt_path = static_cast<float>(i - static_cast<int64_t>(pathc) * cspan + 1);
    const float f_full = s.scale / static_cast<float>(cspan), f_path = s.scale / cnt_path;
    for (int cs = lane; cs < nc; cs += 32) {
      const int c = cand[cs];
      const int ch0 = 2 * c, ch1 = 2 * c + 1;
      const bool rv = static_cast<int64_t>(ch1) * cspan <= i;
      float lv[8], rw[8];
      if (pre) {
        const float* cf = cfirst + ((head * s.N + i) * kFirstChildren + ch0) * G;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          lv[h] = h < G ? cf[h] : 0.f;
          rw[h] = h < G && rv ? cf[G + h] : 0.f;
        }
      } else {
        const float4 a = *reinterpret_cast<const float4*>(&cd[cs].v[0][0]);
        const float4 b = *reinterpret_cast<const float4*>(&cd[cs].v[0][4]);
        lv[0] = a.x; lv[1] = a.y; lv[2] = a.z; lv[3] = a.w; lv[4] = b.x; lv[5] = b.y; lv[6] = b.z; lv[7] = b.w;
      }
      if (pre) {
        // both children from the prefix pass (above)
      } else if (have_pdot) {
        const int ps = s_par[warp][cs];
        const float* par = pdots[kslot[ps >> 1]].v[ps & 1];
        const float4 a = *reinterpret_cast<const float4*>(par), b = *reinterpret_cast<const float4*>(par + 4);
        rw[0] = a.x - lv[0]; rw[1] = a.y - lv[1]; rw[2] = a.z - lv[2]; rw[3] = a.w - lv[3];
        rw[4] = b.x - lv[4]; rw[5] = b.y - lv[5]; rw[6] = b.z - lv[6]; rw[7] = b.w - lv[7];
      } else {
        const float4 a = *reinterpret_cast<const float4*>(&cd[cs].v[1][0]);
        const float4 b = *reinterpret_cast<const float4*>(&cd[cs].v[1][4]);
        rw[0] = a.x; rw[1] = a.y; rw[2] = a.z; rw[3] = a.w; rw[4] = b.x; rw[5] = b.y; rw[6] = b.z; rw[7] = b.w;
      }
      float f0 = f_full, f1 = f_full;
      if (ch0 == pathc || ch1 == pathc) {
        const float* pd = s_pd[warp][lam - 1];
        const float4 a = *reinterpret_cast<const float4*>(pd), b = *reinterpret_cast<const float4*>(pd + 4);
        const float pv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (ch0 == pathc) {
          f0 = f_path;
#pragma unroll
          for (int h = 0; h < 8; ++h) lv[h] = pv[h];
        } else {
          f1 = f_path;
#pragma unroll
          for (int h = 0; h < 8; ++h) rw[h] = pv[h];
        }
      }
      *reinterpret_cast<float4*>(&cd[cs].v[0][0]) = make_float4(lv[0], lv[1], lv[2], lv[3]);
      *reinterpret_cast<float4*>(&cd[cs].v[0][4]) = make_float4(lv[4], lv[5], lv[6], lv[7]);
      *reinterpret_cast<float4*>(&cd[cs].v[1][0]) = make_float4(rw[0], rw[1], rw[2], rw[3]);
      *reinterpret_cast<float4*>(&cd[cs].v[1][4]) = make_float4(rw[4], rw[5], rw[6], rw[7]);
      float score = 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h >= G) break;
        float l;
        if constexpr (MEAN) {   // the node's own mean key: (left + right sums) / (their counts)
          const float cnt0 = ch0 == pathc ? cnt_path : static_cast<float>(cspan);
          const float cnt1 = ch1 == pathc ? cnt_path : static_cast<float>(cspan);
          l = rv ? (lv[h] + rw[h]) * (s.scale / (cnt0 + cnt1)) : lv[h] * f0;
        } else {
          const float x0 = lv[h] * f0;
          if (rv) {     // LSE of two terms: max + log(1 + exp(-|difference|))
            const float x1 = rw[h] * f1;
            l = fmaxf(x0, x1) + __logf(1.f + __expf(-fabsf(x0 - x1)));
          } else {
            l = x0;
          }
        }
        score += l;
      }
      key[cs] = node_key(no_nan(score), c);
    }
    __syncwarp();
    for (int s2 = lane; s2 < nc; s2 += 32) {
      const uint64_t my = key[s2];
      const int mi = cand[s2];
      int rank = 0;
#pragma unroll 8
      for (int o = 0; o < nc; ++o) rank += key[o] > my ? 1 : 0;
      if (rank < Ksel) { kept[rank] = mi; kslot[rank] = s2; }
    }
    nkept = Ksel;
    have_pdot = true;
    scored = true;
    cur = nxt;
    __syncwarp();
  }

  // leaf candidates: visible descendants of the kept level-lp nodes (children when lp = 1,
  // grandchildren when lp = 2), or the single leaf
  int32_t* out = cand_out + ((head * s.N) + i) * W;
  int nc = 1;
  if (L == 1) {
    if (lane == 0) cand[0] = 0;
  } else if (lp == 1) {
    const int a = lane < nkept ? kept[lane] : -1;
    const bool c0 = a >= 0;
    const bool c1 = a >= 0 && static_cast<int64_t>(2 * a + 1) * C <= i;
    const unsigned m0 = __ballot_sync(0xffffffffu, c0), m1 = __ballot_sync(0xffffffffu, c1);
    const int pos = __popc(m0 & ltm) + __popc(m1 & ltm);
    nc = __popc(m0) + __popc(m1);
    __syncwarp();
    if (c0) cand[pos] = 2 * a;
    if (c1) cand[pos + 1] = 2 * a + 1;
  } else {
    __syncwarp();
    nc = expand4(lane < nkept ? kept[lane] : -1, static_cast<int64_t>(C), i, cand, ltm);
  }
  __syncwarp();
  if constexpr (MEAN) {
    // PISA-1 leaf scores: s q . S(0,t) / count; the query's own leaf uses its causal prefix dot
    const float pd0 = s_pd[warp][0][2 * p], pd1 = s_pd[warp][0][2 * p + 1];
    auto leaf_part = [&](int t, float d0, float d1) {
      if (t < 0) return 0.f;
      float cnt;
      if (t == ti) {
        d0 = pd0;
        d1 = pd1;
        cnt = static_cast<float>(i - t * C + 1);
      } else {
        cnt = static_cast<float>(min(static_cast<int64_t>(t + 1) * C, static_cast<int64_t>(s.N)) -
                                 static_cast<int64_t>(t) * C);
      }
      const float k = s.scale / cnt;
      return (2 * p < G ? d0 * k : 0.f) + (2 * p + 1 < G ? d1 * k : 0.f);
    };
    for (int mt = 0; mt * 16 < nc; ++mt) {
      const int csa = mt * 16 + g, csb = csa + 8;
      const int ta = csa < nc ? cand[csa] : -1, tb = csb < nc ? cand[csb] : -1;
      const bool la = ta >= 0 && ta != ti, lb = tb >= 0 && tb != ti;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint4* ra = spl_h + (la ? (geo.off[0] + ta) * RQ : 0);
      const uint4* rb = spl_h + (lb ? (geo.off[0] + tb) * RQ : 0);
      mma_split_rows<KS>(acc, ra, la, rb, lb, p, qb);
      float pa = leaf_part(ta, acc[0], acc[1]), pb = leaf_part(tb, acc[2], acc[3]);
      pa += __shfl_xor_sync(0xffffffffu, pa, 1);
      pa += __shfl_xor_sync(0xffffffffu, pa, 2);
      pb += __shfl_xor_sync(0xffffffffu, pb, 1);
      pb += __shfl_xor_sync(0xffffffffu, pb, 2);
      if (p == 0 && csa < nc) sc[csa] = no_nan(pa);
      if (p == 0 && csb < nc) sc[csb] = no_nan(pb);
    }
    __syncwarp();
    float* outs = cscore_out + ((head * s.N) + i) * W;
    for (int q = lane; q < W; q += 32) outs[q] = q < nc ? sc[q] : neg_inf();
  }
  for (int q = lane; q < W; q += 32) out[q] = q < nc ? cand[q] : -1;
}

// ---------------------------------------------------------------------------- finish
// One warp per (b, KV head, query): top K of the <= W (<= 64) candidate scores, output
// ascending. Lane l holds candidates l and l + 32 in registers; ranks and output positions
// come from warp shuffles.
// When the status word carries PISA_STATUS_TIMEOUT (a bounded wait of the leaf stage gave up,
// so candidate scores may be missing or stale) every output slot is poisoned instead:
// idx = -1, score = head_lse = NaN.
template <int J>    // candidates per lane: 1 (W <= 32) or 2 (W <= 64)
__global__ void __launch_bounds__(kWarps * 32)
topk_kernel(int64_t units, int W, int Ksel, int N, int G, const int32_t* __restrict__ cand,
            const float* __restrict__ csc, const float* __restrict__ chead, int32_t* __restrict__ idx,
            float* __restrict__ score, float* __restrict__ head_lse, const int32_t* __restrict__ status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t u = blockIdx.x * static_cast<int64_t>(kWarps) + warp;
  if (u >= units) return;
  const int64_t hrow = (u / N) * G * N + u % N;
  if (*status & PISA_STATUS_TIMEOUT) {
    const float nan = __int_as_float(0x7fc00000);
    for (int q = lane; q < Ksel; q += 32) {
      idx[u * Ksel + q] = -1;
      if (score) score[u * Ksel + q] = nan;
      if (head_lse)
        for (int h = 0; h < G; ++h) head_lse[(hrow + static_cast<int64_t>(h) * N) * Ksel + q] = nan;
    }
    return;
  }
  int ci[2] = {-1, -1};
  float cs[2] = {neg_inf(), neg_inf()};
  for (int j = 0; j < J; ++j) {
    const int q = lane + 32 * j;
    if (q < W) {
      ci[j] = cand[u * W + q];
      if (ci[j] >= 0) cs[j] = no_nan(csc[u * W + q]);
    }
  }
  int rank[2] = {0, 0};
#pragma unroll
  for (int jj = 0; jj < J; ++jj)
#pragma unroll 8
    for (int o = 0; o < 32; ++o) {
      const float so = __shfl_sync(0xffffffffu, cs[jj], o);
      const int io = __shfl_sync(0xffffffffu, ci[jj], o);
      if (io < 0) continue;
#pragma unroll
      for (int j = 0; j < J; ++j) rank[j] += beats(so, io, cs[j], ci[j]) ? 1 : 0;
    }
  bool keep[2] = {false, false};
  int pos[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < J; ++j) keep[j] = ci[j] >= 0 && rank[j] < Ksel;
#pragma unroll
  for (int jj = 0; jj < J; ++jj)
#pragma unroll 8
    for (int o = 0; o < 32; ++o) {
      const int io = __shfl_sync(0xffffffffu, keep[jj] ? ci[jj] : -1, o);
      if (io < 0) continue;
#pragma unroll
      for (int j = 0; j < J; ++j) pos[j] += io < ci[j] ? 1 : 0;
    }
  const int nk = __popc(__ballot_sync(0xffffffffu, keep[0])) + __popc(__ballot_sync(0xffffffffu, keep[1]));
  // unit u = (b*Hkv + kv)*N + i -> head_lse rows (b*Hq + kv*G + h)*N + i
  const int64_t hrow0 = hrow;
  for (int j = 0; j < J; ++j) {
    if (!keep[j]) continue;
    idx[u * Ksel + pos[j]] = ci[j];
    if (score) score[u * Ksel + pos[j]] = cs[j];
    if (head_lse) {
      const float* src = chead + (u * W + lane + 32 * j) * G;
      for (int h = 0; h < G; ++h) head_lse[(hrow0 + static_cast<int64_t>(h) * N) * Ksel + pos[j]] = src[h];
    }
  }
  for (int q = nk + lane; q < Ksel; q += 32) {
    idx[u * Ksel + q] = -1;
    if (score) score[u * Ksel + q] = neg_inf();
    if (head_lse)
      for (int h = 0; h < G; ++h) head_lse[(hrow0 + static_cast<int64_t>(h) * N) * Ksel + q] = neg_inf();
  }
}

// One thread per (b, KV head, query) for W <= 32: the warp version above spends most of its
// time in shuffles (two per candidate and lane). Here a CTA stages its units' candidate rows
// in shared memory with coalesced loads, and every thread sorts its own row in registers with
// two bitonic networks: the (score, leaf) pairs by the selection order, then the first K of
// them by leaf index. A pair is one 64-bit key, the order-preserving bits of the score above
// the complemented leaf index (lower leaf wins a tie) and the candidate slot; an empty slot
// is key 0, below every candidate. Same outputs and poisoning as the warp version.
#ifndef PISA_TOPK_THREAD
#define PISA_TOPK_THREAD 1
#endif
constexpr int kTopkUnits = 128;   // units (threads) per CTA
constexpr uint32_t kLeafMask = (1u << 26) - 1;   // leaf indices < 2^26 (N < 2^32 tokens of C = 64)


template <typename T>
__device__ __forceinline__ void bitonic32(T (&a)[32], bool descending) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const bool first_high = ((i & k) == 0) == descending;   // a[i] should end up the larger
          const T x = a[i], y = a[l];
          const bool sw = first_high ? x < y : x > y;
          a[i] = sw ? y : x;
          a[l] = sw ? x : y;
        }
      }
}

__global__ void __launch_bounds__(kTopkUnits)
topk_thread_kernel(int64_t units, int W, int Ksel, int N, int G, const int32_t* __restrict__ cand,
                   const float* __restrict__ csc, const float* __restrict__ chead, int32_t* __restrict__ idx,
                   float* __restrict__ score, float* __restrict__ head_lse, const int32_t* __restrict__ status) {
  __shared__ int32_t s_c[kTopkUnits * 33];
  __shared__ float s_s[kTopkUnits * 33];
  const int tid = threadIdx.x;
  const int64_t u0 = blockIdx.x * static_cast<int64_t>(kTopkUnits);
  const int nu = static_cast<int>(min(static_cast<int64_t>(kTopkUnits), units - u0));
  const int stride = W | 1;                  // odd row stride: a thread's row reads are conflict-free
  const bool timeout = (*status & PISA_STATUS_TIMEOUT) != 0;
  if (!timeout) {
    for (int e = tid; e < nu * W; e += kTopkUnits) {
      const int r = e / W, c = e - r * W;
      s_c[r * stride + c] = cand[u0 * W + e];
      s_s[r * stride + c] = csc[u0 * W + e];
    }
  }
  __syncthreads();
  if (timeout) {
    if (tid >= nu) return;
    const int64_t u = u0 + tid;
    const int64_t hrow = (u / N) * G * N + u % N;    // head_lse row of head 0
    const float nan = __int_as_float(0x7fc00000);
    for (int q = 0; q < Ksel; ++q) {
      idx[u * Ksel + q] = -1;
      if (score) score[u * Ksel + q] = nan;
      if (head_lse)
        for (int h = 0; h < G; ++h) head_lse[(hrow + static_cast<int64_t>(h) * N) * Ksel + q] = nan;
    }
    return;
  }
  if (tid < nu) {
    uint64_t key[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      key[j] = 0;
      if (j < W) {
        const int c = s_c[tid * stride + j];
        if (c >= 0)
          key[j] = (static_cast<uint64_t>(ordered_bits(no_nan(s_s[tid * stride + j]))) << 32) |
                   ((kLeafMask - static_cast<uint32_t>(c)) << 6) | static_cast<uint32_t>(j);
      }
    }
    bitonic32(key, true);
    // the first K non-empty keys, re-keyed as (leaf, slot) and sorted by leaf; the rest last
    uint32_t k2[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool keep = j < Ksel && key[j] != 0;
      const uint32_t lo = static_cast<uint32_t>(key[j]);
      k2[j] = keep ? (((kLeafMask - (lo >> 6)) << 6) | (lo & 63u)) : 0xffffffffu;
    }
    bitonic32(k2, false);
    // the thread's own row, overwritten in place: slot q < K holds (leaf << 6 | source slot)
    // or -1, and the score (read before any write: a source slot may lie below q)
    float sq[32];
#pragma unroll
    for (int q = 0; q < 32; ++q)
      sq[q] = q < Ksel && k2[q] != 0xffffffffu ? no_nan(s_s[tid * stride + (k2[q] & 63u)]) : neg_inf();
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      if (q >= Ksel) break;
      s_c[tid * stride + q] = k2[q] == 0xffffffffu ? -1 : static_cast<int32_t>(k2[q]);
      s_s[tid * stride + q] = sq[q];
    }
  }
  __syncthreads();
  // coalesced stores: the CTA's units are consecutive, so its idx / score rows are one range,
  // and per head its head_lse rows are one range within each (batch, KV head)
  for (int e = tid; e < nu * Ksel; e += kTopkUnits) {
    const int t = e / Ksel, q = e - t * Ksel;
    const int32_t v = s_c[t * stride + q];
    idx[u0 * Ksel + e] = v < 0 ? -1 : (v >> 6);
    if (score) score[u0 * Ksel + e] = s_s[t * stride + q];
  }
  if (head_lse) {
    // a lane reads one kept candidate's G per-head terms (one contiguous row) and writes them
    // to the G head rows: per head, the warp's stores are consecutive
    for (int e = tid; e < nu * Ksel; e += kTopkUnits) {
      const int t = e / Ksel, q = e - t * Ksel;
      const int64_t u = u0 + t;
      const int32_t v = s_c[t * stride + q];
      float hv[8];
      const float* src = chead + (u * W + (v & 63)) * G;
      if (v >= 0 && G % 4 == 0) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(src));
        hv[0] = a.x; hv[1] = a.y; hv[2] = a.z; hv[3] = a.w;
        if (G == 8) {
          const float4 c = __ldg(reinterpret_cast<const float4*>(src) + 1);
          hv[4] = c.x; hv[5] = c.y; hv[6] = c.z; hv[7] = c.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < 8; ++h) hv[h] = v >= 0 && h < G ? src[h] : neg_inf();
      }
      float* dst = head_lse + ((u / N) * G * N + u % N) * Ksel + q;
#pragma unroll
      for (int h = 0; h < 8; ++h)
        if (h < G) dst[static_cast<int64_t>(h) * N * Ksel] = hv[h];
    }
  }
}

// ---------------------------------------------------------------------------- flat BSA
// One CTA per (query leaf block tq, KV head, batch), 4 warps x 16 queries. Leaf t < tq is
// scored by s * qbar . S(0,t) / C with qbar = sum_h q_h (a dot product is linear, so the
// head sum moves inside) using a 3-term bf16 split (hi*hi + hi*lo + lo*hi); the query's own
// leaf by s * sum_{j<=i} qbar . k_j / (i - tq*C + 1). Each lane keeps a streaming top-K for
// its two rows in shared memory; the four lanes of a row are merged at the end.
template <int D>
__global__ void __launch_bounds__(kWarps * 32)
flat_kernel(Dims s, Geo geo, const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
            const uint4* __restrict__ spl, int32_t* __restrict__ idx, float* __restrict__ score) {
  constexpr int KS = D / 16, RQ = D / 4;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_keep[kWarps][2 * kMaxCand];
  const int Ksel = s.K;
  // lists: [warp][row 0..1][k][lane] scores and indices
  float* ls = reinterpret_cast<float*>(smem_raw);
  int* li = reinterpret_cast<int*>(ls + kWarps * 2 * Ksel * 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
  const int tq = gridDim.x - 1 - blockIdx.x;
  const int kv = blockIdx.y, b = blockIdx.z;
  const int C = s.C, G = s.G;
  const int qbase = tq * C + warp * 16;
  if (qbase >= s.N) return;
  const int64_t head = static_cast<int64_t>(b) * s.Hkv + kv;                       // selection unit
  const int64_t head_k = static_cast<int64_t>(b) * s.Hkv_r + kv / s.kvr;           // its KV head
  const int i0 = qbase + g, i1 = qbase + g + 8;
  const bool ok0 = i0 < s.N, ok1 = i1 < s.N;

  uint32_t ahi[KS][4], alo[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    float f0[4] = {0.f, 0.f, 0.f, 0.f}, f1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int h = 0; h < G; ++h) {
      if (ok0) {
        uint2 v = ldg_u2(Q + ((static_cast<int64_t>(b) * s.N + i0) * s.Hq + kv * G + h) * D + kdim(ks, p));
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
        for (int u = 0; u < 4; ++u) f0[u] += __bfloat162float(e[u]);
      }
      if (ok1) {
        uint2 v = ldg_u2(Q + ((static_cast<int64_t>(b) * s.N + i1) * s.Hq + kv * G + h) * D + kdim(ks, p));
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
        for (int u = 0; u < 4; ++u) f1[u] += __bfloat162float(e[u]);
      }
    }
    __nv_bfloat16 h0[4], l0[4], h1[4], l1[4];
    for (int u = 0; u < 4; ++u) {
      split_bf16(f0[u], h0[u], l0[u]);
      split_bf16(f1[u], h1[u], l1[u]);
    }
    auto pk = [](__nv_bfloat16 x, __nv_bfloat16 y) {
      return (uint32_t)__bfloat16_as_ushort(x) | ((uint32_t)__bfloat16_as_ushort(y) << 16);
    };
    ahi[ks][0] = pk(h0[0], h0[1]); ahi[ks][2] = pk(h0[2], h0[3]);
    ahi[ks][1] = pk(h1[0], h1[1]); ahi[ks][3] = pk(h1[2], h1[3]);
    alo[ks][0] = pk(l0[0], l0[1]); alo[ks][2] = pk(l0[2], l0[3]);
    alo[ks][1] = pk(l1[0], l1[1]); alo[ks][3] = pk(l1[2], l1[3]);
  }

  // streaming lists
  float* L0s = ls + (warp * 2 + 0) * Ksel * 32;
  float* L1s = ls + (warp * 2 + 1) * Ksel * 32;
  int* L0i = li + (warp * 2 + 0) * Ksel * 32;
  int* L1i = li + (warp * 2 + 1) * Ksel * 32;
  int n0c = 0, n1c = 0, w0 = 0, w1 = 0;   // counts and worst slots
  auto insert = [&](float* Ls, int* Li, int& n, int& w, float sv, int iv) {
    sv = no_nan(sv);
    if (n < Ksel) {
      Ls[n * 32 + lane] = sv;
      Li[n * 32 + lane] = iv;
      if (n == 0 || beats(Ls[w * 32 + lane], Li[w * 32 + lane], sv, iv)) w = n;
      ++n;
      return;
    }
    if (!beats(sv, iv, Ls[w * 32 + lane], Li[w * 32 + lane])) return;
    Ls[w * 32 + lane] = sv;
    Li[w * 32 + lane] = iv;
    int nw = 0;
    for (int k = 1; k < Ksel; ++k)
      if (beats(Ls[nw * 32 + lane], Li[nw * 32 + lane], Ls[k * 32 + lane], Li[k * 32 + lane])) nw = k;
    w = nw;
  };

  const float inv_c = s.scale / static_cast<float>(C);
  const uint4* spl0 = spl + (head_k * geo.nodes + geo.off[0]) * RQ;
  for (int nt = 0; nt * 8 < tq; ++nt) {
    const int tl = nt * 8 + g;
    const bool vb = tl < tq;
    const uint4* row = spl0 + static_cast<int64_t>(vb ? tl : 0) * RQ;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {
      uint4 xx[2];
      ldg_pair(row + 8 * kp + 2 * p, xx[0], xx[1]);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int ks = 2 * kp + e;
        const uint4 x = vb ? xx[e] : make_uint4(0, 0, 0, 0);
        mma_bf16(acc, ahi[ks], x.x, x.y);
        mma_bf16(acc, ahi[ks], x.z, x.w);
        mma_bf16(acc, alo[ks], x.x, x.y);
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = nt * 8 + 2 * p + e;
      if (t < tq) {
        if (ok0) insert(L0s, L0i, n0c, w0, acc[e] * inv_c, t);
        if (ok1) insert(L1s, L1i, n1c, w1, acc[2 + e] * inv_c, t);
      }
    }
  }
  // own leaf tq: prefix over keys j <= i
  {
    float r0 = 0.f, r1 = 0.f;
    const int64_t kb = static_cast<int64_t>(tq) * C;
    for (int nt = 0; nt < 8; ++nt) {
      const int64_t j = kb + nt * 8 + g;
      const bool vk = j < s.N;
      const __nv_bfloat16* kr = K + ((static_cast<int64_t>(b) * s.N + (vk ? j : 0)) * s.Hkv_r + kv / s.kvr) * D;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
        const uint4 x = vk ? ldg_u4(kr + kdim(2 * kp, p)) : make_uint4(0, 0, 0, 0);
        mma_bf16(acc, ahi[2 * kp], x.x, x.y);
        mma_bf16(acc, alo[2 * kp], x.x, x.y);
        mma_bf16(acc, ahi[2 * kp + 1], x.z, x.w);
        mma_bf16(acc, alo[2 * kp + 1], x.z, x.w);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t key = kb + nt * 8 + 2 * p + e;
        if (key <= i0) r0 += acc[e];
        if (key <= i1) r1 += acc[2 + e];
      }
    }
    r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
    r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
    if (p == 0) {
      if (ok0) insert(L0s, L0i, n0c, w0, s.scale * r0 / static_cast<float>(i0 - kb + 1), tq);
      if (ok1) insert(L1s, L1i, n1c, w1, s.scale * r1 / static_cast<float>(i1 - kb + 1), tq);
    }
  }
  // pad unused list slots
  for (int k = n0c; k < Ksel; ++k) { L0s[k * 32 + lane] = neg_inf(); L0i[k * 32 + lane] = -1; }
  for (int k = n1c; k < Ksel; ++k) { L1s[k * 32 + lane] = neg_inf(); L1i[k * 32 + lane] = -1; }
  __syncwarp();

  // merge: row r (0..15) lives in lanes 4*(r&7) + {0..3}, list (r>>3); E = 4K entries
  const int E = 4 * Ksel;
  int* keep = s_keep[warp];
  for (int r = 0; r < 16; ++r) {
    const int i = qbase + r;
    if (i >= s.N) break;
    const float* Ls = ls + (warp * 2 + (r >> 3)) * Ksel * 32;
    const int* Li = li + (warp * 2 + (r >> 3)) * Ksel * 32;
    const int lbase = 4 * (r & 7);
    constexpr int kReps = (2 * kMaxCand) / 32;      // E <= 4*32 entries, 32 per pass
    int myi[kReps];
    float mys[kReps];
    for (int rep = 0; rep < kReps; ++rep) {
      const int eidx = lane + 32 * rep;
      myi[rep] = -1;
      mys[rep] = 0.f;
      if (eidx >= E) continue;
      const int ln = lbase + (eidx & 3), k = eidx >> 2;
      mys[rep] = Ls[k * 32 + ln];
      myi[rep] = Li[k * 32 + ln];
      int kept = 0;
      if (myi[rep] >= 0) {
        int rank = 0;
        for (int o = 0; o < E; ++o) {
          const int lo_ = lbase + (o & 3), ko = o >> 2;
          const int io = Li[ko * 32 + lo_];
          if (io >= 0 && beats(Ls[ko * 32 + lo_], io, mys[rep], myi[rep])) ++rank;
        }
        kept = rank < Ksel;
      }
      keep[eidx] = kept ? myi[rep] : -1;
    }
    __syncwarp();
    int nk = 0;
    for (int o = 0; o < E; ++o) nk += keep[o] >= 0 ? 1 : 0;
    int32_t* orow = idx + (head * s.N + i) * Ksel;
    float* srow = score ? score + (head * s.N + i) * Ksel : nullptr;
    for (int rep = 0; rep < kReps; ++rep) {
      const int eidx = lane + 32 * rep;
      if (eidx >= E || keep[eidx] < 0) continue;
      int pos = 0;
      for (int o = 0; o < E; ++o) pos += (keep[o] >= 0 && keep[o] < myi[rep]) ? 1 : 0;
      orow[pos] = myi[rep];
      if (srow) srow[pos] = mys[rep];
    }
    for (int q = nk + lane; q < Ksel; q += 32) {
      orow[q] = -1;
      if (srow) srow[q] = neg_inf();
    }
    __syncwarp();
  }
}

// Stage-2 grouping: query chunks of about 64 MiB of one KV head's query rows; about 4096
// (query, head) rows per work item (with the dynamic item order, longer items measured faster:
// 1.60 -> 1.53 ms at 64K, and fewer bins shorten the scans).
#ifndef PISA_LEAF_CHUNK_MIB
#define PISA_LEAF_CHUNK_MIB 64
#endif
#ifndef PISA_LEAF_ITEM_ROWS
#define PISA_LEAF_ITEM_ROWS 4096
#endif
#ifndef PISA_LEAF_PAIRS
#define PISA_LEAF_PAIRS 1
#endif
// The leaf candidates of a query come as sibling pairs (2m, 2m + 1) in adjacent slots (the
// visible children of a kept node; with g = 4 its visible grandchildren 4a .. 4a + 3 in order),
// so the leaf stage groups them by pair: a work item holds both leaves' 128 keys and gathers each
// query row once for the two of them.
GroupPlan leaf_plan(const Dims& s) {
  const int64_t per_query = static_cast<int64_t>(s.G) * s.d * 2;
  return make_group_plan(s, s.g * s.K, (int64_t(PISA_LEAF_CHUNK_MIB) << 20) / per_query, PISA_LEAF_ITEM_ROWS / s.G,
                         PISA_LEAF_PAIRS);
}

inline int grid_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  return static_cast<int>(b < 1 ? 1 : (b > 152 * 32 ? 152 * 32 : b));
}

}  // namespace

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The top-K finish over `units` rows of W candidates (ascending output, -1 / -inf padding,
// poisoned outputs when the status word reports a timeout).
int launch_topk(const Dims& s, int W, const int32_t* cand, const float* cscore, const float* chead,
                int32_t* idx, float* score, float* head_lse, const int32_t* status, cudaStream_t st) {
  const int64_t units = static_cast<int64_t>(s.B) * s.Hkv * s.N;
  ProfScope ps(st, "topk");
  // one thread per unit pays once there are a few CTAs per SM (0.078 against 0.116 ms at 131072
  // units); below, the warp version's parallelism wins (0.011 against 0.021 ms at 4096 units)
  if (W <= 32 && PISA_TOPK_THREAD && units >= 32768)
    topk_thread_kernel<<<static_cast<unsigned>((units + kTopkUnits - 1) / kTopkUnits), kTopkUnits, 0, st>>>(
        units, W, s.K, s.N, s.G, cand, cscore, chead, idx, score, head_lse, status);
  else
    (W > 32 ? topk_kernel<2> : topk_kernel<1>)<<<static_cast<unsigned>((units + kWarps - 1) / kWarps), kWarps * 32,
                                                  0, st>>>(units, W, s.K, s.N, s.G, cand, cscore, chead, idx, score,
                                                           head_lse, status);
  return cudaGetLastError();
}

// Path-prefix levels the descent can score: l < LP for every scored level l + 1 (a level
// scores only when it holds more than K nodes); at least level 0 (the PISA-1 leaf scores).
int prefix_levels(const Dims& s, const Geo& g) {
  int lp = 1;
  for (int l = 1; l < g.n_levels; ++l)
    if (g.size[l] > s.K) lp = l;
  return lp;
}

// The prefix pass also computes the first scored level's child dots when that level's children
// fit its slots (fan-out 2, K <= 16) and G <= 4. The dots make a round trip through HBM
// (kFirstChildren x G x 4 bytes per query), which pays where the descent's own gathers of that
// level cost more: at the G = 4 sweep shape 0.21 + 2.79 -> 0.47 + 2.31 ms (prefix pass + descent),
// at the G = 8 64K workload 0.109 + 0.745 -> 0.227 + 0.662 ms.
bool first_level_pre(const Dims& s) { return s.g == 2 && 4 * s.K <= kFirstChildren && s.G <= 4; }

int launch_route_prefix(const Dims& s, const Geo& g, const void* Q, const void* K, const uint4* spl, float* pd,
                        float* cfirst, cudaStream_t st) {
  const int per_cta = 16 / s.G * prefix_warps(s.G);   // queries per CTA (one leaf at most)
  dim3 grid((s.N + per_cta - 1) / per_cta, s.Hkv, s.B);
  const int lp = prefix_levels(s, g);
  const auto* q = static_cast<const __nv_bfloat16*>(Q);
  const auto* k = static_cast<const __nv_bfloat16*>(K);
  ProfScope ps(st, "route_prefix");
  const int dyn = cfirst != nullptr ? kFirstChildren * s.d / 4 * 16 : 0;   // split rows of the first-level children
#define PISA_PREFIX_CASE(DD, GG)                                                                             \
  if (s.d == DD && s.G == GG) {                                                                              \
    cudaError_t e = cudaFuncSetAttribute(route_prefix_kernel<DD, GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn); \
    if (e != cudaSuccess) return e;                                                                          \
    route_prefix_kernel<DD, GG><<<grid, prefix_warps(GG) * 32, dyn, st>>>(s, g, lp, q, k, spl, pd, cfirst);  \
  }
  PISA_PREFIX_CASE(128, 1) PISA_PREFIX_CASE(128, 2) PISA_PREFIX_CASE(128, 4) PISA_PREFIX_CASE(128, 8)
  PISA_PREFIX_CASE(64, 1) PISA_PREFIX_CASE(64, 2) PISA_PREFIX_CASE(64, 4) PISA_PREFIX_CASE(64, 8)
#undef PISA_PREFIX_CASE
  return cudaGetLastError();
}

SelectWs select_ws(const Dims& s, const Geo& g, bool first) {
  SelectWs w{};
  const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.N;
  const size_t W = static_cast<size_t>(s.g) * s.K;
  size_t o = 0;
  w.status = o; o += 256;          // first: the caller finds the status word at offset 0
  w.split = o;  o += align256(static_cast<size_t>(s.B) * s.Hkv_r * g.nodes * s.d * 4);
  w.pd = o;     o += align256(units * prefix_levels(s, g) * s.G * 4);
  w.cfirst = o; o += first && first_level_pre(s) ? align256(units * kFirstChildren * s.G * 4) : 0;
  w.cand = o;   o += align256(units * W * 4);
  w.cscore = o; o += align256(units * W * 4);
  w.mean_end = o;                  // the PISA-1 path needs nothing past here
  w.group = o;
  o = group_ws(leaf_plan(s), o).end;
  w.total = o;           // without the per-head terms
  w.chead = o;  o += align256(units * W * s.G * 4);
  w.total_head = o;      // with them (head_lse requested)
  return w;
}

size_t flat_ws(const Dims& s, const Geo& g) {
  return 256 + align256(static_cast<size_t>(s.B) * s.Hkv_r * g.nodes * s.d * 4);   // status word, split rows
}

int launch_split(const Dims& s, const Geo& g, const float* pyr, uint4* spl, cudaStream_t st) {
  const int64_t n4 = static_cast<int64_t>(s.B) * s.Hkv_r * g.nodes * s.d / 4;
  ProfScope ps(st, "split_pyramid");
  split_kernel<<<grid_for(n4, 256), 256, 0, st>>>(reinterpret_cast<const float4*>(pyr), spl, n4);
  return cudaGetLastError();
}

int launch_select(const Dims& s, const Geo& g, const void* Q, const void* K, const float* pyr,
                  int32_t* idx, float* score, float* head_lse, char* ws, void* stream, bool first) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const SelectWs w = select_ws(s, g, first);
  uint4* spl = reinterpret_cast<uint4*>(ws + w.split);
  int32_t* cand = reinterpret_cast<int32_t*>(ws + w.cand);
  float* cscore = reinterpret_cast<float*>(ws + w.cscore);
  float* chead = head_lse ? reinterpret_cast<float*>(ws + w.chead) : nullptr;
  const GroupPlan gp = leaf_plan(s);
  const GroupWs gw = group_ws(gp, w.group);
  float* pd = reinterpret_cast<float*>(ws + w.pd);
  float* cfirst = first && first_level_pre(s) ? reinterpret_cast<float*>(ws + w.cfirst) : nullptr;
  const int lp = prefix_levels(s, g);
  int err = launch_split(s, g, pyr, spl, st);
  if (err) return err;
  if ((err = cudaMemsetAsync(ws + w.status, 0, 256, st))) return err;
  if ((err = launch_route_prefix(s, g, Q, K, spl, pd, cfirst, st))) return err;
  dim3 rgrid((s.N + kWarps - 1) / kWarps, s.Hkv, s.B);
  {
  ProfScope ps(st, "route");
#define PISA_ROUTE(DD, MM) \
  route_kernel<DD, MM, false><<<rgrid, kWarps * 32, 0, st>>>(s, g, lp, static_cast<const __nv_bfloat16*>(Q), pd, \
                                                           cfirst, spl, cand, nullptr)
  if (s.d == 128) {
    if (s.g * s.K <= 32) PISA_ROUTE(128, 32); else PISA_ROUTE(128, 64);
  } else {
    if (s.g * s.K <= 32) PISA_ROUTE(64, 32); else PISA_ROUTE(64, 64);
  }
#undef PISA_ROUTE
  }
  if ((err = cudaGetLastError())) return err;
  const int W = s.g * s.K;
  if ((err = launch_group_items(gp, cand, ws, gw, st))) return err;
  const int32_t* list = reinterpret_cast<const int32_t*>(ws + gw.list);
  const int4* items = reinterpret_cast<const int4*>(ws + gw.items);
  const int32_t* n_items = reinterpret_cast<const int32_t*>(ws + gw.icount) + gp.bins;
  if ((err = launch_leaf_tc(s, gp, Q, K, list, items, n_items, W, cscore, chead,
                            reinterpret_cast<int32_t*>(ws + w.status), st)))
    return err;
  return launch_topk(s, W, cand, cscore, chead, idx, score, head_lse, reinterpret_cast<const int32_t*>(ws + w.status),
                     st);
}

// PISA-1 ablation: the descent with mean scores at every level, the leaf candidates scored by
// their mean keys inside the routing kernel, then the final top K (no exact leaf stage).
int launch_select_mean(const Dims& s, const Geo& g, const void* Q, const void* K, const float* pyr,
                       int32_t* idx, float* score, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const SelectWs w = select_ws(s, g);
  uint4* spl = reinterpret_cast<uint4*>(ws + w.split);
  int32_t* cand = reinterpret_cast<int32_t*>(ws + w.cand);
  float* cscore = reinterpret_cast<float*>(ws + w.cscore);
  float* pd = reinterpret_cast<float*>(ws + w.pd);
  float* cfirst = first_level_pre(s) ? reinterpret_cast<float*>(ws + w.cfirst) : nullptr;
  const int lp = prefix_levels(s, g);
  int err = launch_split(s, g, pyr, spl, st);
  if (err) return err;
  if ((err = cudaMemsetAsync(ws + w.status, 0, 256, st))) return err;
  if ((err = launch_route_prefix(s, g, Q, K, spl, pd, cfirst, st))) return err;
  dim3 rgrid((s.N + kWarps - 1) / kWarps, s.Hkv, s.B);
  {
    ProfScope ps(st, "route_mean");
#define PISA_ROUTE(DD, MM) \
  route_kernel<DD, MM, true><<<rgrid, kWarps * 32, 0, st>>>(s, g, lp, static_cast<const __nv_bfloat16*>(Q), pd, \
                                                          cfirst, spl, cand, cscore)
    if (s.d == 128) {
      if (s.g * s.K <= 32) PISA_ROUTE(128, 32); else PISA_ROUTE(128, 64);
    } else {
      if (s.g * s.K <= 32) PISA_ROUTE(64, 32); else PISA_ROUTE(64, 64);
    }
#undef PISA_ROUTE
  }
  if ((err = cudaGetLastError())) return err;
  return launch_topk(s, s.g * s.K, cand, cscore, nullptr, idx, score, nullptr,
                     reinterpret_cast<const int32_t*>(ws + w.status), st);
}

int launch_select_flat(const Dims& s, const Geo& g, const void* Q, const void* K,
                       const float* pyr, int32_t* idx, float* score, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint4* spl = reinterpret_cast<uint4*>(ws + 256);
  int err = cudaMemsetAsync(ws, 0, 256, st);      // status word (no bounded waits here: stays 0)
  if (err) return err;
  if ((err = launch_split(s, g, pyr, spl, st))) return err;
  dim3 grid(s.n0, s.Hkv, s.B);
  const size_t smem = static_cast<size_t>(kWarps) * 2 * s.K * 32 * 8;
  ProfScope ps(st, "flat_select");
  if (s.d == 128) {
    cudaFuncSetAttribute(flat_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    flat_kernel<128><<<grid, kWarps * 32, smem, st>>>(s, g, static_cast<const __nv_bfloat16*>(Q),
                                                      static_cast<const __nv_bfloat16*>(K), spl, idx, score);
  } else {
    cudaFuncSetAttribute(flat_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    flat_kernel<64><<<grid, kWarps * 32, smem, st>>>(s, g, static_cast<const __nv_bfloat16*>(Q),
                                                     static_cast<const __nv_bfloat16*>(K), spl, idx, score);
  }
  return cudaGetLastError();
}

}  // namespace pisa
