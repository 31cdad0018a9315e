// Causal block-sparse attention forward on the fifth-generation tensor cores (tcgen05).
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value
// of the work": queries that use the same leaf key block are grouped into tiles so the
// block's keys are read once per tile, and attention runs only over the selected blocks.
// One CTA takes one work item (a leaf block of one KV head and up to 2048 (query, head)
// rows that selected it) in tiles of 128 rows:
//   * the item's pair list is staged in shared memory; the leaf's K (64 x d) and V^T
//     (d x 64) are staged once in the K-major 128-byte-swizzled layout;
//   * the next tile's 128 query rows are gathered with cp.async into the other half of a
//     double-buffered Q tile while the current tile computes;
//   * S = Q K^T (M=128, N=64) and O = P V (M=128, N=d) run as tcgen05.mma issued by one
//     thread, accumulating in TMEM; completion is tracked with mbarriers;
//   * each thread owns one row: it reads its S row from TMEM, applies the causal mask and
//     the block softmax, writes P (bf16) into the first K-block of the current Q buffer
//     (Q is no longer needed once S is done), then reads its O row, normalises it and
//     stores the (row, block) partial and the block LSE;
//   * a second kernel merges every row's block partials, one warp per row with all of its
//     slots in flight: lse = log sum_t exp(lse_t), o = sum_t exp(lse_t - lse) o_t.
// Every mbarrier wait is bounded: if one gives up, the kernel records PISA_ETIMEOUT in the
// status word, lets its outstanding copies finish, frees its TMEM and returns.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"

namespace pisa {

namespace {

constexpr int kRows = 128;
constexpr int kMaxItem = 1024;       // entries per work item (queries)

template <int D>
struct TcFwdSmem {
  static constexpr int KB = D / 64;                 // K-blocks along the head dim
  static constexpr int Q_BYTES = KB * kRows * 128;  // one Q tile
  static constexpr int K_BYTES = KB * 64 * 128;
  static constexpr int V_BYTES = D * 128;           // V^T: D rows of 64 keys
  static constexpr int oQ0 = 0, oK = 2 * Q_BYTES, oV = oK + K_BYTES;
  static constexpr int bytes = oV + V_BYTES + 1024; // + alignment slack
  static constexpr int tmem_cols = (64 + D) <= 128 ? 128 : 256;
};

template <int D, int G>
__global__ void __launch_bounds__(kRows, 1)
attn_fwd_tc_kernel(Dims s, GroupPlan gp, const __nv_bfloat16* __restrict__ Q,
                   const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                   const int32_t* __restrict__ list, const int4* __restrict__ items,
                   const int32_t* __restrict__ n_items, __nv_bfloat16* __restrict__ part_o,
                   float* __restrict__ part_lse, int32_t* status) {
  using L = TcFwdSmem<D>;
  constexpr int EPT = kRows / G;          // entries (queries) per tile
  constexpr int CH = D / 8;               // 16-byte chunks per row
  extern __shared__ unsigned char smraw[];
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_list[kMaxItem];        // the item's (query << 6 | slot) entries
  __shared__ int s_abort;

  if (static_cast<int>(blockIdx.x) >= *n_items) return;
  const int4 item = items[blockIdx.x];
  const int beg = item.y, n_ent = item.z;
  const int t = gp.leaf_of(item.x);
  const int64_t head = gp.head_of(item.x);
  const int b = static_cast<int>(head / s.Hkv), kv = static_cast<int>(head % s.Hkv);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int Ksel = s.K;
  const int kbase = t * 64;
  const int n_tiles = (n_ent + EPT - 1) / EPT;

  unsigned char* sm = smraw + ((1024 - (tc::su32(smraw) & 1023)) & 1023);
  const uint32_t aQ0 = tc::su32(sm + L::oQ0);     // Q buffer `buf` starts at aQ0 + buf * Q_BYTES
  const uint32_t aK = tc::su32(sm + L::oK), aV = tc::su32(sm + L::oV);
  constexpr uint32_t idS = tc::idesc_bf16(kRows, 64), idO = tc::idesc_bf16(kRows, D);

  if (tid == 0) {
    tc::bar_init(&bar[0], 1);
    tc::bar_init(&bar[1], 1);
    tc::fence_bar_init();
    s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, L::tmem_cols);
  for (int e = tid; e < n_ent; e += kRows) s_list[e] = list[beg + e];
  // entry e of tile j: query s_list[j*EPT + e] >> 6, slot & 63 (query -1 past the end)
  auto entry_query = [&](int j, int e) {
    const int ge = j * EPT + e;
    return ge < n_ent ? (s_list[ge] >> 6) : -1;
  };
  auto gather_q = [&](int j, int buf) {
    const uint32_t dstb = aQ0 + buf * L::Q_BYTES;
    for (int lin = tid; lin < kRows * CH; lin += kRows) {
      const int r = lin / CH, c = lin % CH;
      const int i = entry_query(j, r / G);
      const __nv_bfloat16* src =
          Q + ((static_cast<int64_t>(b) * s.N + (i < 0 ? 0 : i)) * s.Hq + kv * G + (r % G)) * D + c * 8;
      tc::cp_async16(dstb + (c >> 3) * (kRows * 128) + tc::sw128(r, (c & 7) * 8), src, i >= 0);
    }
  };
  __syncthreads();
  gather_q(0, 0);
  // leaf K tile (async) and V^T, transposed by the threads (lanes walk keys: no bank conflicts)
  for (int lin = tid; lin < 64 * CH; lin += kRows) {
    const int r = lin / CH, c = lin % CH;
    const int64_t j = static_cast<int64_t>(kbase) + r;
    const bool ok = j < s.N;
    const __nv_bfloat16* src = K + ((static_cast<int64_t>(b) * s.N + (ok ? j : 0)) * s.Hkv + kv) * D + c * 8;
    tc::cp_async16(aK + (c >> 3) * (64 * 128) + tc::sw128(r, (c & 7) * 8), src, ok);
  }
  tc::cp_async_commit();
  for (int lin = tid; lin < 64 * CH; lin += kRows) {
    const int r = lin % 64, c = lin / 64;   // key r, dims c*8 .. c*8+7
    const int64_t j = static_cast<int64_t>(kbase) + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < s.N) v = ldg_u4(V + ((static_cast<int64_t>(b) * s.N + j) * s.Hkv + kv) * D + c * 8);
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<__nv_bfloat16*>(sm + L::oV + tc::sw128(c * 8 + u, r)) = e[u];
  }
  tc::before_sync();
  __syncthreads();
  tc::after_sync();
  const uint32_t tS = tmem_base, tO = tmem_base + 64;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  for (int jt = 0; jt < n_tiles; ++jt) {
    const int buf = jt & 1;
    const uint32_t aQb = aQ0 + buf * L::Q_BYTES;
    // prefetch the next tile's rows into the other buffer (its last reader, the previous
    // tile's P V MMA, has completed)
    if (jt + 1 < n_tiles) gather_q(jt + 1, buf ^ 1);
    tc::cp_async_commit();
    tc::cp_async_wait<1>();              // this tile's rows (and the K tile) have landed
    tc::fence_async_smem();
    tc::before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::after_sync();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc::mma(tS, tc::desc(aQb + (ks >> 2) * (kRows * 128) + (ks & 3) * 32),
                tc::desc(aK + (ks >> 2) * (64 * 128) + (ks & 3) * 32), idS, ks > 0);
      tc::commit(&bar[0]);
    }
    if (!tc::bar_wait(&bar[0], jt & 1)) atomicOr(&s_abort, 1);
    tc::after_sync();
    // softmax of this thread's row; P goes into the (now free) first K-block of Q[buf]
    const int r = tid, e = r / G, h = r % G;
    const int qi = entry_query(jt, e);
    float m, l = 0.f;
    {
      float sv[64];
      tc::tmem_ld64(tS + lane_off, sv);
      float mx = neg_inf();
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        sv[c] = (kbase + c <= qi) ? s.scale * sv[c] : neg_inf();
        mx = fmaxf(mx, sv[c]);
      }
      m = mx == neg_inf() ? 0.f : mx;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        sv[c] = expf(sv[c] - m);
        l += sv[c];
      }
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4 pk;
        pk.x = pack_bf16(sv[cc * 8 + 0], sv[cc * 8 + 1]);
        pk.y = pack_bf16(sv[cc * 8 + 2], sv[cc * 8 + 3]);
        pk.z = pack_bf16(sv[cc * 8 + 4], sv[cc * 8 + 5]);
        pk.w = pack_bf16(sv[cc * 8 + 6], sv[cc * 8 + 7]);
        *reinterpret_cast<uint4*>(sm + L::oQ0 + buf * L::Q_BYTES + tc::sw128(r, cc * 8)) = pk;
      }
    }
    tc::fence_async_smem();
    tc::before_sync();
    __syncthreads();
    if (s_abort) break;
    if (tid == 0) {
      tc::after_sync();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma(tO, tc::desc(aQb + kk * 32), tc::desc(aV + kk * 32), idO, kk > 0);
      tc::commit(&bar[1]);
    }
    if (!tc::bar_wait(&bar[1], jt & 1)) atomicOr(&s_abort, 1);
    tc::after_sync();
    // epilogue: this thread's normalised partial row and its block LSE
    const int64_t row = (static_cast<int64_t>(b) * s.N + (qi < 0 ? 0 : qi)) * s.Hq + kv * G + h;
    const int slot = qi >= 0 ? (s_list[jt * EPT + e] & 63) : 0;
    const float rl = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* dst = part_o + (row * Ksel + slot) * D;
#pragma unroll
    for (int half = 0; half < D / 64; ++half) {
      float ov[64];
      tc::tmem_ld64(tO + lane_off + half * 64, ov);
      if (qi >= 0) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 pk;
          pk.x = pack_bf16(ov[cc * 8 + 0] * rl, ov[cc * 8 + 1] * rl);
          pk.y = pack_bf16(ov[cc * 8 + 2] * rl, ov[cc * 8 + 3] * rl);
          pk.z = pack_bf16(ov[cc * 8 + 4] * rl, ov[cc * 8 + 5] * rl);
          pk.w = pack_bf16(ov[cc * 8 + 6] * rl, ov[cc * 8 + 7] * rl);
          *reinterpret_cast<uint4*>(dst + half * 64 + cc * 8) = pk;
        }
      }
    }
    if (qi >= 0) part_lse[row * Ksel + slot] = l > 0.f ? m + logf(l) : neg_inf();
    tc::before_sync();
    __syncthreads();
    if (s_abort) break;
  }
  tc::cp_async_wait<0>();
  tc::before_sync();
  __syncthreads();
  if (s_abort && tid == 0) atomicOr(status, PISA_ETIMEOUT);
  if (warp == 0) tc::tmem_free(tmem_base, L::tmem_cols);
}

// One warp per (b, query, head) row: merges the row's <= K block partials. Lane q < K
// holds slot q's LSE, the weights come from warp reductions, and each lane then owns D/32
// dimensions, with every slot's load issued before any is used.
template <int D>
__global__ void __launch_bounds__(256)
attn_combine_kernel(Dims s, const int32_t* __restrict__ idx, const __nv_bfloat16* __restrict__ part_o,
                    const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ O,
                    float* __restrict__ lse_out) {
  constexpr int PER = D / 32;
  const int64_t row = blockIdx.x * 8LL + (threadIdx.x >> 5);       // (b*N + i)*Hq + h
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(s.B) * s.N * s.Hq) return;
  const int h = static_cast<int>(row % s.Hq);
  const int64_t bi = row / s.Hq;
  const int i = static_cast<int>(bi % s.N), b = static_cast<int>(bi / s.N);
  const int64_t unit = (static_cast<int64_t>(b) * s.Hkv + h / s.G) * s.N + i;
  const bool valid = lane < s.K && idx[unit * s.K + lane] >= 0;
  const float my = valid ? part_lse[row * s.K + lane] : neg_inf();
  float m = my;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float w = (valid && m != neg_inf()) ? expf(my - m) : 0.f;
  const float den = warp_sum(w);
  const unsigned vmask = __ballot_sync(0xffffffffu, valid);
  const float r = den > 0.f ? 1.f / den : 0.f;
  const __nv_bfloat16* src = part_o + row * s.K * D + lane * PER;
  float acc[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) acc[u] = 0.f;
  uint2 v[32];
#pragma unroll
  for (int q = 0; q < 32; ++q)
    if ((vmask >> q) & 1u) v[q] = __ldg(reinterpret_cast<const uint2*>(src + q * D));
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    const float wq = __shfl_sync(0xffffffffu, w, q);
    if ((vmask >> q) & 1u) {
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v[q]);
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] += wq * __bfloat162float(e[u]);
    }
  }
  __nv_bfloat16* dst = O + row * D + lane * PER;
#pragma unroll
  for (int u = 0; u < PER; u += 2) *reinterpret_cast<uint32_t*>(dst + u) = pack_bf16(acc[u] * r, acc[u + 1] * r);
  if (lane == 0)
    lse_out[(static_cast<int64_t>(b) * s.Hq + h) * s.N + i] = den > 0.f ? m + logf(den) : neg_inf();
}

template <int D, int G>
int tc_launch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
              const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
              __nv_bfloat16* po, float* pl, void* O, float* lse, int32_t* status, cudaStream_t st) {
  const int smem = TcFwdSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  {
    ProfScope ps(st, "attn_fwd_tc");
    attn_fwd_tc_kernel<D, G><<<static_cast<unsigned>(gp.max_items), kRows, smem, st>>>(
        s, gp, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
        static_cast<const __nv_bfloat16*>(V), list, items, n_items, po, pl, status);
  }
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  ProfScope ps(st, "attn_combine");
  attn_combine_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      s, idx, po, pl, static_cast<__nv_bfloat16*>(O), lse);
  return cudaGetLastError();
}

}  // namespace

// Tensor-core forward for d in {64, 128} and G in {1, 2, 4, 8}.
int launch_attn_fwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       __nv_bfloat16* po, float* pl, void* O, float* lse, int32_t* status, cudaStream_t st) {
#define PISA_TC_CASE(DD, GG)                                                                          \
  if (s.d == DD && s.G == GG)                                                                         \
    return tc_launch<DD, GG>(s, gp, Q, K, V, idx, list, items, n_items, po, pl, O, lse, status, st);
  PISA_TC_CASE(128, 1) PISA_TC_CASE(128, 2) PISA_TC_CASE(128, 4) PISA_TC_CASE(128, 8)
  PISA_TC_CASE(64, 1) PISA_TC_CASE(64, 2) PISA_TC_CASE(64, 4) PISA_TC_CASE(64, 8)
#undef PISA_TC_CASE
  return static_cast<int>(cudaErrorNotSupported);
}

}  // namespace pisa
