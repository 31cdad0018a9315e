// Causal block-sparse attention forward on the fifth-generation tensor cores (tcgen05).
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value
// of the work": queries that use the same leaf key block are grouped into tiles so the
// block's keys are read once per tile, and attention runs only over the selected blocks.
//
// The softmax normaliser of row (query i, head h) is lse = log sum_k exp(lse_k) over the
// LSEs lse_k of its selected blocks, which the selection already computed exactly (they
// are the per-head terms of its leaf scores). With lse known before any key is visited,
// every block's contribution exp(s q.k - lse) v is already final: the blocks of a row are
// summed, not merged, so they can be added straight into an fp32 accumulator in any order.
//
// One CTA takes one work item (a leaf block of one KV head and up to 2048 (query, head)
// rows that selected it) in tiles of 128 rows:
//   * the item's pair list is staged in shared memory; the leaf's K (64 x d) and V^T
//     (d x 64) are staged once in the K-major 128-byte-swizzled layout;
//   * the next tile's 128 query rows are gathered with cp.async into the other half of a
//     double-buffered Q tile while the current tile computes;
//   * S = Q K^T (M=128, N=64) and O = P V (M=128, N=d) run as tcgen05.mma issued by one
//     thread, accumulating in TMEM; completion is tracked with mbarriers;
//   * each thread owns one row: it reads its S row from TMEM, applies the causal mask,
//     P = exp(s S - lse) (bf16) goes into the first K-block of the current Q buffer (Q is
//     no longer needed once S is done); after P V, the thread copies its O row, 64 columns
//     at a time, into a padded staging row in that same buffer and hands it to the TMA
//     unit as one bulk fp32 reduce-add into the accumulator (coalesced 256-byte requests
//     instead of 32 rows per warp store; the accumulator rows of a query chunk stay in L2).
// The LSE mode runs the same tiles through S only and writes every (row, block) LSE, for
// callers that do not pass the selection's. Every mbarrier wait is bounded: if one gives
// up, the kernel records PISA_ETIMEOUT in the status word, lets its outstanding copies
// finish, frees its TMEM and returns.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"

namespace pisa {

namespace {

constexpr int kRows = 128;
constexpr int kMaxItem = 1024;       // entries per work item (queries)
constexpr int kModeLse = 0, kModeOut = 1;

constexpr int round1024(int x) { return (x + 1023) / 1024 * 1024; }
constexpr int imax(int a, int b) { return a > b ? a : b; }

template <int D, int MODE>
struct TcFwdSmem {
  static constexpr int KB = D / 64;                 // K-blocks along the head dim
  static constexpr int Q_BYTES = KB * kRows * 128;  // one Q tile
  static constexpr int STG_ROW = 64 * 4 + 16;       // 64 fp32 of an O row + 16 B (no bank conflicts)
  static constexpr int BUF = MODE == kModeOut ? round1024(imax(Q_BYTES, kRows * STG_ROW)) : Q_BYTES;
  static constexpr int K_BYTES = KB * 64 * 128;
  static constexpr int V_BYTES = MODE == kModeOut ? D * 128 : 0;   // V^T: D rows of 64 keys
  static constexpr int oQ0 = 0, oK = 2 * BUF, oV = oK + K_BYTES;
  static constexpr int bytes = oV + V_BYTES + 1024; // + alignment slack
  static constexpr int tmem_cols = MODE == kModeOut ? ((64 + D) <= 128 ? 128 : 256) : 64;
};

template <int D, int G, int MODE>
__global__ void __launch_bounds__(kRows, 1)
attn_fwd_tc_kernel(Dims s, GroupPlan gp, const __nv_bfloat16* __restrict__ Q,
                   const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                   const int32_t* __restrict__ list, const int4* __restrict__ items,
                   const int32_t* __restrict__ n_items, const float* __restrict__ lse_rows,
                   float* __restrict__ block_lse, float* __restrict__ o_acc, int32_t* status) {
  using L = TcFwdSmem<D, MODE>;
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
  const int kbase = t * 64;
  const int n_tiles = (n_ent + EPT - 1) / EPT;

  unsigned char* sm = smraw + ((1024 - (tc::su32(smraw) & 1023)) & 1023);
  const uint32_t aQ0 = tc::su32(sm + L::oQ0);     // Q buffer `buf` starts at aQ0 + buf * BUF
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
    const uint32_t dstb = aQ0 + buf * L::BUF;
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
  if constexpr (MODE == kModeOut) {
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
  }
  tc::before_sync();
  __syncthreads();
  tc::after_sync();
  const uint32_t tS = tmem_base, tO = tmem_base + 64;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const int r = tid, h = r % G;

  for (int jt = 0; jt < n_tiles; ++jt) {
    const int buf = jt & 1;
    const uint32_t aQb = aQ0 + buf * L::BUF;
    // prefetch the next tile's rows into the other buffer (its last readers, the previous
    // tile's MMAs and bulk reductions, have completed)
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
    const int qi = entry_query(jt, r / G);
    const int64_t lrow_at = (static_cast<int64_t>(b) * s.Hq + kv * G + h) * s.N + (qi < 0 ? 0 : qi);
    float lrow = 0.f;
    if (MODE == kModeOut && qi >= 0) lrow = lse_rows[lrow_at];   // in flight during the MMA
    if (!tc::bar_wait(&bar[0], jt & 1)) atomicOr(&s_abort, 1);
    tc::after_sync();
    float sv[64];
    tc::tmem_ld64(tS + lane_off, sv);
    if constexpr (MODE == kModeLse) {
      float mx = neg_inf(), l = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        sv[c] = (kbase + c <= qi) ? s.scale * sv[c] : neg_inf();
        mx = fmaxf(mx, sv[c]);
      }
      const float m = mx == neg_inf() ? 0.f : mx;
#pragma unroll
      for (int c = 0; c < 64; ++c) l += expf(sv[c] - m);
      if (qi >= 0)
        block_lse[lrow_at * s.K + (s_list[jt * EPT + r / G] & 63)] = l > 0.f ? m + logf(l) : neg_inf();
      tc::before_sync();
      __syncthreads();
      if (s_abort) break;
    } else {
      // P = exp(s S - lse) on the visible keys; into the (now free) first K-block of Q[buf]
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float pv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = cc * 8 + u;
          pv[u] = (kbase + c <= qi) ? expf(fmaf(s.scale, sv[c], -lrow)) : 0.f;
        }
        uint4 pk;
        pk.x = pack_bf16(pv[0], pv[1]);
        pk.y = pack_bf16(pv[2], pv[3]);
        pk.z = pack_bf16(pv[4], pv[5]);
        pk.w = pack_bf16(pv[6], pv[7]);
        *reinterpret_cast<uint4*>(sm + L::oQ0 + buf * L::BUF + tc::sw128(r, cc * 8)) = pk;
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
      // epilogue: the O row, 64 columns at a time, through this thread's staging row in the
      // now free Q[buf] and one bulk reduce-add each into the accumulator row
      const int64_t row = (static_cast<int64_t>(b) * s.N + (qi < 0 ? 0 : qi)) * s.Hq + kv * G + h;
      float4* stg = reinterpret_cast<float4*>(sm + L::oQ0 + buf * L::BUF + r * L::STG_ROW);
      const uint32_t a_stg = tc::su32(stg);
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        float ov[64];
        tc::tmem_ld64(tO + lane_off + half * 64, ov);
        if (half > 0) tc::bulk_wait_read<0>();      // the staging row was read out
#pragma unroll
        for (int c = 0; c < 16; ++c) stg[c] = make_float4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
        tc::fence_async_smem();
        if (qi >= 0) {
          tc::bulk_reduce_add_f32(o_acc + row * D + half * 64, a_stg, 256);
          tc::bulk_commit();
        }
      }
      tc::bulk_wait_read<0>();                     // Q[buf] is gathered into again next tile
      tc::before_sync();
      __syncthreads();
      if (s_abort) break;
    }
  }
  tc::cp_async_wait<0>();
  tc::bulk_wait<0>();                              // reductions complete before exit
  tc::before_sync();
  __syncthreads();
  if (s_abort && tid == 0) atomicOr(status, PISA_ETIMEOUT);
  if (warp == 0) tc::tmem_free(tmem_base, L::tmem_cols);
}

// One warp per (b, query, head) row: lse = log sum_k exp(block_lse_k) over the row's valid
// slots (lane k < K holds slot k), written to the caller's lse; the row's accumulator is
// cleared for the reduce-adds.
template <int D>
__global__ void __launch_bounds__(256)
attn_rows_kernel(Dims s, const int32_t* __restrict__ idx, const float* __restrict__ block_lse,
                 float* __restrict__ lse_out, float4* __restrict__ o_acc) {
  const int64_t row = blockIdx.x * 8LL + (threadIdx.x >> 5);       // (b*N + i)*Hq + h
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(s.B) * s.N * s.Hq) return;
  const int h = static_cast<int>(row % s.Hq);
  const int64_t bi = row / s.Hq;
  const int i = static_cast<int>(bi % s.N), b = static_cast<int>(bi / s.N);
  const int64_t unit = (static_cast<int64_t>(b) * s.Hkv + h / s.G) * s.N + i;
  const int64_t lrow = (static_cast<int64_t>(b) * s.Hq + h) * s.N + i;
  const bool valid = lane < s.K && idx[unit * s.K + lane] >= 0;
  const float my = valid ? block_lse[lrow * s.K + lane] : neg_inf();
  float m = my;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float den = warp_sum((valid && m != neg_inf()) ? expf(my - m) : 0.f);
  if (lane == 0) lse_out[lrow] = den > 0.f ? m + logf(den) : neg_inf();
  for (int c = lane; c < D / 4; c += 32) o_acc[row * (D / 4) + c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// O = bf16(accumulator), 8 elements per thread.
__global__ void __launch_bounds__(256)
attn_out_kernel(int64_t n8, const float4* __restrict__ o_acc, uint4* __restrict__ O) {
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n8;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = o_acc[2 * q], c = o_acc[2 * q + 1];
    O[q] = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(c.x, c.y), pack_bf16(c.z, c.w));
  }
}

template <int D, int G, int MODE>
int tc_launch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
              const int32_t* list, const int4* items, const int32_t* n_items, const float* lse_rows,
              float* block_lse, float* o_acc, int32_t* status, cudaStream_t st) {
  const int smem = TcFwdSmem<D, MODE>::bytes;
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_tc_kernel<D, G, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope ps(st, MODE == kModeOut ? "attn_fwd_tc" : "attn_lse_tc");
  attn_fwd_tc_kernel<D, G, MODE><<<static_cast<unsigned>(gp.max_items), kRows, smem, st>>>(
      s, gp, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
      static_cast<const __nv_bfloat16*>(V), list, items, n_items, lse_rows, block_lse, o_acc, status);
  return cudaGetLastError();
}

template <int MODE>
int tc_dispatch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                const int32_t* list, const int4* items, const int32_t* n_items, const float* lse_rows,
                float* block_lse, float* o_acc, int32_t* status, cudaStream_t st) {
#define PISA_TC_CASE(DD, GG)                                                                          \
  if (s.d == DD && s.G == GG)                                                                         \
    return tc_launch<DD, GG, MODE>(s, gp, Q, K, V, list, items, n_items, lse_rows, block_lse, o_acc, \
                                   status, st);
  PISA_TC_CASE(128, 1) PISA_TC_CASE(128, 2) PISA_TC_CASE(128, 4) PISA_TC_CASE(128, 8)
  PISA_TC_CASE(64, 1) PISA_TC_CASE(64, 2) PISA_TC_CASE(64, 4) PISA_TC_CASE(64, 8)
#undef PISA_TC_CASE
  return static_cast<int>(cudaErrorNotSupported);
}

}  // namespace

// Tensor-core forward for d in {64, 128} and G in {1, 2, 4, 8}: [block LSE pass when
// head_lse is NULL] -> row LSE + accumulator clear -> output pass -> bf16 conversion.
int launch_attn_fwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       const float* head_lse, float* block_lse_ws, float* o_acc, void* O, float* lse,
                       int32_t* status, cudaStream_t st) {
  const float* hl = head_lse;
  int err;
  if (!hl) {
    err = tc_dispatch<kModeLse>(s, gp, Q, K, V, list, items, n_items, nullptr, block_lse_ws, nullptr, status, st);
    if (err) return err;
    hl = block_lse_ws;
  }
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  {
    ProfScope ps(st, "attn_rows");
    if (s.d == 128)
      attn_rows_kernel<128><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
          s, idx, hl, lse, reinterpret_cast<float4*>(o_acc));
    else
      attn_rows_kernel<64><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
          s, idx, hl, lse, reinterpret_cast<float4*>(o_acc));
  }
  if ((err = cudaGetLastError())) return err;
  err = tc_dispatch<kModeOut>(s, gp, Q, K, V, list, items, n_items, lse, nullptr, o_acc, status, st);
  if (err) return err;
  {
    ProfScope ps(st, "attn_out");
    const int64_t n8 = rows * s.d / 8;
    const int64_t nb = (n8 + 255) / 256;
    attn_out_kernel<<<static_cast<unsigned>(nb < 152 * 32 ? nb : 152 * 32), 256, 0, st>>>(
        n8, reinterpret_cast<const float4*>(o_acc), static_cast<uint4*>(O));
  }
  return cudaGetLastError();
}

}  // namespace pisa
