// Causal block-sparse attention forward on the fifth-generation tensor cores (tcgen05), and
// its block-LSE pass.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value
// of the work": queries that use the same leaf key block are grouped into tiles so the
// block's keys are read once per tile, and attention runs only over the selected blocks.
//
// Attention normaliser. Row (query i, head h) has lse = log sum_k exp(lse_k) over the LSEs
// lse_k of its selected blocks, which the selection already computed exactly (the per-head
// terms of its leaf scores). With lse known before any key is visited, every block's
// contribution exp(s q.k - lse) v is final: the blocks of a row are summed, not merged, and
// go straight into an fp32 accumulator in any order.
//
// One CTA (8 warps) takes one work item: a leaf block of one KV head and up to 2048
// (query, head) rows that chose it, in tiles of 128 rows (row = TMEM lane; the two
// warpgroups split the columns of every tile):
//   * the leaf's K (64 x d) arrives by TMA tile load, V^T (d x 64) is transposed by the
//     threads once per item, both in the K-major 128-byte-swizzled layout;
//   * the tiles' query rows are gathered with cp.async (each thread copies half a row) into
//     a double-buffered Q tile; a thread confirms its copies of a tile one tile later
//     (wait, proxy fence, mbarrier arrival), so the MMA issuer never waits on a fresh copy;
//   * S = Q K^T (M=128, N=64) into one of two TMEM buffers, issued for the next tile as soon
//     as its rows have landed, so it overlaps this tile's softmax; O = P V (M=128, N=d);
//   * output mode: P = 2^(s log2(e) S - log2(e) lse) on the visible keys (bf16, into the
//     free first K-block of the tile's Q buffer); after P V, each warpgroup moves its half
//     of O through a swizzled staging tile in the same buffer, and one lane per query adds
//     its G heads x 32 columns into the accumulator with a single TMA tensor reduce-add;
//   * the LSE mode (for callers without the selection's LSEs) stops after S: each
//     warpgroup reduces its 32 columns to a (max, sum) pair, the halves merge in shared
//     memory, and the row LSE is written per (row, block).
// Every mbarrier wait is bounded: if one gives up, the kernel records PISA_ETIMEOUT in the
// status word, lets its outstanding copies finish, frees its TMEM and returns.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"
#include "tmap.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 128;
constexpr int kMaxItem = 1024;       // entries per work item (queries)
constexpr int kModeLse = 0, kModeOut = 1;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int imax(int a, int b) { return a > b ? a : b; }

template <int D, int MODE>
struct TcSmem {
  static constexpr int KB = D / 64;                 // K-blocks along the head dim
  static constexpr int Q_BYTES = KB * kRows * 128;  // one Q tile
  static constexpr int STAGE = kRows * 128;         // one warpgroup's 32-column fp32 staging tile
  static constexpr int BUF = MODE == kModeOut ? imax(Q_BYTES, 2 * STAGE) : Q_BYTES;
  static constexpr int K_BYTES = KB * 64 * 128;
  static constexpr int V_BYTES = MODE == kModeOut ? D * 128 : 0;   // V^T: D rows of 64 keys
  static constexpr int oQ0 = 0, oK = 2 * BUF, oV = oK + K_BYTES;
  static constexpr int bytes = oV + V_BYTES + 1024; // + alignment slack
  // TMEM: S0 | S1 (64 columns each) | O (D columns)
  static constexpr int tmem_cols = MODE == kModeOut ? 256 : 128;
};

struct TcArgs {
  Dims s;
  GroupPlan gp;
  const __nv_bfloat16* Q;
  const __nv_bfloat16* V;
  const int32_t* list;
  const int4* items;
  const int32_t* n_items;
  const float* lse_rows;   // output mode: [B,Hq,N]
  float* out;              // LSE mode: block LSE [B,Hq,N,K]
  int32_t* status;
};

template <int D, int G, int MODE>
__global__ void __launch_bounds__(kThreads, 2)
block_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap omap) {
  using L = TcSmem<D, MODE>;
  constexpr int EPT = kRows / G;          // entries (queries) per tile
  constexpr int KB = L::KB;
  constexpr int HC = D / 16;              // 16-byte chunks per half row
  extern __shared__ unsigned char smraw[];
  __shared__ __align__(8) uint64_t bar_q[2], bar_s[2], bar_k, bar_o;
  __shared__ uint32_t tmem_base;
  __shared__ int s_list[kMaxItem];        // the item's (query << 6 | slot) entries
  __shared__ float2 s_ml[2][kRows];       // LSE mode: the second warpgroup's (max, sum) per row

  const Dims& s = a.s;
  if (static_cast<int>(blockIdx.x) >= *a.n_items) return;
  const int4 item = a.items[blockIdx.x];
  const int beg = item.y, n_ent = item.z;
  const int t = a.gp.leaf_of(item.x);
  const int64_t head = a.gp.head_of(item.x);
  const int b = static_cast<int>(head / s.Hkv), kv = static_cast<int>(head % s.Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;                       // column half of every tile
  const int r = (warp & 3) * 32 + lane;           // tile row = TMEM lane
  const int h = r % G;
  const int kbase = t * 64;
  const int n_tiles = (n_ent + EPT - 1) / EPT;

  unsigned char* sm = smraw + ((1024 - (tc::su32(smraw) & 1023)) & 1023);
  const uint32_t aQ0 = tc::su32(sm + L::oQ0);     // Q buffer `bf` starts at aQ0 + bf * BUF
  const uint32_t aK = tc::su32(sm + L::oK), aV = tc::su32(sm + L::oV);
  constexpr uint32_t idS = tc::idesc_bf16(kRows, 64), idO = tc::idesc_bf16(kRows, D);

  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      tc::bar_init(&bar_q[k], kThreads);   // every thread confirms its copies
      tc::bar_init(&bar_s[k], 1);
    }
    tc::bar_init(&bar_k, 1);
    tc::bar_init(&bar_o, 1);
    tc::fence_bar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, L::tmem_cols);
  for (int e = tid; e < n_ent; e += kThreads) s_list[e] = a.list[beg + e];
  tc::before_sync();
  __syncthreads();
  tc::after_sync();

  // query of row rr of tile j (-1 past the end of the item)
  auto query_of = [&](int j, int rr) {
    const int e = j * EPT + rr / G;
    return e < n_ent ? (s_list[e] >> 6) : -1;
  };
  bool bad = false;                 // this thread saw a bounded wait give up
  // all threads: cp.async of tile j's 128 query rows into Q buffer bf, one commit group;
  // thread t copies half row t >> 1 (zero-filled past the end of the item)
  auto gather = [&](int j, int bf) {
    const int rr = tid >> 1, qi = query_of(j, rr);
    const __nv_bfloat16* src =
        a.Q + ((static_cast<int64_t>(b) * s.N + (qi < 0 ? 0 : qi)) * s.Hq + kv * G + rr % G) * D;
    const uint32_t dst = aQ0 + bf * L::BUF;
#pragma unroll
    for (int u = 0; u < HC; ++u) {
      const int c = (tid & 1) * HC + u;
      tc::cp_async16(dst + (c >> 3) * (kRows * 128) + tc::sw128(rr, (c & 7) * 8), src + c * 8, qi >= 0);
    }
    tc::cp_async_commit();
  };
  // this thread's copies of the tile in buffer bf have landed (all but `newer` groups):
  // make them visible to the tensor cores and arrive on the buffer's barrier
  auto confirm = [&](int bf, bool newer) {
    if (newer) tc::cp_async_wait<1>(); else tc::cp_async_wait<0>();
    tc::fence_async_smem();
    tc::bar_arrive(&bar_q[bf]);
  };
  // thread 0: S(j) = Q(j) K^T into TMEM buffer j & 1, once tile j's rows (and K) have landed
  auto issue_s = [&](int j) {
    const int bf = j & 1;
    bool ok = tc::bar_wait(&bar_q[bf], (j >> 1) & 1);
    if (j == 0) ok = tc::bar_wait(&bar_k, 0) && ok;
    if (!ok) bad = true;
    tc::after_sync();
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      tc::mma(tmem_base + 64 * bf, tc::desc(aQ0 + bf * L::BUF + (ks >> 2) * (kRows * 128) + (ks & 3) * 32),
              tc::desc(aK + (ks >> 2) * (64 * 128) + (ks & 3) * 32), idS, ks > 0);
    tc::commit(&bar_s[bf]);
  };

  if (tid == 0) {
    tc::bar_expect_tx(&bar_k, L::K_BYTES);
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) tc::tma_load4(aK + kb * (64 * 128), &kmap, kb * 64, kv, kbase, b, &bar_k);
  }
  gather(0, 0);
  if (n_tiles > 1) gather(1, 1);
  confirm(0, n_tiles > 1);
  if constexpr (MODE == kModeOut) {
    // V^T, transposed by the threads (lanes walk keys: no bank conflicts); rows past N are 0
    for (int lin = tid; lin < 64 * (D / 8); lin += kThreads) {
      const int key = lin % 64, c = lin / 64;   // dims c*8 .. c*8+7
      const int64_t j = static_cast<int64_t>(kbase) + key;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (j < s.N) v = ldg_u4(a.V + ((static_cast<int64_t>(b) * s.N + j) * s.Hkv + kv) * D + c * 8);
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int u = 0; u < 8; ++u) *reinterpret_cast<__nv_bfloat16*>(sm + L::oV + tc::sw128(c * 8 + u, key)) = e[u];
    }
    tc::fence_async_smem();
    tc::before_sync();
    __syncthreads();
  }
  if (tid == 0) issue_s(0);
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const float c1 = s.scale * kLog2e;              // logits in base-2 units

  for (int jt = 0; jt < n_tiles; ++jt) {
    const int bf = jt & 1;
    const int qi = query_of(jt, r);
    const int lim = qi - kbase - 32 * wg;        // this half's column c is visible iff c <= lim
    const int slot = qi >= 0 ? (s_list[jt * EPT + r / G] & 63) : 0;
    float lrow2 = 0.f;
    if (MODE == kModeOut && qi >= 0)               // in flight during the MMA wait
      lrow2 = a.lse_rows[(static_cast<int64_t>(b) * s.Hq + kv * G + h) * s.N + qi] * kLog2e;
    if (!tc::bar_wait(&bar_s[bf], (jt >> 1) & 1)) bad = true;
    tc::after_sync();

    if constexpr (MODE == kModeLse) {
      // Q[bf] is free (S(jt) is done): tile jt+2's rows go there; tile jt+1's rows (copied
      // one tile ago) are confirmed and S(jt+1) starts now
      if (jt + 2 < n_tiles) gather(jt + 2, bf);
      if (jt + 1 < n_tiles) confirm(bf ^ 1, jt + 2 < n_tiles);
      if (tid == 0 && jt + 1 < n_tiles) issue_s(jt + 1);
      float sv[32];
      tc::tmem_ld32(tmem_base + 64 * bf + 32 * wg + lane_off, sv);
      float mx = -INFINITY;
      if (lim >= 31) {
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = fmaxf(mx, sv[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sv[c] = c <= lim ? sv[c] : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      }
      float l = 0.f, m2 = -INFINITY;
      if (mx != -INFINITY) {
        m2 = mx * c1;
#pragma unroll
        for (int c = 0; c < 32; ++c) l += tc::ex2(fmaf(sv[c], c1, -m2));
      }
      if (wg == 1) s_ml[bf][r] = make_float2(m2, l);
      tc::before_sync();
      const bool stop = __syncthreads_or(bad);
      if (wg == 0 && !stop) {
        const float2 o = s_ml[bf][r];
        const float M = fmaxf(m2, o.x);
        float lse = -INFINITY;
        if (M != -INFINITY) {
          const float Lsum = l * tc::ex2(m2 - M) + o.y * tc::ex2(o.x - M);
          lse = (M + tc::lg2(Lsum)) * kLn2;
        }
        if (qi >= 0) a.out[((static_cast<int64_t>(b) * s.Hq + kv * G + h) * s.N + qi) * s.K + slot] = lse;
      }
      if (stop) break;
    } else {
      // P = 2^(c1 S - log2e lse) on the visible keys, this half's 32 keys of the row, into
      // the first K-block of Q[bf]
      float sv[32];
      tc::tmem_ld32(tmem_base + 64 * bf + 32 * wg + lane_off, sv);
      if (lim >= 31) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = tc::ex2(fmaf(sv[c], c1, -lrow2));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = c <= lim ? tc::ex2(fmaf(sv[c], c1, -lrow2)) : 0.f;
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint4 pk;
        pk.x = pack_bf16(sv[cc * 8 + 0], sv[cc * 8 + 1]);
        pk.y = pack_bf16(sv[cc * 8 + 2], sv[cc * 8 + 3]);
        pk.z = pack_bf16(sv[cc * 8 + 4], sv[cc * 8 + 5]);
        pk.w = pack_bf16(sv[cc * 8 + 6], sv[cc * 8 + 7]);
        *reinterpret_cast<uint4*>(sm + L::oQ0 + bf * L::BUF + tc::sw128(r, 32 * wg + cc * 8)) = pk;
      }
      if (jt + 1 < n_tiles) confirm(bf ^ 1, false);   // tile jt+1's rows, copied last tile
      tc::fence_async_smem();
      tc::before_sync();
      if (__syncthreads_or(bad)) break;
      if (tid == 0) {
        tc::after_sync();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma(tmem_base + 128, tc::desc(aQ0 + bf * L::BUF + kk * 32), tc::desc(aV + kk * 32), idO, kk > 0);
        tc::commit(&bar_o);
        if (jt + 1 < n_tiles) issue_s(jt + 1);   // overlaps this tile's epilogue
      }
      if (!tc::bar_wait(&bar_o, jt & 1)) bad = true;
      tc::after_sync();
      // epilogue: this warpgroup's D/2 columns in rounds of 32 through its staging tile
      // (row r at +128 r, 16-byte chunks swizzled by r & 7); the lane holding a query's
      // first head adds the query's G x 32 box into the accumulator
      const uint32_t stg = aQ0 + bf * L::BUF + wg * L::STAGE;
      unsigned char* stg_p = sm + L::oQ0 + bf * L::BUF + wg * L::STAGE;
      const bool issuer = h == 0 && qi >= 0;
      const int unit = (b * s.N + (qi < 0 ? 0 : qi)) * s.Hkv + kv;
#pragma unroll
      for (int rd = 0; rd < D / 64; ++rd) {
        const int c0 = wg * (D / 2) + 32 * rd;
        float ov[32];
        tc::tmem_ld32(tmem_base + 128 + c0 + lane_off, ov);
        if (rd > 0) {
          if (issuer) tc::bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(stg_p + r * 128 + ((c ^ (r & 7)) << 4)) =
              make_float4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
        tc::fence_async_smem();
        __syncwarp();
        if (issuer) {
          tc::tma_reduce_add3(&omap, c0, 0, unit, stg + r * 128);
          tc::bulk_commit();
        }
      }
      if (issuer) tc::bulk_wait_read<0>();          // Q[bf] is gathered into again below
      tc::before_sync();
      if (__syncthreads_or(bad)) break;
      if (jt + 2 < n_tiles) gather(jt + 2, bf);
    }
  }
  tc::cp_async_wait<0>();                          // copies still in flight after an abort
  tc::bulk_wait<0>();                              // reductions complete before exit
  tc::before_sync();
  if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, PISA_ETIMEOUT);
  if (warp == 0) tc::tmem_free(tmem_base, L::tmem_cols);
}

// lse = log sum_k exp(block_lse_k) over each row's valid slots, written to the caller's lse
// ([B,Hq,N]); one thread per row, rows in lse order (consecutive threads read consecutive
// rows of block_lse and idx).
__global__ void __launch_bounds__(256)
attn_rows_kernel(Dims s, const int32_t* __restrict__ idx, const float* __restrict__ block_lse,
                 float* __restrict__ lse_out) {
  const int64_t lrow = blockIdx.x * 256LL + threadIdx.x;            // (b*Hq + h)*N + i
  if (lrow >= static_cast<int64_t>(s.B) * s.N * s.Hq) return;
  const int i = static_cast<int>(lrow % s.N);
  const int64_t bh = lrow / s.N;
  const int h = static_cast<int>(bh % s.Hq), b = static_cast<int>(bh / s.Hq);
  const int32_t* id = idx + ((static_cast<int64_t>(b) * s.Hkv + h / s.G) * s.N + i) * s.K;
  const float* bl = block_lse + lrow * s.K;
  float m = neg_inf();
  for (int k = 0; k < s.K; ++k)
    if (id[k] >= 0) m = fmaxf(m, bl[k]);
  float den = 0.f;
  if (m != neg_inf())
    for (int k = 0; k < s.K; ++k)
      if (id[k] >= 0) den += expf(bl[k] - m);
  lse_out[lrow] = den > 0.f ? m + logf(den) : neg_inf();
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

// Tensor maps: K as 4-D [B, N, Hkv, d] (boxes of 64 tokens x 64 of one KV head), the
// accumulator as 3-D [B*N*Hkv, G, d] fp32 (boxes of one query's G heads x 32 columns).
int make_maps(const Dims& s, const void* K, const float* o_acc, CUtensorMap* km, CUtensorMap* om) {
  const uint64_t d = static_cast<uint64_t>(s.d);
  {
    const uint64_t dims[4] = {d, static_cast<uint64_t>(s.Hkv), static_cast<uint64_t>(s.N),
                              static_cast<uint64_t>(s.B)};
    const uint64_t st[3] = {d * 2, d * 2 * s.Hkv, d * 2 * s.Hkv * s.N};
    const uint32_t box[4] = {64, 1, 64, 1};
    if (int e = encode_tmap(km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, K, dims, st, box)) return e;
  }
  if (o_acc) {
    const uint64_t dims[3] = {d, static_cast<uint64_t>(s.G), static_cast<uint64_t>(s.B) * s.N * s.Hkv};
    const uint64_t st[2] = {d * 4, d * 4 * s.G};
    const uint32_t box[3] = {32, static_cast<uint32_t>(s.G), 1};
    if (int e = encode_tmap(om, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, o_acc, dims, st, box)) return e;
  } else {
    *om = *km;                                      // not read outside the output mode
  }
  return 0;
}

template <int D, int G, int MODE>
int tc_launch(const TcArgs& a, const CUtensorMap& km, const CUtensorMap& om, const char* name, cudaStream_t st) {
  const int smem = TcSmem<D, MODE>::bytes;
  cudaError_t e =
      cudaFuncSetAttribute(block_tc_kernel<D, G, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope ps(st, name);
  block_tc_kernel<D, G, MODE><<<static_cast<unsigned>(a.gp.max_items), kThreads, smem, st>>>(a, km, om);
  return cudaGetLastError();
}

template <int MODE>
int tc_dispatch(const TcArgs& a, const CUtensorMap& km, const CUtensorMap& om, const char* name, cudaStream_t st) {
#define PISA_TC_CASE(DD, GG) \
  if (a.s.d == DD && a.s.G == GG) return tc_launch<DD, GG, MODE>(a, km, om, name, st);
  PISA_TC_CASE(128, 1) PISA_TC_CASE(128, 2) PISA_TC_CASE(128, 4) PISA_TC_CASE(128, 8)
  PISA_TC_CASE(64, 1) PISA_TC_CASE(64, 2) PISA_TC_CASE(64, 4) PISA_TC_CASE(64, 8)
#undef PISA_TC_CASE
  return static_cast<int>(cudaErrorNotSupported);
}

TcArgs base_args(const Dims& s, const GroupPlan& gp, const void* Q, const int32_t* list, const int4* items,
                 const int32_t* n_items, int32_t* status) {
  TcArgs a{};
  a.s = s;
  a.Q = static_cast<const __nv_bfloat16*>(Q);
  a.gp = gp;
  a.list = list;
  a.items = items;
  a.n_items = n_items;
  a.status = status;
  return a;
}

}  // namespace

// Attention forward for d in {64, 128} and G in {1, 2, 4, 8}: [block LSE pass when
// head_lse is NULL] -> accumulator clear, row LSE -> output pass -> bf16 conversion.
int launch_attn_fwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       const float* head_lse, float* block_lse_ws, float* o_acc, void* O, float* lse,
                       int32_t* status, cudaStream_t st) {
  CUtensorMap km, om;
  int err = make_maps(s, K, o_acc, &km, &om);
  if (err) return err;
  TcArgs a = base_args(s, gp, Q, list, items, n_items, status);
  a.V = static_cast<const __nv_bfloat16*>(V);
  const float* hl = head_lse;
  if (!hl) {
    a.out = block_lse_ws;
    if ((err = tc_dispatch<kModeLse>(a, km, om, "attn_lse_tc", st))) return err;
    hl = block_lse_ws;
  }
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  {
    ProfScope ps(st, "attn_clear");
    if ((err = cudaMemsetAsync(o_acc, 0, static_cast<size_t>(rows) * s.d * 4, st))) return err;
  }
  {
    ProfScope ps(st, "attn_rows");
    attn_rows_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(s, idx, hl, lse);
  }
  if ((err = cudaGetLastError())) return err;
  a.lse_rows = lse;
  a.out = nullptr;
  if ((err = tc_dispatch<kModeOut>(a, km, om, "attn_fwd_tc", st))) return err;
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
