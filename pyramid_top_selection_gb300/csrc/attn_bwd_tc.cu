// Backward of the causal block-sparse attention on the fifth-generation tensor cores (d = 128).
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value of
// the work": during training the gradient passes only through the selected attention; the
// discrete selection takes none. With P = exp(s q.k - lse) (lse from the forward),
// D_i = dO_i . O_i and dS = P (dO . v - D):  dQ = s dS K,  dK = s dS^T Q,  dV = P^T dO.
//
// One CTA per work item (a leaf block of one selection unit and the rows = (query, head) that
// selected it, grouped as for the forward), 8 warps, one CTA per SM. The item's 64 keys and
// values arrive once by TMA; its rows come in tiles of 128 (row = TMEM lane), gathered by
// cp.async into two buffers (the next tile's Q and dO rows land while this one is computed).
// Per tile, one thread issues
//     S = Q K^T and dP = dO V^T          (M = 128 rows, N = 64 keys, K = d; K-major operands)
// into TMEM; every row's P and dS are computed by two threads (32 keys each) and written as
// bf16 tiles [row][key]; then
//     dV^T += dO^T P and dK^T += Q^T dS  (M = d, N = 64 keys, K = 128 rows; MN-major operands,
//                                         accumulated in TMEM over the whole item)
//     dQ = dS K                          (M = 128 rows, N = d, K = 64 keys; K MN-major)
// and dQ (scaled by s) leaves TMEM through a staging tile as TMA tensor reduce-adds into the
// fp32 dQ accumulator (the rows of a query chunk stay in L2). At the item's end its dK^T and
// dV^T columns are added into the fp32 key/value accumulators. Every wait is bounded (the
// launch's wait limit); a wait that gives up makes the whole CTA leave its loop, drain the MMAs,
// copies and reductions it issued, free its tensor memory and OR PISA_STATUS_TIMEOUT into the
// status word, which the output conversion turns into poisoned (NaN) gradients.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"
#include "tiles.cuh"
#include "tmap.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 128;                     // tile rows = TMEM lanes
constexpr int kD = 128;                        // head dimension of this kernel
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound of the drain waits (work already issued)

// TMEM columns: S, dP, dV^T, dK^T (64 each), dQ (128).
constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 128, kColDK = 192, kColDQ = 256;

struct Smem {
  static constexpr int KV = 2 * 64 * 128;            // [64 keys x 128 dims] bf16, two SW128 chunks
  static constexpr int TILE = 2 * kRows * 128;       // [128 rows x 128 dims] bf16, two SW128 chunks
  static constexpr int PS = kRows * 128;             // [128 rows x 64 keys] bf16, SW128
  static constexpr int STG = kRows * 128;            // [128 rows x 32] fp32, SW128 chunks
  static constexpr int oK = 0, oV = oK + KV, oQ = oV + KV, odO = oQ + 2 * TILE, oP = odO + 2 * TILE,
                       odS = oP + PS, oS = odS + PS;
  static constexpr int bytes = oS + STG + 1024;
};

struct BwdTcArgs {
  Dims s;
  ItemSource src;
  const __nv_bfloat16* Q;
  const __nv_bfloat16* dO;
  const float* lse;        // [B, Hq, N]
  const float* delta;      // [B, N, Hq]
  const int32_t* n_items;
  float* dk_acc;           // [B, N, Hkv_r, d] fp32
  float* dv_acc;
  int32_t* status;
  uint64_t wait_ns;
  int stall;
};

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_tc_kernel(const BwdTcArgs a, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
  using L = Smem;
  constexpr int EPT = kRows / G;                     // list entries (queries) per tile
  extern __shared__ unsigned char smraw[];
  __shared__ __align__(8) uint64_t kv_bar, mma_bar, drain, never;
  __shared__ uint32_t tmem_base;
  __shared__ float m_lse2[2][kRows], m_D[2][kRows];
  __shared__ int m_qi[2][kRows];

  const Dims& s = a.s;
  if (static_cast<int>(blockIdx.x) >= *a.n_items) return;
  const ItemView v = view_of(a.src, a.src.items[blockIdx.x]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* sm = smraw + ((1024 - (tc::su32(smraw) & 1023)) & 1023);
  const uint32_t aK = tc::su32(sm + L::oK), aV = tc::su32(sm + L::oV), aQ = tc::su32(sm + L::oQ),
                 adO = tc::su32(sm + L::odO), aP = tc::su32(sm + L::oP), adS = tc::su32(sm + L::odS),
                 aS = tc::su32(sm + L::oS);
  const int n_tiles = (v.n_ent + EPT - 1) / EPT;
  const int kvk = v.kv / s.kvr;                      // the unit's KV head

  if (tid == 0) {
    tc::bar_init(&kv_bar, 1);
    tc::bar_init(&mma_bar, 1);
    tc::bar_init(&drain, 1);
    tc::bar_init(&never, 1);
    tc::fence_bar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  tc::before_sync();
  __syncthreads();
  tc::after_sync();
  const uint32_t tm = tmem_base;

  // the item's keys and values: two 64-dim boxes each, one transaction barrier
  if (tid == 0) {
    tc::bar_expect_tx(&kv_bar, 2 * L::KV);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load4(aK + kb * (64 * 128), &kmap, kb * 64, kvk, v.kbase, v.b, &kv_bar);
      tc::tma_load4(aV + kb * (64 * 128), &vmap, kb * 64, kvk, v.kbase, v.b, &kv_bar);
    }
  }

  // A tile's list entries, loaded one tile ahead of its gather: entries of the thread's 8
  // gather rows ((tid >> 4) + 16u) and, for threads < 128, of metadata row tid.
  struct Entries {
    int pk[8];
    int mpk;
  };
  auto load_entries = [&](int j, Entries& en) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = j * EPT + ((tid >> 4) + 16 * u) / G;
      en.pk[u] = e < v.n_ent ? a.src.list[v.beg + e] : -1;
    }
    const int e = j * EPT + (tid & (kRows - 1)) / G;
    en.mpk = tid < kRows && e < v.n_ent ? a.src.list[v.beg + e] : -1;
  };
  // gather of a tile into buffer bf: the thread copies 16-byte chunk (tid & 15) of its rows
  auto gather = [&](const Entries& en, int bf) {
    const int c = tid & 15;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = (tid >> 4) + 16 * u, pk = en.pk[u];
      const int64_t row = (static_cast<int64_t>(v.b) * s.N + (pk < 0 ? 0 : (pk >> 6))) * s.Hq + v.kv * G + r % G;
      const uint32_t off = bf * L::TILE + (c >> 3) * (kRows * 128) + tc::sw128(r, (c & 7) * 8);
      tc::cp_async16(aQ + off, a.Q + row * kD + c * 8, pk >= 0);
      tc::cp_async16(adO + off, a.dO + row * kD + c * 8, pk >= 0);
    }
    tc::cp_async_commit();
  };
  // metadata of row tid (threads < 128): lse * log2e, D, query (-1: padding); loaded into
  // registers when the tile's gather is issued, stored to shared memory a phase later
  float ml2 = 0.f, mD = 0.f;
  int mqi = -1;
  auto meta_load = [&](const Entries& en) {
    const int h = tid % G;
    mqi = en.mpk < 0 ? -1 : (en.mpk >> 6);
    ml2 = mD = 0.f;
    if (mqi >= 0) {
      ml2 = a.lse[(static_cast<int64_t>(v.b) * s.Hq + v.kv * G + h) * s.N + mqi] * kLog2e;
      mD = a.delta[(static_cast<int64_t>(v.b) * s.N + mqi) * s.Hq + v.kv * G + h];
    }
  };
  auto meta_store = [&](int bf) {
    if (tid < kRows) {
      m_lse2[bf][tid] = ml2;
      m_D[bf][tid] = mD;
      m_qi[bf][tid] = mqi;
    }
  };

  bool ok = true;
  bool mma_issued = false, kv_landed = false;
  const int r = tid & (kRows - 1), hf = tid >> 7;      // a thread's tile row and half of it
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const float c1 = s.scale * kLog2e;
  constexpr uint32_t idS = tc::idesc_bf16(kRows, 64);                  // S, dP
  constexpr uint32_t idKV = tc::idesc_bf16_major(kD, 64, true, true);   // dV^T, dK^T
  constexpr uint32_t idQ = tc::idesc_bf16_major(kRows, kD, false, true);  // dQ
  uint32_t mma_phase = 0;
  auto wait_mma = [&]() {
    const bool w = tc::bar_wait(&mma_bar, mma_phase, a.wait_ns);
    mma_phase ^= 1;
    return w;
  };
  // dQ of the previous tile, row r, columns 64 hf .. 64 hf + 63 (scaled by s), and its query
  float dqr[2][32];
  int dq_qi = -1;
  // the previous tile's dQ into the fp32 accumulator: two rounds of 32 columns per thread half,
  // staged in the P and dS tiles (free once that tile's MMAs completed), one TMA reduce-add per
  // query (its G rows) and staging buffer
  auto dq_out = [&]() {
    const bool issuer = dq_qi >= 0 && r % G == 0;
    const int unit = (v.b * s.N + (dq_qi < 0 ? 0 : dq_qi)) * s.Hkv + v.kv;
    const uint32_t stg_a = hf == 0 ? aP : adS;
    unsigned char* stg = sm + (hf == 0 ? L::oP : L::odS);
#pragma unroll
    for (int rd = 0; rd < 2; ++rd) {
      const float* x = dqr[rd];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(stg + r * 128 + ((c ^ (r & 7)) << 4)) =
            make_float4(s.scale * x[4 * c], s.scale * x[4 * c + 1], s.scale * x[4 * c + 2], s.scale * x[4 * c + 3]);
      tc::fence_async_smem();
      __syncthreads();
      if (issuer) {
        tc::tma_reduce_add3(&qmap, 64 * hf + 32 * rd, 0, unit, stg_a + r * 128);
        tc::bulk_commit();
        tc::bulk_wait_read<0>();
      }
      __syncthreads();
    }
  };

  Entries ent;
  if (n_tiles > 0) {
    load_entries(0, ent);
    gather(ent, 0);
    meta_load(ent);
    meta_store(0);
    if (n_tiles > 1) load_entries(1, ent);
  }
  for (int j = 0; j < n_tiles; ++j) {
    const int bf = j & 1;
    if (j + 1 < n_tiles) {
      gather(ent, bf ^ 1);                        // buffer bf ^ 1: tile j - 1's MMAs are complete
      meta_load(ent);                             // in flight; stored below
      if (j + 2 < n_tiles) load_entries(j + 2, ent);
      tc::cp_async_wait<1>();
    } else {
      tc::cp_async_wait<0>();
    }
    tc::fence_async_smem();                       // the copies land in the async proxy's view
    __syncthreads();
    // S and dP of tile j
    if (tid == 0) {
      if (!kv_landed) {
        kv_landed = tc::bar_wait(&kv_bar, 0, a.wait_ns);
        ok = kv_landed;
        if (ok && a.stall) ok = tc::bar_wait(&never, 0, a.wait_ns);   // test aid: runs out
      }
      if (ok) {
        tc::after_sync();
        const uint32_t q = aQ + bf * L::TILE, o = adO + bf * L::TILE;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t ka = (k >> 2) * (kRows * 128) + (k & 3) * 32, kb = (k >> 2) * (64 * 128) + (k & 3) * 32;
          tc::mma(tm + kColS, tc::desc(q + ka), tc::desc(aK + kb), idS, k > 0);
          tc::mma(tm + kColDP, tc::desc(o + ka), tc::desc(aV + kb), idS, k > 0);
        }
        tc::commit(&mma_bar);
        mma_issued = true;
      }
    }
    if (!__syncthreads_and(ok)) break;
    // meanwhile, the previous tile's dQ leaves through the P/dS tiles
    if (j > 0) dq_out();
    ok = wait_mma();
    if (!__syncthreads_and(ok)) break;
    tc::after_sync();
    // P and dS of the thread's 32 keys of row r
    {
      float sv[32], dp[32];
      tc::tmem_ld32(tm + kColS + 32 * hf + lane_off, sv);
      tc::tmem_ld32(tm + kColDP + 32 * hf + lane_off, dp);
      const int qi = m_qi[bf][r];
      const int lim = qi < 0 ? -1 : qi - v.kbase - 32 * hf;   // key c of the half visible iff c <= lim
      const float l2 = m_lse2[bf][r], D = m_D[bf][r];
      const uint64_t cc = tc::pack2(c1, c1), ll = tc::pack2(-l2, -l2), dd = tc::pack2(-D, -D);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {           // packed pairs: exponent arguments, dP - D, P (dP - D)
        float y0, y1, e0, e1;
        tc::unpack2(tc::fma2(tc::pack2(sv[c], sv[c + 1]), cc, ll), y0, y1);
        const float p0 = c <= lim ? tc::ex2(y0) : 0.f, p1 = c + 1 <= lim ? tc::ex2(y1) : 0.f;
        sv[c] = p0;
        sv[c + 1] = p1;
        tc::unpack2(tc::add2(tc::pack2(dp[c], dp[c + 1]), dd), e0, e1);
        dp[c] = p0 * e0;
        dp[c + 1] = p1 * e1;
      }
      unsigned char* pt = sm + L::oP;
      unsigned char* st = sm + L::odS;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t off = tc::sw128(r, 32 * hf + cc * 8);
        *reinterpret_cast<uint4*>(pt + off) =
            make_uint4(pack_bf16(sv[cc * 8 + 0], sv[cc * 8 + 1]), pack_bf16(sv[cc * 8 + 2], sv[cc * 8 + 3]),
                       pack_bf16(sv[cc * 8 + 4], sv[cc * 8 + 5]), pack_bf16(sv[cc * 8 + 6], sv[cc * 8 + 7]));
        *reinterpret_cast<uint4*>(st + off) =
            make_uint4(pack_bf16(dp[cc * 8 + 0], dp[cc * 8 + 1]), pack_bf16(dp[cc * 8 + 2], dp[cc * 8 + 3]),
                       pack_bf16(dp[cc * 8 + 4], dp[cc * 8 + 5]), pack_bf16(dp[cc * 8 + 6], dp[cc * 8 + 7]));
      }
      dq_qi = qi;                                 // this tile's query of row r, for its dQ
    }
    tc::fence_async_smem();
    tc::before_sync();
    __syncthreads();
    // dV^T += dO^T P, dK^T += Q^T dS (over the tile's 128 rows), dQ = dS K (over the 64 keys)
    if (tid == 0) {
      tc::after_sync();
      const uint32_t q = aQ + bf * L::TILE, o = adO + bf * L::TILE;
#pragma unroll
      for (int k = 0; k < kRows / 16; ++k) {
        const uint32_t rk = k * 2048;             // 16 rows of an MN-major operand
        tc::mma(tm + kColDV, tc::desc_mn(o + rk, kRows * 128), tc::desc_mn(aP + rk, 0), idKV, j > 0 || k > 0);
        tc::mma(tm + kColDK, tc::desc_mn(q + rk, kRows * 128), tc::desc_mn(adS + rk, 0), idKV, j > 0 || k > 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma(tm + kColDQ, tc::desc(adS + k * 32), tc::desc_mn(aK + k * 2048, 64 * 128), idQ, k > 0);
      tc::commit(&mma_bar);
    }
    if (j + 1 < n_tiles) meta_store(bf ^ 1);      // the next tile's metadata (loads issued above)
    ok = wait_mma();
    if (!__syncthreads_and(ok)) break;
    tc::after_sync();
    tc::tmem_ld32(tm + kColDQ + 64 * hf + lane_off, dqr[0]);
    tc::tmem_ld32(tm + kColDQ + 64 * hf + 32 + lane_off, dqr[1]);
    tc::before_sync();
  }
  if (__syncthreads_and(ok) && n_tiles > 0) dq_out();   // the last tile's dQ
  // every thread takes the same branch below (a loop left early leaves per-thread flags apart)
  const bool all_ok = __syncthreads_and(ok);
  // the item's dK and dV columns: warps 0-3 read dV^T, warps 4-7 dK^T (thread = dimension)
  if (all_ok && n_tiles > 0) {
    tc::after_sync();
    float x[2][32];
    const uint32_t col = warp < 4 ? kColDV : kColDK;
    tc::tmem_ld32(tm + col + lane_off, x[0]);
    tc::tmem_ld32(tm + col + 32 + lane_off, x[1]);
    float* acc = warp < 4 ? a.dv_acc : a.dk_acc;
    const int dim = (warp & 3) * 32 + lane;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int64_t jk = static_cast<int64_t>(v.kbase) + 32 * h2 + c;
        if (jk < s.N)
          atomicAdd(acc + ((static_cast<int64_t>(v.b) * s.N + jk) * s.Hkv_r + kvk) * kD + dim, x[h2][c]);
      }
  }
  // drain what was issued, then free the tensor memory
  tc::cp_async_wait<0>();
  tc::bulk_wait<0>();
  if (tid == 0) {
    if (!kv_landed) tc::bar_wait(&kv_bar, 0, kDrainNs);
    if (mma_issued) {
      tc::commit(&drain);
      tc::bar_wait(&drain, 0, kDrainNs);
    }
    if (!all_ok) atomicOr(a.status, PISA_STATUS_TIMEOUT);
  }
  tc::before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::after_sync();
    tc::tmem_free(tm, 512);
  }
}

}  // namespace

// Tensor-core backward pass over the grouped (selected leaf, rows) work items, d = 128:
// dQ scaled by s into dq_acc [B, N, Hq, d] fp32, dK (unscaled) and dV into dk_acc / dv_acc
// [B, N, Hkv_r, d] fp32.
int launch_attn_bwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const void* dO, const float* lse, const float* delta, const int32_t* list,
                       const int4* items, const int32_t* n_items, float* dq_acc, float* dk_acc, float* dv_acc,
                       int32_t* status, cudaStream_t st) {
  if (s.d != kD) return static_cast<int>(cudaErrorNotSupported);
  CUtensorMap km, vm, qm;
  const uint64_t d = kD;
  {
    const uint64_t dims[4] = {d, static_cast<uint64_t>(s.Hkv_r), static_cast<uint64_t>(s.N),
                              static_cast<uint64_t>(s.B)};
    const uint64_t strides[3] = {d * 2, d * 2 * s.Hkv_r, d * 2 * s.Hkv_r * s.N};
    const uint32_t box[4] = {64, 1, 64, 1};
    if (int e = encode_tmap(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, K, dims, strides, box)) return e;
    if (int e = encode_tmap(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, V, dims, strides, box)) return e;
  }
  {
    const uint64_t dims[3] = {d, static_cast<uint64_t>(s.G), static_cast<uint64_t>(s.B) * s.N * s.Hkv};
    const uint64_t strides[2] = {d * 4, d * 4 * s.G};
    const uint32_t box[3] = {32, static_cast<uint32_t>(s.G), 1};
    if (int e = encode_tmap(&qm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dq_acc, dims, strides, box)) return e;
  }
  BwdTcArgs a{};
  a.s = s;
  a.src.gp = gp;
  a.src.items = items;
  a.src.list = list;
  a.src.Hkv = s.Hkv;
  a.Q = static_cast<const __nv_bfloat16*>(Q);
  a.dO = static_cast<const __nv_bfloat16*>(dO);
  a.lse = lse;
  a.delta = delta;
  a.n_items = n_items;
  a.dk_acc = dk_acc;
  a.dv_acc = dv_acc;
  a.status = status;
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  const int smem = Smem::bytes;
  auto run = [&](auto kernel) -> int {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ProfScope ps(st, "attn_bwd");
    kernel<<<static_cast<unsigned>(gp.max_items), kThreads, smem, st>>>(a, km, vm, qm);
    return cudaGetLastError();
  };
  switch (s.G) {
    case 1: return run(attn_bwd_tc_kernel<1>);
    case 2: return run(attn_bwd_tc_kernel<2>);
    case 4: return run(attn_bwd_tc_kernel<4>);
    default: return run(attn_bwd_tc_kernel<8>);
  }
}

}  // namespace pisa
