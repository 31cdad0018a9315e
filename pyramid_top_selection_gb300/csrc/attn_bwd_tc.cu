// Backward of the causal block-sparse attention on the fifth-generation tensor cores (d = 128).
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value of
// the work": during training the gradient passes only through the selected attention; the
// discrete selection takes none. With P = exp(s q.k - lse) (lse from the forward),
// D_i = dO_i . O_i and dS = P (dO . v - D):  dQ = s dS K,  dK = s dS^T Q,  dV = P^T dO.
//
// One CTA per work item (a leaf block of one selection unit and the rows = (query, head) that
// selected it, grouped as for the forward), one CTA per SM, warp-specialised so that the tensor
// cores, the softmax arithmetic, the row gathers and the dQ reductions of different tiles run at
// the same time. The item's 64 keys and values arrive once by TMA; its rows come in tiles of 128
// (row = TMEM lane). Roles, connected by mbarriers:
//   * producers (warps 12-15): gather a tile's Q and dO rows by cp.async into one of two stages;
//   * control (warp 16, one thread): per tile T, S = Q K^T and dP = dO V^T (M = 128 rows, N = 64
//     keys, K = d; K-major operands) into one of two TMEM stages, issued before tile T - 1's
//     second group; once T's P and dS tiles are written,
//         dV^T += dO^T P and dK^T += Q^T dS  (M = d, N = 64 keys, K = 128 rows; MN-major operands,
//                                             accumulated in TMEM over the whole item)
//         dQ = dS K                          (M = 128 rows, N = d, K = 64 keys; K MN-major)
//   * softmax (warps 0-7, two threads per row, 32 keys each): P = exp(s S - lse) and
//     dS = P (dP - D) from TMEM into bf16 tiles [row][key];
//   * dQ epilogue (warps 8-11): dQ (scaled by s) from TMEM, 32 columns per round, through two
//     swizzled staging tiles as TMA tensor reduce-adds of each query's G rows into the fp32 dQ
//     accumulator (the rows of a query chunk stay in L2); after the item's last tile, its dK^T
//     and dV^T columns are added into the fp32 key/value accumulators.
// Every wait is bounded (the launch's wait limit); a wait that gives up sets the CTA's abort
// flag and every role leaves its loop at its next wait; the CTA drains the MMAs, copies and
// reductions it issued, frees its tensor memory and ORs PISA_STATUS_TIMEOUT into the status
// word, which the output conversion turns into poisoned (NaN) gradients.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"
#include "tiles.cuh"
#include "tmap.h"

namespace pisa {

namespace {

constexpr int kThreads = 544;                  // softmax 0-255, epilogue 256-383, producers 384-511, control
constexpr int kRows = 128;                     // tile rows = TMEM lanes
constexpr int kD = 128;                        // head dimension of this kernel
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound of the drain waits (work already issued)

// TMEM columns: S and dP of stage st at 128 st and 128 st + 64; dV^T, dK^T (64 each); dQ (128).
constexpr uint32_t kColDV = 256, kColDK = 320, kColDQ = 384;

struct Smem {
  static constexpr int KV = 2 * 64 * 128;            // [64 keys x 128 dims] bf16, two SW128 chunks
  static constexpr int TILE = 2 * kRows * 128;       // [128 rows x 128 dims] bf16, two SW128 chunks
  static constexpr int PS = kRows * 128;             // [128 rows x 64 keys] bf16, SW128
  static constexpr int STG = kRows * 128;            // [128 rows x 32] fp32, SW128
  static constexpr int oK = 0, oV = oK + KV, oQ = oV + KV, odO = oQ + 2 * TILE, oP = odO + 2 * TILE,
                       odS = oP + PS, oS = odS + PS;
  static constexpr int bytes = oS + 2 * STG + 1024;
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
  __shared__ __align__(8) uint64_t kv_bar, q_full[2], q_empty[2], s_full[2], s_empty[2], p_full, p_empty,
      dq_full, dq_empty, drain, never;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;

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
  // list entry of tile j's row r (-1: padding), packed as query << 6 | slot
  auto entry = [&](int j, int r) {
    const int e = j * EPT + r / G;
    return e < v.n_ent ? a.src.list[v.beg + e] : -1;
  };

  if (tid == 0) {
    tc::bar_init(&kv_bar, 1);
    for (int k = 0; k < 2; ++k) {
      tc::bar_init(&q_full[k], kRows);
      tc::bar_init(&q_empty[k], 1);
      tc::bar_init(&s_full[k], 1);
      tc::bar_init(&s_empty[k], 2 * kRows);
    }
    tc::bar_init(&p_full, 2 * kRows);
    tc::bar_init(&p_empty, 1);
    tc::bar_init(&dq_full, 1);
    tc::bar_init(&dq_empty, kRows);
    tc::bar_init(&drain, 1);
    tc::bar_init(&never, 1);
    tc::fence_bar_init();
    s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  tc::before_sync();
  __syncthreads();
  tc::after_sync();
  const uint32_t tm = tmem_base;
  auto give_up = [&]() { atomicOr(&s_abort, 1); };
  auto wait = [&](uint64_t* bar, uint32_t parity) { return tc::bar_wait(bar, parity, a.wait_ns); };

  if (warp >= 12 && warp < 16) {
    // ---------------------------------------------------------------- producers
    // thread: chunk (lane & 15) of two rows per instruction, rows wr .. wr + 31 of the tile; the
    // tile's copies are waited for and confirmed before the next stage is awaited, so no
    // unconfirmed copies are held while blocking (the stages are released only after the
    // second MMA group, which needs the next tile's S)
    const int wr = (warp - 12) * 32, c = lane & 15;
    int pk = n_tiles > 0 ? entry(0, wr + lane) : -1;
    for (int T = 0; T < n_tiles; ++T) {
      const int pk_n = T + 1 < n_tiles ? entry(T + 1, wr + lane) : -1;   // in flight meanwhile
      const int st = T & 1;
      const bool ok = wait(&q_empty[st], ((T >> 1) & 1) ^ 1);
      if (!__all_sync(0xffffffffu, ok)) { give_up(); break; }
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int rl = 2 * k + (lane >> 4);
        const int qpk = __shfl_sync(0xffffffffu, pk, rl);
        const int r = wr + rl;
        const int64_t row = (static_cast<int64_t>(v.b) * s.N + (qpk < 0 ? 0 : (qpk >> 6))) * s.Hq + v.kv * G + r % G;
        const uint32_t off = st * L::TILE + (c >> 3) * (kRows * 128) + tc::sw128(r, (c & 7) * 8);
        tc::cp_async16(aQ + off, a.Q + row * kD + c * 8, qpk >= 0);
        tc::cp_async16(adO + off, a.dO + row * kD + c * 8, qpk >= 0);
      }
      tc::cp_async_commit();
      tc::cp_async_wait<0>();
      tc::fence_async_smem();
      tc::bar_arrive(&q_full[st]);
      pk = pk_n;
    }
    tc::cp_async_wait<0>();
  } else if (warp == 16) {
    // ---------------------------------------------------------------- control
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kRows, 64);                   // S, dP
      constexpr uint32_t idKV = tc::idesc_bf16_major(kD, 64, true, true);   // dV^T, dK^T
      constexpr uint32_t idQ = tc::idesc_bf16_major(kRows, kD, false, true);  // dQ
      bool kv_landed = false, mma_issued = false, ok = true;
      tc::bar_expect_tx(&kv_bar, 2 * L::KV);
      for (int kb = 0; kb < 2; ++kb) {
        tc::tma_load4(aK + kb * (64 * 128), &kmap, kb * 64, kvk, v.kbase, v.b, &kv_bar);
        tc::tma_load4(aV + kb * (64 * 128), &vmap, kb * 64, kvk, v.kbase, v.b, &kv_bar);
      }
      auto issue_s = [&](int T) -> bool {            // S and dP of tile T
        const int st = T & 1;
        if (!wait(&q_full[st], (T >> 1) & 1) || !wait(&s_empty[st], ((T >> 1) & 1) ^ 1)) return false;
        tc::after_sync();
        mma_issued = true;
        const uint32_t q = aQ + st * L::TILE, o = adO + st * L::TILE;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t ka = (k >> 2) * (kRows * 128) + (k & 3) * 32, kb = (k >> 2) * (64 * 128) + (k & 3) * 32;
          tc::mma(tm + 128 * st, tc::desc(q + ka), tc::desc(aK + kb), idS, k > 0);
          tc::mma(tm + 128 * st + 64, tc::desc(o + ka), tc::desc(aV + kb), idS, k > 0);
        }
        tc::commit(&s_full[st]);
        return true;
      };
      kv_landed = wait(&kv_bar, 0);
      ok = kv_landed;
      if (ok && a.stall) ok = wait(&never, 0);      // test aid: runs out after the wait limit
      if (ok && n_tiles > 0) ok = issue_s(0);
      for (int T = 0; ok && T < n_tiles; ++T) {
        if (*reinterpret_cast<volatile int*>(&s_abort)) { ok = false; break; }
        if (T + 1 < n_tiles && !issue_s(T + 1)) { ok = false; break; }   // runs under T's softmax
        if (!wait(&p_full, T & 1) || (T > 0 && !wait(&dq_empty, (T - 1) & 1))) { ok = false; break; }
        tc::after_sync();
        const int st = T & 1;
        const uint32_t q = aQ + st * L::TILE, o = adO + st * L::TILE;
#pragma unroll
        for (int k = 0; k < kRows / 16; ++k) {
          const uint32_t rk = k * 2048;             // 16 rows of an MN-major operand
          tc::mma(tm + kColDV, tc::desc_mn(o + rk, kRows * 128), tc::desc_mn(aP + rk, 0), idKV, T > 0 || k > 0);
          tc::mma(tm + kColDK, tc::desc_mn(q + rk, kRows * 128), tc::desc_mn(adS + rk, 0), idKV, T > 0 || k > 0);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma(tm + kColDQ, tc::desc(adS + k * 32), tc::desc_mn(aK + k * 2048, 64 * 128), idQ, k > 0);
        tc::commit(&q_empty[st]);
        tc::commit(&p_empty);
        tc::commit(&dq_full);
      }
      if (!ok) give_up();
      // drain: the key/value tiles land and every MMA issued completes before the CTA leaves
      if (!kv_landed) tc::bar_wait(&kv_bar, 0, kDrainNs);
      if (mma_issued) {
        tc::commit(&drain);
        tc::bar_wait(&drain, 0, kDrainNs);
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax
    // thread: row r (TMEM lane), keys 32 hs .. 32 hs + 31; the next tile's row metadata
    // (lse * log2e, D, query) loads during this tile
    const int r = tid & (kRows - 1), hs = warp >> 2, h = r % G;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c1 = s.scale * kLog2e;
    auto meta = [&](int j, float& l2, float& D) {
      const int pk = entry(j, r);
      l2 = D = 0.f;
      if (pk >= 0) {
        const int qi = pk >> 6;
        l2 = a.lse[(static_cast<int64_t>(v.b) * s.Hq + v.kv * G + h) * s.N + qi] * kLog2e;
        D = a.delta[(static_cast<int64_t>(v.b) * s.N + qi) * s.Hq + v.kv * G + h];
      }
      return pk;
    };
    float l2 = 0.f, D = 0.f;
    int pk = n_tiles > 0 ? meta(0, l2, D) : -1;
    for (int T = 0; T < n_tiles; ++T) {
      float l2_n = 0.f, D_n = 0.f;
      const int pk_n = T + 1 < n_tiles ? meta(T + 1, l2_n, D_n) : -1;
      const int st = T & 1;
      const bool ok = wait(&s_full[st], (T >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { give_up(); break; }
      tc::after_sync();
      float sv[32], dp[32];
      tc::tmem_ld32(tm + 128 * st + 32 * hs + lane_off, sv);
      tc::tmem_ld32(tm + 128 * st + 64 + 32 * hs + lane_off, dp);
      tc::before_sync();
      tc::bar_arrive(&s_empty[st]);
      const int lim = pk < 0 ? -1 : (pk >> 6) - v.kbase - 32 * hs;   // key c of the half visible iff c <= lim
      const uint64_t cc = tc::pack2(c1, c1), ll = tc::pack2(-l2, -l2), dd = tc::pack2(-D, -D);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {             // packed pairs: exponent arguments, dP - D, P (dP - D)
        float y0, y1, e0, e1;
        tc::unpack2(tc::fma2(tc::pack2(sv[c], sv[c + 1]), cc, ll), y0, y1);
        const float p0 = c <= lim ? tc::ex2(y0) : 0.f, p1 = c + 1 <= lim ? tc::ex2(y1) : 0.f;
        sv[c] = p0;
        sv[c + 1] = p1;
        tc::unpack2(tc::add2(tc::pack2(dp[c], dp[c + 1]), dd), e0, e1);
        dp[c] = p0 * e0;
        dp[c + 1] = p1 * e1;
      }
      const bool ok2 = wait(&p_empty, (T & 1) ^ 1);   // tile T - 1's second group has read P and dS
      if (!__all_sync(0xffffffffu, ok2)) { give_up(); break; }
      unsigned char* pt = sm + L::oP;
      unsigned char* dt = sm + L::odS;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t off = tc::sw128(r, 32 * hs + k * 8);
        *reinterpret_cast<uint4*>(pt + off) =
            make_uint4(pack_bf16(sv[k * 8 + 0], sv[k * 8 + 1]), pack_bf16(sv[k * 8 + 2], sv[k * 8 + 3]),
                       pack_bf16(sv[k * 8 + 4], sv[k * 8 + 5]), pack_bf16(sv[k * 8 + 6], sv[k * 8 + 7]));
        *reinterpret_cast<uint4*>(dt + off) =
            make_uint4(pack_bf16(dp[k * 8 + 0], dp[k * 8 + 1]), pack_bf16(dp[k * 8 + 2], dp[k * 8 + 3]),
                       pack_bf16(dp[k * 8 + 4], dp[k * 8 + 5]), pack_bf16(dp[k * 8 + 6], dp[k * 8 + 7]));
      }
      tc::fence_async_smem();
      tc::bar_arrive(&p_full);
      pk = pk_n;
      l2 = l2_n;
      D = D_n;
    }
  } else if (warp < 12) {
    // ---------------------------------------------------------------- dQ epilogue
    // row r's dQ, 32 columns per round, into staging tile (round & 1) at +128 r with 16-byte
    // chunks swizzled by r & 7; every lane commits one bulk group per round (empty unless it
    // issued), so "all but the newest group read out" means the other tile is free again
    const int r = tid - 256, h = r % G;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int pk = n_tiles > 0 ? entry(0, r) : -1;
    int rd_all = 0;
    bool ok = true;
    for (int T = 0; T < n_tiles; ++T) {
      const int pk_n = T + 1 < n_tiles ? entry(T + 1, r) : -1;
      ok = wait(&dq_full, T & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; give_up(); break; }
      tc::after_sync();
      const bool issuer = h == 0 && pk >= 0;
      const int unit = (v.b * s.N + (pk < 0 ? 0 : (pk >> 6))) * s.Hkv + v.kv;
#pragma unroll 1
      for (int rd = 0; rd < kD / 32; ++rd, ++rd_all) {
        float x[32];
        tc::tmem_ld32(tm + kColDQ + 32 * rd + lane_off, x);
        if (rd == kD / 32 - 1) {                      // dQ's columns are free for tile T + 1
          tc::before_sync();
          tc::bar_arrive(&dq_empty);
        }
        const int sb = rd_all & 1;
        tc::bulk_wait_read<1>();
        __syncwarp();
        unsigned char* stg = sm + L::oS + sb * L::STG;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(stg + r * 128 + ((c ^ (r & 7)) << 4)) =
              make_float4(s.scale * x[4 * c], s.scale * x[4 * c + 1], s.scale * x[4 * c + 2], s.scale * x[4 * c + 3]);
        tc::fence_async_smem();
        __syncwarp();
        if (issuer) tc::tma_reduce_add3(&qmap, 32 * rd, 0, unit, aS + sb * L::STG + r * 128);
        tc::bulk_commit();
      }
      pk = pk_n;
    }
    // the item's dK and dV columns (dQ's last commit covers every MMA): thread = dimension r
    if (ok && n_tiles > 0) {
      tc::after_sync();
#pragma unroll 1
      for (int w = 0; w < 2; ++w) {
        float* acc = w == 0 ? a.dv_acc : a.dk_acc;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float x[32];
          tc::tmem_ld32(tm + (w == 0 ? kColDV : kColDK) + 32 * h2 + lane_off, x);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int64_t jk = static_cast<int64_t>(v.kbase) + 32 * h2 + c;
            if (jk < s.N) atomicAdd(acc + ((static_cast<int64_t>(v.b) * s.N + jk) * s.Hkv_r + kvk) * kD + r, x[c]);
          }
        }
      }
    }
    tc::bulk_wait<0>();
  }
  tc::before_sync();
  __syncthreads();
  if (tid == 0 && s_abort) atomicOr(a.status, PISA_STATUS_TIMEOUT);
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
