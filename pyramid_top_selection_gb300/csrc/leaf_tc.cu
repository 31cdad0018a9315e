// Stage-2 exact leaf scoring on the fifth-generation tensor cores: a persistent,
// warp-specialised kernel.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Method key
// points": leaves are scored by the exact LSE over their raw keys and the G query heads of a
// KV head sum their LSEs; "Reference value of the work": the queries that use the same leaf
// block are grouped into tiles so the block's keys are read once per tile.
//
// One CTA per SM takes work items (a candidate leaf of one KV head and the (query, head)
// rows that have it among their candidates; for the selection, a pair of sibling leaves, which
// a query's candidates hold together whenever both are visible, so each query row is gathered
// once for 128 keys and two LSEs: 1.18 -> 0.76 ms at the 64K workload) from a global counter
// through its item queue (tiles.cuh) and walks them in tiles of 128 rows. Roles, connected by
// mbarrier rings so that no role waits on another's latency:
//   * producers (4 warps after the softmax ones, 32 tile rows each): gather the query vectors with cp.async
//     into a 4-stage ring of swizzled Q tiles, each warp instruction copying whole rows
//     (full 32-byte sectors); a thread confirms a tile's copies (wait, proxy fence,
//     arrival) once it has issued the next tile;
//   * control (the next warp, one thread): loads each item's 64 or 128 keys by TMA into a 2-stage ring
//     (the next item's while the current one runs) and issues S = Q K^T (M=128, N=64) as
//     tcgen05.mma into a 4-stage ring of TMEM accumulators;
//   * softmax (two warpgroups, three when G = 8, taking the tiles in turn; thread = TMEM lane =
//     tile row): reads its S row, frees the TMEM stage, and reduces the row to its LSE over
//     the visible keys; the G rows of a query (adjacent lanes) sum their LSEs into the
//     candidate's score;
//   * scheduler (the last warp, one thread): fills the item queue.
// Every wait is bounded (the launch's wait limit); a wait that gives up sets the CTA's abort
// flag and every role leaves its loop at its next tile. Before the CTA frees its tensor memory
// the control thread drains what it issued (key tiles in flight, MMAs), the producers their
// copies; the kernel then ORs PISA_STATUS_TIMEOUT into the status word, and the top-K finish
// reads it and writes poisoned outputs.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"
#include "tiles.cuh"
#include "tmap.h"

namespace pisa {

namespace {

constexpr int kRows = 128;
constexpr int kNQ = 4;            // Q tile stages
constexpr int kNS = 4;            // TMEM S stages (64 columns each)
constexpr int kNK = 2;            // K tile stages
// Softmax warpgroups (tile T goes to group T % SG): three when G = 8 (0.760 -> 0.729 ms at the
// 64K workload), two otherwise (three: 1.433 -> 1.440 ms at the G = 4 sweep shape; 1.24 vs 1.18
// ms at G = 8 with one leaf per item).
#ifndef PISA_LEAF_SG8
#define PISA_LEAF_SG8 3
#endif
__host__ __device__ constexpr int sg_for(int G) { return G >= 8 ? PISA_LEAF_SG8 : 2; }
__host__ __device__ constexpr int threads_for(int G) { return 128 * sg_for(G) + 128 + 64; }   // softmax, producers (4 warps), control, scheduler
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound of the drain waits (work already issued)

// PR = 1: an item is a pair of sibling leaves (128 keys, two LSEs per row); PR = 0: one leaf.
template <int D, int PR>
struct LeafSmem {
  static constexpr int KB = D / 64;
  static constexpr int NK = 64 << PR;             // keys per item
  static constexpr int Q_BYTES = KB * kRows * 128;
  static constexpr int K_BYTES = KB * NK * 128;
  static constexpr int oQ = 0, oK = kNQ * Q_BYTES;
  static constexpr int bytes = oK + kNK * K_BYTES + 1024;
};

struct LeafArgs {
  Dims s;
  ItemSource src;
  const __nv_bfloat16* Q;
  const int32_t* n_items;
  int W;
  float* pair_score;   // [heads, N, W]
  float* pair_head;    // [heads, N, W, G] or NULL
  float* block_lse;    // when set: per-row LSE [B, Hq, N, W] instead of the scores
  int32_t* status;
  int32_t* next_item;  // zeroed item counter
  uint64_t wait_ns;    // bound of every pipeline wait
  int stall;           // test aid: wait on a barrier nothing signals before the first MMA
};

template <int D, int G, int PR>
__global__ void __launch_bounds__(threads_for(G), 1)
leaf_tc_kernel(const LeafArgs a, const __grid_constant__ CUtensorMap kmap) {
  using L = LeafSmem<D, PR>;
  constexpr int NK = L::NK;
  constexpr int EPT = kRows / G;          // entries (queries) per tile
  constexpr int CH = D / 8;               // 16-byte chunks per row
  constexpr int kSG = sg_for(G);          // softmax warpgroups
  constexpr int kWP = 4 * kSG;            // first producer warp
  constexpr int kConsumerWarps = 4 * kSG + 5;
  extern __shared__ unsigned char smraw[];
  __shared__ __align__(8) uint64_t q_full[kNQ], q_empty[kNQ], s_full[kNS], s_empty[kNS], k_full[kNK],
      k_empty[kNK], drain, never;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  __shared__ ItemQueue s_q;

  const Dims& s = a.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* sm = smraw + ((1024 - (tc::su32(smraw) & 1023)) & 1023);
  const uint32_t aQ = tc::su32(sm + L::oQ), aK = tc::su32(sm + L::oK);
  const int n_items = *a.n_items;

  if (tid == 0) {
    for (int k = 0; k < kNQ; ++k) {
      tc::bar_init(&q_full[k], kRows);
      tc::bar_init(&q_empty[k], 1);
    }
    for (int k = 0; k < kNS; ++k) {
      tc::bar_init(&s_full[k], 1);
      tc::bar_init(&s_empty[k], kRows);
    }
    for (int k = 0; k < kNK; ++k) {
      tc::bar_init(&k_full[k], 1);
      tc::bar_init(&k_empty[k], 1);
    }
    tc::bar_init(&drain, 1);
    tc::bar_init(&never, 1);
    queue_init(s_q, kConsumerWarps, a.wait_ns);
    tc::fence_bar_init();
    s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kNS * NK);
  tc::before_sync();
  __syncthreads();
  tc::after_sync();
  auto give_up = [&]() { atomicOr(&s_abort, 1); };
  auto wait = [&](uint64_t* bar, uint32_t parity) { return tc::bar_wait(bar, parity, a.wait_ns); };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };

  if (warp >= kWP && warp < kWP + 4) {
    // ---------------------------------------------------------------- producers
    // the next tile's list entries (and item) load while this tile's copies are issued; lane
    // l holds the entry of the warp's row l, and instruction k copies rows k*RPI .. of the
    // warp's 32, chunk (lane % CH) of row (lane / CH)
    constexpr int RPI = 32 / CH;                      // rows per warp instruction
    const int wr = (warp - kWP) * 32;                 // the warp's first tile row
    DynCursor cur;
    const bool lead = warp == kWP;                    // marks the queue positions demanded
    bool have = dyn_first(s_q, EPT, &s_abort, cur, true, lead);
    int pk = have ? row_entry(a.src, cur, EPT, G, wr + lane) : -1;
    int T = 0;
    while (have && !aborted()) {
      DynCursor nxt = cur;
      const bool have_n = dyn_next(s_q, EPT, &s_abort, nxt, true, lead);
      const int pk_n = have_n ? row_entry(a.src, nxt, EPT, G, wr + lane) : -1;
      const int st = T % kNQ;
      if (!wait(&q_empty[st], ((T / kNQ) & 1) ^ 1)) { give_up(); break; }
      const uint32_t dst = aQ + st * L::Q_BYTES;
      const int c = lane % CH;
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int rl = k * RPI + lane / CH;           // row within the warp's 32
        const int qi = __shfl_sync(0xffffffffu, pk, rl) >> 6;
        const int r = wr + rl;
        const __nv_bfloat16* src =
            a.Q + ((static_cast<int64_t>(cur.v.b) * s.N + (qi < 0 ? 0 : qi)) * s.Hq + cur.v.kv * G + r % G) * D;
        tc::cp_async16(dst + (c >> 3) * (kRows * 128) + tc::sw128(r, (c & 7) * 8), src + c * 8, qi >= 0);
      }
      tc::cp_async_commit();
      if (T > 0) {             // the previous tile's copies have had a tile's time to land
        tc::cp_async_wait<1>();
        tc::fence_async_smem();
        tc::bar_arrive(&q_full[(T - 1) % kNQ]);
      }
      cur = nxt;
      have = have_n;
      pk = pk_n;
      ++T;
    }
    tc::cp_async_wait<0>();
    if (T > 0) {
      tc::fence_async_smem();
      tc::bar_arrive(&q_full[(T - 1) % kNQ]);
    }
  } else if (warp == kWP + 4) {
    // ---------------------------------------------------------------- control
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kRows, NK);
      int k_issued = 0;            // key tiles issued: items 0 .. k_issued - 1
      int k_landed = 0;            // key tiles whose arrival was waited for
      bool mma_issued = false;
      auto load_k = [&](int I, const ItemView& v) {
        const int ks = I % kNK;
        if (!wait(&k_empty[ks], ((I / kNK) & 1) ^ 1)) { give_up(); return; }
        tc::bar_expect_tx(&k_full[ks], L::K_BYTES);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
#pragma unroll
          for (int hp = 0; hp <= PR; ++hp)    // a pair's second leaf may lie past N: zero fill
            tc::tma_load4(aK + ks * L::K_BYTES + kb * (NK * 128) + hp * (64 * 128), &kmap, kb * 64, v.kv / s.kvr,
                          v.kbase + 64 * hp, v.b, &k_full[ks]);
        k_issued = I + 1;
      };
      int T = 0, I = 0;
      ItemView v = queue_take(s_q, 0, &s_abort);
      if (v.n_ent >= 0) load_k(0, v);
      if (a.stall && !wait(&never, 0)) give_up();   // runs out after the wait limit
      for (; v.n_ent >= 0 && !aborted(); ++I) {
        const ItemView v_n = queue_take(s_q, I + 1, &s_abort);
        if (v_n.n_ent >= 0) load_k(I + 1, v_n);
        const int ks = I % kNK;
        if (!wait(&k_full[ks], (I / kNK) & 1)) { give_up(); break; }
        k_landed = I + 1;
        const int n_tiles = (v.n_ent + EPT - 1) / EPT;
        for (int j = 0; j < n_tiles; ++j, ++T) {
          const int st = T % kNQ, ss = T % kNS;
          if (!wait(&q_full[st], (T / kNQ) & 1) || !wait(&s_empty[ss], ((T / kNS) & 1) ^ 1)) {
            give_up();
            break;
          }
          tc::after_sync();
          mma_issued = true;
#pragma unroll
          for (int ks2 = 0; ks2 < D / 16; ++ks2)
            tc::mma(tmem_base + NK * ss,
                    tc::desc(aQ + st * L::Q_BYTES + (ks2 >> 2) * (kRows * 128) + (ks2 & 3) * 32),
                    tc::desc(aK + ks * L::K_BYTES + (ks2 >> 2) * (NK * 128) + (ks2 & 3) * 32), idS, ks2 > 0);
          tc::commit(&s_full[ss]);
          tc::commit(&q_empty[st]);
        }
        tc::commit(&k_empty[ks]);
        v = v_n;
      }
      // Drain before the CTA frees its tensor memory and leaves: key tiles still in flight land
      // (each stage holds at most one: a stage is reloaded only after its item's MMAs), and every
      // MMA issued completes (one commit tracks them all). Both end in bounded time once issued.
      for (int J = k_landed; J < k_issued; ++J) tc::bar_wait(&k_full[J % kNK], (J / kNK) & 1, kDrainNs);
      if (mma_issued) {
        tc::commit(&drain);
        tc::bar_wait(&drain, 0, kDrainNs);
      }
    }
  } else if (warp < kWP) {
    // ---------------------------------------------------------------- softmax
    // warpgroup sg takes the tiles T with T % kSG == sg; its entries for the next such tile
    // load while the current one is reduced
    const int sg = warp >> 2;
    const int r = tid & (kRows - 1);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c1 = s.scale * kLog2e;
    const int h = r % G;
    DynCursor cur;
    bool have = dyn_first(s_q, EPT, &s_abort, cur, true);
    int T = 0;
    for (; have && T < sg; ++T) have = dyn_next(s_q, EPT, &s_abort, cur, true);
    int pk = have ? row_entry(a.src, cur, EPT, G, r) : -1;
    while (have && !aborted()) {
      DynCursor nxt = cur;
      bool have_n = true;
#pragma unroll
      for (int k = 0; k < kSG; ++k)
        if (have_n) have_n = dyn_next(s_q, EPT, &s_abort, nxt, true);
      const int pk_n = have_n ? row_entry(a.src, nxt, EPT, G, r) : -1;   // in flight during this tile
      const int ss = T % kNS;
      const bool ok = wait(&s_full[ss], (T / kNS) & 1);
      if (!__all_sync(0xffffffffu, ok)) { give_up(); break; }   // warp-uniform exit
      tc::after_sync();
      const int qi = pk >> 6;                                  // -1 on padding rows
      // one LSE per leaf of the item: leaf hp's keys are TMEM columns 64 hp .. 64 hp + 63; the
      // pair's second leaf is a candidate of the row iff its first key is visible, and then its
      // slot follows the first leaf's
#pragma unroll 1
      for (int hp = 0; hp <= PR; ++hp) {
        float sv[64];
        tc::tmem_ld64(tmem_base + NK * ss + 64 * hp + lane_off, sv);
        if (hp == PR) {
          tc::before_sync();
          tc::bar_arrive(&s_empty[ss]);
        }
        const int lim = qi - cur.v.kbase - 64 * hp;            // key c is visible iff c <= lim
        if (lim < 63) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sv[c] = c <= lim ? sv[c] : -INFINITY;
        }
        // row max: eight chains of three-input maxima; exponent arguments and the sum on packed
        // pairs (fewer instructions per row: the softmax warps are issue- and latency-bound)
        float mq[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mq[k] = fmaxf(sv[k], sv[k + 8]);
#pragma unroll
          for (int u = 16; u < 64; u += 16) mq[k] = tc::max3(mq[k], sv[k + u], sv[k + u + 8]);
        }
        const float mx = fmaxf(tc::max3(mq[0], mq[1], mq[2]), tc::max3(mq[3], tc::max3(mq[4], mq[5], mq[6]), mq[7]));
        float lse = -INFINITY;
        if (mx != -INFINITY) {
          const float m2 = mx * c1;
          const uint64_t cc = tc::pack2(c1, c1), mm = tc::pack2(-m2, -m2);
          uint64_t lq[4] = {0, 0, 0, 0};            // packed zero pairs
#pragma unroll
          for (int p = 0; p < 32; ++p) {
            float y0, y1;
            tc::unpack2(tc::fma2(tc::pack2(sv[2 * p], sv[2 * p + 1]), cc, mm), y0, y1);
            lq[p & 3] = tc::add2(lq[p & 3], tc::pack2(tc::ex2(y0), tc::ex2(y1)));
          }
          const uint64_t t = tc::add2(tc::add2(lq[0], lq[1]), tc::add2(lq[2], lq[3]));
          float t0, t1;
          tc::unpack2(t, t0, t1);
          lse = (m2 + tc::lg2(t0 + t1)) * kLn2;
        }
        const bool cand = pk >= 0 && lim >= 0;                 // this leaf is one of the row's candidates
        if (a.block_lse) {
          if (cand)
            a.block_lse[((static_cast<int64_t>(cur.v.b) * s.Hq + cur.v.kv * G + h) * s.N + qi) * a.W + (pk & 63)] = lse;
          continue;
        }
        // G adjacent lanes hold the heads of one query (a padding entry is whole)
        float sum = lse;
#pragma unroll
        for (int o = 1; o < G; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (cand) {
          const int64_t at = (cur.v.head * s.N + qi) * a.W + (pk & 63) + hp;
          if (h == 0) a.pair_score[at] = sum;
          if (a.pair_head) a.pair_head[at * G + h] = lse;
        }
      }
      cur = nxt;
      have = have_n;
      pk = pk_n;
      T += kSG;
    }
  } else if (warp == kWP + 5) {
    // ---------------------------------------------------------------- scheduler
    if (lane == 0) queue_fill(s_q, a.src, a.next_item, n_items, &s_abort);
  }
  tc::before_sync();
  __syncthreads();
  if (tid == 0 && s_abort) atomicOr(a.status, PISA_STATUS_TIMEOUT);
  if (warp == 0) {
    tc::after_sync();
    tc::tmem_free(tmem_base, kNS * NK);
  }
}

template <int D, int G, int PR>
int leaf_tc_launch(const LeafArgs& a, const CUtensorMap& km, int grid, cudaStream_t st) {
  const int smem = LeafSmem<D, PR>::bytes;
  cudaError_t e = cudaFuncSetAttribute(leaf_tc_kernel<D, G, PR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope ps(st, a.block_lse ? "attn_lse_tc" : "leaf_score");
  leaf_tc_kernel<D, G, PR><<<static_cast<unsigned>(grid), threads_for(G), smem, st>>>(a, km);
  return cudaGetLastError();
}

}  // namespace

// Streaming multiprocessors of the current device (persistent grids: one CTA per SM).
int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  }
  return n;
}

namespace {

int leaf_tc_run(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const int32_t* list,
                const int4* items, const int32_t* n_items, int W, float* pair_score, float* pair_head,
                float* block_lse, int32_t* status, cudaStream_t st) {
  CUtensorMap km;
  {
    const uint64_t d = static_cast<uint64_t>(s.d);
    const uint64_t dims[4] = {d, static_cast<uint64_t>(s.Hkv_r), static_cast<uint64_t>(s.N),
                              static_cast<uint64_t>(s.B)};
    const uint64_t strides[3] = {d * 2, d * 2 * s.Hkv_r, d * 2 * s.Hkv_r * s.N};
    const uint32_t box[4] = {64, 1, 64, 1};
    if (int e = encode_tmap(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, K, dims, strides, box)) return e;
  }
  LeafArgs a{};
  a.s = s;
  a.src.gp = gp;
  a.src.items = items;
  a.src.list = list;
  a.src.Hkv = s.Hkv;
  a.Q = static_cast<const __nv_bfloat16*>(Q);
  a.n_items = n_items;
  a.W = W;
  a.pair_score = pair_score;
  a.pair_head = pair_head;
  a.block_lse = block_lse;
  a.status = status;
  a.next_item = status + 16;
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  const int64_t mi = gp.max_items;
  const int grid = static_cast<int>(mi < sm_count() ? mi : sm_count());
#define PISA_LEAF_CASE(DD, GG)                                                                     \
  if (s.d == DD && s.G == GG)                                                                    \
    return gp.shift ? leaf_tc_launch<DD, GG, 1>(a, km, grid, st) : leaf_tc_launch<DD, GG, 0>(a, km, grid, st);
  PISA_LEAF_CASE(128, 1) PISA_LEAF_CASE(128, 2) PISA_LEAF_CASE(128, 4) PISA_LEAF_CASE(128, 8)
  PISA_LEAF_CASE(64, 1) PISA_LEAF_CASE(64, 2) PISA_LEAF_CASE(64, 4) PISA_LEAF_CASE(64, 8)
#undef PISA_LEAF_CASE
  return static_cast<int>(cudaErrorNotSupported);
}

}  // namespace

// Exact leaf scores of the grouped (candidate leaf, query) pairs: pair_score[unit, slot] =
// sum over the G heads of the leaf's LSE; per-head terms into pair_head when it is given.
int launch_leaf_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const int32_t* list,
                   const int4* items, const int32_t* n_items, int W, float* pair_score, float* pair_head,
                   int32_t* status, cudaStream_t st) {
  return leaf_tc_run(s, gp, Q, K, list, items, n_items, W, pair_score, pair_head, nullptr, status, st);
}

// Per-(row, block) LSEs of the grouped (selected leaf, query) pairs of an attention call:
// block_lse[b, h, i, slot] = log sum_{j in the leaf, j <= i} exp(s q_{i,h} . k_j).
int launch_block_lse_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const int32_t* list,
                        const int4* items, const int32_t* n_items, float* block_lse, int32_t* status,
                        cudaStream_t st) {
  return leaf_tc_run(s, gp, Q, K, list, items, n_items, s.K, nullptr, nullptr, block_lse, status, st);
}

}  // namespace pisa
