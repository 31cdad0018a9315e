// Causal block-sparse attention forward on the fifth-generation tensor cores: a persistent,
// warp-specialised kernel.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value
// of the work": queries that use the same leaf key block are grouped into tiles so the
// block's keys are read once per tile, and attention runs only over the selected blocks.
//
// Normaliser. Row (query i, head h) has lse = log sum_k exp(lse_k) over the LSEs of its
// selected blocks (the selection's per-head leaf terms, or the LSE pass), known before any
// key is visited; so every block's contribution exp(s q.k - lse) v is final and the blocks
// of a row are summed straight into an fp32 accumulator, in any order.
//
// One CTA per SM takes work items (a selected leaf of one KV head and the (query, head) rows
// that chose it) from a global counter through its item queue (tiles.cuh) and walks them in
// tiles of 128 rows. Roles, connected by mbarrier rings:
//   * producers (warps 12-15): per tile, the query rows gathered with cp.async (whole rows per
//     warp instruction) into a 2-stage ring of swizzled Q tiles, confirmed one tile later;
//   * control (warp 16, one thread): each item's keys and values by TMA into 2-stage rings
//     (the values as stored, [keys][d], read by the P V MMA as an MN-major operand, so no
//     warp transposes them: that took a producer warp 7 % of the kernel's time); S = Q K^T
//     (M=128, N=64) into one of 2 TMEM stages and O = P V (M=128, N=d) into one of 2 TMEM
//     stages, issuing the next tile's S before this tile's P V;
//   * softmax (two warpgroups, warps 0-3 and 4-7, alternate tiles): S row -> P = 2^(s log2e S
//     - log2e lse) on the visible keys, bf16, stored into one of 2 TMEM stages (P V then reads
//     its A operand from tensor memory, no shared-memory tile);
//   * epilogue (warps 8-11): O row from TMEM, 32 columns at a time, through two swizzled
//     staging tiles; the lane holding a query's first head adds the query's G heads x 32
//     columns into the accumulator with one TMA tensor reduce-add;
//   * scheduler (warp 17, one thread): fills the item queue.
// Every wait is bounded (the launch's wait limit); a wait that gives up sets the CTA's abort
// flag and every role leaves its loop at its next tile. Before the CTA frees its tensor memory
// the control thread drains what it issued (key and value tiles in flight, MMAs), the producers and the
// epilogue their copies and reductions; the kernel then ORs PISA_STATUS_TIMEOUT into the
// status word, and the output conversion reads it and writes poisoned outputs.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"
#include "tiles.cuh"
#include "tmap.h"

namespace pisa {

namespace {

constexpr int kRows = 128;
constexpr int kNQ = 2, kNP = 2, kNKV = 2;   // Q, P, K/V stages; S, P and O stages are in TMEM
constexpr int kThreads = 576;               // softmax 0-255, epilogue 256-383, producers 384-511, control, scheduler
constexpr int kConsumerWarps = 17;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound of the drain waits (work already issued)

// PR = 1: an item is a pair of sibling leaves (128 keys) and a row selected one or both of
// them; PR = 0: one leaf.
template <int D, int PR>
struct AttnSmem {
  static constexpr int KB = D / 64;
  static constexpr int NK = 64 << PR;               // keys per item
  static constexpr int Q_BYTES = KB * kRows * 128;
  static constexpr int K_BYTES = KB * NK * 128;
  static constexpr int V_BYTES = KB * NK * 128;     // [NK keys x D] bf16 as K, MN-major operand
  static constexpr int STG = kRows * 128;           // 128 rows x 32 fp32
  static constexpr int oQ = 0, oK = oQ + kNQ * Q_BYTES, oV = oK + kNKV * K_BYTES,
                       oS = oV + kNKV * V_BYTES;
  static constexpr int bytes = oS + 2 * STG + 1024;
  // TMEM columns: S stage k at NK k; O stage k at 2 NK + k D; P stage k (bf16 pairs) at
  // tmem_p + 32 k, or (PR = 1, where S and O fill the 512 columns) over the first NK / 2
  // columns of S stage k, written after the softmax has read them
  static constexpr int tmem_o = 2 * NK;
  static constexpr int tmem_p = 2 * NK + 2 * D;
  static __device__ __forceinline__ uint32_t p_col(int k) { return PR ? NK * k : tmem_p + 32 * k; }
};

struct AttnArgs {
  Dims s;
  ItemSource src;
  const __nv_bfloat16* Q;
  const int32_t* n_items;
  const float* lse_rows;   // [B, Hq, N]
  const int32_t* idx;      // the selection [B, Hkv, N, K] (pairs: which leaves of a pair a row chose)
  int32_t* status;
  int32_t* next_item;      // zeroed item counter
  uint64_t wait_ns;        // bound of every pipeline wait
  int stall;               // test aid: wait on a barrier nothing signals before the first MMA
};

template <int D, int G, int PR>
__global__ void __launch_bounds__(kThreads, 1)
attn_ws_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap omap) {
  using L = AttnSmem<D, PR>;
  constexpr int NK = L::NK;
  constexpr int EPT = kRows / G;
  constexpr int CH = D / 8;               // 16-byte chunks per Q / V row
  extern __shared__ unsigned char smraw[];
  __shared__ __align__(8) uint64_t q_full[kNQ], q_empty[kNQ], s_full[2], s_empty[2], p_full[kNP], p_empty[kNP],
      o_full[2], o_empty[2], k_full[kNKV], k_empty[kNKV], v_full[kNKV], v_empty[kNKV], drain, never;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  __shared__ ItemQueue s_q;

  const Dims& s = a.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* sm = smraw + ((1024 - (tc::su32(smraw) & 1023)) & 1023);
  const uint32_t aQ = tc::su32(sm + L::oQ), aK = tc::su32(sm + L::oK),
                 aV = tc::su32(sm + L::oV), aS = tc::su32(sm + L::oS);
  const int n_items = *a.n_items;

  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      tc::bar_init(&q_full[k], kRows);
      tc::bar_init(&q_empty[k], 1);
      tc::bar_init(&s_full[k], 1);
      tc::bar_init(&s_empty[k], PR ? 1 : kRows);   // pairs: freed by the P V that read P from it
      tc::bar_init(&p_full[k], kRows);
      tc::bar_init(&p_empty[k], 1);
      tc::bar_init(&o_full[k], 1);
      tc::bar_init(&o_empty[k], kRows);
      tc::bar_init(&k_full[k], 1);
      tc::bar_init(&k_empty[k], 1);
      tc::bar_init(&v_full[k], 1);
      tc::bar_init(&v_empty[k], 1);
    }
    tc::bar_init(&drain, 1);
    tc::bar_init(&never, 1);
    queue_init(s_q, kConsumerWarps, a.wait_ns);
    tc::fence_bar_init();
    s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  tc::before_sync();
  __syncthreads();
  tc::after_sync();
  auto give_up = [&]() { atomicOr(&s_abort, 1); };
  auto wait = [&](uint64_t* bar, uint32_t parity) { return tc::bar_wait(bar, parity, a.wait_ns); };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };

  if (warp >= 12 && warp < 16) {
    // ---------------------------------------------------------------- producers
    constexpr int RPI = 32 / CH;                      // Q rows per warp instruction
    const int wr = (warp - 12) * 32;
    DynCursor cur;
    const bool lead = warp == 12;                     // marks the queue positions demanded
    bool have = dyn_first(s_q, EPT, &s_abort, cur, true, lead);
    int pk = have ? row_entry(a.src, cur, EPT, G, wr + lane) : -1;
    int T = 0;
    bool pending = false;                             // tile T-1 issued, not yet confirmed
    auto confirm_last = [&](bool newer_outstanding) {
      if (newer_outstanding) tc::cp_async_wait<1>(); else tc::cp_async_wait<0>();
      tc::fence_async_smem();
      tc::bar_arrive(&q_full[(T - 1) % kNQ]);
    };
    while (have && !aborted()) {
      DynCursor nxt = cur;
      const bool have_n = dyn_next(s_q, EPT, &s_abort, nxt, true, lead);
      const int pk_n = have_n ? row_entry(a.src, nxt, EPT, G, wr + lane) : -1;
      const int st = T % kNQ;
      if (!wait(&q_empty[st], ((T / kNQ) & 1) ^ 1)) { give_up(); break; }
      const uint32_t dst = aQ + st * L::Q_BYTES;
      const int c = lane % CH;
#pragma unroll 4
      for (int k = 0; k < CH; ++k) {
        const int rl = k * RPI + lane / CH;
        const int qi = __shfl_sync(0xffffffffu, pk, rl) >> 6;
        const int r = wr + rl;
        const __nv_bfloat16* src =
            a.Q + ((static_cast<int64_t>(cur.v.b) * s.N + (qi < 0 ? 0 : qi)) * s.Hq + cur.v.kv * G + r % G) * D;
        tc::cp_async16(dst + (c >> 3) * (kRows * 128) + tc::sw128(r, (c & 7) * 8), src + c * 8, qi >= 0);
      }
      tc::cp_async_commit();
      if (pending) confirm_last(true);                // tile T-1, a tile's time after its copies
      pending = true;
      cur = nxt;
      have = have_n;
      pk = pk_n;
      ++T;
    }
    if (pending) confirm_last(false);
    tc::cp_async_wait<0>();
  } else if (warp == 16) {
    // ---------------------------------------------------------------- control
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kRows, NK);
      constexpr uint32_t idO = tc::idesc_bf16_major(kRows, D, false, true);   // B = V, MN-major
      int k_issued = 0;            // key tiles issued: items 0 .. k_issued - 1
      int k_landed = 0;            // key tiles whose arrival was waited for
      int v_issued = 0, v_landed = 0;   // the same for value tiles
      bool mma_issued = false;
      // K of the CTA's item number I into stage I % 2
      auto load_k = [&](int I, const ItemView& v) {
        const int ks = I % kNKV;
        if (!wait(&k_empty[ks], ((I / kNKV) & 1) ^ 1)) { give_up(); return; }
        tc::bar_expect_tx(&k_full[ks], L::K_BYTES);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
#pragma unroll
          for (int hp = 0; hp <= PR; ++hp)    // a pair's second leaf may lie past N: zero fill
            tc::tma_load4(aK + ks * L::K_BYTES + kb * (NK * 128) + hp * (64 * 128), &kmap, kb * 64, v.kv / s.kvr,
                          v.kbase + 64 * hp, v.b, &k_full[ks]);
        k_issued = I + 1;
      };
      // V of item I into stage I % 2 (its stage was freed by item I - 2's last P V)
      auto load_v = [&](int I, const ItemView& v) {
        const int vs = I % kNKV;
        if (!wait(&v_empty[vs], ((I / kNKV) & 1) ^ 1)) { give_up(); return; }
        tc::bar_expect_tx(&v_full[vs], L::V_BYTES);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
#pragma unroll
          for (int hp = 0; hp <= PR; ++hp)
            tc::tma_load4(aV + vs * L::V_BYTES + kb * (NK * 128) + hp * (64 * 128), &vmap, kb * 64, v.kv / s.kvr,
                          v.kbase + 64 * hp, v.b, &v_full[vs]);
        v_issued = I + 1;
      };
      // S of tile T (cursor c, item number I)
      auto issue_s = [&](const DynCursor& c, int T, int I) -> bool {
        const int ks = I % kNKV, st = T % kNQ, ss = T & 1;
        if (c.j == 0) {
          const ItemView v_n = queue_peek(s_q, c.k + 1, &s_abort);
          if (v_n.n_ent >= 0) load_k(I + 1, v_n);
          if (!wait(&k_full[ks], (I / kNKV) & 1)) return false;
          k_landed = I + 1;
        }
        if (!wait(&q_full[st], (T / kNQ) & 1) || !wait(&s_empty[ss], ((T >> 1) & 1) ^ 1))
          return false;
        tc::after_sync();
        mma_issued = true;
#pragma unroll
        for (int k2 = 0; k2 < D / 16; ++k2)
          tc::mma(tmem_base + NK * ss, tc::desc(aQ + st * L::Q_BYTES + (k2 >> 2) * (kRows * 128) + (k2 & 3) * 32),
                  tc::desc(aK + ks * L::K_BYTES + (k2 >> 2) * (NK * 128) + (k2 & 3) * 32), idS, k2 > 0);
        tc::commit(&s_full[ss]);
        tc::commit(&q_empty[st]);
        if (c.j + 1 == c.n_tiles) tc::commit(&k_empty[ks]);   // the item's last S
        return true;
      };
      // P V of tile T
      auto issue_pv = [&](const DynCursor& c, int T, int I) -> bool {
        const int vs = I % kNKV, ps = T % kNP, os = T & 1;
        if (c.j == 0) {
          if (!wait(&v_full[vs], (I / kNKV) & 1)) return false;
          v_landed = I + 1;
        }
        if (!wait(&p_full[ps], (T / kNP) & 1) || !wait(&o_empty[os], ((T >> 1) & 1) ^ 1))
          return false;
        tc::after_sync();
        // K step kk: keys 16 kk .. 16 kk + 15, 2048 bytes of each 64-column chunk of V
#pragma unroll
        for (int kk = 0; kk < NK / 16; ++kk)
          tc::mma_ts(tmem_base + L::tmem_o + os * D, tmem_base + L::p_col(ps) + 8 * kk,
                     tc::desc_mn(aV + vs * L::V_BYTES + kk * 2048, NK * 128), idO, kk > 0);
        tc::commit(&o_full[os]);
        tc::commit(PR ? &s_empty[ps] : &p_empty[ps]);   // pairs: P lives in its S stage
        if (c.j + 1 == c.n_tiles) tc::commit(&v_empty[vs]);   // the item's last P V
        if (c.j == 0) {                                          // the next item's values: their
          const ItemView v_n = queue_peek(s_q, c.k + 1, &s_abort);   // stage is item I - 1's
          if (v_n.n_ent >= 0) load_v(I + 1, v_n);
        }
        return true;
      };
      // cs (S, one tile ahead) only looks; cp (P V) frees the positions it leaves
      DynCursor cs, cp;
      bool have_s = dyn_first(s_q, EPT, &s_abort, cs, false, false, 1u);
      bool have_p = dyn_first(s_q, EPT, &s_abort, cp, true, false, 1u);
      int Ts = 0, Is = 0, Tp = 0, Ip = 0;
      if (have_s) {
        load_k(0, cs.v);
        load_v(0, cs.v);
        if (a.stall && !wait(&never, 0)) give_up();   // runs out after the wait limit
        if (!aborted() && !issue_s(cs, 0, 0)) give_up();
        Ts = 1;
        have_s = dyn_next(s_q, EPT, &s_abort, cs, false, false, 1u);
        if (have_s && cs.j == 0) Is = 1;
      }
      while (have_p && !aborted()) {
        if (have_s) {                                        // S of the next tile first
          if (!issue_s(cs, Ts, Is)) { give_up(); break; }
          ++Ts;
          have_s = dyn_next(s_q, EPT, &s_abort, cs, false, false, 1u);
          if (have_s && cs.j == 0) ++Is;
        }
        if (!issue_pv(cp, Tp, Ip)) { give_up(); break; }
        ++Tp;
        have_p = dyn_next(s_q, EPT, &s_abort, cp, true, false, 1u);
        if (have_p && cp.j == 0) ++Ip;
      }
      // Drain before the CTA frees its tensor memory and leaves: key tiles still in flight land
      // (each stage holds at most one: a stage is reloaded only after its item's last S), and
      // every MMA issued completes (one commit tracks them all).
      for (int J = k_landed; J < k_issued; ++J) tc::bar_wait(&k_full[J % kNKV], (J / kNKV) & 1, kDrainNs);
      for (int J = v_landed; J < v_issued; ++J) tc::bar_wait(&v_full[J % kNKV], (J / kNKV) & 1, kDrainNs);
      if (mma_issued) {
        tc::commit(&drain);
        tc::bar_wait(&drain, 0, kDrainNs);
      }
    }
  }
  else if (warp < 8) {
    // ---------------------------------------------------------------- softmax
    const int sg = warp >> 2;                         // tiles T with T % 2 == sg
    const int r = tid & (kRows - 1);
    const int h = r % G;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c1 = s.scale * kLog2e;
    auto row_lse2 = [&](const DynCursor& c, int pkv) {
      if (pkv < 0) return 0.f;
      return a.lse_rows[(static_cast<int64_t>(c.v.b) * s.Hq + c.v.kv * G + h) * s.N + (pkv >> 6)] * kLog2e;
    };
    // pairs: bit l set when the row chose leaf l of the pair (its entry holds the slot of the
    // first chosen one; the selection is ascending, so a chosen second leaf follows it)
    auto row_sel = [&](const DynCursor& c, int pkv) -> int {
      if (!PR || pkv < 0) return 1;
      const int64_t base = (c.v.head * s.N + (pkv >> 6)) * s.K;
      const int slot = pkv & 63, t0 = a.idx[base + slot];
      if (t0 & 1) return 2;
      return slot + 1 < s.K && a.idx[base + slot + 1] == t0 + 1 ? 3 : 1;
    };
    DynCursor cur;
    bool have = dyn_first(s_q, EPT, &s_abort, cur, true);
    int T = 0;
    if (have && sg == 1) {
      have = dyn_next(s_q, EPT, &s_abort, cur, true);
      T = 1;
    }
    int pk = have ? row_entry(a.src, cur, EPT, G, r) : -1;
    float l2 = have ? row_lse2(cur, pk) : 0.f;
    int sel = have ? row_sel(cur, pk) : 1;
    while (have && !aborted()) {
      DynCursor nxt = cur;
      bool have_n = dyn_next(s_q, EPT, &s_abort, nxt, true);
      if (have_n) have_n = dyn_next(s_q, EPT, &s_abort, nxt, true);
      const int pk_n = have_n ? row_entry(a.src, nxt, EPT, G, r) : -1;
      const bool ok = wait(&s_full[sg], (T >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { give_up(); break; }
      tc::after_sync();
      const float l2_n = have_n ? row_lse2(nxt, pk_n) : 0.f;   // in flight during the math
      const int sel_n = have_n ? row_sel(nxt, pk_n) : 1;
      const int lim = pk < 0 ? -1 : (pk >> 6) - cur.v.kbase;    // key c is visible iff c <= lim
      const int ps = T % kNP;
      // the row's keys in quarters of 32 (fewer live registers); with pairs, P overwrites the
      // front of the S stage, columns the later quarters do not read
#pragma unroll 1     // rolled, like the epilogue's rounds: instruction-cache footprint
      for (int q = 0; q < NK / 32; ++q) {
        float sv[32];
        tc::tmem_ld32(tmem_base + NK * sg + 32 * q + lane_off, sv);
        if (!PR && q == 1) {                                   // the S stage is free for S(T + 2)
          tc::before_sync();
          tc::bar_arrive(&s_empty[sg]);
        }
        const int lh = (sel >> (q >> 1)) & 1 ? lim - 32 * q : -1;   // a leaf the row did not choose: P = 0
        const uint64_t cc = tc::pack2(c1, c1), ll = tc::pack2(-l2, -l2);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {         // exponent arguments on packed pairs
          float y0, y1;
          tc::unpack2(tc::fma2(tc::pack2(sv[c], sv[c + 1]), cc, ll), y0, y1);
          sv[c] = c <= lh ? tc::ex2(y0) : 0.f;
          sv[c + 1] = c + 1 <= lh ? tc::ex2(y1) : 0.f;
        }
        if (!PR && q == 0) {
          const bool ok2 = wait(&p_empty[ps], ((T / kNP) & 1) ^ 1);
          if (!__all_sync(0xffffffffu, ok2)) {
            give_up();
            break;
          }
        }
        uint32_t pkd[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pkd[c] = pack_bf16(sv[2 * c], sv[2 * c + 1]);
        tc::tmem_st16(tmem_base + L::p_col(ps) + 16 * q + lane_off, pkd);
      }
      if (aborted()) break;
      tc::tmem_wait_st();                                      // P in TMEM before the arrival
      tc::before_sync();
      tc::bar_arrive(&p_full[ps]);
      cur = nxt;
      have = have_n;
      pk = pk_n;
      l2 = l2_n;
      sel = sel_n;
      T += 2;
    }
  } else if (warp < 12) {
    // ---------------------------------------------------------------- epilogue
    // row r's O, 32 columns per round, into staging tile (round & 1) at +128 r with 16-byte
    // chunks swizzled by r & 7; every lane commits one bulk group per round (empty unless it
    // issued), so "all but the newest group read out" means the other tile is free again
    const int r = tid - 256;
    const int h = r % G;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    DynCursor cur;
    bool have = dyn_first(s_q, EPT, &s_abort, cur, true);
    int pk = have ? row_entry(a.src, cur, EPT, G, r) : -1;
    int T = 0, rd_all = 0;
    while (have && !aborted()) {
      DynCursor nxt = cur;
      const bool have_n = dyn_next(s_q, EPT, &s_abort, nxt, true);
      const int pk_n = have_n ? row_entry(a.src, nxt, EPT, G, r) : -1;
      const int os = T & 1;
      const bool ok = wait(&o_full[os], (T >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { give_up(); break; }
      tc::after_sync();
      const bool issuer = h == 0 && pk >= 0;
      const int unit = (cur.v.b * s.N + (pk < 0 ? 0 : (pk >> 6))) * s.Hkv + cur.v.kv;
#pragma unroll 1     // rolled: a smaller kernel body keeps the roles' code in the instruction cache
      for (int rd = 0; rd < D / 32; ++rd, ++rd_all) {
        float ov[32];
        tc::tmem_ld32(tmem_base + L::tmem_o + os * D + 32 * rd + lane_off, ov);
        if (rd == D / 32 - 1) {                        // the O stage is free for P V of T + 2
          tc::before_sync();
          tc::bar_arrive(&o_empty[os]);
        }
        const int sb = rd_all & 1;
        tc::bulk_wait_read<1>();
        __syncwarp();
        unsigned char* stg = sm + L::oS + sb * L::STG;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(stg + r * 128 + ((c ^ (r & 7)) << 4)) =
              make_float4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
        tc::fence_async_smem();
        __syncwarp();
        if (issuer) tc::tma_reduce_add3(&omap, 32 * rd, 0, unit, aS + sb * L::STG + r * 128);
        tc::bulk_commit();
      }
      cur = nxt;
      have = have_n;
      pk = pk_n;
      ++T;
    }
    tc::bulk_wait<0>();
  } else if (warp == 17) {
    // ---------------------------------------------------------------- scheduler
    if (lane == 0) queue_fill(s_q, a.src, a.next_item, n_items, &s_abort);
  }
  tc::before_sync();
  __syncthreads();
  if (tid == 0 && s_abort) atomicOr(a.status, PISA_STATUS_TIMEOUT);
  if (warp == 0) {
    tc::after_sync();
    tc::tmem_free(tmem_base, 512);
  }
}

template <int D, int G, int PR>
int attn_ws_launch(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& om, int grid,
                   cudaStream_t st) {
  const int smem = AttnSmem<D, PR>::bytes;
  cudaError_t e = cudaFuncSetAttribute(attn_ws_kernel<D, G, PR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope ps(st, "attn_fwd_tc");
  attn_ws_kernel<D, G, PR><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a, km, vm, om);
  return cudaGetLastError();
}

}  // namespace

// Attention output pass over the grouped (selected leaf, query) entries: adds every row's
// normalised block contributions into the fp32 accumulator o_acc [B, N, Hq, d]. With a plan
// of sibling pairs (gp.shift = 1, deduplicated) an item covers both leaves of a pair and a
// row's entry stands for the members it selected (read back from idx).
int launch_attn_out_ws(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       const float* lse_rows, float* o_acc, int32_t* status, cudaStream_t st) {
  CUtensorMap km, vm, om;
  const uint64_t d = static_cast<uint64_t>(s.d);
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
    if (int e = encode_tmap(&om, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, o_acc, dims, strides, box)) return e;
  }
  AttnArgs a{};
  a.s = s;
  a.src.gp = gp;
  a.src.items = items;
  a.src.list = list;
  a.src.Hkv = s.Hkv;
  a.Q = static_cast<const __nv_bfloat16*>(Q);
  a.n_items = n_items;
  a.lse_rows = lse_rows;
  a.idx = idx;
  a.status = status;
  a.next_item = status + 32;
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  const int64_t mi = gp.max_items;
  const int grid = static_cast<int>(mi < sm_count() ? mi : sm_count());
#define PISA_ATTN_CASE(DD, GG)                                                                         \
  if (s.d == DD && s.G == GG)                                                                          \
    return gp.shift ? attn_ws_launch<DD, GG, 1>(a, km, vm, om, grid, st)                               \
                    : attn_ws_launch<DD, GG, 0>(a, km, vm, om, grid, st);
  PISA_ATTN_CASE(128, 1) PISA_ATTN_CASE(128, 2) PISA_ATTN_CASE(128, 4) PISA_ATTN_CASE(128, 8)
  PISA_ATTN_CASE(64, 1) PISA_ATTN_CASE(64, 2) PISA_ATTN_CASE(64, 4) PISA_ATTN_CASE(64, 8)
#undef PISA_ATTN_CASE
  return static_cast<int>(cudaErrorNotSupported);
}

}  // namespace pisa
