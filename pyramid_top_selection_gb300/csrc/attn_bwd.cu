// Backward of the causal block-sparse attention; the discrete selection takes no gradient.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value
// of the work": during training the gradient passes only through the selected attention,
// so the block selection can be dropped into an existing model as a sparse module.
//
// With P = exp(s q.k - lse) (lse from the forward), D_i = dO_i . O_i and
// dS = P (dO . v - D):  dQ = s dS K,  dK = s dS^T Q,  dV = P^T dO.
//
// Block-major: the selected (leaf, query) pairs are grouped by (KV head, query chunk, leaf)
// and cut into work items; one CTA takes one item (a leaf block of one KV head and a run of
// the rows = (query, head of the group) that selected it) and adds its share of that
// block's dK/dV into fp32 accumulators with vector reductions. Each of the 4
// warps owns 16 of the 64 keys and keeps their dK/dV in registers across all row chunks;
// rows come in chunks of 32, staged in shared memory row-major by cp.async into two buffers
// (the next chunk's rows land while this one is computed); the operands that contract over
// rows or keys (dO and Q for dV/dK, K for dQ) are read transposed by ldmatrix.trans.
// dQ of a (row, block) pair is added into an fp32 accumulator with vector reductions (the
// rows of a query chunk stay in L2); a last kernel converts dQ, dK and dV to bf16.
#include "device.cuh"
#include "group.h"
#include "profile.h"
#include "tc.cuh"

namespace pisa {

size_t align256(size_t x);
int launch_attn_bwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const void* dO, const float* lse, const float* delta, const int32_t* list,
                       const int4* items, const int32_t* n_items, float* dq_acc, float* dk_acc, float* dv_acc,
                       int32_t* status, cudaStream_t st);

namespace {

constexpr int kWarps = 4;
constexpr int kRows = 32;       // rows per chunk

template <int D>
struct BwdSmem {
  static constexpr int KROW = D + 16;     // row-major tiles (8-byte fragment loads, 16-byte ldmatrix rows)
  static constexpr int SROW = 64 + 8;     // dS [row][key]
  static constexpr int oK = 0;
  static constexpr int oV = oK + 64 * KROW;
  static constexpr int oQ = oV + 64 * KROW;            // two buffers each of Q and dO rows
  static constexpr int odO = oQ + 2 * kRows * KROW;
  static constexpr int odS = odO + 2 * kRows * KROW;
  static constexpr int n_bf16 = odS + kRows * SROW;
  static constexpr int bytes = n_bf16 * 2 + 2 * kRows * (4 + 4 + 4 + 4);
};

// Four 8x8 bf16 matrices, transposed: the B fragments (k = 16 rows from `row0`, n = dims
// n8*8.. and n8*8+8..) of two m16n8k16 MMAs from a row-major [k][n] tile with `stride`
// elements per row. Lane l addresses row row0 + (l & 15), column block n8 + (l >> 4).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&b)[4], const __nv_bfloat16* tile, int stride, int row0,
                                              int n8) {
  const int lane = threadIdx.x & 31;
  const uint32_t a = static_cast<uint32_t>(
      __cvta_generic_to_shared(tile + (row0 + (lane & 15)) * stride + (n8 + (lane >> 4)) * 8));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
               : "r"(a));
}

// D_row = dO_row . O_row (fp32), one warp per row.
template <int D>
__global__ void __launch_bounds__(256)
delta_kernel(int64_t rows, const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
             float* __restrict__ delta) {
  const int64_t row = blockIdx.x * 8LL + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int PER = D / 32;
  float acc = 0.f;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int64_t o = row * D + lane * PER + u;
    acc += __bfloat162float(O[o]) * __bfloat162float(dO[o]);
  }
  acc = warp_sum(acc);
  if (lane == 0) delta[row] = acc;
}

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
attn_bwd_kernel(Dims s, GroupPlan gp, const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                const __nv_bfloat16* __restrict__ V, const __nv_bfloat16* __restrict__ dO,
                const float* __restrict__ lse, const float* __restrict__ delta,
                const int32_t* __restrict__ list, const int4* __restrict__ items,
                const int32_t* __restrict__ n_items, float* __restrict__ dq_acc,
                float* __restrict__ dk_acc, float* __restrict__ dv_acc) {
  using L = BwdSmem<D>;
  constexpr int KS = D / 16, ND = D / 8, QPC = kRows / G;
  extern __shared__ __align__(16) unsigned char smraw[];
  __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(smraw);
  __nv_bfloat16 *sK = sb + L::oK, *sV = sb + L::oV, *sdS = sb + L::odS;
  // per row buffer: lse, D, query, head (kRows words each)
  int* s_meta = reinterpret_cast<int*>(sb + L::n_bf16);

  if (static_cast<int>(blockIdx.x) >= *n_items) return;
  const int4 item = items[blockIdx.x];
  const int t = gp.leaf_of(item.x);
  const int64_t head = gp.head_of(item.x);
  const int b = static_cast<int>(head / s.Hkv), kv = static_cast<int>(head % s.Hkv);
  const int beg = item.y, end = item.y + item.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
  const int kbase = t * 64;

  // leaf tiles: K, V row-major
  for (int it = threadIdx.x; it < 64 * (D / 8); it += blockDim.x) {
    const int r = it / (D / 8), c = it % (D / 8);
    const int64_t j = static_cast<int64_t>(kbase) + r;
    uint4 kk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (j < s.N && beg < end) {
      const int64_t o = ((static_cast<int64_t>(b) * s.N + j) * s.Hkv_r + kv / s.kvr) * D + c * 8;
      kk = ldg_u4(K + o);
      vv = ldg_u4(V + o);
    }
    *reinterpret_cast<uint4*>(&sK[r * L::KROW + c * 8]) = kk;
    *reinterpret_cast<uint4*>(&sV[r * L::KROW + c * 8]) = vv;
  }

  float dv[ND][4], dk[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) dv[nd][e] = dk[nd][e] = 0.f;

  const int n_ent = end - beg;
  const int key0 = 16 * warp;        // this warp's keys: key0 + g, key0 + g + 8
  // chunk staging: thread tid copies chunk (tid % CPR) of rows tid / CPR + RSTEP * u
  constexpr int CPR = D / 8, NIT = kRows * CPR / (kWarps * 32), RSTEP = kWarps * 32 / CPR;
  const int sc_c = threadIdx.x % CPR, sc_r = threadIdx.x / CPR;
  auto entries = [&](int e0, int (&pk)[NIT]) {     // list entries of the thread's rows (-1: none)
#pragma unroll
    for (int u = 0; u < NIT; ++u) {
      const int e = e0 + (sc_r + RSTEP * u) / G;
      pk[u] = e < n_ent ? list[beg + e] : -1;
    }
  };
  auto issue = [&](int bf, const int (&pk)[NIT]) {
#pragma unroll
    for (int u = 0; u < NIT; ++u) {
      const int r = sc_r + RSTEP * u, h = r % G;
      const int64_t row = (static_cast<int64_t>(b) * s.N + (pk[u] < 0 ? 0 : (pk[u] >> 6))) * s.Hq + kv * G + h;
      const uint32_t o = static_cast<uint32_t>(((bf * kRows + r) * L::KROW + sc_c * 8) * 2);
      tc::cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(sb + L::oQ)) + o, Q + row * D + sc_c * 8, pk[u] >= 0);
      tc::cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(sb + L::odO)) + o, dO + row * D + sc_c * 8,
                     pk[u] >= 0);
    }
  };
  // row metadata of a chunk (threads < kRows), loaded into registers and stored later
  struct Meta { float lse, delta; int i, h; };  // delta: D_i = dO_i . O_i
  auto meta_load = [&](int e0) {
    Meta m{__int_as_float(0x7f800000), 0.f, -1, 0};      // +inf lse: P = 0 on padding rows
    const int r = threadIdx.x, e = e0 + r / G, h = r % G;
    if (e < n_ent) {
      const int pk = list[beg + e];
      const int i = pk >> 6;
      const int64_t row = (static_cast<int64_t>(b) * s.N + i) * s.Hq + kv * G + h;
      m.lse = lse[(static_cast<int64_t>(b) * s.Hq + kv * G + h) * s.N + i];
      m.delta = delta[row];
      m.i = i;
      m.h = h;
    }
    return m;
  };
  auto meta_store = [&](int bf, const Meta& m) {
    int* mb = s_meta + bf * 4 * kRows;
    const int r = threadIdx.x;
    mb[r] = __float_as_int(m.lse);
    mb[kRows + r] = __float_as_int(m.delta);
    mb[2 * kRows + r] = m.i;
    mb[3 * kRows + r] = m.h;
  };
  int pk_next[NIT];
  Meta m_next{};
  if (n_ent > 0) {
    entries(0, pk_next);
    issue(0, pk_next);
    if (threadIdx.x < kRows) meta_store(0, meta_load(0));
    entries(QPC, pk_next);
  }
  tc::cp_async_commit();
  for (int e0 = 0, bf = 0; e0 < n_ent; e0 += QPC, bf ^= 1) {
    // the next chunk's rows into the other buffer (freed by the previous iteration's last
    // barrier); its list entries for the chunk after it load meanwhile
    const bool more = e0 + QPC < n_ent;
    if (more) {
      issue(bf ^ 1, pk_next);
      if (threadIdx.x < kRows) m_next = meta_load(e0 + QPC);
      entries(e0 + 2 * QPC, pk_next);
    }
    tc::cp_async_commit();
    tc::cp_async_wait<1>();
    __syncthreads();                 // this chunk's rows and metadata are in place
    const __nv_bfloat16* sQ = sb + L::oQ + bf * kRows * L::KROW;
    const __nv_bfloat16* sdO = sb + L::odO + bf * kRows * L::KROW;
    const int* mb = s_meta + bf * 4 * kRows;
    const float* s_lse = reinterpret_cast<const float*>(mb);
    const float* s_D = reinterpret_cast<const float*>(mb + kRows);
    const int* s_i = mb + 2 * kRows;
    const int* s_h = mb + 3 * kRows;

    // S^T and dP^T for keys key0+{g, g+8} x the 32 rows (4 n-tiles of 8 rows)
    float st[4][4], dp[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[nt][e] = dp[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint2 k0 = *reinterpret_cast<const uint2*>(&sK[(key0 + g) * L::KROW + 16 * ks + 4 * p]);
      const uint2 k1 = *reinterpret_cast<const uint2*>(&sK[(key0 + g + 8) * L::KROW + 16 * ks + 4 * p]);
      const uint2 v0 = *reinterpret_cast<const uint2*>(&sV[(key0 + g) * L::KROW + 16 * ks + 4 * p]);
      const uint2 v1 = *reinterpret_cast<const uint2*>(&sV[(key0 + g + 8) * L::KROW + 16 * ks + 4 * p]);
      const uint32_t ak[4] = {k0.x, k1.x, k0.y, k1.y};
      const uint32_t av[4] = {v0.x, v1.x, v0.y, v1.y};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint2 q = *reinterpret_cast<const uint2*>(&sQ[(nt * 8 + g) * L::KROW + 16 * ks + 4 * p]);
        const uint2 o = *reinterpret_cast<const uint2*>(&sdO[(nt * 8 + g) * L::KROW + 16 * ks + 4 * p]);
        mma_bf16(st[nt], ak, q.x, q.y);
        mma_bf16(dp[nt], av, o.x, o.y);
      }
    }
    // P^T, dS^T (in place: st <- P, dp <- dS)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = nt * 8 + 2 * p + (e & 1);
        const int key = kbase + key0 + g + ((e >> 1) << 3);
        const float pr = (s_i[r] >= 0 && key <= s_i[r]) ? expf(s.scale * st[nt][e] - s_lse[r]) : 0.f;
        st[nt][e] = pr;
        dp[nt][e] = pr * (dp[nt][e] - s_D[r]);
      }
    // dV += P^T dO, dK += dS^T Q   (contraction over the 32 rows: 2 k-steps)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t ap[4] = {pack_bf16(st[2 * kk][0], st[2 * kk][1]), pack_bf16(st[2 * kk][2], st[2 * kk][3]),
                              pack_bf16(st[2 * kk + 1][0], st[2 * kk + 1][1]),
                              pack_bf16(st[2 * kk + 1][2], st[2 * kk + 1][3])};
      const uint32_t as[4] = {pack_bf16(dp[2 * kk][0], dp[2 * kk][1]), pack_bf16(dp[2 * kk][2], dp[2 * kk][3]),
                              pack_bf16(dp[2 * kk + 1][0], dp[2 * kk + 1][1]),
                              pack_bf16(dp[2 * kk + 1][2], dp[2 * kk + 1][3])};
#pragma unroll
      for (int nd = 0; nd < ND; nd += 2) {
        uint32_t bo[4], bq[4];
        ldsm_x4_trans(bo, sdO, L::KROW, 16 * kk, nd);
        ldsm_x4_trans(bq, sQ, L::KROW, 16 * kk, nd);
        mma_bf16(dv[nd], ap, bo[0], bo[1]);
        mma_bf16(dv[nd + 1], ap, bo[2], bo[3]);
        mma_bf16(dk[nd], as, bq[0], bq[1]);
        mma_bf16(dk[nd + 1], as, bq[2], bq[3]);
      }
    }
    // dS -> shared memory as [row][key] for dQ
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = nt * 8 + 2 * p + (e & 1);
        const int key = key0 + g + ((e >> 1) << 3);
        sdS[r * L::SROW + key] = __float2bfloat16_rn(dp[nt][e]);
      }
    __syncthreads();
    // dQ partial = s dS K for 16 rows x D/2 dims per warp
    {
      const int r0 = (warp & 1) * 16, d0 = (warp >> 1) * (D / 2);
      float dq[ND / 2][4];
#pragma unroll
      for (int nd = 0; nd < ND / 2; ++nd)
#pragma unroll
        for (int e = 0; e < 4; ++e) dq[nd][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const __nv_bfloat16* a0 = &sdS[(r0 + g) * L::SROW + 16 * kk + 2 * p];
        const __nv_bfloat16* a1 = &sdS[(r0 + g + 8) * L::SROW + 16 * kk + 2 * p];
        const uint32_t a[4] = {*reinterpret_cast<const uint32_t*>(a0), *reinterpret_cast<const uint32_t*>(a1),
                               *reinterpret_cast<const uint32_t*>(a0 + 8), *reinterpret_cast<const uint32_t*>(a1 + 8)};
#pragma unroll
        for (int nd = 0; nd < ND / 2; nd += 2) {
          uint32_t bk[4];
          ldsm_x4_trans(bk, sK, L::KROW, 16 * kk, d0 / 8 + nd);
          mma_bf16(dq[nd], a, bk[0], bk[1]);
          mma_bf16(dq[nd + 1], a, bk[2], bk[3]);
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = r0 + g + 8 * half;
        if (s_i[r] < 0) continue;
        const int64_t row = (static_cast<int64_t>(b) * s.N + s_i[r]) * s.Hq + kv * G + s_h[r];
        float* dst = dq_acc + row * D + d0;
#pragma unroll
        for (int nd = 0; nd < ND / 2; ++nd)
          atomicAdd(reinterpret_cast<float2*>(dst + nd * 8 + 2 * p),
                    make_float2(s.scale * dq[nd][2 * half], s.scale * dq[nd][2 * half + 1]));
      }
    }
    if (more && threadIdx.x < kRows) meta_store(bf ^ 1, m_next);
    __syncthreads();                 // this chunk's buffers are free for the chunk after next
  }
  tc::cp_async_wait<0>();
  // this item's share of the leaf block's dK and dV (unscaled dK), added into fp32
  // accumulators with vector reductions: items of one leaf run in different CTAs
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int64_t j = static_cast<int64_t>(kbase) + key0 + g + 8 * half;
    if (j >= s.N) continue;
    const int64_t o = ((static_cast<int64_t>(b) * s.N + j) * s.Hkv_r + kv / s.kvr) * D;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      atomicAdd(reinterpret_cast<float2*>(dk_acc + o + nd * 8 + 2 * p), make_float2(dk[nd][2 * half], dk[nd][2 * half + 1]));
      atomicAdd(reinterpret_cast<float2*>(dv_acc + o + nd * 8 + 2 * p), make_float2(dv[nd][2 * half], dv[nd][2 * half + 1]));
    }
  }
}

constexpr uint32_t kNaN2 = 0x7fc07fc0u;   // two bf16 NaNs

// dK = bf16(s * dK_acc), dV = bf16(dV_acc), 8 elements per thread; NaN everywhere when the
// status word reports a bounded wait that gave up (the accumulators are then incomplete).
__global__ void dkdv_convert_kernel(int64_t n8, float scale, const float4* __restrict__ dk_acc,
                                    const float4* __restrict__ dv_acc, uint4* __restrict__ dK,
                                    uint4* __restrict__ dV, const int32_t* __restrict__ status) {
  const bool poison = (*status & PISA_STATUS_TIMEOUT) != 0;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n8;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (poison) {
      dK[q] = dV[q] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
      continue;
    }
    const float4 a = dk_acc[2 * q], c = dk_acc[2 * q + 1], e = dv_acc[2 * q], f = dv_acc[2 * q + 1];
    dK[q] = make_uint4(pack_bf16(scale * a.x, scale * a.y), pack_bf16(scale * a.z, scale * a.w),
                       pack_bf16(scale * c.x, scale * c.y), pack_bf16(scale * c.z, scale * c.w));
    dV[q] = make_uint4(pack_bf16(e.x, e.y), pack_bf16(e.z, e.w), pack_bf16(f.x, f.y), pack_bf16(f.z, f.w));
  }
}

// dQ = bf16(dQ_acc), 8 elements per thread (NaN when the status word reports a timeout).
__global__ void dq_convert_kernel(int64_t n8, const float4* __restrict__ dq_acc, uint4* __restrict__ dQ,
                                  const int32_t* __restrict__ status) {
  const bool poison = (*status & PISA_STATUS_TIMEOUT) != 0;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n8;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (poison) {
      dQ[q] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
      continue;
    }
    const float4 a = dq_acc[2 * q], c = dq_acc[2 * q + 1];
    dQ[q] = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(c.x, c.y), pack_bf16(c.z, c.w));
  }
}

template <int D, int G>
int bwd_launch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
               const void* dO, const float* lse, const float* delta, const int32_t* list,
               const int4* items, const int32_t* n_items, float* dqa, float* dk_acc,
               float* dv_acc, cudaStream_t st) {
  const int smem = BwdSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope ps(st, "attn_bwd");
  attn_bwd_kernel<D, G><<<static_cast<unsigned>(gp.max_items), kWarps * 32, smem, st>>>(
      s, gp, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
      static_cast<const __nv_bfloat16*>(V), static_cast<const __nv_bfloat16*>(dO), lse, delta, list,
      items, n_items, dqa, dk_acc, dv_acc);
  return cudaGetLastError();
}

template <int D>
int bwd_dispatch(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                 const void* dO, const float* lse, const float* delta, const int32_t* list,
                 const int4* items, const int32_t* n_items, float* dqa, float* dk_acc,
                 float* dv_acc, cudaStream_t st) {
  switch (s.G) {
    case 1: return bwd_launch<D, 1>(s, gp, Q, K, V, dO, lse, delta, list, items, n_items, dqa, dk_acc, dv_acc, st);
    case 2: return bwd_launch<D, 2>(s, gp, Q, K, V, dO, lse, delta, list, items, n_items, dqa, dk_acc, dv_acc, st);
    case 4: return bwd_launch<D, 4>(s, gp, Q, K, V, dO, lse, delta, list, items, n_items, dqa, dk_acc, dv_acc, st);
    default: return bwd_launch<D, 8>(s, gp, Q, K, V, dO, lse, delta, list, items, n_items, dqa, dk_acc, dv_acc, st);
  }
}

// Query chunks of about 16 MiB of one head's Q and dO rows (their fp32 dQ rows stay in L2);
// about 4096 (query, head) rows per work item.
#ifndef PISA_BWD_CHUNK_MIB
#define PISA_BWD_CHUNK_MIB 16
#endif
#ifndef PISA_BWD_ITEM_ROWS
#define PISA_BWD_ITEM_ROWS 4096
#endif
GroupPlan bwd_plan(const Dims& s) {
  const int64_t per_query = static_cast<int64_t>(s.G) * s.d * 2 * 2;
  return make_group_plan(s, s.K, (int64_t(PISA_BWD_CHUNK_MIB) << 20) / per_query, PISA_BWD_ITEM_ROWS / s.G);
}

}  // namespace

AttnBwdWs attn_bwd_ws(const Dims& s) {
  AttnBwdWs w{};
  const size_t rows = static_cast<size_t>(s.B) * s.N * s.Hq;
  const size_t kvel = static_cast<size_t>(s.B) * s.N * s.Hkv_r * s.d;
  w.status = 0;                         // first: the caller finds the status word at offset 0
  size_t o = group_ws(bwd_plan(s), 256).end;
  w.delta = o;   o += align256(rows * 4);
  w.dq_acc = o;  o += align256(rows * s.d * 4);
  w.dk_acc = o;  o += align256(kvel * 4);
  w.dv_acc = o;  o += align256(kvel * 4);
  w.total = o;
  return w;
}

int launch_attn_bwd(const Dims& s, const void* Q, const void* K, const void* V, const void* O,
                    const float* lse, const void* dO, const int32_t* idx, void* dQ, void* dK,
                    void* dV, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnBwdWs w = attn_bwd_ws(s);
  const GroupPlan gp = bwd_plan(s);
  const GroupWs g = group_ws(gp, 256);
  float* delta = reinterpret_cast<float*>(ws + w.delta);
  float* dqa = reinterpret_cast<float*>(ws + w.dq_acc);
  float* dk_acc = reinterpret_cast<float*>(ws + w.dk_acc);
  float* dv_acc = reinterpret_cast<float*>(ws + w.dv_acc);
  const size_t kvel = static_cast<size_t>(s.B) * s.N * s.Hkv_r * s.d;
  int err = launch_group_items(gp, idx, ws, g, st);
  if (err) return err;
  cudaError_t e = cudaMemsetAsync(ws + w.status, 0, 256, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dk_acc, 0, kvel * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv_acc, 0, kvel * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dqa, 0, static_cast<size_t>(s.B) * s.N * s.Hq * s.d * 4, st);
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  {
    ProfScope ps(st, "attn_bwd_delta");
    if (s.d == 128)
      delta_kernel<128><<<blocks, 256, 0, st>>>(rows, static_cast<const __nv_bfloat16*>(O),
                                                static_cast<const __nv_bfloat16*>(dO), delta);
    else
      delta_kernel<64><<<blocks, 256, 0, st>>>(rows, static_cast<const __nv_bfloat16*>(O),
                                               static_cast<const __nv_bfloat16*>(dO), delta);
  }
  if ((err = cudaGetLastError())) return err;
  const int32_t* list = reinterpret_cast<const int32_t*>(ws + g.list);
  const int4* items = reinterpret_cast<const int4*>(ws + g.items);
  const int32_t* n_items = reinterpret_cast<const int32_t*>(ws + g.icount) + gp.bins;
  // d = 128 on the tensor-core kernel (attn_bwd_tc.cu); d = 64 on the warp-MMA kernel above
  err = s.d == 128 ? launch_attn_bwd_tc(s, gp, Q, K, V, dO, lse, delta, list, items, n_items, dqa, dk_acc, dv_acc,
                                        reinterpret_cast<int32_t*>(ws + w.status), st)
                   : bwd_dispatch<64>(s, gp, Q, K, V, dO, lse, delta, list, items, n_items, dqa, dk_acc, dv_acc, st);
  if (err) return err;
  {
    ProfScope ps(st, "attn_bwd_dkdv");
    const int64_t n8 = static_cast<int64_t>(kvel / 8);
    const int64_t nb = (n8 + 255) / 256;
    dkdv_convert_kernel<<<static_cast<unsigned>(nb < 152 * 32 ? nb : 152 * 32), 256, 0, st>>>(
        n8, s.scale, reinterpret_cast<const float4*>(dk_acc), reinterpret_cast<const float4*>(dv_acc),
        static_cast<uint4*>(dK), static_cast<uint4*>(dV), reinterpret_cast<const int32_t*>(ws + w.status));
  }
  {
    ProfScope ps(st, "attn_bwd_dq");
    const int64_t n8 = rows * s.d / 8;
    const int64_t nb = (n8 + 255) / 256;
    dq_convert_kernel<<<static_cast<unsigned>(nb < 152 * 32 ? nb : 152 * 32), 256, 0, st>>>(
        n8, reinterpret_cast<const float4*>(dqa), static_cast<uint4*>(dQ),
        reinterpret_cast<const int32_t*>(ws + w.status));
  }
  return cudaGetLastError();
}

}  // namespace pisa
