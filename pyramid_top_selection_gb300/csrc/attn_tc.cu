// Causal block-sparse attention forward: orchestration of the passes, and the two small
// row-wise kernels around the tensor-core output pass (attn_ws.cu).
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference value
// of the work": attention runs only over the selected blocks. Row (query i, head h) has
// lse = log sum_k exp(lse_k) over the LSEs of its selected blocks. The selection computes
// those block LSEs exactly (the per-head terms of its leaf scores) and hands them over;
// without them, the leaf-scoring kernel computes them over the selected pairs first. With
// lse known up front, every block's contribution is final and is added into an fp32
// accumulator, which a last kernel converts to bf16.
#include "device.cuh"
#include "group.h"
#include "profile.h"

namespace pisa {

int launch_block_lse_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const int32_t* list,
                        const int4* items, const int32_t* n_items, float* block_lse, int32_t* status,
                        cudaStream_t st);
int launch_attn_out_ws(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       const float* lse_rows, float* o_acc, int32_t* status, cudaStream_t st);

namespace {

// lse = log sum_k exp(block_lse_k) over each row's valid slots, written to the caller's lse
// ([B,Hq,N]); rows in lse order, one thread per row. A row's K block LSEs are contiguous, and
// so are its slot indices (shared by the G heads of its KV head): 16-byte loads when K is a
// multiple of 4.
constexpr int kRowThreads = 256;
constexpr int kMaxK = 32;

template <bool V4>
__global__ void __launch_bounds__(kRowThreads)
attn_rows_kernel(Dims s, const int32_t* __restrict__ idx, const float* __restrict__ block_lse,
                 float* __restrict__ lse_out) {
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  const int64_t lrow = blockIdx.x * static_cast<int64_t>(kRowThreads) + threadIdx.x;   // (b*Hq + h)*N + i
  if (lrow >= rows) return;
  const int K = s.K;
  const int i = static_cast<int>(lrow % s.N);
  const int64_t bh = lrow / s.N;
  const int h = static_cast<int>(bh % s.Hq), b = static_cast<int>(bh / s.Hq);
  const int32_t* id = idx + ((static_cast<int64_t>(b) * s.Hkv + h / s.G) * s.N + i) * K;
  const float* bl = block_lse + lrow * K;
  float v[kMaxK];
  if constexpr (V4) {
#pragma unroll
    for (int k = 0; k < kMaxK; k += 4) {
      if (k >= K) break;
      const float4 l = __ldg(reinterpret_cast<const float4*>(bl + k));
      const int4 t = __ldg(reinterpret_cast<const int4*>(id + k));
      v[k] = t.x >= 0 ? l.x : neg_inf();
      v[k + 1] = t.y >= 0 ? l.y : neg_inf();
      v[k + 2] = t.z >= 0 ? l.z : neg_inf();
      v[k + 3] = t.w >= 0 ? l.w : neg_inf();
    }
  } else {
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      if (k >= K) break;
      v[k] = __ldg(id + k) >= 0 ? __ldg(bl + k) : neg_inf();
    }
  }
  float m = neg_inf();
#pragma unroll
  for (int k = 0; k < kMaxK; ++k)
    if (k < K) m = fmaxf(m, v[k]);
  float den = 0.f;
  if (m != neg_inf()) {
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
      if (k < K && v[k] != neg_inf()) den += expf(v[k] - m);
  }
  lse_out[lrow] = den > 0.f ? m + logf(den) : neg_inf();
}

// O = bf16(accumulator), 8 elements per thread. When the status word carries
// PISA_STATUS_TIMEOUT (a bounded wait of a tensor-core pass gave up, so some block
// contributions are missing) O and lse are poisoned instead: every element NaN.
__global__ void __launch_bounds__(256)
attn_out_kernel(Dims s, int64_t n8, const float4* __restrict__ o_acc, uint4* __restrict__ O,
                float* __restrict__ lse, const int32_t* __restrict__ status) {
  const bool poison = (*status & PISA_STATUS_TIMEOUT) != 0;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n8;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (poison) {
      O[q] = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
      const int64_t e = q * 8;
      if (e % s.d == 0) {                      // the row's first chunk: row = (b*N + i)*Hq + h
        const int64_t row = e / s.d;
        const int64_t h = row % s.Hq, bi = row / s.Hq;
        lse[((bi / s.N) * s.Hq + h) * s.N + bi % s.N] = __int_as_float(0x7fc00000);
      }
      continue;
    }
    const float4 a = o_acc[2 * q], c = o_acc[2 * q + 1];
    O[q] = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(c.x, c.y), pack_bf16(c.z, c.w));
  }
}

}  // namespace

// Attention forward for d in {64, 128} and G in {1, 2, 4, 8}: [block LSE pass when
// head_lse is NULL] -> accumulator clear, row LSE -> output pass -> bf16 conversion.
int launch_attn_fwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       const float* head_lse, float* block_lse_ws, float* o_acc, void* O, float* lse,
                       int32_t* status, cudaStream_t st) {
  const float* hl = head_lse;
  int err;
  if (!hl) {
    if ((err = launch_block_lse_tc(s, gp, Q, K, list, items, n_items, block_lse_ws, status, st))) return err;
    hl = block_lse_ws;
  }
  const int64_t rows = static_cast<int64_t>(s.B) * s.N * s.Hq;
  {
    ProfScope ps(st, "attn_clear");
    if ((err = cudaMemsetAsync(o_acc, 0, static_cast<size_t>(rows) * s.d * 4, st))) return err;
  }
  {
    ProfScope ps(st, "attn_rows");
    const unsigned nb = static_cast<unsigned>((rows + kRowThreads - 1) / kRowThreads);
    if (s.K % 4 == 0)
      attn_rows_kernel<true><<<nb, kRowThreads, 0, st>>>(s, idx, hl, lse);
    else
      attn_rows_kernel<false><<<nb, kRowThreads, 0, st>>>(s, idx, hl, lse);
  }
  if ((err = cudaGetLastError())) return err;
  if ((err = launch_attn_out_ws(s, gp, Q, K, V, idx, list, items, n_items, lse, o_acc, status, st))) return err;
  {
    ProfScope ps(st, "attn_out");
    const int64_t n8 = rows * s.d / 8;
    const int64_t nb = (n8 + 255) / 256;
    attn_out_kernel<<<static_cast<unsigned>(nb < 152 * 32 ? nb : 152 * 32), 256, 0, st>>>(
        s, n8, reinterpret_cast<const float4*>(o_acc), static_cast<uint4*>(O), lse, status);
  }
  return cudaGetLastError();
}

}  // namespace pisa
