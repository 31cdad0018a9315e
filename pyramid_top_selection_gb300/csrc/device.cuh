// Device helpers shared by the PISA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace pisa {

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col), warp-wide.
// Fragment ownership for lane = 4*g + p (g = lane>>2, p = lane&3):
//   a[0]: A[g][k0,k0+1]   a[1]: A[g+8][k0,k0+1]   a[2]: A[g][k1,k1+1]   a[3]: A[g+8][k1,k1+1]
//   b[0]: B[k0,k0+1][g]   b[1]: B[k1,k1+1][g]
//   d[0..1]: D[g][2p,2p+1]  d[2..3]: D[g+8][2p,2p+1]
// with (k0, k1) = (2p, 2p+8) as MMA k-slots. The kernels map k-slots to physical
// contraction indices so that a lane's four slots (k0,k0+1,k1,k1+1) are four CONSECUTIVE
// elements 16*ks + 4p + {0,1,2,3}: a dot product does not depend on how its terms are
// labelled, as long as A and B use the same labels.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Split x into hi + lo, both bf16, hi = rn(x), lo = rn(x - hi): hi + lo carries ~16
// significant bits, so bf16 MMAs on (hi, lo) reproduce fp32 dot products to ~1e-5 relative.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// Bit mask of the lanes below this one.
__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint2 ldg_u2(const void* p) {
  return __ldg(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ uint4 ldg_u4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// A score that enters a top-K: NaN (only non-finite inputs make one) becomes -inf, so the
// order below stays total and a rank-based top-K never keeps more than K.
__device__ __forceinline__ float no_nan(float x) { return x != x ? neg_inf() : x; }

// Strict "a beats b" order of the selection: higher score, then lower node index (scores
// pass through no_nan first).
__device__ __forceinline__ bool beats(float sa, int ia, float sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}

}  // namespace pisa
