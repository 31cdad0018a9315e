// Causal block-sparse attention over the selected leaf blocks: workspace layout and launch.
//
// "Block Sparse Attention with Log-Linear Complexity", daily digest page, "Reference
// value of the work": attention runs only over the selected blocks and gradients pass
// only through that attention (the discrete selection takes none); the prefill kernel
// groups the queries that use the same leaf key block into tiles so the block's keys are
// read once per tile.
//
// Forward, block-major: the selected (leaf, query) pairs are grouped by (KV head, query
// chunk, leaf) and cut into work items (group.cu); the tensor-core kernel (attn_tc.cu)
// takes one item per CTA. A row's softmax normaliser lse = log sum_t exp(lse_t) comes
// from the per-block LSEs lse_t (the selection's per-head leaf terms, or a first S-only
// pass), so each (row, block) adds its final share exp(s q.k - lse) v into an fp32
// accumulator; a last kernel converts the accumulator to bf16.
#include "device.cuh"
#include "group.h"
#include "profile.h"

namespace pisa {

int launch_attn_fwd_tc(const Dims& s, const GroupPlan& gp, const void* Q, const void* K, const void* V,
                       const int32_t* idx, const int32_t* list, const int4* items, const int32_t* n_items,
                       const float* head_lse, float* block_lse_ws, float* o_acc, void* O, float* lse,
                       int32_t* status, cudaStream_t st);

namespace {

// Query chunks of about 32 MiB of one KV head's fp32 accumulator rows (G heads x d): the
// items running at one time add into one chunk's rows, which then stay in L2. At the 64K
// workload 128 / 48 / 32 / 24 / 16 MiB took 2.13 / 1.68 / 1.67 / 1.70 / 1.74 ms per launch, and
// at 32K the launch moved 1.51 / 1.15 / 1.02 / 0.75 GB of DRAM traffic at 48 / 32 / 24 / 16 MiB
// (smaller chunks keep more of the accumulator in L2 but make smaller work items); at most 512
// queries per work item (1024 measured slower).
#ifndef PISA_FWD_CHUNK_MIB
#define PISA_FWD_CHUNK_MIB 32
#endif
#ifndef PISA_FWD_ITEM_CAP
#define PISA_FWD_ITEM_CAP 512
#endif
// With the per-block LSEs given, the output pass takes sibling leaves (2m, 2m + 1) together:
// a row that selected both is gathered and reduced once for the pair. The S-only LSE pass
// (head_lse NULL) keeps one leaf per item, since it writes one LSE per (row, slot).
#ifndef PISA_FWD_PAIRS
#define PISA_FWD_PAIRS 1
#endif
GroupPlan fwd_plan(const Dims& s, bool pairs) {
  const int64_t per_query = static_cast<int64_t>(s.G) * s.d * 4;
  const int sh = pairs && PISA_FWD_PAIRS ? 1 : 0;
  return make_group_plan(s, s.K, (int64_t(PISA_FWD_CHUNK_MIB) << 20) / per_query, PISA_FWD_ITEM_CAP, sh, sh);
}

}  // namespace

AttnFwdWs attn_fwd_ws(const Dims& s) {
  AttnFwdWs w{};
  const GroupPlan gp = fwd_plan(s, false);   // the larger of the two plans' buffers
  const size_t rows = static_cast<size_t>(s.B) * s.N * s.Hq;
  w.status = 0;                         // first: the caller finds the status word at offset 0
  size_t o = group_ws(gp, 256).end;
  w.block_lse = o; o += align256(rows * s.K * 4);
  w.o_acc = o;     o += align256(rows * s.d * 4);
  w.total = o;
  return w;
}

int launch_attn_fwd(const Dims& s, const void* Q, const void* K, const void* V, const int32_t* idx,
                    const float* head_lse, void* O, float* lse, char* ws, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnFwdWs w = attn_fwd_ws(s);
  const GroupPlan gp = fwd_plan(s, head_lse != nullptr);
  const GroupWs g = group_ws(gp, 256);
  int err = launch_group_items(gp, idx, ws, g, st);
  if (err) return err;
  cudaError_t e = cudaMemsetAsync(ws + w.status, 0, 256, st);
  if (e != cudaSuccess) return e;
  const int32_t* list = reinterpret_cast<const int32_t*>(ws + g.list);
  const int4* items = reinterpret_cast<const int4*>(ws + g.items);
  const int32_t* n_items = reinterpret_cast<const int32_t*>(ws + g.icount) + gp.bins;
  return launch_attn_fwd_tc(s, gp, Q, K, V, idx, list, items, n_items, head_lse,
                            reinterpret_cast<float*>(ws + w.block_lse), reinterpret_cast<float*>(ws + w.o_acc),
                            O, lse, reinterpret_cast<int32_t*>(ws + w.status), st);
}

}  // namespace pisa
