// Host-side declarations shared by the C ABI (api.cpp) and the kernel launchers (*.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/pisa.h"

namespace pisa {

// Pyramid geometry of one (batch, KV head): level l holds size[l] nodes starting at node
// offset off[l]; level 0 = leaves of C tokens, every level halves (rounding up).
struct Geo {
  int32_t n_levels;
  int32_t size[PISA_MAX_LEVELS];
  int64_t off[PISA_MAX_LEVELS];
  int64_t nodes;
};

inline Geo make_geo(int64_t N, int C) {
  Geo g{};
  int64_t n = (N + C - 1) / C;
  int64_t off = 0;
  int l = 0;
  while (true) {
    g.size[l] = static_cast<int32_t>(n);
    g.off[l] = off;
    off += n;
    ++l;
    if (n <= 1 || l >= PISA_MAX_LEVELS) break;
    n = (n + 1) / 2;
  }
  g.n_levels = l;
  g.nodes = off;
  return g;
}

// Plain-old-data view of a prefill shape with derived values, passed to kernels by value.
// Selection units are (b, kv) with kv < Hkv and G query heads kv*G .. kv*G+G-1 each. With a
// per-head selection every query head is a unit of its own: Hkv = Hq and G = 1 here, and the
// keys, values and pyramid of unit kv are those of KV head kv / kvr of the Hkv_r real ones
// (kvr = the real group size). Otherwise Hkv_r = Hkv and kvr = 1. g: candidate fan-out.
struct Dims {
  int32_t B, N, Hq, Hkv, d, C, K, G, n0;
  float scale;
  int32_t Hkv_r, kvr, g;
};

// Workspace carving for each op; every sub-buffer is 256-byte aligned.
// total: without the per-head leaf terms; total_head: with them (head_lse requested);
// mean_end: what the PISA-1 path uses.
// status: the first 256 bytes of every workspace, zeroed before the op's kernels; word 0
// collects PISA_STATUS_* bits (the caller reads it there), words 16 and 32 are the item
// counters of the persistent leaf-scoring and attention kernels.
struct SelectWs {
  size_t status, split, pd, cfirst, cand, cscore, mean_end, group, total, chead, total_head;
};
struct AttnFwdWs {
  size_t block_lse, o_acc, status, total;
};
struct AttnBwdWs {
  size_t status, delta, dq_acc, dk_acc, dv_acc, total;
};
int sm_count();
// first: the first scored level's child dots precomputed where that pays (G <= 4); the
// fixed-scratch entry point turns it off to keep its scratch per query small.
SelectWs select_ws(const Dims& s, const Geo& g, bool first = true);
AttnFwdWs attn_fwd_ws(const Dims& s);
AttnBwdWs attn_bwd_ws(const Dims& s);
size_t flat_ws(const Dims& s, const Geo& g);

// Launchers: return 0 or a cudaError_t value.
int launch_build_pyramid(const Dims& s, const Geo& g, const void* K, const int32_t* len,
                         int64_t tokens_per_seq, float* pyr, void* stream);
int launch_select(const Dims& s, const Geo& g, const void* Q, const void* K, const float* pyr,
                  int32_t* idx, float* score, float* head_lse, char* ws, void* stream, bool first = true);
int launch_select_flat(const Dims& s, const Geo& g, const void* Q, const void* K,
                       const float* pyr, int32_t* idx, float* score, char* ws, void* stream);
int launch_select_mean(const Dims& s, const Geo& g, const void* Q, const void* K,
                       const float* pyr, int32_t* idx, float* score, char* ws, void* stream);
int launch_select_meanvar(const Dims& s, const Geo& g, const void* Q, const void* K,
                          const float* pyr, int32_t* idx, float* score, char* ws, void* stream);
size_t meanvar_ws(const Dims& s, const Geo& g);
int launch_attn_fwd(const Dims& s, const void* Q, const void* K, const void* V, const int32_t* idx,
                    const float* head_lse, void* O, float* lse, char* ws, void* stream);
int launch_attn_bwd(const Dims& s, const void* Q, const void* K, const void* V, const void* O,
                    const float* lse, const void* dO, const int32_t* idx, void* dQ, void* dK,
                    void* dV, char* ws, void* stream);
int launch_decode_step(const Dims& s, int32_t Ncap, const Geo& g, const int32_t* pos,
                       void* Kc, void* Vc, float* pyr, const void* q, const void* k_new,
                       const void* v_new, void* o, int32_t* idx, float* score, int32_t* status,
                       void* stream);
const char* cuda_error_string(int err);
// Bound of every device-side pipeline wait (pisa_set_wait_limit), and the test stall switch
// (pisa_test_stall), as the launchers pass them to the tensor-core kernels.
uint64_t wait_limit_ns();
int test_stall();
size_t noalloc_scratch_bytes();
int noalloc_scratch(void** out);

}  // namespace pisa
