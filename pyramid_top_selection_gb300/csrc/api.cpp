// C ABI of the PISA GB300 library: argument checks on the host (before any CUDA call),
// workspace sizing, and dispatch to the kernel launchers.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "internal.h"

namespace {

thread_local char g_err[512] = "";

constexpr uint64_t kDefaultWaitNs = 1000000000ull;   // one second
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stall{0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptr(const void* p, const char* name, bool nullable = false) {
  if (!p) return nullable ? PISA_OK : fail(PISA_EINVAL, "%s is NULL", name);
  if (!aligned16(p)) return fail(PISA_EINVAL, "%s is not 16-byte aligned", name);
  return PISA_OK;
}

#define PISA_CHECK(expr)          \
  do {                            \
    const int _rc = (expr);       \
    if (_rc != PISA_OK) return _rc; \
  } while (0)

int check_common(int B, int N, int Hq, int Hkv, int d, int C, int K, int g) {
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || d < 1 || C < 1 || K < 1 || g < 1)
    return fail(PISA_EINVAL, "sizes must be positive (B=%d N=%d Hq=%d Hkv=%d d=%d C=%d K=%d g=%d)",
                B, N, Hq, Hkv, d, C, K, g);
  if (Hq % Hkv != 0) return fail(PISA_EINVAL, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  const int G = Hq / Hkv;
  if (d != 64 && d != 128) return fail(PISA_EUNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
  if (C != 64) return fail(PISA_EUNSUPPORTED, "leaf block C=%d (supported: 64)", C);
  if (g != 2 && g != 4)
    return fail(PISA_EUNSUPPORTED, "fan-out g=%d (supported: 2, the merge factor, and 4, two levels per step)", g);
  if (K > 32) return fail(PISA_EUNSUPPORTED, "K=%d (supported: 1..32)", K);
  if (g * K > 64) return fail(PISA_EUNSUPPORTED, "g*K=%d candidates (supported: at most 64)", g * K);
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(PISA_EUNSUPPORTED, "GQA group G=%d (supported: 1, 2, 4, 8)", G);
  if (N > (1 << 24)) return fail(PISA_EUNSUPPORTED, "N=%d exceeds 2^24", N);
  const int64_t pairs = static_cast<int64_t>(B) * Hkv * N * g * K;
  if (pairs >= (int64_t(1) << 31))
    return fail(PISA_EUNSUPPORTED, "B*Hkv*N*gK=%lld exceeds 2^31", static_cast<long long>(pairs));
  const int64_t rows = static_cast<int64_t>(B) * N * Hq;   // TMA row coordinates are int32
  if (rows >= (int64_t(1) << 31))
    return fail(PISA_EUNSUPPORTED, "B*N*Hq=%lld exceeds 2^31", static_cast<long long>(rows));
  return PISA_OK;
}

int check_shape(const pisa_shape_t* s) {
  if (!s) return fail(PISA_EINVAL, "shape is NULL");
  PISA_CHECK(check_common(s->B, s->N, s->Hq, s->Hkv, s->d, s->C, s->K, s->g));
  if (s->qtile < 0) return fail(PISA_EINVAL, "qtile=%d is negative", s->qtile);
  if (s->per_head != 0 && s->per_head != 1) return fail(PISA_EINVAL, "per_head=%d (0 or 1)", s->per_head);
  if (s->per_head) {          // the units are the query heads
    const int64_t pairs = static_cast<int64_t>(s->B) * s->Hq * s->N * s->g * s->K;
    if (pairs >= (int64_t(1) << 31))
      return fail(PISA_EUNSUPPORTED, "B*Hq*N*gK=%lld exceeds 2^31 (per-head selection)", static_cast<long long>(pairs));
  }
  if (!(s->scale >= 0.f) || std::isinf(s->scale)) return fail(PISA_EINVAL, "scale must be finite and >= 0");
  return PISA_OK;
}

pisa::Dims dims_of(const pisa_shape_t* s) {
  pisa::Dims d{};
  d.B = s->B; d.N = s->N; d.Hq = s->Hq; d.Hkv = s->Hkv; d.d = s->d; d.C = s->C; d.K = s->K;
  d.G = s->Hq / s->Hkv;
  d.n0 = (s->N + s->C - 1) / s->C;
  d.scale = s->scale > 0.f ? s->scale : 1.0f / std::sqrt(static_cast<float>(s->d));
  d.Hkv_r = s->Hkv;
  d.kvr = 1;
  d.g = s->g;
  if (s->per_head) {          // every query head a selection unit of its own
    d.kvr = d.G;
    d.Hkv = s->Hq;
    d.G = 1;
  }
  return d;
}

// The real (per KV head) view of a shape, for the pyramid build: the pyramid always belongs to
// the KV heads.
pisa::Dims kv_dims_of(const pisa_shape_t* s) {
  pisa_shape_t r = *s;
  r.per_head = 0;
  return dims_of(&r);
}

pisa::Dims dims_of(const pisa_decode_shape_t* s) {
  pisa::Dims d{};
  d.B = s->B; d.N = s->Ncap; d.Hq = s->Hq; d.Hkv = s->Hkv; d.d = s->d; d.C = s->C; d.K = s->K;
  d.G = s->Hq / s->Hkv;
  d.n0 = (s->Ncap + s->C - 1) / s->C;
  d.scale = s->scale > 0.f ? s->scale : 1.0f / std::sqrt(static_cast<float>(s->d));
  d.Hkv_r = s->Hkv;
  d.kvr = 1;
  d.g = s->g;
  return d;
}

int cuda_rc(int err, const char* what) {
  if (err == 0) return PISA_OK;
  return fail(PISA_ECUDA, "%s: CUDA error %d (%s)", what, err, pisa::cuda_error_string(err));
}

int layout_out(const pisa::Geo& g, int32_t* n_levels, int64_t* level_offset, int64_t* nodes) {
  if (n_levels) *n_levels = g.n_levels;
  if (level_offset)
    for (int l = 0; l < g.n_levels; ++l) level_offset[l] = g.off[l];
  if (nodes) *nodes = g.nodes;
  return PISA_OK;
}

size_t ws_bytes_for(const pisa::Dims& d, const pisa::Geo& g, int op) {
  switch (op) {
    case PISA_OP_SELECT: return pisa::select_ws(d, g).total_head;
    case PISA_OP_SELECT_MEAN: return pisa::select_ws(d, g).mean_end;
    case PISA_OP_SELECT_MEANVAR: return pisa::meanvar_ws(d, g);
    case PISA_OP_SELECT_FLAT: return pisa::flat_ws(d, g);
    case PISA_OP_ATTN_FWD: return pisa::attn_fwd_ws(d).total;
    case PISA_OP_ATTN_BWD: return pisa::attn_bwd_ws(d).total;
    default: return 0;
  }
}

int check_ws_bytes(size_t need, const void* ws, size_t ws_bytes) {
  if (ws_bytes < need) return fail(PISA_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  if (need > 0 && !ws) return fail(PISA_EWORKSPACE, "workspace is NULL");
  if (ws && !aligned16(ws)) return fail(PISA_EINVAL, "workspace is not 16-byte aligned");
  return PISA_OK;
}

int check_ws(const pisa::Dims& d, const pisa::Geo& g, int op, const void* ws, size_t ws_bytes) {
  return check_ws_bytes(ws_bytes_for(d, g, op), ws, ws_bytes);
}

}  // namespace

namespace pisa {
uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int test_stall() { return g_stall.load(std::memory_order_relaxed); }
}  // namespace pisa

extern "C" {

int pisa_version(void) { return PISA_VERSION; }

const char* pisa_last_error(void) { return g_err; }

int pisa_set_wait_limit(uint64_t limit_ns) {
  g_wait_ns.store(limit_ns == 0 ? kDefaultWaitNs : limit_ns, std::memory_order_relaxed);
  return PISA_OK;
}

int pisa_test_stall(int on) {
  g_stall.store(on ? 1 : 0, std::memory_order_relaxed);
  return PISA_OK;
}

int pisa_pyramid_layout(const pisa_shape_t* shape, int32_t* n_levels, int64_t* level_offset,
                        int64_t* nodes_per_head) {
  PISA_CHECK(check_shape(shape));
  return layout_out(pisa::make_geo(shape->N, shape->C), n_levels, level_offset, nodes_per_head);
}

int pisa_workspace_size(const pisa_shape_t* shape, int op, size_t* bytes) {
  PISA_CHECK(check_shape(shape));
  if (!bytes) return fail(PISA_EINVAL, "bytes is NULL");
  if (op < PISA_OP_SELECT || op > PISA_OP_SELECT_MEANVAR) return fail(PISA_EINVAL, "unknown op %d", op);
  *bytes = ws_bytes_for(dims_of(shape), pisa::make_geo(shape->N, shape->C), op);
  return PISA_OK;
}

int pisa_build_pyramid(const pisa_shape_t* shape, const void* K, float* pyr_sum, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  const pisa::Dims d = kv_dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  return cuda_rc(pisa::launch_build_pyramid(d, g, K, nullptr, d.N, pyr_sum, stream), "pisa_build_pyramid");
}

int pisa_select(const pisa_shape_t* shape, const void* Q, const void* K, const float* pyr_sum,
                int32_t* idx, float* score, float* head_lse, void* ws, size_t ws_bytes, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(Q, "Q"));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  PISA_CHECK(check_ptr(idx, "idx"));
  PISA_CHECK(check_ptr(score, "score", true));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  PISA_CHECK(check_ptr(head_lse, "head_lse", true));
  PISA_CHECK(check_ws(d, g, PISA_OP_SELECT, ws, ws_bytes));
  return cuda_rc(pisa::launch_select(d, g, Q, K, pyr_sum, idx, score, head_lse, static_cast<char*>(ws), stream),
                 "pisa_select");
}

int pisa_select_noalloc(const pisa_shape_t* shape, const void* Q, const void* K,
                        const float* pyr_sum, int32_t* idx, float* score, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(Q, "Q"));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  PISA_CHECK(check_ptr(idx, "idx"));
  PISA_CHECK(check_ptr(score, "score", true));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  const size_t need = pisa::select_ws(d, g, false).total;
  if (need > pisa::noalloc_scratch_bytes())
    return fail(PISA_EUNSUPPORTED,
                "pisa_select_noalloc: this shape needs %zu bytes of scratch, more than the fixed %zu; "
                "use pisa_select with a caller workspace", need, pisa::noalloc_scratch_bytes());
  void* ws = nullptr;
  PISA_CHECK(cuda_rc(pisa::noalloc_scratch(&ws), "pisa_select_noalloc scratch set-up"));
  return cuda_rc(pisa::launch_select(d, g, Q, K, pyr_sum, idx, score, nullptr, static_cast<char*>(ws), stream, false),
                 "pisa_select_noalloc");
}

int pisa_select_flat(const pisa_shape_t* shape, const void* Q, const void* K,
                     const float* pyr_sum, int32_t* idx, float* score, void* ws,
                     size_t ws_bytes, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(Q, "Q"));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  PISA_CHECK(check_ptr(idx, "idx"));
  PISA_CHECK(check_ptr(score, "score", true));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  PISA_CHECK(check_ws(d, g, PISA_OP_SELECT_FLAT, ws, ws_bytes));
  return cuda_rc(pisa::launch_select_flat(d, g, Q, K, pyr_sum, idx, score, static_cast<char*>(ws), stream),
                 "pisa_select_flat");
}

int pisa_select_mean(const pisa_shape_t* shape, const void* Q, const void* K,
                     const float* pyr_sum, int32_t* idx, float* score, void* ws,
                     size_t ws_bytes, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(Q, "Q"));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  PISA_CHECK(check_ptr(idx, "idx"));
  PISA_CHECK(check_ptr(score, "score", true));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  if (shape->g != 2) return fail(PISA_EUNSUPPORTED, "pisa_select_mean: fan-out g=%d (supported: 2)", shape->g);
  PISA_CHECK(check_ws(d, g, PISA_OP_SELECT_MEAN, ws, ws_bytes));
  return cuda_rc(pisa::launch_select_mean(d, g, Q, K, pyr_sum, idx, score, static_cast<char*>(ws), stream),
                 "pisa_select_mean");
}

int pisa_select_meanvar(const pisa_shape_t* shape, const void* Q, const void* K,
                        const float* pyr_sum, int32_t* idx, float* score, void* ws,
                        size_t ws_bytes, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(Q, "Q"));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  PISA_CHECK(check_ptr(idx, "idx"));
  PISA_CHECK(check_ptr(score, "score", true));
  if (shape->g != 2) return fail(PISA_EUNSUPPORTED, "pisa_select_meanvar: fan-out g=%d (supported: 2)", shape->g);
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  PISA_CHECK(check_ws(d, g, PISA_OP_SELECT_MEANVAR, ws, ws_bytes));
  return cuda_rc(pisa::launch_select_meanvar(d, g, Q, K, pyr_sum, idx, score, static_cast<char*>(ws), stream),
                 "pisa_select_meanvar");
}

int pisa_sparse_attn_fwd(const pisa_shape_t* shape, const void* Q, const void* K, const void* V,
                         const int32_t* idx, const float* head_lse, void* O, float* lse, void* ws,
                         size_t ws_bytes, void* stream) {
  PISA_CHECK(check_shape(shape));
  PISA_CHECK(check_ptr(Q, "Q"));
  PISA_CHECK(check_ptr(K, "K"));
  PISA_CHECK(check_ptr(V, "V"));
  PISA_CHECK(check_ptr(idx, "idx"));
  PISA_CHECK(check_ptr(O, "O"));
  PISA_CHECK(check_ptr(lse, "lse"));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  PISA_CHECK(check_ptr(head_lse, "head_lse", true));
  PISA_CHECK(check_ws(d, g, PISA_OP_ATTN_FWD, ws, ws_bytes));
  return cuda_rc(pisa::launch_attn_fwd(d, Q, K, V, idx, head_lse, O, lse, static_cast<char*>(ws), stream),
                 "pisa_sparse_attn_fwd");
}

int pisa_sparse_attn_bwd(const pisa_shape_t* shape, const void* Q, const void* K, const void* V,
                         const void* O, const float* lse, const void* dO, const int32_t* idx,
                         void* dQ, void* dK, void* dV, void* ws, size_t ws_bytes, void* stream) {
  PISA_CHECK(check_shape(shape));
  const void* in[] = {Q, K, V, O, lse, dO, idx, dQ, dK, dV};
  const char* names[] = {"Q", "K", "V", "O", "lse", "dO", "idx", "dQ", "dK", "dV"};
  for (int k = 0; k < 10; ++k) PISA_CHECK(check_ptr(in[k], names[k]));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  PISA_CHECK(check_ws(d, g, PISA_OP_ATTN_BWD, ws, ws_bytes));
  return cuda_rc(pisa::launch_attn_bwd(d, Q, K, V, O, lse, dO, idx, dQ, dK, dV, static_cast<char*>(ws), stream),
                 "pisa_sparse_attn_bwd");
}

int pisa_decode_pyramid_layout(const pisa_decode_shape_t* shape, int32_t* n_levels,
                               int64_t* level_offset, int64_t* nodes_per_head) {
  if (!shape) return fail(PISA_EINVAL, "shape is NULL");
  PISA_CHECK(check_common(shape->B, shape->Ncap, shape->Hq, shape->Hkv, shape->d, shape->C, shape->K, shape->g));
  if (shape->g != 2) return fail(PISA_EUNSUPPORTED, "decode: fan-out g=%d (supported: 2)", shape->g);
  return layout_out(pisa::make_geo(shape->Ncap, shape->C), n_levels, level_offset, nodes_per_head);
}

int pisa_decode_build_pyramid(const pisa_decode_shape_t* shape, const void* Kcache,
                              const int32_t* len, float* pyr_sum, void* stream) {
  if (!shape) return fail(PISA_EINVAL, "shape is NULL");
  PISA_CHECK(check_common(shape->B, shape->Ncap, shape->Hq, shape->Hkv, shape->d, shape->C, shape->K, shape->g));
  if (shape->g != 2) return fail(PISA_EUNSUPPORTED, "decode: fan-out g=%d (supported: 2)", shape->g);
  PISA_CHECK(check_ptr(Kcache, "Kcache"));
  PISA_CHECK(check_ptr(len, "len"));
  PISA_CHECK(check_ptr(pyr_sum, "pyr_sum"));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  return cuda_rc(pisa::launch_build_pyramid(d, g, Kcache, len, d.N, pyr_sum, stream),
                 "pisa_decode_build_pyramid");
}

int pisa_decode_step(const pisa_decode_shape_t* shape, const int32_t* pos, void* Kcache,
                     void* Vcache, float* pyr_sum, const void* q, const void* k_new,
                     const void* v_new, void* o, int32_t* idx, float* score, int32_t* status,
                     void* stream) {
  if (!shape) return fail(PISA_EINVAL, "shape is NULL");
  PISA_CHECK(check_common(shape->B, shape->Ncap, shape->Hq, shape->Hkv, shape->d, shape->C, shape->K, shape->g));
  if (shape->g != 2) return fail(PISA_EUNSUPPORTED, "decode: fan-out g=%d (supported: 2)", shape->g);
  if (!(shape->scale >= 0.f) || std::isinf(shape->scale)) return fail(PISA_EINVAL, "scale must be finite and >= 0");
  const void* in[] = {pos, Kcache, Vcache, pyr_sum, q, k_new, v_new, o, idx, status};
  const char* names[] = {"pos", "Kcache", "Vcache", "pyr_sum", "q", "k_new", "v_new", "o", "idx", "status"};
  for (int k = 0; k < 10; ++k) PISA_CHECK(check_ptr(in[k], names[k]));
  PISA_CHECK(check_ptr(score, "score", true));
  const pisa::Dims d = dims_of(shape);
  const pisa::Geo g = pisa::make_geo(d.N, d.C);
  return cuda_rc(pisa::launch_decode_step(d, shape->Ncap, g, pos, Kcache, Vcache, pyr_sum, q, k_new,
                                          v_new, o, idx, score, status, stream),
                 "pisa_decode_step");
}

}  // extern "C"
