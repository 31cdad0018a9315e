/*
 * pisa.h -- C ABI of the GB300 (sm_103a) PISA hot path.
 *
 * PISA ("Block Sparse Attention with Log-Linear Complexity"): keys are grouped in leaf
 * blocks of C tokens and mean-pooled with merge factor 2 into a pyramid of O(log N)
 * levels; every query descends it from the single top node, scoring at most gK candidate
 * nodes per level with LogSumExp and keeping the top K, down to the leaves; leaves are
 * scored by the exact LSE over their raw keys, intermediate nodes by the LSE over their
 * children's mean keys; the query heads that share a KV head sum their LSEs and share one
 * selection. Attention is then causal softmax attention restricted to the selected leaf
 * blocks. (Problem statement: the arxivdaily page's English abstract. Leaf/intermediate
 * scoring, bounded gK candidates, GQA head sum, two-stage prefill kernel with queries
 * grouped per leaf block, single-kernel decode with an ancestor-path update: the daily
 * digest page, sections "Reference value of the work" and "Method key points".)
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller allocates and frees every buffer (inputs, outputs, workspace).
 *    The library never allocates, frees or synchronises; it only enqueues work.
 *  - Streams: every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream). Outputs are valid once the stream reaches them.
 *  - Layouts: row-major and contiguous. Q/O/dQ/dO [B,N,Hq,d], K/V/dK/dV [B,N,Hkv,d] in
 *    bf16 (token-major); pyramid sums fp32 [B,Hkv,nodes,d] with the levels concatenated
 *    leaves first (offsets from pisa_pyramid_layout); indices int32; scores/LSE fp32.
 *    Every pointer must be 16-byte aligned.
 *  - Query head h uses KV head floor(h / G), G = Hq / Hkv.
 *  - Errors: shapes, pointers, alignment and workspace size are checked on the host before
 *    any CUDA call; a failed check returns PISA_EINVAL / PISA_EUNSUPPORTED /
 *    PISA_EWORKSPACE and enqueues nothing. A launch failure returns PISA_ECUDA. The text
 *    of the last error of the calling thread is returned by pisa_last_error().
 *  - Supported in this build: d in {64,128}, C = 64, g in {2,4} (4 for the entry points
 *    named under pisa_shape_t), 1 <= K <= 32 with gK <= 64, G in {1,2,4,8},
 *    1 <= N <= 2^24, B*U*N*gK < 2^31 (U = Hkv, or Hq for a per-head selection) and
 *    B*N*Hq < 2^31. Anything else returns PISA_EUNSUPPORTED.
 */
#ifndef PISA_H_
#define PISA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PISA_VERSION 4
#define PISA_MAX_LEVELS 32

enum {
  PISA_OK = 0,
  PISA_EINVAL = 1,       /* bad argument (null/misaligned pointer, inconsistent shape) */
  PISA_EUNSUPPORTED = 2, /* valid per the method but not built here (see the list above) */
  PISA_EWORKSPACE = 3,   /* workspace pointer null or smaller than pisa_workspace_size */
  PISA_ECUDA = 4,        /* a kernel launch or async memset failed */
  PISA_ETIMEOUT = 5      /* never returned by a call: the code the Python binding raises when a
                            status word carries PISA_STATUS_TIMEOUT */
};

/* Device status word. Every call that takes a workspace clears the first 4 bytes of it on its
 * stream and ORs PISA_STATUS_* bits into them as its kernels run; read them (one int32) once
 * the stream has passed the call. 0 means every step ran to completion. pisa_decode_step
 * writes the same bits into its `status` argument.
 *   PISA_STATUS_POS_RANGE: a decode position was outside [0, Ncap); that sequence was skipped.
 *   PISA_STATUS_TIMEOUT:   a bounded wait inside a tensor-core kernel gave up (see
 *                          pisa_set_wait_limit). The kernel then stops early, drains the work
 *                          it had issued and frees its tensor memory; the call's outputs are
 *                          poisoned: idx = -1 and score/head_lse = NaN for the selections,
 *                          O = NaN and lse = NaN for the attention forward.
 * The selection entry point without a workspace (pisa_select_noalloc) reports a timeout
 * through the poisoned outputs only. */
enum { PISA_STATUS_POS_RANGE = 1, PISA_STATUS_TIMEOUT = 2 };

/* Operations that need a workspace (pisa_workspace_size's `op`): pisa_select,
 * pisa_select_flat, pisa_sparse_attn_fwd, pisa_sparse_attn_bwd, pisa_select_mean and
 * pisa_select_meanvar. */
enum {
  PISA_OP_SELECT = 0,
  PISA_OP_SELECT_FLAT = 1,
  PISA_OP_ATTN_FWD = 2,
  PISA_OP_ATTN_BWD = 3,
  PISA_OP_SELECT_MEAN = 4,
  PISA_OP_SELECT_MEANVAR = 5
};

/* Prefill/training shape. C = leaf block size in tokens, K = blocks kept per level,
 * g = candidate fan-out per kept node: 2 (the merge factor: candidates are the visible
 * children of the kept nodes) or 4 (two levels per step: the visible grandchildren, the last
 * step one level when that reaches the leaves; pisa_select and pisa_select_noalloc only;
 * the flat comparator has no descent and ignores g), qtile = scheduling hint for how many queries sharing a leaf block
 * form one tile (results never depend on it), scale = LSE and softmax temperature (0 selects
 * 1/sqrt(d)).
 * per_head = 0: the G query heads of a KV head sum their LSEs and share one selection;
 * selections are [B,Hkv,N,K]. per_head = 1 (explainer page, "five pitfalls" item 2: a
 * per-head top-K budget so that no head takes the others' share): every query head selects
 * its own K leaves with its own LSE scores over its KV head's keys; selections (idx, score)
 * are [B,Hq,N,K], and pisa_sparse_attn_fwd/bwd read such a selection per query head. The
 * pyramid always belongs to the KV heads ([B,Hkv,nodes,d]). */
typedef struct {
  int32_t B, N, Hq, Hkv, d, C, K, g, qtile;
  float scale;
  int32_t per_head;
} pisa_shape_t;

/* Decode shape: Ncap = KV-cache capacity in tokens per sequence (g = 2, shared selection). */
typedef struct {
  int32_t B, Ncap, Hq, Hkv, d, C, K, g;
  float scale;
} pisa_decode_shape_t;

int pisa_version(void);

/* Text of the calling thread's last error ("" if none). Owned by the library. */
const char* pisa_last_error(void);

/* Upper bound, in nanoseconds of the GPU's global timer, on every single device-side wait of
 * the tensor-core kernels (a pipeline stage waiting for another). 0 restores the default of
 * one second. Process-wide; applies to launches enqueued after the call. A wait that reaches
 * the bound gives up as described under PISA_STATUS_TIMEOUT. Host-only, no CUDA call. */
int pisa_set_wait_limit(uint64_t limit_ns);

/* Test aid (no counterpart on the pages): with on != 0, the tensor-core kernels of the
 * following pisa_select and pisa_sparse_attn_fwd launches wait, after their first key tile is
 * issued and before their first MMA, on a barrier that nothing signals, so that the wait
 * runs out after the wait limit and the give-up path runs (status PISA_STATUS_TIMEOUT,
 * poisoned outputs). Process-wide; 0 turns it off. Host-only, no CUDA call. */
int pisa_test_stall(int on);

/* Pyramid geometry for N tokens: n_levels = ceil(log2(ceil(N/C))) + 1, node offset of
 * every level inside one head's pyramid (level_offset[l], l < n_levels; may be NULL) and
 * the node count per (batch, KV head). Host-only, no CUDA call. */
int pisa_pyramid_layout(const pisa_shape_t* shape, int32_t* n_levels, int64_t* level_offset,
                        int64_t* nodes_per_head);

/* Bytes of workspace that `op` needs for `shape` (host-only, no CUDA call). The first 256
 * bytes of every workspace are the status block (status word at offset 0). */
int pisa_workspace_size(const pisa_shape_t* shape, int op, size_t* bytes);

/* Key pyramid (digest page, "Method key points": leaf blocks of C tokens, mean pooling
 * with merge factor 2, O(log N) levels). Writes fp32 key SUMS per node:
 *   leaf t:   S(0,t) = sum of k_j over tokens j in [tC, min(tC+C, N)), j ascending,
 *   parents:  S(l,m) = S(l-1,2m) + S(l-1,2m+1) (left alone when 2m+1 does not exist).
 * A node's mean summary is its sum over its token count. K: [B,N,Hkv,d] bf16 (read).
 * pyr_sum: [B,Hkv,nodes_per_head,d] fp32 (written). The summation order is fixed, so the
 * decode path's incremental update reproduces these sums bit for bit. */
int pisa_build_pyramid(const pisa_shape_t* shape, const void* K, float* pyr_sum, void* stream);

/* Pyramid Top-K selection (abstract; digest page "Method key points"): for every
 * (b, KV head, query i) -- (b, query head, i) with per_head -- descend from the top node; at
 * every level whose candidate set (the visible children of the kept nodes, at most gK;
 * grandchildren with g = 4) exceeds K, score the candidates
 * and keep the K best (higher score first, then lower index). Intermediate node m at
 * level l scores sum_{h in group} log sum_{visible child c} exp(s q_{i,h} . mu_i(l-1,c)),
 * leaf t scores sum_h log sum_{j in t, j <= i} exp(s q_{i,h} . k_j). A node is visible to
 * query i when its first token is <= i, and mu_i is the mean of the node's keys j <= i
 * (causal summaries). Two stages: per-query routing over the intermediate levels, then
 * exact leaf scoring with the queries grouped per candidate leaf block.
 *   Q [B,N,Hq,d], K [B,N,Hkv,d] bf16; pyr_sum from pisa_build_pyramid (read).
 *   idx   [B,Hkv,N,K] int32 (written): selected leaves ascending, -1 padded when fewer
 *         than K leaves are visible.
 *   score [B,Hkv,N,K] fp32 (written, may be NULL): leaf scores aligned with idx, -inf pad.
 *   head_lse [B,Hq,N,K] fp32 (written, may be NULL): the per-head terms of the score,
 *         head_lse[b,h,i,k] = log sum_{j in leaf idx[b,h/G,i,k], j <= i} exp(s q_{i,h}.k_j),
 *         -inf pad; the G heads of a KV head sum to its score. pisa_sparse_attn_fwd takes
 *         it to normalise the attention without a second pass over the keys.
 *   ws / ws_bytes: workspace of at least pisa_workspace_size(shape, PISA_OP_SELECT). */
int pisa_select(const pisa_shape_t* shape, const void* Q, const void* K, const float* pyr_sum,
                int32_t* idx, float* score, float* head_lse, void* ws, size_t ws_bytes,
                void* stream);

/* pisa_select without a caller workspace (the pages have no counterpart: this is an
 * integration aid). For callers that cannot hand the library device memory at call time,
 * for instance code running under an engine that owns a fixed device-memory arena and
 * forbids allocations on the serving path, or a plugin whose host exposes no allocator.
 * Same arguments, results and errors as pisa_select minus head_lse and ws/ws_bytes; it allocates
 * nothing and calls no allocating routine. Its scratch is one fixed 32 MiB array inside
 * the library's device image, held on a GPU from the moment that image is loaded there until
 * the process exits. Under CUDA's default lazy module loading the image (the array and the
 * selection kernels) is loaded by the first call on each device, so the driver reserves the
 * 32 MiB inside that first call: callers that forbid device allocation while serving make one
 * warm-up call per device at set-up, or run with CUDA_MODULE_LOADING=EAGER. That first call
 * should also come before any stream capture on the device. Each call looks up the array's
 * device address with the calling device current. Shapes whose selection workspace without
 * head_lse exceeds 32 MiB are rejected with PISA_EUNSUPPORTED before any CUDA call (about
 * B*Hkv*N <= 60K units at K = 16, G = 8; 70K at G = 4). Every call shares the one array and it keeps the last
 * call's contents: the call clears on its stream whatever must start at zero, and calls whose
 * GPU work overlaps in time (different streams or host threads on one device) race on the
 * array. A bounded wait that gives up is reported through poisoned outputs (idx = -1,
 * score = NaN), the array's status word being out of the caller's reach. */
int pisa_select_noalloc(const pisa_shape_t* shape, const void* Q, const void* K,
                        const float* pyr_sum, int32_t* idx, float* score, void* stream);

/* Flat block selection, the O(N^2/C) comparator (digest page, "Motivation": conventional
 * selection scores every query-block pair): leaf t scores sum_h s q_{i,h} . mu_i(0,t)
 * over every visible leaf; top K with the same tie rule and output layout as
 * pisa_select. Workspace: PISA_OP_SELECT_FLAT. */
int pisa_select_flat(const pisa_shape_t* shape, const void* Q, const void* K,
                     const float* pyr_sum, int32_t* idx, float* score, void* ws,
                     size_t ws_bytes, void* stream);

/* PISA-1 ablation selection (digest page, "Method key points": the ablation that scores
 * blocks by the mean instead of the LSE): the same coarse-to-fine descent as pisa_select,
 * but every block, leaves included, scores sum_h s q_{i,h} . mu_i(l,m), its own causal mean
 * key; no exact leaf stage. score (nullable) receives these mean scores of the selected
 * leaves (-inf padding). Same arguments, layouts, tie rule and errors as pisa_select minus
 * head_lse. Workspace: PISA_OP_SELECT_MEAN. */
int pisa_select_mean(const pisa_shape_t* shape, const void* Q, const void* K,
                     const float* pyr_sum, int32_t* idx, float* score, void* ws,
                     size_t ws_bytes, void* stream);

/* PISA-2 ablation selection (digest page, "Method key points": the ablation that scores
 * blocks by mean + variance). The pages give no formula; this library reads it as the
 * second-order cumulant expansion of a block's log-mean-exp with a diagonal covariance:
 * every block m at level l, leaves included, scores
 *     sum_h [ s q_{i,h} . mu_i(l,m) + (s^2 / 2) sum_k q_{i,h,k}^2 var_i(l,m)_k ],
 * mu_i and var_i the mean and the population variance per dimension of the block's keys
 * j <= i. Descent, K, tie rule, outputs and errors as pisa_select_mean; score (nullable)
 * receives these scores of the selected leaves. The call builds the squared-key pyramid it
 * needs inside its workspace (PISA_OP_SELECT_MEANVAR). Runs on the CUDA cores (an ablation,
 * not the method's hot path). */
int pisa_select_meanvar(const pisa_shape_t* shape, const void* Q, const void* K,
                        const float* pyr_sum, int32_t* idx, float* score, void* ws,
                        size_t ws_bytes, void* stream);

/* Causal block-sparse attention forward over the selected leaves (digest page,
 * "Reference value of the work"): o_{i,h} = sum_{j in J_i} softmax_j(s q_{i,h}.k_j) v_j,
 * J_i = keys j <= i inside the leaves idx[b, h/G, i, :] (-1 entries ignored).
 *   Q [B,N,Hq,d], K, V [B,N,Hkv,d] bf16; idx [B,Hkv,N,K] int32 (read).
 *   head_lse [B,Hq,N,K] fp32 (read, may be NULL): the per-block LSEs of these very idx,
 *         as pisa_select writes them. Given, the softmax normaliser lse is known before
 *         any key is visited; NULL, the call first computes them itself (one more pass of
 *         Q.K^T over the selected blocks). Values that are not those LSEs give wrongly
 *         normalised outputs; nothing checks them.
 *   O [B,N,Hq,d] bf16 and lse [B,Hq,N] fp32 = log sum_{j in J_i} exp(s q.k_j) (written);
 *         a row with no selected key gets O = 0 and lse = -inf.
 *   Workspace: PISA_OP_ATTN_FWD. */
int pisa_sparse_attn_fwd(const pisa_shape_t* shape, const void* Q, const void* K, const void* V,
                         const int32_t* idx, const float* head_lse, void* O, float* lse,
                         void* ws, size_t ws_bytes, void* stream);

/* Backward of the selected attention only; the discrete selection takes no gradient
 * (digest page, "Reference value of the work"). With P = exp(s q.k - lse),
 * D_i = dO_i . O_i, dS = P (dO . v - D): dQ = s dS K, dK = s dS^T Q, dV = P^T dO, where
 * dK and dV sum over the G query heads of their KV head.
 *   Q, O, dO [B,N,Hq,d], K, V [B,N,Hkv,d] bf16; lse [B,Hq,N] fp32 from the forward;
 *   idx [B,Hkv,N,K] (read). dQ [B,N,Hq,d], dK, dV [B,N,Hkv,d] bf16 (written).
 *   Workspace: PISA_OP_ATTN_BWD. */
int pisa_sparse_attn_bwd(const pisa_shape_t* shape, const void* Q, const void* K, const void* V,
                         const void* O, const float* lse, const void* dO, const int32_t* idx,
                         void* dQ, void* dK, void* dV, void* ws, size_t ws_bytes, void* stream);

/* Pyramid geometry over the cache capacity Ncap (host-only). */
int pisa_decode_pyramid_layout(const pisa_decode_shape_t* shape, int32_t* n_levels,
                               int64_t* level_offset, int64_t* nodes_per_head);

/* Builds the decode pyramid over Ncap from the first len[b] cached keys of every
 * sequence; nodes (or parts of nodes) past len[b] count as empty (zero sums). Same fixed
 * summation order as pisa_build_pyramid. Kcache [B,Ncap,Hkv,d] bf16, len device [B]
 * int32 (read); pyr_sum [B,Hkv,nodes_per_head(Ncap),d] fp32 (written). */
int pisa_decode_build_pyramid(const pisa_decode_shape_t* shape, const void* Kcache,
                              const int32_t* len, float* pyr_sum, void* stream);

/* One decode step for every sequence in ONE kernel launch (digest page, "Reference value
 * of the work": single kernel over all levels; the cached mean pyramid is updated only on
 * the new token's ancestor path). For sequence b with p = pos[b]:
 *   1. writes k_new/v_new at cache slot p;
 *   2. recomputes the sum of leaf floor(p/C) from its cached keys (pyramid order), then
 *      every ancestor as left + right;
 *   3. selects K leaves for query p exactly as pisa_select would for query p of a prefill
 *      over tokens 0..p, and
 *   4. attends over them.
 *   pos device [B] int32 (read, not advanced: the caller advances it).
 *   Kcache, Vcache [B,Ncap,Hkv,d] bf16 and pyr_sum (read + updated in place).
 *   q [B,Hq,d], k_new, v_new [B,Hkv,d] bf16 (read). o [B,Hq,d] bf16, idx [B,Hkv,K] int32,
 *   score [B,Hkv,K] fp32 (may be NULL) (written).
 *   status: device int32 word; the kernel ORs 1 into it when some pos[b] is outside
 *   [0, Ncap) (that sequence is then left untouched). It never traps. */
int pisa_decode_step(const pisa_decode_shape_t* shape, const int32_t* pos, void* Kcache,
                     void* Vcache, float* pyr_sum, const void* q, const void* k_new,
                     const void* v_new, void* o, int32_t* idx, float* score, int32_t* status,
                     void* stream);

/* Per-kernel timing (no counterpart on the pages: a measurement aid). After
 * pisa_profile_start(), every kernel that the library launches is bracketed by two CUDA
 * events recorded on its launch stream; pisa_profile_read() waits for the recorded events,
 * sums the elapsed time per kernel name into `out` (up to max_entries names; n_entries
 * receives how many), and clears the record. Up to 16384 launches are recorded between
 * reads; past that, launches go unrecorded and the read returns PISA_EWORKSPACE.
 * Host-thread: one thread at a time. Returns PISA_ECUDA if an event call fails. */
typedef struct {
  char name[48];
  int32_t launches;
  double total_ms;
} pisa_profile_entry_t;

int pisa_profile_start(void);
int pisa_profile_stop(void);
int pisa_profile_read(pisa_profile_entry_t* out, int32_t max_entries, int32_t* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* PISA_H_ */
