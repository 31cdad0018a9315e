"""PISA fp64 CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may import this
module. The product (the CUDA library and its Python binding) never calls it, and this
module imports nothing from the product: the two share no code. The only thing both sides
share is the seeded input generator module, which holds none of the method's arithmetic.

What is computed, and where it comes from ("Block Sparse Attention with Log-Linear
Complexity", PISA; three web pages about it):
  * the abstract (arxivdaily page, "English abstract"): a coarse-to-fine hierarchy of keys
    built by pooling, O(log N) levels, LogSumExp scoring of a bounded candidate set at
    every level, from the coarsest level down to the finest;
  * the daily digest page, section "Method key points": leaf blocks of C tokens, mean
    pooling with merge factor 2, the candidate set starts with 1 node, each level scores at
    most gK candidates, keeps the top K, expands only the kept nodes' children, down to
    the leaves; leaves are scored by exact LSE over raw keys, intermediate nodes by LSE
    over their children's mean summaries; under GQA the query heads that share a KV head
    share one selection (their LSEs are summed); gradients flow only through the selected
    attention;
  * the same page, section "Reference value of the work": the decode path keeps a cached
    mean pyramid and updates only the ancestor path of the new token.

Readings taken where the pages are silent (each one is listed in the design notes):
  R2  g = 2 (fan-out equals the merge factor), so a level holds at most 2K candidates.
  R24 g = 4 (a fan-out above the merge factor 2): each descent step goes down two levels,
      the candidates being the visible grandchildren of the kept nodes (at most 4K); a last
      step of one level reaches the leaves when the level count is odd. A candidate is still
      scored by the LSE over its two children's means (leaves: exact LSE).
  R25 per-head selection (the explainer's remedy for one head taking the shared budget):
      every query head selects its own K leaves with its own LSE scores, no sum over the
      group; the key summaries are those of its KV head.
  R3  the descent starts at the single top node; levels with <= K candidates keep all.
  R7  the LSE temperature is the attention scale s (default 1/sqrt(d)).
  R8  an intermediate node is scored with its (at most 2) immediate children, each
      represented by its mean key.
  R10 query head h belongs to KV head floor(h / G), G = Hq / Hkv.
  R11 causal summaries: every summary that query i sees is built only from keys j <= i;
      a node is visible to i iff its first token is <= i.
  R12 the query's own leaf is not forced; it is scored like any other leaf.
  R13 fewer than K visible leaves -> all visible leaves, padded with -1.
  R14 ties: higher score first, then lower node index.
  R15 the output leaf list is sorted ascending.
  R22 the digest's PISA-1 ablation ("scored by the mean"): every block, leaves included, is
      scored by sum_h s q_h . mu_i(l,m), its own causal mean key; descent and ties unchanged.
  R23 the digest's PISA-2 ablation ("mean + variance"): every block, leaves included, is
      scored by sum_h [s q_h . mu + (s^2 / 2) sum_k q_hk^2 var_k] over its causal keys, with
      var_k the population variance of dimension k: the second-order cumulant expansion of
      the block's log-mean-exp with a diagonal covariance; descent and ties unchanged.
Parity unpinned: R7, R8, R11, R12, R14, R22 and R23 are readings that nothing the pages print
can confirm; the pins in the tests check the oracle against the mathematics of those readings.

Precision: every input is the exact bf16 value promoted to float64; all arithmetic is fp64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------------------
# Pyramid geometry (digest page, "Method key points": leaf blocks of C tokens, merge 2)
# --------------------------------------------------------------------------------------
def level_sizes(N: int, C: int) -> list[int]:
    """Node counts per level, leaves first, up to the single top node."""
    sizes = [-(-N // C)]
    while sizes[-1] > 1:
        sizes.append(-(-sizes[-1] // 2))
    return sizes


def node_range(l: int, m: int, C: int, N: int) -> tuple[int, int]:
    """Token range [start, end) of node m at level l."""
    span = C << l
    return m * span, min((m + 1) * span, N)


def pyramid_sums(K_bk: np.ndarray, C: int) -> list[np.ndarray]:
    """Key sums of every node, computed straight from the definition (sum over the node's
    token range). K_bk: [N, d] keys of one (batch, KV head). Returns [n_l, d] per level.
    The pyramid's mean summary of a node is this sum divided by its token count."""
    N, d = K_bk.shape
    out = []
    for l, n in enumerate(level_sizes(N, C)):
        S = np.zeros((n, d), dtype=np.float64)
        for m in range(n):
            s, e = node_range(l, m, C, N)
            S[m] = K_bk[s:e].sum(axis=0)
        out.append(S)
    return out


@dataclass
class CausalKeySummaries:
    """Mean key summaries as seen by a query at token i (reading R11).

    A full node (last token <= i) uses the pyramid's mean; the node that holds i uses the
    mean of its keys j <= i (a prefix of the node), taken from an fp64 running sum."""
    K_bk: np.ndarray
    C: int
    sums: list = field(init=False)
    csum: np.ndarray = field(init=False)

    def __post_init__(self):
        self.N = self.K_bk.shape[0]
        self.sizes = level_sizes(self.N, self.C)
        self.sums = pyramid_sums(self.K_bk, self.C)
        self.csum = np.concatenate([np.zeros((1, self.K_bk.shape[1])), np.cumsum(self.K_bk, axis=0)])

    @property
    def top(self) -> int:
        return len(self.sizes) - 1

    def visible(self, l: int, m: int, i: int) -> bool:
        return 0 <= m < self.sizes[l] and node_range(l, m, self.C, self.N)[0] <= i

    def means(self, l: int, nodes: np.ndarray, i: int) -> np.ndarray:
        """[len(nodes), d] causal means of visible nodes at level l for query i."""
        out = np.empty((len(nodes), self.K_bk.shape[1]))
        for r, m in enumerate(nodes):
            s, e = node_range(l, int(m), self.C, self.N)
            if e - 1 <= i:
                out[r] = self.sums[l][m] / (e - s)
            else:
                out[r] = (self.csum[i + 1] - self.csum[s]) / (i + 1 - s)
        return out

    def variances(self, l: int, nodes: np.ndarray, i: int) -> np.ndarray:
        """[len(nodes), d] population variance, per dimension, of the causal keys of visible
        nodes at level l for query i (mean of squares minus squared mean)."""
        if not hasattr(self, "sq_sums"):
            self.sq_sums = pyramid_sums(self.K_bk * self.K_bk, self.C)
            self.csq = np.concatenate([np.zeros((1, self.K_bk.shape[1])), np.cumsum(self.K_bk * self.K_bk, axis=0)])
        mu = self.means(l, nodes, i)
        out = np.empty_like(mu)
        for r, m in enumerate(nodes):
            s, e = node_range(l, int(m), self.C, self.N)
            if e - 1 <= i:
                out[r] = self.sq_sums[l][m] / (e - s)
            else:
                out[r] = (self.csq[i + 1] - self.csq[s]) / (i + 1 - s)
        return out - mu * mu


# --------------------------------------------------------------------------------------
# Scores (digest page, "Method key points": exact LSE for leaves, LSE over child means for
# intermediate nodes; GQA heads sum their LSE -- "Reference value of the work")
# --------------------------------------------------------------------------------------
def _logsumexp(x: np.ndarray, axis: int) -> np.ndarray:
    m = np.max(x, axis=axis, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    s = np.sum(np.exp(x - m_safe), axis=axis, keepdims=True)
    with np.errstate(divide="ignore"):
        r = np.log(s) + m_safe
    return np.squeeze(r, axis=axis)


def leaf_scores(q: np.ndarray, i: int, leaves: np.ndarray, K_bk: np.ndarray, C: int,
                scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Exact leaf score S_i(0,t) = sum_h log sum_{j in leaf t, j <= i} exp(s q_h . k_j).

    q: [G, d]. Returns (summed score [n], per-head LSE [n, G])."""
    N = K_bk.shape[0]
    tot = np.empty(len(leaves))
    per_head = np.empty((len(leaves), q.shape[0]))
    for r, t in enumerate(leaves):
        s, e = node_range(0, int(t), C, N)
        e = min(e, i + 1)
        logits = scale * (q @ K_bk[s:e].T)          # [G, n_keys]
        per_head[r] = _logsumexp(logits, axis=1)
        tot[r] = per_head[r].sum()
    return tot, per_head


def node_scores(q: np.ndarray, i: int, l: int, nodes: np.ndarray, summ: CausalKeySummaries,
                scale: float) -> np.ndarray:
    """Intermediate score S_i(l,m) = sum_h log sum_{visible child c} exp(s q_h . mu_i(l-1,c))."""
    tot = np.empty(len(nodes))
    for r, m in enumerate(nodes):
        kids = [c for c in (2 * int(m), 2 * int(m) + 1) if summ.visible(l - 1, c, i)]
        mu = summ.means(l - 1, np.asarray(kids), i)   # [n_kids, d]
        logits = scale * (q @ mu.T)                    # [G, n_kids]
        tot[r] = _logsumexp(logits, axis=1).sum()
    return tot


def _top_k(cand: np.ndarray, scores: np.ndarray, K: int) -> tuple[np.ndarray, float]:
    """Keep the K best by (score descending, node index ascending); also the K-th vs
    (K+1)-th margin (inf when nothing is pruned)."""
    order = sorted(range(len(cand)), key=lambda r: (-scores[r], int(cand[r])))
    if len(cand) <= K:
        return cand[order], np.inf
    margin = scores[order[K - 1]] - scores[order[K]]
    return cand[order[:K]], float(margin)


# --------------------------------------------------------------------------------------
# Coarse-to-fine descent (abstract; digest page "Method key points": the candidate set
# starts with one node, at most gK candidates per level, keep the top K, expand children)
# --------------------------------------------------------------------------------------
@dataclass
class UnitSelection:
    leaves: np.ndarray           # ascending, len <= K
    scores: np.ndarray           # S_i(0,t) aligned with leaves
    head_lse: np.ndarray         # [len, G] per-head leaf LSE
    min_margin: float            # smallest K-th vs (K+1)-th margin over pruning levels
    cand_sizes: list             # |Cand| per level, top level first
    leaf_candidates: np.ndarray  # the (<= gK) leaves that reached exact scoring


def select_unit(q: np.ndarray, i: int, summ: CausalKeySummaries, K: int, scale: float,
                g: int = 2) -> UnitSelection:
    """Pyramid Top-K selection for one query i of one (batch, KV head); q: [G, d] (the heads
    whose LSEs are summed: the whole group, or one head for a per-head selection).

    g = 2: every step goes one level down (candidates = visible children of the kept nodes);
    g = 4: two levels (visible grandchildren), the last step one level when that reaches the
    leaves (reading R24)."""
    assert g in (2, 4), "fan-out g: 2 (the merge factor) or 4 (two levels per step)"
    step = 1 if g == 2 else 2
    kept = np.array([0], dtype=np.int64)            # A at the top level
    min_margin = np.inf
    cand_sizes = []
    cand = kept                                     # a single leaf: the top node
    l = summ.top
    while l > 0:
        nl = max(l - step, 0)
        t = l - nl                                  # levels this step goes down
        cand = np.array([c for a in kept for c in range(int(a) << t, (int(a) + 1) << t)
                         if summ.visible(nl, c, i)], dtype=np.int64)
        cand_sizes.append(len(cand))
        assert len(cand) <= g * K
        l = nl
        if l == 0:
            break
        if len(cand) <= K:
            kept = cand
            continue
        sc = node_scores(q, i, l, cand, summ, scale)
        kept, margin = _top_k(cand, sc, K)
        min_margin = min(min_margin, margin)
    leaf_cand = cand
    sc, ph = leaf_scores(q, i, leaf_cand, summ.K_bk, summ.C, scale)
    kept, margin = _top_k(leaf_cand, sc, K)
    min_margin = min(min_margin, margin)
    order = np.argsort(kept)
    kept = kept[order]
    pos = [int(np.nonzero(leaf_cand == t)[0][0]) for t in kept]
    return UnitSelection(kept, sc[pos], ph[pos], min_margin, cand_sizes, leaf_cand)


# --------------------------------------------------------------------------------------
# PISA-1 ablation (digest page, "Method key points": in the ablation, PISA-1 scores blocks
# by the mean instead of the LSE; the full LSE is reported to work better)
# --------------------------------------------------------------------------------------
def mean_scores(q: np.ndarray, i: int, l: int, nodes: np.ndarray, summ: CausalKeySummaries,
                scale: float) -> np.ndarray:
    """PISA-1 score of nodes at level l (l = 0: leaves): sum_h s q_h . mu_i(l, m)."""
    mu = summ.means(l, nodes, i)                      # [n, d]
    return (scale * (q @ mu.T)).sum(axis=0)


def meanvar_scores(q: np.ndarray, i: int, l: int, nodes: np.ndarray, summ: CausalKeySummaries,
                   scale: float) -> np.ndarray:
    """PISA-2 score of nodes at level l (l = 0: leaves):
    sum_h [s q_h . mu_i(l, m) + (s^2 / 2) sum_k q_hk^2 var_i(l, m)_k]."""
    mu = summ.means(l, nodes, i)                      # [n, d]
    var = summ.variances(l, nodes, i)                 # [n, d]
    return (scale * (q @ mu.T) + 0.5 * scale * scale * ((q * q) @ var.T)).sum(axis=0)


def select_unit_mean(q: np.ndarray, i: int, summ: CausalKeySummaries, K: int, scale: float,
                     g: int = 2, score_fn=None) -> tuple[np.ndarray, np.ndarray, float]:
    """The coarse-to-fine descent with one block score at every level, leaves included
    (PISA-1 mean scores by default, PISA-2 with score_fn=meanvar_scores); returns the
    ascending leaves, their scores and the smallest pruning margin."""
    assert g == 2, "the pyramid's merge factor is 2, so a node has 2 children"
    mean_scores_ = score_fn or mean_scores
    kept = np.array([0], dtype=np.int64)
    min_margin = np.inf
    cand = kept
    for l in range(summ.top - 1, -1, -1):
        cand = np.array([c for a in kept for c in (2 * int(a), 2 * int(a) + 1)
                         if summ.visible(l, c, i)], dtype=np.int64)
        if l == 0:
            break
        if len(cand) <= K:
            kept = cand
            continue
        kept, margin = _top_k(cand, mean_scores_(q, i, l, cand, summ, scale), K)
        min_margin = min(min_margin, margin)
    sc = mean_scores_(q, i, 0, cand, summ, scale)
    kept, margin = _top_k(cand, sc, K)
    min_margin = min(min_margin, margin)
    kept = np.sort(kept)
    pos = [int(np.nonzero(cand == t)[0][0]) for t in kept]
    return kept, sc[pos], min_margin


def select_meanvar(Q, K, C: int, K_sel: int, scale: float | None = None, queries=None, per_head: bool = False):
    """PISA-2 selection (reading R23), same outputs as select_mean."""
    return select_mean(Q, K, C, K_sel, scale, queries, score_fn=meanvar_scores, per_head=per_head)


def _units(Hq: int, Hkv: int, per_head: bool):
    """Selection units per batch and query heads per unit: the KV heads with their groups, or
    every query head on its own (per-head selection, reading R25)."""
    return (Hq, 1) if per_head else (Hkv, Hq // Hkv)


def select_mean(Q, K, C: int, K_sel: int, scale: float | None = None, queries=None, score_fn=None,
                per_head: bool = False):
    """PISA-1 selection for every (batch, unit, query): idx [B,U,N,K] ascending (-1 pad),
    score [B,U,N,K] (the PISA-1 leaf scores, -inf pad), margin [B,U,N]; U = Hkv, or Hq with
    per_head."""
    Q, K = _as64(Q), _as64(K)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    U, per = _units(Hq, Hkv, per_head)
    s = default_scale(d) if scale is None else float(scale)
    qs = range(N) if queries is None else [int(x) for x in queries]
    idx = np.full((B, U, N, K_sel), -1, dtype=np.int32)
    score = np.full((B, U, N, K_sel), np.nan)
    margin = np.full((B, U, N), np.nan)
    for b in range(B):
        for kv in range(Hkv):
            summ = CausalKeySummaries(K[b, :, kv, :], C)
            for un in range(kv * G // per, (kv + 1) * G // per):
                for i in qs:
                    leaves, sc, mg = select_unit_mean(Q[b, i, un * per:(un + 1) * per, :], i, summ, K_sel, s,
                                                      score_fn=score_fn)
                    idx[b, un, i, :len(leaves)] = leaves
                    score[b, un, i, :] = NEG_INF
                    score[b, un, i, :len(leaves)] = sc
                    margin[b, un, i] = mg
    return dict(idx=idx, score=score, margin=margin)


def _as64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def select(Q, K, C: int, K_sel: int, scale: float | None = None, queries=None, g: int = 2,
           per_head: bool = False):
    """Pyramid Top-K selection for every (batch, KV head, query), or with per_head for every
    (batch, query head, query) (reading R25). U = Hkv units per batch, or Hq with per_head.

    Q [B,N,Hq,d], K [B,N,Hkv,d]. Returns a dict with
      idx   int32 [B,U,N,K]    selected leaves, ascending, -1 padded
      score f64   [B,U,N,K]    S_i(0,t) (-inf on padding)
      head_lse f64 [B,Hq,N,K]  per-head leaf LSE of the selected leaves (-inf padding)
      margin f64  [B,U,N]      smallest pruning margin over all levels (inf if none)
      cand  int32 [B,U,N,gK]   leaf candidates that reached exact scoring (-1 padded)
    Only the queries listed in `queries` (default: all) are filled; the rest stay -1/nan."""
    Q, K = _as64(Q), _as64(K)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    U, per = _units(Hq, Hkv, per_head)
    s = default_scale(d) if scale is None else float(scale)
    qs = range(N) if queries is None else [int(x) for x in queries]
    idx = np.full((B, U, N, K_sel), -1, dtype=np.int32)
    score = np.full((B, U, N, K_sel), np.nan)
    head_lse = np.full((B, Hq, N, K_sel), np.nan)
    margin = np.full((B, U, N), np.nan)
    cand = np.full((B, U, N, g * K_sel), -1, dtype=np.int32)
    for b in range(B):
        for kv in range(Hkv):
            summ = CausalKeySummaries(K[b, :, kv, :], C)
            for un in range(kv * G // per, (kv + 1) * G // per):
                hs = slice(un * per, (un + 1) * per)
                for i in qs:
                    u = select_unit(Q[b, i, hs, :], i, summ, K_sel, s, g)
                    n = len(u.leaves)
                    idx[b, un, i, :n] = u.leaves
                    score[b, un, i, :] = NEG_INF
                    score[b, un, i, :n] = u.scores
                    head_lse[b, hs, i, :] = NEG_INF
                    head_lse[b, hs, i, :n] = u.head_lse.T
                    margin[b, un, i] = u.min_margin
                    cand[b, un, i, :len(u.leaf_candidates)] = np.sort(u.leaf_candidates)
    return dict(idx=idx, score=score, head_lse=head_lse, margin=margin, cand=cand)


# --------------------------------------------------------------------------------------
# Comparators: flat block selection (digest page, "Motivation": conventional block
# selection scores every query-block pair, O(N^2/C)) and exhaustive exact scoring
# --------------------------------------------------------------------------------------
def select_unit_flat(q: np.ndarray, i: int, summ: CausalKeySummaries, K: int,
                     scale: float) -> tuple[np.ndarray, np.ndarray, float]:
    """Flat BSA for one query i of one (batch, KV head): every visible leaf t scores
    sum_h s q_h . mu_i(0,t); returns the K best ascending, their scores and the margin."""
    vis = np.arange(i // summ.C + 1)
    sc = (scale * (q @ summ.means(0, vis, i).T)).sum(axis=0)
    kept, mg = _top_k(vis, sc, K)
    kept = np.sort(kept)
    return kept, sc[kept], mg


def select_flat(Q, K, C: int, K_sel: int, scale: float | None = None, queries=None, per_head: bool = False):
    """Flat BSA: score every visible leaf by sum_h s q_h . mu_i(0,t), keep the top K (per
    (batch, KV head, query), or per query head with per_head)."""
    Q, K = _as64(Q), _as64(K)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    U, per = _units(Hq, Hkv, per_head)
    s = default_scale(d) if scale is None else float(scale)
    qs = range(N) if queries is None else [int(x) for x in queries]
    idx = np.full((B, U, N, K_sel), -1, dtype=np.int32)
    score = np.full((B, U, N, K_sel), np.nan)
    margin = np.full((B, U, N), np.nan)
    for b in range(B):
        for kv in range(Hkv):
            summ = CausalKeySummaries(K[b, :, kv, :], C)
            for un in range(kv * G // per, (kv + 1) * G // per):
                for i in qs:
                    kept, sc, mg = select_unit_flat(Q[b, i, un * per:(un + 1) * per, :], i, summ, K_sel, s)
                    idx[b, un, i, :len(kept)] = kept
                    score[b, un, i, :] = NEG_INF
                    score[b, un, i, :len(kept)] = sc
                    margin[b, un, i] = mg
    return dict(idx=idx, score=score, margin=margin)


def select_exhaustive(Q, K, C: int, K_sel: int, scale: float | None = None, queries=None):
    """Exact leaf score for every visible leaf, then the top K (no pyramid)."""
    Q, K = _as64(Q), _as64(K)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    s = default_scale(d) if scale is None else float(scale)
    qs = range(N) if queries is None else [int(x) for x in queries]
    idx = np.full((B, Hkv, N, K_sel), -1, dtype=np.int32)
    score = np.full((B, Hkv, N, K_sel), np.nan)
    for b in range(B):
        for kv in range(Hkv):
            for i in qs:
                vis = np.arange(i // C + 1)
                sc, _ = leaf_scores(Q[b, i, kv * G:(kv + 1) * G, :], i, vis, K[b, :, kv, :], C, s)
                kept, _ = _top_k(vis, sc, K_sel)
                kept = np.sort(kept)
                idx[b, kv, i, :len(kept)] = kept
                score[b, kv, i, :] = NEG_INF
                score[b, kv, i, :len(kept)] = sc[kept]
    return dict(idx=idx, score=score)


# --------------------------------------------------------------------------------------
# Causal block-sparse attention over the selected leaves (digest page, "Reference value
# of the work": the discrete selection takes no gradient, only the selected attention)
# --------------------------------------------------------------------------------------
def selected_keys(idx_row: np.ndarray, i: int, C: int, N: int) -> np.ndarray:
    """J_i: token indices j <= i inside the selected leaves (ascending)."""
    js = []
    for t in sorted(int(t) for t in idx_row if t >= 0):
        s, e = node_range(0, t, C, N)
        js.extend(range(s, min(e, i + 1)))
    return np.asarray(js, dtype=np.int64)


def selected_head_lse(Q, K, idx, C: int, scale: float | None = None, queries=None):
    """Per-head LSE of every selected leaf: log sum_{j in leaf idx[b,kv,i,k], j <= i}
    exp(s q_{i,h} . k_j) for h in KV head kv's group (the exact leaf score of the digest
    page's "Method key points" before the GQA heads are summed).

    idx: [B,Hkv,N,K] (a selection shared by the group) or [B,Hq,N,K] (per head).
    Returns [B,Hq,N,K] f64: -inf for -1 slots, nan for queries not computed."""
    Q, K = _as64(Q), _as64(K)
    idx = np.asarray(idx)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    Ksel = idx.shape[-1]
    s = default_scale(d) if scale is None else float(scale)
    qs = range(N) if queries is None else [int(x) for x in queries]
    out = np.full((B, Hq, N, Ksel), np.nan)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            for i in qs:
                row = _idx_row(idx, b, h, G, Hkv, i)
                for k in range(Ksel):
                    t = int(row[k])
                    if t < 0:
                        out[b, h, i, k] = -np.inf
                        continue
                    lo, hi = node_range(0, t, C, N)
                    logits = s * (Q[b, i, h, :] @ K[b, lo:min(hi, i + 1), kv, :].T)   # [n]
                    out[b, h, i, k] = _logsumexp(logits, axis=0)
    return out


def _idx_row(idx: np.ndarray, b: int, h: int, G: int, Hkv: int, i: int) -> np.ndarray:
    """The selection row of query head h: its KV head's row of a selection shared by the
    group (idx [B,Hkv,N,K]) or its own row of a per-head selection (idx [B,Hq,N,K])."""
    return idx[b, h // G, i] if idx.shape[1] == Hkv else idx[b, h, i]


def sparse_attn_fwd(Q, K, V, idx, C: int, scale: float | None = None, queries=None):
    """o_{i,h} = sum_{j in J_i} softmax_j(s q_{i,h} . k_j) v_j ; lse_{i,h} = log sum exp.

    idx: [B,Hkv,N,K] (shared by the group) or [B,Hq,N,K] (per head).
    Returns O [B,N,Hq,d] f64 and lse [B,Hq,N] f64 (nan where not computed)."""
    Q, K, V = _as64(Q), _as64(K), _as64(V)
    idx = np.asarray(idx)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    s = default_scale(d) if scale is None else float(scale)
    qs = range(N) if queries is None else [int(x) for x in queries]
    O = np.full((B, N, Hq, d), np.nan)
    lse = np.full((B, Hq, N), np.nan)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            for i in qs:
                J = selected_keys(_idx_row(idx, b, h, G, Hkv, i), i, C, N)
                logits = s * (Q[b, i, h, :] @ K[b, J, kv, :].T)   # [|J|]
                l = _logsumexp(logits, axis=0)
                O[b, i, h, :] = np.exp(logits - l) @ V[b, J, kv, :]
                lse[b, h, i] = l
    return O, lse


def sparse_attn_bwd(Q, K, V, dO, idx, C: int, scale: float | None = None):
    """Gradients of sum(O * dO) w.r.t. Q, K, V with the selection held constant.

    P_ij = exp(s q_i.k_j - lse_i), D_i = dO_i . o_i, dS_ij = P_ij (dO_i . v_j - D_i),
    dQ_i = s sum_j dS_ij k_j, dK_j = s sum_{i,h in group} dS_ij q_i,
    dV_j = sum_{i,h in group} P_ij dO_i.
    idx: [B,Hkv,N,K] (shared by the group) or [B,Hq,N,K] (per head)."""
    Q, K, V, dO = _as64(Q), _as64(K), _as64(V), _as64(dO)
    idx = np.asarray(idx)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    s = default_scale(d) if scale is None else float(scale)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            for i in range(N):
                J = selected_keys(_idx_row(idx, b, h, G, Hkv, i), i, C, N)
                q, kJ, vJ, do = Q[b, i, h, :], K[b, J, kv, :], V[b, J, kv, :], dO[b, i, h, :]
                logits = s * (kJ @ q)
                P = np.exp(logits - _logsumexp(logits, axis=0))            # [|J|]
                D = do @ (P @ vJ)
                dS = P * (vJ @ do - D)
                dQ[b, i, h, :] = s * (dS @ kJ)
                dK[b, J, kv, :] += s * np.outer(dS, q)
                dV[b, J, kv, :] += np.outer(P, do)
    return dQ, dK, dV


# --------------------------------------------------------------------------------------
# Decode (digest page, "Reference value of the work": a cached mean pyramid that, for each
# new token, is updated only along that token's ancestor path; amortised O(log N))
# --------------------------------------------------------------------------------------
class DecodeState:
    """KV cache plus a cached key-sum pyramid over the cache capacity Ncap.

    Node sums cover only the tokens present so far (0..p); absent tokens count as zero,
    and a node's summary is its sum over its present tokens divided by their number."""

    def __init__(self, Kcache, Vcache, length: int, C: int):
        self.K = _as64(Kcache).copy()     # [B, Ncap, Hkv, d]
        self.V = _as64(Vcache).copy()
        self.B, self.Ncap, self.Hkv, self.d = self.K.shape
        self.C = C
        self.sizes = level_sizes(self.Ncap, C)
        self.len = np.full(self.B, int(length), dtype=np.int64)
        self.sums = [np.zeros((self.B, self.Hkv, n, self.d)) for n in self.sizes]
        for b in range(self.B):
            L = int(self.len[b])
            for l, n in enumerate(self.sizes):
                for m in range(n):
                    s, e = node_range(l, m, C, self.Ncap)
                    e = min(e, L)
                    if e > s:
                        self.sums[l][b, :, m, :] = self.K[b, s:e].sum(axis=0)

    def append(self, b: int, k_new: np.ndarray, v_new: np.ndarray) -> int:
        """Write token p = len[b] and update only its ancestor path."""
        p = int(self.len[b])
        assert p < self.Ncap
        self.K[b, p] = k_new
        self.V[b, p] = v_new
        t = p // self.C
        self.sums[0][b, :, t, :] = self.K[b, t * self.C:p + 1].sum(axis=0)   # leaf recompute
        m = t
        for l in range(1, len(self.sizes)):
            m //= 2
            left = self.sums[l - 1][b, :, 2 * m, :]
            right = self.sums[l - 1][b, :, 2 * m + 1, :] if 2 * m + 1 < self.sizes[l - 1] else 0.0
            self.sums[l][b, :, m, :] = left + right
        self.len[b] = p + 1
        return p

    def _mean(self, b, kv, l, m, p):
        s, e = node_range(l, m, self.C, self.Ncap)
        cnt = min(e, p + 1) - s
        return self.sums[l][b, kv, m, :] / cnt

    def select(self, b: int, kv: int, q: np.ndarray, K_sel: int, scale: float) -> UnitSelection:
        """Descent for the newest token p from the cached (partial-node) summaries."""
        p = int(self.len[b]) - 1
        vis = lambda l, m: m < self.sizes[l] and node_range(l, m, self.C, self.Ncap)[0] <= p
        kept = np.array([0], dtype=np.int64)
        min_margin = np.inf
        top = len(self.sizes) - 1
        cand = kept
        for l in range(top - 1, -1, -1):
            cand = np.array([c for a in kept for c in (2 * int(a), 2 * int(a) + 1) if vis(l, c)],
                            dtype=np.int64)
            if l == 0:
                break
            if len(cand) <= K_sel:
                kept = cand
                continue
            sc = np.empty(len(cand))
            for r, m in enumerate(cand):
                kids = [c for c in (2 * int(m), 2 * int(m) + 1) if vis(l - 1, c)]
                mu = np.stack([self._mean(b, kv, l - 1, c, p) for c in kids])
                sc[r] = _logsumexp(scale * (q @ mu.T), axis=1).sum()
            kept, mg = _top_k(cand, sc, K_sel)
            min_margin = min(min_margin, mg)
        sc, ph = leaf_scores(q, p, cand, self.K[b, :, kv, :], self.C, scale)
        kept, mg = _top_k(cand, sc, K_sel)
        min_margin = min(min_margin, mg)
        kept = np.sort(kept)
        pos = [int(np.nonzero(cand == t)[0][0]) for t in kept]
        return UnitSelection(kept, sc[pos], ph[pos], min_margin, [], cand)

    def step(self, q, k_new, v_new, K_sel: int, scale: float | None = None):
        """One decode step for every sequence: append, select, attend.

        q [B,Hq,d], k_new/v_new [B,Hkv,d]. Returns o [B,Hq,d], idx [B,Hkv,K],
        score [B,Hkv,K], margin [B,Hkv]."""
        q, k_new, v_new = _as64(q), _as64(k_new), _as64(v_new)
        Hq = q.shape[1]
        G = Hq // self.Hkv
        s = default_scale(self.d) if scale is None else float(scale)
        o = np.zeros((self.B, Hq, self.d))
        idx = np.full((self.B, self.Hkv, K_sel), -1, dtype=np.int32)
        score = np.full((self.B, self.Hkv, K_sel), NEG_INF)
        margin = np.full((self.B, self.Hkv), np.inf)
        for b in range(self.B):
            p = self.append(b, k_new[b], v_new[b])
            for kv in range(self.Hkv):
                hs = slice(kv * G, (kv + 1) * G)
                u = self.select(b, kv, q[b, hs, :], K_sel, s)
                idx[b, kv, :len(u.leaves)] = u.leaves
                score[b, kv, :len(u.leaves)] = u.scores
                margin[b, kv] = u.min_margin
                J = selected_keys(idx[b, kv], p, self.C, self.Ncap)
                logits = s * (q[b, hs, :] @ self.K[b, J, kv, :].T)
                P = np.exp(logits - _logsumexp(logits, axis=1)[:, None])
                o[b, hs, :] = P @ self.V[b, J, kv, :]
        return o, idx, score, margin


def sparse_attn_bwd_sampled(Q, K, V, dO, idx, C: int, scale: float | None = None,
                            queries=(), leaves=()):
    """The backward's definitions evaluated only where asked: dQ of the listed queries (all
    heads) and dK/dV of the keys of the listed (b, KV head, leaf) triples. dK/dV of a key
    sums over every (query, head) whose selection holds the key's leaf and sees the key.
    idx: [B,Hkv,N,K] (shared by the group) or [B,Hq,N,K] (per head).

    Returns (dQ {(b, i): [Hq, d]}, dK {(b, kv, t): [n_keys, d]}, dV {...})."""
    Q, K, V, dO = _as64(Q), _as64(K), _as64(V), _as64(dO)
    idx = np.asarray(idx)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    s = default_scale(d) if scale is None else float(scale)

    def row_terms(b, h, i):
        kv = h // G
        J = selected_keys(_idx_row(idx, b, h, G, Hkv, i), i, C, N)
        q, kJ, vJ, do = Q[b, i, h, :], K[b, J, kv, :], V[b, J, kv, :], dO[b, i, h, :]
        logits = s * (kJ @ q)
        P = np.exp(logits - _logsumexp(logits, axis=0))
        D = do @ (P @ vJ)
        dS = P * (vJ @ do - D)
        return J, q, kJ, do, P, dS

    dQ = {}
    for (b, i) in queries:
        out = np.zeros((Hq, d))
        for h in range(Hq):
            J, q, kJ, do, P, dS = row_terms(b, h, i)
            out[h] = s * (dS @ kJ)
        dQ[(b, i)] = out
    dK, dV = {}, {}
    for (b, kv, t) in leaves:
        s0, e0 = node_range(0, t, C, N)
        gk = np.zeros((e0 - s0, d))
        gv = np.zeros((e0 - s0, d))
        for h in range(kv * G, (kv + 1) * G):
            rows = idx[b, kv] if idx.shape[1] == Hkv else idx[b, h]
            for i in np.nonzero((rows == t).any(axis=-1))[0]:
                J, q, kJ, do, P, dS = row_terms(b, h, int(i))
                for c, j in enumerate(J):
                    if s0 <= j < e0:
                        gk[j - s0] += s * dS[c] * q
                        gv[j - s0] += P[c] * do
        dK[(b, kv, t)] = gk
        dV[(b, kv, t)] = gv
    return dQ, dK, dV
