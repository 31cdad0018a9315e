"""Seeded synthetic inputs for the PISA hot path (shared by the CUDA path and the oracle).

This module holds no arithmetic of the method itself: it only draws random tensors and
plants "needles" into keys. Both the CUDA library and the fp64 oracle read the very same
bf16 bits that these functions return.

Workloads follow the shapes of "Block Sparse Attention with Log-Linear Complexity"
(PISA): bf16 Q/K/V drawn i.i.d. N(0, 1), optionally with needle-planted key blocks so
that block selection has a correct answer.

Seeds (seed = 0 by default):
  Q = seed, K = seed + 1, V = seed + 2, needle leaves = seed + 3, upstream dO = seed + 4,
  decode token stream = seed + 5.

Needles (per batch b and KV head kappa): u = unit(sum over tokens i and query heads h of
group kappa of q[b, i, h]) computed in fp32; 8 distinct leaf blocks are drawn uniformly
from [0, n_leaves); every key of those blocks becomes bf16(k + 3 u).
"""
from __future__ import annotations

import torch


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """fp32 N(0,1) draws from a seeded generator, rounded to bf16 (round-to-nearest-even)."""
    x = torch.randn(*shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def needle_direction(Q: torch.Tensor, Hkv: int, b: int, kv: int) -> torch.Tensor:
    """u = unit(sum over tokens and the group's query heads of q), fp32 [d]."""
    G = Q.shape[2] // Hkv
    u = Q[b, :, kv * G:(kv + 1) * G, :].to(torch.float32).sum(dim=(0, 1))
    return u / u.norm().clamp_min(1e-30)


def needle_leaves(B: int, Hkv: int, n0: int, seed: int, n_needles: int = 8, device="cpu"):
    """The needle leaf indices [b][kv] -> list, drawn exactly as plant_needles draws them."""
    g = _gen(device, seed)
    n_pick = min(n_needles, n0)
    return [[torch.randperm(n0, generator=g, device=device)[:n_pick].tolist() for _ in range(Hkv)]
            for _ in range(B)]


def plant_needles(Q: torch.Tensor, K: torch.Tensor, C: int, seed: int, n_needles: int = 8,
                  strength: float = 3.0) -> torch.Tensor:
    """Return a copy of K [B,N,Hkv,d] with needle leaf blocks planted (see module doc)."""
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    n0 = (N + C - 1) // C
    K = K.clone()
    leaves = needle_leaves(B, Hkv, n0, seed, n_needles, K.device)
    for b in range(B):
        for kv in range(Hkv):
            u = needle_direction(Q, Hkv, b, kv)
            for t in leaves[b][kv]:
                s, e = t * C, min((t + 1) * C, N)
                K[b, s:e, kv, :] = (K[b, s:e, kv, :].to(torch.float32) + strength * u).to(torch.bfloat16)
    return K


def make_prefill(B: int, N: int, Hq: int, Hkv: int, d: int, C: int = 64, seed: int = 0,
                 needles: bool = False, device="cpu"):
    """Q [B,N,Hq,d], K [B,N,Hkv,d], V [B,N,Hkv,d] bf16, token-major and contiguous."""
    Q = randn_bf16((B, N, Hq, d), seed, device)
    K = randn_bf16((B, N, Hkv, d), seed + 1, device)
    V = randn_bf16((B, N, Hkv, d), seed + 2, device)
    if needles:
        K = plant_needles(Q, K, C, seed + 3)
    return Q, K, V


def make_grad_out(B: int, N: int, Hq: int, d: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Upstream gradient dO [B,N,Hq,d] bf16 N(0,1)."""
    return randn_bf16((B, N, Hq, d), seed + 4, device)


def make_decode_stream(B: int, steps: int, Hq: int, Hkv: int, d: int, seed: int = 0, device="cpu"):
    """Fresh per-step decode tokens: q [steps,B,Hq,d], k/v [steps,B,Hkv,d] bf16 N(0,1)."""
    q = randn_bf16((steps, B, Hq, d), seed + 5, device)
    k = randn_bf16((steps, B, Hkv, d), seed + 6, device)
    v = randn_bf16((steps, B, Hkv, d), seed + 7, device)
    return q, k, v


def query_subsample(N: int, every: int = 7, tail: int = 4096) -> torch.Tensor:
    """Deterministic query subsample for full-size parity: every `every`-th query + the last `tail`."""
    idx = set(range(0, N, every)) | set(range(max(0, N - tail), N))
    return torch.tensor(sorted(idx), dtype=torch.int64)


def random_selection(B: int, Hkv: int, N: int, C: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """A uniformly random valid selection: for every (b, KV head, query i), K distinct leaves
    among the visible ones 0..floor(i/C) (all of them if fewer), ascending, -1 padded.
    Returns int32 [B, Hkv, N, K]."""
    n0 = (N + C - 1) // C
    g = _gen(device, seed)
    r = torch.rand(B, Hkv, N, n0, generator=g, device=device)
    vis = torch.arange(n0, device=device).view(1, 1, 1, n0) <= (torch.arange(N, device=device) // C).view(1, 1, N, 1)
    r = torch.where(vis, r, torch.full_like(r, -1.0))
    k = min(K, n0)
    val, pick = torch.topk(r, k, dim=-1)
    pick = torch.where(val >= 0, pick, torch.full_like(pick, n0 + 1))
    pick = torch.sort(pick, dim=-1).values
    pick = torch.where(pick > n0, torch.full_like(pick, -1), pick)
    out = torch.full((B, Hkv, N, K), -1, dtype=torch.int32, device=device)
    out[..., :k] = pick.to(torch.int32)
    return out
