"""fp64 CPU oracle: exact scaled-dot-product attention, per-tile partials and the LSE merge.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module; the product path (the C-ABI library and its
Python binding) never calls it and shares no code with it.

What it computes (written from the definitions, not from any printed listing):

* Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V -- the left-hand side of the
  decomposition formula in the Ring-Attention blog's "理论奠基" (evolution / theory)
  section.  The right-hand side printed there sums separately normalised block
  softmaxes and is NOT an identity; this oracle does not use it.
* The row log-sum-exp LSE_i = ln sum_j exp(s_ij), natural log of the scaled scores, the
  quantity the same blog's "数值稳定性" (numerical stability) section carries between
  devices (m_i, l_i of FlashAttention's forward pass).
* Merge of partial results: given per-part (O_t, lse_t), lse = ln sum_t exp(lse_t) and
  O = sum_t exp(lse_t - lse) O_t.  This is the exact re-association Mesh-Attention relies
  on when a Q partition's keys are split over the tiles of one mesh row (Mesh-Attention
  tutorial, "从一维环到二维网" and the arXiv abstract: each GPU computes a 2D tile and
  the partial outputs go back to the Q owner).

Conventions (readings where the pages are silent):
* scale defaults to 1/sqrt(d);
* causal: key j is visible to query i iff j <= i (global token positions);
* GQA: query head h reads kv head h // (Hq // Hkv);
* a row with no visible key has O = 0 and lse = -inf.

Evaluation is a plain two-pass computation: pass 1 takes the row maximum of the masked
scaled scores, pass 2 sums exp(s - m) and exp(s - m) * v.  Keys are visited in chunks
only to bound memory; every chunk is an ordinary fp64 matrix product.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import torch

F64 = torch.float64


def _as64(x) -> torch.Tensor:
    t = torch.as_tensor(x)
    return t.to(device="cpu", dtype=F64)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def attention_rows(q, q_pos, k, v, scale: float, causal: bool, key_pos=None,
                   key_chunk: int = 4096) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention of query rows q [n, d] at global positions q_pos [n] over keys k [m, d]
    and values v [m, dv] at positions key_pos [m] (default 0..m-1).

    Returns (O [n, dv], lse [n]) in fp64.
    """
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    n, m = q.shape[0], k.shape[0]
    q_pos = torch.as_tensor(q_pos, dtype=torch.int64).reshape(n)
    key_pos = (torch.arange(m, dtype=torch.int64) if key_pos is None
               else torch.as_tensor(key_pos, dtype=torch.int64).reshape(m))
    neg_inf = torch.tensor(float("-inf"), dtype=F64)

    def scores(c0: int, c1: int) -> torch.Tensor:
        s = scale * (q @ k[c0:c1].T)
        if causal:
            visible = key_pos[c0:c1][None, :] <= q_pos[:, None]
            s = torch.where(visible, s, neg_inf)
        return s

    # pass 1: row maximum over the visible keys
    mx = torch.full((n,), float("-inf"), dtype=F64)
    for c0 in range(0, m, key_chunk):
        c1 = min(m, c0 + key_chunk)
        mx = torch.maximum(mx, scores(c0, c1).max(dim=1).values)
    empty = torch.isneginf(mx)
    shift = torch.where(empty, torch.zeros_like(mx), mx)

    # pass 2: sum of exp(s - m) and of exp(s - m) v
    ell = torch.zeros(n, dtype=F64)
    acc = torch.zeros(n, v.shape[1], dtype=F64)
    for c0 in range(0, m, key_chunk):
        c1 = min(m, c0 + key_chunk)
        e = torch.exp(scores(c0, c1) - shift[:, None])
        ell += e.sum(dim=1)
        acc += e @ v[c0:c1]

    lse = torch.where(empty, neg_inf, shift + torch.log(torch.where(empty, torch.ones_like(ell), ell)))
    out = torch.where(empty[:, None], torch.zeros_like(acc), acc / torch.where(empty, torch.ones_like(ell), ell)[:, None])
    return out, lse


def attention_bhsd(Q, K, V, causal: bool, scale: Optional[float] = None,
                   rows=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention for Q [B,Hq,S,d], K/V [B,Hkv,S,d] (any float dtype, upcast exactly).

    rows: None (all rows) or an int array [B, Hq, n] of query rows per head.
    Returns O [B,Hq,n,d] and LSE [B,Hq,n] in fp64.
    """
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    assert Hq % Hkv == 0
    g = Hq // Hkv
    scale = default_scale(d) if scale is None else scale
    n = S if rows is None else rows.shape[-1]
    O = torch.empty(B, Hq, n, V.shape[-1], dtype=F64)
    LSE = torch.empty(B, Hq, n, dtype=F64)
    for b in range(B):
        for kh in range(Hkv):
            k64 = _as64(K[b, kh])
            v64 = _as64(V[b, kh])
            for h in range(kh * g, (kh + 1) * g):
                pos = torch.arange(S) if rows is None else torch.as_tensor(rows[b, h], dtype=torch.int64)
                O[b, h], LSE[b, h] = attention_rows(_as64(Q[b, h])[pos], pos, k64, v64, scale, causal)
    return O, LSE


def merge(partials: Sequence[Tuple[torch.Tensor, torch.Tensor]]) -> Tuple[torch.Tensor, torch.Tensor]:
    """LSE merge of partial results [(O_t [n, d], lse_t [n]), ...] into (O [n, d], lse [n]).

    lse = M + ln sum_t exp(lse_t - M) with M = max_t lse_t; O = sum_t exp(lse_t - lse) O_t.
    Parts with lse_t = -inf carry weight 0; if every part is -inf the row is O = 0, lse = -inf.
    """
    if len(partials) == 0:
        raise ValueError("merge needs at least one partial")
    lses = torch.stack([_as64(l) for _, l in partials])  # [T, n]
    outs = torch.stack([_as64(o) for o, _ in partials])  # [T, n, d]
    M = lses.max(dim=0).values
    empty = torch.isneginf(M)
    Ms = torch.where(empty, torch.zeros_like(M), M)
    w = torch.exp(lses - Ms[None, :])  # exp(-inf) = 0 for empty parts
    tot = w.sum(dim=0)
    lse = torch.where(empty, M, Ms + torch.log(torch.where(empty, torch.ones_like(tot), tot)))
    wn = torch.where(empty[None, :], torch.zeros_like(w), w / torch.where(empty, torch.ones_like(tot), tot)[None, :])
    out = (wn[:, :, None] * outs).sum(dim=0)
    return out, lse


def split_attention(q, q_pos, k, v, scale: float, causal: bool,
                    key_parts: Iterable[Sequence[int]]) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention computed part by part over a split of the key indices, then merged.

    Each part is attended separately (attention_rows over that subset of keys, keeping
    their global positions) and the parts are combined with merge().  Equals
    attention_rows over all keys for any split -- the invariant tiled attention rests on.
    """
    k = _as64(k)
    v = _as64(v)
    parts = []
    for idx in key_parts:
        idx = torch.as_tensor(list(idx), dtype=torch.int64)
        parts.append(attention_rows(q, q_pos, k[idx], v[idx], scale, causal, key_pos=idx))
    return merge(parts)
