"""fp64 CPU oracle of the attention backward pass and of its per-tile partial sums.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module; the product path never calls it.

The pages describe the forward pass only.  Mesh-Attention targets training (the tutorial's
end-to-end training speedups and its closing remarks on large-model training), so the
backward pass follows the forward's tile structure: each tile produces partial gradients over
its own (query, key) blocks, dQ partials are summed along the mesh row (like the forward's
partial outputs) and dK / dV partials along the mesh column.

What it computes is the derivative of the forward definition (the left-hand side of the
Ring-Attention blog's "理论奠基" formula, softmax(Q K^T / sqrt(d_k)) V), by the chain rule:
with s_ij = scale q_i . k_j over the visible keys, P_ij = exp(s_ij - LSE_i),
O_i = sum_j P_ij v_j and an upstream gradient dO,

    dV_j  = sum_i P_ij dO_i
    dP_ij = dO_i . v_j
    D_i   = sum_j P_ij dP_ij  (= dO_i . O_i)
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = scale sum_j dS_ij k_j
    dK_j  = scale sum_i dS_ij q_i

Grouped-query attention: a key / value head receives the sum over its query heads.  The
per-tile partials are the same sums restricted to the tile's keys (dQ) or to the tile's query
rows (dK, dV), with the global LSE_i and D_i; summed over the tiles they give the full
gradients exactly.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from oracle.attention import F64, _as64, attention_bhsd, attention_rows, default_scale


def bwd_rows(q, q_pos, k, v, do, lse, dsum, scale: float, causal: bool, key_pos=None,
             key_chunk: int = 4096, want_kv: bool = True, absolute: bool = False,
             dmag=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Gradient sums over the (row, key) pairs of query rows q [n, d] (global positions q_pos,
    global LSE lse [n], D = dO . O dsum [n], upstream gradient do [n, dv]) and keys k [m, d],
    v [m, dv] at positions key_pos (default 0..m-1).  want_kv=False skips dk and dv (returned as
    zeros).  absolute=True returns instead the magnitudes that scale the rounding error of a
    computation that rounds dS and P to a short format and takes D from a rounded O:
    scale sum_j (|dS_ij| + dmag_i P_ij) |k_j|, scale sum_i (|dS_ij| + dmag_i P_ij) |q_i| and
    sum_i P_ij |dO_i| (elementwise absolute values), with dmag [n] the rows' magnitude of D
    (see attention_bwd_bhsd).

    Returns (dq [n, d], dk [m, d], dv [m, dv]) in fp64: dq_i = scale sum_j dS_ij k_j over these
    keys, dk_j = scale sum_i dS_ij q_i and dv_j = sum_i P_ij dO_i over these rows.  Rows with
    lse = -inf (no visible key anywhere) contribute nothing.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    lse, dsum = _as64(lse), _as64(dsum)
    n, m = q.shape[0], k.shape[0]
    q_pos = torch.as_tensor(q_pos, dtype=torch.int64).reshape(n)
    key_pos = (torch.arange(m, dtype=torch.int64) if key_pos is None
               else torch.as_tensor(key_pos, dtype=torch.int64).reshape(m))
    live = ~torch.isneginf(lse)
    lse_s = torch.where(live, lse, torch.zeros_like(lse))
    dq = torch.zeros(n, q.shape[1], dtype=F64)
    dk = torch.zeros(m, k.shape[1], dtype=F64)
    dv = torch.zeros(m, v.shape[1], dtype=F64)
    for c0 in range(0, m, key_chunk):
        c1 = min(m, c0 + key_chunk)
        s = scale * (q @ k[c0:c1].T)
        p = torch.exp(s - lse_s[:, None])
        visible = live[:, None].expand(n, c1 - c0)
        if causal:
            visible = visible & (key_pos[c0:c1][None, :] <= q_pos[:, None])
        p = torch.where(visible, p, torch.zeros_like(p))
        dp = do @ v[c0:c1].T
        ds = p * (dp - dsum[:, None])
        kc, qq, dd = k[c0:c1], q, do
        if absolute:
            ds = ds.abs() + (0.0 if dmag is None else _as64(dmag)[:, None] * p)
            kc, qq, dd = kc.abs(), q.abs(), do.abs()
        dq += scale * (ds @ kc)
        if want_kv:
            dk[c0:c1] = scale * (ds.T @ qq)
            dv[c0:c1] = p.T @ dd
    return dq, dk, dv


def attention_bwd_bhsd(Q, K, V, dO, causal: bool, scale: Optional[float] = None, absolute: bool = False):
    """Full backward for Q [B,Hq,S,d], K/V [B,Hkv,S,d], dO [B,Hq,S,d] (any float dtype, upcast
    exactly).  The forward quantities O, LSE come from the forward oracle.  absolute=True gives
    the magnitude sums of bwd_rows in place of dQ, dK, dV, and in place of D the rows' magnitude
    of D, dmag_i = sum_e |dO_ie| (|O_ie| + sum_j P_ij |v_je|): a rounding of O by a relative u
    (plus a rounding of P by u inside O) moves D_i by at most u dmag_i.

    Returns dQ [B,Hq,S,d], dK, dV [B,Hkv,S,d], LSE [B,Hq,S] and D [B,Hq,S], all fp64.
    """
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    scale = default_scale(d) if scale is None else scale
    O, LSE = attention_bhsd(Q, K, V, causal, scale)
    D = (_as64(dO) * O).sum(dim=-1)
    if absolute:
        O_abs, _ = attention_bhsd(Q, K, _as64(V).abs(), causal, scale)
        D = (_as64(dO).abs() * (O.abs() + O_abs)).sum(dim=-1)
    dQ = torch.zeros(B, Hq, S, d, dtype=F64)
    dK = torch.zeros(B, Hkv, S, d, dtype=F64)
    dV = torch.zeros(B, Hkv, S, V.shape[-1], dtype=F64)
    pos = torch.arange(S)
    for b in range(B):
        for kh in range(Hkv):
            k64, v64 = _as64(K[b, kh]), _as64(V[b, kh])
            for h in range(kh * g, (kh + 1) * g):
                dsum = (_as64(dO[b, h]) * O[b, h]).sum(dim=-1)
                dq, dk, dv = bwd_rows(_as64(Q[b, h]), pos, k64, v64, _as64(dO[b, h]), LSE[b, h], dsum,
                                      scale, causal, absolute=absolute, dmag=D[b, h] if absolute else None)
                dQ[b, h] = dq
                dK[b, kh] += dk
                dV[b, kh] += dv
    return dQ, dK, dV, LSE, D


def _forward_with_magnitude(q, pos, k64, v64, do, scale: float, causal: bool):
    """Forward of rows q at positions pos with values [v, |v|] in one pass: LSE, D = dO . O and
    the rows' magnitude of D, dmag = sum_e |dO_e| (|O_e| + sum_j P_j |v_je|)."""
    dv = v64.shape[1]
    o2, lse = attention_rows(q, pos, k64, torch.cat([v64, v64.abs()], dim=1), scale, causal)
    o, o_abs = o2[:, :dv], o2[:, dv:]
    return lse, (do * o).sum(dim=-1), (do.abs() * (o.abs() + o_abs)).sum(dim=-1)


def dq_rows(Q, K, V, dO, causal: bool, rows, scale: Optional[float] = None, absolute: bool = False):
    """dQ on sampled query rows only: rows is an int array [B, Hq, n].  Each row needs only its
    own forward (LSE_i, O_i, hence D_i) and all keys.  Returns dQ [B, Hq, n, d] in fp64; with
    absolute=True also the rows' magnitude sums of bwd_rows (a second tensor of the same shape)."""
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    scale = default_scale(d) if scale is None else scale
    out = torch.empty(B, Hq, rows.shape[-1], d, dtype=F64)
    mag = torch.empty_like(out) if absolute else None
    for b in range(B):
        for kh in range(Hkv):
            k64, v64 = _as64(K[b, kh]), _as64(V[b, kh])
            for h in range(kh * g, (kh + 1) * g):
                pos = torch.as_tensor(rows[b, h], dtype=torch.int64)
                q = _as64(Q[b, h])[pos]
                do = _as64(dO[b, h])[pos]
                lse, dsum, dmag = _forward_with_magnitude(q, pos, k64, v64, do, scale, causal)
                out[b, h], _, _ = bwd_rows(q, pos, k64, v64, do, lse, dsum, scale, causal, want_kv=False)
                if absolute:
                    mag[b, h], _, _ = bwd_rows(q, pos, k64, v64, do, lse, dsum, scale, causal, want_kv=False,
                                               absolute=True, dmag=dmag)
    return (out, mag) if absolute else out


def dkdv_keys(Q, K, V, dO, causal: bool, b: int, kh: int, keys, scale: Optional[float] = None,
              row_chunk: int = 4096):
    """dK and dV of KV head kh (batch b) on the sampled key rows `keys` (global positions), with
    the magnitude sums of bwd_rows.  A key's gradient sums over every query row that sees it, in
    every query head of the group, so this needs the forward (LSE_i, D_i, dmag_i) of all rows
    of those heads.  Returns (dk, dv, dk_mag, dv_mag), each [n_keys, d] in fp64."""
    B, Hq, S, d = Q.shape
    g = Hq // K.shape[1]
    scale = default_scale(d) if scale is None else scale
    keys = torch.as_tensor(keys, dtype=torch.int64)
    k64, v64 = _as64(K[b, kh]), _as64(V[b, kh])
    ks, vs = k64[keys], v64[keys]
    dk = torch.zeros(len(keys), d, dtype=F64)
    dv = torch.zeros(len(keys), V.shape[-1], dtype=F64)
    dk_mag, dv_mag = torch.zeros_like(dk), torch.zeros_like(dv)
    for h in range(kh * g, (kh + 1) * g):
        for r0 in range(0, S, row_chunk):
            pos = torch.arange(r0, min(S, r0 + row_chunk))
            q = _as64(Q[b, h])[pos]
            do = _as64(dO[b, h])[pos]
            lse, dsum, dmag = _forward_with_magnitude(q, pos, k64, v64, do, scale, causal)
            _, a, c = bwd_rows(q, pos, ks, vs, do, lse, dsum, scale, causal, key_pos=keys)
            dk += a
            dv += c
            _, a, c = bwd_rows(q, pos, ks, vs, do, lse, dsum, scale, causal, key_pos=keys, absolute=True,
                               dmag=dmag)
            dk_mag += a
            dv_mag += c
    return dk, dv, dk_mag, dv_mag
