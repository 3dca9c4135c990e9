"""Shared helpers of the GPU parity tests: run the C-ABI path and the fp64 oracle on the same
seeded inputs and compare element by element."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import attention as OA

# tolerances of the comparison against the fp64 oracle (max absolute error)
TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 1e-3)}

# unit roundoff of bf16: 8 significant bits, round to nearest even
U_BF16 = 2.0 ** -8


def bf16_grad_bound(ref, mag, n_terms: int):
    """Elementwise error bound of a gradient computed from bf16 inputs, derived term by term from
    the arithmetic of the tile backward (ref: the fp64 oracle's gradient, mag: the oracle's
    magnitude sums for it, n_terms: the most products one element sums).

    * u |ref|: the result is rounded to bf16 once.
    * u mag: the products take P (dV) and dS (dQ, dK) rounded to bf16 once, and D from the
      forward's bf16 O; mag carries exactly these terms (scale sum (|dS| + dmag P) |k| for dQ,
      the transposed sum for dK, sum P |dO| for dV).
    * 2^-9 mag: P is recomputed from the forward's LSE, which is within 1e-3 of the exact one
      (the forward's LSE tolerance), so P is off by a relative 1e-3; the fp32 recomputation of
      the scores and of dP over d <= 128 exact bf16 products adds under 2^-16 relative.
    * n 2^-23 mag: fp32 accumulation of n terms, worst case with adders that truncate (one ulp,
      2^-23 relative, per addition).
    Plus 1e-6 absolute for elements whose terms all cancel."""
    return U_BF16 * ref.abs() + (U_BF16 + 2.0 ** -9 + n_terms * 2.0 ** -23) * mag + 1e-6


def run_gpu(lib, w, q, k, v, kvr=None, greedy=None):
    """Whole path through the binding; returns device tensors O, LSE, partial O, partial LSE and the plan."""
    plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr if kvr is None else kvr,
                                     w.greedy if greedy is None else greedy)
    O, LSE, po, pl = lib.mesh_attention(q.cuda(), k.cuda(), v.cuda(), w.P, w.causal, plan=plan,
                                        return_partials=True)
    torch.cuda.synchronize()
    return O, LSE, po, pl, plan


def max_err(a: torch.Tensor, b: torch.Tensor) -> float:
    a = a.double().cpu()
    b = b.double().cpu()
    fa, fb = torch.isfinite(a), torch.isfinite(b)
    assert torch.equal(fa, fb), "non-finite pattern differs"
    if not fa.any():
        return 0.0
    assert torch.equal(a[~fa], b[~fb]), "infinities differ"
    return (a[fa] - b[fb]).abs().max().item()


def check_full(w, O, LSE, q, k, v):
    Or, Lr = OA.attention_bhsd(q, k, v, w.causal)
    to, tl = TOL[w.dtype]
    eo, el = max_err(O, Or), max_err(LSE, Lr)
    print(f"[parity] {w.name}: max|dO| = {eo:.3e} (tol {to}), max|dLSE| = {el:.3e} (tol {tl})")
    assert eo <= to and el <= tl, f"{w.name}: max|dO| = {eo:.3e} (tol {to}), max|dLSE| = {el:.3e} (tol {tl})"
    return eo, el


def check_partials(lib, w, plan, po, pl, q, k, v):
    """Every slot's partial O_t and lse_t against attention over that tile's keys."""
    B, Hq, S, d = q.shape
    g = Hq // k.shape[1]
    n = plan.n_slots
    L = plan.L
    po = po[: B * Hq * n * L * d].view(B, Hq, n, L, d).cpu()
    pl = pl[: B * Hq * n * L].view(B, Hq, n, L).cpu()
    items, _, kvs = lib.mesh_attn_plan_order(plan)
    to, tl = TOL[w.dtype]
    scale = 1.0 / math.sqrt(d)
    worst = (0.0, 0.0)
    for b in range(B):
        for h in range(Hq):
            k64, v64 = OA._as64(k[b, h // g]), OA._as64(v[b, h // g])
            q64 = OA._as64(q[b, h])
            for (p, t, slot), kl in zip(items, kvs):
                rows = torch.arange(p * L, (p + 1) * L)
                keys = torch.cat([torch.arange(x * L, (x + 1) * L) for x in kl])
                Or, Lr = OA.attention_rows(q64[rows], rows, k64[keys], v64[keys], scale, w.causal, key_pos=keys)
                eo, el = max_err(po[b, h, slot], Or), max_err(pl[b, h, slot], Lr)
                assert eo <= to and el <= tl, f"slot {slot} (p={p}, t={t}) b={b} h={h}: {eo:.3e} {el:.3e}"
                worst = (max(worst[0], eo), max(worst[1], el))
    return worst


def check_sampled(w, O, LSE, q, k, v, rows: np.ndarray):
    """O and LSE on seeded sampled rows per head against the oracle computed on those rows."""
    Or, Lr = OA.attention_bhsd(q, k, v, w.causal, rows=rows)
    idx = torch.as_tensor(rows)
    Og = torch.stack([torch.stack([O[b, h].cpu()[idx[b, h]] for h in range(w.Hq)]) for b in range(w.B)])
    Lg = torch.stack([torch.stack([LSE[b, h].cpu()[idx[b, h]] for h in range(w.Hq)]) for b in range(w.B)])
    to, tl = TOL[w.dtype]
    eo, el = max_err(Og, Or), max_err(Lg, Lr)
    print(f"[parity] {w.name} (sampled rows): max|dO| = {eo:.3e} (tol {to}), max|dLSE| = {el:.3e} (tol {tl})")
    assert eo <= to and el <= tl, f"{w.name}: max|dO| = {eo:.3e} (tol {to}), max|dLSE| = {el:.3e} (tol {tl})"
    return eo, el
