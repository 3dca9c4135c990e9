"""GPU parity of the backward pass: the C-ABI path (bwd_prep, tile_bwd, bwd_reduce, fed by the
C-ABI forward's O and LSE) against the fp64 backward oracle on the same seeded inputs, element
by element, plus every partial slot against the oracle's sums restricted to that slot."""
import math

import pytest
import torch

from mesh_inputs import WORKLOADS, Workload, make_do, make_qkv
from oracle import backward as OB
from tests.gpu_helpers import max_err

pytestmark = pytest.mark.gpu

# fp32: the fp32 tolerance of the forward (1e-4 absolute).  bf16: see BWD_TOL_BF16.
F32_CASES = [
    WORKLOADS["tiny_f32"],
    Workload(140, "f32_bwd_causal_ragged_L100", 1, 2, 1, 900, 128, "f32", True, 9),
    Workload(141, "f32_bwd_gqa_d64", 1, 4, 2, 512, 64, "f32", False, 4),
    Workload(142, "f32_bwd_batch2_causal", 2, 2, 2, 256, 64, "f32", True, 4),
]


def run_backward(lib, w, q, k, v, dO, plan=None):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    plan = plan or lib.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
    O, LSE = lib.mesh_attention(qd, kd, vd, w.P, w.causal, plan=plan)
    out = lib.mesh_attention_backward(qd, kd, vd, O, LSE, dod, w.P, w.causal, plan=plan, return_partials=True)
    torch.cuda.synchronize()
    return out, plan, LSE


def bwd_tol(w, ref):
    if w.dtype == "f32":
        return 1e-4
    return BWD_TOL_BF16(ref)


def BWD_TOL_BF16(ref):
    """bf16 gradients: products take bf16 P and dS, and dQ / dK / dV are rounded to bf16 at the
    end (half an ulp: 2^-9 of the value); absolute error <= 2^-7 of the largest gradient
    magnitude, and at least 2e-3."""
    return max(2e-3, ref.abs().max().item() * 2.0 ** -7)


def check_gradients(w, got, q, k, v, dO, tag=""):
    dQ, dK, dV = got[:3]
    rQ, rK, rV, _, _ = OB.attention_bwd_bhsd(q, k, v, dO, w.causal)
    for name, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        e = max_err(g, r)
        t = bwd_tol(w, r)
        print(f"[parity-bwd] {w.name}{tag} {name}: max|err| = {e:.3e} (tol {t:.3e}, max|ref| {r.abs().max().item():.3e})")
        assert e <= t, f"{w.name} {name}: {e:.3e} > {t:.3e}"


def check_backward_partials(lib, w, plan, got, q, k, v, dO, LSE):
    """Each dq partial slot against the oracle's dQ sum over that item's keys, each dk / dv slot
    against the oracle's sums over that KV slot's query rows (and the KV head's query heads),
    with the GPU forward's LSE and the oracle's D."""
    _, _, _, dq_p, dk_p, dv_p = got
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    L = plan.L
    n, m = plan.n_slots, plan.n_kv_slots
    dq_p = dq_p[: B * Hq * n * L * d].view(B, Hq, n, L, d).cpu()
    dk_p = dk_p[: B * Hkv * m * L * d].view(B, Hkv, m, L, d).cpu()
    dv_p = dv_p[: B * Hkv * m * L * d].view(B, Hkv, m, L, d).cpu()
    _, _, _, LSE64, D64 = OB.attention_bwd_bhsd(q, k, v, dO, w.causal)
    items, _, kvs = lib.mesh_attn_plan_order(plan)
    _, kv_items, kv_q = lib.mesh_attn_plan_kv_slots(plan)
    scale = 1.0 / math.sqrt(d)
    tol = 1e-4 if w.dtype == "f32" else None
    for b in range(B):
        for hk in range(Hkv):
            K64, V64 = k[b, hk].double(), v[b, hk].double()
            acc_k = {s: torch.zeros(L, d, dtype=torch.float64) for _, _, s in kv_items}
            acc_v = {s: torch.zeros(L, d, dtype=torch.float64) for _, _, s in kv_items}
            for h in range(hk * g, (hk + 1) * g):
                Q64, G64 = q[b, h].double(), dO[b, h].double()
                for (p, t, slot), kl in zip(items, kvs):
                    rows = torch.arange(p * L, (p + 1) * L)
                    keys = torch.cat([torch.arange(x * L, (x + 1) * L) for x in kl])
                    r, _, _ = OB.bwd_rows(Q64[rows], rows, K64[keys], V64[keys], G64[rows], LSE64[b, h, rows],
                                          D64[b, h, rows], scale, w.causal, key_pos=keys, want_kv=False)
                    t_ = tol or BWD_TOL_BF16(r)
                    assert max_err(dq_p[b, h, slot], r) <= t_, f"dq slot {slot} (p={p}, t={t})"
                for (kk, t, slot), ql in zip(kv_items, kv_q):
                    keys = torch.arange(kk * L, (kk + 1) * L)
                    rows = torch.cat([torch.arange(x * L, (x + 1) * L) for x in ql])
                    _, rk, rv = OB.bwd_rows(Q64[rows], rows, K64[keys], V64[keys], G64[rows], LSE64[b, h, rows],
                                            D64[b, h, rows], scale, w.causal, key_pos=keys)
                    acc_k[slot] += rk
                    acc_v[slot] += rv
            for (kk, t, slot) in kv_items:
                tk = tol or BWD_TOL_BF16(acc_k[slot])
                tv = tol or BWD_TOL_BF16(acc_v[slot])
                assert max_err(dk_p[b, hk, slot], acc_k[slot]) <= tk, f"dk slot {slot} (k={kk}, t={t})"
                assert max_err(dv_p[b, hk, slot], acc_v[slot]) <= tv, f"dv slot {slot} (k={kk}, t={t})"


@pytest.mark.parametrize("w", F32_CASES, ids=lambda w: w.name)
def test_backward_f32_against_oracle(lib, w):
    q, k, v = make_qkv(w)
    dO = make_do(w)
    got, plan, LSE = run_backward(lib, w, q, k, v, dO)
    assert got[0].dtype == torch.float32
    check_gradients(w, got, q, k, v, dO)
    check_backward_partials(lib, w, plan, got, q, k, v, dO, LSE)


def test_backward_f32_plan_variants(lib):
    """KVR, greedy and the ring plan change the tiles, slots and order, not the gradients."""
    w = F32_CASES[1]
    q, k, v = make_qkv(w)
    dO = make_do(w)
    for kvr, greedy in ((0, 0), (1, 0), (0, 1)):
        plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, kvr, greedy)
        got, plan, _ = run_backward(lib, w, q, k, v, dO, plan=plan)
        check_gradients(w, got, q, k, v, dO, tag=f" kvr={kvr} greedy={greedy}")
    ring = lib.mesh_attn_plan_create_ring(w.S, w.P, w.causal)
    got, plan, _ = run_backward(lib, w, q, k, v, dO, plan=ring)
    check_gradients(w, got, q, k, v, dO, tag=" ring")


def test_backward_f32_closed_form_constant_values(lib):
    """Constant V: dQ = dK = 0 (exactly, up to fp32 rounding of the cancelling terms)."""
    w = F32_CASES[2]
    q, k, v = make_qkv(w)
    v = torch.full_like(v, 0.5)
    dO = make_do(w)
    got, _, _ = run_backward(lib, w, q, k, v, dO)
    assert got[0].abs().max().item() <= 1e-5 and got[1].abs().max().item() <= 1e-5
