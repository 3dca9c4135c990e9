"""GPU parity of the backward pass: the C-ABI path (bwd_prep, tile_bwd, bwd_reduce, fed by the
C-ABI forward's O and LSE) against the fp64 backward oracle on the same seeded inputs, element
by element, plus every partial slot against the oracle's sums restricted to that slot."""
import math

import pytest
import torch

from mesh_inputs import WORKLOADS, Workload, make_do, make_qkv
from oracle import backward as OB
from tests.gpu_helpers import bf16_grad_bound


pytestmark = pytest.mark.gpu

# fp32: the fp32 tolerance of the forward (1e-4 absolute).  bf16: bf16_grad_bound, elementwise.
F32_CASES = [
    WORKLOADS["tiny_f32"],
    Workload(140, "f32_bwd_causal_ragged_L100", 1, 2, 1, 900, 128, "f32", True, 9),
    Workload(141, "f32_bwd_gqa_d64", 1, 4, 2, 512, 64, "f32", False, 4),
    Workload(142, "f32_bwd_batch2_causal", 2, 2, 2, 256, 64, "f32", True, 4),
]


BF16_CASES = [
    Workload(150, "bf16_bwd_causal_L1024", 1, 2, 2, 4096, 128, "bf16", True, 4),
    Workload(151, "bf16_bwd_gqa_noncausal", 1, 4, 2, 2048, 128, "bf16", False, 4),
    Workload(152, "bf16_bwd_ragged_L200_causal", 1, 2, 1, 800, 128, "bf16", True, 4),
    Workload(153, "bf16_bwd_d64_P9", 1, 2, 2, 3456, 64, "bf16", True, 9),
    Workload(154, "bf16_bwd_batch2_ragged_d64", 2, 2, 1, 900, 64, "bf16", False, 9),
    Workload(155, "bf16_bwd_single_partition", 1, 2, 1, 640, 128, "bf16", True, 1),
    Workload(156, "bf16_bwd_peaked_k4", 1, 2, 1, 2048, 128, "bf16", True, 16, k_scale=4.0),
]


def run_backward(lib, w, q, k, v, dO, plan=None):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    plan = plan or lib.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
    O, LSE = lib.mesh_attention(qd, kd, vd, w.P, w.causal, plan=plan)
    out = lib.mesh_attention_backward(qd, kd, vd, O, LSE, dod, w.P, w.causal, plan=plan, return_partials=True)
    torch.cuda.synchronize()
    return out, plan, LSE


def n_terms(w, grad: str) -> int:
    """Most products one gradient element sums: the keys of a query row (dQ), the query rows of
    every head of the group (dK, dV)."""
    return w.S if grad == "dQ" else w.S * (w.Hq // w.Hkv)


def compare(w, got, ref, mag, n):
    """(max |err|, max err / bound) of one gradient tensor."""
    e = (got.double().cpu() - ref).abs()
    if w.dtype == "f32":
        return e.max().item(), e.max().item() / 1e-4
    return e.max().item(), (e / bf16_grad_bound(ref, mag, n)).max().item()


def check_gradients(w, got, q, k, v, dO, tag=""):
    dQ, dK, dV = got[:3]
    rQ, rK, rV, _, _ = OB.attention_bwd_bhsd(q, k, v, dO, w.causal)
    mags = OB.attention_bwd_bhsd(q, k, v, dO, w.causal, absolute=True)[:3] if w.dtype == "bf16" else (None,) * 3
    for name, g, r, m in (("dQ", dQ, rQ, mags[0]), ("dK", dK, rK, mags[1]), ("dV", dV, rV, mags[2])):
        e, ratio = compare(w, g, r, m, n_terms(w, name))
        print(f"[parity-bwd] {w.name}{tag} {name}: max|err| = {e:.3e}, max err/bound = {ratio:.3f} "
              f"(max|ref| {r.abs().max().item():.3e})")
        assert ratio <= 1.0, f"{w.name} {name}: error {ratio:.3f}x the bound"


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
    DM64 = OB.attention_bwd_bhsd(q, k, v, dO, w.causal, absolute=True)[4] if w.dtype == "bf16" else None
    items, _, kvs = lib.mesh_attn_plan_order(plan)
    _, kv_items, kv_q = lib.mesh_attn_plan_kv_slots(plan)
    scale = 1.0 / math.sqrt(d)
    bf = w.dtype == "bf16"

    def ok(got_, ref_, mag_, n):
        e = (got_.double() - ref_).abs()
        return bool((e <= (bf16_grad_bound(ref_, mag_, n) if bf else 1e-4)).all())

    for b in range(B):
        for hk in range(Hkv):
            K64, V64 = k[b, hk].double(), v[b, hk].double()
            acc_k = {s: torch.zeros(L, d, dtype=torch.float64) for _, _, s in kv_items}
            acc_v = {s: torch.zeros(L, d, dtype=torch.float64) for _, _, s in kv_items}
            mag_k = {s: torch.zeros(L, d, dtype=torch.float64) for _, _, s in kv_items}
            mag_v = {s: torch.zeros(L, d, dtype=torch.float64) for _, _, s in kv_items}
            for h in range(hk * g, (hk + 1) * g):
                Q64, G64 = q[b, h].double(), dO[b, h].double()
                for (p, t, slot), kl in zip(items, kvs):
                    rows = torch.arange(p * L, (p + 1) * L)
                    keys = torch.cat([torch.arange(x * L, (x + 1) * L) for x in kl])
                    args = (Q64[rows], rows, K64[keys], V64[keys], G64[rows], LSE64[b, h, rows], D64[b, h, rows],
                            scale, w.causal)
                    r, _, _ = OB.bwd_rows(*args, key_pos=keys, want_kv=False)
                    m = OB.bwd_rows(*args, key_pos=keys, want_kv=False, absolute=True,
                                    dmag=DM64[b, h, rows])[0] if bf else None
                    assert ok(dq_p[b, h, slot], r, m, n_terms(w, "dQ")), f"dq slot {slot} (p={p}, t={t})"
                for (kk, t, slot), ql in zip(kv_items, kv_q):
                    keys = torch.arange(kk * L, (kk + 1) * L)
                    rows = torch.cat([torch.arange(x * L, (x + 1) * L) for x in ql])
                    args = (Q64[rows], rows, K64[keys], V64[keys], G64[rows], LSE64[b, h, rows], D64[b, h, rows],
                            scale, w.causal)
                    _, rk, rv = OB.bwd_rows(*args, key_pos=keys)
                    acc_k[slot] += rk
                    acc_v[slot] += rv
                    if bf:
                        _, mk, mv = OB.bwd_rows(*args, key_pos=keys, absolute=True, dmag=DM64[b, h, rows])
                        mag_k[slot] += mk
                        mag_v[slot] += mv
            nk = n_terms(w, "dK")
            for (kk, t, slot) in kv_items:
                assert ok(dk_p[b, hk, slot], acc_k[slot], mag_k[slot], nk), f"dk slot {slot} (k={kk}, t={t})"
                assert ok(dv_p[b, hk, slot], acc_v[slot], mag_v[slot], nk), f"dv slot {slot} (k={kk}, t={t})"


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


@pytest.mark.parametrize("w", BF16_CASES, ids=lambda w: w.name)
def test_backward_bf16_against_oracle(lib, w):
    q, k, v = make_qkv(w)
    dO = make_do(w)
    got, plan, LSE = run_backward(lib, w, q, k, v, dO)
    assert got[0].dtype == torch.bfloat16
    check_gradients(w, got, q, k, v, dO)
    if w.S <= 2048:
        check_backward_partials(lib, w, plan, got, q, k, v, dO, LSE)


def test_backward_bf16_plan_variants(lib):
    w = BF16_CASES[2]
    q, k, v = make_qkv(w)
    dO = make_do(w)
    for kvr, greedy in ((0, 0), (0, 1)):
        plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, kvr, greedy)
        got, _, _ = run_backward(lib, w, q, k, v, dO, plan=plan)
        check_gradients(w, got, q, k, v, dO, tag=f" kvr={kvr} greedy={greedy}")
    got, _, _ = run_backward(lib, w, q, k, v, dO, plan=lib.mesh_attn_plan_create_ring(w.S, w.P, w.causal))
    check_gradients(w, got, q, k, v, dO, tag=" ring")


def test_backward_bf16_several_units_per_cta(lib):
    """A mid-size case whose persistent backward kernels take several units per CTA: with
    P = 16 partitions of 512 tokens and 4 heads the dK/dV kernel has 640 units and the dQ kernel
    928, against one CTA per SM.  So the cross-unit code (the next unit's resident loads, the
    drain and overwrite barriers, barrier phases counted over a CTA's whole sequence of blocks)
    runs under an elementwise check of dQ, dK and dV and of every partial slot."""
    w = Workload(157, "bf16_bwd_multi_unit", 1, 4, 4, 8192, 128, "bf16", True, 16)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v = make_qkv(w)
    dO = make_do(w)
    got, plan, LSE = run_backward(lib, w, q, k, v, dO)
    blocks = plan.L // 128
    units_dkdv = plan.n_kv_slots * w.B * w.Hkv * blocks
    units_dq = plan.n_slots * w.B * w.Hq * blocks
    print(f"[parity-bwd] {w.name}: {units_dkdv} dK/dV units, {units_dq} dQ units, {sms} SMs")
    assert units_dkdv >= 4 * sms and units_dq >= 6 * sms
    check_gradients(w, got, q, k, v, dO)
    check_backward_partials(lib, w, plan, got, q, k, v, dO, LSE)


@pytest.mark.parametrize("name", ["bf16_causal_16k", "gqa_causal_64k"])
def test_backward_full_size(lib, name):
    """Full-size workloads (the forward's bench configurations), elementwise on seeded samples:
    dQ on sampled query rows (each needs only its own forward row), and on the bf16 causal 16K
    workload dK and dV on sampled key rows of two KV heads (each sums over every query row that
    sees it, so the oracle runs the forward of all rows of those heads), all against the derived
    bound.  Besides, two identities that hold at any size for every KV head and column:
    sum_j dK_j = scale sum_i q_i sum_j dS_ij = 0 and sum_j dV_j = sum_i dO_i (rows of P sum to 1),
    each within 2^-7 of the sum of the terms' magnitudes."""
    import numpy as np
    from mesh_inputs import forced_rows
    w = WORKLOADS[name]
    q, k, v = make_qkv(w)
    dO = make_do(w)
    got, plan, _ = run_backward(lib, w, q, k, v, dO)
    dQ, dK, dV = (t.double().cpu() for t in got[:3])
    del got
    g = w.Hq // w.Hkv
    dk_sum = dK.sum(dim=2)
    dk_abs = dK.abs().sum(dim=2)
    assert (dk_sum.abs() <= 2.0 ** -7 * dk_abs + 1e-3).all(), (dk_sum.abs() / dk_abs).max().item()
    dv_sum = dV.sum(dim=2)
    want = dO.double().view(w.B, w.Hkv, g, w.S, w.d).sum(dim=(2, 3))
    dv_abs = dV.abs().sum(dim=2)
    assert ((dv_sum - want).abs() <= 2.0 ** -7 * dv_abs + 1e-3).all()
    rng = np.random.default_rng(w.cfg_id)
    forced = np.array(forced_rows(w.S, w.P))
    pool = np.setdiff1d(np.arange(w.S), forced)

    def draw(n):
        return np.sort(np.concatenate([forced, rng.choice(pool, n - len(forced), replace=False)]))

    rows = np.stack([np.stack([draw(24) for _ in range(w.Hq)]) for _ in range(w.B)])
    ref, mag = OB.dq_rows(q, k, v, dO, w.causal, rows, absolute=True)
    got_rows = torch.stack([torch.stack([dQ[b, h, torch.as_tensor(rows[b, h])] for h in range(w.Hq)])
                            for b in range(w.B)])
    r = ((got_rows - ref).abs() / bf16_grad_bound(ref, mag, n_terms(w, "dQ"))).max().item()
    print(f"[parity-bwd] {name} sampled dQ rows: max|err| = {(got_rows - ref).abs().max().item():.3e}, "
          f"max err/bound = {r:.3f}")
    assert r <= 1.0
    if name != "bf16_causal_16k":
        return
    for hk in (0, w.Hkv - 5):
        keys = draw(32)
        rk, rv, mk, mv = OB.dkdv_keys(q, k, v, dO, w.causal, 0, hk, keys)
        idx = torch.as_tensor(keys)
        for nm, got_k, ref_k, mag_k in (("dK", dK[0, hk, idx], rk, mk), ("dV", dV[0, hk, idx], rv, mv)):
            e = (got_k - ref_k).abs()
            r = (e / bf16_grad_bound(ref_k, mag_k, n_terms(w, nm))).max().item()
            print(f"[parity-bwd] {name} KV head {hk} sampled {nm} rows: max|err| = {e.max().item():.3e}, "
                  f"max err/bound = {r:.3f}")
            assert r <= 1.0, f"{nm} of KV head {hk}: {r:.3f}x the bound"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 3, 37), (2, 5, 301)], ids=["one_row", "rows111", "rows3010"])
def test_prep_row_sums(lib, dtype, d, shape):
    """D_i = dO_i . O_i from the prep call against the fp64 sum over the same stored values, for
    row counts that leave every CTA shape ragged.  fp32 accumulation of d products: within
    d 2^-24 sum |dO O| (taken as 1e-5 sum |dO O| + 1e-7)."""
    B, H, S = shape
    g = torch.Generator().manual_seed(7000 + d + S)
    O = torch.randn(B, H, S, d, generator=g).to(dtype)
    dO = torch.randn(B, H, S, d, generator=g).to(dtype)
    D = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    lib.mesh_attn_bwd_prep(O.cuda(), dO.cuda(), D, status)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    prod = O.double() * dO.double()
    ref = prod.sum(dim=-1)
    tol = 1e-5 * prod.abs().sum(dim=-1) + 1e-7
    err = (D.double().cpu() - ref).abs()
    assert torch.isfinite(D).all()
    assert (err <= tol).all(), err.max().item()
