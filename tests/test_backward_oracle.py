"""Pins of the backward-pass oracle against things other than itself: central finite differences
of the forward oracle (the gradient is the derivative of <O, dO>), closed forms (constant V,
causal row 0, a single key), exact identities of the softmax gradient, PyTorch autograd on a
plain fp64 attention, and the tile decomposition of the partial gradients."""
import math

import pytest
import torch

from oracle import attention as OA
from oracle import backward as OB
from oracle import planner as PL

F64 = torch.float64


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * scale


def _case(B, Hq, Hkv, S, d, seed):
    return (_rand((B, Hq, S, d), seed), _rand((B, Hkv, S, d), seed + 1), _rand((B, Hkv, S, d), seed + 2),
            _rand((B, Hq, S, d), seed + 3))


def _loss(Q, K, V, dO, causal):
    O, _ = OA.attention_bhsd(Q, K, V, causal)
    return float((O * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_finite_differences(causal, Hq, Hkv):
    """<dX, U> equals d/de <O(X + eU), dO> for X in (Q, K, V) and random directions U."""
    Q, K, V, dO = _case(1, Hq, Hkv, 13, 8, 11 + Hq)
    dQ, dK, dV, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
    eps = 1e-5
    for which, grad in (("q", dQ), ("k", dK), ("v", dV)):
        base = {"q": Q, "k": K, "v": V}[which]
        U = _rand(base.shape, 99)
        args_p = {"q": Q, "k": K, "v": V}
        args_m = dict(args_p)
        args_p[which] = base + eps * U
        args_m[which] = base - eps * U
        fd = (_loss(args_p["q"], args_p["k"], args_p["v"], dO, causal)
              - _loss(args_m["q"], args_m["k"], args_m["v"], dO, causal)) / (2 * eps)
        an = float((grad * U).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (which, fd, an)


def test_constant_values_give_zero_q_and_k_gradients():
    """V rows all equal c: O = c for every row whatever P is, so dQ = dK = 0 and
    dV_j = sum_i P_ij dO_i (whose sum over j is sum_i dO_i)."""
    Q, K, V, dO = _case(1, 2, 1, 20, 8, 5)
    V = torch.full_like(V, 0.75)
    for causal in (False, True):
        dQ, dK, dV, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
        assert dQ.abs().max() < 1e-13 and dK.abs().max() < 1e-13
        assert torch.allclose(dV.sum(dim=2), dO.sum(dim=(1, 2))[:, None], atol=1e-12)


def test_causal_row_zero_and_single_key():
    """Causal row 0 sees only key 0: P_00 = 1, so dS_00 = dO_0.v_0 - dO_0.O_0 = 0 and dQ_0 = 0.
    With S = 1 every gradient but dV vanishes and dV = sum over heads of dO."""
    Q, K, V, dO = _case(1, 2, 1, 9, 8, 7)
    dQ, _, _, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, True)
    assert dQ[:, :, 0].abs().max() < 1e-14
    Q1, K1, V1, dO1 = _case(1, 2, 1, 1, 8, 8)
    dQ, dK, dV, _, _ = OB.attention_bwd_bhsd(Q1, K1, V1, dO1, False)
    assert dQ.abs().max() < 1e-14 and dK.abs().max() < 1e-14
    assert torch.allclose(dV[0, 0], dO1[0].sum(dim=0), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(causal):
    """sum_j dS_ij = D_i - D_i = 0, hence sum_j dK_j = 0; rows of P sum to 1, hence
    sum_j dV_j = sum over the group's heads and rows of dO."""
    Q, K, V, dO = _case(2, 4, 2, 24, 16, 21)
    _, dK, dV, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
    assert dK.sum(dim=2).abs().max() < 1e-11
    want = dO.view(2, 2, 2, 24, 16).sum(dim=(2, 3))
    assert torch.allclose(dV.sum(dim=2), want, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_against_autograd(causal):
    """PyTorch autograd through a plain fp64 softmax attention gives the same gradients."""
    Q, K, V, dO = _case(1, 4, 2, 17, 8, 31)
    g = 2
    q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
    kk = k.repeat_interleave(g, dim=1)
    vv = v.repeat_interleave(g, dim=1)
    s = (q @ kk.transpose(-1, -2)) / math.sqrt(8)
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(17, 17, dtype=torch.bool), 1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ vv
    (o * dO).sum().backward()
    dQ, dK, dV, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
    assert torch.allclose(dQ, q.grad, atol=1e-12)
    assert torch.allclose(dK, k.grad, atol=1e-12)
    assert torch.allclose(dV, v.grad, atol=1e-12)


def test_dq_rows_matches_full():
    Q, K, V, dO = _case(1, 4, 2, 40, 8, 41)
    import numpy as np
    rows = np.array([[[0, 5, 39], [1, 2, 3], [39, 20, 10], [7, 8, 9]]])
    for causal in (False, True):
        dQ, *_ = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
        got = OB.dq_rows(Q, K, V, dO, causal, rows)
        for h in range(4):
            assert torch.allclose(got[0, h], dQ[0, h, torch.as_tensor(rows[0, h])], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kvr", [False, True])
def test_tile_partials_sum_to_full(causal, kvr):
    """Per-tile partial gradients, restricted to each tile's (Q partition, KV partition) blocks
    with the global LSE and D, summed over the tiles of a mesh row (dQ) or column (dK, dV) give
    the full gradients."""
    P, L, d = 4, 6, 8
    S = P * L
    Q, K, V, dO = _case(1, 2, 2, S, d, 51)
    dQ, dK, dV, LSE, D = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
    plan = PL.make_plan(S, P, causal, kvr, True)
    ks = PL.kv_slots(plan)
    scale = 1.0 / math.sqrt(d)
    acc_q = torch.zeros_like(dQ)
    acc_k = torch.zeros_like(dK)
    acc_v = torch.zeros_like(dV)
    for h in range(2):
        for (p, t, slot), kl in zip(plan.items, plan.item_kv):
            rows = torch.arange(p * L, (p + 1) * L)
            keys = torch.cat([torch.arange(k * L, (k + 1) * L) for k in kl])
            dq, _, _ = OB.bwd_rows(Q[0, h, rows], rows, K[0, h, keys], V[0, h, keys], dO[0, h, rows],
                                   LSE[0, h, rows], D[0, h, rows], scale, causal, key_pos=keys)
            acc_q[0, h, rows] += dq
        for (k, t, slot), ql in zip(ks.kv_items, ks.kv_item_q):
            keys = torch.arange(k * L, (k + 1) * L)
            rows = torch.cat([torch.arange(p * L, (p + 1) * L) for p in ql])
            _, dk, dv = OB.bwd_rows(Q[0, h, rows], rows, K[0, h, keys], V[0, h, keys], dO[0, h, rows],
                                    LSE[0, h, rows], D[0, h, rows], scale, causal, key_pos=keys)
            acc_k[0, h, keys] += dk
            acc_v[0, h, keys] += dv
    assert torch.allclose(acc_q, dQ, atol=1e-12)
    assert torch.allclose(acc_k, dK, atol=1e-12)
    assert torch.allclose(acc_v, dV, atol=1e-12)


@pytest.mark.parametrize("P", [1, 4, 9, 16, 64])
def test_kv_slot_closed_forms(P):
    """KVR mesh: KV partition k = aR + c lies in the R tiles of mesh column c; tile row r has a
    live block for it iff its last Q partition rR + R - 1 >= k, i.e. r >= a.  So causal plans
    have R - floor(k/R) slots for k (R^2 (R+1)/2 in all), non-causal ones R (P R in all); every
    live block lies in exactly one slot."""
    R = math.isqrt(P)
    for causal in (False, True):
        plan = PL.make_plan(P * 4, P, causal, True, True)
        ks = PL.kv_slots(plan)
        for k in range(P):
            want = (R - k // R) if causal else R
            assert ks.kv_slot_off[k + 1] - ks.kv_slot_off[k] == want
        assert len(ks.kv_items) == (R * R * (R + 1) // 2 if causal else P * R)
        assert sum(len(q) for q in ks.kv_item_q) == plan.n_live_blocks
        assert [s for _, _, s in ks.kv_items] == list(range(len(ks.kv_items)))


def test_kv_slots_ring_and_empty():
    ring = PL.make_ring_plan(5 * 3, 3, True)
    ks = PL.kv_slots(ring)
    assert ks.kv_items == [(0, 0, 0), (0, 1, 1), (0, 2, 2), (1, 1, 3), (1, 2, 4), (2, 2, 5)]
    assert ks.kv_item_q == [[0], [1], [2], [1], [2], [2]]
    assert ks.kv_slot_off == [0, 3, 5, 6]
    empty = PL.kv_slots(PL.make_plan(0, 4, True, True, True))
    assert empty.kv_items == [] and empty.kv_slot_off == [0] * 5


@pytest.mark.parametrize("causal", [False, True])
def test_magnitude_sums_bound_the_gradients(causal):
    """The magnitude sums bound the gradients elementwise (triangle inequality), and equal dV when
    every term P_ij dO_i is non-negative (dO >= 0)."""
    Q, K, V, dO = _case(1, 4, 2, 19, 8, 61)
    g = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
    m = OB.attention_bwd_bhsd(Q, K, V, dO, causal, absolute=True)
    for a, b in zip(g[:3], m[:3]):
        assert (a.abs() <= b + 1e-12).all()
    dOp = dO.abs()
    g = OB.attention_bwd_bhsd(Q, K, V, dOp, causal)
    m = OB.attention_bwd_bhsd(Q, K, V, dOp, causal, absolute=True)
    assert torch.allclose(g[2], m[2], atol=1e-12)
    assert (m[0] > g[0].abs()).any()  # dS changes sign: the dQ magnitude is a strict bound somewhere
    # the magnitude of D bounds |D| = |dO . O| (and equals 2 sum |dO| |O| when V >= 0)
    assert (m[4] >= g[4].abs() - 1e-12).all()
    Vp = V.abs()
    O, _ = OA.attention_bhsd(Q, K, Vp, causal)
    mp = OB.attention_bwd_bhsd(Q, K, Vp, dOp, causal, absolute=True)
    assert torch.allclose(mp[4], 2 * (dOp * O).sum(dim=-1), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_key_and_row_gradients_match_full(causal):
    """dkdv_keys (dK, dV on chosen key rows, with magnitudes) and dq_rows with magnitudes equal
    the full backward (itself pinned above by finite differences and autograd) on those rows."""
    Q, K, V, dO = _case(1, 4, 2, 37, 8, 41)
    dQ, dK, dV, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, causal)
    mQ, mK, mV, _, _ = OB.attention_bwd_bhsd(Q, K, V, dO, causal, absolute=True)
    keys = [0, 5, 17, 36]
    for kh in range(2):
        dk, dv, mk, mv = OB.dkdv_keys(Q, K, V, dO, causal, 0, kh, keys, row_chunk=16)
        for got, ref in ((dk, dK[0, kh, keys]), (dv, dV[0, kh, keys]), (mk, mK[0, kh, keys]), (mv, mV[0, kh, keys])):
            assert torch.allclose(got, ref, atol=1e-12, rtol=1e-12)
    import numpy as np
    rows = np.array([[[0, 3, 36], [1, 2, 30], [4, 9, 33], [0, 20, 36]]])
    got, mag = OB.dq_rows(Q, K, V, dO, causal, rows, absolute=True)
    for h in range(4):
        assert torch.allclose(got[0, h], dQ[0, h, rows[0, h]], atol=1e-12, rtol=1e-12)
        assert torch.allclose(mag[0, h], mQ[0, h, rows[0, h]], atol=1e-12, rtol=1e-12)


def test_bf16_gradient_bound_rejects_one_missing_block():
    """The elementwise bound of the bf16 GPU gradients is tight enough to catch the loss of a
    single 128-wide block of the sum: on a bf16-rounded causal case (S = 2048, d = 128), dropping
    one key block from dQ, or one query block from dK and dV, moves some element outside the
    bound -- also among rows and keys at least 512 positions away from the dropped block, where
    the block is a small share of the sum.  (The perturbation is made on the oracle's result.)"""
    from mesh_inputs import Workload, make_do, make_qkv
    from tests.gpu_helpers import bf16_grad_bound
    w = Workload(150, "bound_check", 1, 1, 1, 2048, 128, "bf16", True, 4)
    q, k, v = make_qkv(w)
    dO = make_do(w)
    rQ, rK, rV, LSE, D = OB.attention_bwd_bhsd(q, k, v, dO, True)
    mQ, mK, mV, _, _ = OB.attention_bwd_bhsd(q, k, v, dO, True, absolute=True)
    Q64, K64, V64, G64 = (t[0, 0].double() for t in (q, k, v, dO))
    pos = torch.arange(w.S)
    scale = 1.0 / math.sqrt(w.d)
    for blk in (0, 3, 8):
        span = torch.arange(blk * 128, (blk + 1) * 128)
        # dQ without key block blk: the error is that block's contribution
        drop_q, _, _ = OB.bwd_rows(Q64, pos, K64[span], V64[span], G64, LSE[0, 0], D[0, 0], scale, True,
                                   key_pos=span, want_kv=False)
        ratio_q = drop_q.abs() / bf16_grad_bound(rQ[0, 0], mQ[0, 0], w.S)
        far_rows = pos >= (blk + 1) * 128 + 512
        assert ratio_q.max() > 1.0 and ratio_q[far_rows].max() > 1.0, (blk, ratio_q[far_rows].max())
        # dK and dV without query block blk
        _, drop_k, drop_v = OB.bwd_rows(Q64[span], span, K64, V64, G64[span], LSE[0, 0, span], D[0, 0, span],
                                        scale, True)
        ratio_k = drop_k.abs() / bf16_grad_bound(rK[0, 0], mK[0, 0], w.S)
        ratio_v = drop_v.abs() / bf16_grad_bound(rV[0, 0], mV[0, 0], w.S)
        assert ratio_k.max() > 1.0 and ratio_v.max() > 1.0, blk
        if blk >= 8:
            far_keys = pos < blk * 128 - 512
            assert ratio_k[far_keys].max() > 1.0 and ratio_v[far_keys].max() > 1.0, blk
