"""Pins for the fp64 attention oracle, independent of the oracle's own code path.

* brute force: a pure-Python triple loop (math.fsum / math.exp) on tiny inputs;
* closed forms: equal keys, Q = 0, constant V, causal row 0;
* invariants: key shift, linearity in V, joint key/value permutation, any key split
  merged by LSE equals the unsplit result;
* the negative case: summing separately normalised block softmaxes (the right-hand
  side of the decomposition formula in the Ring-Attention blog, §"理论奠基") is not
  attention, so the oracle must disagree with it.
"""
import math
import random

import numpy as np
import pytest
import torch

from oracle import attention as A

F64 = torch.float64


def brute(q, k, v, scale, causal, q_pos=None):
    """Plain Python attention: lists of lists in, (O, lse) lists out."""
    n, m = len(q), len(k)
    q_pos = list(range(n)) if q_pos is None else list(q_pos)
    O, LSE = [], []
    for i in range(n):
        vis = [j for j in range(m) if (not causal or j <= q_pos[i])]
        if not vis:
            O.append([0.0] * len(v[0]))
            LSE.append(float("-inf"))
            continue
        s = {j: scale * math.fsum(q[i][e] * k[j][e] for e in range(len(q[i]))) for j in vis}
        mx = max(s.values())
        w = {j: math.exp(s[j] - mx) for j in vis}
        z = math.fsum(w.values())
        LSE.append(mx + math.log(z))
        O.append([math.fsum(w[j] * v[j][e] for j in vis) / z for e in range(len(v[0]))])
    return O, LSE


def rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * scale


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,m,d,seed", [(1, 1, 1, 0), (5, 5, 3, 1), (8, 8, 4, 2), (3, 7, 2, 3), (7, 3, 4, 4)])
def test_brute_force(causal, n, m, d, seed):
    q, k, v = rand((n, d), seed), rand((m, d), seed + 100, 2.0), rand((m, d + 1), seed + 200)
    scale = 0.7
    qpos = list(range(m - n, m)) if m >= n else list(range(n))
    O, L = A.attention_rows(q, qpos, k, v, scale, causal, key_chunk=3)
    Ob, Lb = brute(q.tolist(), k.tolist(), v.tolist(), scale, causal, qpos)
    Ob = torch.tensor(Ob, dtype=F64)
    Lb = torch.tensor(Lb, dtype=F64)
    fin = torch.isfinite(Lb)
    assert torch.equal(fin, torch.isfinite(L))
    assert torch.allclose(L[fin], Lb[fin], atol=1e-12, rtol=0)
    assert torch.allclose(O, Ob, atol=1e-12, rtol=0)


def test_brute_force_bhsd_gqa():
    """Head mapping: query head h reads kv head h // (Hq // Hkv)."""
    B, Hq, Hkv, S, d = 2, 4, 2, 6, 3
    Q, K, V = rand((B, Hq, S, d), 7), rand((B, Hkv, S, d), 8), rand((B, Hkv, S, d), 9)
    O, L = A.attention_bhsd(Q, K, V, causal=True)
    for b in range(B):
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            Ob, Lb = brute(Q[b, h].tolist(), K[b, kh].tolist(), V[b, kh].tolist(), 1 / math.sqrt(d), True)
            assert torch.allclose(O[b, h], torch.tensor(Ob, dtype=F64), atol=1e-12, rtol=0)
            assert torch.allclose(L[b, h], torch.tensor(Lb, dtype=F64), atol=1e-12, rtol=0)


def test_sampled_rows_match_full():
    B, Hq, Hkv, S, d = 1, 2, 1, 40, 4
    Q, K, V = rand((B, Hq, S, d), 11), rand((B, Hkv, S, d), 12), rand((B, Hkv, S, d), 13)
    rows = np.array([[[0, 5, 17, 39], [1, 2, 3, 38]]])
    O, L = A.attention_bhsd(Q, K, V, causal=True)
    Os, Ls = A.attention_bhsd(Q, K, V, causal=True, rows=rows)
    for h in range(Hq):
        assert torch.equal(Os[0, h], O[0, h, rows[0, h]])
        assert torch.equal(Ls[0, h], L[0, h, rows[0, h]])


@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_closed_form(causal):
    """All keys equal: every visible score is s_i, so O_i = mean of visible V rows and
    LSE_i = ln|visible| + s_i."""
    n, d = 33, 8
    q = rand((n, d), 21)
    k1 = rand((1, d), 22)
    k = k1.repeat(n, 1)
    v = rand((n, d), 23)
    scale = 1 / math.sqrt(d)
    O, L = A.attention_rows(q, torch.arange(n), k, v, scale, causal, key_chunk=7)
    for i in range(n):
        cnt = i + 1 if causal else n
        s_i = scale * float(q[i] @ k1[0])
        assert abs(float(L[i]) - (math.log(cnt) + s_i)) < 1e-12
        assert torch.allclose(O[i], v[:cnt].mean(dim=0), atol=1e-13, rtol=0)


def test_zero_query_closed_form():
    n, d = 20, 4
    O, L = A.attention_rows(torch.zeros(n, d), torch.arange(n), rand((n, d), 31), rand((n, d), 32), 0.5, True)
    for i in range(n):
        assert abs(float(L[i]) - math.log(i + 1)) < 1e-13


def test_constant_v_closed_form():
    n, d = 50, 16
    v = torch.full((n, d), -1.75, dtype=F64)
    O, _ = A.attention_rows(rand((n, d), 41), torch.arange(n), rand((n, d), 42, 3.0), v, 0.25, True)
    assert torch.allclose(O, v, atol=1e-14, rtol=0)


def test_causal_row0_closed_form():
    n, d = 17, 5
    q, k, v = rand((n, d), 51), rand((n, d), 52), rand((n, d), 53)
    O, L = A.attention_rows(q, torch.arange(n), k, v, 0.3, True)
    assert torch.allclose(O[0], v[0], atol=1e-15, rtol=0)
    assert abs(float(L[0]) - 0.3 * float(q[0] @ k[0])) < 1e-14


def test_key_shift_invariant():
    n, d = 24, 6
    q, k, v = rand((n, d), 61), rand((n, d), 62), rand((n, d), 63)
    u = rand((d,), 64)
    sc = 0.4
    O1, L1 = A.attention_rows(q, torch.arange(n), k, v, sc, True)
    O2, L2 = A.attention_rows(q, torch.arange(n), k + u, v, sc, True)
    assert torch.allclose(O1, O2, atol=1e-12, rtol=0)
    assert torch.allclose(L2, L1 + sc * (q @ u), atol=1e-12, rtol=0)


def test_linear_in_v():
    n, d = 19, 5
    q, k = rand((n, d), 71), rand((n, d), 72)
    v1, v2 = rand((n, d), 73), rand((n, d), 74)
    O1, _ = A.attention_rows(q, torch.arange(n), k, v1, 0.5, False)
    O2, _ = A.attention_rows(q, torch.arange(n), k, v2, 0.5, False)
    O3, _ = A.attention_rows(q, torch.arange(n), k, 2.5 * v1 - 0.5 * v2, 0.5, False)
    assert torch.allclose(O3, 2.5 * O1 - 0.5 * O2, atol=1e-12, rtol=0)


def test_joint_permutation_invariant():
    n, m, d = 9, 31, 4
    q, k, v = rand((n, d), 81), rand((m, d), 82), rand((m, d), 83)
    perm = torch.randperm(m, generator=torch.Generator().manual_seed(84))
    O1, L1 = A.attention_rows(q, torch.arange(n), k, v, 0.6, False)
    O2, L2 = A.attention_rows(q, torch.arange(n), k[perm], v[perm], 0.6, False)
    assert torch.allclose(O1, O2, atol=1e-12, rtol=0)
    assert torch.allclose(L1, L2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", range(6))
def test_split_merge_equals_unsplit(causal, seed):
    """Any split of the keys (including empty parts), each part attended separately and
    merged by LSE, equals attention over all keys."""
    rng = random.Random(seed)
    n, m, d = 23, 57, 8
    q, k, v = rand((n, d), 90 + seed), rand((m, d), 190 + seed, 2.0), rand((m, d), 290 + seed)
    qpos = torch.arange(m - n, m)
    idx = list(range(m))
    rng.shuffle(idx)
    cuts = sorted(rng.sample(range(m + 1), rng.randint(1, 6)))
    parts = [idx[a:b] for a, b in zip([0] + cuts, cuts + [m])]
    parts.append([])  # an empty part must carry weight 0
    O1, L1 = A.attention_rows(q, qpos, k, v, 0.35, causal)
    O2, L2 = A.split_attention(q, qpos, k, v, 0.35, causal, parts)
    assert torch.allclose(O1, O2, atol=1e-12, rtol=0)
    assert torch.allclose(L1, L2, atol=1e-12, rtol=0)


def test_merge_special_cases():
    n, d = 6, 3
    o, l = rand((n, d), 1), rand((n,), 2)
    # a part merged with an identical copy: same O, lse + ln 2
    O, L = A.merge([(o, l), (o, l)])
    assert torch.allclose(O, o, atol=1e-15, rtol=0)
    assert torch.allclose(L, l + math.log(2), atol=1e-15, rtol=0)
    # an empty part (lse = -inf) changes nothing
    ninf = torch.full((n,), float("-inf"), dtype=F64)
    O, L = A.merge([(o, l), (torch.zeros(n, d, dtype=F64), ninf)])
    assert torch.equal(O, o) and torch.equal(L, l)
    # every part empty: O = 0, lse = -inf, no NaN
    O, L = A.merge([(torch.zeros(n, d, dtype=F64), ninf)] * 3)
    assert torch.equal(O, torch.zeros(n, d, dtype=F64)) and bool(torch.isneginf(L).all())
    # two parts, hand computed weights e^1 / (e^1 + e^0)
    a = torch.tensor([[1.0, 0.0]], dtype=F64)
    b = torch.tensor([[0.0, 1.0]], dtype=F64)
    O, L = A.merge([(a, torch.tensor([1.0], dtype=F64)), (b, torch.tensor([0.0], dtype=F64))])
    w = math.e / (math.e + 1)
    assert abs(float(O[0, 0]) - w) < 1e-15 and abs(float(O[0, 1]) - (1 - w)) < 1e-15
    assert abs(float(L[0]) - math.log(math.e + 1)) < 1e-15


def test_empty_rows_and_keys():
    d = 4
    q = rand((3, d), 5)
    O, L = A.attention_rows(q, [0, 1, 2], torch.zeros(0, d, dtype=F64), torch.zeros(0, d, dtype=F64), 1.0, False)
    assert torch.equal(O, torch.zeros(3, d, dtype=F64)) and bool(torch.isneginf(L).all())
    # causal: keys all after the query -> empty row
    O, L = A.attention_rows(q, [0, 1, 2], rand((2, d), 6), rand((2, d), 7), 1.0, True, key_pos=[5, 6])
    assert bool(torch.isneginf(L).all()) and not torch.isnan(O).any()


def test_summed_block_softmax_is_not_attention():
    """With V constant c and T key blocks, sum_i softmax(Q K_i^T) V_i = T*c while
    attention gives c: the blog's right-hand side is not an identity."""
    n, d, T = 8, 4, 4
    q, k = rand((n, d), 3), rand((n * T, d), 4)
    v = torch.full((n * T, d), 0.5, dtype=F64)
    O, _ = A.attention_rows(q, torch.arange(n), k, v, 0.5, False)
    rhs = torch.zeros(n, d, dtype=F64)
    for i in range(T):
        sl = slice(i * n, (i + 1) * n)
        rhs += torch.softmax(0.5 * q @ k[sl].T, dim=1) @ v[sl]
    assert torch.allclose(O, v[:n], atol=1e-14)
    assert torch.allclose(rhs, T * v[:n], atol=1e-14)
    assert not torch.allclose(O, rhs, atol=1e-3)


def test_bf16_inputs_upcast_exactly():
    """bf16 values enter the oracle unchanged (bf16 -> fp64 is exact)."""
    x = torch.randn(16, 8).to(torch.bfloat16)
    assert torch.equal(A._as64(x), x.double())
