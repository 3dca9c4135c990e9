"""Pins for the plain-Python planner oracle: hand-worked plans, closed forms, coverage,
locality, greedy maximality and the O(sqrt(N)) versus O(N) receive count."""
import itertools
import json
import math
import os

import pytest

from oracle import planner as PL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["plan_p4_causal_kvr_greedy.json", "plan_p4_causal_nokvr_rowmajor.json"])
def test_hand_worked_plan(name):
    g = load(name)
    p = PL.make_plan(g["S"], g["P"], g["causal"], g["kvr"], g["greedy"])
    assert p.q_parts == g["q_parts"]
    assert p.kv_parts == g["kv_parts"]
    assert p.slot_off == g["slot_off"]
    assert [list(i) for i in p.items] == g["items"]
    assert p.item_kv == g["item_kv"]
    assert p.item_step == g["item_step"]
    assert [list(r) for r in p.recv] == g["recv"]
    assert p.n_live_blocks == g["n_live_blocks"]


@pytest.mark.parametrize("row", load("plan_counts.json")["rows"], ids=lambda r: r["name"])
def test_workload_counts(row):
    P, causal = row["P"], row["causal"]
    if P > 256:
        pytest.skip("P=1024 is checked against the C++ planner; the Python oracle takes minutes there")
    R = math.isqrt(P)
    a = PL.make_plan(P * 128, P, causal, True, False)
    b = PL.make_plan(P * 128, P, causal, False, False)
    assert a.slot_off[-1] == row["slots_kvr"]
    assert b.slot_off[-1] == row["slots_nokvr"]
    assert a.n_live_blocks == row["live_blocks"]
    idle_b = sum(1 for t in range(P) if not any(i[1] == t for i in b.items))
    idle_a = sum(1 for t in range(P) if not any(i[1] == t for i in a.items))
    assert idle_b == row["idle_nokvr"]
    assert idle_a == 0
    # closed forms
    if causal:
        assert a.slot_off[-1] == sum(min(p + 1, R) for p in range(P))
        assert b.slot_off[-1] == sum(p // R + 1 for p in range(P))
        assert a.n_live_blocks == P * (P + 1) // 2
    else:
        assert a.slot_off[-1] == P * R
        assert a.n_live_blocks == P * P


def check_plan_invariants(p: PL.Plan):
    P, R = p.P, p.R
    # each item is a slot exactly once, the order is a permutation of the slots
    slots = sorted(i[2] for i in p.items)
    assert slots == list(range(p.slot_off[-1]))
    for (pp, t, s), kvs in zip(p.items, p.item_kv):
        assert p.slot_off[pp] <= s < p.slot_off[pp + 1]
        assert pp in p.q_parts[t]
        assert sorted(kvs) == sorted(k for k in p.kv_parts[t] if PL.live(pp, k, p.causal))
        assert len(set(kvs)) == len(kvs) > 0
    # coverage: every live block is computed by exactly one item
    seen = {}
    for (pp, t, _), kvs in zip(p.items, p.item_kv):
        for k in kvs:
            assert (pp, k) not in seen
            seen[(pp, k)] = t
    assert set(seen) == {(a, k) for a in range(P) for k in range(P) if PL.live(a, k, p.causal)}
    # locality: Q from the own mesh row, KV from the own mesh column (with KVR) and the
    # diagonal block (v, v) in device v's own tile
    for v in range(P):
        r, c = divmod(v, R)
        assert all(q // R == r for q in p.q_parts[v])
        if p.kvr:
            assert all(k % R == c for k in p.kv_parts[v])
            assert v in p.kv_parts[v] and v in p.q_parts[v]
    # slots of p are in increasing tile column
    for pp in range(P):
        ts = sorted((s, t) for (q, t, s) in p.items if q == pp)
        assert [t for _, t in ts] == sorted(t for _, t in ts)


@pytest.mark.parametrize("P", [1, 4, 9, 16, 25, 36, 64])
@pytest.mark.parametrize("causal,kvr,greedy", list(itertools.product([False, True], repeat=3)))
def test_plan_invariants(P, causal, kvr, greedy):
    check_plan_invariants(PL.make_plan(P * 8, P, causal, kvr, greedy))


def brute_greedy_steps(v, qset, kvset, causal):
    """Independent greedy maximality check: at each step, every remaining transfer's gain
    recomputed from scratch over the full block set of the tile."""
    blocks = {(p, k) for p in qset for k in kvset if PL.live(p, k, causal)}
    need_q = {p for p, _ in blocks}
    need_kv = {k for _, k in blocks}
    have_q = {v} & need_q
    have_kv = {v} & need_kv
    gains = []
    while (need_q - have_q) or (need_kv - have_kv):
        def unlocked(hq, hk):
            return {(p, k) for (p, k) in blocks if p in hq and k in hk}
        base = len(unlocked(have_q, have_kv))
        opts = [(len(unlocked(have_q, have_kv | {k})) - base, 0, k) for k in need_kv - have_kv]
        opts += [(len(unlocked(have_q | {p}, have_kv)) - base, 1, p) for p in need_q - have_q]
        best = max(o[0] for o in opts)
        gains.append(best)
        choice = min((o for o in opts if o[0] == best), key=lambda o: (o[1], o[2]))
        (have_kv if choice[1] == 0 else have_q).add(choice[2])
    return gains


@pytest.mark.parametrize("P", [4, 9, 16])
@pytest.mark.parametrize("causal,kvr", list(itertools.product([False, True], repeat=2)))
def test_greedy_takes_max_gain_each_step(P, causal, kvr):
    R = math.isqrt(P)
    qs, ks = PL.tile_sets(P, R, kvr)
    for v in range(P):
        arr_q, arr_kv = PL.greedy_device(v, qs[v], ks[v], causal)
        # replay the oracle's choices and count the gain of each
        events = sorted([(s, 1, p) for p, s in arr_q.items() if s > 0] + [(s, 0, k) for k, s in arr_kv.items() if s > 0])
        hq = {p for p, s in arr_q.items() if s == 0}
        hk = {k for k, s in arr_kv.items() if s == 0}
        got = []
        for _, kind, x in events:
            if kind == 0:
                got.append(sum(1 for p in hq if PL.live(p, x, causal)))
                hk.add(x)
            else:
                got.append(sum(1 for k in hk if PL.live(x, k, causal)))
                hq.add(x)
        assert got == brute_greedy_steps(v, qs[v], ks[v], causal)
        assert sorted(s for s in list(arr_q.values()) + list(arr_kv.values()) if s > 0) == list(range(1, len(events) + 1))


@pytest.mark.parametrize("P", [4, 16, 64, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_receive_counts_closed_forms(P, causal):
    """With KVR every device receives at most R-1 Q, R-1 KV and R-1 partial-O partitions;
    Ring receives P-1.  The mesh/ring ratio 3(R-1)/(P-1) falls like 1/sqrt(P): the
    O(sqrt(N)) versus O(N) claim counted in partitions."""
    R = math.isqrt(P)
    a = PL.make_plan(P * 4, P, causal, True, True)
    mx = tuple(max(r[i] for r in a.recv) for i in range(3))
    assert mx == (R - 1, R - 1, R - 1)
    if not causal:
        assert all(r == (R - 1, R - 1, R - 1) for r in a.recv)
        b = PL.make_plan(P * 4, P, causal, False, True)
        # without KVR an off-diagonal device lacks its own KV partition: R KV receives
        for v, r in enumerate(b.recv):
            assert r[1] == (R - 1 if v // R == v % R else R)
    ring = PL.ring_recv_partitions(P)
    assert ring == P - 1
    ratio = sum(mx) / ring
    assert abs(ratio - 3 * (R - 1) / (P - 1)) < 1e-12
    assert ratio * math.sqrt(P) <= 3.0 + 1e-12


def test_volume_bytes():
    p = PL.make_plan(16384, 16, True, True, True)
    per, ring = PL.volume_bytes(p, 16, 16, 128, 2)
    mx = max(sum(x) for x in per)
    assert ring == 15 * 2 * 1024 * 16 * 128 * 2
    # Q, KV and fp32 partial (O plus LSE) of one partition, three of each at most
    assert mx == 3 * (1024 * 16 * 128 * 2) + 3 * (2 * 1024 * 16 * 128 * 2) + 3 * (1024 * 16 * (4 * 128 + 4))


def test_empty_sequence_and_bad_args():
    p = PL.make_plan(0, 4, True, True, True)
    assert p.slot_off == [0] * 5 and p.items == [] and p.n_live_blocks == 0
    for S, P in [(10, 4), (16, 8), (16, 0), (-4, 4)]:
        with pytest.raises(ValueError):
            PL.make_plan(S, P, True, True, True)


@pytest.mark.parametrize("P", [1, 2, 3, 4, 7, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_plan(P, causal):
    """Ring-Attention rows: one slot per Q partition covering every live KV partition, visited in
    ring order (own partition first), P - 1 KV receives per device and nothing else."""
    p = PL.make_ring_plan(P * 4, P, causal)
    assert p.slot_off == list(range(P + 1))
    assert sorted(i[0] for i in p.items) == list(range(P))
    for (q, t, slot), kvs in zip(p.items, p.item_kv):
        assert q == t == slot
        assert kvs[0] == q  # the device's own KV first
        assert sorted(kvs) == [k for k in range(P) if PL.live(q, k, causal)]
        assert kvs == [k for k in [(q - i) % P for i in range(P)] if PL.live(q, k, causal)]
    assert all(r == (0, P - 1, 0) for r in p.recv)
    assert p.n_live_blocks == (P * (P + 1) // 2 if causal else P * P)
    steps = p.item_step
    assert steps == sorted(steps)
    if causal:  # device v's last live block (KV 0) arrives after v hops
        assert sorted(steps) == list(range(P))


def test_ring_plan_hand_worked():
    """P = 3 causal, worked by hand: device 2 sees KV 2, 1, 0 (steps 0, 1, 2); device 1 sees KV 1
    then (ring step 1) KV 0; device 0 only its own KV 0."""
    p = PL.make_ring_plan(12, 3, True)
    assert [list(i) for i in p.items] == [[0, 0, 0], [1, 1, 1], [2, 2, 2]]
    assert p.item_kv == [[0], [1, 0], [2, 1, 0]]
    assert p.item_step == [0, 1, 2]
