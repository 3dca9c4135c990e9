"""Plain-Python oracle of the Mesh-Attention tile planner.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module; the C++ planner in the product library shares
no code with it.

It restates, set by set, how Mesh-Attention assigns the Q-KV interaction matrix to a
sqrt(P) x sqrt(P) mesh of devices:

* Q-KV interaction matrix: P x P blocks, row = Q partition, column = KV partition
  ("Mesh-Attention" tutorial, §"Mesh-Attention：从一维'环'到二维'网'"; arXiv abstract).
* Ring-Attention gives a device a whole row; Mesh-Attention gives device v a 2D tile and
  lets it talk only to its own mesh row and column (same section, items (a) and (b)).
* KV Partition Rotation ("索引旋转", same section, item (c); the abstract's "KVR") changes
  which KV partitions a tile holds so that each device keeps its own Q *and* KV partition
  local.
* Greedy scheduling (tutorial §"贪心算法：寻找最优的'流水线'", rule 1): the next transfer
  is the one that unlocks the most compute blocks.  Rule 2 (hold some compute back to fill
  later waits) only matters with real transfers and is not modelled.
* Communication volume O(sqrt(N)) per device instead of Ring's O(N) (same section as
  the tiles; abstract).

Readings adopted where the pages leave a step open:
* device v owns Q partition v and KV partition v and sits at mesh position (v // R, v % R);
* tile t = v holds Q partitions {r*R + j} (its mesh row's contiguous group) and KV
  partitions {k*R + c : k < R} with KVR (its mesh column, strided), or {c*R + k : k < R}
  without KVR;
* causal: block (p, k) is live iff k <= p; non-causal: every block is live;
* a (p, t) pair with at least one live block is a partial slot; the slots of partition p
  are numbered consecutively in increasing tile column;
* greedy ties: a KV transfer before a Q transfer, then the lower partition index; a
  work item (p, t) completes at the step that unlocks its last live block; the global
  order lists items by (completion step, device, p); each item's KV partitions are
  visited in the order they reached the device;
* without greedy: items in (tile, p) order with KV partitions ascending.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Tuple


@dataclasses.dataclass
class Plan:
    S: int
    P: int
    R: int
    L: int
    causal: bool
    kvr: bool
    greedy: bool
    q_parts: List[List[int]]  # [P][R]
    kv_parts: List[List[int]]  # [P][R]
    slot_off: List[int]  # [P+1]
    items: List[Tuple[int, int, int]]  # (p, t, slot) in execution order
    item_kv: List[List[int]]  # KV partitions of each item, in visiting order
    item_step: List[int]  # greedy completion step of each item (0 without greedy)
    recv: List[Tuple[int, int, int]]  # per device (Q, KV, partial-O) partitions received
    n_live_blocks: int


def live(p: int, k: int, causal: bool) -> bool:
    return (k <= p) if causal else True


def tile_sets(P: int, R: int, kvr: bool):
    q_parts, kv_parts = [], []
    for t in range(P):
        r, c = divmod(t, R)
        q_parts.append([r * R + j for j in range(R)])
        kv_parts.append([k * R + c for k in range(R)] if kvr else [c * R + k for k in range(R)])
    return q_parts, kv_parts


def greedy_device(v: int, qset: List[int], kvset: List[int], causal: bool):
    """Greedy receive order of device v on its own tile.

    Returns (arrival step of each needed Q partition, of each needed KV partition).
    """
    need_q = [p for p in qset if any(live(p, k, causal) for k in kvset)]
    need_kv = [k for k in kvset if any(live(p, k, causal) for p in qset)]
    arr_q: Dict[int, int] = {}
    arr_kv: Dict[int, int] = {}
    if v in need_q:
        arr_q[v] = 0
    if v in need_kv:
        arr_kv[v] = 0
    step = 0
    while True:
        cands = []
        for k in need_kv:
            if k not in arr_kv:
                gain = sum(1 for p in arr_q if live(p, k, causal))
                cands.append((gain, 0, k))  # kind 0 = KV
        for p in need_q:
            if p not in arr_q:
                gain = sum(1 for k in arr_kv if live(p, k, causal))
                cands.append((gain, 1, p))  # kind 1 = Q
        if not cands:
            break
        step += 1
        best = max(cands, key=lambda c: (c[0], -c[1], -c[2]))
        (arr_kv if best[1] == 0 else arr_q)[best[2]] = step
    return arr_q, arr_kv


def make_plan(S: int, P: int, causal: bool, kvr: bool, greedy: bool) -> Plan:
    if P < 1:
        raise ValueError("P must be >= 1")
    R = math.isqrt(P)
    if R * R != P:
        raise ValueError("P must be a perfect square")
    if S < 0 or S % P != 0:
        raise ValueError("S must be a non-negative multiple of P")
    L = S // P
    q_parts, kv_parts = tile_sets(P, R, kvr)
    empty = (S == 0)

    # partial slots, grouped by Q partition, tile column ascending
    slot_of: Dict[Tuple[int, int], int] = {}
    slot_off = [0]
    for p in range(P):
        r = p // R
        for c in range(R):
            t = r * R + c
            if not empty and any(live(p, k, causal) for k in kv_parts[t]):
                slot_of[(p, t)] = len(slot_of)
        slot_off.append(len(slot_of))

    n_live = 0 if empty else sum(1 for p in range(P) for k in range(P) if live(p, k, causal))

    items: List[Tuple[int, int, int]] = []
    item_kv: List[List[int]] = []
    item_step: List[int] = []
    recv: List[Tuple[int, int, int]] = []
    keyed = []
    for t in range(P):
        v = t
        qset, kvset = q_parts[t], kv_parts[t]
        if empty:
            recv.append((0, 0, 0))
            continue
        arr_q, arr_kv = greedy_device(v, qset, kvset, causal)
        n_slots_v = slot_off[v + 1] - slot_off[v]
        recv.append((len([p for p in arr_q if p != v]),
                     len([k for k in arr_kv if k != v]),
                     n_slots_v - (1 if (v, t) in slot_of else 0)))
        for p in qset:
            if (p, t) not in slot_of:
                continue
            kvs = [k for k in kvset if live(p, k, causal)]
            if greedy:
                done = max(max(arr_q[p], arr_kv[k]) for k in kvs)
                kvs = sorted(kvs, key=lambda k: arr_kv[k])
                keyed.append(((done, t, p), (p, t, slot_of[(p, t)]), kvs, done))
            else:
                keyed.append(((0, t, p), (p, t, slot_of[(p, t)]), sorted(kvs), 0))
    keyed.sort(key=lambda e: e[0])
    for _, it, kvs, st in keyed:
        items.append(it)
        item_kv.append(kvs)
        item_step.append(st)

    return Plan(S, P, R, L, causal, kvr, greedy, q_parts, kv_parts, slot_off, items, item_kv,
                item_step, recv, n_live)


def make_ring_plan(S: int, P: int, causal: bool) -> Plan:
    """Ring-Attention's assignment as a plan of the same shape: device v owns Q partition v and
    computes its whole row of the Q-KV matrix ("Mesh-Attention" tutorial, the 1D ring of item
    (a) and the section on Ring-Attention's bottleneck: no Q moves, every KV partition passes
    through every device).

    Readings: KV partitions reach device v in ring order v, v-1, v-2, ... (its own first, one
    neighbour hop per step); an item completes at the step its last live block arrives; items are
    ordered by (step, device); each device receives P-1 KV partitions (a plain ring forwards all
    of them) and no Q or partial output.
    """
    if P < 1:
        raise ValueError("P must be >= 1")
    if S < 0 or S % P != 0:
        raise ValueError("S must be a non-negative multiple of P")
    L = S // P
    empty = S == 0
    q_parts = [[v] for v in range(P)]
    kv_parts = [[(v - i) % P for i in range(P)] for v in range(P)]
    slot_off = [0] + [0 if empty else p + 1 for p in range(P)]
    keyed = []
    for v in range(P):
        if empty:
            continue
        kvs = [k for k in kv_parts[v] if live(v, k, causal)]
        done = max(i for i, k in enumerate(kv_parts[v]) if live(v, k, causal))
        keyed.append(((done, v), (v, v, v), kvs, done))
    keyed.sort(key=lambda e: e[0])
    recv = [(0, 0 if empty else P - 1, 0) for _ in range(P)]
    n_live = 0 if empty else sum(1 for p in range(P) for k in range(P) if live(p, k, causal))
    return Plan(S, P, 1, L, causal, False, True, q_parts, kv_parts, slot_off, [e[1] for e in keyed],
                [e[2] for e in keyed], [e[3] for e in keyed], recv, n_live)


def ring_recv_partitions(P: int) -> int:
    """KV partitions a device receives in plain Ring-Attention: every other one."""
    return P - 1


def volume_bytes(plan: Plan, Hq: int, Hkv: int, d: int, elem_bytes: int):
    """Per-device received bytes (Q, KV, partial O+LSE) and Ring's per-device KV bytes.

    A Q partition is L*Hq*d elements, a KV partition 2*L*Hkv*d elements (K and V), a
    partial L*Hq*(d+1) fp32 values (normalised O and the LSE).
    """
    qb = plan.L * Hq * d * elem_bytes
    kvb = 2 * plan.L * Hkv * d * elem_bytes
    ob = plan.L * Hq * (4 * d + 4)
    per = [(q * qb, kv * kvb, o * ob) for (q, kv, o) in plan.recv]
    return per, ring_recv_partitions(plan.P) * kvb


@dataclasses.dataclass
class KvSlots:
    """Backward pass: the partial dK / dV slots of a plan."""
    kv_slot_off: List[int]  # [P+1]: the slots of KV partition k are kv_slot_off[k] .. kv_slot_off[k+1]-1
    kv_items: List[Tuple[int, int, int]]  # (k, t, kv_slot) in slot order
    kv_item_q: List[List[int]]  # the tile's Q partitions with a live block for k, ascending


def kv_slots(plan: Plan) -> KvSlots:
    """The (KV partition k, tile t) pairs of a plan that hold at least one live block.

    In the backward pass tile t sums dK and dV of each of its KV partitions over its own Q
    partitions; those partial sums go back along the mesh column to k's owner, as the forward's
    partial outputs go back along the mesh row to the Q owner.  Readings: slots are grouped by k,
    tiles ascending within a group, and the backward visits them in slot order.
    """
    P = plan.P
    off = [0]
    items: List[Tuple[int, int, int]] = []
    item_q: List[List[int]] = []
    empty = plan.S == 0
    for k in range(P):
        for t in range(len(plan.q_parts)):
            if empty or k not in plan.kv_parts[t]:
                continue
            qs = sorted(p for p in plan.q_parts[t] if live(p, k, plan.causal))
            if qs:
                items.append((k, t, len(items)))
                item_q.append(qs)
        off.append(len(items))
    return KvSlots(off, items, item_q)
