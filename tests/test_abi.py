"""CPU tests of the C ABI: the library loads, exports every declared entry point, the C++
planner matches the plain-Python planner oracle bit for bit, and host-side validation
returns the documented status codes before touching the GPU."""
import ctypes
import itertools
import json
import math
import os
import re

import pytest

from oracle import planner as PL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mesh_attn.h")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mesh_attn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 15
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), f"{n} declared in mesh_attn.h but not exported"
    assert set(names) == set(lib._SIGS), "binding and header disagree"


def cpp_plan(lib, S, P, causal, kvr, greedy):
    p = lib.mesh_attn_plan_create(S, P, causal, kvr, greedy)
    q, kv = lib.mesh_attn_plan_tiles(p)
    off = lib.mesh_attn_plan_slots(p)
    items, steps, kvs = lib.mesh_attn_plan_order(p)
    counts, _, _ = lib.mesh_attn_plan_volumes(p, 1, 1, 1)
    return p, q, kv, off, items, steps, kvs, counts


@pytest.mark.parametrize("P", [1, 4, 9, 16, 25, 64, 256])
@pytest.mark.parametrize("causal,kvr,greedy", list(itertools.product([0, 1], repeat=3)))
def test_planner_matches_oracle(lib, P, causal, kvr, greedy):
    S = P * 3
    ref = PL.make_plan(S, P, bool(causal), bool(kvr), bool(greedy))
    p, q, kv, off, items, steps, kvs, counts = cpp_plan(lib, S, P, causal, kvr, greedy)
    assert q == ref.q_parts and kv == ref.kv_parts
    assert off == ref.slot_off
    assert [list(i) for i in items] == [list(i) for i in ref.items]
    assert steps == ref.item_step
    assert kvs == ref.item_kv
    assert [list(c) for c in counts] == [list(r) for r in ref.recv]
    assert p.n_live_blocks == ref.n_live_blocks
    assert p.n_kv_entries == ref.n_live_blocks
    assert p.L == 3 and p.R == math.isqrt(P)


@pytest.mark.parametrize("name", ["plan_p4_causal_kvr_greedy.json", "plan_p4_causal_nokvr_rowmajor.json"])
def test_hand_worked_plan_cpp(lib, name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    p, q, kv, off, items, steps, kvs, counts = cpp_plan(lib, g["S"], g["P"], g["causal"], g["kvr"], g["greedy"])
    assert q == g["q_parts"] and kv == g["kv_parts"] and off == g["slot_off"]
    assert [list(i) for i in items] == g["items"]
    assert kvs == g["item_kv"] and steps == g["item_step"]
    assert [list(c) for c in counts] == g["recv"]


@pytest.mark.parametrize("row", json.load(open(os.path.join(GOLDEN, "plan_counts.json")))["rows"],
                         ids=lambda r: r["name"])
def test_workload_counts_cpp(lib, row):
    P, causal = row["P"], row["causal"]
    R = math.isqrt(P)
    a = lib.mesh_attn_plan_create(P * 256, P, causal, True, True)
    b = lib.mesh_attn_plan_create(P * 256, P, causal, False, True)
    assert a.n_slots == row["slots_kvr"] and b.n_slots == row["slots_nokvr"]
    assert a.n_live_blocks == row["live_blocks"]
    items_b, _, _ = lib.mesh_attn_plan_order(b)
    assert P - len({t for _, t, _ in items_b}) == row["idle_nokvr"]
    counts, _, ring = lib.mesh_attn_plan_volumes(a, 1, 1, 1)
    assert tuple(max(c[i] for c in counts) for i in range(3)) == (R - 1, R - 1, R - 1)


def test_volume_bytes_match_oracle(lib):
    for causal in (False, True):
        ref = PL.make_plan(16384, 16, causal, True, True)
        per, ring = PL.volume_bytes(ref, 16, 16, 128, 2)
        p = lib.mesh_attn_plan_create(16384, 16, causal, True, True)
        _, byts, ring_c = lib.mesh_attn_plan_volumes(p, 16, 16, 128)
        assert [tuple(b) for b in byts] == [tuple(x) for x in per]
        assert ring_c == ring


def test_planner_large_p_consistency(lib):
    """P = 1024 (the stress workload): slot closed form, coverage of live blocks, order is a
    permutation of the slots, and each item's KV list lies in its tile's mesh column."""
    P, R = 1024, 32
    p = lib.mesh_attn_plan_create(P * 256, P, True, True, True)
    items, steps, kvs = lib.mesh_attn_plan_order(p)
    assert p.n_slots == sum(min(x + 1, R) for x in range(P))
    assert sorted(s for _, _, s in items) == list(range(p.n_slots))
    assert sum(len(k) for k in kvs) == P * (P + 1) // 2
    assert steps == sorted(steps)
    for (q, t, _), kl in zip(items, kvs):
        assert all(k % R == t % R and k <= q for k in kl)


def test_status_codes(lib):
    so = lib._lib
    h = ctypes.c_void_p()
    assert so.mesh_attn_plan_create(100, 8, 1, 1, 1, ctypes.byref(h)) == 1  # P not a square
    assert "square" in so.mesh_attn_last_error().decode()
    assert so.mesh_attn_plan_create(10, 4, 1, 1, 1, ctypes.byref(h)) == 1  # S % P
    assert so.mesh_attn_plan_create(16, 4, 2, 1, 1, ctypes.byref(h)) == 1  # flag not 0/1
    assert so.mesh_attn_plan_create(16, 0, 1, 1, 1, ctypes.byref(h)) == 1
    assert so.mesh_attn_plan_create(-4, 4, 1, 1, 1, ctypes.byref(h)) == 1
    assert so.mesh_attn_plan_create(16 * 4225, 4225, 1, 1, 1, ctypes.byref(h)) == 1  # P > 4096
    assert so.mesh_attn_plan_create(16, 4, 1, 1, 1, None) == 1
    plan = lib.mesh_attn_plan_create(1024, 4, True)
    ws = lib.mesh_attn_workspace_size(plan)
    fake = ctypes.c_void_p(1 << 20)
    args = lambda **kw: dict(dict(plan=plan.handle, dt=1, B=1, Hq=2, Hkv=1, d=128, Q=fake, K=fake, V=fake,
                                  scale=0.1, po=fake, pl=fake, ws=fake, wsb=ws, st=fake, stream=None), **kw)

    def call(**kw):
        a = args(**kw)
        return so.mesh_attn_tile_fwd(a["plan"], a["dt"], a["B"], a["Hq"], a["Hkv"], a["d"], a["Q"], a["K"], a["V"],
                                     a["scale"], a["po"], a["pl"], a["ws"], a["wsb"], a["st"], a["stream"])

    assert call(plan=None) == 1
    assert call(d=96) == 2
    assert call(Hkv=3) == 1
    assert call(dt=7) == 1
    assert call(scale=0.0) == 1
    assert call(scale=float("nan")) == 1
    assert call(Q=None) == 1
    assert call(K=ctypes.c_void_p((1 << 20) + 8)) == 3
    assert call(wsb=ws - 1) == 9
    assert call(B=-1) == 1
    assert call(B=0) == 0 and call(Hq=0) == 0  # nothing to do: no launch, no CUDA call
    assert call(B=1 << 20, Hq=1 << 10) == 2    # rows beyond 32-bit coordinates
    # merge validation
    assert so.mesh_attn_merge(plan.handle, 5, 1, 2, 128, fake, fake, fake, fake, fake, ws, fake, None) == 1
    assert so.mesh_attn_merge(plan.handle, 1, 1, 2, 128, fake, fake, fake, fake, fake, ws - 1, fake, None) == 9
    assert so.mesh_attn_merge(plan.handle, 1, 1, 2, 100, fake, fake, fake, fake, fake, ws, fake, None) == 2
    assert so.mesh_attn_set_wait_limit_ns(-1) == 1
    for c in range(10):
        assert so.mesh_attn_status_string(c)
    assert so.mesh_attn_plan_destroy(None) == 0


def test_empty_sequence_plan(lib):
    p = lib.mesh_attn_plan_create(0, 16, True)
    assert p.n_slots == 0 and p.n_live_blocks == 0 and p.L == 0
    assert lib.mesh_attn_partials_size(p, 2, 4, 128) == (0, 0)
    # an empty plan enqueues nothing: NULL tensors are accepted
    rc = lib._lib.mesh_attn_tile_fwd(p.handle, 1, 1, 2, 1, 128, None, None, None, 0.1, None, None, None, 0, None, None)
    assert rc == 0
    rc = lib._lib.mesh_attn_merge(p.handle, 1, 1, 2, 128, None, None, None, None, None, 0, None, None)
    assert rc == 0


def test_partials_and_workspace_sizes(lib):
    p = lib.mesh_attn_plan_create(16384, 16, True)
    assert lib.mesh_attn_partials_size(p, 1, 16, 128) == (16 * 58 * 1024 * 128, 16 * 58 * 1024)
    assert lib.mesh_attn_workspace_size(p) >= 17 * 4 + 58 * 16 + 136 * 4


@pytest.mark.parametrize("P", [1, 2, 3, 4, 7, 16, 100])
@pytest.mark.parametrize("causal", [0, 1])
def test_ring_planner_matches_oracle(lib, P, causal):
    S = P * 5
    ref = PL.make_ring_plan(S, P, bool(causal))
    p = lib.mesh_attn_plan_create_ring(S, P, causal)
    assert p.layout == 1 and p.tile_q == 1 and p.tile_kv == P and p.R == 0
    q, kv = lib.mesh_attn_plan_tiles(p)
    assert q == ref.q_parts and kv == ref.kv_parts
    assert lib.mesh_attn_plan_slots(p) == ref.slot_off
    items, steps, kvs = lib.mesh_attn_plan_order(p)
    assert [list(i) for i in items] == [list(i) for i in ref.items]
    assert steps == ref.item_step and kvs == ref.item_kv
    counts, _, ring = lib.mesh_attn_plan_volumes(p, 1, 1, 1)
    assert [list(c) for c in counts] == [list(r) for r in ref.recv]


def test_ring_plan_errors(lib):
    so = lib._lib
    h = ctypes.c_void_p()
    assert so.mesh_attn_plan_create_ring(10, 3, 1, ctypes.byref(h)) == 1
    assert so.mesh_attn_plan_create_ring(12, 0, 1, ctypes.byref(h)) == 1
    assert so.mesh_attn_plan_create_ring(12, 3, 2, ctypes.byref(h)) == 1
    p = lib.mesh_attn_plan_create_ring(0, 3, True)
    assert p.n_slots == 0


@pytest.mark.parametrize("P", [1, 4, 9, 16, 64])
@pytest.mark.parametrize("causal,kvr", list(itertools.product([0, 1], repeat=2)))
def test_kv_slots_match_oracle(lib, P, causal, kvr):
    """Backward KV slots of the C++ planner equal the plain-Python planner's, bit for bit."""
    S = P * 3
    ref = PL.kv_slots(PL.make_plan(S, P, bool(causal), bool(kvr), True))
    p = lib.mesh_attn_plan_create(S, P, causal, kvr, True)
    off, items, qs = lib.mesh_attn_plan_kv_slots(p)
    assert p.n_kv_slots == len(ref.kv_items)
    assert off == ref.kv_slot_off
    assert [list(i) for i in items] == [list(i) for i in ref.kv_items]
    assert qs == ref.kv_item_q


@pytest.mark.parametrize("P", [1, 3, 7])
def test_kv_slots_ring_match_oracle(lib, P):
    for causal in (0, 1):
        ref = PL.kv_slots(PL.make_ring_plan(P * 2, P, bool(causal)))
        p = lib.mesh_attn_plan_create_ring(P * 2, P, causal)
        off, items, qs = lib.mesh_attn_plan_kv_slots(p)
        assert off == ref.kv_slot_off and [list(i) for i in items] == [list(i) for i in ref.kv_items]
        assert qs == ref.kv_item_q


def test_backward_sizes_and_status_codes(lib):
    so = lib._lib
    p = lib.mesh_attn_plan_create(16384, 16, True)
    assert p.n_kv_slots == 40  # R^2 (R + 1) / 2 for R = 4
    assert lib.mesh_attn_bwd_partials_size(p, 1, 16, 4, 128) == (16 * 58 * 1024 * 128, 4 * 40 * 1024 * 128)
    ws = lib.mesh_attn_bwd_workspace_size(p)
    assert ws >= 17 * 4 + 58 * 16 + 136 * 4 + 17 * 4 + 40 * 16 + 136 * 4 + 512
    fake = ctypes.c_void_p(1 << 20)

    def tile(**kw):
        a = dict(plan=p.handle, dt=1, B=1, Hq=2, Hkv=1, d=128, scale=0.1, wsb=ws, dO=fake)
        a.update(kw)
        return so.mesh_attn_tile_bwd(a["plan"], a["dt"], a["B"], a["Hq"], a["Hkv"], a["d"], fake, fake, fake, a["dO"],
                                     fake, fake, a["scale"], fake, fake, fake, fake, a["wsb"], fake, None)

    assert tile(plan=None) == 1
    assert tile(d=96) == 2
    assert tile(Hkv=3) == 1
    assert tile(dt=7) == 1
    assert tile(scale=-1.0) == 1
    assert tile(dO=None) == 1
    assert tile(dO=ctypes.c_void_p((1 << 20) + 4)) == 3
    assert tile(wsb=ws - 1) == 9
    assert tile(B=0) == 0 and tile(Hq=0) == 0
    assert so.mesh_attn_bwd_prep(1, 1, 2, 1024, 100, fake, fake, fake, fake, None) == 2
    assert so.mesh_attn_bwd_prep(5, 1, 2, 1024, 128, fake, fake, fake, fake, None) == 1
    assert so.mesh_attn_bwd_prep(1, 0, 2, 1024, 128, None, None, None, None, None) == 0
    assert so.mesh_attn_bwd_reduce(p.handle, 1, 1, 2, 1, 128, fake, fake, fake, fake, fake, fake, fake, ws - 1, fake,
                                   None) == 9
    assert so.mesh_attn_bwd_reduce(p.handle, 1, 1, 2, 3, 128, fake, fake, fake, fake, fake, fake, fake, ws, fake,
                                   None) == 1
    empty = lib.mesh_attn_plan_create(0, 16, True)
    assert empty.n_kv_slots == 0
    assert lib.mesh_attn_bwd_partials_size(empty, 2, 4, 2, 128) == (0, 0)
    assert so.mesh_attn_tile_bwd(empty.handle, 1, 1, 2, 1, 128, None, None, None, None, None, None, 0.1, None, None,
                                 None, None, 0, None, None) == 0
    assert so.mesh_attn_bwd_reduce(empty.handle, 1, 1, 2, 1, 128, None, None, None, None, None, None, None, 0, None,
                                   None) == 0


def test_workspace_size_for_fp32_pieces(lib):
    """fp32 inputs need room for three bf16 pieces of Q, K and V after the work list; bf16 inputs
    need the work list only."""
    p = lib.mesh_attn_plan_create(16384, 16, True)
    base = lib.mesh_attn_workspace_size(p)
    assert lib.mesh_attn_workspace_size_for(p, lib.torch.bfloat16, 1, 16, 4, 128) == base
    up = lambda x: (x + 255) // 256 * 256
    q, kv = 3 * 16 * 16384 * 128 * 2, 3 * 4 * 16384 * 128 * 2
    assert lib.mesh_attn_workspace_size_for(p, lib.torch.float32, 1, 16, 4, 128) == up(base) + up(q) + 2 * up(kv)
    fake = ctypes.c_void_p(1 << 20)
    so = lib._lib
    # an fp32 call with only the bf16-sized workspace is refused before anything is enqueued
    assert so.mesh_attn_tile_fwd(p.handle, 0, 1, 16, 4, 128, fake, fake, fake, 0.1, fake, fake, fake, base, fake,
                                 None) == 9


@pytest.mark.parametrize("P", [1, 4, 16, 64, 256])
@pytest.mark.parametrize("causal,kvr,greedy", list(itertools.product([0, 1], repeat=3)))
def test_launch_order_keeps_each_device_sequence(lib, P, causal, kvr, greedy):
    """The kernels take the work items tile after tile (row-major over the mesh), each tile's
    items in that virtual device's order from the plan: a permutation of the plan's items whose
    tiles never decrease and whose positions in the plan's order increase within a tile."""
    S = 64 * P
    plan = lib.mesh_attn_plan_create(S, P, causal, kvr, greedy)
    items, steps, _ = lib.mesh_attn_plan_order(plan)
    order = lib.mesh_attn_plan_launch_order(plan)
    assert sorted(order) == list(range(len(items)))
    tiles = [items[i][1] for i in order]
    assert tiles == sorted(tiles)
    for a, b in zip(order, order[1:]):
        if items[a][1] == items[b][1]:
            assert a < b and steps[a] <= steps[b]


@pytest.mark.parametrize("P", [1, 5, 16])
def test_launch_order_of_ring_plan_is_its_order(lib, P):
    plan = lib.mesh_attn_plan_create_ring(32 * P, P, True)
    assert lib.mesh_attn_plan_launch_order(plan) == list(range(P))
