"""The no-allocation tile forward against the workspace entry point and the oracle.

mesh_attn_tile_fwd_noalloc serves callers that may not call cudaMalloc -- code running under a
framework whose caching allocator already owns the device memory, inside allocator callbacks,
or under a fixed memory budget -- and therefore cannot hand the library a workspace.  It keeps
the plan's work list in one fixed device array inside the library instead.  It runs the same
kernel on the same inputs as mesh_attn_tile_fwd, and every work item is computed by one CTA in
a fixed order, so its partial outputs must equal the workspace entry point's bit for bit.  Two
calls in a row with different plans show that each call rewrites everything the kernel reads
from that shared array.

This file is collected last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from mesh_inputs import Workload, make_qkv
from tests.gpu_helpers import check_partials

pytestmark = pytest.mark.gpu

CASES = [
    Workload(130, "noalloc_gqa_causal", 1, 4, 2, 4096, 128, "bf16", True, 16),
    Workload(131, "noalloc_ragged", 1, 2, 1, 800, 128, "bf16", False, 4),
    Workload(132, "noalloc_f32_pieces_in_scratch", 1, 2, 2, 512, 64, "f32", True, 4),
]


def test_noalloc_matches_workspace_entry_point(lib):
    for i, w in enumerate(CASES):  # calls in a row, different plans sharing the one scratch array
        q, k, v = make_qkv(w)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
        ref_o, ref_l = lib.new_partials(plan, w.B, w.Hq, w.d)
        ws = lib.new_workspace(plan, "cuda", qd, kd)
        st_ref = lib.new_status()
        lib.mesh_attn_tile_fwd(plan, qd, kd, vd, None, ref_o, ref_l, ws, st_ref)
        out_o, out_l = lib.new_partials(plan, w.B, w.Hq, w.d)
        out_o.fill_(float("nan"))  # a slot the call never writes stays NaN and fails the comparison
        out_l.fill_(float("nan"))
        st = lib.new_status()
        lib.mesh_attn_tile_fwd_noalloc(plan, qd, kd, vd, None, out_o, out_l, st)
        assert lib.mesh_attn_read_status(st_ref) == 0
        assert lib.mesh_attn_read_status(st) == 0, st.tolist()
        n_o, n_l = lib.mesh_attn_partials_size(plan, w.B, w.Hq, w.d)
        assert torch.equal(out_o[:n_o], ref_o[:n_o]), w.name
        assert torch.equal(out_l[:n_l], ref_l[:n_l]), w.name
        if i == 0:  # and directly against the oracle, slot by slot
            check_partials(lib, w, plan, out_o, out_l, q, k, v)


def test_noalloc_rejects_plans_beyond_its_scratch(lib):
    """P = 4096 causal needs more than MESH_ATTN_NOALLOC_SCRATCH_BYTES of work list.  The call gets
    B = 0 and NULL tensor pointers: the scratch-size check comes first and must answer
    MESH_ATTN_ERR_WORKSPACE; should it ever be skipped, the call would end at the empty-batch
    return or the NULL check without launching anything."""
    plan = lib.mesh_attn_plan_create(4096 * 8, 4096, True)
    st = lib.new_status()
    rc = lib._lib.mesh_attn_tile_fwd_noalloc(plan.handle, 1, 0, 1, 1, 128, None, None, None, 0.125, None, None,
                                             ctypes.c_void_p(st.data_ptr()), None)
    assert rc == 9
    assert "at most" in lib._lib.mesh_attn_last_error().decode()
    assert lib.mesh_attn_read_status(st) == 0
