"""The no-allocation tile forward against the workspace entry point.

mesh_attn_tile_fwd_noalloc serves callers that may not call cudaMalloc -- code running under a
framework whose caching allocator already owns the device memory, inside allocator callbacks,
or under a fixed memory budget -- and therefore cannot hand the library a workspace.  It keeps
the plan's work list in one fixed device array inside the library instead, and must produce
exactly what mesh_attn_tile_fwd produces.  Two calls in a row with different plans show that
each call rewrites everything the kernel reads from that shared array.

This file is collected last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from mesh_inputs import Workload, make_qkv
from tests.gpu_helpers import TOL, max_err

pytestmark = pytest.mark.gpu

CASES = [
    Workload(130, "noalloc_gqa_causal", 1, 4, 2, 4096, 128, "bf16", True, 16),
    Workload(131, "noalloc_ragged", 1, 2, 1, 800, 128, "bf16", False, 4),
    Workload(132, "noalloc_f32_pieces_in_scratch", 1, 2, 2, 512, 64, "f32", True, 4),
]


def test_noalloc_matches_workspace_entry_point(lib):
    for w in CASES:  # two calls in a row, different plans sharing the one scratch array
        q, k, v = (t.cuda() for t in make_qkv(w))
        plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
        ref_o, ref_l = lib.new_partials(plan, w.B, w.Hq, w.d)
        ws = lib.new_workspace(plan, "cuda", q, k)
        st_ref = lib.new_status()
        lib.mesh_attn_tile_fwd(plan, q, k, v, None, ref_o, ref_l, ws, st_ref)
        out_o, out_l = lib.new_partials(plan, w.B, w.Hq, w.d)
        out_o.fill_(float("nan"))
        out_l.fill_(float("nan"))
        st = lib.new_status()
        lib.mesh_attn_tile_fwd_noalloc(plan, q, k, v, None, out_o, out_l, st)
        assert lib.mesh_attn_read_status(st_ref) == 0
        assert lib.mesh_attn_read_status(st) == 0, st.tolist()
        n_o, n_l = lib.mesh_attn_partials_size(plan, w.B, w.Hq, w.d)
        tol_o, tol_l = TOL[w.dtype]
        assert max_err(out_o[:n_o], ref_o[:n_o]) <= tol_o
        assert max_err(out_l[:n_l], ref_l[:n_l]) <= tol_l


def test_noalloc_rejects_plans_beyond_its_scratch(lib):
    """P = 4096 causal needs more than MESH_ATTN_NOALLOC_SCRATCH_BYTES of work list."""
    plan = lib.mesh_attn_plan_create(4096 * 8, 4096, True)
    st = lib.new_status()
    fake = ctypes.c_void_p(1 << 20)
    rc = lib._lib.mesh_attn_tile_fwd_noalloc(plan.handle, 1, 1, 1, 1, 128, fake, fake, fake, 0.125, fake, fake,
                                             ctypes.c_void_p(st.data_ptr()), None)
    assert rc == 9
    assert "at most" in lib._lib.mesh_attn_last_error().decode()
    assert lib.mesh_attn_read_status(st) == 0
