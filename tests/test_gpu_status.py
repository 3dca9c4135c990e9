"""Device-side failure reporting without a GPU fault.

The wait limit is set to 0 so every device wait that is not already satisfied gives up at
once: the tile kernel must record MESH_ATTN_ERR_DEVICE_TIMEOUT in the status block, drain its
copies, free its tensor memory and return.  Later kernels see the non-zero status and skip
their work.  After clearing the status and restoring the limit, the same context computes
correct results again.
"""
import pytest
import torch

from mesh_inputs import Workload, make_qkv
from tests.gpu_helpers import check_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_wait_timeout_reports_status_and_context_survives(lib, dtype):
    """Both forward kernels; in the fp32 one the waits include the per-block swap of half-row
    maxima between the two softmax warps of a row, which must give up as the others do."""
    w = Workload(120, "status", 1, 2, 1, 2048, 128, dtype, True, 4)
    q, k, v = make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, True, True)
    po, pl = lib.new_partials(plan, 1, 2, 128)
    ws = lib.new_workspace(plan, "cuda", qd, kd)
    st = lib.new_status()
    O = torch.full_like(qd, 7.0)
    LSE = torch.full((1, 2, w.S), 7.0, device="cuda")
    lib.mesh_attn_set_wait_limit_ns(0)
    try:
        lib.mesh_attn_tile_fwd(plan, qd, kd, vd, None, po, pl, ws, st)
        code = lib.mesh_attn_read_status(st)
    finally:
        lib.mesh_attn_set_wait_limit_ns(2_000_000_000)
    assert code == 5, f"status block {st.tolist()}"
    assert st[1].item() in (1, 2, 3, 5)  # softmax, MMA, load or relay role gave up
    # a set status makes later kernels skip their work
    lib.mesh_attn_merge(plan, 1, 2, 128, po, pl, O, LSE, ws, st)
    assert lib.mesh_attn_read_status(st) == 5
    assert bool((O == 7.0).all()) and bool((LSE == 7.0).all())
    # the context is still usable
    st.zero_()
    lib.mesh_attn_tile_fwd(plan, qd, kd, vd, None, po, pl, ws, st)
    lib.mesh_attn_merge(plan, 1, 2, 128, po, pl, O, LSE, ws, st)
    assert lib.mesh_attn_read_status(st) == 0
    check_full(w, O, LSE, q, k, v)


def test_empty_and_degenerate_launches(lib):
    """B = 0, Hq = 0 and an empty sequence enqueue nothing and leave outputs untouched."""
    plan = lib.mesh_attn_plan_create(0, 4, True)
    st = lib.new_status()
    O = torch.full((1, 2, 0, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((1, 2, 0), device="cuda")
    ws = lib.new_workspace(plan)
    po, pl = lib.new_partials(plan, 1, 2, 128)
    q = torch.zeros((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    lib.mesh_attn_tile_fwd(plan, q, q[:, :1], q[:, :1], None, po, pl, ws, st)
    lib.mesh_attn_merge(plan, 1, 2, 128, po, pl, O, LSE, ws, st)
    assert lib.mesh_attn_read_status(st) == 0


def test_backward_wait_timeout_reports_status_and_context_survives(lib):
    """The tensor-core backward kernels under a zero wait limit: status DEVICE_TIMEOUT, the reduce
    skips its work, and after a reset the same context produces correct gradients."""
    from mesh_inputs import make_do
    from tests.test_gpu_backward import check_gradients
    w = Workload(121, "status_bwd", 1, 2, 1, 2048, 128, "bf16", True, 4)
    q, k, v = make_qkv(w)
    dO = make_do(w)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, True, True)
    O, LSE = lib.mesh_attention(qd, kd, vd, w.P, w.causal, plan=plan)
    dq_p, dk_p, dv_p = lib.new_bwd_partials(plan, 1, 2, 1, 128)
    ws = lib.new_bwd_workspace(plan)
    st = lib.new_status()
    D = torch.empty(1, 2, w.S, device="cuda")
    dQ, dK, dV = (torch.full_like(t, 7.0) for t in (qd, kd, vd))
    lib.mesh_attn_bwd_prep(O, dod, D, st)
    lib.mesh_attn_set_wait_limit_ns(0)
    try:
        lib.mesh_attn_tile_bwd(plan, qd, kd, vd, dod, LSE, D, None, dq_p, dk_p, dv_p, ws, st)
        code = lib.mesh_attn_read_status(st)
    finally:
        lib.mesh_attn_set_wait_limit_ns(2_000_000_000)
    assert code == 5, f"status block {st.tolist()}"
    assert st[1].item() in (1, 2, 3)
    lib.mesh_attn_bwd_reduce(plan, 1, 2, 1, 128, dq_p, dk_p, dv_p, dQ, dK, dV, ws, st)
    assert lib.mesh_attn_read_status(st) == 5
    assert bool((dQ == 7.0).all()) and bool((dK == 7.0).all()) and bool((dV == 7.0).all())
    st.zero_()
    got = lib.mesh_attention_backward(qd, kd, vd, O, LSE, dod, w.P, w.causal, plan=plan)
    check_gradients(w, got, q, k, v, dO)
