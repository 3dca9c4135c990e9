"""The autograd binding: gradients from loss.backward() equal the explicit backward call on the
same dO, bit for bit (the same kernels on the same inputs), for bf16 and fp32 inputs."""
import pytest
import torch

from mesh_inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

CASES = [
    Workload(170, "autograd_bf16_gqa_causal", 1, 4, 2, 1024, 128, "bf16", True, 4),
    Workload(171, "autograd_f32_d64", 2, 2, 2, 512, 64, "f32", False, 4),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_autograd_matches_explicit_backward(lib, w):
    q, k, v = (t.cuda() for t in make_qkv(w))
    qg, kg, vg = (t.clone().requires_grad_(True) for t in (q, k, v))
    O, LSE = lib.mesh_attention_autograd(qg, kg, vg, w.P, w.causal, w.kvr, w.greedy)
    assert not LSE.requires_grad
    g = torch.Generator(device="cpu").manual_seed(w.cfg_id)
    W = torch.randn(O.shape, generator=g, dtype=torch.float32).cuda()
    (O.float() * W).sum().backward()
    dO = W.to(O.dtype)  # the gradient autograd hands to the attention output
    O2, LSE2 = lib.mesh_attention(q, k, v, w.P, w.causal, w.kvr, w.greedy)
    assert torch.equal(O.detach(), O2) and torch.equal(LSE, LSE2)
    dQ, dK, dV = lib.mesh_attention_backward(q, k, v, O2, LSE2, dO, w.P, w.causal, w.kvr, w.greedy)
    for got, ref in ((qg.grad, dQ), (kg.grad, dK), (vg.grad, dV)):
        assert got.dtype == ref.dtype and got.shape == ref.shape
        assert torch.equal(got, ref)
