"""GPU parity: the C-ABI path (planner, tile kernels, merge) against the fp64 oracle on the
same seeded inputs, element by element.

Small cases span several 128-row tiles, ragged partitions (L not a multiple of 128, an odd
number of query tiles), GQA, batch > 1, causal and non-causal masks and every plan variant;
each also checks every partial slot.  The full-size workloads are compared on 4096 seeded
rows per head.
"""
import math

import pytest
import torch

from mesh_inputs import WORKLOADS, Workload, make_qkv, sample_rows
from tests.gpu_helpers import TOL, check_full, check_partials, check_sampled, max_err, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    WORKLOADS["tiny_f32"],
    Workload(101, "bf16_L128_causal", 1, 2, 2, 2048, 128, "bf16", True, 16),
    Workload(102, "bf16_gqa4_L1024_causal", 1, 4, 1, 4096, 128, "bf16", True, 4),
    Workload(103, "bf16_ragged_L200", 1, 2, 1, 800, 128, "bf16", False, 4),
    Workload(104, "bf16_ragged_L200_causal", 1, 2, 1, 800, 128, "bf16", True, 4),
    Workload(105, "bf16_oddtiles_L384_d64", 1, 2, 2, 3456, 64, "bf16", True, 9),
    Workload(106, "bf16_batch2", 2, 2, 2, 1024, 128, "bf16", False, 4),
    Workload(107, "f32_ragged_L100_causal", 1, 2, 1, 900, 128, "f32", True, 9),
    Workload(108, "bf16_peaked_k4", 1, 2, 1, 4096, 128, "bf16", True, 16, k_scale=4.0),
    Workload(109, "bf16_single_partition", 1, 1, 1, 640, 128, "bf16", True, 1),
    Workload(111, "bf16_one_token_partitions", 1, 2, 1, 16, 128, "bf16", True, 16),
    Workload(112, "bf16_tiny_partitions_L8", 1, 2, 2, 512, 128, "bf16", True, 64),
    Workload(113, "bf16_batch2_gqa_ragged_causal", 2, 4, 2, 800, 128, "bf16", True, 4),
    Workload(114, "bf16_mqa_32_heads", 1, 32, 1, 1024, 128, "bf16", True, 4),
    Workload(115, "f32_gqa_d64", 1, 4, 2, 765, 64, "f32", False, 9),
    Workload(116, "bf16_noncausal_d64_L1000", 1, 2, 1, 4000, 64, "bf16", False, 4),
    # fp32 inputs through the same edge cases: batch, GQA and ragged partitions together; MQA at
    # d = 64; partitions of 8 and of 1 token, where one softmax warp of each row holds no key
    Workload(119, "f32_batch2_gqa_ragged_causal", 2, 4, 2, 800, 128, "f32", True, 4),
    Workload(120, "f32_mqa_8_heads_d64", 1, 8, 1, 1024, 64, "f32", True, 4),
    Workload(121, "f32_tiny_partitions_L8", 1, 2, 2, 512, 128, "f32", True, 64),
    Workload(122, "f32_one_token_partitions", 1, 2, 1, 16, 128, "f32", True, 16),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_against_oracle(lib, w):
    q, k, v = make_qkv(w)
    O, LSE, po, pl, plan = run_gpu(lib, w, q, k, v)
    assert O.dtype == q.dtype and LSE.dtype == torch.float32
    check_full(w, O, LSE, q, k, v)
    check_partials(lib, w, plan, po, pl, q, k, v)


@pytest.mark.parametrize("kvr,greedy", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("name", ["bf16_L128_causal", "bf16_ragged_L200_causal"])
def test_plan_variants_agree(lib, name, kvr, greedy):
    """KVR on/off and greedy on/off change the tiles and the order, not the result."""
    w = next(x for x in SMALL if x.name == name)
    q, k, v = make_qkv(w)
    O, LSE, po, pl, plan = run_gpu(lib, w, q, k, v, kvr=bool(kvr), greedy=bool(greedy))
    check_full(w, O, LSE, q, k, v)
    check_partials(lib, w, plan, po, pl, q, k, v)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("ramp", [6.0, -0.9])
def test_growing_and_shrinking_scores(lib, ramp, causal):
    """Keys scaled by a ramp along the sequence.  Growing: the row maximum rises block after
    block, so the running reference of the online softmax is raised (and O and l rescaled) many
    times inside one work unit.  Shrinking: the first block holds the maximum and later blocks
    only add small terms.  The growing ramp makes attention so peaked that O is close to single
    rows of V, and with |V| up to 4.7 the two roundings the bf16 path makes add up past the
    absolute 2e-2: O rounded to bf16 (half an ulp, 2^-6 for |O| in [4, 8)) plus P rounded to
    bf16 in the PV product (2^-9 of the second-largest weight times |V|); unscaled the worst row
    measures 2.11e-2.  V is scaled by 1/4 (exact in bf16), which scales both roundings by 1/4,
    while a wrong rescale factor would still be off by O(|O|)."""
    w = Workload(117, "bf16_ramp", 1, 2, 1, 4096, 128, "bf16", causal, 4)
    q, k, v = make_qkv(w)
    ramp_k = 1.0 + ramp * torch.arange(w.S, dtype=torch.float32) / w.S
    k = (k.float() * ramp_k[None, None, :, None]).to(k.dtype)
    v = v * 0.25
    O, LSE, po, pl, plan = run_gpu(lib, w, q, k, v)
    check_full(w, O, LSE, q, k, v)
    check_partials(lib, w, plan, po, pl, q, k, v)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("ramp", [6.0, -0.9])
def test_growing_and_shrinking_scores_f32(lib, ramp, causal):
    """The same ramps with fp32 inputs, at the fp32 tolerance and with V unscaled: the growing
    ramp raises the running reference (and rescales O and l) many times per unit, which in the
    fp32 kernel the two softmax warps of each row decide together from their swapped half-row
    maxima, each rescaling its half of O.  Scores reach ~35 here, so fp32 accumulation of the
    score's 768 piece products is what the LSE error measures (about 1e-5)."""
    w = Workload(118, "f32_ramp", 1, 2, 1, 4096, 128, "f32", causal, 4)
    q, k, v = make_qkv(w)
    ramp_k = 1.0 + ramp * torch.arange(w.S, dtype=torch.float32) / w.S
    k = k * ramp_k[None, None, :, None]
    O, LSE, po, pl, plan = run_gpu(lib, w, q, k, v)
    check_full(w, O, LSE, q, k, v)
    check_partials(lib, w, plan, po, pl, q, k, v)


def test_closed_forms_on_gpu(lib):
    """Constant V gives O = V; causal row 0 gives O_0 = V_0 and LSE_0 = scale q_0 . k_0; equal
    keys give the mean of the visible values and LSE = ln(count) + score."""
    w = Workload(110, "closed", 1, 2, 1, 1024, 128, "bf16", True, 4)
    q, k, v = make_qkv(w)
    vc = torch.full_like(v, 0.375)
    O, LSE, *_ = run_gpu(lib, w, q, k, vc)
    assert max_err(O, vc.expand(1, 2, 1024, 128)) <= 1e-6
    O, LSE, *_ = run_gpu(lib, w, q, k, v)
    for h in range(2):
        assert torch.equal(O[0, h, 0].cpu(), v[0, 0, 0])
        s0 = (q[0, h, 0].double() @ k[0, 0, 0].double()).item() / math.sqrt(128)
        assert abs(LSE[0, h, 0].item() - s0) <= 1e-4
    ke = k[:, :, :1].expand_as(k).contiguous()
    O, LSE, *_ = run_gpu(lib, w, q, ke, v)
    csum = v[0, 0].double().cumsum(0) / torch.arange(1, 1025, dtype=torch.float64)[:, None]
    s = (q[0].double() @ k[0, 0, 0].double()) / math.sqrt(128)
    for h in range(2):
        assert max_err(O[0, h], csum) <= 2e-2
        assert max_err(LSE[0, h], torch.log(torch.arange(1, 1025, dtype=torch.float64)) + s[h]) <= 1e-3


FULL = ["bf16_causal_16k", "gqa_causal_64k", "long_128k", "long_128k_causal", "stress_256k", "long_1m_causal"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(lib, name):
    """The full-size workloads, in the launch configuration the benchmark times, on 4096 seeded
    sampled query rows per head (forced rows: 0, S-1, first/last of partitions 0, 1, P/2, P-1)."""
    w = WORKLOADS[name]
    plan = lib.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
    no, nl = lib.mesh_attn_partials_size(plan, w.B, w.Hq, w.d)
    need = 4 * (no + nl) + 2 * (2 * w.B * w.Hq * w.S * w.d + 2 * w.B * w.Hkv * w.S * w.d)
    free, _ = torch.cuda.mem_get_info()
    if need > free * 0.9:
        pytest.skip(f"needs about {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} GiB free")
    q, k, v = make_qkv(w)
    O, LSE, po, pl, plan = run_gpu(lib, w, q, k, v)
    del po, pl
    rows = sample_rows(w)
    check_sampled(w, O, LSE, q, k, v, rows)
    # causal row 0 closed form on every head
    if w.causal:
        g = w.Hq // w.Hkv
        for h in range(w.Hq):
            assert torch.equal(O[0, h, 0].cpu(), v[0, h // g, 0])


@pytest.mark.parametrize("name", ["bf16_causal_16k", "gqa_causal_64k"])
def test_full_size_f32_sampled_rows(lib, name):
    """The fp32 tensor-core path (three-piece split, six products, two S buffers) at full size:
    the 16K causal and 64K GQA causal shapes with fp32 inputs, on 4096 sampled query rows per
    head at the fp32 tolerance.  A unit here runs up to 128 key blocks of 64 keys (a 1,024-row
    partition against up to 8 KV partitions), so the block pipeline, the K/V stage rings and the
    running-maximum rescale all go round many times."""
    w = WORKLOADS[name]
    w = w.with_(dtype="f32", name=w.name + "_f32")
    q, k, v = make_qkv(w)
    O, LSE, po, pl, plan = run_gpu(lib, w, q, k, v)
    del po, pl
    check_sampled(w, O, LSE, q, k, v, sample_rows(w))
    # causal row 0 sees key 0 alone: O = V[0] up to the fp32 accumulation of its three pieces
    g = w.Hq // w.Hkv
    for h in range(w.Hq):
        assert torch.allclose(O[0, h, 0].cpu(), v[0, h // g, 0], rtol=0, atol=1e-6)


@pytest.mark.parametrize("name", ["tiny_f32", "bf16_L128_causal", "bf16_ragged_L200", "bf16_gqa4_L1024_causal"])
def test_ring_plan_through_kernels(lib, name):
    """Ring-Attention's row assignment (one slot per Q partition holding every live KV partition)
    through the same tile and merge kernels gives the same attention."""
    w = next(x for x in SMALL if x.name == name)
    q, k, v = make_qkv(w)
    plan = lib.mesh_attn_plan_create_ring(w.S, w.P, w.causal)
    O, LSE, po, pl = lib.mesh_attention(q.cuda(), k.cuda(), v.cuda(), w.P, w.causal, plan=plan, return_partials=True)
    torch.cuda.synchronize()
    check_full(w, O, LSE, q, k, v)
    check_partials(lib, w, plan, po, pl, q, k, v)
