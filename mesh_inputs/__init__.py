"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds the workload table and the random draws only.  It contains none
of the attention arithmetic, imports neither the oracle nor the CUDA binding, and
is the one piece of code both sides of a parity test may share.

Workloads are the long-context shapes of the Mesh-Attention write-ups ("Mesh-Attention:
A New Communication-Efficient Distributed Attention with Improved Data Locality",
abstract: 1M-token sequences on clusters; no dataset is named), restated as five
single-GPU configurations.  Inputs are i.i.d. N(0, 1) draws from NumPy's PCG64,
seeded with ``SeedSequence([20251224, cfg_id, tensor_id])`` where tensor_id is
Q=0, K=1, V=2, the sampled-row stream 3 and the backward pass's upstream gradient
dO 4.  bf16 inputs are the float32 draw rounded to nearest even.  The stress workload
multiplies K by 4 after rounding, which is exact in bf16 (a power of two).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

SEED_ROOT = 20251224
TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_ROWS, TENSOR_DO = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, masking and the mesh it is planned on."""

    cfg_id: int
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    d: int
    dtype: str  # "f32" or "bf16"
    causal: bool
    P: int
    kvr: bool = True
    greedy: bool = True
    k_scale: float = 1.0
    sampled_rows: Optional[int] = None  # None: every row is checked

    @property
    def L(self) -> int:
        return self.S // self.P

    @property
    def R(self) -> int:
        return int(round(self.P ** 0.5))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five single-GPU configurations (tiny exact check, bf16 causal, GQA causal,
# long context, merge-heavy stress).
WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload(1, "tiny_f32", 1, 2, 2, 512, 64, "f32", False, 4),
    "bf16_causal_16k": Workload(2, "bf16_causal_16k", 1, 16, 16, 16384, 128, "bf16", True, 16,
                                sampled_rows=4096),
    "gqa_causal_64k": Workload(3, "gqa_causal_64k", 1, 32, 8, 65536, 128, "bf16", True, 64,
                               sampled_rows=4096),
    "long_128k": Workload(4, "long_128k", 1, 32, 8, 131072, 128, "bf16", False, 256,
                          sampled_rows=4096),
    "long_128k_causal": Workload(4, "long_128k_causal", 1, 32, 8, 131072, 128, "bf16", True, 256,
                                 sampled_rows=4096),
    "stress_256k": Workload(5, "stress_256k", 1, 16, 4, 262144, 128, "bf16", True, 1024,
                            k_scale=4.0, sampled_rows=4096),
    # a profiling-size slice of the stress workload: the same partition length (256 tokens),
    # GQA group (4), K scaling and mask, with a quarter of the sequence and half of the heads,
    # so that a replayed counter capture holds about 4 GB on the device
    "stress_64k": Workload(6, "stress_64k", 1, 8, 2, 65536, 128, "bf16", True, 256,
                           k_scale=4.0, sampled_rows=4096),
    # the 1M-token sequence length the pages measure across GPUs, on one GPU: 8 query heads and
    # 2 KV heads so that its fp32 partials (32,272 slots of 1,024 rows, 136 GB) fit in HBM
    "long_1m_causal": Workload(7, "long_1m_causal", 1, 8, 2, 1048576, 128, "bf16", True, 1024,
                               sampled_rows=1024),
}


def _rng(cfg_id: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([SEED_ROOT, cfg_id, tensor_id])))


def normal_tensor(cfg_id: int, tensor_id: int, shape, dtype: str, scale: float = 1.0) -> torch.Tensor:
    """N(0,1) draw of `shape` from the (cfg_id, tensor_id) stream, as a CPU tensor.

    The draw is made slice by slice along the first axes so that large tensors never
    hold a second full-size float32 copy; the values do not depend on the slicing.
    """
    rng = _rng(cfg_id, tensor_id)
    tdtype = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    out = torch.empty(shape, dtype=tdtype)
    flat = out.view(-1, shape[-1])
    rows_per_chunk = max(1, (1 << 24) // shape[-1])
    for r0 in range(0, flat.shape[0], rows_per_chunk):
        r1 = min(flat.shape[0], r0 + rows_per_chunk)
        x = rng.standard_normal((r1 - r0, shape[-1]), dtype=np.float32)
        t = torch.from_numpy(x).to(tdtype)
        if scale != 1.0:
            t = t * scale
        flat[r0:r1] = t
    return out


def make_qkv(w: Workload, seed_offset: int = 0):
    """Q [B,Hq,S,d], K and V [B,Hkv,S,d] as CPU tensors of the workload's dtype."""
    cid = w.cfg_id + 1000 * seed_offset
    q = normal_tensor(cid, TENSOR_Q, (w.B, w.Hq, w.S, w.d), w.dtype)
    k = normal_tensor(cid, TENSOR_K, (w.B, w.Hkv, w.S, w.d), w.dtype, scale=w.k_scale)
    v = normal_tensor(cid, TENSOR_V, (w.B, w.Hkv, w.S, w.d), w.dtype)
    return q, k, v


def make_do(w: Workload, seed_offset: int = 0) -> torch.Tensor:
    """The upstream gradient dO [B,Hq,S,d] of the backward pass: N(0,1) in the workload's dtype."""
    cid = w.cfg_id + 1000 * seed_offset
    return normal_tensor(cid, TENSOR_DO, (w.B, w.Hq, w.S, w.d), w.dtype)


def forced_rows(S: int, P: int) -> List[int]:
    """Rows always checked: 0, S-1 and the first and last row of partitions 0, 1, P/2, P-1."""
    L = S // P
    rows = {0, S - 1}
    for p in {0, min(1, P - 1), P // 2, P - 1}:
        rows.add(p * L)
        rows.add(p * L + L - 1)
    return sorted(r for r in rows if 0 <= r < S)


def sample_rows(w: Workload, n: Optional[int] = None) -> np.ndarray:
    """Sorted distinct query rows per (b, h): int64 array [B, Hq, n].

    Each head gets its own draw from the rows stream: the forced rows plus rows drawn
    uniformly without replacement from the rest.  With n >= S every row is returned.
    """
    n = w.sampled_rows if n is None else n
    if n is None or n >= w.S:
        base = np.arange(w.S, dtype=np.int64)
        return np.broadcast_to(base, (w.B, w.Hq, w.S)).copy()
    rng = _rng(w.cfg_id, TENSOR_ROWS)
    forced = np.array(forced_rows(w.S, w.P), dtype=np.int64)
    out = np.empty((w.B, w.Hq, n), dtype=np.int64)
    mask = np.ones(w.S, dtype=bool)
    mask[forced] = False
    pool = np.nonzero(mask)[0]
    for b in range(w.B):
        for h in range(w.Hq):
            extra = rng.choice(pool, size=n - len(forced), replace=False)
            out[b, h] = np.sort(np.concatenate([forced, extra]))
    return out
