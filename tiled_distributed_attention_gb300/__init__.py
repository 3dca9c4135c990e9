"""Python binding of libmesh_attn.so, the single-GPU Mesh-Attention hot path for sm_103a.

Argument marshalling only: every step of the computation (tile map, greedy order, tile
attention, LSE merge) runs in the C++ planner and the CUDA kernels behind the C ABI declared
in include/mesh_attn.h.  The functions carry the same names as the C entry points.  PyTorch
supplies device memory and streams; nothing here computes attention, and there is no CPU
fallback: if the library is missing, load_library() raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmesh_attn.so")

MESH_ATTN_OK = 0
MESH_ATTN_F32 = 0
MESH_ATTN_BF16 = 1
MESH_ATTN_STATUS_WORDS = 4
STATUS_NAMES = {
    0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_MISALIGNED", 4: "ERR_CUDA",
    5: "ERR_DEVICE_TIMEOUT", 6: "ERR_OUT_OF_RANGE", 7: "ERR_INTERNAL", 8: "ERR_NO_MEMORY",
    9: "ERR_WORKSPACE",
}

_lib: Optional[ctypes.CDLL] = None

c_i32, c_i64, c_sz, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
P_i32 = ctypes.POINTER(c_i32)
P_i64 = ctypes.POINTER(c_i64)
P_sz = ctypes.POINTER(c_sz)


class PlanInfo(ctypes.Structure):
    _fields_ = [("S", c_i64), ("L", c_i64), ("P", c_i32), ("R", c_i32), ("causal", c_i32), ("kvr", c_i32),
                ("greedy", c_i32), ("n_slots", c_i32), ("n_steps", c_i32), ("layout", c_i32), ("tile_q", c_i32),
                ("tile_kv", c_i32), ("n_kv_entries", c_i64), ("n_live_blocks", c_i64), ("n_kv_slots", c_i32),
                ("reserved", c_i32)]


_SIGS = {
    "mesh_attn_plan_create": (c_i32, [c_i64, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_vp)]),
    "mesh_attn_plan_create_ring": (c_i32, [c_i64, c_i32, c_i32, ctypes.POINTER(c_vp)]),
    "mesh_attn_plan_destroy": (c_i32, [c_vp]),
    "mesh_attn_plan_get_info": (c_i32, [c_vp, ctypes.POINTER(PlanInfo)]),
    "mesh_attn_plan_tiles": (c_i32, [c_vp, P_i32, P_i32]),
    "mesh_attn_plan_slots": (c_i32, [c_vp, P_i32]),
    "mesh_attn_plan_order": (c_i32, [c_vp, P_i32, P_i32, P_i32, P_i32]),
    "mesh_attn_plan_volumes": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, P_i32, P_i64, P_i64]),
    "mesh_attn_plan_launch_order": (c_i32, [c_vp, P_i32]),
    "mesh_attn_partials_size": (c_i32, [c_vp, c_i32, c_i32, c_i32, P_sz, P_sz]),
    "mesh_attn_workspace_size": (c_i32, [c_vp, P_sz]),
    "mesh_attn_workspace_size_for": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, P_sz]),
    "mesh_attn_tile_fwd": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_f32, c_vp, c_vp,
                                   c_vp, c_sz, c_vp, c_vp]),
    "mesh_attn_tile_fwd_noalloc": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_f32, c_vp,
                                           c_vp, c_vp, c_vp]),
    "mesh_attn_merge": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "mesh_attn_plan_kv_slots": (c_i32, [c_vp, P_i32, P_i32, P_i32, P_i32]),
    "mesh_attn_bwd_partials_size": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, P_sz, P_sz]),
    "mesh_attn_bwd_workspace_size": (c_i32, [c_vp, P_sz]),
    "mesh_attn_bwd_prep": (c_i32, [c_i32, c_i32, c_i32, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "mesh_attn_tile_bwd": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                   c_f32, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "mesh_attn_bwd_reduce": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                     c_vp, c_sz, c_vp, c_vp]),
    "mesh_attn_read_status": (c_i32, [c_vp, c_vp, P_i32]),
    "mesh_attn_status_string": (ctypes.c_char_p, [c_i32]),
    "mesh_attn_last_error": (ctypes.c_char_p, []),
    "mesh_attn_set_wait_limit_ns": (c_i32, [c_i64]),
}


class MeshAttnError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmesh_attn.so (built by __graft_entry__.build()) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != MESH_ATTN_OK:
        msg = _lib.mesh_attn_last_error().decode()
        raise MeshAttnError(code, where, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return MESH_ATTN_BF16
    if dt == torch.float32:
        return MESH_ATTN_F32
    raise TypeError(f"unsupported dtype {dt}: use torch.bfloat16 or torch.float32")


class Plan:
    """Owning handle of a mesh_attn_plan (host memory, immutable)."""

    def __init__(self, handle: ctypes.c_void_p):
        self._h = handle
        info = PlanInfo()
        _check(_lib.mesh_attn_plan_get_info(self._h, ctypes.byref(info)), "mesh_attn_plan_get_info")
        self.info = info

    @property
    def handle(self):
        return self._h

    def __getattr__(self, name):
        if name in ("S", "L", "P", "R", "causal", "kvr", "greedy", "n_slots", "n_steps", "n_kv_entries",
                    "n_live_blocks", "layout", "tile_q", "tile_kv", "n_kv_slots"):
            return getattr(self.__dict__["info"], name)
        raise AttributeError(name)

    def close(self):
        if self._h is not None and _lib is not None:
            _lib.mesh_attn_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _i32(n: int):
    return (c_i32 * max(n, 1))()


def mesh_attn_plan_create(S: int, P: int, causal: bool, kvr: bool = True, greedy: bool = True) -> Plan:
    load_library()
    h = c_vp()
    _check(_lib.mesh_attn_plan_create(S, P, int(causal), int(kvr), int(greedy), ctypes.byref(h)),
           "mesh_attn_plan_create")
    return Plan(h)


def mesh_attn_plan_create_ring(S: int, P: int, causal: bool) -> Plan:
    load_library()
    h = c_vp()
    _check(_lib.mesh_attn_plan_create_ring(S, P, int(causal), ctypes.byref(h)), "mesh_attn_plan_create_ring")
    return Plan(h)


def mesh_attn_plan_tiles(plan: Plan):
    a, b = plan.tile_q, plan.tile_kv
    q, kv = _i32(plan.P * a), _i32(plan.P * b)
    _check(_lib.mesh_attn_plan_tiles(plan.handle, q, kv), "mesh_attn_plan_tiles")
    return ([list(q[t * a:(t + 1) * a]) for t in range(plan.P)], [list(kv[t * b:(t + 1) * b]) for t in range(plan.P)])


def mesh_attn_plan_slots(plan: Plan):
    off = _i32(plan.P + 1)
    _check(_lib.mesh_attn_plan_slots(plan.handle, off), "mesh_attn_plan_slots")
    return list(off[:plan.P + 1])


def mesh_attn_plan_order(plan: Plan):
    n = plan.n_slots
    items, steps, kv_off, kv_list = _i32(3 * n), _i32(n), _i32(n + 1), _i32(plan.n_kv_entries)
    _check(_lib.mesh_attn_plan_order(plan.handle, items, steps, kv_off, kv_list), "mesh_attn_plan_order")
    off = list(kv_off[:n + 1])
    kvl = list(kv_list[:plan.n_kv_entries])
    return ([tuple(items[3 * i:3 * i + 3]) for i in range(n)], list(steps[:n]),
            [kvl[off[i]:off[i + 1]] for i in range(n)])


def mesh_attn_plan_launch_order(plan: Plan):
    """Indices into mesh_attn_plan_order's item list, in the order the kernels take the items."""
    n = plan.n_slots
    out = (c_i32 * max(n, 1))()
    _check(_lib.mesh_attn_plan_launch_order(plan.handle, out), "mesh_attn_plan_launch_order")
    return [out[i] for i in range(n)]


def mesh_attn_plan_volumes(plan: Plan, Hq: int, Hkv: int, d: int, dtype: torch.dtype = torch.bfloat16):
    counts = _i32(3 * plan.P)
    byts = (c_i64 * (3 * plan.P))()
    ring = c_i64()
    _check(_lib.mesh_attn_plan_volumes(plan.handle, Hq, Hkv, d, _dtype_code(dtype), counts, byts, ctypes.byref(ring)),
           "mesh_attn_plan_volumes")
    P = plan.P
    return ([tuple(counts[3 * v:3 * v + 3]) for v in range(P)], [tuple(byts[3 * v:3 * v + 3]) for v in range(P)],
            ring.value)


def mesh_attn_partials_size(plan: Plan, B: int, Hq: int, d: int) -> Tuple[int, int]:
    o, l = c_sz(), c_sz()
    _check(_lib.mesh_attn_partials_size(plan.handle, B, Hq, d, ctypes.byref(o), ctypes.byref(l)),
           "mesh_attn_partials_size")
    return o.value, l.value


def mesh_attn_workspace_size(plan: Plan) -> int:
    n = c_sz()
    _check(_lib.mesh_attn_workspace_size(plan.handle, ctypes.byref(n)), "mesh_attn_workspace_size")
    return n.value


def mesh_attn_workspace_size_for(plan: Plan, dtype: torch.dtype, B: int, Hq: int, Hkv: int, d: int) -> int:
    n = c_sz()
    _check(_lib.mesh_attn_workspace_size_for(plan.handle, _dtype_code(dtype), B, Hq, Hkv, d, ctypes.byref(n)),
           "mesh_attn_workspace_size_for")
    return n.value


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status block (MESH_ATTN_STATUS_WORDS int32)."""
    return torch.zeros(MESH_ATTN_STATUS_WORDS, dtype=torch.int32, device=device or "cuda")


def new_workspace(plan: Plan, device=None, q: Optional[torch.Tensor] = None, k: Optional[torch.Tensor] = None
                  ) -> torch.Tensor:
    """Workspace for mesh_attn_tile_fwd and mesh_attn_merge; pass q and k (fp32 inputs need room
    for their bf16 pieces)."""
    if q is not None and k is not None:
        B, Hq, _, d = q.shape
        n = mesh_attn_workspace_size_for(plan, q.dtype, B, Hq, k.shape[1], d)
    else:
        n = mesh_attn_workspace_size(plan)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def new_partials(plan: Plan, B: int, Hq: int, d: int, device=None):
    no, nl = mesh_attn_partials_size(plan, B, Hq, d)
    dev = device or "cuda"
    return (torch.empty(max(no, 4), dtype=torch.float32, device=dev),
            torch.empty(max(nl, 4), dtype=torch.float32, device=dev))


def mesh_attn_tile_fwd(plan: Plan, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float],
                       partial_o: torch.Tensor, partial_lse: torch.Tensor, workspace: torch.Tensor,
                       status: torch.Tensor, stream=None) -> None:
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    _check(_lib.mesh_attn_tile_fwd(plan.handle, _dtype_code(q.dtype), B, Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v),
                                   float(scale), _ptr(partial_o), _ptr(partial_lse), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(status),
                                   _stream_handle(stream)), "mesh_attn_tile_fwd")


def mesh_attn_tile_fwd_noalloc(plan: Plan, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               scale: Optional[float], partial_o: torch.Tensor, partial_lse: torch.Tensor,
                               status: torch.Tensor, stream=None) -> None:
    """mesh_attn_tile_fwd without a workspace: for callers that may not allocate device memory.
    The work list goes into the library's fixed scratch array; calls overlapping on the GPU race."""
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    _check(_lib.mesh_attn_tile_fwd_noalloc(plan.handle, _dtype_code(q.dtype), B, Hq, Hkv, d, _ptr(q), _ptr(k),
                                           _ptr(v), float(scale), _ptr(partial_o), _ptr(partial_lse), _ptr(status),
                                           _stream_handle(stream)), "mesh_attn_tile_fwd_noalloc")


def mesh_attn_merge(plan: Plan, B: int, Hq: int, d: int, partial_o: torch.Tensor, partial_lse: torch.Tensor,
                    O: torch.Tensor, LSE: torch.Tensor, workspace: torch.Tensor, status: torch.Tensor,
                    stream=None) -> None:
    _check(_lib.mesh_attn_merge(plan.handle, _dtype_code(O.dtype), B, Hq, d, _ptr(partial_o), _ptr(partial_lse),
                                _ptr(O), _ptr(LSE), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(status), _stream_handle(stream)), "mesh_attn_merge")


def mesh_attn_plan_kv_slots(plan: Plan):
    """Backward KV slots: (kv_slot_off [P+1], [(k, t, kv_slot)], [[Q partitions] per slot])."""
    n = plan.n_kv_slots
    off, items, q_off, q_list = _i32(plan.P + 1), _i32(3 * n), _i32(n + 1), _i32(plan.n_live_blocks)
    _check(_lib.mesh_attn_plan_kv_slots(plan.handle, off, items, q_off, q_list), "mesh_attn_plan_kv_slots")
    qo = list(q_off[:n + 1])
    ql = list(q_list[:plan.n_live_blocks])
    return (list(off[:plan.P + 1]), [tuple(items[3 * i:3 * i + 3]) for i in range(n)],
            [ql[qo[i]:qo[i + 1]] for i in range(n)])


def mesh_attn_bwd_partials_size(plan: Plan, B: int, Hq: int, Hkv: int, d: int) -> Tuple[int, int]:
    q, kv = c_sz(), c_sz()
    _check(_lib.mesh_attn_bwd_partials_size(plan.handle, B, Hq, Hkv, d, ctypes.byref(q), ctypes.byref(kv)),
           "mesh_attn_bwd_partials_size")
    return q.value, kv.value


def mesh_attn_bwd_workspace_size(plan: Plan) -> int:
    n = c_sz()
    _check(_lib.mesh_attn_bwd_workspace_size(plan.handle, ctypes.byref(n)), "mesh_attn_bwd_workspace_size")
    return n.value


def new_bwd_workspace(plan: Plan, device=None) -> torch.Tensor:
    return torch.empty(max(mesh_attn_bwd_workspace_size(plan), 16), dtype=torch.uint8, device=device or "cuda")


def new_bwd_partials(plan: Plan, B: int, Hq: int, Hkv: int, d: int, device=None):
    nq, nkv = mesh_attn_bwd_partials_size(plan, B, Hq, Hkv, d)
    dev = device or "cuda"
    return tuple(torch.empty(max(n, 4), dtype=torch.float32, device=dev) for n in (nq, nkv, nkv))


def mesh_attn_bwd_prep(O: torch.Tensor, dO: torch.Tensor, D: torch.Tensor, status: torch.Tensor,
                       stream=None) -> None:
    B, Hq, S, d = O.shape
    if O.dtype != dO.dtype or not O.is_contiguous() or not dO.is_contiguous():
        raise ValueError("O and dO must be contiguous and of one dtype")
    _check(_lib.mesh_attn_bwd_prep(_dtype_code(O.dtype), B, Hq, S, d, _ptr(O), _ptr(dO), _ptr(D), _ptr(status),
                                   _stream_handle(stream)), "mesh_attn_bwd_prep")


def mesh_attn_tile_bwd(plan: Plan, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dO: torch.Tensor,
                       LSE: torch.Tensor, D: torch.Tensor, scale: Optional[float], dq_partial: torch.Tensor,
                       dk_partial: torch.Tensor, dv_partial: torch.Tensor, workspace: torch.Tensor,
                       status: torch.Tensor, stream=None) -> None:
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (q, k, v, dO):
        if not t.is_contiguous():
            raise ValueError("q, k, v and dO must be contiguous")
    _check(_lib.mesh_attn_tile_bwd(plan.handle, _dtype_code(q.dtype), B, Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(dO), _ptr(LSE), _ptr(D), float(scale), _ptr(dq_partial), _ptr(dk_partial),
                                   _ptr(dv_partial), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(status), _stream_handle(stream)), "mesh_attn_tile_bwd")


def mesh_attn_bwd_reduce(plan: Plan, B: int, Hq: int, Hkv: int, d: int, dq_partial: torch.Tensor,
                         dk_partial: torch.Tensor, dv_partial: torch.Tensor, dQ: torch.Tensor, dK: torch.Tensor,
                         dV: torch.Tensor, workspace: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    if not (dQ.dtype == dK.dtype == dV.dtype):
        raise ValueError("dQ, dK and dV must share one dtype")
    _check(_lib.mesh_attn_bwd_reduce(plan.handle, _dtype_code(dQ.dtype), B, Hq, Hkv, d, _ptr(dq_partial),
                                     _ptr(dk_partial), _ptr(dv_partial), _ptr(dQ), _ptr(dK), _ptr(dV),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
                                     _stream_handle(stream)), "mesh_attn_bwd_reduce")


def mesh_attention_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, O: torch.Tensor,
                            LSE: torch.Tensor, dO: torch.Tensor, P: int, causal: bool, kvr: bool = True,
                            greedy: bool = True, scale: Optional[float] = None, plan: Optional[Plan] = None,
                            return_partials: bool = False, check_status: bool = True):
    """Whole backward on the current stream: D = dO . O, tile backward, reduce.

    q [B,Hq,S,d], k/v [B,Hkv,S,d], O and dO [B,Hq,S,d] (one dtype, bf16 or fp32), LSE [B,Hq,S]
    fp32 from the forward.  Returns (dQ, dK, dV) in q's dtype; with return_partials also the
    fp32 partials (dq, dk, dv).
    """
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    plan = plan or mesh_attn_plan_create(S, P, causal, kvr, greedy)
    dq_p, dk_p, dv_p = new_bwd_partials(plan, B, Hq, Hkv, d, q.device)
    ws = new_bwd_workspace(plan, q.device)
    st = new_status(q.device)
    D = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    mesh_attn_bwd_prep(O, dO, D, st)
    mesh_attn_tile_bwd(plan, q, k, v, dO, LSE, D, scale, dq_p, dk_p, dv_p, ws, st)
    mesh_attn_bwd_reduce(plan, B, Hq, Hkv, d, dq_p, dk_p, dv_p, dQ, dK, dV, ws, st)
    if check_status:
        code = mesh_attn_read_status(st)
        if code != 0:
            raise MeshAttnError(code, "device", f"status block {st.tolist()}")
    if return_partials:
        return dQ, dK, dV, dq_p, dk_p, dv_p
    return dQ, dK, dV


def mesh_attn_read_status(status: torch.Tensor, stream=None) -> int:
    out = c_i32()
    _check(_lib.mesh_attn_read_status(_ptr(status), _stream_handle(stream), ctypes.byref(out)),
           "mesh_attn_read_status")
    return out.value


def mesh_attn_set_wait_limit_ns(ns: int) -> None:
    load_library()
    _check(_lib.mesh_attn_set_wait_limit_ns(int(ns)), "mesh_attn_set_wait_limit_ns")


def mesh_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, causal: bool, kvr: bool = True,
                   greedy: bool = True, scale: Optional[float] = None, plan: Optional[Plan] = None,
                   return_partials: bool = False, check_status: bool = True):
    """Whole hot path on the current stream: plan, tile forward, LSE merge.

    q [B,Hq,S,d], k/v [B,Hkv,S,d] CUDA tensors (bf16 or fp32).  Returns (O, LSE) with O in
    q's dtype and LSE fp32; with return_partials also (partial_o, partial_lse).
    """
    B, Hq, S, d = q.shape
    plan = plan or mesh_attn_plan_create(S, P, causal, kvr, greedy)
    po, pl = new_partials(plan, B, Hq, d, q.device)
    ws = new_workspace(plan, q.device, q, k)
    st = new_status(q.device)
    O = torch.empty_like(q)
    LSE = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    mesh_attn_tile_fwd(plan, q, k, v, scale, po, pl, ws, st)
    mesh_attn_merge(plan, B, Hq, d, po, pl, O, LSE, ws, st)
    if check_status:
        code = mesh_attn_read_status(st)
        if code != 0:
            raise MeshAttnError(code, "device", f"status block {st.tolist()}")
    if return_partials:
        return O, LSE, po, pl
    return O, LSE


class MeshAttentionFunction(torch.autograd.Function):
    """torch.autograd binding of the two public calls: the forward runs mesh_attention and keeps
    q, k, v, O and LSE; the backward runs mesh_attention_backward with the incoming dO.  Gradients
    reach q, k and v; LSE is returned as a non-differentiable output (no gradient flows through
    it).  Argument marshalling only: every step runs in the library's kernels."""

    @staticmethod
    def forward(ctx, q, k, v, P, causal, kvr, greedy, scale):
        plan = mesh_attn_plan_create(q.shape[2], P, causal, kvr, greedy)
        O, LSE = mesh_attention(q, k, v, P, causal, kvr, greedy, scale, plan=plan)
        ctx.save_for_backward(q, k, v, O, LSE)
        ctx.plan = plan
        ctx.args = (P, causal, kvr, greedy, scale)
        ctx.mark_non_differentiable(LSE)
        return O, LSE

    @staticmethod
    def backward(ctx, dO, dLSE):
        q, k, v, O, LSE = ctx.saved_tensors
        P, causal, kvr, greedy, scale = ctx.args
        dQ, dK, dV = mesh_attention_backward(q, k, v, O, LSE, dO.contiguous(), P, causal, kvr, greedy, scale,
                                             plan=ctx.plan)
        return dQ, dK, dV, None, None, None, None, None


def mesh_attention_autograd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, causal: bool,
                            kvr: bool = True, greedy: bool = True, scale: Optional[float] = None):
    """mesh_attention with autograd: returns (O, LSE); O.backward(...) fills q.grad, k.grad and v.grad
    through the tile backward."""
    return MeshAttentionFunction.apply(q, k, v, P, causal, kvr, greedy, scale)
