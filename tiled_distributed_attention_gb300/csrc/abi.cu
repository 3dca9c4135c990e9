// extern "C" entry points declared in mesh_attn.h: argument validation, plan access, work-list
// upload into the caller's workspace and kernel dispatch.  No exception crosses this layer and
// nothing is enqueued before every host-side check has passed.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <new>
#include <stdexcept>
#include <string>

#include "internal.h"

namespace {

thread_local std::string g_err;
std::atomic<int64_t> g_wait_limit_ns{2000000000LL};

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what, const std::string& extra = std::string()) {
  g_err = std::string(what) + ": " + cudaGetErrorString(e) + (extra.empty() ? "" : " (" + extra + ")");
  return MESH_ATTN_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename F>
int guarded(F&& f) {
  try {
    g_err.clear();
    return f();
  } catch (const std::bad_alloc&) {
    return fail(MESH_ATTN_ERR_NO_MEMORY, "host allocation failed");
  } catch (const std::invalid_argument& e) {
    return fail(MESH_ATTN_ERR_INVALID_ARG, e.what());
  } catch (const std::exception& e) {
    return fail(MESH_ATTN_ERR_INTERNAL, e.what());
  } catch (...) {
    return fail(MESH_ATTN_ERR_INTERNAL, "unknown exception");
  }
}

int check_common(const mesh_attn_plan* plan, int32_t B, int32_t Hq, int32_t d) {
  if (!plan) return fail(MESH_ATTN_ERR_INVALID_ARG, "plan is NULL");
  if (B < 0 || Hq < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "B and Hq must be >= 0");
  if (d != 64 && d != 128) return fail(MESH_ATTN_ERR_UNSUPPORTED, "d must be 64 or 128");
  const mesh::Plan& pl = plan->p;
  // rows are addressed with 32-bit TMA coordinates and 32-bit grid indices
  if ((int64_t)B * Hq * pl.S >= (int64_t)1 << 31)
    return fail(MESH_ATTN_ERR_UNSUPPORTED, "B * Hq * S must be < 2^31");
  return MESH_ATTN_OK;
}

}  // namespace

namespace mesh {
int set_last_error(int code, const std::string& msg) { return fail(code, msg); }
int64_t current_wait_limit_ns() { return g_wait_limit_ns.load(); }
}  // namespace mesh

extern "C" {

int mesh_attn_plan_create(int64_t S, int32_t P, int32_t causal, int32_t kvr, int32_t greedy,
                          mesh_attn_plan** out) {
  return guarded([&] {
    if (!out) return fail(MESH_ATTN_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    for (int32_t f : {causal, kvr, greedy})
      if (f != 0 && f != 1) return fail(MESH_ATTN_ERR_INVALID_ARG, "causal, kvr and greedy must be 0 or 1");
    mesh_attn_plan* p = new mesh_attn_plan();
    try {
      mesh::build_plan(p->p, S, P, causal != 0, kvr != 0, greedy != 0);
    } catch (...) {
      delete p;
      throw;
    }
    *out = p;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_create_ring(int64_t S, int32_t P, int32_t causal, mesh_attn_plan** out) {
  return guarded([&] {
    if (!out) return fail(MESH_ATTN_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (causal != 0 && causal != 1) return fail(MESH_ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
    mesh_attn_plan* p = new mesh_attn_plan();
    try {
      mesh::build_ring_plan(p->p, S, P, causal != 0);
    } catch (...) {
      delete p;
      throw;
    }
    *out = p;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_destroy(mesh_attn_plan* plan) {
  delete plan;
  return MESH_ATTN_OK;
}

int mesh_attn_plan_get_info(const mesh_attn_plan* plan, mesh_attn_plan_info* out) {
  return guarded([&] {
    if (!plan || !out) return fail(MESH_ATTN_ERR_INVALID_ARG, "plan or out is NULL");
    const mesh::Plan& p = plan->p;
    std::memset(out, 0, sizeof(*out));
    out->S = p.S;
    out->L = p.L;
    out->P = p.P;
    out->R = p.R;
    out->causal = p.causal;
    out->kvr = p.kvr;
    out->greedy = p.greedy;
    out->n_slots = p.n_slots();
    out->n_steps = p.n_steps;
    out->layout = p.layout;
    out->tile_q = p.tile_q;
    out->tile_kv = p.tile_kv;
    out->n_kv_entries = (int64_t)p.kv_list.size();
    out->n_live_blocks = p.n_live;
    out->n_kv_slots = p.n_kv_slots();
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_tiles(const mesh_attn_plan* plan, int32_t* q_parts, int32_t* kv_parts) {
  return guarded([&] {
    if (!plan || !q_parts || !kv_parts) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    std::memcpy(q_parts, plan->p.q_parts.data(), plan->p.q_parts.size() * sizeof(int32_t));
    std::memcpy(kv_parts, plan->p.kv_parts.data(), plan->p.kv_parts.size() * sizeof(int32_t));
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_slots(const mesh_attn_plan* plan, int32_t* slot_off) {
  return guarded([&] {
    if (!plan || !slot_off) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    std::memcpy(slot_off, plan->p.slot_off.data(), plan->p.slot_off.size() * sizeof(int32_t));
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_order(const mesh_attn_plan* plan, int32_t* items, int32_t* item_step, int32_t* kv_off,
                         int32_t* kv_list) {
  return guarded([&] {
    if (!plan) return fail(MESH_ATTN_ERR_INVALID_ARG, "plan is NULL");
    const mesh::Plan& p = plan->p;
    if (items) std::memcpy(items, p.items.data(), p.items.size() * sizeof(int32_t));
    if (item_step) std::memcpy(item_step, p.item_step.data(), p.item_step.size() * sizeof(int32_t));
    if (kv_off) std::memcpy(kv_off, p.kv_off.data(), p.kv_off.size() * sizeof(int32_t));
    if (kv_list) std::memcpy(kv_list, p.kv_list.data(), p.kv_list.size() * sizeof(int32_t));
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_launch_order(const mesh_attn_plan* plan, int32_t* order) {
  return guarded([&] {
    if (!plan) return fail(MESH_ATTN_ERR_INVALID_ARG, "plan is NULL");
    const mesh::Plan& p = plan->p;
    if (order && !p.launch.empty()) std::memcpy(order, p.launch.data(), p.launch.size() * sizeof(int32_t));
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_volumes(const mesh_attn_plan* plan, int32_t Hq, int32_t Hkv, int32_t d, mesh_attn_dtype dtype,
                           int32_t* counts, int64_t* bytes, int64_t* ring_bytes) {
  return guarded([&] {
    if (!plan) return fail(MESH_ATTN_ERR_INVALID_ARG, "plan is NULL");
    if (Hq < 0 || Hkv < 0 || d < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "Hq, Hkv and d must be >= 0");
    if (dtype != MESH_ATTN_F32 && dtype != MESH_ATTN_BF16) return fail(MESH_ATTN_ERR_INVALID_ARG, "bad dtype");
    const mesh::Plan& p = plan->p;
    const int64_t es = dtype == MESH_ATTN_BF16 ? 2 : 4;
    const int64_t qb = p.L * Hq * d * es;
    const int64_t kvb = 2 * p.L * Hkv * d * es;
    const int64_t ob = p.L * Hq * (4 * (int64_t)d + 4);
    for (int32_t v = 0; v < p.P; ++v) {
      const int32_t* c = &p.recv[(size_t)v * 3];
      if (counts) {
        counts[3 * v + 0] = c[0];
        counts[3 * v + 1] = c[1];
        counts[3 * v + 2] = c[2];
      }
      if (bytes) {
        bytes[3 * v + 0] = c[0] * qb;
        bytes[3 * v + 1] = c[1] * kvb;
        bytes[3 * v + 2] = c[2] * ob;
      }
    }
    if (ring_bytes) *ring_bytes = (int64_t)(p.P - 1) * kvb;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_partials_size(const mesh_attn_plan* plan, int32_t B, int32_t Hq, int32_t d, size_t* o_elems,
                            size_t* lse_elems) {
  return guarded([&] {
    if (!plan || !o_elems || !lse_elems) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    if (B < 0 || Hq < 0 || d < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "B, Hq and d must be >= 0");
    const size_t rows = (size_t)B * Hq * plan->p.n_slots() * (size_t)plan->p.L;
    *lse_elems = rows;
    *o_elems = rows * (size_t)d;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_workspace_size(const mesh_attn_plan* plan, size_t* bytes) {
  return guarded([&] {
    if (!plan || !bytes) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    *bytes = mesh::workspace_layout(plan->p).total;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_workspace_size_for(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B, int32_t Hq,
                                 int32_t Hkv, int32_t d, size_t* bytes) {
  return guarded([&] {
    if (!plan || !bytes) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    if (in_dtype != MESH_ATTN_F32 && in_dtype != MESH_ATTN_BF16)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "in_dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    if (B < 0 || Hq < 0 || Hkv < 0 || d < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "B, Hq, Hkv and d must be >= 0");
    const size_t base = mesh::workspace_layout(plan->p).total;
    *bytes = in_dtype == MESH_ATTN_F32
                 ? ((base + 255) & ~(size_t)255) + mesh::f32_pieces_layout(B, Hq, Hkv, plan->p.S, d).total
                 : base;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_tile_fwd(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                       int32_t d, const void* Q, const void* K, const void* V, float scale, float* partial_o,
                       float* partial_lse, void* workspace, size_t workspace_bytes, int32_t* d_status,
                       void* stream) {
  return guarded([&] {
    int rc = check_common(plan, B, Hq, d);
    if (rc) return rc;
    if (in_dtype != MESH_ATTN_F32 && in_dtype != MESH_ATTN_BF16)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "in_dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    if (Hkv < 1 || Hq % Hkv != 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "need Hkv >= 1 and Hq % Hkv == 0");
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MESH_ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    const mesh::Plan& pl = plan->p;
    if (pl.n_slots() == 0 || B == 0 || Hq == 0) return (int)MESH_ATTN_OK;
    if (!Q || !K || !V || !partial_o || !partial_lse || !workspace || !d_status)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "a tensor, workspace or status pointer is NULL");
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(partial_o, 16) ||
        !aligned(partial_lse, 4) || !aligned(workspace, 16) || !aligned(d_status, 4))
      return fail(MESH_ATTN_ERR_MISALIGNED, "Q, K, V, partial_o and workspace must be 16-byte aligned");
    const mesh::WorkspaceLayout wl = mesh::workspace_layout(pl);
    // fp32 inputs: the bf16 pieces of Q, K and V follow the work list
    const size_t pieces_off = (wl.total + 255) & ~(size_t)255;
    const size_t need = in_dtype == MESH_ATTN_F32 ? pieces_off + mesh::f32_pieces_layout(B, Hq, Hkv, pl.S, d).total
                                                  : wl.total;
    if (workspace_bytes < need)
      return fail(MESH_ATTN_ERR_WORKSPACE, "workspace needs " + std::to_string(need) + " bytes");
    char* ws = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(ws + wl.items_off, pl.dev_items.data(), wl.items_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "work-list upload");
    e = cudaMemcpyAsync(ws + wl.kv_off, pl.kv_list.data(), wl.kv_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "KV-list upload");
    e = cudaMemsetAsync(ws + wl.counter_off, 0, 256, st);  // the kernel's unit counter starts at 0
    if (e != cudaSuccess) return cuda_fail(e, "counter reset");
    mesh::TileArgs a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.part_o = partial_o;
    a.part_lse = partial_lse;
    a.items = reinterpret_cast<const mesh::DevItem*>(ws + wl.items_off);
    a.kv_list = reinterpret_cast<const int32_t*>(ws + wl.kv_off);
    a.counter = reinterpret_cast<uint32_t*>(ws + wl.counter_off);
    a.status = d_status;
    a.S = pl.S;
    a.L = pl.L;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.P = pl.P;
    a.n_items = pl.n_slots();
    a.n_slots = pl.n_slots();
    a.causal = pl.causal ? 1 : 0;
    a.scale = scale;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.pieces = ws + pieces_off;
    std::string err;
    const int ce = (in_dtype == MESH_ATTN_BF16) ? mesh::launch_tile_fwd_tc(a, stream, &err)
                                                : mesh::launch_tile_fwd_tc32(a, stream, &err);
    if (ce != (int)cudaSuccess) return fail(MESH_ATTN_ERR_CUDA, err.empty() ? cudaGetErrorString((cudaError_t)ce) : err);
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_merge(const mesh_attn_plan* plan, mesh_attn_dtype out_dtype, int32_t B, int32_t Hq, int32_t d,
                    const float* partial_o, const float* partial_lse, void* O, float* LSE, void* workspace,
                    size_t workspace_bytes, int32_t* d_status, void* stream) {
  return guarded([&] {
    int rc = check_common(plan, B, Hq, d);
    if (rc) return rc;
    if (out_dtype != MESH_ATTN_F32 && out_dtype != MESH_ATTN_BF16)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "out_dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    const mesh::Plan& pl = plan->p;
    if (pl.S == 0 || B == 0 || Hq == 0) return (int)MESH_ATTN_OK;
    if (!partial_o || !partial_lse || !O || !LSE || !workspace || !d_status)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "a tensor, workspace or status pointer is NULL");
    if (!aligned(partial_o, 16) || !aligned(partial_lse, 4) || !aligned(O, 16) || !aligned(LSE, 4) ||
        !aligned(workspace, 16) || !aligned(d_status, 4))
      return fail(MESH_ATTN_ERR_MISALIGNED, "partial_o, O and workspace must be 16-byte aligned");
    const mesh::WorkspaceLayout wl = mesh::workspace_layout(pl);
    if (workspace_bytes < wl.total)
      return fail(MESH_ATTN_ERR_WORKSPACE, "workspace needs " + std::to_string(wl.total) + " bytes");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(workspace, pl.slot_off.data(), wl.slot_off_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "slot-offset upload");
    mesh::MergeArgs a{};
    a.part_o = partial_o;
    a.part_lse = partial_lse;
    a.slot_off = static_cast<const int32_t*>(workspace);
    a.O = O;
    a.LSE = LSE;
    a.status = d_status;
    a.S = pl.S;
    a.L = pl.L;
    a.B = B;
    a.Hq = Hq;
    a.d = d;
    a.P = pl.P;
    a.n_slots = pl.n_slots();
    std::string err;
    const int ce = mesh::launch_merge(a, out_dtype, stream, &err);
    if (ce != (int)cudaSuccess) return fail(MESH_ATTN_ERR_CUDA, err.empty() ? cudaGetErrorString((cudaError_t)ce) : err);
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_plan_kv_slots(const mesh_attn_plan* plan, int32_t* kv_slot_off, int32_t* kv_items, int32_t* q_off,
                            int32_t* q_list) {
  return guarded([&] {
    if (!plan) return fail(MESH_ATTN_ERR_INVALID_ARG, "plan is NULL");
    const mesh::Plan& p = plan->p;
    if (kv_slot_off) std::memcpy(kv_slot_off, p.kv_slot_off.data(), p.kv_slot_off.size() * sizeof(int32_t));
    if (kv_items) std::memcpy(kv_items, p.kv_items.data(), p.kv_items.size() * sizeof(int32_t));
    if (q_off) std::memcpy(q_off, p.kv_q_off.data(), p.kv_q_off.size() * sizeof(int32_t));
    if (q_list) std::memcpy(q_list, p.kv_q_list.data(), p.kv_q_list.size() * sizeof(int32_t));
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_bwd_partials_size(const mesh_attn_plan* plan, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                                size_t* dq_elems, size_t* dkv_elems) {
  return guarded([&] {
    if (!plan || !dq_elems || !dkv_elems) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    if (B < 0 || Hq < 0 || Hkv < 0 || d < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "B, Hq, Hkv and d must be >= 0");
    const mesh::Plan& p = plan->p;
    *dq_elems = (size_t)B * Hq * p.n_slots() * (size_t)p.L * d;
    *dkv_elems = (size_t)B * Hkv * p.n_kv_slots() * (size_t)p.L * d;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_bwd_workspace_size(const mesh_attn_plan* plan, size_t* bytes) {
  return guarded([&] {
    if (!plan || !bytes) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    *bytes = mesh::bwd_workspace_layout(plan->p).total;
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_bwd_prep(mesh_attn_dtype dtype, int32_t B, int32_t Hq, int64_t S, int32_t d, const void* O,
                       const void* dO, float* D, int32_t* d_status, void* stream) {
  return guarded([&] {
    if (dtype != MESH_ATTN_F32 && dtype != MESH_ATTN_BF16)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    if (B < 0 || Hq < 0 || S < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "B, Hq and S must be >= 0");
    if (d != 64 && d != 128) return fail(MESH_ATTN_ERR_UNSUPPORTED, "d must be 64 or 128");
    if (B == 0 || Hq == 0 || S == 0) return (int)MESH_ATTN_OK;
    if (!O || !dO || !D || !d_status) return fail(MESH_ATTN_ERR_INVALID_ARG, "a tensor or status pointer is NULL");
    if (!aligned(O, 16) || !aligned(dO, 16) || !aligned(D, 4) || !aligned(d_status, 4))
      return fail(MESH_ATTN_ERR_MISALIGNED, "O and dO must be 16-byte aligned");
    mesh::PrepArgs a{};
    a.O = O;
    a.dO = dO;
    a.D = D;
    a.status = d_status;
    a.S = S;
    a.B = B;
    a.H = Hq;
    a.d = d;
    std::string err;
    const int ce = mesh::launch_bwd_prep(a, dtype, stream, &err);
    if (ce != (int)cudaSuccess) return fail(MESH_ATTN_ERR_CUDA, err.empty() ? cudaGetErrorString((cudaError_t)ce) : err);
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_tile_bwd(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                       int32_t d, const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                       const float* D, float scale, float* dq_partial, float* dk_partial, float* dv_partial,
                       void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
  return guarded([&] {
    int rc = check_common(plan, B, Hq, d);
    if (rc) return rc;
    if (in_dtype != MESH_ATTN_F32 && in_dtype != MESH_ATTN_BF16)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "in_dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    if (Hkv < 1 || Hq % Hkv != 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "need Hkv >= 1 and Hq % Hkv == 0");
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MESH_ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    const mesh::Plan& pl = plan->p;
    if (pl.n_slots() == 0 || B == 0 || Hq == 0) return (int)MESH_ATTN_OK;
    if (!Q || !K || !V || !dO || !LSE || !D || !dq_partial || !dk_partial || !dv_partial || !workspace || !d_status)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "a tensor, workspace or status pointer is NULL");
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(dO, 16) || !aligned(LSE, 4) ||
        !aligned(D, 4) || !aligned(dq_partial, 16) || !aligned(dk_partial, 16) || !aligned(dv_partial, 16) ||
        !aligned(workspace, 16) || !aligned(d_status, 4))
      return fail(MESH_ATTN_ERR_MISALIGNED, "tensors and workspace must be 16-byte aligned");
    const mesh::BwdWorkspaceLayout wl = mesh::bwd_workspace_layout(pl);
    if (workspace_bytes < wl.total)
      return fail(MESH_ATTN_ERR_WORKSPACE, "workspace needs " + std::to_string(wl.total) + " bytes");
    char* ws = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    struct Up { size_t off; const void* src; size_t bytes; const char* what; };
    const Up ups[] = {{wl.items_off, pl.dev_items.data(), wl.items_bytes, "work-list upload"},
                      {wl.kv_off, pl.kv_list.data(), wl.kv_bytes, "KV-list upload"},
                      {wl.kv_items_off, pl.dev_kv_items.data(), wl.kv_items_bytes, "KV-slot upload"},
                      {wl.q_list_off, pl.kv_q_list.data(), wl.q_list_bytes, "Q-list upload"}};
    for (const Up& u : ups) {
      if (u.bytes == 0) continue;
      cudaError_t e = cudaMemcpyAsync(ws + u.off, u.src, u.bytes, cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) return cuda_fail(e, u.what);
    }
    cudaError_t e = cudaMemsetAsync(ws + wl.counter_off, 0, 512, st);  // both scheduling counters start at 0
    if (e != cudaSuccess) return cuda_fail(e, "counter reset");
    mesh::BwdArgs a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.dO = dO;
    a.LSE = LSE;
    a.D = D;
    a.dq_part = dq_partial;
    a.dk_part = dk_partial;
    a.dv_part = dv_partial;
    a.items = reinterpret_cast<const mesh::DevItem*>(ws + wl.items_off);
    a.kv_list = reinterpret_cast<const int32_t*>(ws + wl.kv_off);
    a.kv_items = reinterpret_cast<const mesh::DevItem*>(ws + wl.kv_items_off);
    a.q_list = reinterpret_cast<const int32_t*>(ws + wl.q_list_off);
    a.counters = reinterpret_cast<uint32_t*>(ws + wl.counter_off);
    a.status = d_status;
    a.S = pl.S;
    a.L = pl.L;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.P = pl.P;
    a.n_items = pl.n_slots();
    a.n_slots = pl.n_slots();
    a.n_kv_items = pl.n_kv_slots();
    a.n_kv_slots = pl.n_kv_slots();
    a.causal = pl.causal ? 1 : 0;
    a.scale = scale;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.wait_limit_ns = g_wait_limit_ns.load();
    std::string err;
    const int ce = (in_dtype == MESH_ATTN_BF16) ? mesh::launch_tile_bwd_tc(a, stream, &err)
                                                : mesh::launch_tile_bwd_simt(a, stream, &err);
    if (ce != (int)cudaSuccess) return fail(MESH_ATTN_ERR_CUDA, err.empty() ? cudaGetErrorString((cudaError_t)ce) : err);
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_bwd_reduce(const mesh_attn_plan* plan, mesh_attn_dtype out_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                         int32_t d, const float* dq_partial, const float* dk_partial, const float* dv_partial,
                         void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int32_t* d_status,
                         void* stream) {
  return guarded([&] {
    int rc = check_common(plan, B, Hq, d);
    if (rc) return rc;
    if (out_dtype != MESH_ATTN_F32 && out_dtype != MESH_ATTN_BF16)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "out_dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    if (Hkv < 1 || Hq % Hkv != 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "need Hkv >= 1 and Hq % Hkv == 0");
    const mesh::Plan& pl = plan->p;
    if (pl.S == 0 || B == 0 || Hq == 0) return (int)MESH_ATTN_OK;
    if (!dq_partial || !dk_partial || !dv_partial || !dQ || !dK || !dV || !workspace || !d_status)
      return fail(MESH_ATTN_ERR_INVALID_ARG, "a tensor, workspace or status pointer is NULL");
    if (!aligned(dq_partial, 16) || !aligned(dk_partial, 16) || !aligned(dv_partial, 16) || !aligned(dQ, 16) ||
        !aligned(dK, 16) || !aligned(dV, 16) || !aligned(workspace, 16) || !aligned(d_status, 4))
      return fail(MESH_ATTN_ERR_MISALIGNED, "tensors and workspace must be 16-byte aligned");
    const mesh::BwdWorkspaceLayout wl = mesh::bwd_workspace_layout(pl);
    if (workspace_bytes < wl.total)
      return fail(MESH_ATTN_ERR_WORKSPACE, "workspace needs " + std::to_string(wl.total) + " bytes");
    char* ws = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(ws + wl.slot_off_off, pl.slot_off.data(), wl.slot_off_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "slot-offset upload");
    e = cudaMemcpyAsync(ws + wl.kv_slot_off_off, pl.kv_slot_off.data(), wl.kv_slot_off_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "KV-slot-offset upload");
    std::string err;
    struct Job { const float* part; size_t off; void* out; int32_t H, n; };
    const Job jobs[] = {{dq_partial, wl.slot_off_off, dQ, Hq, pl.n_slots()},
                        {dk_partial, wl.kv_slot_off_off, dK, Hkv, pl.n_kv_slots()},
                        {dv_partial, wl.kv_slot_off_off, dV, Hkv, pl.n_kv_slots()}};
    for (const Job& j : jobs) {
      mesh::ReduceArgs a{};
      a.part = j.part;
      a.off = reinterpret_cast<const int32_t*>(ws + j.off);
      a.out = j.out;
      a.status = d_status;
      a.S = pl.S;
      a.L = pl.L;
      a.B = B;
      a.H = j.H;
      a.d = d;
      a.P = pl.P;
      a.n_slots = j.n;
      const int ce = mesh::launch_bwd_reduce(a, out_dtype, stream, &err);
      if (ce != (int)cudaSuccess) return fail(MESH_ATTN_ERR_CUDA, err.empty() ? cudaGetErrorString((cudaError_t)ce) : err);
    }
    return (int)MESH_ATTN_OK;
  });
}

int mesh_attn_read_status(const int32_t* d_status, void* stream, int32_t* out) {
  return guarded([&] {
    if (!d_status || !out) return fail(MESH_ATTN_ERR_INVALID_ARG, "NULL argument");
    int32_t h = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "status copy");
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
    *out = h;
    return (int)MESH_ATTN_OK;
  });
}

const char* mesh_attn_status_string(int status) {
  switch (status) {
    case MESH_ATTN_OK: return "ok";
    case MESH_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case MESH_ATTN_ERR_UNSUPPORTED: return "unsupported";
    case MESH_ATTN_ERR_MISALIGNED: return "misaligned pointer";
    case MESH_ATTN_ERR_CUDA: return "CUDA error";
    case MESH_ATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MESH_ATTN_ERR_OUT_OF_RANGE: return "device index out of range";
    case MESH_ATTN_ERR_INTERNAL: return "internal error";
    case MESH_ATTN_ERR_NO_MEMORY: return "host out of memory";
    case MESH_ATTN_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

const char* mesh_attn_last_error(void) { return g_err.c_str(); }

int mesh_attn_set_wait_limit_ns(int64_t ns) {
  if (ns < 0) return fail(MESH_ATTN_ERR_INVALID_ARG, "ns must be >= 0");
  g_wait_limit_ns.store(ns);
  return MESH_ATTN_OK;
}

}  // extern "C"
