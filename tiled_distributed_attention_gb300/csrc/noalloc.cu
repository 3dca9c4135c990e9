// mesh_attn_tile_fwd_noalloc: the tile forward for callers that cannot allocate device
// memory, so cannot provide the workspace mesh_attn_tile_fwd asks for.  Typical cases: code
// running under a framework whose caching allocator already owns the device memory pool (a
// direct cudaMalloc would fail or bypass its accounting), code running inside an allocator
// or memory-pressure callback, and embedded callers with a fixed, pre-reserved budget.
//
// Instead of a caller workspace, the plan's work list (items, KV lists and the scheduling
// counter) is copied into one fixed array of device memory owned by this library, declared
// below at file scope.  Every GPU that loads the library holds that array until the process
// exits.  This entry point calls no cudaMalloc, cudaFree or allocating library routine; its
// only CUDA runtime calls are cudaGetDevice, cudaGetSymbolAddress (first call on a device),
// cudaMemcpyAsync, cudaMemsetAsync and the kernel launch.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <string>

#include "internal.h"

namespace {

// Device-side scratch shared by every call on a device.  In host code this name is only a
// host-side stand-in for the symbol: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MESH_ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device with
// that device current.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int mesh_attn_tile_fwd_noalloc(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B,
                                          int32_t Hq, int32_t Hkv, int32_t d, const void* Q, const void* K,
                                          const void* V, float scale, float* partial_o, float* partial_lse,
                                          int32_t* d_status, void* stream) {
  const auto noalloc_fail = mesh::set_last_error;
  try {
    if (!plan) return noalloc_fail(MESH_ATTN_ERR_INVALID_ARG, "plan is NULL");
    const mesh::Plan& pl = plan->p;
    if (B < 0 || Hq < 0) return noalloc_fail(MESH_ATTN_ERR_INVALID_ARG, "B and Hq must be >= 0");
    if (d != 64 && d != 128) return noalloc_fail(MESH_ATTN_ERR_UNSUPPORTED, "d must be 64 or 128");
    if ((int64_t)B * Hq * pl.S >= (int64_t)1 << 31)
      return noalloc_fail(MESH_ATTN_ERR_UNSUPPORTED, "B * Hq * S must be < 2^31");
    if (in_dtype != MESH_ATTN_F32 && in_dtype != MESH_ATTN_BF16)
      return noalloc_fail(MESH_ATTN_ERR_INVALID_ARG, "in_dtype must be MESH_ATTN_F32 or MESH_ATTN_BF16");
    if (Hkv < 1 || Hq % Hkv != 0) return noalloc_fail(MESH_ATTN_ERR_INVALID_ARG, "need Hkv >= 1 and Hq % Hkv == 0");
    if (!(scale > 0.f) || !std::isfinite(scale))
      return noalloc_fail(MESH_ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    const mesh::WorkspaceLayout wl = mesh::workspace_layout(pl);
    // the scratch holds [items | KV lists | counter]; the slot offsets are the merge's
    const size_t items_off = 0;
    const size_t kv_off = (wl.items_bytes + 255) & ~(size_t)255;
    const size_t counter_off = kv_off + ((wl.kv_bytes + 255) & ~(size_t)255);
    // fp32 inputs also keep the bf16 pieces of Q, K and V in the scratch
    const size_t pieces_off = counter_off + 256;
    const size_t need = in_dtype == MESH_ATTN_F32 ? pieces_off + mesh::f32_pieces_layout(B, Hq, Hkv, pl.S, d).total
                                                  : pieces_off;
    if (need > MESH_ATTN_NOALLOC_SCRATCH_BYTES)
      return noalloc_fail(MESH_ATTN_ERR_WORKSPACE,
                          "plan work list (and fp32 input pieces) need " + std::to_string(need) +
                          " bytes of scratch; the no-allocation entry point holds at most " +
                          std::to_string((size_t)MESH_ATTN_NOALLOC_SCRATCH_BYTES) +
                          " bytes: use mesh_attn_tile_fwd with a workspace");
    if (pl.n_slots() == 0 || B == 0 || Hq == 0) return noalloc_fail(MESH_ATTN_OK, "");
    if (!Q || !K || !V || !partial_o || !partial_lse || !d_status)
      return noalloc_fail(MESH_ATTN_ERR_INVALID_ARG, "a tensor or status pointer is NULL");
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(partial_o, 16) ||
        !aligned(partial_lse, 4) || !aligned(d_status, 4))
      return noalloc_fail(MESH_ATTN_ERR_MISALIGNED, "Q, K, V and partial_o must be 16-byte aligned");
    void* base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess)
      return noalloc_fail(MESH_ATTN_ERR_CUDA, std::string("scratch address lookup: ") + cudaGetErrorString(e));
    char* ws = static_cast<char*>(base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // every region the kernel reads is rewritten by this call; the counter must start at 0
    e = cudaMemcpyAsync(ws + items_off, pl.dev_items.data(), wl.items_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + kv_off, pl.kv_list.data(), wl.kv_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws + counter_off, 0, 256, st);
    if (e != cudaSuccess) return noalloc_fail(MESH_ATTN_ERR_CUDA, std::string("scratch upload: ") + cudaGetErrorString(e));
    mesh::TileArgs a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.part_o = partial_o;
    a.part_lse = partial_lse;
    a.items = reinterpret_cast<const mesh::DevItem*>(ws + items_off);
    a.kv_list = reinterpret_cast<const int32_t*>(ws + kv_off);
    a.counter = reinterpret_cast<uint32_t*>(ws + counter_off);
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
    a.wait_limit_ns = mesh::current_wait_limit_ns();
    a.pieces = ws + pieces_off;
    std::string err;
    const int ce = (in_dtype == MESH_ATTN_BF16) ? mesh::launch_tile_fwd_tc(a, stream, &err)
                                                : mesh::launch_tile_fwd_tc32(a, stream, &err);
    if (ce != (int)cudaSuccess)
      return noalloc_fail(MESH_ATTN_ERR_CUDA, err.empty() ? cudaGetErrorString((cudaError_t)ce) : err);
    return noalloc_fail(MESH_ATTN_OK, "");
  } catch (const std::bad_alloc&) {
    return noalloc_fail(MESH_ATTN_ERR_NO_MEMORY, "host allocation failed");
  } catch (...) {
    return noalloc_fail(MESH_ATTN_ERR_INTERNAL, "unexpected exception");
  }
}
