// Tile attention forward on the CUDA cores, fp32 throughout: the path for fp32 inputs, whose
// tolerance (1e-4 absolute on O and LSE) the bf16 tensor-core products cannot meet.
//
// Same work decomposition and output as the tensor-core kernel (Mesh-Attention tiles and
// partials; online m_i / l_i softmax of "环形注意力：突破长序列处理瓶颈的分布式计算范式",
// §"数值稳定性：Log-Sum-Exp技术的分布式应用"), mapped for the FP32 pipe:
//   a CTA of 4 warps owns 32 query rows of one (item, batch, head); each warp owns 8 rows;
//   keys are staged 32 at a time in shared memory; lane j scores key j against the warp's 8
//   rows (float4 dot products), the warp reduces max and sum with shuffles, and each lane
//   accumulates d/32 output columns of the 8 rows from the probabilities in shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace simt {

constexpr int ROWS = 32;   // query rows per CTA
constexpr int RPW = 8;     // rows per warp
constexpr int CHUNK = 32;  // keys per staged chunk
constexpr int THREADS = 128;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T, int D>
__global__ void __launch_bounds__(THREADS) tile_fwd_simt_kernel(const TileArgs a, int n_rb) {
  constexpr int KP = D + 4;  // padded key row: conflict-free float4 reads across lanes
  constexpr int E = D / 32;  // output columns per lane
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [ROWS][D]
  float* Ks = Qs + ROWS * D;                    // [CHUNK][KP]
  float* Vs = Ks + CHUNK * KP;                  // [CHUNK][D]
  float* Ps = Vs + CHUNK * D;                   // [4][RPW][CHUNK]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int64_t u = blockIdx.x;
  const int rb = (int)(u % n_rb); u /= n_rb;
  const int h = (int)(u % a.Hq); u /= a.Hq;
  const int b = (int)(u % a.B);
  const int item_idx = (int)(u / a.B);
  if (*reinterpret_cast<volatile int32_t*>(a.status) != 0) return;
  const DevItem it = a.items[item_idx];
  if (it.p < 0 || it.p >= a.P || it.slot < 0 || it.slot >= a.n_slots || it.n_kv < 1 || it.kv_off < 0) {
    if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 4, (int32_t)blockIdx.x);
    return;
  }
  const int64_t L = a.L;
  const int hk = h / (a.Hq / a.Hkv);
  const int64_t row0 = (int64_t)rb * ROWS;  // first row of the CTA within the partition
  const T* Qg = reinterpret_cast<const T*>(a.Q) + (((int64_t)b * a.Hq + h) * a.S + (int64_t)it.p * L) * D;
  const T* Kg = reinterpret_cast<const T*>(a.K) + ((int64_t)b * a.Hkv + hk) * a.S * D;
  const T* Vg = reinterpret_cast<const T*>(a.V) + ((int64_t)b * a.Hkv + hk) * a.S * D;

  for (int i = tid; i < ROWS * D; i += THREADS) {
    const int r = i / D;
    Qs[i] = (row0 + r < L) ? to_f(Qg[(row0 + r) * D + (i % D)]) : 0.f;
  }

  float m[RPW], l[RPW], acc[RPW][E];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  }
  const int wrow0 = warp * RPW;  // warp's first row within the CTA

  for (int ki = 0; ki < it.n_kv; ++ki) {
    const int k = a.kv_list[it.kv_off + ki];
    if (k < 0 || k >= a.P) {
      if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 3, (int32_t)blockIdx.x);
      return;
    }
    const bool diag = a.causal && k == it.p;
    const int64_t n_keys = diag ? min(L, row0 + ROWS) : L;
    for (int64_t c0 = 0; c0 < n_keys; c0 += CHUNK) {
      __syncthreads();
      for (int i = tid; i < CHUNK * D; i += THREADS) {
        const int j = i / D, e = i % D;
        const int64_t key = c0 + j;
        const bool in = key < n_keys;
        const int64_t g = ((int64_t)k * L + key) * D + e;
        Ks[j * KP + e] = in ? to_f(Kg[g]) : 0.f;
        Vs[j * D + e] = in ? to_f(Vg[g]) : 0.f;
      }
      __syncthreads();
      // scores of key (c0 + lane) against the warp's rows
      float s[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) s[i] = 0.f;
      const float4* kr = reinterpret_cast<const float4*>(Ks + lane * KP);
#pragma unroll 4
      for (int e4 = 0; e4 < D / 4; ++e4) {
        const float4 kv = kr[e4];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          const float4 q = reinterpret_cast<const float4*>(Qs + (wrow0 + i) * D)[e4];
          s[i] = fmaf(q.x, kv.x, fmaf(q.y, kv.y, fmaf(q.z, kv.z, fmaf(q.w, kv.w, s[i]))));
        }
      }
      const int64_t key = c0 + lane;
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const int64_t row = row0 + wrow0 + i;
        const bool vis = key < n_keys && (!diag || key <= row);
        const float s2 = vis ? s[i] * a.scale_log2 : -INFINITY;
        const float cmax = warp_max(s2);
        const float m_new = fmaxf(m[i], cmax);
        const float mref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - mref);
        const float pj = vis ? exp2f(s2 - mref) : 0.f;
        l[i] = l[i] * alpha + warp_sum(pj);
        m[i] = m_new;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] *= alpha;
        Ps[(warp * RPW + i) * CHUNK + lane] = pj;
      }
      __syncwarp();
#pragma unroll 4
      for (int j = 0; j < CHUNK; ++j) {
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = Vs[j * D + lane + 32 * e];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          const float pj = Ps[(warp * RPW + i) * CHUNK + j];
#pragma unroll
          for (int e = 0; e < E; ++e) acc[i][e] = fmaf(pj, v[e], acc[i][e]);
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int64_t row = row0 + wrow0 + i;
    if (row >= L) continue;
    const int64_t prow = (((int64_t)b * a.Hq + h) * a.n_slots + it.slot) * L + row;
    const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) a.part_o[prow * D + lane + 32 * e] = acc[i][e] * inv;
    if (lane == 0) a.part_lse[prow] = l[i] > 0.f ? (m[i] + log2f(l[i])) * 0.69314718055994531f : -INFINITY;
  }
}

template <typename T, int D>
static int launch(const TileArgs& a, void* stream, std::string* err) {
  const int64_t n_rb = (a.L + ROWS - 1) / ROWS;
  const int64_t blocks = (int64_t)a.n_items * a.B * a.Hq * n_rb;
  if (blocks <= 0) return (int)cudaSuccess;
  if (blocks > 0x7fffffff) {
    *err = "too many work units for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  const size_t smem = sizeof(float) * (ROWS * D + CHUNK * (D + 4) + CHUNK * D + 4 * RPW * CHUNK);
  auto kern = tile_fwd_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  kern<<<dim3((unsigned)blocks), dim3(THREADS), smem, (cudaStream_t)stream>>>(a, (int)n_rb);
  e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("tile_fwd_simt launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace simt

int launch_tile_fwd_simt(const TileArgs& a, mesh_attn_dtype dt, void* stream, std::string* err) {
  if (dt == MESH_ATTN_F32) {
    if (a.d == 128) return simt::launch<float, 128>(a, stream, err);
    if (a.d == 64) return simt::launch<float, 64>(a, stream, err);
  } else {
    if (a.d == 128) return simt::launch<__nv_bfloat16, 128>(a, stream, err);
    if (a.d == 64) return simt::launch<__nv_bfloat16, 64>(a, stream, err);
  }
  *err = "CUDA-core tile kernel supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
