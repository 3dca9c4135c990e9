// LSE merge of the partial outputs of one Q partition's tiles: for every (batch, head, row),
//   M = max_t lse_t,  lse = M + ln sum_t exp(lse_t - M),  O = sum_t exp(lse_t - lse) O_t.
// This is the combine step the Mesh-Attention Q owner performs on the partial results its
// mesh row sends back ("Mesh-Attention: A New Communication-Efficient Distributed Attention
// with Improved Data Locality", tutorial §"Mesh-Attention：从一维'环'到二维'网'"), with the
// log-sum-exp rescaling of "环形注意力：突破长序列处理瓶颈的分布式计算范式",
// §"数值稳定性：Log-Sum-Exp技术的分布式应用".
//
// A streaming HBM-bound kernel: one warp per output row.  Lane t first reads lse of slot t
// (the slots of a row are L rows apart), the warp reduces max and sum with shuffles, then each
// lane streams its d/32 contiguous columns of every slot's O_t row (16-byte loads for d = 128,
// 512 contiguous bytes per slot per warp) and writes d/32 output values (8-byte bf16 or
// 16-byte fp32 stores).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace merge {

constexpr int THREADS = 256;

template <int E>
struct Vec;
template <>
struct Vec<4> {
  using T = float4;
  static __device__ __forceinline__ void fma_into(float* acc, float w, const T& v) {
    acc[0] = fmaf(w, v.x, acc[0]);
    acc[1] = fmaf(w, v.y, acc[1]);
    acc[2] = fmaf(w, v.z, acc[2]);
    acc[3] = fmaf(w, v.w, acc[3]);
  }
};
template <>
struct Vec<2> {
  using T = float2;
  static __device__ __forceinline__ void fma_into(float* acc, float w, const T& v) {
    acc[0] = fmaf(w, v.x, acc[0]);
    acc[1] = fmaf(w, v.y, acc[1]);
  }
};

template <int E>
__device__ __forceinline__ void store_out(float* o, const float* acc) {
  if constexpr (E == 4) *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  else *reinterpret_cast<float2*>(o) = make_float2(acc[0], acc[1]);
}
template <int E>
__device__ __forceinline__ void store_out(__nv_bfloat16* o, const float* acc) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0], acc[1]);
  if constexpr (E == 4) {
    const __nv_bfloat162 c = __floats2bfloat162_rn(acc[2], acc[3]);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&c);
    *reinterpret_cast<uint2*>(o) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(o) = a;
  }
}

template <int D, typename OutT>
__global__ void __launch_bounds__(THREADS) merge_kernel(const MergeArgs a) {
  constexpr int E = D / 32;
  using V = Vec<E>;
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)a.B * a.Hq * a.S;
  const int64_t warps = ((int64_t)gridDim.x * THREADS) >> 5;
  if (*reinterpret_cast<volatile int32_t*>(a.status) != 0) return;
  for (int64_t w = ((int64_t)blockIdx.x * THREADS + threadIdx.x) >> 5; w < total; w += warps) {
    const int64_t bh = w / a.S;
    const int64_t i = w - bh * a.S;
    const int p = (int)(i / a.L);
    const int64_t r = i - (int64_t)p * a.L;
    const int s0 = __ldg(a.slot_off + p);
    const int ns = __ldg(a.slot_off + p + 1) - s0;
    const int64_t base = (bh * a.n_slots + s0) * a.L + r;  // row of slot s0; slot t is t*L rows further
    const float* lse_p = a.part_lse + base;
    const typename V::T* o_p = reinterpret_cast<const typename V::T*>(a.part_o + base * D) + lane;
    const int64_t o_stride = a.L * (D / E);  // in vectors, one slot

    float M = -INFINITY;
    for (int t = lane; t < ns; t += 32) M = fmaxf(M, __ldg(lse_p + (int64_t)t * a.L));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Ms = (M == -INFINITY) ? 0.f : M;
    float W = 0.f;
    for (int t = lane; t < ns; t += 32) W += expf(__ldg(lse_p + (int64_t)t * a.L) - Ms);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    const float invW = W > 0.f ? 1.f / W : 0.f;

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int g = 0; g < ns; g += 32) {
      const int n = min(32, ns - g);
      const float wl = (lane < n) ? expf(__ldg(lse_p + (int64_t)(g + lane) * a.L) - Ms) * invW : 0.f;
      int t = 0;
      for (; t + 4 <= n; t += 4) {
        typename V::T v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = __ldcs(o_p + (int64_t)(g + t + q) * o_stride);
#pragma unroll
        for (int q = 0; q < 4; ++q) V::fma_into(acc, __shfl_sync(0xffffffffu, wl, t + q), v[q]);
      }
      for (; t < n; ++t) {
        const typename V::T v = __ldcs(o_p + (int64_t)(g + t) * o_stride);
        V::fma_into(acc, __shfl_sync(0xffffffffu, wl, t), v);
      }
    }
    store_out<E>(reinterpret_cast<OutT*>(a.O) + (bh * a.S + i) * D + lane * E, acc);
    if (lane == 0) a.LSE[bh * a.S + i] = (W > 0.f) ? Ms + logf(W) : -INFINITY;
  }
}

template <int D, typename OutT>
static int launch(const MergeArgs& a, void* stream, std::string* err) {
  const int64_t rows = (int64_t)a.B * a.Hq * a.S;
  if (rows <= 0) return (int)cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (rows + (THREADS / 32) - 1) / (THREADS / 32);
  const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 64;  // enough resident warps, grid-stride beyond
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  merge_kernel<D, OutT><<<blocks, THREADS, 0, (cudaStream_t)stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("merge launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace merge

int launch_merge(const MergeArgs& a, mesh_attn_dtype out_dtype, void* stream, std::string* err) {
  if (out_dtype == MESH_ATTN_BF16) {
    if (a.d == 128) return merge::launch<128, __nv_bfloat16>(a, stream, err);
    if (a.d == 64) return merge::launch<64, __nv_bfloat16>(a, stream, err);
  } else {
    if (a.d == 128) return merge::launch<128, float>(a, stream, err);
    if (a.d == 64) return merge::launch<64, float>(a, stream, err);
  }
  *err = "merge supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
