// LSE merge of the partial outputs of one Q partition's tiles: for every (batch, head, row),
//   M = max_t lse_t,  lse = M + ln sum_t exp(lse_t - M),  O = sum_t exp(lse_t - lse) O_t.
// This is the combine step the Mesh-Attention Q owner performs on the partial results its
// mesh row sends back ("Mesh-Attention: A New Communication-Efficient Distributed Attention
// with Improved Data Locality", tutorial §"Mesh-Attention：从一维'环'到二维'网'"), with the
// log-sum-exp rescaling of "环形注意力：突破长序列处理瓶颈的分布式计算范式",
// §"数值稳定性：Log-Sum-Exp技术的分布式应用".
//
// A streaming HBM-bound kernel.  One CTA of 256 threads owns ROWS consecutive rows of one
// (batch, head, partition); because the slots of a partition hold the same rows at a stride of
// L rows, the CTA's share of each slot is one contiguous block of ROWS * d floats (16 KB).
//   0. the loads of the first two slots' blocks go out first (they do not need the weights);
//   1. the CTA reads its ROWS x n_slots LSE values (coalesced per slot) into shared memory;
//   2. one warp turns them into per-row weights exp(lse_t - lse) and writes the row LSE;
//   3. every thread streams 16-byte pieces of each slot's contiguous block (consecutive
//      threads, consecutive addresses), scales them by the row weight and accumulates;
//   4. the d/4 float4 sums per row are written as 8-byte bf16 (or 16-byte fp32) stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace merge {

constexpr int THREADS = 256;
constexpr int MAX_SLOTS = 64;  // R <= 64 for P <= 4096

template <typename OutT>
__device__ __forceinline__ void store4(OutT* o, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* o, float4 v) {
  *reinterpret_cast<float4*>(o) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* o, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(o) = w;
}

template <int D, typename OutT>
__global__ void __launch_bounds__(THREADS) merge_kernel(const MergeArgs a, int n_rblk) {
  constexpr int ROWS = 4096 / D;                // 16 KB of fp32 per slot per CTA
  constexpr int V4_PER_ROW = D / 4;
  constexpr int PER_THREAD = ROWS * V4_PER_ROW / THREADS;  // float4 outputs per thread (4)
  __shared__ float w_s[MAX_SLOTS][ROWS];
  if (*reinterpret_cast<volatile int32_t*>(a.status) != 0) return;
  const int tid = threadIdx.x;
  // CTA -> (bh, p, row block); 32-bit arithmetic: B*Hq*P*n_rblk < 2^31 is checked on the host
  const int rb = (int)(blockIdx.x % (unsigned)n_rblk);
  const int bhp = (int)(blockIdx.x / (unsigned)n_rblk);
  const int p = bhp % a.P;
  const int bh = bhp / a.P;
  const int L = (int)a.L;
  const int r0 = rb * ROWS;
  const int nrows = min(ROWS, L - r0);
  const int s0 = __ldg(a.slot_off + p);
  const int ns = __ldg(a.slot_off + p + 1) - s0;
  if (ns > MAX_SLOTS) {
    if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 5, (int32_t)blockIdx.x);
    return;
  }
  const int64_t row_base = ((int64_t)bh * a.n_slots + s0) * L + r0;  // slot s0, row r0
  const float4* src = reinterpret_cast<const float4*>(a.part_o + row_base * D);
  const int64_t slot_stride = (int64_t)L * V4_PER_ROW;  // float4 per slot

  // 0. the first two slots' blocks do not depend on the weights: their loads go out first and
  //    land while the LSEs are read and the weights computed
  float4 v[2][PER_THREAD];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int k = 0; k < PER_THREAD; ++k) {
      const int idx = tid + k * THREADS;
      v[q][k] = (q < ns && idx / V4_PER_ROW < nrows) ? __ldcs(src + q * slot_stride + idx)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }

  // 1. slot LSEs of the CTA's rows
  for (int i = tid; i < ns * ROWS; i += THREADS) {
    const int t = i / ROWS, r = i - t * ROWS;
    w_s[t][r] = (r < nrows) ? __ldg(a.part_lse + row_base + (int64_t)t * L + r) : -INFINITY;
  }
  __syncthreads();
  // 2. weights exp(lse_t - lse) and the row LSE
  if (tid < ROWS) {
    const int r = tid;
    float M = -INFINITY;
    for (int t = 0; t < ns; ++t) M = fmaxf(M, w_s[t][r]);
    const float Ms = (M == -INFINITY) ? 0.f : M;
    float W = 0.f;
    for (int t = 0; t < ns; ++t) {
      const float e = __expf(w_s[t][r] - Ms);
      w_s[t][r] = e;
      W += e;
    }
    const float invW = W > 0.f ? 1.f / W : 0.f;
    for (int t = 0; t < ns; ++t) w_s[t][r] *= invW;
    if (r < nrows) a.LSE[(int64_t)bh * a.S + (int64_t)p * L + r0 + r] = (W > 0.f) ? Ms + logf(W) : -INFINITY;
  }
  __syncthreads();
  // 3. stream each slot's contiguous block (slots 0 and 1 are already in registers)
  float4 acc[PER_THREAD];
#pragma unroll
  for (int k = 0; k < PER_THREAD; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < 2; ++q)
    if (q < ns) {
#pragma unroll
      for (int k = 0; k < PER_THREAD; ++k) {
        const float w = w_s[q][(tid + k * THREADS) / V4_PER_ROW];
        acc[k].x = fmaf(w, v[q][k].x, acc[k].x);
        acc[k].y = fmaf(w, v[q][k].y, acc[k].y);
        acc[k].z = fmaf(w, v[q][k].z, acc[k].z);
        acc[k].w = fmaf(w, v[q][k].w, acc[k].w);
      }
    }
  int t = 2;
  for (; t + 2 <= ns; t += 2) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < PER_THREAD; ++k) {
        const int idx = tid + k * THREADS;
        v[q][k] = (idx / V4_PER_ROW < nrows) ? __ldcs(src + (t + q) * slot_stride + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < PER_THREAD; ++k) {
        const float w = w_s[t + q][(tid + k * THREADS) / V4_PER_ROW];
        acc[k].x = fmaf(w, v[q][k].x, acc[k].x);
        acc[k].y = fmaf(w, v[q][k].y, acc[k].y);
        acc[k].z = fmaf(w, v[q][k].z, acc[k].z);
        acc[k].w = fmaf(w, v[q][k].w, acc[k].w);
      }
  }
  for (; t < ns; ++t) {
#pragma unroll
    for (int k = 0; k < PER_THREAD; ++k) {
      const int idx = tid + k * THREADS;
      if (idx / V4_PER_ROW < nrows) {
        const float4 v = __ldcs(src + t * slot_stride + idx);
        const float w = w_s[t][idx / V4_PER_ROW];
        acc[k].x = fmaf(w, v.x, acc[k].x);
        acc[k].y = fmaf(w, v.y, acc[k].y);
        acc[k].z = fmaf(w, v.z, acc[k].z);
        acc[k].w = fmaf(w, v.w, acc[k].w);
      }
    }
  }
  // 4. output rows r0 .. r0 + nrows of O[bh, p*L + r, :]
  OutT* out = reinterpret_cast<OutT*>(a.O) + ((int64_t)bh * a.S + (int64_t)p * L + r0) * D;
#pragma unroll
  for (int k = 0; k < PER_THREAD; ++k) {
    const int idx = tid + k * THREADS;
    if (idx / V4_PER_ROW < nrows) store4<OutT>(out + (int64_t)idx * 4, acc[k]);
  }
}

template <int D, typename OutT>
static int launch(const MergeArgs& a, void* stream, std::string* err) {
  constexpr int ROWS = 4096 / D;
  const int64_t n_rblk = (a.L + ROWS - 1) / ROWS;
  const int64_t blocks = (int64_t)a.B * a.Hq * a.P * n_rblk;
  if (blocks <= 0) return (int)cudaSuccess;
  if (blocks > 0x7fffffff || a.L > 0x7fffffff) {
    *err = "too many merge blocks for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  merge_kernel<D, OutT><<<(unsigned)blocks, THREADS, 0, (cudaStream_t)stream>>>(a, (int)n_rblk);
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
