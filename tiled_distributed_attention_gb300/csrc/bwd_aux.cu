// The two streaming (HBM-bound) kernels around the tile backward:
//   prep:   D_i = dO_i . O_i per (batch, head, row), the row term of dS_ij = P_ij (dP_ij - D_i);
//   reduce: sum of the partial gradients of a partition over its slots -- dQ partials along the
//           mesh row (the slots of a Q partition, as the forward merges partial outputs) and dK /
//           dV partials along the mesh column (the KV slots of a KV partition) -- rounded to the
//           output type.  Mesh-Attention tile structure: "Mesh-Attention: A New
//           Communication-Efficient Distributed Attention with Improved Data Locality", tutorial
//           §"Mesh-Attention：从一维'环'到二维'网'".
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace baux {

template <typename T>
__device__ __forceinline__ void store4(T* o, float4 v);
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

// 16 bytes of a row as floats: 8 bf16 or 4 fp32 elements.
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* out) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    out[0] = v.x, out[1] = v.y, out[2] = v.z, out[3] = v.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* out) {
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
      out[2 * i] = f.x, out[2 * i + 1] = f.y;
    }
  }
};

// A row is read by LPR = D / (16 / sizeof(T)) lanes with one 16-byte load each of O and dO; a
// warp covers 32 / LPR rows per step and PREP_STEPS steps, all loads issued before the first
// product, so that every thread keeps 2 PREP_STEPS 16-byte loads in flight.
constexpr int PREP_STEPS = 4;
template <typename T, int D>
struct PrepShape {
  static constexpr int LPR = D / Vec16<T>::N;        // lanes per row
  static constexpr int RPS = 32 / LPR;               // rows per warp step
  static constexpr int ROWS_PER_WARP = RPS * PREP_STEPS;
  static constexpr int ROWS_PER_CTA = 8 * ROWS_PER_WARP;
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must split evenly over the lanes");
};

template <typename T, int D>
__global__ void __launch_bounds__(256) prep_kernel(const T* O, const T* dO, float* Dsum, int32_t* status,
                                                   int64_t rows) {
  using Sh = PrepShape<T, D>;
  constexpr int N = Vec16<T>::N;
  if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
  const int lane = threadIdx.x & 31;
  const int sub = lane / Sh::LPR, col = (lane % Sh::LPR) * N;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * Sh::ROWS_PER_WARP + sub;
  float o[PREP_STEPS][N], g[PREP_STEPS][N];
#pragma unroll
  for (int st = 0; st < PREP_STEPS; ++st) {
    const int64_t row = row0 + (int64_t)st * Sh::RPS;
    if (row < rows) {
      Vec16<T>::load(O + row * D + col, o[st]);
      Vec16<T>::load(dO + row * D + col, g[st]);
    }
  }
#pragma unroll
  for (int st = 0; st < PREP_STEPS; ++st) {
    const int64_t row = row0 + (int64_t)st * Sh::RPS;
    float acc = 0.f;
    if (row < rows) {
#pragma unroll
      for (int e = 0; e < N; ++e) acc = fmaf(o[st][e], g[st][e], acc);
    }
    // sum over the LPR lanes of the row (aligned groups of lanes)
#pragma unroll
    for (int off = Sh::LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && lane % Sh::LPR == 0) Dsum[row] = acc;
  }
}

// One CTA of 256 threads per ROWS consecutive rows of one (batch, head, partition): its share of
// each slot is one contiguous block of ROWS * D floats (16 KB), streamed with consecutive
// 16-byte loads and summed.
template <int D, typename OutT>
__global__ void __launch_bounds__(256) reduce_kernel(const ReduceArgs a, int n_rblk) {
  constexpr int ROWS = 4096 / D;
  constexpr int V4_PER_ROW = D / 4;
  constexpr int PER_THREAD = ROWS * V4_PER_ROW / 256;
  if (*reinterpret_cast<volatile int32_t*>(a.status) != 0) return;
  const int tid = threadIdx.x;
  const int rb = (int)(blockIdx.x % (unsigned)n_rblk);
  const int hp = (int)(blockIdx.x / (unsigned)n_rblk);
  const int part = hp % a.P;
  const int bh = hp / a.P;
  const int L = (int)a.L;
  const int r0 = rb * ROWS;
  const int nrows = min(ROWS, L - r0);
  const int s0 = __ldg(a.off + part);
  const int ns = __ldg(a.off + part + 1) - s0;
  if (s0 < 0 || ns < 0 || s0 + ns > a.n_slots) {
    if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 6, (int32_t)blockIdx.x);
    return;
  }
  const float4* src = reinterpret_cast<const float4*>(a.part + (((int64_t)bh * a.n_slots + s0) * L + r0) * D);
  const int64_t slot_stride = (int64_t)L * V4_PER_ROW;
  float4 acc[PER_THREAD];
#pragma unroll
  for (int k = 0; k < PER_THREAD; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t = 0; t < ns; ++t) {
#pragma unroll
    for (int k = 0; k < PER_THREAD; ++k) {
      const int idx = tid + k * 256;
      if (idx / V4_PER_ROW < nrows) {
        const float4 v = __ldcs(src + t * slot_stride + idx);
        acc[k].x += v.x;
        acc[k].y += v.y;
        acc[k].z += v.z;
        acc[k].w += v.w;
      }
    }
  }
  OutT* out = reinterpret_cast<OutT*>(a.out) + ((int64_t)bh * a.S + (int64_t)part * L + r0) * D;
#pragma unroll
  for (int k = 0; k < PER_THREAD; ++k) {
    const int idx = tid + k * 256;
    if (idx / V4_PER_ROW < nrows) store4<OutT>(out + (int64_t)idx * 4, acc[k]);
  }
}

template <typename T, int D>
int launch_prep(const PrepArgs& a, void* stream, std::string* err) {
  const int64_t rows = (int64_t)a.B * a.H * a.S;
  constexpr int64_t per_cta = PrepShape<T, D>::ROWS_PER_CTA;
  const int64_t blocks = (rows + per_cta - 1) / per_cta;
  if (blocks <= 0) return (int)cudaSuccess;
  if (blocks > 0x7fffffff) {
    *err = "too many rows for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  prep_kernel<T, D><<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      static_cast<const T*>(a.O), static_cast<const T*>(a.dO), a.D, a.status, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("bwd prep launch: ") + cudaGetErrorString(e);
  return (int)e;
}

template <int D, typename OutT>
int launch_reduce(const ReduceArgs& a, void* stream, std::string* err) {
  constexpr int ROWS = 4096 / D;
  const int64_t n_rblk = (a.L + ROWS - 1) / ROWS;
  const int64_t blocks = (int64_t)a.B * a.H * a.P * n_rblk;
  if (blocks <= 0) return (int)cudaSuccess;
  if (blocks > 0x7fffffff || a.L > 0x7fffffff) {
    *err = "too many reduce blocks for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  reduce_kernel<D, OutT><<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a, (int)n_rblk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("bwd reduce launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace baux

int launch_bwd_prep(const PrepArgs& a, mesh_attn_dtype dt, void* stream, std::string* err) {
  if (dt == MESH_ATTN_BF16) {
    if (a.d == 128) return baux::launch_prep<__nv_bfloat16, 128>(a, stream, err);
    if (a.d == 64) return baux::launch_prep<__nv_bfloat16, 64>(a, stream, err);
  } else {
    if (a.d == 128) return baux::launch_prep<float, 128>(a, stream, err);
    if (a.d == 64) return baux::launch_prep<float, 64>(a, stream, err);
  }
  *err = "backward prep supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

int launch_bwd_reduce(const ReduceArgs& a, mesh_attn_dtype out_dtype, void* stream, std::string* err) {
  if (out_dtype == MESH_ATTN_BF16) {
    if (a.d == 128) return baux::launch_reduce<128, __nv_bfloat16>(a, stream, err);
    if (a.d == 64) return baux::launch_reduce<64, __nv_bfloat16>(a, stream, err);
  } else {
    if (a.d == 128) return baux::launch_reduce<128, float>(a, stream, err);
    if (a.d == 64) return baux::launch_reduce<64, float>(a, stream, err);
  }
  *err = "backward reduce supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
