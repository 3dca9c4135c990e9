// Tile attention backward on the CUDA cores, fp32 throughout: the path for fp32 inputs.
//
// The gradients of the forward definition, per tile (the Mesh-Attention tile structure of the
// forward, "Mesh-Attention: A New Communication-Efficient Distributed Attention with Improved
// Data Locality", tutorial §"Mesh-Attention：从一维'环'到二维'网'"):
//   P_ij = exp(s_ij - LSE_i) with the global LSE, dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - D_i)
//   with D_i = dO_i . O_i;  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
//   dV_j = sum_i P_ij dO_i.
// Two kernels, each writing fp32 partial sums that the reduce kernel adds up:
//   dq:   per forward work item (p, t): the sums over the tile's KV partitions of p, into the
//         item's partial slot.  A CTA of 4 warps owns 32 query rows; keys are staged 32 at a
//         time; lane j forms s, dP and dS of key j against the warp's 8 rows, and each lane
//         accumulates d/32 columns of dQ for the 8 rows.
//   dkdv: per KV slot (k, t): the sums over the tile's live Q partitions for k and over the
//         query heads of k's KV head, into the slot.  A CTA owns 32 keys (8 per warp); query
//         rows are staged 32 at a time; lane i forms P and dS of row i against the warp's keys,
//         and each lane accumulates d/32 columns of dK and dV for the 8 keys.
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace bsimt {

constexpr int BLK = 32;     // rows (dq) or keys (dkdv) per CTA
constexpr int PER_W = 8;    // per warp
constexpr int CHUNK = 32;   // staged keys (dq) or rows (dkdv)
constexpr int THREADS = 128;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}

template <int D>
__global__ void __launch_bounds__(THREADS) dq_kernel(const BwdArgs a, int n_rb) {
  constexpr int KP = D + 4;  // padded rows: conflict-free float4 reads across lanes
  constexpr int E = D / 32;
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [BLK][D]
  float* Gs = Qs + BLK * D;                     // dO rows [BLK][D]
  float* Ks = Gs + BLK * D;                     // [CHUNK][KP]
  float* Vs = Ks + CHUNK * KP;                  // [CHUNK][KP]
  float* Ds = Vs + CHUNK * KP;                  // dS [4][PER_W][CHUNK]
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
  const int64_t row0 = (int64_t)rb * BLK;
  const int64_t grow0 = (int64_t)it.p * L + row0;  // global position of the CTA's first row
  const int64_t qbase = ((int64_t)b * a.Hq + h) * a.S;
  const float* Qg = static_cast<const float*>(a.Q) + (qbase + grow0) * D;
  const float* Gg = static_cast<const float*>(a.dO) + (qbase + grow0) * D;
  const float* Kg = static_cast<const float*>(a.K) + ((int64_t)b * a.Hkv + hk) * a.S * D;
  const float* Vg = static_cast<const float*>(a.V) + ((int64_t)b * a.Hkv + hk) * a.S * D;
  for (int i = tid; i < BLK * D; i += THREADS) {
    const bool in = row0 + i / D < L;
    Qs[i] = in ? Qg[i] : 0.f;
    Gs[i] = in ? Gg[i] : 0.f;
  }
  const int wrow0 = warp * PER_W;
  float lse2[PER_W], dsum[PER_W], acc[PER_W][E];
#pragma unroll
  for (int i = 0; i < PER_W; ++i) {
    const int64_t row = row0 + wrow0 + i;
    const bool in = row < L;
    const float lse = in ? a.LSE[qbase + grow0 + wrow0 + i] : -INFINITY;
    lse2[i] = lse * LOG2E;  // -inf for a row with no visible key: it contributes nothing
    dsum[i] = in ? a.D[qbase + grow0 + wrow0 + i] : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  }

  for (int ki = 0; ki < it.n_kv; ++ki) {
    const int k = a.kv_list[it.kv_off + ki];
    if (k < 0 || k >= a.P) {
      if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 3, (int32_t)blockIdx.x);
      return;
    }
    const bool diag = a.causal && k == it.p;
    const int64_t n_keys = diag ? min(L, row0 + BLK) : L;
    for (int64_t c0 = 0; c0 < n_keys; c0 += CHUNK) {
      __syncthreads();
      for (int i = tid; i < CHUNK * D; i += THREADS) {
        const int j = i / D, e = i % D;
        const int64_t key = c0 + j;
        const bool in = key < n_keys;
        const int64_t g = ((int64_t)k * L + key) * D + e;
        Ks[j * KP + e] = in ? Kg[g] : 0.f;
        Vs[j * KP + e] = in ? Vg[g] : 0.f;
      }
      __syncthreads();
      float s[PER_W], dp[PER_W];
#pragma unroll
      for (int i = 0; i < PER_W; ++i) s[i] = dp[i] = 0.f;
      const float4* kr = reinterpret_cast<const float4*>(Ks + lane * KP);
      const float4* vr = reinterpret_cast<const float4*>(Vs + lane * KP);
#pragma unroll 4
      for (int e4 = 0; e4 < D / 4; ++e4) {
        const float4 kv = kr[e4], vv = vr[e4];
#pragma unroll
        for (int i = 0; i < PER_W; ++i) {
          s[i] = dot4(reinterpret_cast<const float4*>(Qs + (wrow0 + i) * D)[e4], kv, s[i]);
          dp[i] = dot4(reinterpret_cast<const float4*>(Gs + (wrow0 + i) * D)[e4], vv, dp[i]);
        }
      }
      const int64_t key = c0 + lane;
#pragma unroll
      for (int i = 0; i < PER_W; ++i) {
        const int64_t row = row0 + wrow0 + i;
        const bool vis = key < n_keys && (!diag || key <= row) && lse2[i] > -INFINITY;
        const float p = vis ? exp2f(s[i] * a.scale_log2 - lse2[i]) : 0.f;
        Ds[(warp * PER_W + i) * CHUNK + lane] = p * (dp[i] - dsum[i]);
      }
      __syncwarp();
#pragma unroll 4
      for (int j = 0; j < CHUNK; ++j) {
        float kc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) kc[e] = Ks[j * KP + lane + 32 * e];
#pragma unroll
        for (int i = 0; i < PER_W; ++i) {
          const float ds = Ds[(warp * PER_W + i) * CHUNK + j];
#pragma unroll
          for (int e = 0; e < E; ++e) acc[i][e] = fmaf(ds, kc[e], acc[i][e]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < PER_W; ++i) {
    const int64_t row = row0 + wrow0 + i;
    if (row >= L) continue;
    const int64_t prow = (((int64_t)b * a.Hq + h) * a.n_slots + it.slot) * L + row;
#pragma unroll
    for (int e = 0; e < E; ++e) a.dq_part[prow * D + lane + 32 * e] = acc[i][e] * a.scale;
  }
}

template <int D>
__global__ void __launch_bounds__(THREADS) dkdv_kernel(const BwdArgs a, int n_kb) {
  constexpr int KP = D + 4;
  constexpr int E = D / 32;
  extern __shared__ float4 smem4[];
  float* Ks = reinterpret_cast<float*>(smem4);  // [BLK][D] the CTA's keys
  float* Vs = Ks + BLK * D;                     // [BLK][D]
  float* Qs = Vs + BLK * D;                     // [CHUNK][KP] staged query rows
  float* Gs = Qs + CHUNK * KP;                  // [CHUNK][KP] their dO rows
  float* Ps = Gs + CHUNK * KP;                  // P  [4][PER_W][CHUNK]
  float* Ds = Ps + 4 * PER_W * CHUNK;           // dS [4][PER_W][CHUNK]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int64_t u = blockIdx.x;
  const int kb = (int)(u % n_kb); u /= n_kb;
  const int hk = (int)(u % a.Hkv); u /= a.Hkv;
  const int b = (int)(u % a.B);
  const int idx = (int)(u / a.B);
  if (*reinterpret_cast<volatile int32_t*>(a.status) != 0) return;
  const DevItem it = a.kv_items[idx];  // {k, kv slot, q_off, n_q}
  if (it.p < 0 || it.p >= a.P || it.slot < 0 || it.slot >= a.n_kv_slots || it.n_kv < 1 || it.kv_off < 0) {
    if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 4, (int32_t)blockIdx.x);
    return;
  }
  const int k = it.p;
  const int64_t L = a.L;
  const int g = a.Hq / a.Hkv;
  const int64_t key0 = (int64_t)kb * BLK;           // first key of the CTA within partition k
  const int64_t gkey0 = (int64_t)k * L + key0;
  const int64_t kvbase = ((int64_t)b * a.Hkv + hk) * a.S;
  const float* Kg = static_cast<const float*>(a.K) + (kvbase + gkey0) * D;
  const float* Vg = static_cast<const float*>(a.V) + (kvbase + gkey0) * D;
  for (int i = tid; i < BLK * D; i += THREADS) {
    const bool in = key0 + i / D < L;
    Ks[i] = in ? Kg[i] : 0.f;
    Vs[i] = in ? Vg[i] : 0.f;
  }
  const int wkey0 = warp * PER_W;
  float dk[PER_W][E], dv[PER_W][E];
#pragma unroll
  for (int j = 0; j < PER_W; ++j)
#pragma unroll
    for (int e = 0; e < E; ++e) dk[j][e] = dv[j][e] = 0.f;

  for (int hh = 0; hh < g; ++hh) {
    const int h = hk * g + hh;
    const int64_t qbase = ((int64_t)b * a.Hq + h) * a.S;
    for (int qi = 0; qi < it.n_kv; ++qi) {
      const int p = a.q_list[it.kv_off + qi];
      if (p < 0 || p >= a.P) {
        if (tid == 0) record_error(a.status, MESH_ATTN_ERR_OUT_OF_RANGE, 3, (int32_t)blockIdx.x);
        return;
      }
      const bool diag = a.causal && p == k;
      // on the diagonal partition, rows before the CTA's first key see none of its keys
      const int64_t r_begin = diag ? (key0 / CHUNK) * CHUNK : 0;
      for (int64_t c0 = r_begin; c0 < L; c0 += CHUNK) {
        __syncthreads();
        for (int i = tid; i < CHUNK * D; i += THREADS) {
          const int r = i / D, e = i % D;
          const bool in = c0 + r < L;
          const int64_t gi = (qbase + (int64_t)p * L + c0 + r) * D + e;
          Qs[r * KP + e] = in ? static_cast<const float*>(a.Q)[gi] : 0.f;
          Gs[r * KP + e] = in ? static_cast<const float*>(a.dO)[gi] : 0.f;
        }
        __syncthreads();
        const int64_t row = c0 + lane;
        const bool row_in = row < L;
        const float lse2 = row_in ? a.LSE[qbase + (int64_t)p * L + row] * LOG2E : -INFINITY;
        const float dsum = row_in ? a.D[qbase + (int64_t)p * L + row] : 0.f;
        float s[PER_W], dp[PER_W];
#pragma unroll
        for (int j = 0; j < PER_W; ++j) s[j] = dp[j] = 0.f;
        const float4* qr = reinterpret_cast<const float4*>(Qs + lane * KP);
        const float4* gr = reinterpret_cast<const float4*>(Gs + lane * KP);
#pragma unroll 4
        for (int e4 = 0; e4 < D / 4; ++e4) {
          const float4 qv = qr[e4], gv = gr[e4];
#pragma unroll
          for (int j = 0; j < PER_W; ++j) {
            s[j] = dot4(qv, reinterpret_cast<const float4*>(Ks + (wkey0 + j) * D)[e4], s[j]);
            dp[j] = dot4(gv, reinterpret_cast<const float4*>(Vs + (wkey0 + j) * D)[e4], dp[j]);
          }
        }
#pragma unroll
        for (int j = 0; j < PER_W; ++j) {
          const int64_t key = key0 + wkey0 + j;
          const bool vis = row_in && key < L && (!diag || key <= row) && lse2 > -INFINITY;
          const float pj = vis ? exp2f(s[j] * a.scale_log2 - lse2) : 0.f;
          Ps[(warp * PER_W + j) * CHUNK + lane] = pj;
          Ds[(warp * PER_W + j) * CHUNK + lane] = pj * (dp[j] - dsum);
        }
        __syncwarp();
#pragma unroll 4
        for (int r = 0; r < CHUNK; ++r) {
          float qc[E], gc[E];
#pragma unroll
          for (int e = 0; e < E; ++e) {
            qc[e] = Qs[r * KP + lane + 32 * e];
            gc[e] = Gs[r * KP + lane + 32 * e];
          }
#pragma unroll
          for (int j = 0; j < PER_W; ++j) {
            const float pj = Ps[(warp * PER_W + j) * CHUNK + r];
            const float ds = Ds[(warp * PER_W + j) * CHUNK + r];
#pragma unroll
            for (int e = 0; e < E; ++e) {
              dv[j][e] = fmaf(pj, gc[e], dv[j][e]);
              dk[j][e] = fmaf(ds, qc[e], dk[j][e]);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < PER_W; ++j) {
    const int64_t key = key0 + wkey0 + j;
    if (key >= L) continue;
    const int64_t prow = (((int64_t)b * a.Hkv + hk) * a.n_kv_slots + it.slot) * L + key;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      a.dk_part[prow * D + lane + 32 * e] = dk[j][e] * a.scale;
      a.dv_part[prow * D + lane + 32 * e] = dv[j][e];
    }
  }
}

template <int D>
static int launch(const BwdArgs& a, void* stream, std::string* err) {
  const int64_t n_b = (a.L + BLK - 1) / BLK;
  const int64_t dq_blocks = (int64_t)a.n_items * a.B * a.Hq * n_b;
  const int64_t kv_blocks = (int64_t)a.n_kv_items * a.B * a.Hkv * n_b;
  if (dq_blocks > 0x7fffffff || kv_blocks > 0x7fffffff) {
    *err = "too many work units for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  const size_t dq_smem = sizeof(float) * (2 * BLK * D + 2 * CHUNK * (D + 4) + 4 * PER_W * CHUNK);
  const size_t kv_smem = sizeof(float) * (2 * BLK * D + 2 * CHUNK * (D + 4) + 8 * PER_W * CHUNK);
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dq_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kv_smem);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  if (dq_blocks > 0)
    dq_kernel<D><<<dim3((unsigned)dq_blocks), dim3(THREADS), dq_smem, (cudaStream_t)stream>>>(a, (int)n_b);
  if (kv_blocks > 0)
    dkdv_kernel<D><<<dim3((unsigned)kv_blocks), dim3(THREADS), kv_smem, (cudaStream_t)stream>>>(a, (int)n_b);
  e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("tile_bwd_simt launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace bsimt

int launch_tile_bwd_simt(const BwdArgs& a, void* stream, std::string* err) {
  if (a.d == 128) return bsimt::launch<128>(a, stream, err);
  if (a.d == 64) return bsimt::launch<64>(a, stream, err);
  *err = "CUDA-core backward supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
