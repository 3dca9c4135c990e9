// Tile attention backward on the 5th-generation tensor cores (sm_103a), bf16 inputs.
//
// The gradients of the forward definition (the left-hand side of "环形注意力：突破长序列处理
// 瓶颈的分布式计算范式", §"理论奠基"), per tile of the Mesh-Attention plan ("Mesh-Attention: A New
// Communication-Efficient Distributed Attention with Improved Data Locality", tutorial
// §"Mesh-Attention：从一维'环'到二维'网'"), with the forward's global LSE and D_i = dO_i . O_i:
//   P_ij = exp(s_ij - LSE_i),  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
// Two kernels; one CTA owns one 128-row tile of one unit (no persistence) with 10 warps:
//   warps 0-7  elementwise: two warps per TMEM lane quadrant, one thread per TMEM lane (a key row
//              in dkdv, a query row in dq), each warp taking 64 of the block's 128 columns
//   warp 8     MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M = N = 128, K = 16, issued by an
//              elected lane of the converged warp; completion by tcgen05.commit
//   warp 9     producer: TMA loads of 128 x 64 bf16 boxes with 128-byte swizzle
//
// dkdv (unit = KV slot, batch, KV head, 128-key block): K and V stay in shared memory; Q and dO
// blocks of the slot's query rows (over the KV head's query heads) stream through three and two
// stages (Q feeds S^T one block ahead of its last use).
//   TMEM: S^T | dP^T | dV | dK   (S^T = K Q^T and dP^T = V dO^T have lanes = keys; P^T and dS^T
//   are written back as bf16 into the first half of their columns and feed dV += P^T dO and
//   dK += dS^T Q from TMEM).  Issue order per query block i:
//     [P^T(i) ready] dV(i), S^T(i+1)   [dS^T(i) ready] dK(i), dP^T(i+1)
//   so the exponentials of block i+1 overlap dK(i) and dP^T(i+1), and dS^T(i+1) overlaps
//   dV(i+1) and S^T(i+2).  LSE and D of the block's query columns are broadcast from shared
//   memory.
// dq (unit = forward work item, batch, head, 128-row block): Q and dO stay in shared memory; K
//   and V blocks of the item's KV partitions stream through three and two stages.
//   TMEM: S(even) | S(odd) | dP | dQ: S(j+2) is issued as soon as its K block has landed, so
//   the exponentials of block j+1 run while dQ(j) and dP(j+1) execute.  LSE and D of a row are
//   thread-local.
// Every mbarrier wait is bounded; a timeout records MESH_ATTN_ERR_DEVICE_TIMEOUT, the CTA stops,
// drains its copies and products and frees its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace btc {

constexpr int BM = 128;  // rows per tile = TMEM lanes = keys / queries per block
constexpr int NUM_THREADS = 320;
constexpr int N_EW = 8;  // elementwise warps: two per TMEM lane quadrant, 64 columns each
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
// The bf16 P / dS written back into TMEM by column half `hf` land in packed columns
// [64 hf, 64 hf + 32) of their region -- inside the half's own input columns, so the halves never
// overwrite values the other still has to read -- and the MMAs that take them as A read K-step kk
// (16 elements = 8 packed columns) from here:
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }
constexpr int64_t DRAIN_NS = 200000000;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int ROLE_EW = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_ITEM = 4;

struct Params {
  const DevItem* items;
  const int32_t* kv_list;
  const DevItem* kv_items;
  const int32_t* q_list;
  const float* lse;
  const float* dsum;
  float* dq_part;
  float* dk_part;
  float* dv_part;
  int32_t* status;
  int64_t S, L;
  int32_t B, Hq, Hkv, P, n_items, n_slots, n_kv_items, n_kv_slots, nb, causal;
  float scale, scale_log2;
  int64_t wait_limit_ns;
};

// Shared memory: the resident pair (K, V in dkdv; Q, dO in dq), NSA stages of stream A (the
// operand of the S product, needed two blocks ahead: Q in dkdv, K in dq) and NSB stages of
// stream B (dO in dkdv, V in dq).  224 KB for d = 128 leaves no room to align the base by hand:
// the kernels check that the dynamic shared window starts 1024-aligned (it does on sm_100-class
// parts, whose window starts at a 1 KB-aligned offset) and report MESH_ATTN_ERR_INTERNAL if not.
template <int D>
struct Layout {
  static constexpr uint32_t TILE = BM * D * 2;  // one 128-row bf16 block
  static constexpr uint32_t BOX = BM * 64 * 2;  // one 128 x 64 TMA box
  static constexpr int NSA = 3, NSB = 2;
  static constexpr uint32_t RES0 = 0, RES1 = TILE;
  static constexpr uint32_t A0 = 2 * TILE;             // stream A stage s at A0 + s TILE
  static constexpr uint32_t B0 = A0 + NSA * TILE;      // stream B stage s at B0 + s TILE
  static constexpr uint32_t VEC_OFF = B0 + NSB * TILE;  // dkdv: lse2[2][128], dsum[2][128] fp32
  static constexpr uint32_t BAR_OFF = VEC_OFF + 4 * BM * 4;
  static constexpr int B_RES = 0, B_AF = 1, B_AE = B_AF + NSA, B_BF = B_AE + NSA, B_BE = B_BF + NSB,
                       B_S = B_BE + NSB, B_DP = B_S + 2, B_P = B_DP + 1, B_DS = B_P + 1, B_ACC = B_DS + 1,
                       B_DRAIN = B_ACC + 1, B_VEC = B_DRAIN + 1, NBARS = B_VEC + 2;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr uint32_t TOTAL = MISC_OFF + 16;
  static constexpr uint32_t ALLOC = TOTAL;
};

// 128-row blocks of partition `k` (keys, dq kernel) visited by query block `qb` of partition
// `p`: on the causal diagonal partition only blocks up to the query block.
__device__ __forceinline__ int kblocks_of(int k, int p, int causal, int nb, int qb) {
  return (causal && k == p) ? min(nb, qb + 1) : nb;
}
// query blocks of partition `p` visited by key block `kb` of partition `k` (dkdv kernel)
__device__ __forceinline__ int qblock_begin(int k, int p, int causal, int kb) { return (causal && k == p) ? kb : 0; }

__device__ __forceinline__ float4 shfl4(float4 x, int src) {
  x.x = __shfl_sync(0xffffffffu, x.x, src);
  x.y = __shfl_sync(0xffffffffu, x.y, src);
  x.z = __shfl_sync(0xffffffffu, x.z, src);
  x.w = __shfl_sync(0xffffffffu, x.w, src);
  return x;
}

// Store one warp's 32 x 32 fp32 chunk -- lane r holds columns [c, c + 32) of row row0 + r, times
// `mul` -- into a row-major [rows][D] buffer.  Each group of four lanes transposes its 4 x 4
// matrix of 16-byte pieces (two exchange steps: lanes ^ 2, then lanes ^ 1), after which lane
// 4a + i holds piece i of rows 4a .. 4a + 3; so each store instruction writes eight 64-byte row
// segments (whole sectors) instead of 32 scattered 16-byte pieces, without shared memory.  Rows
// from `rows_valid` on are not written.
template <int D>
__device__ __forceinline__ void store_rows(const float (&v)[32], float mul, float* dst, int64_t row0,
                                           int rows_valid, int c, int lane) {
  const int i = lane & 3, rbase = lane & ~3;
  const bool hi = (i & 2) != 0, odd = (i & 1) != 0;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float4 e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int o = 16 * blk + 4 * q;
      e[q] = make_float4(v[o] * mul, v[o + 1] * mul, v[o + 2] * mul, v[o + 3] * mul);
    }
    {  // swap the off-diagonal 2 x 2 blocks with lane ^ 2
      const float4 r0 = shfl4(hi ? e[0] : e[2], lane ^ 2), r1 = shfl4(hi ? e[1] : e[3], lane ^ 2);
      if (hi) {
        e[0] = r0;
        e[1] = r1;
      } else {
        e[2] = r0;
        e[3] = r1;
      }
    }
    {  // swap within the 2 x 2 blocks with lane ^ 1
      const float4 r0 = shfl4(odd ? e[0] : e[1], lane ^ 1), r1 = shfl4(odd ? e[2] : e[3], lane ^ 1);
      if (odd) {
        e[0] = r0;
        e[2] = r1;
      } else {
        e[1] = r0;
        e[3] = r1;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (rbase + j < rows_valid)
        *reinterpret_cast<float4*>(dst + (row0 + rbase + j) * D + c + 16 * blk + 4 * i) = e[j];
  }
}

// Walk over the key blocks of a dq unit in the order the producer loads them: the tile's KV
// partitions, then the partition's blocks (on the causal diagonal only up to the query block).
struct KCursor {
  int ki, kp, kb, n;
  __device__ __forceinline__ void load(const Params& prm, const DevItem& it, int p, int qb) {
    kp = __ldg(prm.kv_list + it.kv_off + ki);
    kb = 0;
    n = kblocks_of(kp, p, prm.causal, prm.nb, qb);
  }
  __device__ __forceinline__ void start(const Params& prm, const DevItem& it, int p, int qb) {
    ki = 0;
    load(prm, it, p, qb);
  }
  __device__ __forceinline__ void step(const Params& prm, const DevItem& it, int p, int qb) {
    if (++kb < n) return;
    ++ki;
    if (ki < it.n_kv) load(prm, it, p, qb);
    else kp = -1;
  }
};

// Walk over the query blocks of a dkdv unit in the order the producer loads them: heads of the
// group, then the slot's Q partitions, then the partition's blocks.
struct QCursor {
  int h, qi, p, qb;
  __device__ __forceinline__ void load(const Params& prm, const DevItem& it, int k, int kb) {
    p = __ldg(prm.q_list + it.kv_off + qi);
    qb = qblock_begin(k, p, prm.causal, kb);
  }
  __device__ __forceinline__ void start(const Params& prm, const DevItem& it, int k, int kb, int h0) {
    h = h0;
    qi = 0;
    load(prm, it, k, kb);
  }
  __device__ __forceinline__ void step(const Params& prm, const DevItem& it, int k, int kb) {
    if (++qb < prm.nb) return;
    if (++qi >= it.n_kv) {
      qi = 0;
      ++h;
    }
    load(prm, it, k, kb);
  }
};

// Descriptor offsets (16-byte units) of a 128-row operand made of 64-column SW128 boxes.
template <int D>
__device__ __forceinline__ uint64_t kmaj_off(int kk) {
  return (uint64_t)((kk >> 2) * (Layout<D>::BOX >> 4) + (kk & 3) * 2);
}

// ================================================================== dK / dV
template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const Params prm) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = smem_u32(smem_raw);
  if (sb & 1023u) {  // 128-byte swizzle atoms need 1024-aligned operands (see Layout)
    if (threadIdx.x == 0) record_error(prm.status, MESH_ATTN_ERR_INTERNAL, ROLE_ITEM, (int32_t)blockIdx.x);
    return;
  }
  uint8_t* smem = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + Ly::BAR_OFF + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 4);
  float* nlse_s = reinterpret_cast<float*>(smem + Ly::VEC_OFF);  // [2][BM] -LSE log2 e of the query columns
  float* ndsum_s = nlse_s + 2 * BM;                              // [2][BM] -D
  const int64_t L = prm.L;

  // unit -> (KV slot, batch, KV head, key block)
  int64_t uu = blockIdx.x;
  const int kb = (int)(uu % prm.nb); uu /= prm.nb;
  const int hk = (int)(uu % prm.Hkv); uu /= prm.Hkv;
  const int b = (int)(uu % prm.B);
  const int idx = (int)(uu / prm.B);
  const DevItem it = prm.kv_items[idx];  // {k, kv slot, q_off, n_q}
  const bool unit_ok = it.p >= 0 && it.p < prm.P && it.slot >= 0 && it.slot < prm.n_kv_slots && it.n_kv >= 1 &&
                       it.kv_off >= 0;
  const int k = it.p;
  const int g = prm.Hq / prm.Hkv;
  // query blocks of the unit: heads of the group x Q partitions of the slot x blocks
  int NBQ = 0;
  if (unit_ok)
    for (int qi = 0; qi < it.n_kv; ++qi) {
      const int p = __ldg(prm.q_list + it.kv_off + qi);
      NBQ += prm.nb - qblock_begin(k, p, prm.causal, kb);
    }
  NBQ *= g;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_RES), 1);
    for (int s = 0; s < Ly::NSA; ++s) {
      mbar_init(bar(Ly::B_AF + s), 1);
      mbar_init(bar(Ly::B_AE + s), 1);
    }
    for (int s = 0; s < Ly::NSB; ++s) {
      mbar_init(bar(Ly::B_BF + s), 1);
      mbar_init(bar(Ly::B_BE + s), 1);
    }
    mbar_init(bar(Ly::B_S), 1);
    mbar_init(bar(Ly::B_S + 1), 1);
    mbar_init(bar(Ly::B_DP), 1);
    mbar_init(bar(Ly::B_P), N_EW);  // one lane of each elementwise warp
    mbar_init(bar(Ly::B_DS), N_EW);
    mbar_init(bar(Ly::B_ACC), 1);
    mbar_init(bar(Ly::B_DRAIN), 1);
    mbar_init(bar(Ly::B_VEC), BM);  // every elementwise thread has written its LSE / D value
    mbar_init(bar(Ly::B_VEC + 1), BM);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(prm.status) != 0 || !unit_ok) ? 1 : 0;
    if (!unit_ok) record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_ITEM, (int32_t)blockIdx.x);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == WARP_LOAD && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmG);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = *abort_flag == 0;

  // the i-th query block of the unit: head, partition, block
  auto block_at = [&](int i, int& h, int& p, int& qb) {
    const int per_head = NBQ / g;
    h = hk * g + i / per_head;
    int r = i % per_head;
    for (int qi = 0; qi < it.n_kv; ++qi) {
      p = __ldg(prm.q_list + it.kv_off + qi);
      const int b0 = qblock_begin(k, p, prm.causal, kb);
      if (r < prm.nb - b0) {
        qb = b0 + r;
        return;
      }
      r -= prm.nb - b0;
    }
    p = -1;
    qb = 0;
  };

  if (warp < N_EW) {
    // ================================================================ elementwise
    const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
    const int row = wq * 32 + lane;           // TMEM lane = key row within the block
    const int c_base = hf * 64;               // this warp's query columns [c_base, c_base + 64)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_s = tmem + lane_base;           // S^T, then P^T (bf16)
    const uint32_t tm_dp = tmem + lane_base + 128u;   // dP^T, then dS^T (bf16)
    const uint32_t tm_dv = tmem + lane_base + 256u;
    const uint32_t tm_dk = tmem + lane_base + 256u + (uint32_t)D;
    bool ok = run;
    // Query-block cursors: `cur` is block i, `nxt` block i + 1.  Stepping them keeps the global
    // reads of the slot's partition list off the per-block path (one read per partition change).
    QCursor cur, nxt;
    cur.start(prm, it, k, kb, hk * g);
    nxt = cur;
    // LSE and D of query column `row` for the next block, loaded raw one block ahead by the first
    // column half and only used (scaled, published) at the top of the next iteration, so that the
    // loads never stall the block in flight
    float raw_lse = 0.f, raw_d = 0.f;
    bool raw_in = false;
    auto fetch = [&](const QCursor& c) {
      const int64_t ql = (int64_t)c.qb * BM + row;
      raw_in = c.p >= 0 && c.p < prm.P && ql < L;
      if (raw_in) {
        const int64_t gi = ((int64_t)b * prm.Hq + c.h) * prm.S + (int64_t)c.p * L + ql;
        raw_lse = __ldg(prm.lse + gi);
        raw_d = __ldg(prm.dsum + gi);
      }
    };
    if (ok && NBQ > 0 && hf == 0) fetch(cur);
    for (int i = 0; i < NBQ && ok; ++i) {
      const int vb = i & 1;
      if (i > 0) cur = nxt;
      if (i + 1 < NBQ) nxt.step(prm, it, k, kb);
      // publish this column's values, then wait (bounded) until all 128 columns are written; a
      // buffer is rewritten two blocks later, after every writer has arrived for the block between
      if (hf == 0) {
        // no such query row: exp2(s - inf) = 0, so it needs no mask
        nlse_s[vb * BM + row] = raw_in ? -raw_lse * LOG2E : -INFINITY;
        ndsum_s[vb * BM + row] = raw_in ? -raw_d : 0.f;
        mbar_arrive(bar(Ly::B_VEC + vb));
        if (i + 1 < NBQ) fetch(nxt);
      }
      ok = mbar_wait(bar(Ly::B_VEC + vb), (uint32_t)((i >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_EW, i);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int p = cur.p, qb = cur.qb;
      // causal diagonal block: query columns before this key row are masked (query rows past the
      // partition end carry -inf in place of -LSE and need no mask)
      const int lo = (prm.causal && p == k && qb == kb) ? row - c_base : 0;
      ok = mbar_wait(bar(Ly::B_S), (uint32_t)(i & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, i);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float pv[64];
      tmem_ld32(tm_s + (uint32_t)c_base, pv);
      tmem_ld32(tm_s + (uint32_t)c_base + 32u, pv + 32);
      tc_wait_ld();
      if (__any_sync(0xffffffffu, lo > 0)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < lo) pv[c] = -INFINITY;
      }
      const float4* lv = reinterpret_cast<const float4*>(nlse_s + vb * BM + c_base);
      const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = lv[c / 4];
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(pv[c], pv[c + 1]), sc2, f2_pack(l4.x, l4.y)), x0, x1);
        f2_unpack(f2_fma(f2_pack(pv[c + 2], pv[c + 3]), sc2, f2_pack(l4.z, l4.w)), x2, x3);
        pv[c] = fast_exp2(x0);
        pv[c + 1] = fast_exp2(x1);
        pv[c + 2] = fast_exp2(x2);
        pv[c + 3] = fast_exp2(x3);
        pk[c / 2] = pack_bf16x2(pv[c], pv[c + 1]);
        pk[c / 2 + 1] = pack_bf16x2(pv[c + 2], pv[c + 3]);
      }
      tmem_st32(tm_s + (uint32_t)c_base, pk);  // P^T columns of this half (see packed_col)
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_P));
      ok = mbar_wait(bar(Ly::B_DP), (uint32_t)(i & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, i);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      {
        float dp[64];
        tmem_ld32(tm_dp + (uint32_t)c_base, dp);
        tmem_ld32(tm_dp + (uint32_t)c_base + 32u, dp + 32);
        tc_wait_ld();
        const float4* dv_ = reinterpret_cast<const float4*>(ndsum_s + vb * BM + c_base);
        uint32_t ds2[32];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 d4 = dv_[c / 4];
          float a0, a1, a2, a3;
          f2_unpack(f2_mul(f2_add(f2_pack(dp[c], dp[c + 1]), f2_pack(d4.x, d4.y)), f2_pack(pv[c], pv[c + 1])), a0, a1);
          f2_unpack(f2_mul(f2_add(f2_pack(dp[c + 2], dp[c + 3]), f2_pack(d4.z, d4.w)), f2_pack(pv[c + 2], pv[c + 3])),
                    a2, a3);
          ds2[c / 2] = pack_bf16x2(a0, a1);
          ds2[c / 2 + 1] = pack_bf16x2(a2, a3);
        }
        tmem_st32(tm_dp + (uint32_t)c_base, ds2);  // dS^T columns of this half
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_DS));
    }
    // ---- epilogue: this half's columns of the dV and dK rows of this key block
    if (ok) {
      ok = mbar_wait(bar(Ly::B_ACC), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, -1);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const int64_t row0 = (((int64_t)b * prm.Hkv + hk) * prm.n_kv_slots + it.slot) * L + (int64_t)kb * BM + wq * 32;
      const int rows_valid = (int)max((int64_t)0, min((int64_t)32, L - ((int64_t)kb * BM + wq * 32)));
#pragma unroll 1
      for (int c = hf * (D / 2); c < (hf + 1) * (D / 2); c += 32) {
        float v[32];
        tmem_ld32(tm_dv + (uint32_t)c, v);
        tc_wait_ld();
        store_rows<D>(v, 1.f, prm.dv_part, row0, rows_valid, c, lane);
        tmem_ld32(tm_dk + (uint32_t)c, v);
        tc_wait_ld();
        store_rows<D>(v, prm.scale, prm.dk_part, row0, rows_valid, c, lane);
      }
    }
  } else if (warp == WARP_MMA) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_ss = idesc_bf16_f32(BM, BM, false);  // S^T, dP^T: K-major A and B
    constexpr uint32_t idesc_ts = idesc_bf16_f32(BM, D, true);    // dV, dK: B MN-major
    const uint64_t kdesc = smem_desc_sw128(sb + Ly::RES0, 16u, 1024u);
    const uint64_t vdesc = smem_desc_sw128(sb + Ly::RES1, 16u, 1024u);
    constexpr uint64_t TILE16 = Ly::TILE >> 4;
    const uint64_t a_kmaj = smem_desc_sw128(sb + Ly::A0, 16u, 1024u);   // Q stages
    const uint64_t a_mn = smem_desc_sw128(sb + Ly::A0, Ly::BOX, 1024u);
    const uint64_t b_kmaj = smem_desc_sw128(sb + Ly::B0, 16u, 1024u);   // dO stages
    const uint64_t b_mn = smem_desc_sw128(sb + Ly::B0, Ly::BOX, 1024u);
    auto issue_s = [&](int sa) {  // S^T = K Q^T
      const uint64_t qd = a_kmaj + (uint64_t)sa * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_warp(tmem, kdesc + kmaj_off<D>(kk), qd + kmaj_off<D>(kk), idesc_ss, kk > 0);
      tc_commit_warp(bar(Ly::B_S));
    };
    auto issue_dp = [&](int sbb) {  // dP^T = V dO^T
      const uint64_t gd = b_kmaj + (uint64_t)sbb * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_warp(tmem + 128u, vdesc + kmaj_off<D>(kk), gd + kmaj_off<D>(kk), idesc_ss, kk > 0);
      tc_commit_warp(bar(Ly::B_DP));
    };
    auto issue_dv = [&](int sbb, bool first) {  // dV += P^T dO
      const uint64_t gd = b_mn + (uint64_t)sbb * TILE16;
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        tc_mma_ts_warp(tmem + 256u, tmem + packed_col(kk), gd + (uint64_t)(kk * 128), idesc_ts,
                       (!first || kk > 0) ? 1u : 0u);
    };
    auto issue_dk = [&](int sa, bool first) {  // dK += dS^T Q
      const uint64_t qd = a_mn + (uint64_t)sa * TILE16;
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        tc_mma_ts_warp(tmem + 256u + (uint32_t)D, tmem + 128u + packed_col(kk), qd + (uint64_t)(kk * 128),
                       idesc_ts, (!first || kk > 0) ? 1u : 0u);
    };
    auto wait_a = [&](int i) {  // Q(i) landed
      return mbar_wait_warp(bar(Ly::B_AF + i % Ly::NSA), (uint32_t)((i / Ly::NSA) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, ROLE_MMA, i);
    };
    auto wait_b = [&](int i) {  // dO(i) landed
      return mbar_wait_warp(bar(Ly::B_BF + i % Ly::NSB), (uint32_t)((i / Ly::NSB) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, ROLE_MMA, i);
    };
    bool ok = run && NBQ > 0;
    if (ok) ok = mbar_wait_warp(bar(Ly::B_RES), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, -1);
    if (ok) ok = wait_a(0) && wait_b(0);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int i = 0; i < NBQ && ok; ++i) {
      ok = mbar_wait_warp(bar(Ly::B_P), (uint32_t)(i & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, i);
      if (!ok) break;
      tc_fence_after();
      issue_dv(i % Ly::NSB, i == 0);
      tc_commit_warp(bar(Ly::B_BE + i % Ly::NSB));  // dO(i): read by dP^T(i) and dV(i)
      if (i + 1 < NBQ) {
        ok = wait_a(i + 1);
        if (!ok) break;
        tc_fence_after();
        issue_s((i + 1) % Ly::NSA);
      }
      ok = mbar_wait_warp(bar(Ly::B_DS), (uint32_t)(i & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, i);
      if (!ok) break;
      tc_fence_after();
      issue_dk(i % Ly::NSA, i == 0);
      tc_commit_warp(bar(Ly::B_AE + i % Ly::NSA));  // Q(i): read by S^T(i) and dK(i)
      if (i + 1 < NBQ) {
        ok = wait_b(i + 1);
        if (!ok) break;
        tc_fence_after();
        issue_dp((i + 1) % Ly::NSB);
      }
    }
    if (ok) tc_commit_warp(bar(Ly::B_ACC));
    tc_commit_warp(bar(Ly::B_DRAIN));
    mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
  } else if (warp == WARP_LOAD && lane == 0) {
    // ================================================================ producer
    bool ok = run && NBQ > 0;
    const int64_t kvrow = ((int64_t)b * prm.Hkv + hk) * prm.S + (int64_t)k * L + (int64_t)kb * BM;
    if (ok) {
      mbar_expect_tx(bar(Ly::B_RES), 2 * Ly::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(sb + Ly::RES0 + (uint32_t)c * Ly::BOX, &tmK, c * 64, (int32_t)kvrow, bar(Ly::B_RES));
        tma_load_2d(sb + Ly::RES1 + (uint32_t)c * Ly::BOX, &tmV, c * 64, (int32_t)kvrow, bar(Ly::B_RES));
      }
    }
    int issued_a = 0, issued_b = 0;
    for (int i = 0; i < NBQ && ok; ++i) {
      int h, p, qb;
      block_at(i, h, p, qb);
      if (p < 0 || p >= prm.P) {
        record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, (int32_t)blockIdx.x);
        *abort_flag = 1;
        break;
      }
      const int32_t qrow = (int32_t)(((int64_t)b * prm.Hq + h) * prm.S + (int64_t)p * L + (int64_t)qb * BM);
      const int sa = i % Ly::NSA, sbb = i % Ly::NSB;
      if (i >= Ly::NSA) {
        ok = mbar_wait(bar(Ly::B_AE + sa), (uint32_t)((i / Ly::NSA - 1) & 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, i);
        if (!ok) break;
      }
      mbar_expect_tx(bar(Ly::B_AF + sa), Ly::TILE);
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sb + Ly::A0 + (uint32_t)sa * Ly::TILE + (uint32_t)c * Ly::BOX, &tmQ, c * 64, qrow,
                    bar(Ly::B_AF + sa));
      ++issued_a;
      if (i >= Ly::NSB) {
        ok = mbar_wait(bar(Ly::B_BE + sbb), (uint32_t)((i / Ly::NSB - 1) & 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, i);
        if (!ok) break;
      }
      mbar_expect_tx(bar(Ly::B_BF + sbb), Ly::TILE);
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sb + Ly::B0 + (uint32_t)sbb * Ly::TILE + (uint32_t)c * Ly::BOX, &tmG, c * 64, qrow,
                    bar(Ly::B_BF + sbb));
      ++issued_b;
    }
    // exit-path drain: every load issued lands before the CTA exits
    if (run && NBQ > 0) mbar_drain(bar(Ly::B_RES), 0u, DRAIN_NS);
    for (int j = (issued_a > Ly::NSA ? issued_a - Ly::NSA : 0); j < issued_a; ++j)
      mbar_drain(bar(Ly::B_AF + j % Ly::NSA), (uint32_t)((j / Ly::NSA) & 1), DRAIN_NS);
    for (int j = (issued_b > Ly::NSB ? issued_b - Ly::NSB : 0); j < issued_b; ++j)
      mbar_drain(bar(Ly::B_BF + j % Ly::NSB), (uint32_t)((j / Ly::NSB) & 1), DRAIN_NS);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================== dQ
template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                  const Params prm) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = smem_u32(smem_raw);
  if (sb & 1023u) {  // 128-byte swizzle atoms need 1024-aligned operands (see Layout)
    if (threadIdx.x == 0) record_error(prm.status, MESH_ATTN_ERR_INTERNAL, ROLE_ITEM, (int32_t)blockIdx.x);
    return;
  }
  uint8_t* smem = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + Ly::BAR_OFF + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 4);
  const int64_t L = prm.L;

  // unit -> (work item, batch, head, query block)
  int64_t uu = blockIdx.x;
  const int qb = (int)(uu % prm.nb); uu /= prm.nb;
  const int h = (int)(uu % prm.Hq); uu /= prm.Hq;
  const int b = (int)(uu % prm.B);
  const int idx = (int)(uu / prm.B);
  const DevItem it = prm.items[idx];  // {p, slot, kv_off, n_kv}
  const bool unit_ok = it.p >= 0 && it.p < prm.P && it.slot >= 0 && it.slot < prm.n_slots && it.n_kv >= 1 &&
                       it.kv_off >= 0;
  const int p = it.p;
  const int hk = h / (prm.Hq / prm.Hkv);
  int NB = 0;
  if (unit_ok)
    for (int ki = 0; ki < it.n_kv; ++ki) NB += kblocks_of(__ldg(prm.kv_list + it.kv_off + ki), p, prm.causal, prm.nb, qb);

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_RES), 1);
    for (int s = 0; s < Ly::NSA; ++s) {
      mbar_init(bar(Ly::B_AF + s), 1);
      mbar_init(bar(Ly::B_AE + s), 1);
    }
    for (int s = 0; s < Ly::NSB; ++s) {
      mbar_init(bar(Ly::B_BF + s), 1);
      mbar_init(bar(Ly::B_BE + s), 1);
    }
    mbar_init(bar(Ly::B_S), 1);
    mbar_init(bar(Ly::B_S + 1), 1);
    mbar_init(bar(Ly::B_DP), 1);
    mbar_init(bar(Ly::B_DS), N_EW);  // one lane of each elementwise warp
    mbar_init(bar(Ly::B_ACC), 1);
    mbar_init(bar(Ly::B_DRAIN), 1);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(prm.status) != 0 || !unit_ok) ? 1 : 0;
    if (!unit_ok) record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_ITEM, (int32_t)blockIdx.x);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == WARP_LOAD && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmG);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = *abort_flag == 0;

  // the j-th key block of the unit: KV partition and block
  auto block_at = [&](int j, int& kp, int& kbk) {
    int r = j;
    for (int ki = 0; ki < it.n_kv; ++ki) {
      kp = __ldg(prm.kv_list + it.kv_off + ki);
      const int n = kblocks_of(kp, p, prm.causal, prm.nb, qb);
      if (r < n) {
        kbk = r;
        return;
      }
      r -= n;
    }
    kp = -1;
    kbk = 0;
  };

  if (warp < N_EW) {
    // ================================================================ elementwise
    const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
    const int row = wq * 32 + lane;           // TMEM lane = query row within the block
    const int c_base = hf * 64;               // this warp's key columns [c_base, c_base + 64)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_dp = tmem + lane_base + 256u;  // dP, then dS (bf16)
    const uint32_t tm_dq = tmem + lane_base + 384u;
    const int64_t q_local = (int64_t)qb * BM + row;
    const int64_t grow = ((int64_t)b * prm.Hq + h) * prm.S + (int64_t)p * L + q_local;
    const bool row_in = q_local < L;
    const float lse2 = row_in ? __ldg(prm.lse + grow) * LOG2E : INFINITY;
    const float dsum = row_in ? __ldg(prm.dsum + grow) : 0.f;
    bool ok = run;
    KCursor cur;
    cur.start(prm, it, p, qb);
    for (int j = 0; j < NB && ok; ++j) {
      if (j > 0) cur.step(prm, it, p, qb);
      const int kp = cur.kp, kbk = cur.kb;
      const int64_t kvalid = L - (int64_t)kbk * BM;
      int hi = (int)min((int64_t)BM, kvalid);                         // keys past the partition end
      if (prm.causal && kp == p && kbk == qb) hi = min(hi, row + 1);  // diagonal block
      hi -= c_base;                                                   // in this half's columns
      const bool any_mask = __any_sync(0xffffffffu, hi < 64);
      const uint32_t tm_s = tmem + lane_base + (uint32_t)((j & 1) * 128);
      ok = mbar_wait(bar(Ly::B_S + (j & 1)), (uint32_t)((j >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_EW, j);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float pv[64];
      tmem_ld32(tm_s + (uint32_t)c_base, pv);
      tmem_ld32(tm_s + (uint32_t)c_base + 32u, pv + 32);
      tc_wait_ld();
      if (any_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= hi) pv[c] = -INFINITY;
      }
      const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2);
      const uint64_t nl2 = f2_pack(-lse2, -lse2);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(pv[c], pv[c + 1]), sc2, nl2), x0, x1);
        pv[c] = fast_exp2(x0);
        pv[c + 1] = fast_exp2(x1);
      }
      ok = mbar_wait(bar(Ly::B_DP), (uint32_t)(j & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, j);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      {
        const uint64_t nd2 = f2_pack(-dsum, -dsum);
        float dp[64];
        tmem_ld32(tm_dp + (uint32_t)c_base, dp);
        tmem_ld32(tm_dp + (uint32_t)c_base + 32u, dp + 32);
        tc_wait_ld();
        uint32_t ds2[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float a0, a1;
          f2_unpack(f2_mul(f2_add(f2_pack(dp[c], dp[c + 1]), nd2), f2_pack(pv[c], pv[c + 1])), a0, a1);
          ds2[c / 2] = pack_bf16x2(a0, a1);
        }
        tmem_st32(tm_dp + (uint32_t)c_base, ds2);  // dS columns of this half (see packed_col)
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_DS));
    }
    if (ok) {
      ok = mbar_wait(bar(Ly::B_ACC), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, -1);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const int64_t row0 = (((int64_t)b * prm.Hq + h) * prm.n_slots + it.slot) * L + (int64_t)qb * BM + wq * 32;
      const int rows_valid = (int)max((int64_t)0, min((int64_t)32, L - ((int64_t)qb * BM + wq * 32)));
#pragma unroll 1
      for (int c = hf * (D / 2); c < (hf + 1) * (D / 2); c += 32) {
        float v[32];
        tmem_ld32(tm_dq + (uint32_t)c, v);
        tc_wait_ld();
        store_rows<D>(v, prm.scale, prm.dq_part, row0, rows_valid, c, lane);
      }
    }
  } else if (warp == WARP_MMA) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_ss = idesc_bf16_f32(BM, BM, false);  // S = Q K^T, dP = dO V^T
    constexpr uint32_t idesc_ts = idesc_bf16_f32(BM, D, true);    // dQ += dS K, K MN-major
    const uint64_t qdesc = smem_desc_sw128(sb + Ly::RES0, 16u, 1024u);
    const uint64_t gdesc = smem_desc_sw128(sb + Ly::RES1, 16u, 1024u);
    constexpr uint64_t TILE16 = Ly::TILE >> 4;
    const uint64_t a_kmaj = smem_desc_sw128(sb + Ly::A0, 16u, 1024u);  // K stages
    const uint64_t a_mn = smem_desc_sw128(sb + Ly::A0, Ly::BOX, 1024u);
    const uint64_t b_kmaj = smem_desc_sw128(sb + Ly::B0, 16u, 1024u);  // V stages
    auto issue_s = [&](int sa, int buf) {  // S = Q K^T into S buffer `buf`
      const uint64_t kd = a_kmaj + (uint64_t)sa * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_warp(tmem + (uint32_t)(buf * 128), qdesc + kmaj_off<D>(kk), kd + kmaj_off<D>(kk), idesc_ss, kk > 0);
      tc_commit_warp(bar(Ly::B_S + buf));
    };
    auto issue_dp = [&](int sbb) {  // dP = dO V^T; V(j) is read by this product only
      const uint64_t vd = b_kmaj + (uint64_t)sbb * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_warp(tmem + 256u, gdesc + kmaj_off<D>(kk), vd + kmaj_off<D>(kk), idesc_ss, kk > 0);
      tc_commit_warp(bar(Ly::B_DP));
      tc_commit_warp(bar(Ly::B_BE + sbb));
    };
    auto issue_dq = [&](int sa, bool first) {  // dQ += dS K
      const uint64_t kd = a_mn + (uint64_t)sa * TILE16;
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        tc_mma_ts_warp(tmem + 384u, tmem + 256u + packed_col(kk), kd + (uint64_t)(kk * 128), idesc_ts,
                       (!first || kk > 0) ? 1u : 0u);
    };
    auto wait_a = [&](int j) {  // K(j) landed
      return mbar_wait_warp(bar(Ly::B_AF + j % Ly::NSA), (uint32_t)((j / Ly::NSA) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, ROLE_MMA, j);
    };
    auto wait_b = [&](int j) {  // V(j) landed
      return mbar_wait_warp(bar(Ly::B_BF + j % Ly::NSB), (uint32_t)((j / Ly::NSB) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, ROLE_MMA, j);
    };
    bool ok = run && NB > 0;
    if (ok) ok = mbar_wait_warp(bar(Ly::B_RES), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, -1);
    if (ok) ok = wait_a(0);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      ok = wait_b(0);
    }
    if (ok) {
      tc_fence_after();
      issue_dp(0);
      if (NB > 1) {
        ok = wait_a(1);
        if (ok) {
          tc_fence_after();
          issue_s(1, 1);
        }
      }
    }
    for (int j = 0; j < NB && ok; ++j) {
      // dS(j) is in TMEM, and S(j) has been read, so its buffer is free for S(j+2).  (One barrier per
      // block, passed in order: a second "S read" barrier could complete for block j+1, whose S is
      // issued two blocks ahead, before this warp observed block j -- two phases ahead of its
      // parity wait.)
      ok = mbar_wait_warp(bar(Ly::B_DS), (uint32_t)(j & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, j);
      if (!ok) break;
      tc_fence_after();
      issue_dq(j % Ly::NSA, j == 0);
      tc_commit_warp(bar(Ly::B_AE + j % Ly::NSA));  // K(j): read by S(j) and dQ(j)
      if (j + 1 < NB) {
        ok = wait_b(j + 1);
        if (!ok) break;
        tc_fence_after();
        issue_dp((j + 1) % Ly::NSB);
      }
      if (j + 2 < NB) {
        ok = wait_a(j + 2);
        if (!ok) break;
        tc_fence_after();
        issue_s((j + 2) % Ly::NSA, j & 1);
      }
    }
    if (ok) tc_commit_warp(bar(Ly::B_ACC));
    tc_commit_warp(bar(Ly::B_DRAIN));
    mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
  } else if (warp == WARP_LOAD && lane == 0) {
    // ================================================================ producer
    bool ok = run && NB > 0;
    const int64_t qrow = ((int64_t)b * prm.Hq + h) * prm.S + (int64_t)p * L + (int64_t)qb * BM;
    const int64_t kvbase = ((int64_t)b * prm.Hkv + hk) * prm.S;
    if (ok) {
      mbar_expect_tx(bar(Ly::B_RES), 2 * Ly::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(sb + Ly::RES0 + (uint32_t)c * Ly::BOX, &tmQ, c * 64, (int32_t)qrow, bar(Ly::B_RES));
        tma_load_2d(sb + Ly::RES1 + (uint32_t)c * Ly::BOX, &tmG, c * 64, (int32_t)qrow, bar(Ly::B_RES));
      }
    }
    int issued_a = 0, issued_b = 0;
    for (int j = 0; j < NB && ok; ++j) {
      int kp, kbk;
      block_at(j, kp, kbk);
      if (kp < 0 || kp >= prm.P) {
        record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, (int32_t)blockIdx.x);
        *abort_flag = 1;
        break;
      }
      const int32_t krow = (int32_t)(kvbase + (int64_t)kp * L + (int64_t)kbk * BM);
      const int sa = j % Ly::NSA, sbb = j % Ly::NSB;
      if (j >= Ly::NSA) {
        ok = mbar_wait(bar(Ly::B_AE + sa), (uint32_t)((j / Ly::NSA - 1) & 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, j);
        if (!ok) break;
      }
      mbar_expect_tx(bar(Ly::B_AF + sa), Ly::TILE);
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sb + Ly::A0 + (uint32_t)sa * Ly::TILE + (uint32_t)c * Ly::BOX, &tmK, c * 64, krow,
                    bar(Ly::B_AF + sa));
      ++issued_a;
      if (j >= Ly::NSB) {
        ok = mbar_wait(bar(Ly::B_BE + sbb), (uint32_t)((j / Ly::NSB - 1) & 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, j);
        if (!ok) break;
      }
      mbar_expect_tx(bar(Ly::B_BF + sbb), Ly::TILE);
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sb + Ly::B0 + (uint32_t)sbb * Ly::TILE + (uint32_t)c * Ly::BOX, &tmV, c * 64, krow,
                    bar(Ly::B_BF + sbb));
      ++issued_b;
    }
    if (run && NB > 0) mbar_drain(bar(Ly::B_RES), 0u, DRAIN_NS);
    for (int j = (issued_a > Ly::NSA ? issued_a - Ly::NSA : 0); j < issued_a; ++j)
      mbar_drain(bar(Ly::B_AF + j % Ly::NSA), (uint32_t)((j / Ly::NSA) & 1), DRAIN_NS);
    for (int j = (issued_b > Ly::NSB ? issued_b - Ly::NSB : 0); j < issued_b; ++j)
      mbar_drain(bar(Ly::B_BF + j % Ly::NSB), (uint32_t)((j / Ly::NSB) & 1), DRAIN_NS);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode(std::string* err) {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return nullptr;
  }
  fn = reinterpret_cast<EncodeTiledFn>(ptr);
  return fn;
}

// [rows, d] bf16 row-major tensor, boxes of 128 rows x 64 columns with 128-byte swizzle.
static bool make_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t rows, int d, std::string* err) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)BM};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

template <int D>
static int launch(const BwdArgs& a, void* stream, std::string* err) {
  const int64_t nb = (a.L + BM - 1) / BM;
  const int64_t dq_units = (int64_t)a.n_items * a.B * a.Hq * nb;
  const int64_t kv_units = (int64_t)a.n_kv_items * a.B * a.Hkv * nb;
  if (dq_units <= 0 && kv_units <= 0) return (int)cudaSuccess;
  if (dq_units > 0x7fffffff || kv_units > 0x7fffffff) {
    *err = "too many work units for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  EncodeTiledFn enc = get_encode(err);
  if (!enc) return (int)cudaErrorNotSupported;
  CUtensorMap mq, mk, mv, mg;
  if (!make_map(enc, &mq, a.Q, (uint64_t)a.B * a.Hq * a.S, D, err) ||
      !make_map(enc, &mk, a.K, (uint64_t)a.B * a.Hkv * a.S, D, err) ||
      !make_map(enc, &mv, a.V, (uint64_t)a.B * a.Hkv * a.S, D, err) ||
      !make_map(enc, &mg, a.dO, (uint64_t)a.B * a.Hq * a.S, D, err))
    return (int)cudaErrorInvalidValue;
  Params prm;
  prm.items = a.items;
  prm.kv_list = a.kv_list;
  prm.kv_items = a.kv_items;
  prm.q_list = a.q_list;
  prm.lse = a.LSE;
  prm.dsum = a.D;
  prm.dq_part = a.dq_part;
  prm.dk_part = a.dk_part;
  prm.dv_part = a.dv_part;
  prm.status = a.status;
  prm.S = a.S;
  prm.L = a.L;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.P = a.P;
  prm.n_items = a.n_items;
  prm.n_slots = a.n_slots;
  prm.n_kv_items = a.n_kv_items;
  prm.n_kv_slots = a.n_kv_slots;
  prm.nb = (int32_t)nb;
  prm.causal = a.causal;
  prm.scale = a.scale;
  prm.scale_log2 = a.scale_log2;
  prm.wait_limit_ns = a.wait_limit_ns;
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Layout<D>::ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<D>::ALLOC);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (kv_units > 0)
    bwd_dkdv_kernel<D><<<dim3((unsigned)kv_units), dim3(NUM_THREADS), Layout<D>::ALLOC, st>>>(mq, mk, mv, mg, prm);
  if (dq_units > 0)
    bwd_dq_kernel<D><<<dim3((unsigned)dq_units), dim3(NUM_THREADS), Layout<D>::ALLOC, st>>>(mq, mk, mv, mg, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("tile_bwd_tc launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace btc

int launch_tile_bwd_tc(const BwdArgs& a, void* stream, std::string* err) {
  if (a.d == 128) return btc::launch<128>(a, stream, err);
  if (a.d == 64) return btc::launch<64>(a, stream, err);
  *err = "tensor-core backward supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
