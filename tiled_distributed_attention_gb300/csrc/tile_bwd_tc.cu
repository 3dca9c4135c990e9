// Tile attention backward on the 5th-generation tensor cores (sm_103a), bf16 inputs.
//
// The gradients of the forward definition (the left-hand side of "环形注意力：突破长序列处理
// 瓶颈的分布式计算范式", §"理论奠基"), per tile of the Mesh-Attention plan ("Mesh-Attention: A New
// Communication-Efficient Distributed Attention with Improved Data Locality", tutorial
// §"Mesh-Attention：从一维'环'到二维'网'"), with the forward's global LSE and D_i = dO_i . O_i:
//   P_ij = exp(s_ij - LSE_i),  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
// Two persistent kernels: one CTA per SM takes units (one 128-row tile each) from a global
// counter; the producer decodes a unit and publishes it through a two-entry shared-memory ring.
// 16 warps in four warpgroups, registers rebalanced with setmaxnreg:
//   warps 0-7   elementwise: two warps per TMEM lane quadrant, one thread per TMEM lane (a key row
//               in dkdv, a query row in dq), each warp taking 64 of the block's 128 columns
//   warp 8      MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M = N = 128, K = 16, issued by an
//               elected lane of the converged warp; completion by tcgen05.commit
//   warp 9      producer: TMA loads of 128 x 64 bf16 boxes with 128-byte swizzle
//   warps 10-11 idle
//   warps 12-15 (dq only) epilogue: one per TMEM lane quadrant; copies each unit's Q and dO into
//               TMEM, and drains the unit's dQ accumulator and stores its partial rows while the
//               other roles run the next unit.  In dkdv the elementwise warps drain dV and dK at
//               the unit boundary instead: drained during the next unit, the TMEM reads of the
//               two accumulators slowed that unit's products down.
// Across units: the next unit's resident block loads as soon as the last products reading the
// current one have completed, its first products are issued right after the current unit's
// last accumulation, and an accumulator is overwritten only after it has been copied out.
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
// dq (unit = forward work item, batch, head, 128-row block): Q and dO are copied once per unit
//   from shared memory into TMEM by the epilogue warps and feed S = Q K^T and dP = dO V^T as
//   A operands from TMEM, so those products read only the streamed K or V block from shared
//   memory; K and V blocks of the item's KV partitions stream through three and two stages.
//   TMEM: S | dP | dQ | Q | dO (bf16).  S(j+1) is issued as soon as the elementwise warps have
//   read S(j) into registers, so it computes while they exponentiate block j; LSE and D of a
//   row are thread-local.
// Every mbarrier wait is bounded; a timeout records MESH_ATTN_ERR_DEVICE_TIMEOUT, the CTA stops,
// drains its copies and products and frees its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace btc {

constexpr int BM = 128;  // rows per tile = TMEM lanes = keys / queries per block
constexpr int NUM_THREADS = 512;
constexpr int N_EW = 8;  // elementwise warps: two per TMEM lane quadrant, 64 columns each
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
constexpr int WARP_EPI = 12;  // warps 12-15: epilogue, one per TMEM lane quadrant (warps 10-11 idle)
constexpr int N_EPI = 4;
// Register budgets after setmaxnreg, per warpgroup: elementwise (warps 0-7), MMA / producer
// (8-11), epilogue (12-15).  They add up to the 512 x 128 registers of the launch; the launcher
// checks the kernels' register count against that before launching.
constexpr int EW_REGS = 168, MMA_REGS = 104, EPI_REGS = 72;
static_assert(2 * 128 * EW_REGS + 128 * MMA_REGS + 128 * EPI_REGS <= NUM_THREADS * 128, "register split");
// The bf16 P / dS written back into TMEM by column half `hf` land in packed columns
// [64 hf, 64 hf + 32) of their region -- inside the half's own input columns, so the halves never
// overwrite values the other still has to read -- and the MMAs that take them as A read K-step kk
// (16 elements = 8 packed columns) from here:
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }
constexpr int64_t DRAIN_NS = 200000000;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int ROLE_EW = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_ITEM = 4, ROLE_EPI = 5;

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
  uint32_t* counter_dq;  // unit counters of the two kernels, 0 at launch
  uint32_t* counter_kv;
  int64_t S, L;
  int32_t B, Hq, Hkv, P, n_items, n_slots, n_kv_items, n_kv_slots, nb, causal;
  int32_t n_dq_units, n_kv_units;
  float scale, scale_log2;
  int64_t wait_limit_ns;
};

// Shared memory: the resident pair (K, V in dkdv; in dq the landing buffers of Q and dO, which
// the epilogue warps copy into TMEM), NSA stages of stream A (the operand of the S product, which
// the next block's S needs while the current block's dK or dQ still reads it: Q in dkdv, K in
// dq) and NSB stages of stream B (dO in dkdv, V in dq).  224 KB for d = 128 leaves no room to align the base by hand:
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
                       B_DRAIN = B_ACC + 1, B_VEC = B_DRAIN + 1, B_RESE = B_VEC + 2, B_ACCE = B_RESE + 1,
                       B_UF = B_ACCE + 1, B_UE = B_UF + 2, B_ACC2 = B_UE + 2, B_ACCE2 = B_ACC2 + 1,
                       B_SREAD = B_ACCE2 + 1, B_QTF = B_SREAD + 1, B_QTE = B_QTF + 1, NBARS = B_QTE + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr uint32_t RING_OFF = MISC_OFF + 16;         // unit ring: 2 decoded units, 16 ints each
  static constexpr uint32_t TOTAL = RING_OFF + 2 * 64;
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
// unit -> (KV slot, batch, KV head, 128-key block), key block fastest
struct KvUnit {
  int kb, hk, b, NBQ;
  DevItem it;  // {k, kv slot, q_off, n_q}
  bool ok;
};
__device__ __forceinline__ KvUnit kv_unit(int u, const Params& prm) {
  KvUnit x;
  int64_t uu = u;
  x.kb = (int)(uu % prm.nb); uu /= prm.nb;
  x.hk = (int)(uu % prm.Hkv); uu /= prm.Hkv;
  x.b = (int)(uu % prm.B);
  const int idx = (int)(uu / prm.B);
  x.NBQ = 0;
  x.ok = idx >= 0 && idx < prm.n_kv_items;
  if (!x.ok) return x;
  x.it = prm.kv_items[idx];
  x.ok = x.it.p >= 0 && x.it.p < prm.P && x.it.slot >= 0 && x.it.slot < prm.n_kv_slots && x.it.n_kv >= 1 &&
         x.it.kv_off >= 0;
  // query blocks of the unit: heads of the group x Q partitions of the slot x blocks
  if (x.ok)
    for (int qi = 0; qi < x.it.n_kv; ++qi)
      x.NBQ += prm.nb - qblock_begin(x.it.p, __ldg(prm.q_list + x.it.kv_off + qi), prm.causal, x.kb);
  x.NBQ *= prm.Hq / prm.Hkv;
  return x;
}
// A unit travels through the shared-memory ring decoded (16 ints per entry), so that consumers
// never wait on the global reads of the decode.
__device__ __forceinline__ void put_unit(volatile int32_t* e, int u, const KvUnit& x) {
  e[0] = u;
  e[1] = x.kb, e[2] = x.hk, e[3] = x.b, e[4] = x.NBQ, e[5] = x.ok ? 1 : 0;
  e[6] = x.it.p, e[7] = x.it.slot, e[8] = x.it.kv_off, e[9] = x.it.n_kv;
}
__device__ __forceinline__ int get_unit(const volatile int32_t* e, KvUnit& x) {
  x.kb = e[1], x.hk = e[2], x.b = e[3], x.NBQ = e[4], x.ok = e[5] != 0;
  x.it.p = e[6], x.it.slot = e[7], x.it.kv_off = e[8], x.it.n_kv = e[9];
  return e[0];
}

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
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + Ly::RING_OFF);
  float* nlse_s = reinterpret_cast<float*>(smem + Ly::VEC_OFF);  // [2][BM] -LSE log2 e of the query columns
  float* ndsum_s = nlse_s + 2 * BM;                              // [2][BM] -D
  const int64_t L = prm.L;
  const int g = prm.Hq / prm.Hkv;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_RES), 1);
    mbar_init(bar(Ly::B_RESE), 1);
    for (int s = 0; s < Ly::NSA; ++s) {
      mbar_init(bar(Ly::B_AF + s), 1);
      mbar_init(bar(Ly::B_AE + s), 1);
    }
    for (int s = 0; s < Ly::NSB; ++s) {
      mbar_init(bar(Ly::B_BF + s), 1);
      mbar_init(bar(Ly::B_BE + s), 1);
    }
    mbar_init(bar(Ly::B_S), 1);
    mbar_init(bar(Ly::B_DP), 1);
    mbar_init(bar(Ly::B_P), N_EW);  // one lane of each elementwise warp
    mbar_init(bar(Ly::B_DS), N_EW);
    mbar_init(bar(Ly::B_ACC), 1);
    mbar_init(bar(Ly::B_ACCE), N_EW);  // one lane of each elementwise warp
    mbar_init(bar(Ly::B_ACC2), 1);
    mbar_init(bar(Ly::B_ACCE2), N_EW);
    mbar_init(bar(Ly::B_DRAIN), 1);
    mbar_init(bar(Ly::B_VEC), BM);  // every elementwise thread has written its LSE / D value
    mbar_init(bar(Ly::B_VEC + 1), BM);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ly::B_UF + s), 1);
      mbar_init(bar(Ly::B_UE + s), N_EW + 1);  // the elementwise warps and the MMA warp read a unit
    }
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(prm.status) != 0) ? 1 : 0;
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

  int nu = 0;
  auto take = [&](int& v, KvUnit& y, int role) -> bool {
    const int slot = nu & 1;
    bool r = mbar_wait_warp(bar(Ly::B_UF + slot), (uint32_t)((nu >> 1) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, role, -1);
    if (!r) return false;
    v = get_unit(unit_ring + 16 * slot, y);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(Ly::B_UE + slot));
    ++nu;
    return true;
  };
  auto bad_unit = [&](int u, int role) {
    if (lane == 0) {
      record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, role, u);
      *abort_flag = 1;
    }
    __syncwarp();
  };

  if (warp < N_EW) {
    // ================================================================ elementwise
    regs_inc<EW_REGS>();
    const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
    const int row = wq * 32 + lane;           // TMEM lane = key row within the block
    const int c_base = hf * 64;               // this warp's query columns [c_base, c_base + 64)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_s = tmem + lane_base;           // S^T, then P^T (bf16)
    const uint32_t tm_dp = tmem + lane_base + 128u;   // dP^T, then dS^T (bf16)
    bool ok = run;
    // LSE and D of query column `row` for the next block, loaded raw one block ahead by the first
    // column half and only used (scaled, published) at the top of the next iteration, so that the
    // loads never stall the block in flight; across units, the next unit's first block is
    // loaded before this unit's epilogue
    float raw_lse = 0.f, raw_d = 0.f;
    bool raw_in = false;
    auto fetch = [&](const KvUnit& y, const QCursor& c) {
      const int64_t ql = (int64_t)c.qb * BM + row;
      raw_in = c.p >= 0 && c.p < prm.P && ql < L;
      if (raw_in) {
        const int64_t gi = ((int64_t)y.b * prm.Hq + c.h) * prm.S + (int64_t)c.p * L + ql;
        raw_lse = __ldg(prm.lse + gi);
        raw_d = __ldg(prm.dsum + gi);
      }
    };
    int v = -1;
    KvUnit x;
    if (ok) ok = take(v, x, ROLE_EW);
    // Query-block cursors: `cur` is block i, `nxt` block i + 1.  Stepping them keeps the global
    // reads of the slot's partition list off the per-block path (one read per partition change).
    QCursor cur, nxt;
    if (ok && v >= 0) {
      if (x.ok) {
        cur.start(prm, x.it, x.it.p, x.kb, x.hk * g);
        if (hf == 0) fetch(x, cur);
      }
    }
    int64_t g0 = 0;  // global index of the unit's first query block
    int k_unit = 0;
    while (ok && v >= 0) {
      if (!x.ok || x.NBQ < 1) {
        bad_unit(v, ROLE_EW);
        ok = false;
        break;
      }
      const int k = x.it.p, kb = x.kb, NBQ = x.NBQ;
      nxt = cur;
      for (int i = 0; i < NBQ && ok; ++i) {
        const int64_t gi = g0 + i;
        const int vb = (int)(gi & 1);
        if (i > 0) cur = nxt;
        if (i + 1 < NBQ) nxt.step(prm, x.it, k, kb);
        // publish this column's values, then wait (bounded) until all 128 columns are written; a
        // buffer is rewritten two blocks later, after every writer has arrived for the block between
        if (hf == 0) {
          // no such query row: exp2(s - inf) = 0, so it needs no mask
          nlse_s[vb * BM + row] = raw_in ? -raw_lse * LOG2E : -INFINITY;
          ndsum_s[vb * BM + row] = raw_in ? -raw_d : 0.f;
          mbar_arrive(bar(Ly::B_VEC + vb));
          if (i + 1 < NBQ) fetch(x, nxt);
        }
        ok = mbar_wait(bar(Ly::B_VEC + vb), (uint32_t)((gi >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                       ROLE_EW, i);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const int p = cur.p, qb = cur.qb;
        // causal diagonal block: query columns before this key row are masked (query rows past the
        // partition end carry -inf in place of -LSE and need no mask)
        const int lo = (prm.causal && p == k && qb == kb) ? row - c_base : 0;
        ok = mbar_wait(bar(Ly::B_S), (uint32_t)(gi & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, i);
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
        ok = mbar_wait(bar(Ly::B_DP), (uint32_t)(gi & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, i);
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
            f2_unpack(f2_mul(f2_add(f2_pack(dp[c], dp[c + 1]), f2_pack(d4.x, d4.y)), f2_pack(pv[c], pv[c + 1])), a0,
                      a1);
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
      if (!ok) break;
      // the next unit, and its first block's LSE and D, before this unit's epilogue
      int vn = -1;
      KvUnit xn;
      ok = take(vn, xn, ROLE_EW);
      if (!ok) break;
      if (vn >= 0) {
        if (xn.ok) {
          cur.start(prm, xn.it, xn.it.p, xn.kb, xn.hk * g);
          if (hf == 0) fetch(xn, cur);
        }
      }
      // ---- epilogue: this half's columns of the dV and dK rows of this key block.  It runs here,
      // at the unit boundary where the tensor pipe has little else to do: drained by separate
      // warps during the next unit, the TMEM reads slowed that unit's products down.
      ok = mbar_wait(bar(Ly::B_ACC2), (uint32_t)(k_unit & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW,
                     -1);  // dK's last product, and so dV's, has completed
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      {
        const uint32_t tm_dv = tmem + lane_base + 256u + (uint32_t)(hf * (D / 2));
        const uint32_t tm_dk = tm_dv + (uint32_t)D;
        const int64_t row0 =
            (((int64_t)x.b * prm.Hkv + x.hk) * prm.n_kv_slots + x.it.slot) * L + (int64_t)kb * BM + wq * 32;
        const int rows_valid = (int)max((int64_t)0, min((int64_t)32, L - ((int64_t)kb * BM + wq * 32)));
        float acc[D / 2];
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) tmem_ld32(tm_dv + (uint32_t)c, acc + c);
        tc_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 2; c += 32)
          store_rows<D>(*reinterpret_cast<const float(*)[32]>(acc + c), 1.f, prm.dv_part, row0, rows_valid,
                        hf * (D / 2) + c, lane);
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) tmem_ld32(tm_dk + (uint32_t)c, acc + c);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {  // both accumulators are copied out: the next unit may overwrite them
          mbar_arrive(bar(Ly::B_ACCE));
          mbar_arrive(bar(Ly::B_ACCE2));
        }
#pragma unroll
        for (int c = 0; c < D / 2; c += 32)
          store_rows<D>(*reinterpret_cast<const float(*)[32]>(acc + c), prm.scale, prm.dk_part, row0, rows_valid,
                        hf * (D / 2) + c, lane);
      }
      ++k_unit;
      g0 += NBQ;
      v = vn;
      x = xn;
    }
  } else if (warp < WARP_EPI) {
    regs_dec<MMA_REGS>();
    if (warp == WARP_MMA) {
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
    auto issue_s = [&](int64_t gi) {  // S^T = K Q(gi)^T
      const uint64_t qd = a_kmaj + (uint64_t)(gi % Ly::NSA) * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_warp(tmem, kdesc + kmaj_off<D>(kk), qd + kmaj_off<D>(kk), idesc_ss, kk > 0);
      tc_commit_warp(bar(Ly::B_S));
    };
    auto issue_dp = [&](int64_t gi) {  // dP^T = V dO(gi)^T
      const uint64_t gd = b_kmaj + (uint64_t)(gi % Ly::NSB) * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_warp(tmem + 128u, vdesc + kmaj_off<D>(kk), gd + kmaj_off<D>(kk), idesc_ss, kk > 0);
      tc_commit_warp(bar(Ly::B_DP));
    };
    auto issue_dv = [&](int64_t gi, bool first) {  // dV += P^T dO(gi)
      const int sbb = (int)(gi % Ly::NSB);
      const uint64_t gd = b_mn + (uint64_t)sbb * TILE16;
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        tc_mma_ts_warp(tmem + 256u, tmem + packed_col(kk), gd + (uint64_t)(kk * 128), idesc_ts,
                       (!first || kk > 0) ? 1u : 0u);
      tc_commit_warp(bar(Ly::B_BE + sbb));  // dO(gi): read by dP^T(gi) and dV(gi)
    };
    auto issue_dk = [&](int64_t gi, bool first) {  // dK += dS^T Q(gi)
      const int sa = (int)(gi % Ly::NSA);
      const uint64_t qd = a_mn + (uint64_t)sa * TILE16;
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        tc_mma_ts_warp(tmem + 256u + (uint32_t)D, tmem + 128u + packed_col(kk), qd + (uint64_t)(kk * 128),
                       idesc_ts, (!first || kk > 0) ? 1u : 0u);
      tc_commit_warp(bar(Ly::B_AE + sa));  // Q(gi): read by S^T(gi) and dK(gi)
    };
    auto wait_a = [&](int64_t gi) {  // Q(gi) landed
      return mbar_wait_warp(bar(Ly::B_AF + (int)(gi % Ly::NSA)), (uint32_t)((gi / Ly::NSA) & 1), prm.wait_limit_ns,
                            abort_flag, prm.status, ROLE_MMA, (int32_t)gi);
    };
    auto wait_b = [&](int64_t gi) {  // dO(gi) landed
      return mbar_wait_warp(bar(Ly::B_BF + (int)(gi % Ly::NSB)), (uint32_t)((gi / Ly::NSB) & 1), prm.wait_limit_ns,
                            abort_flag, prm.status, ROLE_MMA, (int32_t)gi);
    };
    int nres = 0;
    // S^T(0) and dP^T(0) of a unit whose first block is gi, as soon as its resident K and V have
    // landed (for every unit but the first, after the previous unit's last dK)
    auto start_unit = [&](const KvUnit& y, int64_t gi) -> bool {
      if (!mbar_wait_warp(bar(Ly::B_RES), (uint32_t)(nres & 1), prm.wait_limit_ns, abort_flag, prm.status,
                          ROLE_MMA, -1))
        return false;
      ++nres;
      if (!wait_a(gi)) return false;
      tc_fence_after();
      issue_s(gi);
      if (!wait_b(gi)) return false;
      tc_fence_after();
      issue_dp(gi);
      if (y.NBQ == 1) tc_commit_warp(bar(Ly::B_RESE));  // the unit's last S^T and dP^T are issued
      return true;
    };
    bool ok = run;
    int v = -1;
    KvUnit x;
    if (ok) ok = take(v, x, ROLE_MMA);
    if (ok && v >= 0) {
      if (!x.ok || x.NBQ < 1) {
        bad_unit(v, ROLE_MMA);
        ok = false;
      } else {
        ok = start_unit(x, 0);
      }
    }
    int64_t g0 = 0;
    int k_unit = 0;
    while (ok && v >= 0) {
      const int NBQ = x.NBQ;
      for (int i = 0; i < NBQ && ok; ++i) {
        const int64_t gi = g0 + i;
        ok = mbar_wait_warp(bar(Ly::B_P), (uint32_t)(gi & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, i);
        if (!ok) break;
        if (i == 0 && k_unit > 0) {  // the previous unit's dV has been copied out of TMEM
          ok = mbar_wait_warp(bar(Ly::B_ACCE), (uint32_t)((k_unit - 1) & 1), prm.wait_limit_ns, abort_flag,
                              prm.status, ROLE_MMA, -1);
          if (!ok) break;
        }
        tc_fence_after();
        issue_dv(gi, i == 0);
        if (i + 1 == NBQ) tc_commit_warp(bar(Ly::B_ACC));  // dV complete: the epilogue may drain it
        if (i + 1 < NBQ) {
          ok = wait_a(gi + 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(gi + 1);
        }
        ok = mbar_wait_warp(bar(Ly::B_DS), (uint32_t)(gi & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, i);
        if (!ok) break;
        if (i == 0 && k_unit > 0) {  // the previous unit's dK has been copied out of TMEM
          ok = mbar_wait_warp(bar(Ly::B_ACCE2), (uint32_t)((k_unit - 1) & 1), prm.wait_limit_ns, abort_flag,
                              prm.status, ROLE_MMA, -1);
          if (!ok) break;
        }
        tc_fence_after();
        issue_dk(gi, i == 0);
        if (i + 1 == NBQ) tc_commit_warp(bar(Ly::B_ACC2));  // dK complete
        if (i + 1 < NBQ) {
          ok = wait_b(gi + 1);
          if (!ok) break;
          tc_fence_after();
          issue_dp(gi + 1);
          if (i + 2 == NBQ) tc_commit_warp(bar(Ly::B_RESE));  // the unit's last S^T and dP^T are issued
        }
      }
      if (!ok) break;
      int vn = -1;
      ok = take(vn, x, ROLE_MMA);
      if (!ok) break;
      g0 += NBQ;
      ++k_unit;
      v = vn;
      if (v < 0) break;
      if (!x.ok || x.NBQ < 1) {
        bad_unit(v, ROLE_MMA);
        ok = false;
        break;
      }
      ok = start_unit(x, g0);
    }
    // exit-path drain: every MMA issued completes before TMEM is freed
    tc_commit_warp(bar(Ly::B_DRAIN));
    mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
    } else if (warp == WARP_LOAD && lane == 0) {
    // ================================================================ producer
    bool ok = run;
    int np = 0;  // units published
    auto publish = [&](KvUnit& y) -> int {
      const int slot = np & 1;
      ok = mbar_wait(bar(Ly::B_UE + slot), (uint32_t)(((np >> 1) & 1) ^ 1), prm.wait_limit_ns, abort_flag,
                     prm.status, ROLE_LOAD, -1);
      if (!ok) return -1;
      int u = (int)atomicAdd(prm.counter_kv, 1u);
      if (u >= prm.n_kv_units) u = -1;
      if (u >= 0) y = kv_unit(u, prm);
      put_unit(unit_ring + 16 * slot, u, y);
      mbar_arrive(bar(Ly::B_UF + slot));
      ++np;
      return u;
    };
    int nres = 0;
    int64_t ga = 0, gb = 0;  // Q and dO blocks issued
    KvUnit x, y;
    int u = ok ? publish(x) : -1;
    while (ok && u >= 0) {
      if (!x.ok || x.NBQ < 1) {
        record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, u);
        *abort_flag = 1;
        break;
      }
      // publish the following unit now and pull its K, V rows into L2
      const int un = publish(y);
      if (!ok) break;
      if (un >= 0) {
        if (y.ok) {
          const int64_t kn = ((int64_t)y.b * prm.Hkv + y.hk) * prm.S + (int64_t)y.it.p * L + (int64_t)y.kb * BM;
          for (int c = 0; c < D / 64; ++c) {
            tma_prefetch_l2_2d(&tmK, c * 64, (int32_t)kn);
            tma_prefetch_l2_2d(&tmV, c * 64, (int32_t)kn);
          }
        }
      }
      // resident K and V: the previous unit's last S^T and dP^T products must be done with them
      ok = mbar_wait(bar(Ly::B_RESE), (uint32_t)((nres & 1) ^ 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_LOAD, u);
      if (!ok) break;
      const int64_t kvrow = ((int64_t)x.b * prm.Hkv + x.hk) * prm.S + (int64_t)x.it.p * L + (int64_t)x.kb * BM;
      mbar_expect_tx(bar(Ly::B_RES), 2 * Ly::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(sb + Ly::RES0 + (uint32_t)c * Ly::BOX, &tmK, c * 64, (int32_t)kvrow, bar(Ly::B_RES));
        tma_load_2d(sb + Ly::RES1 + (uint32_t)c * Ly::BOX, &tmV, c * 64, (int32_t)kvrow, bar(Ly::B_RES));
      }
      ++nres;
      QCursor cur;
      cur.start(prm, x.it, x.it.p, x.kb, x.hk * g);
      for (int i = 0; i < x.NBQ && ok; ++i) {
        if (i > 0) cur.step(prm, x.it, x.it.p, x.kb);
        if (cur.p < 0 || cur.p >= prm.P) {
          record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, u);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int32_t qrow =
            (int32_t)(((int64_t)x.b * prm.Hq + cur.h) * prm.S + (int64_t)cur.p * L + (int64_t)cur.qb * BM);
        const int sa = (int)(ga % Ly::NSA), sbb = (int)(gb % Ly::NSB);
        if (ga >= Ly::NSA) {
          ok = mbar_wait(bar(Ly::B_AE + sa), (uint32_t)((ga / Ly::NSA - 1) & 1), prm.wait_limit_ns, abort_flag,
                         prm.status, ROLE_LOAD, i);
          if (!ok) break;
        }
        mbar_expect_tx(bar(Ly::B_AF + sa), Ly::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::A0 + (uint32_t)sa * Ly::TILE + (uint32_t)c * Ly::BOX, &tmQ, c * 64, qrow,
                      bar(Ly::B_AF + sa));
        ++ga;
        if (gb >= Ly::NSB) {
          ok = mbar_wait(bar(Ly::B_BE + sbb), (uint32_t)((gb / Ly::NSB - 1) & 1), prm.wait_limit_ns, abort_flag,
                         prm.status, ROLE_LOAD, i);
          if (!ok) break;
        }
        mbar_expect_tx(bar(Ly::B_BF + sbb), Ly::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::B0 + (uint32_t)sbb * Ly::TILE + (uint32_t)c * Ly::BOX, &tmG, c * 64, qrow,
                      bar(Ly::B_BF + sbb));
        ++gb;
      }
      u = un;
      x = y;
    }
    // exit-path drain: every load issued lands before the CTA exits
    if (nres > 0) mbar_drain(bar(Ly::B_RES), (uint32_t)((nres - 1) & 1), DRAIN_NS);
    for (int64_t j = (ga > Ly::NSA ? ga - Ly::NSA : 0); j < ga; ++j)
      mbar_drain(bar(Ly::B_AF + (int)(j % Ly::NSA)), (uint32_t)((j / Ly::NSA) & 1), DRAIN_NS);
    for (int64_t j = (gb > Ly::NSB ? gb - Ly::NSB : 0); j < gb; ++j)
      mbar_drain(bar(Ly::B_BF + (int)(j % Ly::NSB)), (uint32_t)((j / Ly::NSB) & 1), DRAIN_NS);
    }
  } else {
    // warps 12-15 have no role in this kernel (the elementwise warps drain the accumulators)
    regs_dec<EPI_REGS>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================== dQ
// unit -> (work item, batch, head, 128-row query block), query block fastest
struct DqUnit {
  int qb, h, b, hk, NB;
  DevItem it;
  bool ok;
};
__device__ __forceinline__ DqUnit dq_unit(int u, const Params& prm) {
  DqUnit x;
  int64_t uu = u;
  x.qb = (int)(uu % prm.nb); uu /= prm.nb;
  x.h = (int)(uu % prm.Hq); uu /= prm.Hq;
  x.b = (int)(uu % prm.B);
  const int idx = (int)(uu / prm.B);
  x.hk = x.h / (prm.Hq / prm.Hkv);
  x.NB = 0;
  x.ok = idx >= 0 && idx < prm.n_items;
  if (!x.ok) return x;
  x.it = prm.items[idx];  // {p, slot, kv_off, n_kv}
  x.ok = x.it.p >= 0 && x.it.p < prm.P && x.it.slot >= 0 && x.it.slot < prm.n_slots && x.it.n_kv >= 1 &&
         x.it.kv_off >= 0;
  if (x.ok)
    for (int ki = 0; ki < x.it.n_kv; ++ki)
      x.NB += kblocks_of(__ldg(prm.kv_list + x.it.kv_off + ki), x.it.p, prm.causal, prm.nb, x.qb);
  return x;
}
__device__ __forceinline__ void put_unit(volatile int32_t* e, int u, const DqUnit& x) {
  e[0] = u;
  e[1] = x.qb, e[2] = x.h, e[3] = x.b, e[4] = x.NB, e[5] = x.ok ? 1 : 0, e[10] = x.hk;
  e[6] = x.it.p, e[7] = x.it.slot, e[8] = x.it.kv_off, e[9] = x.it.n_kv;
}
__device__ __forceinline__ int get_unit(const volatile int32_t* e, DqUnit& x) {
  x.qb = e[1], x.h = e[2], x.b = e[3], x.NB = e[4], x.ok = e[5] != 0, x.hk = e[10];
  x.it.p = e[6], x.it.slot = e[7], x.it.kv_off = e[8], x.it.n_kv = e[9];
  return e[0];
}

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
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + Ly::RING_OFF);
  const int64_t L = prm.L;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_RES), 1);
    mbar_init(bar(Ly::B_RESE), N_EPI);  // the epilogue warps have copied Q and dO into TMEM
    for (int s = 0; s < Ly::NSA; ++s) {
      mbar_init(bar(Ly::B_AF + s), 1);
      mbar_init(bar(Ly::B_AE + s), 1);
    }
    for (int s = 0; s < Ly::NSB; ++s) {
      mbar_init(bar(Ly::B_BF + s), 1);
      mbar_init(bar(Ly::B_BE + s), 1);
    }
    mbar_init(bar(Ly::B_S), 1);
    mbar_init(bar(Ly::B_SREAD), N_EW);  // S has been loaded by every elementwise warp
    mbar_init(bar(Ly::B_QTF), N_EPI);   // Q and dO of the unit are in TMEM
    mbar_init(bar(Ly::B_QTE), 1);       // the unit's last S and dP products are done with them
    mbar_init(bar(Ly::B_DP), 1);
    mbar_init(bar(Ly::B_DS), N_EW);  // one lane of each elementwise warp
    mbar_init(bar(Ly::B_ACC), 1);
    mbar_init(bar(Ly::B_ACCE), N_EPI);  // one lane of each epilogue warp
    mbar_init(bar(Ly::B_DRAIN), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ly::B_UF + s), 1);
      mbar_init(bar(Ly::B_UE + s), N_EW + 1 + N_EPI);  // elementwise, MMA and epilogue warps read a unit
    }
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(prm.status) != 0) ? 1 : 0;
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

  // the next unit from the ring (consumers: every lane of the warp waits, one lane frees the slot)
  int nu = 0;
  auto take = [&](int& v, DqUnit& y, int role) -> bool {
    const int slot = nu & 1;
    bool r = mbar_wait_warp(bar(Ly::B_UF + slot), (uint32_t)((nu >> 1) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, role, -1);
    if (!r) return false;
    v = get_unit(unit_ring + 16 * slot, y);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(Ly::B_UE + slot));
    ++nu;
    return true;
  };
  auto bad_unit = [&](int u, int role) {
    if (lane == 0) {
      record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, role, u);
      *abort_flag = 1;
    }
    __syncwarp();
  };

  if (warp < N_EW) {
    // ================================================================ elementwise
    regs_inc<EW_REGS>();
    const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
    const int row = wq * 32 + lane;           // TMEM lane = query row within the block
    const int c_base = hf * 64;               // this warp's key columns [c_base, c_base + 64)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_s = tmem + lane_base;          // S
    const uint32_t tm_dp = tmem + lane_base + 128u;  // dP, then dS (bf16)
    bool ok = run;
    int v = -1;
    DqUnit x;
    if (ok) ok = take(v, x, ROLE_EW);
    // LSE and D of this thread's row, loaded as soon as the unit is known and used a phase later
    float raw_lse = 0.f, raw_d = 0.f;
    bool row_in = false;
    auto fetch = [&](const DqUnit& y) {
      const int64_t ql = (int64_t)y.qb * BM + row;
      row_in = ql < L;
      if (row_in) {
        const int64_t gi = ((int64_t)y.b * prm.Hq + y.h) * prm.S + (int64_t)y.it.p * L + ql;
        raw_lse = __ldg(prm.lse + gi);
        raw_d = __ldg(prm.dsum + gi);
      }
    };
    if (ok && v >= 0 && x.ok) fetch(x);
    int64_t g0 = 0;  // global index of the unit's first key block
    while (ok && v >= 0) {
      if (!x.ok || x.NB < 1) {
        bad_unit(v, ROLE_EW);
        ok = false;
        break;
      }
      const int p = x.it.p, qb = x.qb;
      const float lse2 = row_in ? raw_lse * LOG2E : INFINITY;
      const float dsum = row_in ? raw_d : 0.f;
      KCursor cur;
      cur.start(prm, x.it, p, qb);
      for (int j = 0; j < x.NB && ok; ++j) {
        if (j > 0) cur.step(prm, x.it, p, qb);
        const int64_t g = g0 + j;
        const int kp = cur.kp, kbk = cur.kb;
        const int64_t kvalid = L - (int64_t)kbk * BM;
        int hi = (int)min((int64_t)BM, kvalid);                         // keys past the partition end
        if (prm.causal && kp == p && kbk == qb) hi = min(hi, row + 1);  // diagonal block
        hi -= c_base;                                                   // in this half's columns
        const bool any_mask = __any_sync(0xffffffffu, hi < 64);
        ok = mbar_wait(bar(Ly::B_S), (uint32_t)(g & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, j);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float pv[64];
        tmem_ld32(tm_s + (uint32_t)c_base, pv);
        tmem_ld32(tm_s + (uint32_t)c_base + 32u, pv + 32);
        tc_wait_ld();
        // S(g) is in registers: the next block's S may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ly::B_SREAD));
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
        ok = mbar_wait(bar(Ly::B_DP), (uint32_t)(g & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_EW, j);
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
      if (!ok) break;
      // the next unit, and its row's LSE and D (the epilogue warps drain this one)
      int vn = -1;
      DqUnit xn;
      ok = take(vn, xn, ROLE_EW);
      if (!ok) break;
      if (vn >= 0 && xn.ok) fetch(xn);
      g0 += x.NB;
      v = vn;
      x = xn;
    }
  } else if (warp < WARP_EPI) {
    regs_dec<MMA_REGS>();
    if (warp == WARP_MMA) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_sk = idesc_bf16_f32(BM, BM, false);  // S = Q K^T, dP = dO V^T: K-major B
    constexpr uint32_t idesc_ts = idesc_bf16_f32(BM, D, true);    // dQ += dS K, K MN-major
    const uint32_t tm_qt = tmem + 384u, tm_gt = tmem + 384u + (uint32_t)(D / 2);  // Q and dO (bf16)
    constexpr uint64_t TILE16 = Ly::TILE >> 4;
    const uint64_t a_kmaj = smem_desc_sw128(sb + Ly::A0, 16u, 1024u);  // K stages
    const uint64_t a_mn = smem_desc_sw128(sb + Ly::A0, Ly::BOX, 1024u);
    const uint64_t b_kmaj = smem_desc_sw128(sb + Ly::B0, 16u, 1024u);  // V stages
    // Q and dO come from TMEM (copied there once per unit), so these products read only the
    // streamed K or V block from shared memory
    auto issue_s = [&](int64_t g) {  // S(g) = Q K(g)^T
      const uint64_t kd = a_kmaj + (uint64_t)(g % Ly::NSA) * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ts_warp(tmem, tm_qt + (uint32_t)(kk * 8), kd + kmaj_off<D>(kk), idesc_sk, kk > 0 ? 1u : 0u);
      tc_commit_warp(bar(Ly::B_S));
    };
    auto issue_dp = [&](int64_t g) {  // dP(g) = dO V(g)^T; V(g) is read by this product only
      const int sbb = (int)(g % Ly::NSB);
      const uint64_t vd = b_kmaj + (uint64_t)sbb * TILE16;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ts_warp(tmem + 128u, tm_gt + (uint32_t)(kk * 8), vd + kmaj_off<D>(kk), idesc_sk, kk > 0 ? 1u : 0u);
      tc_commit_warp(bar(Ly::B_DP));
      tc_commit_warp(bar(Ly::B_BE + sbb));
    };
    auto issue_dq = [&](int64_t g, bool first) {  // dQ += dS(g) K(g)
      const uint64_t kd = a_mn + (uint64_t)(g % Ly::NSA) * TILE16;
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        tc_mma_ts_warp(tmem + 256u, tmem + 128u + packed_col(kk), kd + (uint64_t)(kk * 128), idesc_ts,
                       (!first || kk > 0) ? 1u : 0u);
      tc_commit_warp(bar(Ly::B_AE + (int)(g % Ly::NSA)));  // K(g): read by S(g) and dQ(g)
    };
    auto wait_a = [&](int64_t g) {  // K(g) landed
      return mbar_wait_warp(bar(Ly::B_AF + (int)(g % Ly::NSA)), (uint32_t)((g / Ly::NSA) & 1), prm.wait_limit_ns,
                            abort_flag, prm.status, ROLE_MMA, (int32_t)g);
    };
    auto wait_b = [&](int64_t g) {  // V(g) landed
      return mbar_wait_warp(bar(Ly::B_BF + (int)(g % Ly::NSB)), (uint32_t)((g / Ly::NSB) & 1), prm.wait_limit_ns,
                            abort_flag, prm.status, ROLE_MMA, (int32_t)g);
    };
    int nqt = 0;
    // S(0) and dP(0) of a unit whose first block is g: issued as soon as its Q and dO are in TMEM
    // (for every unit but the first, after the previous unit's last dQ)
    auto start_unit = [&](const DqUnit& y, int64_t g) -> bool {
      if (!mbar_wait_warp(bar(Ly::B_QTF), (uint32_t)(nqt & 1), prm.wait_limit_ns, abort_flag, prm.status,
                          ROLE_MMA, -1))
        return false;
      ++nqt;
      if (!wait_a(g)) return false;
      tc_fence_after();
      issue_s(g);
      if (!wait_b(g)) return false;
      tc_fence_after();
      issue_dp(g);
      if (y.NB == 1) tc_commit_warp(bar(Ly::B_QTE));  // the unit's last S and dP are issued
      return true;
    };
    bool ok = run;
    int v = -1;
    DqUnit x;
    if (ok) ok = take(v, x, ROLE_MMA);
    if (ok && v >= 0) {
      if (!x.ok || x.NB < 1) {
        bad_unit(v, ROLE_MMA);
        ok = false;
      } else {
        ok = start_unit(x, 0);
      }
    }
    int64_t g0 = 0;
    int k_unit = 0;
    while (ok && v >= 0) {
      const int NB = x.NB;
      for (int j = 0; j < NB && ok; ++j) {
        const int64_t g = g0 + j;
        // S(g) has been read into registers: S(g+1) may overwrite it.  (The next block's S is
        // issued only after this wait, so the barrier cannot run a phase ahead of it.)
        if (j + 1 < NB) {
          ok = mbar_wait_warp(bar(Ly::B_SREAD), (uint32_t)(g & 1), prm.wait_limit_ns, abort_flag, prm.status,
                              ROLE_MMA, j);
          if (!ok) break;
          ok = wait_a(g + 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(g + 1);
        }
        ok = mbar_wait_warp(bar(Ly::B_DS), (uint32_t)(g & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, j);
        if (!ok) break;
        if (j == 0 && k_unit > 0) {  // the previous unit's dQ has been copied out of TMEM
          ok = mbar_wait_warp(bar(Ly::B_ACCE), (uint32_t)((k_unit - 1) & 1), prm.wait_limit_ns, abort_flag,
                              prm.status, ROLE_MMA, -1);
          if (!ok) break;
        }
        tc_fence_after();
        issue_dq(g, j == 0);
        if (j + 1 == NB) tc_commit_warp(bar(Ly::B_ACC));
        if (j + 1 < NB) {
          ok = wait_b(g + 1);
          if (!ok) break;
          tc_fence_after();
          issue_dp(g + 1);
          if (j + 2 == NB) tc_commit_warp(bar(Ly::B_QTE));  // the unit's last S and dP are issued
        }
      }
      if (!ok) break;
      int vn = -1;
      ok = take(vn, x, ROLE_MMA);
      if (!ok) break;
      g0 += NB;
      ++k_unit;
      v = vn;
      if (v < 0) break;
      if (!x.ok || x.NB < 1) {
        bad_unit(v, ROLE_MMA);
        ok = false;
        break;
      }
      ok = start_unit(x, g0);
    }
    // exit-path drain: every MMA issued completes before TMEM is freed
    tc_commit_warp(bar(Ly::B_DRAIN));
    mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
    } else if (warp == WARP_LOAD && lane == 0) {
    // ================================================================ producer
    bool ok = run;
    int np = 0;  // units published
    auto publish = [&](DqUnit& y) -> int {
      const int slot = np & 1;
      ok = mbar_wait(bar(Ly::B_UE + slot), (uint32_t)(((np >> 1) & 1) ^ 1), prm.wait_limit_ns, abort_flag,
                     prm.status, ROLE_LOAD, -1);
      if (!ok) return -1;
      int u = (int)atomicAdd(prm.counter_dq, 1u);
      if (u >= prm.n_dq_units) u = -1;
      if (u >= 0) y = dq_unit(u, prm);
      put_unit(unit_ring + 16 * slot, u, y);
      mbar_arrive(bar(Ly::B_UF + slot));
      ++np;
      return u;
    };
    int nres = 0;
    int64_t ga = 0, gb = 0;  // K and V blocks issued
    DqUnit x, y;
    int u = ok ? publish(x) : -1;
    while (ok && u >= 0) {
      if (!x.ok || x.NB < 1) {
        record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, u);
        *abort_flag = 1;
        break;
      }
      // publish the following unit now and pull its Q, dO rows and first K, V block into L2
      const int un = publish(y);
      if (!ok) break;
      if (un >= 0) {
        if (y.ok) {
          const int64_t qn = ((int64_t)y.b * prm.Hq + y.h) * prm.S + (int64_t)y.it.p * L + (int64_t)y.qb * BM;
          for (int c = 0; c < D / 64; ++c) {
            tma_prefetch_l2_2d(&tmQ, c * 64, (int32_t)qn);
            tma_prefetch_l2_2d(&tmG, c * 64, (int32_t)qn);
          }
          const int kn = __ldg(prm.kv_list + y.it.kv_off);
          if (kn >= 0 && kn < prm.P) {
            const int64_t krn = ((int64_t)y.b * prm.Hkv + y.hk) * prm.S + (int64_t)kn * L;
            for (int c = 0; c < D / 64; ++c) {
              tma_prefetch_l2_2d(&tmK, c * 64, (int32_t)krn);
              tma_prefetch_l2_2d(&tmV, c * 64, (int32_t)krn);
            }
          }
        }
      }
      // resident Q and dO: the previous unit's last S and dP products must be done with them
      ok = mbar_wait(bar(Ly::B_RESE), (uint32_t)((nres & 1) ^ 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_LOAD, u);
      if (!ok) break;
      const int64_t qrow = ((int64_t)x.b * prm.Hq + x.h) * prm.S + (int64_t)x.it.p * L + (int64_t)x.qb * BM;
      mbar_expect_tx(bar(Ly::B_RES), 2 * Ly::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(sb + Ly::RES0 + (uint32_t)c * Ly::BOX, &tmQ, c * 64, (int32_t)qrow, bar(Ly::B_RES));
        tma_load_2d(sb + Ly::RES1 + (uint32_t)c * Ly::BOX, &tmG, c * 64, (int32_t)qrow, bar(Ly::B_RES));
      }
      ++nres;
      const int64_t kvbase = ((int64_t)x.b * prm.Hkv + x.hk) * prm.S;
      KCursor cur;
      cur.start(prm, x.it, x.it.p, x.qb);
      for (int j = 0; j < x.NB && ok; ++j) {
        if (j > 0) cur.step(prm, x.it, x.it.p, x.qb);
        if (cur.kp < 0 || cur.kp >= prm.P) {
          record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, u);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int32_t krow = (int32_t)(kvbase + (int64_t)cur.kp * L + (int64_t)cur.kb * BM);
        const int sa = (int)(ga % Ly::NSA), sbb = (int)(gb % Ly::NSB);
        if (ga >= Ly::NSA) {
          ok = mbar_wait(bar(Ly::B_AE + sa), (uint32_t)((ga / Ly::NSA - 1) & 1), prm.wait_limit_ns, abort_flag,
                         prm.status, ROLE_LOAD, j);
          if (!ok) break;
        }
        mbar_expect_tx(bar(Ly::B_AF + sa), Ly::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::A0 + (uint32_t)sa * Ly::TILE + (uint32_t)c * Ly::BOX, &tmK, c * 64, krow,
                      bar(Ly::B_AF + sa));
        ++ga;
        if (gb >= Ly::NSB) {
          ok = mbar_wait(bar(Ly::B_BE + sbb), (uint32_t)((gb / Ly::NSB - 1) & 1), prm.wait_limit_ns, abort_flag,
                         prm.status, ROLE_LOAD, j);
          if (!ok) break;
        }
        mbar_expect_tx(bar(Ly::B_BF + sbb), Ly::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::B0 + (uint32_t)sbb * Ly::TILE + (uint32_t)c * Ly::BOX, &tmV, c * 64, krow,
                      bar(Ly::B_BF + sbb));
        ++gb;
      }
      u = un;
      x = y;
    }
    // exit-path drain: every load issued lands before the CTA exits
    if (nres > 0) mbar_drain(bar(Ly::B_RES), (uint32_t)((nres - 1) & 1), DRAIN_NS);
    for (int64_t j = (ga > Ly::NSA ? ga - Ly::NSA : 0); j < ga; ++j)
      mbar_drain(bar(Ly::B_AF + (int)(j % Ly::NSA)), (uint32_t)((j / Ly::NSA) & 1), DRAIN_NS);
    for (int64_t j = (gb > Ly::NSB ? gb - Ly::NSB : 0); j < gb; ++j)
      mbar_drain(bar(Ly::B_BF + (int)(j % Ly::NSB)), (uint32_t)((j / Ly::NSB) & 1), DRAIN_NS);
    }
  } else {
    // ================================================================ epilogue
    // Per unit: copy its resident Q and dO from shared memory into TMEM (as the A operands of S
    // and dP) as soon as the previous unit's last S and dP products are done with the TMEM copy,
    // releasing the shared buffers to the producer; then drain the previous unit's dQ while the
    // other roles run this one, releasing it (so the next unit may overwrite it) once its last
    // TMEM load has completed.
    regs_dec<EPI_REGS>();
    const int wq = warp & 3;  // TMEM lane quadrant
    const int r = wq * 32 + lane;  // this thread's row of the 128-row block
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_dq = tmem + lane_base + 256u;
    const uint32_t tm_qt = tmem + lane_base + 384u, tm_gt = tm_qt + (uint32_t)(D / 2);
    bool ok = run;
    int v = -1, k_unit = 0, ncopy = 0;
    DqUnit x;
    // row r of a 128 x D bf16 block landed by TMA in 64-column boxes with 128-byte swizzle (the
    // 16-byte chunk j of a 128-byte row sits at chunk j ^ (r mod 8)), packed two columns per TMEM
    // column from column `dst`
    auto copy_row = [&](uint32_t src_off, uint32_t dst) {
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        const uint8_t* rowp = smem + src_off + (uint32_t)c * Ly::BOX + (uint32_t)r * 128u;
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 q = *reinterpret_cast<const uint4*>(rowp + ((j ^ (r & 7)) << 4));
          w[4 * j] = q.x, w[4 * j + 1] = q.y, w[4 * j + 2] = q.z, w[4 * j + 3] = q.w;
        }
        tmem_st32(dst + (uint32_t)(32 * c), w);
      }
    };
    auto copy_in = [&]() -> bool {
      if (!mbar_wait_warp(bar(Ly::B_RES), (uint32_t)(ncopy & 1), prm.wait_limit_ns, abort_flag, prm.status,
                          ROLE_EPI, -1))
        return false;
      if (ncopy > 0 && !mbar_wait_warp(bar(Ly::B_QTE), (uint32_t)((ncopy - 1) & 1), prm.wait_limit_ns, abort_flag,
                                       prm.status, ROLE_EPI, -1))
        return false;
      tc_fence_after();
      copy_row(Ly::RES0, tm_qt);
      copy_row(Ly::RES1, tm_gt);
      tc_wait_st();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads done before the next TMA write
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(Ly::B_QTF));
        mbar_arrive(bar(Ly::B_RESE));
      }
      ++ncopy;
      return true;
    };
    if (ok) ok = take(v, x, ROLE_EPI);
    if (ok && v >= 0 && x.ok && x.NB >= 1) ok = copy_in();
    while (ok && v >= 0) {
      if (!x.ok || x.NB < 1) {
        bad_unit(v, ROLE_EPI);
        ok = false;
        break;
      }
      int vn = -1;
      DqUnit xn;
      ok = take(vn, xn, ROLE_EPI);
      if (!ok) break;
      if (vn >= 0 && xn.ok && xn.NB >= 1) {
        ok = copy_in();
        if (!ok) break;
      }
      const int64_t row0 =
          (((int64_t)x.b * prm.Hq + x.h) * prm.n_slots + x.it.slot) * L + (int64_t)x.qb * BM + wq * 32;
      const int rows_valid = (int)max((int64_t)0, min((int64_t)32, L - ((int64_t)x.qb * BM + wq * 32)));
      ok = mbar_wait_warp(bar(Ly::B_ACC), (uint32_t)(k_unit & 1), prm.wait_limit_ns, abort_flag, prm.status,
                          ROLE_EPI, -1);
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float t[32];
        tmem_ld32(tm_dq + (uint32_t)c, t);
        tc_wait_ld();
        if (c + 32 == D) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Ly::B_ACCE));
        }
        store_rows<D>(t, prm.scale, prm.dq_part, row0, rows_valid, c, lane);
      }
      ++k_unit;
      v = vn;
      x = xn;
    }
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
  prm.counter_dq = a.counters;
  prm.counter_kv = a.counters + 64;  // the second 256-byte counter slot
  prm.n_dq_units = (int32_t)dq_units;
  prm.n_kv_units = (int32_t)kv_units;
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
  // setmaxnreg hands registers between warpgroups within the launch's pool: the split must fit
  // the registers each kernel is launched with, or a raising warpgroup would wait forever
  for (const void* fn : {(const void*)bwd_dkdv_kernel<D>, (const void*)bwd_dq_kernel<D>}) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncGetAttributes: ") + cudaGetErrorString(e);
      return (int)e;
    }
    if (fa.numRegs * NUM_THREADS < 2 * 128 * EW_REGS + 128 * MMA_REGS + 128 * EPI_REGS) {
      *err = "backward kernels built with " + std::to_string(fa.numRegs) +
             " registers per thread, fewer than their warpgroups' register split needs";
      return (int)cudaErrorInvalidConfiguration;
    }
  }
  // persistent grids: one CTA per SM, units handed out by the counters
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || sms < 1) {
    *err = std::string("SM count: ") + cudaGetErrorString(e);
    return (int)(e != cudaSuccess ? e : cudaErrorInvalidDevice);
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (kv_units > 0)
    bwd_dkdv_kernel<D><<<dim3((unsigned)std::min<int64_t>(kv_units, sms)), dim3(NUM_THREADS), Layout<D>::ALLOC, st>>>(
        mq, mk, mv, mg, prm);
  if (dq_units > 0)
    bwd_dq_kernel<D><<<dim3((unsigned)std::min<int64_t>(dq_units, sms)), dim3(NUM_THREADS), Layout<D>::ALLOC, st>>>(
        mq, mk, mv, mg, prm);
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
