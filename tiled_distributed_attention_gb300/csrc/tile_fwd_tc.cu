// Tile attention forward on the 5th-generation tensor cores (sm_103a).
//
// A work unit is (work item = (Q partition p, tile), batch b, query head h, pair of 128-row
// query tiles of partition p).  For each unit the kernel visits the item's KV partitions in
// planned order, 128 keys at a time, and writes for every query row the partial output
// O_t = acc / l and lse_t = m + ln l.  The per-block recurrence is the online softmax with a
// running maximum m_i and running sum l_i ("环形注意力：突破长序列处理瓶颈的分布式计算范式",
// §"数值稳定性：Log-Sum-Exp技术的分布式应用"); the tile / partial-output structure is
// Mesh-Attention's ("Mesh-Attention: A New Communication-Efficient Distributed Attention with
// Improved Data Locality", tutorial §"Mesh-Attention：从一维'环'到二维'网'": each tile sends its
// partial results back to the Q owner, which merges them).
//
// GB300 mapping: a persistent grid of one CTA per SM; 12 warps = 3 warpgroups.
//   warp 9      producer: takes the next unit from a global counter (units are numbered
//               KV-head-major over the plan's launch order), publishes it through a 2-slot ring in shared
//               memory, then TMA-loads the unit's two Q tiles and streams K and V blocks
//               (128 rows x 64 columns, 128-byte swizzle) through a 2-stage mbarrier ring.
//   warp 8      MMA issuer (one elected lane of a converged warp): S_t = Q_t K^T and O_t += P_t V with
//               tcgen05.mma.cta_group::1.kind::f16 (M = N = 128, K = 16), fp32 accumulators in
//               tensor memory, completion signalled with tcgen05.commit.
//   warps 0-7   softmax, one warpgroup per query tile; thread i owns row i (TMEM lane i), so
//               row max and row sum are thread-local (3-input max and packed f32x2 FMA / ADD in
//               independent chains).  P goes back to TMEM as bf16 in the columns S occupied and
//               feeds the PV product from TMEM.  At the end of a unit the warpgroup copies O_t
//               out of TMEM into registers, releases it (so the next unit's PV can start), and
//               stores the rows through a shared-memory stage as whole 128-byte lines.
//   warps 10-11 idle; warpgroup 2 gives registers to the softmax warpgroups (setmaxnreg).
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  Issue order per block: PV_0(j), S_0(j+1),
// PV_1(j), S_1(j+1), so the softmax of one tile overlaps the other tile's MMAs.  O is
// rescaled only when the running max grows by more than 2^8.
//
// Every mbarrier wait is bounded: a timeout records MESH_ATTN_ERR_DEVICE_TIMEOUT in the status
// block, every role of the CTA stops, in-flight copies and MMAs are drained and TMEM is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace tc {

constexpr int BM = 128;  // query rows per tile = TMEM lanes
constexpr int BN = 128;  // keys per KV block
constexpr int NST = 2;   // K/V ring stages
constexpr int NUM_THREADS = 384;
constexpr int SOFTMAX_REGS = 200;  // 2 x 128 x 200 + 128 x 104 <= 384 x 168 registers at launch
constexpr int OTHER_REGS = 104;
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
constexpr float LOG2_RESCALE = 8.0f;
// Row sum of one block accepted without a max pass: every term is then at most 2^16, and a sum
// this large implies a row maximum more than 2^LOG2_RESCALE above the reference (2^16 / BN > 2^8).
constexpr float SUM_ACCEPT = 65536.0f;
constexpr int64_t DRAIN_NS = 200000000;  // exit-path waits for copies in flight

// roles recorded with an error
constexpr int ROLE_SOFTMAX = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_ITEM = 4;

template <int D>
struct Layout {
  static constexpr uint32_t TILE = BM * D * 2;  // bytes of one Q tile / K block / V block
  static constexpr uint32_t BOX = BM * 64 * 2;  // one 128 x 64 bf16 TMA box (16 KB)
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + 2 * TILE;
  static constexpr uint32_t V_OFF = K_OFF + NST * TILE;
  static constexpr uint32_t EPI_OFF = V_OFF + NST * TILE;  // 8 softmax warps x 32 x 32 fp32
  static constexpr uint32_t BAR_OFF = EPI_OFF + 8 * 4096;
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + NST,
                       B_VFULL = B_KEMPTY + NST, B_VEMPTY = B_VFULL + NST, B_SFULL = B_VEMPTY + NST,
                       B_PFULL = B_SFULL + 2, B_OFINAL = B_PFULL + 2, B_OFREE = B_OFINAL + 2,
                       B_UFULL = B_OFREE + 2, B_UEMPTY = B_UFULL + 2, B_DRAIN = B_UEMPTY + 2,
                       NBARS = B_DRAIN + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag, unit ring[2]
  static constexpr uint32_t TOTAL = MISC_OFF + 16;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
};

struct Params {
  const DevItem* items;
  const int32_t* kv_list;
  float* part_o;
  float* part_lse;
  int32_t* status;
  uint32_t* counter;
  int64_t S, L;
  int32_t B, Hq, Hkv, P, n_items, n_slots, n_pairs, n_units, causal;
  float scale_log2;
  int64_t wait_limit_ns;
};

// What every role derives from a unit index.  Units are numbered KV-head-major: (batch, KV head,
// work item in the plan's launch order, query head of the group, tile pair), so the units running
// at once on the grid share one KV head's partitions and the query heads of a group share them in
// L2.
struct Unit {
  int b, h, qp;
  DevItem it;
  bool ok;      // item indices in range
  int ntiles;   // 1 or 2 query tiles (2 unless the partition has an odd number of tiles)
  int a0;       // first query tile index within the partition
  int a_max;    // last query tile index
  int nb;       // 128-key blocks per KV partition
};

__device__ __forceinline__ Unit decode(int u, const Params& prm) {
  Unit x;
  const int g = prm.Hq / prm.Hkv;
  x.qp = u % prm.n_pairs;
  u /= prm.n_pairs;
  const int gi = u % g;
  u /= g;
  const int item = u % prm.n_items;
  u /= prm.n_items;
  const int hk = u % prm.Hkv;
  x.b = u / prm.Hkv;
  x.h = hk * g + gi;
  x.it = prm.items[item];
  x.ok = x.b < prm.B && x.it.p >= 0 && x.it.p < prm.P && x.it.slot >= 0 && x.it.slot < prm.n_slots &&
         x.it.n_kv >= 1 && x.it.kv_off >= 0;
  x.nb = (int)((prm.L + BN - 1) / BN);
  x.a0 = 2 * x.qp;
  x.ntiles = ((int64_t)(x.a0 + 1) * BM < prm.L) ? 2 : 1;
  x.a_max = x.a0 + x.ntiles - 1;
  return x;
}

// 128-key blocks of KV partition k visited for Q partition p by a unit whose last query tile
// is a_max: only the causal diagonal partition is cut short.
__device__ __forceinline__ int blocks_of(int k, int p, int causal, int nb, int a_max) {
  return (causal && k == p) ? min(nb, a_max + 1) : nb;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tile_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params prm) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;  // 1024-aligned base (128-byte swizzle atoms)
  uint8_t* smem = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + Ly::BAR_OFF + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 4);
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 8);
  const int64_t L = prm.L;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_QFULL), 1);
    mbar_init(bar(Ly::B_QEMPTY), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(Ly::B_KFULL + s), 1);
      mbar_init(bar(Ly::B_KEMPTY + s), 1);
      mbar_init(bar(Ly::B_VFULL + s), 1);
      mbar_init(bar(Ly::B_VEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Ly::B_SFULL + t), 1);
      mbar_init(bar(Ly::B_PFULL + t), BM);
      mbar_init(bar(Ly::B_OFINAL + t), 1);
      mbar_init(bar(Ly::B_OFREE + t), BM);
      mbar_init(bar(Ly::B_UFULL + t), 1);
      mbar_init(bar(Ly::B_UEMPTY + t), 1 + 8);  // one lane of the MMA warp and of each softmax warp
    }
    mbar_init(bar(Ly::B_DRAIN), 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ================================================================ softmax warpgroups
    regs_inc<SOFTMAX_REGS>();
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_s = tmem + lane_base + (uint32_t)(t * 128);
    const uint32_t tm_o = tmem + lane_base + 256u + (uint32_t)(t * 128);
    float* epi = reinterpret_cast<float*>(smem + Ly::EPI_OFF + (uint32_t)warp * 4096u);
    int nu = 0, cnt = 0, uses = 0;
    bool ok = true;
    while (ok) {
      const int slot = nu & 1;
      ok = mbar_wait(bar(Ly::B_UFULL + slot), (uint32_t)((nu >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_SOFTMAX, -1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int u = unit_ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_UEMPTY + slot));
      ++nu;
      if (u < 0) break;
      const Unit x = decode(u, prm);
      if (!x.ok) break;
      if (t >= x.ntiles) continue;
      const int p = x.it.p;
      const int a_t = x.a0 + t;
      const int32_t* kvl = prm.kv_list + x.it.kv_off;
      float m_used = -INFINITY, l_sum = 0.f;
      for (int ki = 0; ki < x.it.n_kv && ok; ++ki) {
        const int k = __ldg(kvl + ki);
        const bool diag = prm.causal && k == p;
        const int nbk = blocks_of(k, p, prm.causal, x.nb, x.a_max);
        for (int jb = 0; jb < nbk; ++jb, ++cnt) {
          ok = mbar_wait(bar(Ly::B_SFULL + t), (uint32_t)(cnt & 1), prm.wait_limit_ns, abort_flag, prm.status,
                         ROLE_SOFTMAX, u);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          // mask: causal diagonal block (key column > query row) and keys past the partition
          const int kv_valid = (int)min((int64_t)BN, L - (int64_t)jb * BN);
          int lim = BN - 1;
          if (diag) lim = (jb < a_t) ? BN - 1 : (jb == a_t ? row : -1);
          lim = min(lim, kv_valid - 1);
          // The exponentials use the row's running reference m_used, which only ever grows.  A
          // block whose row maximum stays within 2^LOG2_RESCALE of it needs no maximum at all, so
          // the common case skips the max pass: exponentiate against m_used and accept the block
          // when its row sum is at most SUM_ACCEPT (every term is then bounded as well).  A row
          // without a reference yet (first block of the unit), or a block whose sum is too large
          // or not finite, takes the row maximum first, raising m_used (and rescaling O and l)
          // when it grew by more than 2^LOG2_RESCALE, and the exponentials are redone.
          bool need_max = __any_sync(0xffffffffu, m_used == -INFINITY);
          float factor = 1.f, blk = 0.f;
          uint32_t pk[BN / 2];
#pragma unroll 1
          for (int pass = 0;; ++pass) {
            // S_t stays in TMEM until P_t is written, so a second pass reloads it rather than
            // keeping 128 scores live across the pass
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN; c += 32) tmem_ld32(tm_s + (uint32_t)c, s + c);
            tc_wait_ld();
            if (lim < BN - 1) {
#pragma unroll
              for (int c = 0; c < BN; ++c)
                if (c > lim) s[c] = -INFINITY;
            }
            if (need_max) {
              // row max: four independent chains of 3-input max
              float mc[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float v = max3f(s[32 * q], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
                for (int i = 3; i + 1 < 32; i += 2) v = max3f(v, s[32 * q + i], s[32 * q + i + 1]);
                mc[q] = fmaxf(v, s[32 * q + 31]);
              }
              const float m_new = fmaxf(max3f(mc[0], mc[1], mc[2]), mc[3]) * prm.scale_log2;
              if (m_new > -INFINITY) {
                if (m_used == -INFINITY) {
                  m_used = m_new;
                } else if (m_new > m_used + LOG2_RESCALE) {
                  factor *= fast_exp2(m_used - m_new);
                  m_used = m_new;
                }
              }
            }
            const float mref = (m_used == -INFINITY) ? 0.f : m_used;
            // p = 2^(s * scale * log2 e - m): two elements per FMA, four independent sum chains
            const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2);
            const uint64_t nm2 = f2_pack(-mref, -mref);
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sc2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              acc2[c & 3] = f2_add(acc2[c & 3], f2_pack(p0, p1));
              pk[c] = pack_bf16x2(p0, p1);
            }
            float sa, sb2;
            f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), sa, sb2);
            blk = sa + sb2;
            // NaN fails the comparison: a NaN row takes the max pass once and is then accepted
            if (pass == 1 || __all_sync(0xffffffffu, blk <= SUM_ACCEPT)) break;
            need_max = true;
          }
          if (__any_sync(0xffffffffu, factor != 1.f)) {
            // O_t holds every earlier PV product of this unit: S_t(j) was issued after
            // PV_t(j-1) and its completion covers all earlier tensor-core work.
            l_sum *= factor;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              float o[32];
              tmem_ld32(tm_o + (uint32_t)c, o);
              tc_wait_ld();
              uint32_t w[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(o[e] * factor);
              tmem_st32(tm_o + (uint32_t)c, w);
            }
          }
          l_sum += blk;
          tmem_st32(tm_s, pk);
          tmem_st32(tm_s + 32u, pk + 32);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(bar(Ly::B_PFULL + t));
        }
      }
      if (!ok) break;
      // ---- epilogue: copy O_t out of TMEM, release it, store through the shared stage
      ok = mbar_wait(bar(Ly::B_OFINAL + t), (uint32_t)(uses & 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_SOFTMAX, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float o[D];
#pragma unroll
      for (int c = 0; c < D; c += 32) tmem_ld32(tm_o + (uint32_t)c, o + c);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(Ly::B_OFREE + t));
      ++uses;
      const int64_t row_local = (int64_t)a_t * BM + row;
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const int64_t prow = (((int64_t)x.b * prm.Hq + x.h) * prm.n_slots + x.it.slot) * L + row_local;
      const int64_t wrow0 = row_local - lane;          // warp's first row in the partition
      float* dst0 = prm.part_o + (prow - lane) * D;    // that row in the slot
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        // 32 rows x 32 columns: 16-byte chunks swizzled by row, read back 4 rows per store
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(epi + lane * 32 + ((q ^ (lane & 7)) * 4)) =
              make_float4(o[c + 4 * q] * inv, o[c + 4 * q + 1] * inv, o[c + 4 * q + 2] * inv,
                          o[c + 4 * q + 3] * inv);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = i * 4 + (lane >> 3), qq = lane & 7;
          const float4 v = *reinterpret_cast<const float4*>(epi + r * 32 + ((qq ^ (r & 7)) * 4));
          if (wrow0 + r < L) *reinterpret_cast<float4*>(dst0 + (int64_t)r * D + c + qq * 4) = v;
        }
        __syncwarp();
      }
      if (row_local < L)
        prm.part_lse[prow] = l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
    }
  } else {
    regs_dec<OTHER_REGS>();
    if (warp == WARP_MMA) {
      // ================================================================ MMA issuer
      // The whole warp runs this loop converged; tcgen05.mma and tcgen05.commit are issued by
      // one elected lane (tc_*_warp), every wait is warp-uniform (mbar_wait_warp).
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
      // Base descriptors are built once; per instruction only the start-address field (the
      // low 14 bits, address / 16) advances by a compile-time offset.  Shared addresses stay
      // below 256 KB, so the addition never carries out of that field.  Keeping the issuing
      // warp's work per MMA to a few independent adds on uniform values is what lets one warp
      // keep the tensor pipe fed.
      const uint64_t q_desc0 = smem_desc_sw128(sb + Ly::Q_OFF, 16u, 1024u);
      const uint64_t k_desc0 = smem_desc_sw128(sb + Ly::K_OFF, 16u, 1024u);
      const uint64_t v_desc0 = smem_desc_sw128(sb + Ly::V_OFF, Ly::BOX, 1024u);
      constexpr uint64_t TILE16 = Ly::TILE >> 4, BOX16 = Ly::BOX >> 4;
      // K-major operand (Q or K): K-step kk of 16 elements sits in box kk/4 at byte 32*(kk%4)
      auto kmaj_off = [](int kk) { return (uint64_t)((kk >> 2) * BOX16 + (kk & 3) * 2); };
      // MN-major V: K-step kk covers key rows 16kk..16kk+15 (two 8-row swizzle atoms, 2048
      // bytes); the second 64-column half of d is the next box (leading byte offset)
      auto issue_s = [&](int t, int stage) {
        const uint64_t qd = q_desc0 + (uint64_t)t * TILE16;
        const uint64_t kd = k_desc0 + (uint64_t)stage * TILE16;
        const uint32_t d_tm = tmem + (uint32_t)(t * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) tc_mma_ss_warp(d_tm, qd + kmaj_off(kk), kd + kmaj_off(kk), idesc_qk, kk > 0);
        tc_commit_warp(bar(Ly::B_SFULL + t));
      };
      auto issue_pv = [&](int t, int stage, bool first) {
        const uint64_t vd = v_desc0 + (uint64_t)stage * TILE16;
        const uint32_t tm_p = tmem + (uint32_t)(t * 128);
        const uint32_t tm_o = tmem + 256u + (uint32_t)(t * 128);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc_mma_ts_warp(tm_o, tm_p + (uint32_t)(kk * 8), vd + (uint64_t)(kk * 128), idesc_pv, (!first || kk > 0) ? 1u : 0u);
      };
      int nu = 0, nblk = 0;
      int cnt[2] = {0, 0}, uses[2] = {0, 0};
      bool ok = true;
      while (ok) {
        const int slot = nu & 1;
        ok = mbar_wait_warp(bar(Ly::B_UFULL + slot), (uint32_t)((nu >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                       ROLE_MMA, -1);
        if (!ok) break;
        const int u = unit_ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ly::B_UEMPTY + slot));
        __syncwarp();
        const int uidx = nu++;
        if (u < 0) break;
        const Unit x = decode(u, prm);
        if (!x.ok) break;
        const int32_t* kvl = prm.kv_list + x.it.kv_off;
        int NB = 0;
        for (int ki = 0; ki < x.it.n_kv; ++ki) NB += blocks_of(__ldg(kvl + ki), x.it.p, prm.causal, x.nb, x.a_max);
        ok = mbar_wait_warp(bar(Ly::B_QFULL), (uint32_t)(uidx & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, u);
        if (ok)
          ok = mbar_wait_warp(bar(Ly::B_KFULL + nblk % NST), (uint32_t)((nblk / NST) & 1), prm.wait_limit_ns, abort_flag,
                         prm.status, ROLE_MMA, u);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < x.ntiles; ++t) issue_s(t, nblk % NST);
        if (NB == 1) tc_commit_warp(bar(Ly::B_QEMPTY));
        tc_commit_warp(bar(Ly::B_KEMPTY + nblk % NST));
        for (int j = 0; j < NB && ok; ++j) {
          const int g = nblk + j;
          const int st = g % NST;
          ok = mbar_wait_warp(bar(Ly::B_VFULL + st), (uint32_t)((g / NST) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                         ROLE_MMA, u);
          for (int t = 0; t < x.ntiles && ok; ++t) {
            ok = mbar_wait_warp(bar(Ly::B_PFULL + t), (uint32_t)(cnt[t] & 1), prm.wait_limit_ns, abort_flag, prm.status,
                           ROLE_MMA, u);
            if (ok && j == 0 && uses[t] > 0)  // the previous unit's epilogue has copied O_t out
              ok = mbar_wait_warp(bar(Ly::B_OFREE + t), (uint32_t)((uses[t] - 1) & 1), prm.wait_limit_ns, abort_flag,
                             prm.status, ROLE_MMA, u);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, st, j == 0);
            ++cnt[t];
            if (j + 1 == NB) {  // tile t's last product of the unit: its epilogue may start
              tc_commit_warp(bar(Ly::B_OFINAL + t));
              ++uses[t];
            }
            if (j + 1 < NB) {
              const int sn = (g + 1) % NST;
              if (t == 0) {
                ok = mbar_wait_warp(bar(Ly::B_KFULL + sn), (uint32_t)(((g + 1) / NST) & 1), prm.wait_limit_ns, abort_flag,
                               prm.status, ROLE_MMA, u);
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(t, sn);
            }
          }
          if (!ok) break;
          if (j + 1 < NB) tc_commit_warp(bar(Ly::B_KEMPTY + (g + 1) % NST));
          if (j + 2 == NB) tc_commit_warp(bar(Ly::B_QEMPTY));  // the unit's last S products are issued
          tc_commit_warp(bar(Ly::B_VEMPTY + st));
        }
        if (!ok) break;
        nblk += NB;
      }
      // exit-path drain: every MMA issued completes before TMEM is freed
      tc_commit_warp(bar(Ly::B_DRAIN));
      mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
    } else if (warp == WARP_LOAD && lane == 0) {
      // ================================================================ producer
      int nu = 0, nq = 0, nk = 0, nv = 0;
      bool ok = *abort_flag == 0;
      // take the next unit from the global counter and publish it to the consumers' ring
      auto publish = [&]() -> int {
        const int slot = nu & 1;
        ok = mbar_wait(bar(Ly::B_UEMPTY + slot), (uint32_t)(((nu >> 1) & 1) ^ 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, -1);
        if (!ok) return -1;
        int v = (int)atomicAdd(prm.counter, 1u);
        if (v >= prm.n_units) v = -1;
        unit_ring[slot] = v;
        mbar_arrive(bar(Ly::B_UFULL + slot));
        ++nu;
        return v;
      };
      int u = ok ? publish() : -1;
      while (ok && u >= 0) {
        const Unit x = decode(u, prm);
        if (!x.ok) {
          record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_ITEM, u);
          *abort_flag = 1;
          break;
        }
        // publish the following unit now and pull its Q tiles and first K/V block into L2, so
        // the unit boundary does not wait on DRAM
        const int un = publish();
        if (!ok) break;
        if (un >= 0) {
          const Unit xn = decode(un, prm);
          if (xn.ok) {
            const int64_t qn = ((int64_t)xn.b * prm.Hq + xn.h) * prm.S + (int64_t)xn.it.p * L + (int64_t)xn.a0 * BM;
            for (int t = 0; t < xn.ntiles; ++t)
              for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_2d(&tmQ, c * 64, (int32_t)(qn + (int64_t)t * BM));
            const int kn = __ldg(prm.kv_list + xn.it.kv_off);
            if (kn >= 0 && kn < prm.P) {
              const int64_t krn = ((int64_t)xn.b * prm.Hkv + xn.h / (prm.Hq / prm.Hkv)) * prm.S + (int64_t)kn * L;
              for (int c = 0; c < D / 64; ++c) {
                tma_prefetch_l2_2d(&tmK, c * 64, (int32_t)krn);
                tma_prefetch_l2_2d(&tmV, c * 64, (int32_t)krn);
              }
            }
          }
        }
        // Q tiles: the previous unit's last S products must be done with the Q buffer
        ok = mbar_wait(bar(Ly::B_QEMPTY), (uint32_t)((nq & 1) ^ 1), prm.wait_limit_ns, abort_flag, prm.status,
                       ROLE_LOAD, u);
        if (!ok) break;
        const int64_t qrow0 = ((int64_t)x.b * prm.Hq + x.h) * prm.S + (int64_t)x.it.p * L + (int64_t)x.a0 * BM;
        mbar_expect_tx(bar(Ly::B_QFULL), (uint32_t)x.ntiles * Ly::TILE);
        for (int t = 0; t < x.ntiles; ++t)
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sb + Ly::Q_OFF + (uint32_t)t * Ly::TILE + (uint32_t)c * Ly::BOX, &tmQ, c * 64,
                        (int32_t)(qrow0 + (int64_t)t * BM), bar(Ly::B_QFULL));
        ++nq;
        const int hk = x.h / (prm.Hq / prm.Hkv);
        const int64_t kvbase = ((int64_t)x.b * prm.Hkv + hk) * prm.S;
        const int32_t* kvl = prm.kv_list + x.it.kv_off;
        for (int ki = 0; ki < x.it.n_kv && ok; ++ki) {
          const int k = __ldg(kvl + ki);
          if (k < 0 || k >= prm.P) {
            record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, u);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const int nbk = blocks_of(k, x.it.p, prm.causal, x.nb, x.a_max);
          for (int jb = 0; jb < nbk; ++jb) {
            const int st = nk % NST;
            const uint32_t ph = (uint32_t)((nk / NST) & 1);
            const int32_t krow = (int32_t)(kvbase + (int64_t)k * L + (int64_t)jb * BN);
            ok = mbar_wait(bar(Ly::B_KEMPTY + st), ph ^ 1u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_LOAD, u);
            if (!ok) break;
            mbar_expect_tx(bar(Ly::B_KFULL + st), Ly::TILE);
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(sb + Ly::K_OFF + (uint32_t)st * Ly::TILE + (uint32_t)c * Ly::BOX, &tmK, c * 64, krow,
                          bar(Ly::B_KFULL + st));
            ++nk;
            ok = mbar_wait(bar(Ly::B_VEMPTY + st), ph ^ 1u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_LOAD, u);
            if (!ok) break;
            mbar_expect_tx(bar(Ly::B_VFULL + st), Ly::TILE);
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(sb + Ly::V_OFF + (uint32_t)st * Ly::TILE + (uint32_t)c * Ly::BOX, &tmV, c * 64, krow,
                          bar(Ly::B_VFULL + st));
            ++nv;
          }
        }
        u = un;
      }
      // exit-path drain: every load issued lands before the CTA exits
      if (nq > 0) mbar_drain(bar(Ly::B_QFULL), (uint32_t)((nq - 1) & 1), DRAIN_NS);
      for (int jj = (nk > NST ? nk - NST : 0); jj < nk; ++jj)
        mbar_drain(bar(Ly::B_KFULL + jj % NST), (uint32_t)((jj / NST) & 1), DRAIN_NS);
      for (int jj = (nv > NST ? nv - NST : 0); jj < nv; ++jj)
        mbar_drain(bar(Ly::B_VFULL + jj % NST), (uint32_t)((jj / NST) & 1), DRAIN_NS);
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
static int launch(const TileArgs& a, void* stream, std::string* err) {
  const int64_t n_tiles = (a.L + BM - 1) / BM;
  const int64_t n_pairs = (n_tiles + 1) / 2;
  const int64_t units = (int64_t)a.n_items * a.B * a.Hq * n_pairs;
  if (units <= 0) return (int)cudaSuccess;
  if (units > 0x7fffffff) {
    *err = "too many work units for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  EncodeTiledFn enc = get_encode(err);
  if (!enc) return (int)cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_map(enc, &mq, a.Q, (uint64_t)a.B * a.Hq * a.S, D, err) ||
      !make_map(enc, &mk, a.K, (uint64_t)a.B * a.Hkv * a.S, D, err) ||
      !make_map(enc, &mv, a.V, (uint64_t)a.B * a.Hkv * a.S, D, err))
    return (int)cudaErrorInvalidValue;
  Params prm;
  prm.items = a.items;
  prm.kv_list = a.kv_list;
  prm.part_o = a.part_o;
  prm.part_lse = a.part_lse;
  prm.status = a.status;
  prm.counter = a.counter;
  prm.S = a.S;
  prm.L = a.L;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.P = a.P;
  prm.n_items = a.n_items;
  prm.n_slots = a.n_slots;
  prm.n_pairs = (int32_t)n_pairs;
  prm.n_units = (int32_t)units;
  prm.causal = a.causal;
  prm.scale_log2 = a.scale_log2;
  prm.wait_limit_ns = a.wait_limit_ns;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    *err = std::string("device query: ") + cudaGetErrorString(e);
    return (int)e;
  }
  auto kern = tile_fwd_tc_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<D>::ALLOC);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  const unsigned grid = (unsigned)(units < sms ? units : sms);  // persistent: one CTA per SM
  kern<<<dim3(grid), dim3(NUM_THREADS), Layout<D>::ALLOC, (cudaStream_t)stream>>>(mq, mk, mv, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("tile_fwd_tc launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace tc

int launch_tile_fwd_tc(const TileArgs& a, void* stream, std::string* err) {
  if (a.d == 128) return tc::launch<128>(a, stream, err);
  if (a.d == 64) return tc::launch<64>(a, stream, err);
  *err = "tensor-core tile kernel supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
