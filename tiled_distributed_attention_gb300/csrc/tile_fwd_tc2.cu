// Tile attention forward on SM pairs: 5th-generation tensor-core products shared by two CTAs
// (tcgen05.mma.cta_group::2), d = 128, bf16 inputs.
//
// What it computes is what the one-SM kernel computes: for each work unit (work item = (Q
// partition p, tile), batch b, query head h, pair of 128-row query tiles of p) it visits the
// item's KV partitions in planned order, 128 keys at a time, and writes for every query row the
// partial output O_t = acc / l and lse_t = m + ln l (the online-softmax recurrence with running
// maximum m_i and running sum l_i of "环形注意力：突破长序列处理瓶颈的分布式计算范式",
// §"数值稳定性：Log-Sum-Exp技术的分布式应用"; partial outputs per tile as in "Mesh-Attention: A
// New Communication-Efficient Distributed Attention with Improved Data Locality", tutorial
// §"Mesh-Attention：从一维'环'到二维'网'").
//
// GB300 mapping: a cluster of two CTAs on two SMs takes one unit at a time; CTA rank r owns
// query tile a0 + r (128 rows = its TMEM lanes).  The even CTA issues the pair's products with
// M = 256: S = Q K^T with each CTA holding 64 of a block's 128 keys (the B operand's N halves),
// and O += P V with each CTA holding 64 of V's 128 columns.  Each SM therefore loads half of
// every K and V block and reads half of every B operand from its own shared memory, which is
// what leaves room for a double-buffered S in TMEM:
//   TMEM per CTA (512 columns): S_0 | S_1 | O_a | O_b.
// The two softmax warpgroups of a CTA split the keys of a block: warpgroup a takes keys 0-63,
// warpgroup b keys 64-127, each with its own running maximum, running sum and accumulator
// (O_a += P_a V[0:64), O_b += P_b V[64:128)), so neither waits for the other inside a unit; the
// two halves are merged by the same LSE rule once per unit in the epilogue.  With S(j+2) issued
// as soon as PV(j) is, the softmax of block j+1 overlaps the products of blocks j and j+2.
//
// Warp roles (12 warps, both CTAs):
//   warp 9      producer: loads the CTA's Q tile and its halves of K and V blocks by TMA
//               through 4-stage rings (128-byte swizzle); in the even CTA it also takes units
//               from the global counter and publishes them to both CTAs' unit rings.
//   warp 8      even CTA: MMA issuer (one elected lane of a converged warp).  Odd CTA: relay --
//               it waits for the odd CTA's own loads to land and arrives on the even CTA's
//               "full" barriers, so the issuer knows both halves of an operand are resident.
//   warps 0-7   softmax (warpgroup a: warps 0-3, b: warps 4-7); thread = row (TMEM lane).
//   warps 10-11 idle; warpgroup 2 gives registers to the softmax warpgroups (setmaxnreg).
// Barriers the issuer waits on live in the even CTA (the odd CTA arrives remotely); completion
// of products is multicast to the barrier of the same offset in both CTAs.
//
// Every mbarrier wait is bounded: a timeout records MESH_ATTN_ERR_DEVICE_TIMEOUT, both CTAs of
// the pair stop, in-flight copies and products are drained, and TMEM is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace tc2 {

constexpr int D = 128;   // head dimension
constexpr int BM = 128;  // query rows per CTA (TMEM lanes); a pair covers 256
constexpr int BN = 128;  // keys per block; each CTA holds 64 of them
constexpr int HALF = 64;
constexpr int NSTK = 4;  // K ring stages
constexpr int NSTV = 4;  // V ring stages
constexpr int NUM_THREADS = 384;
constexpr int SOFTMAX_REGS = 208;  // 2 x 128 x 208 + 128 x 88 = 384 x 168 registers at launch
constexpr int OTHER_REGS = 88;
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
constexpr float LOG2_RESCALE = 8.0f;
// Half-row sum of one block accepted without a max pass: every term is then at most 2^16, and a
// sum this large implies a maximum more than 2^LOG2_RESCALE above the reference (2^16 / 64 > 2^8).
constexpr float SUM_ACCEPT = 65536.0f;
constexpr int64_t DRAIN_NS = 200000000;  // exit-path waits for copies and products in flight
constexpr uint16_t PAIR = 0x3;           // both CTAs of the cluster

constexpr int ROLE_SOFTMAX = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_ITEM = 4, ROLE_RELAY = 5;

struct Layout {
  static constexpr uint32_t QBOX = BM * 64 * 2;    // 128 rows x 64 columns (16 KB)
  static constexpr uint32_t KBOX = HALF * 64 * 2;  // 64 keys x 64 columns (8 KB)
  static constexpr uint32_t Q_BYTES = 2 * QBOX;    // the CTA's Q tile
  static constexpr uint32_t K_STAGE = 2 * KBOX;    // the CTA's 64 keys x 128 columns
  static constexpr uint32_t V_STAGE = BN * 64 * 2; // 128 keys x the CTA's 64 columns (16 KB)
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + NSTK * K_STAGE;
  static constexpr uint32_t EPI_OFF = V_OFF + NSTV * V_STAGE;  // 8 softmax warps x 32 x 32 fp32
  static constexpr uint32_t XCH_OFF = EPI_OFF + 8 * 4096;      // [unit parity][warpgroup][row] (m, l)
  static constexpr uint32_t BAR_OFF = XCH_OFF + 2 * 2 * BM * 8;
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + NSTK, B_VFULL = B_KEMPTY + NSTK,
                       B_VEMPTY = B_VFULL + NSTV, B_SFULL = B_VEMPTY + NSTV, B_PFULL = B_SFULL + 2,
                       B_PVDONE = B_PFULL + 4, B_OFINAL = B_PVDONE + 2, B_OFREE = B_OFINAL + 1,
                       B_XCH = B_OFREE + 1, B_UFULL = B_XCH + 1, B_UEMPTY = B_UFULL + 2, B_DRAIN = B_UEMPTY + 2,
                       NBARS = B_DRAIN + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag, unit ring[2]
  static constexpr uint32_t TOTAL = MISC_OFF + 16;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
};
static_assert(Layout::ALLOC <= 227 * 1024, "shared memory layout exceeds the per-CTA limit");
static_assert(Layout::Q_OFF % 1024 == 0 && Layout::K_OFF % 1024 == 0 && Layout::V_OFF % 1024 == 0,
              "operand tiles must start on 1024-byte swizzle atoms");

// arrivals the even CTA's unit-ring "empty" barrier takes per unit: its MMA warp and 8 softmax
// warps, the odd CTA's producer, relay and 8 softmax warps
constexpr uint32_t UEMPTY_ARRIVALS = 1 + 8 + 1 + 1 + 8;

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
// work item in planned order, query head of the group, tile pair), so the units running at once
// on the grid share one KV head's partitions and the query heads of a group share them in L2.
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

__global__ void __launch_bounds__(NUM_THREADS, 1)
    tile_fwd_tc2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Params prm) {
  using Ly = Layout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;  // 1024-aligned base, the same offset in both CTAs
  uint8_t* smem = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  auto bar = [&](int i) { return sb + Ly::BAR_OFF + 8u * (uint32_t)i; };
  // the even CTA's barrier i, as an address of the cluster window
  auto bar0 = [&](int i) { return mapa_shared(bar(i), 0u); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 4);
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 8);
  const uint32_t peer_abort = mapa_shared(sb + Ly::MISC_OFF + 4, rank ^ 1u);
  const int64_t L = prm.L;
  // stop both CTAs of the pair: the peer's waits see its own flag
  auto abort_pair = [&]() {
    *abort_flag = 1;
    st_shared_cluster(peer_abort, 1u);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_QFULL), even ? 2 : 1);  // own expect_tx (+ the odd CTA's relay)
    mbar_init(bar(Ly::B_QEMPTY), 1);
    for (int s = 0; s < NSTK; ++s) {
      mbar_init(bar(Ly::B_KFULL + s), even ? 2 : 1);
      mbar_init(bar(Ly::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NSTV; ++s) {
      mbar_init(bar(Ly::B_VFULL + s), even ? 2 : 1);
      mbar_init(bar(Ly::B_VEMPTY + s), 1);
    }
    for (int t = 0; t < 4; ++t) mbar_init(bar(Ly::B_PFULL + t), 8);  // 4 warps of the warpgroup in each CTA
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Ly::B_SFULL + t), 1);
      mbar_init(bar(Ly::B_PVDONE + t), 1);
      mbar_init(bar(Ly::B_UFULL + t), 1);
      mbar_init(bar(Ly::B_UEMPTY + t), UEMPTY_ARRIVALS);
    }
    mbar_init(bar(Ly::B_OFINAL), 1);
    mbar_init(bar(Ly::B_OFREE), 16);  // 8 softmax warps in each CTA
    mbar_init(bar(Ly::B_XCH), 8);     // this CTA's 8 softmax warps
    mbar_init(bar(Ly::B_DRAIN), 1);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(prm.status) != 0) ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == WARP_MMA) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  if (warp == WARP_LOAD && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // consumers take a unit from their CTA's ring and release the slot on the even CTA's barrier
  auto take_unit = [&](int nu, int role, bool arrive) -> int {
    const int slot = nu & 1;
    bool ok = mbar_wait_cl(bar(Ly::B_UFULL + slot), (uint32_t)((nu >> 1) & 1), prm.wait_limit_ns, abort_flag,
                           prm.status, role, -1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return -2;
    const int u = unit_ring[slot];
    __syncwarp();
    if (arrive && lane == 0) mbar_arrive_cluster(bar0(Ly::B_UEMPTY + slot));
    __syncwarp();
    return u;
  };

  if (warp < 8) {
    // ================================================================ softmax warpgroups
    regs_inc<SOFTMAX_REGS>();
    const int wg = warp >> 2;  // 0: keys 0-63 of a block, accumulator O_a; 1: keys 64-127, O_b
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // row within the CTA's tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_o_own = tmem + lane_base + 256u + (uint32_t)(wg * 128);
    float* epi = reinterpret_cast<float*>(smem + Ly::EPI_OFF + (uint32_t)warp * 4096u);
    float2* xch = reinterpret_cast<float2*>(smem + Ly::XCH_OFF);
    int nu = 0, cnt = 0, uses = 0;
    bool ok = true;
    while (ok) {
      const int u = take_unit(nu++, ROLE_SOFTMAX, true);
      if (u == -2) {
        ok = false;
        break;
      }
      if (u < 0) break;
      const Unit x = decode(u, prm);
      if (!x.ok) break;
      const int p = x.it.p;
      const int a_t = x.a0 + (int)rank;  // this CTA's query tile
      const int32_t* kvl = prm.kv_list + x.it.kv_off;
      float m_used = -INFINITY, l_sum = 0.f;
      bool first_block = true;
      for (int ki = 0; ki < x.it.n_kv && ok; ++ki) {
        const int k = __ldg(kvl + ki);
        const bool diag = prm.causal && k == p;
        const int nbk = blocks_of(k, p, prm.causal, x.nb, x.a_max);
        for (int jb = 0; jb < nbk; ++jb, ++cnt) {
          const int buf = cnt & 1;
          ok = mbar_wait(bar(Ly::B_SFULL + buf), (uint32_t)((cnt >> 1) & 1), prm.wait_limit_ns, abort_flag,
                         prm.status, ROLE_SOFTMAX, u);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tm_s = tmem + lane_base + (uint32_t)(buf * 128 + wg * HALF);
          // visible keys of this row in the block, as columns 0..lim of the block: causal
          // diagonal block (key column > query row) and keys past the partition end
          const int kv_valid = (int)min((int64_t)BN, L - (int64_t)jb * BN);
          int lim = BN - 1;
          if (diag) lim = (jb < a_t) ? BN - 1 : (jb == a_t ? row : -1);
          lim = min(lim, kv_valid - 1) - wg * HALF;  // in this warpgroup's 64 columns
          // Exponentials against the running reference m_used (never decreasing); the half-row
          // block is accepted without a max pass when its sum is at most SUM_ACCEPT.  The first
          // block, or a block whose sum is too large or not finite, takes the maximum first and
          // raises m_used (rescaling O and l) when it grew by more than 2^LOG2_RESCALE.
          bool need_max = __any_sync(0xffffffffu, m_used == -INFINITY);
          float factor = 1.f, blk = 0.f;
          uint32_t pk[HALF / 2];
#pragma unroll 1
          for (int pass = 0;; ++pass) {
            float s[HALF];
            tmem_ld32(tm_s, s);
            tmem_ld32(tm_s + 32u, s + 32);
            tc_wait_ld();
            if (lim < HALF - 1) {
#pragma unroll
              for (int c = 0; c < HALF; ++c)
                if (c > lim) s[c] = -INFINITY;
            }
            if (need_max) {
              float mc[2];
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                float v = max3f(s[32 * q], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
                for (int i = 3; i + 1 < 32; i += 2) v = max3f(v, s[32 * q + i], s[32 * q + i + 1]);
                mc[q] = fmaxf(v, s[32 * q + 31]);
              }
              const float m_new = fmaxf(mc[0], mc[1]) * prm.scale_log2;
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
            const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2);
            const uint64_t nm2 = f2_pack(-mref, -mref);
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int c = 0; c < HALF / 2; ++c) {
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
            // O_own must hold every earlier PV product of this warpgroup before it is rescaled:
            // wait for the previous block's product (the first block of a unit never rescales).
            // S(j) completed, so PV(j-2) has, and the barrier is at most one phase behind.
            if (!first_block) {
              ok = mbar_wait(bar(Ly::B_PVDONE + wg), (uint32_t)((cnt - 1) & 1), prm.wait_limit_ns, abort_flag,
                             prm.status, ROLE_SOFTMAX, u);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
              tc_fence_after();
            }
            l_sum *= factor;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              float o[32];
              tmem_ld32(tm_o_own + (uint32_t)c, o);
              tc_wait_ld();
              uint32_t w[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(o[e] * factor);
              tmem_st32(tm_o_own + (uint32_t)c, w);
            }
          }
          l_sum += blk;
          first_block = false;
          tmem_st32(tm_s, pk);  // P of these 64 keys, bf16, into the first 32 columns of the half
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          // "P ready" barriers per S buffer: a warpgroup may finish block j + 1 before the issuer
          // has seen block j complete, but not block j + 2 (S(j + 2) follows PV(j))
          if (lane == 0) mbar_arrive_cluster(bar0(Ly::B_PFULL + 2 * wg + buf));
        }
      }
      if (!ok) break;
      // ---- epilogue: merge the two warpgroups' halves of each row, store O_t and lse_t
      ok = mbar_wait(bar(Ly::B_OFINAL), (uint32_t)(uses & 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_SOFTMAX, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float2* xs = xch + (uses & 1) * 2 * BM;
      xs[wg * BM + row] = make_float2(m_used, l_sum);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_XCH));
      ok = mbar_wait(bar(Ly::B_XCH), (uint32_t)(uses & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_SOFTMAX,
                     u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const float2 ma = xs[row], mb = xs[BM + row];
      const float m = fmaxf(ma.x, mb.x);
      const float wa = (ma.x == -INFINITY) ? 0.f : fast_exp2(ma.x - m);
      const float wb = (mb.x == -INFINITY) ? 0.f : fast_exp2(mb.x - m);
      const float l = wa * ma.y + wb * mb.y;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // this warpgroup finishes columns [64 wg, 64 wg + 64) of both accumulators:
      // o = (wa O_a + wb O_b) / l, taking O_b in two 32-column pieces to bound registers
      const float ca = wa * inv, cb = wb * inv;
      float o[HALF];
      const uint32_t tm_oa = tmem + lane_base + 256u + (uint32_t)(wg * HALF);
      const uint32_t tm_ob = tm_oa + 128u;
      tmem_ld32(tm_oa, o);
      tmem_ld32(tm_oa + 32u, o + 32);
      tc_wait_ld();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float ob[32];
        tmem_ld32(tm_ob + (uint32_t)(32 * hh), ob);
        tc_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) o[32 * hh + c] = o[32 * hh + c] * ca + ob[c] * cb;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar0(Ly::B_OFREE));  // the next unit's PV may start
      ++uses;
      const bool mine = a_t < x.a0 + x.ntiles;  // the odd CTA of a one-tile unit stores nothing
      const int64_t row_local = (int64_t)a_t * BM + row;
      const int64_t prow = (((int64_t)x.b * prm.Hq + x.h) * prm.n_slots + x.it.slot) * L + row_local;
      const int64_t wrow0 = row_local - lane;
      float* dst0 = prm.part_o + (prow - lane) * D + wg * HALF;
      if (mine) {
#pragma unroll
        for (int c = 0; c < HALF; c += 32) {
          // 32 rows x 32 columns: 16-byte chunks swizzled by row, read back 4 rows per store
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(epi + lane * 32 + ((q ^ (lane & 7)) * 4)) =
                make_float4(o[c + 4 * q], o[c + 4 * q + 1], o[c + 4 * q + 2], o[c + 4 * q + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = i * 4 + (lane >> 3), qq = lane & 7;
            const float4 v = *reinterpret_cast<const float4*>(epi + r * 32 + ((qq ^ (r & 7)) * 4));
            if (wrow0 + r < L) *reinterpret_cast<float4*>(dst0 + (int64_t)r * D + c + qq * 4) = v;
          }
          __syncwarp();
        }
        if (wg == 0 && row_local < L)
          prm.part_lse[prow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
    if (!ok) abort_pair();
  } else {
    regs_dec<OTHER_REGS>();
    if (warp == WARP_MMA && even) {
      // ================================================================ MMA issuer (even CTA)
      constexpr uint32_t idesc_qk = idesc_bf16_f32(2 * BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(2 * BM, D, true);
      // Base descriptors are built once; per instruction only the start-address field (address
      // / 16) advances by a compile-time offset (shared addresses stay below 256 KB, so it never
      // carries out of the field).
      const uint64_t q_desc0 = smem_desc_sw128(sb + Ly::Q_OFF, 16u, 1024u);
      const uint64_t k_desc0 = smem_desc_sw128(sb + Ly::K_OFF, 16u, 1024u);
      const uint64_t v_desc0 = smem_desc_sw128(sb + Ly::V_OFF, Ly::V_STAGE, 1024u);
      constexpr uint64_t QBOX16 = Ly::QBOX >> 4, KBOX16 = Ly::KBOX >> 4, KST16 = Ly::K_STAGE >> 4,
                         VST16 = Ly::V_STAGE >> 4;
      // K-major operands (Q, K): K-step kk of 16 elements sits in 64-column box kk/4 at byte 32 (kk%4)
      // MN-major V: K-step kk covers keys 16kk .. 16kk+15, 2048 bytes further each
      auto issue_s = [&](int G) -> bool {
        const int st = G % NSTK;
        bool ok = mbar_wait_cl_warp(bar(Ly::B_KFULL + st), (uint32_t)((G / NSTK) & 1), prm.wait_limit_ns, abort_flag,
                                    prm.status, ROLE_MMA, G);
        if (!ok) return false;
        tc_fence_after();
        const uint64_t kd = k_desc0 + (uint64_t)st * KST16;
        const uint32_t d_tm = tmem + (uint32_t)((G & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc2_mma_ss_warp(d_tm, q_desc0 + (uint64_t)((kk >> 2) * QBOX16 + (kk & 3) * 2),
                          kd + (uint64_t)((kk >> 2) * KBOX16 + (kk & 3) * 2), idesc_qk, kk > 0);
        tc2_commit_mc_warp(bar(Ly::B_SFULL + (G & 1)), PAIR);
        tc2_commit_mc_warp(bar(Ly::B_KEMPTY + st), PAIR);
        return true;
      };
      int nu = 0, nblk = 0, uses = 0;
      bool ok = true;
      while (ok) {
        const int u = take_unit(nu, ROLE_MMA, true);
        const int uidx = nu++;
        if (u == -2) {
          ok = false;
          break;
        }
        if (u < 0) break;
        const Unit x = decode(u, prm);
        if (!x.ok) break;
        const int32_t* kvl = prm.kv_list + x.it.kv_off;
        int NB = 0;
        for (int ki = 0; ki < x.it.n_kv; ++ki) NB += blocks_of(__ldg(kvl + ki), x.it.p, prm.causal, x.nb, x.a_max);
        ok = mbar_wait_cl_warp(bar(Ly::B_QFULL), (uint32_t)(uidx & 1), prm.wait_limit_ns, abort_flag, prm.status,
                               ROLE_MMA, u);
        if (ok) ok = issue_s(nblk);
        if (ok && NB > 1) ok = issue_s(nblk + 1);
        if (!ok) break;
        if (NB <= 2) tc2_commit_mc_warp(bar(Ly::B_QEMPTY), PAIR);  // the unit's last S products are issued
        for (int j = 0; j < NB && ok; ++j) {
          const int G = nblk + j;
          const int sv = G % NSTV;
          ok = mbar_wait_cl_warp(bar(Ly::B_VFULL + sv), (uint32_t)((G / NSTV) & 1), prm.wait_limit_ns, abort_flag,
                                 prm.status, ROLE_MMA, u);
          for (int w = 0; w < 2 && ok; ++w) {
            ok = mbar_wait_cl_warp(bar(Ly::B_PFULL + 2 * w + (G & 1)), (uint32_t)((G >> 1) & 1), prm.wait_limit_ns,
                                   abort_flag, prm.status, ROLE_MMA, u);
            if (ok && j == 0 && w == 0 && uses > 0)  // both CTAs' epilogues have copied O_a, O_b out
              ok = mbar_wait_cl_warp(bar(Ly::B_OFREE), (uint32_t)((uses - 1) & 1), prm.wait_limit_ns, abort_flag,
                                     prm.status, ROLE_MMA, u);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tm_p = tmem + (uint32_t)((G & 1) * 128 + w * HALF);
            const uint32_t tm_o = tmem + 256u + (uint32_t)(w * 128);
            const uint64_t vd = v_desc0 + (uint64_t)sv * VST16;
#pragma unroll
            for (int kk = 0; kk < HALF / 16; ++kk)
              tc2_mma_ts_warp(tm_o, tm_p + (uint32_t)(kk * 8), vd + (uint64_t)((w * 4 + kk) * (2048 >> 4)), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
            tc2_commit_mc_warp(bar(Ly::B_PVDONE + w), PAIR);
          }
          if (!ok) break;
          tc2_commit_mc_warp(bar(Ly::B_VEMPTY + sv), PAIR);
          if (j + 1 == NB) {
            tc2_commit_mc_warp(bar(Ly::B_OFINAL), PAIR);  // the unit's epilogues may start
            ++uses;
          }
          if (j + 2 < NB) {
            ok = issue_s(G + 2);  // into the buffer PV(j) has just read (products run in issue order)
            if (!ok) break;
            if (j + 3 == NB) tc2_commit_mc_warp(bar(Ly::B_QEMPTY), PAIR);
          }
        }
        if (!ok) break;
        nblk += NB;
      }
      if (!ok) abort_pair();
      // exit-path drain: every product issued completes before TMEM is freed
      tc2_commit_mc_warp(bar(Ly::B_DRAIN), 0x1);
      mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
    } else if (warp == WARP_MMA) {
      // ================================================================ relay (odd CTA)
      // In the order the issuer consumes them (Q, K(0), K(1), then V(j), K(j+2) per block),
      // wait for this CTA's loads to land and arrive on the even CTA's "full" barriers.
      int nu = 0, nq = 0, nk = 0, nv = 0;
      bool ok = true;
      auto relay = [&](int b_full, int idx, int nst) -> bool {
        const bool r = mbar_wait_warp(bar(b_full + idx % nst), (uint32_t)((idx / nst) & 1), prm.wait_limit_ns,
                                      abort_flag, prm.status, ROLE_RELAY, idx);
        if (r && lane == 0) mbar_arrive_cluster(bar0(b_full + idx % nst));
        __syncwarp();
        return r;
      };
      while (ok) {
        const int u = take_unit(nu++, ROLE_RELAY, true);
        if (u == -2) {
          ok = false;
          break;
        }
        if (u < 0) break;
        const Unit x = decode(u, prm);
        if (!x.ok) break;
        const int32_t* kvl = prm.kv_list + x.it.kv_off;
        int NB = 0;
        for (int ki = 0; ki < x.it.n_kv; ++ki) NB += blocks_of(__ldg(kvl + ki), x.it.p, prm.causal, x.nb, x.a_max);
        ok = mbar_wait_warp(bar(Ly::B_QFULL), (uint32_t)(nq & 1), prm.wait_limit_ns, abort_flag, prm.status,
                            ROLE_RELAY, u);
        if (!ok) break;
        if (lane == 0) mbar_arrive_cluster(bar0(Ly::B_QFULL));
        __syncwarp();
        ++nq;
        ok = relay(Ly::B_KFULL, nk++, NSTK);
        if (ok && NB > 1) ok = relay(Ly::B_KFULL, nk++, NSTK);
        for (int j = 0; j < NB && ok; ++j) {
          ok = relay(Ly::B_VFULL, nv++, NSTV);
          if (ok && j + 2 < NB) ok = relay(Ly::B_KFULL, nk++, NSTK);
        }
      }
      if (!ok) abort_pair();
    } else if (warp == WARP_LOAD && lane == 0) {
      // ================================================================ producer
      int nu = 0, nq = 0, nk = 0, nv = 0;
      bool ok = *abort_flag == 0;
      const uint32_t peer_ring = mapa_shared(sb + Ly::MISC_OFF + 8, 1u);
      // even CTA: take the next unit from the global counter and publish it to both CTAs' rings
      auto publish = [&]() -> int {
        const int slot = nu & 1;
        ok = mbar_wait_cl(bar(Ly::B_UEMPTY + slot), (uint32_t)(((nu >> 1) & 1) ^ 1), prm.wait_limit_ns, abort_flag,
                          prm.status, ROLE_LOAD, -1);
        if (!ok) return -1;
        int v = (int)atomicAdd(prm.counter, 1u);
        if (v >= prm.n_units) v = -1;
        unit_ring[slot] = v;
        st_shared_cluster(peer_ring + 4u * (uint32_t)slot, (uint32_t)v);
        mbar_arrive(bar(Ly::B_UFULL + slot));
        mbar_arrive_cluster(mapa_shared(bar(Ly::B_UFULL + slot), 1u));
        ++nu;
        return v;
      };
      // odd CTA: read the next unit from its ring
      auto next_odd = [&]() -> int {
        const int slot = nu & 1;
        ok = mbar_wait_cl(bar(Ly::B_UFULL + slot), (uint32_t)((nu >> 1) & 1), prm.wait_limit_ns, abort_flag,
                          prm.status, ROLE_LOAD, -1);
        if (!ok) return -1;
        const int v = unit_ring[slot];
        mbar_arrive_cluster(bar0(Ly::B_UEMPTY + slot));
        ++nu;
        return v;
      };
      auto load_k = [&](int64_t krow) -> bool {
        const int st = nk % NSTK;
        ok = mbar_wait(bar(Ly::B_KEMPTY + st), (uint32_t)(((nk / NSTK) & 1) ^ 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, nk);
        if (!ok) return false;
        mbar_expect_tx(bar(Ly::B_KFULL + st), Ly::K_STAGE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::K_OFF + (uint32_t)st * Ly::K_STAGE + (uint32_t)c * Ly::KBOX, &tmK, c * 64,
                      (int32_t)(krow + (int64_t)rank * HALF), bar(Ly::B_KFULL + st));
        ++nk;
        return true;
      };
      auto load_v = [&](int64_t krow) -> bool {
        const int st = nv % NSTV;
        ok = mbar_wait(bar(Ly::B_VEMPTY + st), (uint32_t)(((nv / NSTV) & 1) ^ 1), prm.wait_limit_ns, abort_flag,
                       prm.status, ROLE_LOAD, nv);
        if (!ok) return false;
        mbar_expect_tx(bar(Ly::B_VFULL + st), Ly::V_STAGE);
        tma_load_2d(sb + Ly::V_OFF + (uint32_t)st * Ly::V_STAGE, &tmV, (int32_t)rank * HALF, (int32_t)krow,
                    bar(Ly::B_VFULL + st));
        ++nv;
        return true;
      };
      int u = ok ? (even ? publish() : next_odd()) : -1;
      while (ok && u >= 0) {
        const Unit x = decode(u, prm);
        if (!x.ok) {
          record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_ITEM, u);
          ok = false;
          break;
        }
        int un = -1;
        if (even) {
          // publish the following unit now and pull its Q tiles and first K/V block into L2, so
          // the unit boundary does not wait on DRAM
          un = publish();
          if (!ok) break;
          if (un >= 0) {
            const Unit xn = decode(un, prm);
            if (xn.ok) {
              const int64_t qn = ((int64_t)xn.b * prm.Hq + xn.h) * prm.S + (int64_t)xn.it.p * L + (int64_t)xn.a0 * BM;
              for (int t = 0; t < xn.ntiles; ++t)
                for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_2d(&tmQ, c * 64, (int32_t)(qn + (int64_t)t * BM));
              const int kn = __ldg(prm.kv_list + xn.it.kv_off);
              if (kn >= 0 && kn < prm.P) {
                const int64_t krn =
                    ((int64_t)xn.b * prm.Hkv + xn.h / (prm.Hq / prm.Hkv)) * prm.S + (int64_t)kn * L;
                for (int c = 0; c < D / 64; ++c) {
                  tma_prefetch_l2_2d(&tmK, c * 64, (int32_t)krn);
                  tma_prefetch_l2_2d(&tmK, c * 64, (int32_t)(krn + HALF));
                  tma_prefetch_l2_2d(&tmV, c * 64, (int32_t)krn);
                }
              }
            }
          }
        }
        // the CTA's Q tile: the previous unit's last S products must be done with the buffer
        ok = mbar_wait(bar(Ly::B_QEMPTY), (uint32_t)((nq & 1) ^ 1), prm.wait_limit_ns, abort_flag, prm.status,
                       ROLE_LOAD, u);
        if (!ok) break;
        const int64_t qrow = ((int64_t)x.b * prm.Hq + x.h) * prm.S + (int64_t)x.it.p * L +
                             (int64_t)(x.a0 + (int)rank) * BM;
        mbar_expect_tx(bar(Ly::B_QFULL), Ly::Q_BYTES);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::Q_OFF + (uint32_t)c * Ly::QBOX, &tmQ, c * 64, (int32_t)qrow, bar(Ly::B_QFULL));
        ++nq;
        // block rows in visiting order
        const int hk = x.h / (prm.Hq / prm.Hkv);
        const int64_t kvbase = ((int64_t)x.b * prm.Hkv + hk) * prm.S;
        const int32_t* kvl = prm.kv_list + x.it.kv_off;
        int NB = 0;
        for (int ki = 0; ki < x.it.n_kv; ++ki) {
          const int k = __ldg(kvl + ki);
          if (k < 0 || k >= prm.P) {
            record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, u);
            ok = false;
            break;
          }
          NB += blocks_of(k, x.it.p, prm.causal, x.nb, x.a_max);
        }
        if (!ok) break;
        // loads in the order the issuer consumes them: K(0), K(1), then V(j), K(j+2)
        int kcur = 0, jk = 0;  // K cursor: KV list index and block within it
        int vcur = 0, jv = 0;  // V cursor
        auto next_row = [&](int& ci, int& jb) -> int64_t {
          const int k = __ldg(kvl + ci);
          const int64_t r = kvbase + (int64_t)k * L + (int64_t)jb * BN;
          if (++jb == blocks_of(k, x.it.p, prm.causal, x.nb, x.a_max)) {
            jb = 0;
            ++ci;
          }
          return r;
        };
        ok = load_k(next_row(kcur, jk));
        if (ok && NB > 1) ok = load_k(next_row(kcur, jk));
        for (int j = 0; j < NB && ok; ++j) {
          ok = load_v(next_row(vcur, jv));
          if (ok && j + 2 < NB) ok = load_k(next_row(kcur, jk));
        }
        if (!ok) break;
        u = even ? un : next_odd();
      }
      if (!ok) abort_pair();
      // exit-path drain: every load issued lands before the CTA exits
      if (nq > 0) mbar_drain(bar(Ly::B_QFULL), (uint32_t)((nq - 1) & 1), DRAIN_NS);
      for (int jj = (nk > NSTK ? nk - NSTK : 0); jj < nk; ++jj)
        mbar_drain(bar(Ly::B_KFULL + jj % NSTK), (uint32_t)((jj / NSTK) & 1), DRAIN_NS);
      for (int jj = (nv > NSTV ? nv - NSTV : 0); jj < nv; ++jj)
        mbar_drain(bar(Ly::B_VFULL + jj % NSTV), (uint32_t)((jj / NSTV) & 1), DRAIN_NS);
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // no product, load or remote arrival of either CTA is still in flight
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
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

// [rows, 128] bf16 row-major tensor, boxes of box_rows rows x 64 columns with 128-byte swizzle.
static bool make_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows,
                     std::string* err) {
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, box_rows};
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
  if (!make_map(enc, &mq, a.Q, (uint64_t)a.B * a.Hq * a.S, BM, err) ||
      !make_map(enc, &mk, a.K, (uint64_t)a.B * a.Hkv * a.S, HALF, err) ||
      !make_map(enc, &mv, a.V, (uint64_t)a.B * a.Hkv * a.S, BN, err))
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
  auto kern = tile_fwd_tc2_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout::ALLOC);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  // persistent: as many CTA pairs as can be resident at once, at most one per unit
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Layout::ALLOC;
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters[64] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *err = std::string("device query: ") + cudaGetErrorString(e);
    return (int)e;
  }
  if (dev < 0 || dev >= 64) {
    *err = "device index out of range";
    return (int)cudaErrorInvalidDevice;
  }
  if (max_clusters[dev] == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3((unsigned)(sms & ~1));
    int n = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess || n <= 0) {
      *err = std::string("cluster occupancy query: ") + (e != cudaSuccess ? cudaGetErrorString(e) : "no cluster fits");
      return (int)(e != cudaSuccess ? e : cudaErrorInvalidConfiguration);
    }
    max_clusters[dev] = n;
  }
  const int64_t clusters = units < max_clusters[dev] ? units : max_clusters[dev];
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, prm);
  if (e != cudaSuccess) *err = std::string("tile_fwd_tc2 launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace tc2

int launch_tile_fwd_tc2(const TileArgs& a, void* stream, std::string* err) {
  if (a.d != 128) {
    *err = "the SM-pair tile kernel supports d = 128";
    return (int)cudaErrorInvalidValue;
  }
  return tc2::launch(a, stream, err);
}

}  // namespace mesh
