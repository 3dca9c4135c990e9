// Tile attention forward for fp32 inputs on the 5th-generation tensor cores (sm_103a), with fp32
// accuracy: every fp32 operand x is split exactly into three bf16 pieces x = x1 + x2 + x3
// (8 + 8 + 8 significant bits), and a product sums the six piece products whose order is at
// least 2^-16 of the whole,
//   x1 y1 + x1 y2 + x2 y1 + x1 y3 + x3 y1 + x2 y2,
// on bf16 tensor-core products with fp32 accumulation.  Q, K and V are split by rounding to
// nearest (x1 = bf16(x), x2 = bf16(x - x1), x3 = bf16(x - x1 - x2): |x2| <= 2^-8 |x|,
// |x3| <= 2^-16 |x|), so the terms left out of Q K^T are below 2^-23 of |q||k|.  The
// probabilities P are split in the softmax by truncation, which takes integer masks and byte
// permutes instead of conversions (|p2| < 2^-7 p, |p3| < 2^-15 p), so the terms left out of
// P V are below 2^-22 of p |v|.  Six bf16 products cost what three tf32 products cost.
//
// Same work decomposition and outputs as the bf16 kernel (Mesh-Attention tiles and partial
// outputs: "Mesh-Attention: A New Communication-Efficient Distributed Attention with Improved
// Data Locality", tutorial §"Mesh-Attention：从一维'环'到二维'网'"; online m_i / l_i softmax of
// "环形注意力：突破长序列处理瓶颈的分布式计算范式", §"数值稳定性：Log-Sum-Exp技术的分布式应用").
//   split_kernel: Q, K and V into their bf16 pieces, [3][rows][d] each, in the caller's
//                 workspace (HBM-bound, one pass).
//   tile_fwd_tc32_kernel: one CTA per (work item, batch, head, 128-row query tile); 10 warps --
//     warps 0-7 softmax (two per TMEM lane quadrant: one thread per row, each warp 32 of a
//     block's 64 keys, the pair swapping half-row maxima through shared memory and a bounded
//     mbarrier), warp 8 MMA issuer (elected lane of a converged warp), warp 9 TMA producer.
//     Q's first two pieces sit in TMEM, written there by the softmax warps at the start of the
//     unit, and are the A operand of five of the six S products, which then read only K from
//     shared memory; shared memory holds Q's third piece and two stages each of K's and V's
//     three pieces (32 + 96 + 96 KB at d = 128), 64 keys a block.  TMEM: S of even blocks (64
//     columns) | S of odd blocks (64) | P (three packed bf16 pieces, 96) | O (d) | Q1, Q2 (d / 2
//     each, packed pairs).  Issue order S(0), S(1), then per block PV(j), S(j+2): with S
//     double-buffered and P in its own columns, the S products of the next block run while the
//     softmax works on this one.  The softmax stores P(j) once PV(j-1) has completed.  It takes
//     the block maximum every block but raises its reference (and rescales O and l) only when the
//     maximum grew by more than 2^8; the exact three-piece split keeps P's full fp32 value at any
//     magnitude up to that bound.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace mesh {
namespace tc32 {

constexpr int BM = 128;  // query rows per tile = TMEM lanes
constexpr int BN = 64;   // keys per block
constexpr int NUM_THREADS = 320;
constexpr int N_SOFTMAX_WARPS = 8;  // two per TMEM lane quadrant, 32 of a block's 64 keys each
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
constexpr int NPAIR = 6;
constexpr int64_t DRAIN_NS = 200000000;
constexpr int ROLE_SOFTMAX = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_ITEM = 4;

// piece pairs (a, b) of a product, x_a y_b, smallest first: (1,1), (2,0), (0,2), (1,0), (0,1),
// (0,0).  S starts from a zero accumulator every block, so its terms of order 2^-16 and 2^-8 are
// summed at their own magnitude before the leading term is added, instead of each being rounded
// to the leading term's precision.
__device__ __forceinline__ int pair_a(int i) { return i == 0 ? 1 : i == 1 ? 2 : i == 3 ? 1 : 0; }
__device__ __forceinline__ int pair_b(int i) { return i == 0 ? 1 : i == 2 ? 2 : i == 4 ? 1 : 0; }

struct Params {
  const DevItem* items;
  const int32_t* kv_list;
  float* part_o;
  float* part_lse;
  int32_t* status;
  int64_t S, L;
  int64_t q_rows, kv_rows;  // rows of one piece: B*Hq*S and B*Hkv*S
  const uint32_t* q_pieces;  // Q's bf16 pieces [3][q_rows][D], as packed pairs
  int32_t B, Hq, Hkv, P, n_items, n_slots, nqt, nb, causal;
  float scale_log2;
  int64_t wait_limit_ns;
};

// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp writes lane (base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int D>
struct Layout {
  static constexpr uint32_t QP = BM * D * 2;    // one piece of the Q tile
  static constexpr uint32_t KP = BN * D * 2;    // one piece of a K or V block
  static constexpr uint32_t QBOX = BM * 128;    // 128 rows x 64 bf16 columns
  static constexpr uint32_t KBOX = BN * 128;    // 64 rows x 64 bf16 columns
  // Q's third piece (the first two live in TMEM), two K stages, two V stages
  static constexpr uint32_t KSTAGE = 3 * KP;
  static constexpr uint32_t Q_OFF = 0, K_OFF = QP, V_OFF = K_OFF + 2 * KSTAGE;
  static constexpr uint32_t BAR_OFF = V_OFF + 2 * KSTAGE;
  static constexpr int B_QFULL = 0, B_KFULL = 1, B_KEMPTY = 3, B_VFULL = 5, B_VEMPTY = 7, B_SFULL = 9, B_PFULL = 11,
                       B_OFULL = 12, B_DRAIN = 13, B_PVDONE = 14, B_QTMEM = 15, B_XCH = 16, NBARS = 20;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBARS * 8;
  // the two softmax warps of a lane quadrant swap their half-row maxima (and at the end their
  // sums) here: [quadrant 4][phase parity 2][half 2][32 rows] floats
  static constexpr uint32_t XCH_OFF = MISC_OFF + 16;
  static constexpr uint32_t TOTAL = XCH_OFF + 4 * 2 * 2 * 32 * 4;
};

// 64-key blocks of KV partition k seen by query tile qt of partition p: on the causal diagonal
// partition only the blocks up to the tile's last row.
__device__ __forceinline__ int kblocks(int k, int p, int causal, int nb, int qt) {
  return (causal && k == p) ? min(nb, 2 * qt + 2) : nb;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tile_fwd_tc32_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params prm) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = smem_u32(smem_raw);
  if (sb & 1023u) {  // 128-byte swizzle atoms need 1024-aligned operands; no room to align by hand
    if (threadIdx.x == 0) record_error(prm.status, MESH_ATTN_ERR_INTERNAL, ROLE_ITEM, (int32_t)blockIdx.x);
    return;
  }
  uint8_t* smem = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + Ly::BAR_OFF + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 4);
  const int64_t L = prm.L;

  // Units are numbered KV-head-major: (batch, KV head, work item in launch order, query head of
  // the group, query tile), so the CTAs resident together share one KV head's partitions in L2.
  int64_t uu = blockIdx.x;
  const int g = prm.Hq / prm.Hkv;
  const int qt = (int)(uu % prm.nqt); uu /= prm.nqt;
  const int gi = (int)(uu % g); uu /= g;
  const int idx = (int)(uu % prm.n_items); uu /= prm.n_items;
  const int h = (int)(uu % prm.Hkv) * g + gi;
  const int b = (int)(uu / prm.Hkv);
  const DevItem it = prm.items[idx];
  const bool unit_ok = it.p >= 0 && it.p < prm.P && it.slot >= 0 && it.slot < prm.n_slots && it.n_kv >= 1 &&
                       it.kv_off >= 0;
  const int p = it.p;
  const int hk = h / g;
  int NB = 0;
  if (unit_ok)
    for (int ki = 0; ki < it.n_kv; ++ki) NB += kblocks(__ldg(prm.kv_list + it.kv_off + ki), p, prm.causal, prm.nb, qt);
  auto block_at = [&](int j, int& kp, int& kbk) {
    int r = j;
    for (int ki = 0; ki < it.n_kv; ++ki) {
      kp = __ldg(prm.kv_list + it.kv_off + ki);
      const int n = kblocks(kp, p, prm.causal, prm.nb, qt);
      if (r < n) {
        kbk = r;
        return;
      }
      r -= n;
    }
    kp = -1;
    kbk = 0;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_QFULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ly::B_KFULL + s), 1);
      mbar_init(bar(Ly::B_KEMPTY + s), 1);
    }
    mbar_init(bar(Ly::B_QTMEM), N_SOFTMAX_WARPS);  // one lane of each softmax warp
    for (int q = 0; q < 4; ++q) mbar_init(bar(Ly::B_XCH + q), 2);  // the quadrant's two warps
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ly::B_VFULL + s), 1);
      mbar_init(bar(Ly::B_VEMPTY + s), 1);
    }
    mbar_init(bar(Ly::B_SFULL), 1);  // one per S buffer
    mbar_init(bar(Ly::B_SFULL + 1), 1);
    mbar_init(bar(Ly::B_PFULL), N_SOFTMAX_WARPS);  // one lane of each softmax warp
    mbar_init(bar(Ly::B_OFULL), 1);
    mbar_init(bar(Ly::B_DRAIN), 1);
    mbar_init(bar(Ly::B_PVDONE), 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = *abort_flag == 0;
  // TMEM columns: S of block j in [64 (j % 2), + 64); P [128, 224) as three packed bf16 pieces of
  // 32 columns; O [256, 256 + D); Q's first and second pieces [256 + D, + D / 2) each, packed (the
  // A operand of the S products that take them)
  constexpr uint32_t COL_P = 128, COL_O = 256, COL_Q = COL_O + D, QW = D / 2;
  constexpr float LOG2_RESCALE = 8.0f;

  if (warp < N_SOFTMAX_WARPS) {
    // ================================================================ softmax
    // Warp w owns TMEM lane quadrant w % 4 (rows 32 (w % 4) ..) and half w / 4 of each block's 64
    // keys (and of O's columns).  The two warps of a quadrant swap their half-row maxima every
    // block, so they take the same reference m and the same rescale decisions; each keeps the
    // sum of its half, added together at the end.
    const int q4 = warp & 3, hf = warp >> 2;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t tm_s = tmem + lane_base + 32u * (uint32_t)hf;
    const uint32_t tm_o = tmem + lane_base + COL_O + (uint32_t)(hf * (D / 2));
    volatile float* xch = reinterpret_cast<volatile float*>(smem + Ly::XCH_OFF) + q4 * 128;
    const uint32_t xbar = bar(Ly::B_XCH + q4);
    const int64_t q_local = (int64_t)qt * BM + row;
    float m = -INFINITY, l = 0.f;
    bool ok = run;
    if (ok) {
      // Q piece hf of this row into TMEM (lane = row): rows past the tensor read as zero
      const int64_t grow = ((int64_t)b * prm.Hq + h) * prm.S + (int64_t)p * L + q_local;
      uint32_t w[QW];
      if (grow < prm.q_rows) {
        const uint4* src = reinterpret_cast<const uint4*>(prm.q_pieces + ((int64_t)hf * prm.q_rows + grow) * QW);
#pragma unroll
        for (int i = 0; i < QW / 4; ++i) {
          const uint4 v = __ldg(src + i);
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < QW; ++i) w[i] = 0u;
      }
#pragma unroll
      for (int c = 0; c < QW; c += 32) tmem_st32(tmem + lane_base + COL_Q + (uint32_t)(hf * QW + c), w + c);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_QTMEM));
    }
    for (int j = 0; j < NB && ok; ++j) {
      int kp, kbk;
      block_at(j, kp, kbk);
      // visible keys of this row in the block: [0, hi); this warp holds keys [32 hf, 32 hf + 32)
      int hi = (int)min((int64_t)BN, L - (int64_t)kbk * BN);
      if (prm.causal && kp == p) hi = (int)min((int64_t)hi, q_local - (int64_t)kbk * BN + 1);
      const int lim = hi - 32 * hf;
      ok = mbar_wait(bar(Ly::B_SFULL + (j & 1)), (uint32_t)((j >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                     ROLE_SOFTMAX, j);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float s[32];
      tmem_ld32(tm_s + 64u * (uint32_t)(j & 1), s);
      tc_wait_ld();
#pragma unroll
      for (int c = 0; c < 32; ++c) s[c] = (c < lim) ? s[c] * prm.scale_log2 : -INFINITY;
      float mc0 = max3f(s[0], s[1], s[2]), mc1 = max3f(s[16], s[17], s[18]);
#pragma unroll
      for (int c = 3; c + 1 < 16; c += 2) {
        mc0 = max3f(mc0, s[c], s[c + 1]);
        mc1 = max3f(mc1, s[16 + c], s[16 + c + 1]);
      }
      const float mh = max3f(mc0, mc1, fmaxf(s[15], s[31]));
      // swap half-row maxima with the quadrant's other warp (slot j % 2; the barrier cannot run a
      // phase ahead: the other warp's next arrival follows its wait on this phase, which needs
      // this warp's arrival)
      xch[(j & 1) * 64 + hf * 32 + lane] = mh;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      ok = mbar_wait(xbar, (uint32_t)(j & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_SOFTMAX, j);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const float mb = fmaxf(mh, xch[(j & 1) * 64 + (1 - hf) * 32 + lane]);
      // reference m: set by the first visible block, raised only when the maximum grows by more
      // than 2^LOG2_RESCALE (then O and l are rescaled); P = 2^(s - m) <= 2^LOG2_RESCALE
      float factor = 1.f;
      if (mb > -INFINITY) {
        if (m == -INFINITY) {
          m = mb;
        } else if (mb > m + LOG2_RESCALE) {
          factor = fast_exp2(m - mb);
          m = mb;
        }
      }
      const float mref = (m == -INFINITY) ? 0.f : m;
      // PV(j-1) done: O holds every earlier product and P's buffer is free (PV(j) needs this
      // block's P, so the barrier is never a phase ahead of this wait)
      bool pv_done = (j == 0);
      if (__any_sync(0xffffffffu, factor != 1.f)) {
        ok = mbar_wait(bar(Ly::B_PVDONE), (uint32_t)((j - 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                       ROLE_SOFTMAX, j);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        pv_done = true;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
          float o[32];
          tmem_ld32(tm_o + (uint32_t)c, o);
          tc_wait_ld();
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(o[e] * factor);
          tmem_st32(tm_o + (uint32_t)c, w);
        }
      }
      uint32_t p1[16], p2[16], p3[16];
      uint64_t acc2[2] = {0ull, 0ull};
      const uint64_t nm2 = f2_pack(-mref, -mref);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float x0, x1;
        f2_unpack(f2_add(f2_pack(s[c], s[c + 1]), nm2), x0, x1);
        const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
        acc2[(c >> 1) & 1] = f2_add(acc2[(c >> 1) & 1], f2_pack(e0, e1));
        // exact three-piece split of each probability by truncation: x1 = x with the low 16 bits
        // cleared (its top 8 significant bits), r = x - x1 (exact, at most 16 significant bits),
        // x2 = r truncated the same way, x3 = r - x2 (at most 8 significant bits, so a bf16); each
        // piece is the high half of an fp32 whose low half is zero
        const uint32_t u0 = __float_as_uint(e0), u1 = __float_as_uint(e1);
        const float r0 = e0 - __uint_as_float(u0 & 0xffff0000u), r1 = e1 - __uint_as_float(u1 & 0xffff0000u);
        const uint32_t w0 = __float_as_uint(r0), w1 = __float_as_uint(r1);
        const float t0 = r0 - __uint_as_float(w0 & 0xffff0000u), t1 = r1 - __uint_as_float(w1 & 0xffff0000u);
        p1[c / 2] = __byte_perm(u0, u1, 0x7632u);
        p2[c / 2] = __byte_perm(w0, w1, 0x7632u);
        p3[c / 2] = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x7632u);
      }
      float sa, sb2;
      f2_unpack(f2_add(acc2[0], acc2[1]), sa, sb2);
      l = l * factor + (sa + sb2);
      if (!pv_done) {
        ok = mbar_wait(bar(Ly::B_PVDONE), (uint32_t)((j - 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                       ROLE_SOFTMAX, j);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      // this warp's 32 keys are packed columns [16 hf, 16 hf + 16) of each piece
      const uint32_t tm_p = tmem + lane_base + COL_P + 16u * (uint32_t)hf;
      tmem_st16(tm_p, p1);
      tmem_st16(tm_p + 32u, p2);
      tmem_st16(tm_p + 64u, p3);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_PFULL));
    }
    if (ok) {
      // the row's sum: both halves, swapped through the next phase of the quadrant's barrier
      xch[(NB & 1) * 64 + hf * 32 + lane] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      ok = mbar_wait(xbar, (uint32_t)(NB & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_SOFTMAX, -1);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) l += xch[(NB & 1) * 64 + (1 - hf) * 32 + lane];
    }
    if (ok) {
      ok = mbar_wait(bar(Ly::B_OFULL), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_SOFTMAX, -1);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t prow = (((int64_t)b * prm.Hq + h) * prm.n_slots + it.slot) * L + q_local;
#pragma unroll 1
      for (int c = 0; c < D / 2; c += 32) {
        float o[32];
        tmem_ld32(tm_o + (uint32_t)c, o);
        tc_wait_ld();
        if (q_local < L) {
          float4* dst = reinterpret_cast<float4*>(prm.part_o + prow * D + hf * (D / 2) + c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
        }
      }
      if (q_local < L && hf == 0)
        prm.part_lse[prow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  } else if (warp == WARP_MMA) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
    const uint64_t q0 = smem_desc_sw128(sb + Ly::Q_OFF, 16u, 1024u);
    const uint64_t k0 = smem_desc_sw128(sb + Ly::K_OFF, 16u, 1024u);
    const uint64_t v0 = smem_desc_sw128(sb + Ly::V_OFF, Ly::KBOX, 1024u);
    // K-major operand made of 64-column SW128 boxes: K-step kk sits in box kk/4 at byte 32 (kk % 4)
    auto qoff = [](int kk) { return (uint64_t)((kk >> 2) * (Ly::QBOX >> 4) + (kk & 3) * 2); };
    auto koff = [](int kk) { return (uint64_t)((kk >> 2) * (Ly::KBOX >> 4) + (kk & 3) * 2); };
    bool ok = run && NB > 0;
    if (ok) ok = mbar_wait_warp(bar(Ly::B_QFULL), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, -1);
    if (ok) ok = mbar_wait_warp(bar(Ly::B_QTMEM), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, -1);
    // S(j) = Q K(j)^T over the six piece pairs into S buffer j % 2: Q's first two pieces from TMEM
    // (the products read only K from shared memory), its third from shared memory; K(j)'s stage
    // is free once they complete
    auto issue_s = [&](int j) -> bool {
      const int ks = j & 1;
      const uint32_t sd = tmem + 64u * (uint32_t)ks;
      if (!mbar_wait_warp(bar(Ly::B_KFULL + ks), (uint32_t)((j >> 1) & 1), prm.wait_limit_ns, abort_flag, prm.status,
                          ROLE_MMA, j))
        return false;
      tc_fence_after();
      for (int pr = 0; pr < NPAIR; ++pr) {
        const int pa = pair_a(pr);
        const uint64_t kd = k0 + (uint64_t)ks * (Ly::KSTAGE >> 4) + (uint64_t)pair_b(pr) * (Ly::KP >> 4);
        if (pa < 2) {
          const uint32_t qa = tmem + COL_Q + (uint32_t)(pa * QW);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ts_warp(sd, qa + (uint32_t)(kk * 8), kd + koff(kk), idesc_qk, (pr > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ss_warp(sd, q0 + qoff(kk), kd + koff(kk), idesc_qk, (pr > 0 || kk > 0) ? 1u : 0u);
        }
      }
      tc_commit_warp(bar(Ly::B_SFULL + ks));
      tc_commit_warp(bar(Ly::B_KEMPTY + ks));
      return true;
    };
    // Issue order S(0), S(1), then per block PV(j), S(j+2): S(j+1) is computed while the softmax
    // works on block j, and S(j+2) while it works on block j+1.
    if (ok) ok = issue_s(0);
    if (ok && NB > 1) ok = issue_s(1);
    for (int j = 0; j < NB && ok; ++j) {
      ok = mbar_wait_warp(bar(Ly::B_PFULL), (uint32_t)(j & 1), prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, j);
      if (ok)
        ok = mbar_wait_warp(bar(Ly::B_VFULL + (j & 1)), (uint32_t)((j >> 1) & 1), prm.wait_limit_ns, abort_flag,
                            prm.status, ROLE_MMA, j);
      if (!ok) break;
      tc_fence_after();
      // O += P V over the six piece pairs; P's pieces from TMEM, V's MN-major from shared memory
      const uint32_t pbuf = tmem + COL_P;
      for (int pr = 0; pr < NPAIR; ++pr) {
        const uint32_t pa = pbuf + 32u * (uint32_t)pair_a(pr);
        const uint64_t vd = v0 + (uint64_t)(j & 1) * (Ly::KSTAGE >> 4) + (uint64_t)pair_b(pr) * (Ly::KP >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc_mma_ts_warp(tmem + COL_O, pa + (uint32_t)(kk * 8), vd + (uint64_t)(kk * 128), idesc_pv,
                         (j > 0 || pr > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit_warp(bar(Ly::B_VEMPTY + (j & 1)));  // V(j)'s stage free once these products complete
      tc_commit_warp(bar(Ly::B_PVDONE));  // O holds PV(0..j) and P is free for block j+1
      // the softmax read S(j) before it wrote P(j), so S(j+2) may overwrite S buffer j % 2
      if (j + 2 < NB) ok = issue_s(j + 2);
    }
    if (ok) tc_commit_warp(bar(Ly::B_OFULL));
    tc_commit_warp(bar(Ly::B_DRAIN));
    mbar_drain(bar(Ly::B_DRAIN), 0u, DRAIN_NS);
  } else if (warp == WARP_LOAD && lane == 0) {
    // ================================================================ producer
    bool ok = run && NB > 0;
    int issued_k = 0, issued_v = 0;
    if (ok) {
      const int64_t qrow = ((int64_t)b * prm.Hq + h) * prm.S + (int64_t)p * L + (int64_t)qt * BM;
      mbar_expect_tx(bar(Ly::B_QFULL), Ly::QP);  // the third piece; the softmax warps put the others in TMEM
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sb + Ly::Q_OFF + (uint32_t)c * Ly::QBOX, &tmQ, c * 64, (int32_t)(qrow + 2 * prm.q_rows),
                    bar(Ly::B_QFULL));
    }
    const int64_t kvbase = ((int64_t)b * prm.Hkv + hk) * prm.S;
    // Two K stages and two V stages.  Products run S(0), S(1), PV(0), S(2), PV(1), S(3), ...; K(j)
    // takes the stage S(j-2) frees and V(j) the one PV(j-2) frees, so the loads follow the
    // products' completion order: K(0), K(1), V(0), V(1), K(2), then K(j), V(j-1) for j >= 3, then
    // the last V.
    auto load_pieces = [&](const CUtensorMap* tm, uint32_t off, int64_t krow, uint32_t fullbar) {
      mbar_expect_tx(fullbar, 3 * Ly::KP);
      for (int a = 0; a < 3; ++a)
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + off + (uint32_t)a * Ly::KP + (uint32_t)c * Ly::KBOX, tm, c * 64,
                      (int32_t)(krow + (int64_t)a * prm.kv_rows), fullbar);
    };
    auto row_of = [&](int j, int64_t& krow) -> bool {
      int kp, kbk;
      block_at(j, kp, kbk);
      if (kp < 0 || kp >= prm.P) {
        record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, (int32_t)blockIdx.x);
        *abort_flag = 1;
        return false;
      }
      krow = kvbase + (int64_t)kp * L + (int64_t)kbk * BN;
      return true;
    };
    auto load_k = [&](int j) -> bool {
      int64_t krow;
      if (!row_of(j, krow)) return false;
      const int ks = j & 1;
      if (j >= 2 && !mbar_wait(bar(Ly::B_KEMPTY + ks), (uint32_t)(((j - 2) >> 1) & 1), prm.wait_limit_ns, abort_flag,
                               prm.status, ROLE_LOAD, j))
        return false;
      load_pieces(&tmK, Ly::K_OFF + (uint32_t)ks * Ly::KSTAGE, krow, bar(Ly::B_KFULL + ks));
      ++issued_k;
      return true;
    };
    auto load_v = [&](int j) -> bool {
      int64_t krow;
      if (!row_of(j, krow)) return false;
      const int vs = j & 1;
      if (j >= 2 && !mbar_wait(bar(Ly::B_VEMPTY + vs), (uint32_t)(((j - 2) >> 1) & 1), prm.wait_limit_ns, abort_flag,
                               prm.status, ROLE_LOAD, j))
        return false;
      load_pieces(&tmV, Ly::V_OFF + (uint32_t)vs * Ly::KSTAGE, krow, bar(Ly::B_VFULL + vs));
      ++issued_v;
      return true;
    };
    if (ok) ok = load_k(0);
    if (ok && NB > 1) ok = load_k(1);
    if (ok) ok = load_v(0);
    if (ok && NB > 1) ok = load_v(1);
    if (ok && NB > 2) ok = load_k(2);
    for (int j = 3; j < NB && ok; ++j) {
      ok = load_k(j);
      if (ok) ok = load_v(j - 1);
    }
    if (ok && NB > 2) ok = load_v(NB - 1);
    if (run && NB > 0) mbar_drain(bar(Ly::B_QFULL), 0u, DRAIN_NS);
    for (int jj = (issued_k > 2 ? issued_k - 2 : 0); jj < issued_k; ++jj)
      mbar_drain(bar(Ly::B_KFULL + (jj & 1)), (uint32_t)((jj >> 1) & 1), DRAIN_NS);
    for (int jj = (issued_v > 2 ? issued_v - 2 : 0); jj < issued_v; ++jj)
      mbar_drain(bar(Ly::B_VFULL + (jj & 1)), (uint32_t)((jj >> 1) & 1), DRAIN_NS);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// fp32 rows -> three bf16 pieces [3][n][...] (x1 = bf16(x), x2 = bf16(x - x1), x3 = bf16(x - x1 - x2))
__global__ void __launch_bounds__(256) split_kernel(const float4* __restrict__ x, uint2* __restrict__ out,
                                                    int64_t n4, int32_t* status) {
  if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= n4) return;
  const float4 v = __ldcs(x + i);
  const float e[4] = {v.x, v.y, v.z, v.w};
  uint32_t w[3][2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(e[2 * h], e[2 * h + 1]);
    const float r0 = e[2 * h] - __low2float(a), r1 = e[2 * h + 1] - __high2float(a);
    const __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
    const __nv_bfloat162 c = __floats2bfloat162_rn(r0 - __low2float(b), r1 - __high2float(b));
    w[0][h] = *reinterpret_cast<const uint32_t*>(&a);
    w[1][h] = *reinterpret_cast<const uint32_t*>(&b);
    w[2][h] = *reinterpret_cast<const uint32_t*>(&c);
  }
#pragma unroll
  for (int a = 0; a < 3; ++a) out[(int64_t)a * n4 + i] = make_uint2(w[a][0], w[a][1]);
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

// [rows, d] bf16 row-major pieces, boxes of box_rows x 64 columns with 128-byte swizzle.
static bool make_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows,
                     std::string* err) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
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

static int split(const float* x, void* out, int64_t n, int32_t* status, cudaStream_t st, std::string* err) {
  const int64_t n4 = n / 4;
  if (n4 <= 0) return (int)cudaSuccess;
  const int64_t blocks = (n4 + 255) / 256;
  if (blocks > 0x7fffffff) {
    *err = "tensor too large to split in one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  split_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(x), static_cast<uint2*>(out), n4,
                                                 status);
  return (int)cudaGetLastError();
}

template <int D>
static int launch(const TileArgs& a, void* stream, std::string* err) {
  const int64_t nqt = (a.L + BM - 1) / BM;
  const int64_t nb = (a.L + BN - 1) / BN;
  const int64_t units = (int64_t)a.n_items * a.B * a.Hq * nqt;
  if (units <= 0) return (int)cudaSuccess;
  const int64_t q_rows = (int64_t)a.B * a.Hq * a.S, kv_rows = (int64_t)a.B * a.Hkv * a.S;
  if (units > 0x7fffffff || 3 * q_rows >= ((int64_t)1 << 31) || 3 * kv_rows >= ((int64_t)1 << 31)) {
    *err = "fp32 tensor-core path: too many rows or work units for one launch";
    return (int)cudaErrorInvalidConfiguration;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const F32Pieces pc = f32_pieces_layout(a.B, a.Hq, a.Hkv, a.S, a.d);
  char* base = static_cast<char*>(a.pieces);
  int ce = split(static_cast<const float*>(a.Q), base + pc.q_off, q_rows * D, a.status, st, err);
  if (ce == (int)cudaSuccess) ce = split(static_cast<const float*>(a.K), base + pc.k_off, kv_rows * D, a.status, st, err);
  if (ce == (int)cudaSuccess) ce = split(static_cast<const float*>(a.V), base + pc.v_off, kv_rows * D, a.status, st, err);
  if (ce != (int)cudaSuccess) {
    if (err->empty()) *err = std::string("split launch: ") + cudaGetErrorString((cudaError_t)ce);
    return ce;
  }
  EncodeTiledFn enc = get_encode(err);
  if (!enc) return (int)cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_map(enc, &mq, base + pc.q_off, (uint64_t)(3 * q_rows), D, BM, err) ||
      !make_map(enc, &mk, base + pc.k_off, (uint64_t)(3 * kv_rows), D, BN, err) ||
      !make_map(enc, &mv, base + pc.v_off, (uint64_t)(3 * kv_rows), D, BN, err))
    return (int)cudaErrorInvalidValue;
  Params prm;
  prm.items = a.items;
  prm.kv_list = a.kv_list;
  prm.part_o = a.part_o;
  prm.part_lse = a.part_lse;
  prm.status = a.status;
  prm.S = a.S;
  prm.L = a.L;
  prm.q_rows = q_rows;
  prm.kv_rows = kv_rows;
  prm.q_pieces = reinterpret_cast<const uint32_t*>(base + pc.q_off);
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.P = a.P;
  prm.n_items = a.n_items;
  prm.n_slots = a.n_slots;
  prm.nqt = (int32_t)nqt;
  prm.nb = (int32_t)nb;
  prm.causal = a.causal;
  prm.scale_log2 = a.scale_log2;
  prm.wait_limit_ns = a.wait_limit_ns;
  auto kern = tile_fwd_tc32_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<D>::TOTAL);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  kern<<<dim3((unsigned)units), dim3(NUM_THREADS), Layout<D>::TOTAL, st>>>(mq, mk, mv, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) *err = std::string("tile_fwd_tc32 launch: ") + cudaGetErrorString(e);
  return (int)e;
}

}  // namespace tc32

F32Pieces f32_pieces_layout(int32_t B, int32_t Hq, int32_t Hkv, int64_t S, int32_t d) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  F32Pieces p{};
  const size_t qb = (size_t)3 * B * Hq * (size_t)S * d * 2, kvb = (size_t)3 * B * Hkv * (size_t)S * d * 2;
  p.q_off = 0;
  p.k_off = up(qb);
  p.v_off = p.k_off + up(kvb);
  p.total = p.v_off + up(kvb);
  return p;
}

int launch_tile_fwd_tc32(const TileArgs& a, void* stream, std::string* err) {
  if (a.d == 128) return tc32::launch<128>(a, stream, err);
  if (a.d == 64) return tc32::launch<64>(a, stream, err);
  *err = "fp32 tensor-core tile kernel supports d = 64 or 128";
  return (int)cudaErrorInvalidValue;
}

}  // namespace mesh
