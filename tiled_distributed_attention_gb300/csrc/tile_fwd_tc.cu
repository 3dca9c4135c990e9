// Tile attention forward on the 5th-generation tensor cores (sm_103a): for one work unit
// (work item = (Q partition p, tile), batch b, query head h, pair of 128-row query tiles) it
// visits the item's KV partitions in planned order, 128 keys at a time, and writes the
// partial output O_t = acc / l and lse_t = m + ln l of each query row.
//
// The per-block recurrence is the online softmax (running max m_i and running sum l_i) that
// "环形注意力：突破长序列处理瓶颈的分布式计算范式" describes in §"数值稳定性：Log-Sum-Exp技术的分布式
// 应用"; the tile/partial structure is Mesh-Attention's ("Mesh-Attention: A New
// Communication-Efficient Distributed Attention with Improved Data Locality", tutorial
// §"Mesh-Attention：从一维'环'到二维'网'": each tile's partial results go back to the Q owner).
//
// GB300 mapping (one CTA of 10 warps per unit, 1 CTA per SM):
//   warp 9      TMA producer: Q tiles once, then K and V blocks through a 2-stage mbarrier ring
//               (128-byte swizzled boxes of 128 rows x 64 columns).
//   warp 8      MMA issuer (one thread): S_t = Q_t K^T and O_t += P_t V with tcgen05.mma,
//               accumulators in tensor memory (TMEM), completion signalled by tcgen05.commit.
//   warps 0-7   softmax, one warpgroup per query tile: thread i owns row i (TMEM lane i), so
//               row max and row sum are thread-local; P is written back to TMEM as bf16 in the
//               columns S occupied and feeds the PV product straight from TMEM.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, 128 columns each.  The two tiles interleave on
// the tensor pipe: while softmax 0 works on S_0(j), the pipe runs PV_1(j-1) and S_1(j).
// O is rescaled only when the running max grows by more than 2^8 (values stay below 256).
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
constexpr int NUM_THREADS = 320;
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
constexpr float LOG2_RESCALE = 8.0f;
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
  static constexpr uint32_t BAR_OFF = V_OFF + NST * TILE;
  // barrier indices
  static constexpr int B_QFULL = 0, B_KFULL = 1, B_KEMPTY = B_KFULL + NST, B_VFULL = B_KEMPTY + NST,
                       B_VEMPTY = B_VFULL + NST, B_SFULL = B_VEMPTY + NST, B_PFULL = B_SFULL + 2,
                       B_OFINAL = B_PFULL + 2, NBARS = B_OFINAL + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr uint32_t TOTAL = MISC_OFF + 16;
  static constexpr uint32_t ALLOC = TOTAL + 1024;
};

struct Params {
  const DevItem* items;
  const int32_t* kv_list;
  float* part_o;
  float* part_lse;
  int32_t* status;
  int64_t S, L;
  int32_t B, Hq, Hkv, P, n_items, n_slots, n_pairs, causal;
  float scale_log2;
  int64_t wait_limit_ns;
};

// Number of 128-key blocks of KV partition k visited for Q partition p by a unit whose last
// query tile is a_max (tile index within the partition).
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
  const uint32_t sb = (raw + 1023u) & ~1023u;  // 1024-aligned base (128B swizzle atoms)
  uint8_t* smem = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + Ly::BAR_OFF + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Ly::MISC_OFF + 4);

  // ---- unit decode: (item, b, h, pair) with the pair fastest
  int64_t u = blockIdx.x;
  const int qp = (int)(u % prm.n_pairs); u /= prm.n_pairs;
  const int h = (int)(u % prm.Hq); u /= prm.Hq;
  const int b = (int)(u % prm.B);
  const int item_idx = (int)(u / prm.B);
  const int unit = (int)blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_QFULL), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(Ly::B_KFULL + s), 1);
      mbar_init(bar(Ly::B_KEMPTY + s), 1);
      mbar_init(bar(Ly::B_VFULL + s), 1);
      mbar_init(bar(Ly::B_VEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Ly::B_SFULL + t), 1);
      mbar_init(bar(Ly::B_PFULL + t), BM);
    }
    mbar_init(bar(Ly::B_OFINAL), 1);
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

  const DevItem it = prm.items[item_idx];
  const int64_t L = prm.L;
  const bool item_ok = it.p >= 0 && it.p < prm.P && it.slot >= 0 && it.slot < prm.n_slots && it.n_kv >= 1 &&
                       it.kv_off >= 0;
  if (!item_ok && threadIdx.x == 0) record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_ITEM, unit);
  const bool run = item_ok && (*abort_flag == 0);
  const int p = it.p;
  const int nb = (int)((L + BN - 1) / BN);
  const int a0 = 2 * qp;
  const bool has1 = (int64_t)(a0 + 1) * BM < L;
  const int ntiles = has1 ? 2 : 1;
  const int a_max = a0 + ntiles - 1;
  const int hk = h / (prm.Hq / prm.Hkv);
  const int32_t* kvl = prm.kv_list + it.kv_off;

  if (run && warp < 8) {
    // ================================================================ softmax warpgroups
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // row within the tile = TMEM lane
    const int a_t = a0 + t;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tm_s = tmem + lane_base + (uint32_t)(t * 128);
    const uint32_t tm_o = tmem + lane_base + 256u + (uint32_t)(t * 128);
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    if (t < ntiles) {
      int j = 0;
      for (int ki = 0; ki < it.n_kv && ok; ++ki) {
        const int k = __ldg(kvl + ki);
        const bool diag = prm.causal && k == p;
        const int nbk = blocks_of(k, p, prm.causal, nb, a_max);
        for (int jb = 0; jb < nbk; ++jb, ++j) {
          ok = mbar_wait(bar(Ly::B_SFULL + t), (uint32_t)(j & 1), prm.wait_limit_ns, abort_flag, prm.status,
                         ROLE_SOFTMAX, unit);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          float s[BN];
#pragma unroll
          for (int c = 0; c < BN; c += 32) tmem_ld32(tm_s + (uint32_t)c, s + c);
          tc_wait_ld();
          const int64_t kv_valid = min((int64_t)BN, L - (int64_t)jb * BN);
          int lim = BN - 1;
          if (diag) lim = (jb < a_t) ? BN - 1 : (jb == a_t ? row : -1);
          lim = min(lim, (int)kv_valid - 1);
          if (lim < BN - 1) {
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (c > lim) s[c] = -INFINITY;
          }
          float mx = s[0];
#pragma unroll
          for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
          const float m_new = mx * prm.scale_log2;
          float factor = 1.f;
          if (m_new > -INFINITY) {
            if (m_used == -INFINITY) {
              m_used = m_new;
            } else if (m_new > m_used + LOG2_RESCALE) {
              factor = fast_exp2(m_used - m_new);
              m_used = m_new;
            }
          }
          if (__any_sync(0xffffffffu, factor != 1.f)) {
            // O_t already holds every earlier PV product: S_t(j) was issued after PV_t(j-1)
            // and its completion covers all earlier tensor-core work of the issuing thread.
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
          const float mref = (m_used == -INFINITY) ? 0.f : m_used;
          float sum = 0.f;
          uint32_t pk[BN / 2];
#pragma unroll
          for (int c = 0; c < BN / 2; ++c) {
            const float p0 = fast_exp2(fmaf(s[2 * c], prm.scale_log2, -mref));
            const float p1 = fast_exp2(fmaf(s[2 * c + 1], prm.scale_log2, -mref));
            sum += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
          }
          l_sum += sum;
          tmem_st32(tm_s, pk);
          tmem_st32(tm_s + 32u, pk + 32);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(bar(Ly::B_PFULL + t));
        }
      }
      if (ok) {
        ok = mbar_wait(bar(Ly::B_OFINAL), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_SOFTMAX, unit);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        const int64_t row_local = (int64_t)a_t * BM + row;
        const bool valid = row_local < L;
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const int64_t prow = (((int64_t)b * prm.Hq + h) * prm.n_slots + it.slot) * L + row_local;
        float* dst = prm.part_o + prow * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tm_o + (uint32_t)c, o);
          tc_wait_ld();
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + c + e) =
                  make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
          }
        }
        if (valid)
          prm.part_lse[prow] = l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
      }
    }
  } else if (run && warp == WARP_MMA) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false);
      const uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
      auto q_addr = [&](int t) { return sb + Ly::Q_OFF + (uint32_t)t * Ly::TILE; };
      auto k_addr = [&](int s) { return sb + Ly::K_OFF + (uint32_t)s * Ly::TILE; };
      auto v_addr = [&](int s) { return sb + Ly::V_OFF + (uint32_t)s * Ly::TILE; };
      // K-major operand (Q or K): K-step kk of 16 elements sits in box kk/4 at byte 32*(kk%4)
      auto kmaj = [&](uint32_t base, int kk) {
        return smem_desc_sw128(base + (uint32_t)(kk >> 2) * Ly::BOX + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
      };
      // MN-major V: K-step kk covers rows 16kk..16kk+15 (2 swizzle atoms of 8 rows); the
      // second 64-column half of d is the next box (leading byte offset)
      auto vdesc = [&](int s, int kk) { return smem_desc_sw128(v_addr(s) + (uint32_t)kk * 2048u, Ly::BOX, 1024u); };
      int NB = 0;
      for (int ki = 0; ki < it.n_kv; ++ki) NB += blocks_of(__ldg(kvl + ki), p, prm.causal, nb, a_max);
      bool ok = mbar_wait(bar(Ly::B_QFULL), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, unit);
      if (ok) ok = mbar_wait(bar(Ly::B_KFULL + 0), 0u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, unit);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ss(tmem + (uint32_t)(t * 128), kmaj(q_addr(t), kk), kmaj(k_addr(0), kk), idesc_qk, kk > 0);
          tc_commit(bar(Ly::B_SFULL + t));
        }
        tc_commit(bar(Ly::B_KEMPTY + 0));
      }
      for (int j = 0; j < NB && ok; ++j) {
        const int st = j % NST;
        const uint32_t ph = (uint32_t)((j / NST) & 1);
        ok = mbar_wait(bar(Ly::B_VFULL + st), ph, prm.wait_limit_ns, abort_flag, prm.status, ROLE_MMA, unit);
        for (int t = 0; t < ntiles && ok; ++t) {
          ok = mbar_wait(bar(Ly::B_PFULL + t), (uint32_t)(j & 1), prm.wait_limit_ns, abort_flag, prm.status,
                         ROLE_MMA, unit);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tm_p = tmem + (uint32_t)(t * 128);
          const uint32_t tm_o = tmem + 256u + (uint32_t)(t * 128);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            tc_mma_ts(tm_o, tm_p + (uint32_t)(kk * 8), vdesc(st, kk), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          if (j + 1 < NB) {
            const int sn = (j + 1) % NST;
            if (t == 0) {
              ok = mbar_wait(bar(Ly::B_KFULL + sn), (uint32_t)(((j + 1) / NST) & 1), prm.wait_limit_ns,
                             abort_flag, prm.status, ROLE_MMA, unit);
              if (!ok) break;
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss(tm_p, kmaj(q_addr(t), kk), kmaj(k_addr(sn), kk), idesc_qk, kk > 0);
            tc_commit(bar(Ly::B_SFULL + t));
          }
        }
        if (!ok) break;
        if (j + 1 < NB) tc_commit(bar(Ly::B_KEMPTY + (j + 1) % NST));
        tc_commit(bar(Ly::B_VEMPTY + st));
      }
      // o_final completes when every MMA above has: the softmax epilogue reads O after it, and
      // it is the exit-path drain before TMEM is freed.
      tc_commit(bar(Ly::B_OFINAL));
      mbar_drain(bar(Ly::B_OFINAL), 0u, DRAIN_NS);
    }
  } else if (run && warp == WARP_LOAD) {
    // ================================================================ TMA producer
    if (lane == 0) {
      const int64_t qrow0 = ((int64_t)b * prm.Hq + h) * prm.S + (int64_t)p * L + (int64_t)a0 * BM;
      mbar_expect_tx(bar(Ly::B_QFULL), (uint32_t)ntiles * Ly::TILE);
      for (int t = 0; t < ntiles; ++t)
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Ly::Q_OFF + (uint32_t)t * Ly::TILE + (uint32_t)c * Ly::BOX, &tmQ, c * 64,
                      (int32_t)(qrow0 + (int64_t)t * BM), bar(Ly::B_QFULL));
      const int64_t kvbase = ((int64_t)b * prm.Hkv + hk) * prm.S;
      int nk = 0, nv = 0;  // K and V block loads issued
      bool ok = true;
      for (int ki = 0; ki < it.n_kv && ok; ++ki) {
        const int k = __ldg(kvl + ki);
        if (k < 0 || k >= prm.P) {
          record_error(prm.status, MESH_ATTN_ERR_OUT_OF_RANGE, ROLE_LOAD, unit);
          *abort_flag = 1;
          break;
        }
        const int nbk = blocks_of(k, p, prm.causal, nb, a_max);
        for (int jb = 0; jb < nbk; ++jb) {
          const int st = nk % NST;
          const uint32_t ph = (uint32_t)((nk / NST) & 1);
          const int32_t krow = (int32_t)(kvbase + (int64_t)k * L + (int64_t)jb * BN);
          ok = mbar_wait(bar(Ly::B_KEMPTY + st), ph ^ 1u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_LOAD,
                         unit);
          if (!ok) break;
          mbar_expect_tx(bar(Ly::B_KFULL + st), Ly::TILE);
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sb + Ly::K_OFF + (uint32_t)st * Ly::TILE + (uint32_t)c * Ly::BOX, &tmK, c * 64, krow,
                        bar(Ly::B_KFULL + st));
          ++nk;
          ok = mbar_wait(bar(Ly::B_VEMPTY + st), ph ^ 1u, prm.wait_limit_ns, abort_flag, prm.status, ROLE_LOAD,
                         unit);
          if (!ok) break;
          mbar_expect_tx(bar(Ly::B_VFULL + st), Ly::TILE);
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sb + Ly::V_OFF + (uint32_t)st * Ly::TILE + (uint32_t)c * Ly::BOX, &tmV, c * 64, krow,
                        bar(Ly::B_VFULL + st));
          ++nv;
        }
      }
      // drain: every load issued must land before the CTA exits (the last NST of each ring)
      mbar_drain(bar(Ly::B_QFULL), 0u, DRAIN_NS);
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
  prm.S = a.S;
  prm.L = a.L;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.P = a.P;
  prm.n_items = a.n_items;
  prm.n_slots = a.n_slots;
  prm.n_pairs = (int32_t)n_pairs;
  prm.causal = a.causal;
  prm.scale_log2 = a.scale_log2;
  prm.wait_limit_ns = a.wait_limit_ns;
  auto kern = tile_fwd_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<D>::ALLOC);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return (int)e;
  }
  kern<<<dim3((unsigned)units), dim3(NUM_THREADS), Layout<D>::ALLOC, (cudaStream_t)stream>>>(mq, mk, mv, prm);
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
