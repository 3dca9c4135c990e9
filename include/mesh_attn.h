/*
 * mesh_attn.h -- C ABI of the single-GPU Mesh-Attention hot path (sm_103a).
 *
 * The operation.  Exact scaled-dot-product attention O = softmax(Q K^T * scale) V with the
 * natural-log row log-sum-exp LSE, computed the way Mesh-Attention decomposes it
 * ("Mesh-Attention: A New Communication-Efficient Distributed Attention with Improved Data
 * Locality", tutorial §"Mesh-Attention：从一维'环'到二维'网'" and the arXiv abstract):
 *   1. the sequence of S tokens is cut into P partitions of L = S/P tokens; the P x P
 *      Q-KV interaction matrix is assigned as 2D tiles to a sqrt(P) x sqrt(P) mesh of
 *      (virtual) devices, with KV Partition Rotation (KVR) and a greedy order
 *      (tutorial §"贪心算法：寻找最优的'流水线'");
 *   2. each tile computes, for every Q partition it holds, a partial output O_t and its
 *      LSE_t over the tile's KV partitions (the online m_i / l_i softmax of
 *      "环形注意力：突破长序列处理瓶颈的分布式计算范式", §"数值稳定性：Log-Sum-Exp技术的分布式应用");
 *   3. the partials of each Q partition are merged by LSE rescaling:
 *      lse = ln sum_t exp(lse_t), O = sum_t exp(lse_t - lse) O_t.
 * On one GPU the mesh devices are virtual: the plan fixes the tiles and the execution
 * order, and the receive volumes a real mesh would move are counted, not performed.
 *
 * Conventions shared by every call.
 *   - Tensors are dense, row-major, contiguous, in device memory owned by the caller:
 *     Q [B, Hq, S, d], K and V [B, Hkv, S, d], O [B, Hq, S, d], LSE [B, Hq, S].
 *     Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *   - Causal masking: key j is visible to query i iff j <= i (same token index space).
 *   - Partials are fp32: partial_o [B, Hq, n_slots, L, d] and partial_lse [B, Hq, n_slots, L],
 *     where the slots of partition p are [slot_off[p], slot_off[p+1]) (see
 *     mesh_attn_plan_slots).  O_t is normalised (acc / l) and lse_t = m + ln l.  A row with no
 *     visible key in a slot has O_t = 0 and lse_t = -inf; the merge gives it weight 0.
 *   - Every function returns a mesh_attn_status.  Nothing throws across the ABI.  All
 *     host-side checks run before anything is enqueued; on error nothing is enqueued.
 *     mesh_attn_last_error() gives a one-line description of the last error on the
 *     calling thread.
 *   - GPU calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and never synchronise, except mesh_attn_read_status.
 *   - Device-side failures (a bounded wait that gave up, a work-list index out of range)
 *     are recorded in the caller's status block d_status: MESH_ATTN_STATUS_WORDS int32 in
 *     device memory, zeroed by the caller before the first call; word 0 holds the first
 *     error code, word 1 the kernel role that raised it, word 2 the work unit.  Kernels
 *     skip their work while word 0 is non-zero.  No kernel traps or asserts.
 */
#ifndef MESH_ATTN_H
#define MESH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MESH_ATTN_OK = 0,
  MESH_ATTN_ERR_INVALID_ARG = 1,    /* bad size, null pointer, P not a square, S % P != 0 */
  MESH_ATTN_ERR_UNSUPPORTED = 2,    /* a valid problem outside what the kernels implement */
  MESH_ATTN_ERR_MISALIGNED = 3,     /* a tensor pointer not 16-byte aligned */
  MESH_ATTN_ERR_CUDA = 4,           /* a CUDA runtime call failed (message in last_error) */
  MESH_ATTN_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up (from d_status) */
  MESH_ATTN_ERR_OUT_OF_RANGE = 6,   /* a device-side index check failed (from d_status) */
  MESH_ATTN_ERR_INTERNAL = 7,       /* an internal invariant failed */
  MESH_ATTN_ERR_NO_MEMORY = 8,      /* a host allocation failed */
  MESH_ATTN_ERR_WORKSPACE = 9       /* the workspace passed is smaller than required */
} mesh_attn_status;

typedef enum { MESH_ATTN_F32 = 0, MESH_ATTN_BF16 = 1 } mesh_attn_dtype;

#define MESH_ATTN_STATUS_WORDS 4

/* Opaque plan: host memory only, immutable after creation, safe to share between threads
 * and streams.  Created and freed by the library. */
typedef struct mesh_attn_plan mesh_attn_plan;

typedef struct {
  int64_t S;              /* tokens */
  int64_t L;              /* tokens per partition, S / P */
  int32_t P;              /* partitions = virtual devices = tiles */
  int32_t R;              /* mesh side sqrt(P) (0 for a ring plan) */
  int32_t causal, kvr, greedy;
  int32_t n_slots;        /* partial slots = work items, (p, tile) pairs with a live block */
  int32_t n_steps;        /* steps of the slowest device (greedy or ring; 0 without greedy) */
  int32_t layout;         /* 0: sqrt(P) x sqrt(P) mesh tiles; 1: ring rows */
  int32_t tile_q;         /* Q partitions per tile: R (mesh) or 1 (ring) */
  int32_t tile_kv;        /* KV partitions per tile: R (mesh) or P (ring) */
  int64_t n_kv_entries;   /* sum over items of their KV partitions = live partition blocks */
  int64_t n_live_blocks;  /* live (p, k) partition blocks of the P x P matrix */
  int32_t n_kv_slots;     /* backward: (KV partition, tile) pairs with a live block */
  int32_t reserved;
} mesh_attn_plan_info;

/* Build the tile plan (tutorial §"Mesh-Attention：从一维'环'到二维'网'", items (b) and (c);
 * §"贪心算法"; abstract: 2D tiles, KVR, greedy scheduling).
 *   S >= 0 tokens, P >= 1 partitions with P a perfect square, P <= 4096, S % P == 0.
 *   causal, kvr, greedy: 0 or 1.
 *   Tile t = device v at mesh position (v / R, v % R) holds Q partitions {r R + j : j < R} and
 *   KV partitions {k R + c : k < R} with KVR (own mesh column; block (v, v) is local) or the
 *   contiguous {c R + k : k < R} without.  Causal: block (p, k) is live iff k <= p.
 *   Greedy: each virtual device repeatedly takes the Q or KV transfer that unlocks the most
 *   live blocks (ties: KV first, then the lower partition index); work items are ordered by
 *   the step that unlocks their last block, devices interleaved step by step; each item
 *   visits its KV partitions in arrival order.  Without greedy: (tile, p) order, KV ascending.
 *   S == 0 gives an empty plan (no slots, every GPU call is a no-op).
 * On success *out owns the plan; free it with mesh_attn_plan_destroy. */
int mesh_attn_plan_create(int64_t S, int32_t P, int32_t causal, int32_t kvr, int32_t greedy,
                          mesh_attn_plan** out);

/* Ring-Attention's work assignment as a plan of the same form, to compare against the mesh
 * through the same kernels (tutorial §"Ring-Attention 的'阿喀琉斯之踵'" and the 1D ring of
 * §"Mesh-Attention：从一维'环'到二维'网'", item (a)): device v owns Q partition v and
 * computes its whole row, visiting KV partitions in ring order v, v-1, ... (own first, one hop
 * per step); one partial slot per Q partition.  Receive counts: P - 1 KV partitions per device,
 * no Q and no partial output.  Any P >= 1 (P <= 4096), S >= 0 with S % P == 0. */
int mesh_attn_plan_create_ring(int64_t S, int32_t P, int32_t causal, mesh_attn_plan** out);

/* Free a plan (NULL is accepted).  The caller must not use it afterwards. */
int mesh_attn_plan_destroy(mesh_attn_plan* plan);

/* Scalar facts of the plan. */
int mesh_attn_plan_get_info(const mesh_attn_plan* plan, mesh_attn_plan_info* out);

/* Tile map: q_parts[t*tile_q + j], kv_parts[t*tile_kv + k] for t < P (caller arrays of
 * P*tile_q and P*tile_kv int32; tile_q = tile_kv = R for a mesh plan). */
int mesh_attn_plan_tiles(const mesh_attn_plan* plan, int32_t* q_parts, int32_t* kv_parts);

/* Partial-slot CSR: slot_off[P + 1] (caller array). */
int mesh_attn_plan_slots(const mesh_attn_plan* plan, int32_t* slot_off);

/* Execution order.  items[3 i + 0..2] = (Q partition p, tile t, slot) of the i-th item,
 * item_step[i] = greedy step that completes it (0 without greedy), the KV partitions of item
 * i in visiting order are kv_list[kv_off[i] .. kv_off[i+1]).  Caller arrays of n_slots*3,
 * n_slots, n_slots + 1 and n_kv_entries int32; any of them may be NULL to skip it. */
int mesh_attn_plan_order(const mesh_attn_plan* plan, int32_t* items, int32_t* item_step,
                         int32_t* kv_off, int32_t* kv_list);

/* The order in which the kernels take the work items: order[j] (n_slots int32, caller array) is
 * the index, in mesh_attn_plan_order's list, of the j-th item the kernels take.  The greedy pass
 * (tutorial §"贪心算法：寻找最优的'流水线'") fixes each virtual device's order of work; the
 * public list interleaves the devices step by step.  One GPU takes the devices' sequences tile
 * after tile (row-major over the mesh), each in its own greedy order, so that the work items
 * running together share a tile's KV partitions and its mesh row's Q partitions in L2.  A ring
 * plan is taken in its public order.  A permutation of 0 .. n_slots - 1. */
int mesh_attn_plan_launch_order(const mesh_attn_plan* plan, int32_t* order);

/* Receive volumes a real mesh would move, per device v (tutorial §"Mesh-Attention：从一维'环'
 * 到二维'网'": per-device traffic grows as O(sqrt(N)) rather than Ring's O(N); abstract: a
 * device gathers only some of the Q and KV partitions).
 *   counts[3 v + 0..2] = Q, KV and partial-O partitions device v receives (may be NULL);
 *   bytes[3 v + 0..2]  = the same in bytes: a Q partition is L*Hq*d elements of `dtype`, a KV
 *                        partition 2*L*Hkv*d elements, a partial L*Hq*(d + 1) fp32 (may be NULL);
 *   *ring_bytes = the KV bytes one device receives in plain Ring-Attention, (P - 1) KV
 *                 partitions (may be NULL). */
int mesh_attn_plan_volumes(const mesh_attn_plan* plan, int32_t Hq, int32_t Hkv, int32_t d,
                           mesh_attn_dtype dtype, int32_t* counts, int64_t* bytes,
                           int64_t* ring_bytes);

/* Element counts of partial_o and partial_lse for a batch of B sequences with Hq heads of
 * size d: B*Hq*n_slots*L*d and B*Hq*n_slots*L. */
int mesh_attn_partials_size(const mesh_attn_plan* plan, int32_t B, int32_t Hq, int32_t d,
                            size_t* o_elems, size_t* lse_elems);

/* Bytes of device workspace mesh_attn_tile_fwd with bf16 inputs, and mesh_attn_merge, need for
 * this plan (the plan's work list, slot offsets and a scheduling counter).  The caller allocates
 * it (16-byte aligned) and may reuse it across calls on one stream; calls that overlap on the GPU
 * need separate workspaces. */
int mesh_attn_workspace_size(const mesh_attn_plan* plan, size_t* bytes);

/* Bytes of device workspace mesh_attn_tile_fwd needs for inputs of `in_dtype` and these sizes:
 * the above for MESH_ATTN_BF16; for MESH_ATTN_F32 also room for the bf16 pieces the fp32 path
 * splits Q, K and V into, 6 * (B*Hq + 2*B*Hkv) * S * d bytes (see mesh_attn_tile_fwd).  Enough for
 * mesh_attn_merge as well. */
int mesh_attn_workspace_size_for(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B,
                                 int32_t Hq, int32_t Hkv, int32_t d, size_t* bytes);

/* Tile attention forward: every (Q partition, tile) item of the plan, for every batch and
 * query head, writes its partial O_t and lse_t (step 2 above).
 *   in_dtype  MESH_ATTN_BF16 (tensor-core kernel: bf16 products, fp32 accumulation, fp32
 *             online softmax, P rounded to bf16 for the PV product) or MESH_ATTN_F32 (tensor-core
 *             kernel with fp32 accuracy: Q, K, V and P are each split exactly into three bf16
 *             pieces x = x1 + x2 + x3 and every product sums the six piece products of order
 *             >= 2^-16, x1y1 + x1y2 + x2y1 + x1y3 + x3y1 + x2y2, with fp32 accumulation; the
 *             pieces go into the workspace, which must then hold mesh_attn_workspace_size_for
 *             bytes).
 *   d         64 or 128.  B >= 0, Hq >= 0, Hkv >= 1, Hq % Hkv == 0.
 *   Q, K, V   device tensors of in_dtype, 16-byte aligned (layouts above).
 *   scale     softmax scale, finite and > 0 (1/sqrt(d) is the usual choice).
 *   partial_o, partial_lse  device fp32 outputs, sizes from mesh_attn_partials_size.
 *   workspace device buffer of at least mesh_attn_workspace_size bytes.
 *   d_status  device status block (see above).
 * Any L >= 1 works: query rows and keys past the end of a partition are masked. */
int mesh_attn_tile_fwd(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B,
                       int32_t Hq, int32_t Hkv, int32_t d, const void* Q, const void* K,
                       const void* V, float scale, float* partial_o, float* partial_lse,
                       void* workspace, size_t workspace_bytes, int32_t* d_status,
                       void* stream);

/* Maximum scratch of mesh_attn_tile_fwd_noalloc: device bytes every GPU that loads the
 * library reserves for it until the process exits. */
#define MESH_ATTN_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Tile attention forward for callers that cannot allocate device memory.  The paper has no
 * counterpart: this is a service of this library.
 * Who needs it: code that runs where it may not call cudaMalloc -- under a framework whose
 * caching allocator already owns the device memory pool (a direct allocation would fail or
 * escape its accounting), inside an allocator or memory-pressure callback, or with a fixed,
 * pre-reserved memory budget -- and so cannot provide the workspace mesh_attn_tile_fwd asks
 * for.  It computes exactly what mesh_attn_tile_fwd computes, with the same arguments minus
 * the workspace; the caller still passes the inputs, the partial outputs and d_status.
 * The plan's work list (and, for fp32 inputs, the bf16 pieces of Q, K and V) goes into one fixed
 * array of MESH_ATTN_NOALLOC_SCRATCH_BYTES inside the library instead.  A call that needs more
 * (a work list of about 2.6 MB for P = 1024 causal; P = 4096 is too large; fp32 inputs above
 * about 4 MB of pieces) returns MESH_ATTN_ERR_WORKSPACE with the size in mesh_attn_last_error().
 * The first call on a device looks up that device's array address (cudaGetSymbolAddress with
 * the device current); make that first call before any stream capture.  No cudaMalloc, cudaFree
 * or other allocating call is made.  All calls on a device share the one array and each call
 * rewrites what the kernel reads from it, so calls that overlap on the GPU (other streams,
 * other host threads) race: serialise them. */
int mesh_attn_tile_fwd_noalloc(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B,
                               int32_t Hq, int32_t Hkv, int32_t d, const void* Q, const void* K,
                               const void* V, float scale, float* partial_o, float* partial_lse,
                               int32_t* d_status, void* stream);

/* LSE merge (step 3): per (batch, head, row) over the slots of the row's partition,
 *   M = max_t lse_t, lse = M + ln sum_t exp(lse_t - M), O = sum_t exp(lse_t - lse) O_t;
 * a row whose slots are all -inf gets O = 0 and lse = -inf.
 *   out_dtype MESH_ATTN_BF16 (O rounded to nearest even) or MESH_ATTN_F32.
 *   partial_o, partial_lse  as written by mesh_attn_tile_fwd (or any values of that layout).
 *   O [B, Hq, S, d] of out_dtype, LSE [B, Hq, S] fp32: device outputs, 16-byte aligned.
 *   workspace, d_status, stream as for mesh_attn_tile_fwd. */
int mesh_attn_merge(const mesh_attn_plan* plan, mesh_attn_dtype out_dtype, int32_t B,
                    int32_t Hq, int32_t d, const float* partial_o, const float* partial_lse,
                    void* O, float* LSE, void* workspace, size_t workspace_bytes,
                    int32_t* d_status, void* stream);

/* ---------------------------------------------------------------- backward pass
 *
 * The pages describe the forward pass; Mesh-Attention is a training method (tutorial: end-to-end
 * training speedups; closing remarks on large-model training), so the backward pass keeps the
 * forward's tile structure.  With the forward's global LSE and an upstream gradient dO:
 *   P_ij = exp(scale q_i.k_j - LSE_i) over the visible keys,  dP_ij = dO_i . v_j,
 *   D_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i,
 * a KV head's dK and dV summing over its query heads.  Tile t computes, for each of its work
 * items (p, t), the dQ sums over its KV partitions into the item's partial slot (the forward's
 * slots: summed along the mesh row), and for each of its KV partitions k with a live block, the
 * dK / dV sums over its Q partitions into a KV slot (summed along the mesh column back to k's
 * owner).  Partials are fp32:
 *   dq_partial [B, Hq, n_slots, L, d];  dk_partial, dv_partial [B, Hkv, n_kv_slots, L, d].
 * Call order: mesh_attn_bwd_prep (D), mesh_attn_tile_bwd, mesh_attn_bwd_reduce. */

/* KV slots: kv_slot_off[P + 1] (the slots of KV partition k are kv_slot_off[k] ..
 * kv_slot_off[k+1] - 1, grouped by k, tiles ascending); kv_items[3 i + 0..2] = (k, tile t,
 * kv slot i); the tile's Q partitions with a live block for k, ascending, are
 * q_list[q_off[i] .. q_off[i+1]).  Caller arrays of P + 1, n_kv_slots * 3, n_kv_slots + 1 and
 * n_live_blocks int32; any may be NULL to skip it. */
int mesh_attn_plan_kv_slots(const mesh_attn_plan* plan, int32_t* kv_slot_off, int32_t* kv_items,
                            int32_t* q_off, int32_t* q_list);

/* Element counts of the backward partials: *dq_elems = B*Hq*n_slots*L*d for dq_partial,
 * *dkv_elems = B*Hkv*n_kv_slots*L*d for each of dk_partial and dv_partial. */
int mesh_attn_bwd_partials_size(const mesh_attn_plan* plan, int32_t B, int32_t Hq, int32_t Hkv,
                                int32_t d, size_t* dq_elems, size_t* dkv_elems);

/* Bytes of device workspace mesh_attn_tile_bwd and mesh_attn_bwd_reduce need (both work lists,
 * both slot CSRs, two scheduling counters); caller-allocated, 16-byte aligned, reusable across
 * calls on one stream. */
int mesh_attn_bwd_workspace_size(const mesh_attn_plan* plan, size_t* bytes);

/* D[b, h, i] = sum_e dO[b, h, i, e] * O[b, h, i, e] in fp32 (the row term of dS).
 *   dtype of O and dO: MESH_ATTN_BF16 or MESH_ATTN_F32; O, dO [B, Hq, S, d] 16-byte aligned;
 *   D [B, Hq, S] fp32; d 64 or 128. */
int mesh_attn_bwd_prep(mesh_attn_dtype dtype, int32_t B, int32_t Hq, int64_t S, int32_t d,
                       const void* O, const void* dO, float* D, int32_t* d_status, void* stream);

/* Tile attention backward: the partial gradients above for every batch and head.
 *   in_dtype  MESH_ATTN_BF16 (tensor-core kernels: bf16 products with fp32 accumulation; P and
 *             dS rounded to bf16 for the products that take them) or MESH_ATTN_F32 (CUDA-core
 *             kernels, fp32 throughout).
 *   Q, K, V, dO of in_dtype (dO [B, Hq, S, d]), 16-byte aligned; LSE [B, Hq, S] fp32 as written by
 *   mesh_attn_merge; D from mesh_attn_bwd_prep; scale as in the forward call.
 *   dq_partial, dk_partial, dv_partial: fp32 outputs, sizes from mesh_attn_bwd_partials_size.
 *   Other arguments as for mesh_attn_tile_fwd.  Rows with LSE = -inf contribute nothing. */
int mesh_attn_tile_bwd(const mesh_attn_plan* plan, mesh_attn_dtype in_dtype, int32_t B, int32_t Hq,
                       int32_t Hkv, int32_t d, const void* Q, const void* K, const void* V,
                       const void* dO, const float* LSE, const float* D, float scale,
                       float* dq_partial, float* dk_partial, float* dv_partial, void* workspace,
                       size_t workspace_bytes, int32_t* d_status, void* stream);

/* Sum the backward partials: dQ [B, Hq, S, d] over the slots of each Q partition, dK and dV
 * [B, Hkv, S, d] over the KV slots of each KV partition, rounded to out_dtype (nearest even for
 * bf16).  Outputs 16-byte aligned; other arguments as for mesh_attn_merge. */
int mesh_attn_bwd_reduce(const mesh_attn_plan* plan, mesh_attn_dtype out_dtype, int32_t B,
                         int32_t Hq, int32_t Hkv, int32_t d, const float* dq_partial,
                         const float* dk_partial, const float* dv_partial, void* dQ, void* dK,
                         void* dV, void* workspace, size_t workspace_bytes, int32_t* d_status,
                         void* stream);

/* Synchronise `stream`, copy word 0 of the device status block to *out (a mesh_attn_status).
 * Returns MESH_ATTN_ERR_CUDA if the copy or the synchronisation failed. */
int mesh_attn_read_status(const int32_t* d_status, void* stream, int32_t* out);

/* Static description of a status code. */
const char* mesh_attn_status_string(int status);

/* One-line description of the last error returned on the calling thread ("" if none). */
const char* mesh_attn_last_error(void);

/* Upper bound, in nanoseconds, on every device-side wait of later launches (process-wide;
 * default 2e9).  A wait that exceeds it records MESH_ATTN_ERR_DEVICE_TIMEOUT and the kernel
 * drains its copies in flight, frees its tensor memory and returns.  ns >= 0; 0 makes every
 * wait that is not already satisfied give up at once (used to test the error path). */
int mesh_attn_set_wait_limit_ns(int64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MESH_ATTN_H */
