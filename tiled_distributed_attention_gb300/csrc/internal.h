// Internal declarations shared by the planner, the C-ABI layer and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "mesh_attn.h"

namespace mesh {

// One work item as the kernels read it: Q partition p, its partial slot, and the item's KV
// partitions kv_list[kv_off .. kv_off + n_kv) in visiting order.
struct alignas(16) DevItem {
  int32_t p;
  int32_t slot;
  int32_t kv_off;
  int32_t n_kv;
};

struct Plan {
  int64_t S = 0, L = 0;
  int32_t P = 0, R = 0;          // R: mesh side (0 for a ring plan)
  int32_t layout = 0;            // 0 mesh, 1 ring
  int32_t tile_q = 0, tile_kv = 0;  // Q and KV partitions per tile
  bool causal = false, kvr = false, greedy = false;
  int32_t n_steps = 0;
  int64_t n_live = 0;
  std::vector<int32_t> q_parts, kv_parts;  // [P*tile_q], [P*tile_kv]
  std::vector<int32_t> slot_off;           // [P+1]
  std::vector<int32_t> items;              // [n*3] (p, t, slot) in execution order
  std::vector<int32_t> item_step;          // [n]
  std::vector<int32_t> kv_off;             // [n+1]
  std::vector<int32_t> kv_list;            // [kv_off[n]]
  std::vector<int32_t> recv;               // [P*3] Q, KV, partial-O partitions received
  std::vector<DevItem> dev_items;          // [n] the kernels' copy of the work list, in launch order
  std::vector<int32_t> launch;             // [n] launch position -> index in `items`
  // Backward pass: the (KV partition k, tile t) pairs with a live block, grouped by k, tiles
  // ascending; each with the tile's Q partitions live for k, ascending.
  std::vector<int32_t> kv_slot_off;        // [P+1]
  std::vector<int32_t> kv_items;           // [m*3] (k, t, kv slot)
  std::vector<int32_t> kv_q_off;           // [m+1]
  std::vector<int32_t> kv_q_list;          // [kv_q_off[m]]
  std::vector<DevItem> dev_kv_items;       // [m] as the kernels read them: {k, kv slot, q_off, n_q}

  int32_t n_slots() const { return (int32_t)item_step.size(); }
  int32_t n_kv_slots() const { return (int32_t)(kv_q_off.empty() ? 0 : kv_q_off.size() - 1); }
};

// Throws std::invalid_argument / std::bad_alloc; the ABI layer converts.
void build_plan(Plan& plan, int64_t S, int32_t P, bool causal, bool kvr, bool greedy);
void build_ring_plan(Plan& plan, int64_t S, int32_t P, bool causal);
// Fills the backward fields from the tile map (called by both builders).
void build_kv_slots(Plan& plan);

// Workspace layout shared by tile_fwd and merge: [slot_off | items | kv_list | counter].
struct WorkspaceLayout {
  size_t slot_off_bytes, items_off, items_bytes, kv_off, kv_bytes, counter_off, total;
};
WorkspaceLayout workspace_layout(const Plan& plan);

struct TileArgs {
  const void* Q;
  const void* K;
  const void* V;
  float* part_o;
  float* part_lse;
  const DevItem* items;
  const int32_t* kv_list;
  uint32_t* counter;
  int32_t* status;
  int64_t S, L;
  int32_t B, Hq, Hkv, d, P, n_items, n_slots;
  int32_t causal;
  float scale;
  float scale_log2;
  int64_t wait_limit_ns;
  void* pieces;  // fp32 inputs: device buffer for the bf16 pieces of Q, K and V (f32_pieces_layout)
};
// Kernel launchers return a cudaError_t value as int; *err gets a message on failure.
int launch_tile_fwd_tc(const TileArgs& a, void* stream, std::string* err);
// fp32 inputs: split Q, K and V into bf16 pieces in a.pieces, then the tensor-core forward.
int launch_tile_fwd_tc32(const TileArgs& a, void* stream, std::string* err);
// Byte layout of the bf16 pieces of fp32 Q, K and V ([3][rows][d] each, 256-byte aligned parts).
struct F32Pieces {
  size_t q_off, k_off, v_off, total;
};
F32Pieces f32_pieces_layout(int32_t B, int32_t Hq, int32_t Hkv, int64_t S, int32_t d);

struct MergeArgs {
  const float* part_o;
  const float* part_lse;
  const int32_t* slot_off;
  void* O;
  float* LSE;
  int32_t* status;
  int64_t S, L;
  int32_t B, Hq, d, P, n_slots;
};
int launch_merge(const MergeArgs& a, mesh_attn_dtype out_dtype, void* stream, std::string* err);

// ---------------------------------------------------------------- backward pass
// Workspace of the backward calls: [slot_off | items | kv_list | kv_slot_off | kv_items |
// kv_q_list | counters (2 x 256 B)].
struct BwdWorkspaceLayout {
  size_t slot_off_off, slot_off_bytes, items_off, items_bytes, kv_off, kv_bytes;
  size_t kv_slot_off_off, kv_slot_off_bytes, kv_items_off, kv_items_bytes, q_list_off, q_list_bytes;
  size_t counter_off, total;
};
BwdWorkspaceLayout bwd_workspace_layout(const Plan& plan);

struct BwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* dO;
  const float* LSE;  // [B, Hq, S] natural log, from the forward merge
  const float* D;    // [B, Hq, S] dO . O
  float* dq_part;    // [B, Hq, n_slots, L, d]
  float* dk_part;    // [B, Hkv, n_kv_slots, L, d]
  float* dv_part;
  const DevItem* items;     // forward work items {p, slot, kv_off, n_kv}
  const int32_t* kv_list;
  const DevItem* kv_items;  // KV slots {k, kv slot, q_off, n_q}
  const int32_t* q_list;
  uint32_t* counters;       // [2] scheduling counters (dq pass, dkdv pass)
  int32_t* status;
  int64_t S, L;
  int32_t B, Hq, Hkv, d, P, n_items, n_slots, n_kv_items, n_kv_slots;
  int32_t causal;
  float scale;
  float scale_log2;
  int64_t wait_limit_ns;
};
int launch_tile_bwd_simt(const BwdArgs& a, void* stream, std::string* err);
int launch_tile_bwd_tc(const BwdArgs& a, void* stream, std::string* err);

struct PrepArgs {
  const void* O;
  const void* dO;
  float* D;
  int32_t* status;
  int64_t S;
  int32_t B, H, d;
};
int launch_bwd_prep(const PrepArgs& a, mesh_attn_dtype dt, void* stream, std::string* err);

// out[b, h, part * L + r, :] = sum over the slots off[part] .. off[part + 1] of part[b, h, slot, r, :]
struct ReduceArgs {
  const float* part;
  const int32_t* off;
  void* out;
  int32_t* status;
  int64_t S, L;
  int32_t B, H, d, P, n_slots;
};
int launch_bwd_reduce(const ReduceArgs& a, mesh_attn_dtype out_dtype, void* stream, std::string* err);

// Record `msg` as the calling thread's last error (mesh_attn_last_error) and return `code`.
int set_last_error(int code, const std::string& msg);
// Current process-wide bound on device-side waits (mesh_attn_set_wait_limit_ns).
int64_t current_wait_limit_ns();

}  // namespace mesh

// The opaque handle of the C ABI.
struct mesh_attn_plan {
  mesh::Plan p;
};
