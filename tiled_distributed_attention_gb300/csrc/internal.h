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
  std::vector<DevItem> dev_items;          // [n] the kernels' copy of the order

  int32_t n_slots() const { return (int32_t)item_step.size(); }
};

// Throws std::invalid_argument / std::bad_alloc; the ABI layer converts.
void build_plan(Plan& plan, int64_t S, int32_t P, bool causal, bool kvr, bool greedy);
void build_ring_plan(Plan& plan, int64_t S, int32_t P, bool causal);

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
};
// Kernel launchers return a cudaError_t value as int; *err gets a message on failure.
int launch_tile_fwd_simt(const TileArgs& a, mesh_attn_dtype dt, void* stream, std::string* err);
int launch_tile_fwd_tc(const TileArgs& a, void* stream, std::string* err);

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

// Record `msg` as the calling thread's last error (mesh_attn_last_error) and return `code`.
int set_last_error(int code, const std::string& msg);
// Current process-wide bound on device-side waits (mesh_attn_set_wait_limit_ns).
int64_t current_wait_limit_ns();

}  // namespace mesh

// The opaque handle of the C ABI.
struct mesh_attn_plan {
  mesh::Plan p;
};
