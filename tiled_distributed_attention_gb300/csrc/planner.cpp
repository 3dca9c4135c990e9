// Host planner: partition -> tile map, KV Partition Rotation, causal pruning, greedy execution
// order and per-device receive counts for Mesh-Attention on a sqrt(P) x sqrt(P) virtual mesh.
//
// Follows "Mesh-Attention: A New Communication-Efficient Distributed Attention with Improved
// Data Locality": the Q-KV interaction matrix cut into 2D tiles, one per device, each device
// talking only to its own mesh row and column, KV Partition Rotation keeping a device's own Q
// and KV partition inside its tile (tutorial §"Mesh-Attention：从一维'环'到二维'网'", items
// (a)-(c); arXiv abstract), and the greedy rule of §"贪心算法：寻找最优的'流水线'" (take the
// transfer that unlocks the most compute).  On one GPU the greedy pass only fixes the order in
// which the tile kernel visits work; nothing is transferred.
//
// Cost: O(P * R^2) for the greedy pass with incrementally maintained gains, O(P^2) for the
// item KV lists (one entry per live partition block).
#include <algorithm>
#include <numeric>
#include <stdexcept>
#include <tuple>

#include "internal.h"

namespace mesh {

namespace {

inline bool live(int32_t p, int32_t k, bool causal) { return !causal || k <= p; }

struct DeviceGreedy {
  std::vector<int32_t> arr_q, arr_kv;  // arrival step per tile-local index, -1 = never needed
  int32_t steps = 0;
};

// Greedy receive order of device v on its tile (qset, kvset, both ascending).
void greedy_device(int32_t v, const int32_t* qset, const int32_t* kvset, int32_t R, bool causal,
                   DeviceGreedy& g) {
  g.arr_q.assign(R, -1);
  g.arr_kv.assign(R, -1);
  g.steps = 0;
  std::vector<char> need_q(R), need_kv(R);
  const int32_t q_max = qset[R - 1];
  const int32_t kv_min = *std::min_element(kvset, kvset + R);
  for (int32_t j = 0; j < R; ++j) need_q[j] = live(qset[j], kv_min, causal);
  for (int32_t i = 0; i < R; ++i) need_kv[i] = live(q_max, kvset[i], causal);
  // gains: live blocks a transfer would unlock given what has arrived
  std::vector<int32_t> gain_q(R, 0), gain_kv(R, 0);
  auto arrive_q = [&](int32_t j, int32_t step) {
    g.arr_q[j] = step;
    for (int32_t i = 0; i < R; ++i)
      if (live(qset[j], kvset[i], causal)) ++gain_kv[i];
  };
  auto arrive_kv = [&](int32_t i, int32_t step) {
    g.arr_kv[i] = step;
    for (int32_t j = 0; j < R; ++j)
      if (live(qset[j], kvset[i], causal)) ++gain_q[j];
  };
  for (int32_t j = 0; j < R; ++j)
    if (qset[j] == v && need_q[j]) arrive_q(j, 0);
  for (int32_t i = 0; i < R; ++i)
    if (kvset[i] == v && need_kv[i]) arrive_kv(i, 0);
  int32_t step = 0;
  for (;;) {
    int32_t best_gain = -1, best_kind = -1, best_idx = -1;
    // KV candidates first, ascending partition; a Q candidate wins only with a larger gain
    for (int32_t i = 0; i < R; ++i)
      if (need_kv[i] && g.arr_kv[i] < 0 && gain_kv[i] > best_gain) {
        best_gain = gain_kv[i]; best_kind = 0; best_idx = i;
      }
    for (int32_t j = 0; j < R; ++j)
      if (need_q[j] && g.arr_q[j] < 0 && gain_q[j] > best_gain) {
        best_gain = gain_q[j]; best_kind = 1; best_idx = j;
      }
    if (best_kind < 0) break;
    ++step;
    if (best_kind == 0) arrive_kv(best_idx, step); else arrive_q(best_idx, step);
  }
  g.steps = step;
}

}  // namespace

void build_plan(Plan& pl, int64_t S, int32_t P, bool causal, bool kvr, bool greedy) {
  if (P < 1) throw std::invalid_argument("P must be >= 1");
  if (P > 4096) throw std::invalid_argument("P must be <= 4096");
  int32_t R = 0;
  while ((R + 1) * (R + 1) <= P) ++R;
  if (R * R != P) throw std::invalid_argument("P must be a perfect square");
  if (S < 0) throw std::invalid_argument("S must be >= 0");
  if (S % P != 0) throw std::invalid_argument("S must be a multiple of P");
  pl = Plan();
  pl.S = S; pl.P = P; pl.R = R; pl.L = S / P;
  pl.layout = 0; pl.tile_q = R; pl.tile_kv = R;
  pl.causal = causal; pl.kvr = kvr; pl.greedy = greedy;
  const bool empty = (S == 0);

  pl.q_parts.resize((size_t)P * R);
  pl.kv_parts.resize((size_t)P * R);
  for (int32_t t = 0; t < P; ++t) {
    const int32_t r = t / R, c = t % R;
    for (int32_t j = 0; j < R; ++j) pl.q_parts[(size_t)t * R + j] = r * R + j;
    for (int32_t k = 0; k < R; ++k) pl.kv_parts[(size_t)t * R + k] = kvr ? k * R + c : c * R + k;
  }
  auto kv_min = [&](int32_t t) {
    const int32_t* kv = &pl.kv_parts[(size_t)t * R];
    return *std::min_element(kv, kv + R);
  };

  // Slot CSR: slots of p over the tiles of its mesh row, column ascending.
  std::vector<int32_t> slot_of((size_t)P * R, -1);  // [p * R + c]
  pl.slot_off.assign(P + 1, 0);
  int32_t n = 0;
  for (int32_t p = 0; p < P; ++p) {
    const int32_t r = p / R;
    for (int32_t c = 0; c < R; ++c) {
      const int32_t t = r * R + c;
      if (!empty && live(p, kv_min(t), causal)) slot_of[(size_t)p * R + c] = n++;
    }
    pl.slot_off[p + 1] = n;
  }
  pl.n_live = empty ? 0 : (causal ? (int64_t)P * (P + 1) / 2 : (int64_t)P * P);

  // Per-device greedy pass, item completion steps and KV visiting order.
  struct Key { int32_t step, t, p, slot; int64_t kv_begin; int32_t n_kv; };
  std::vector<Key> keys;
  keys.reserve(n);
  std::vector<int32_t> kv_scratch;
  kv_scratch.reserve((size_t)pl.n_live);
  pl.recv.assign((size_t)P * 3, 0);
  DeviceGreedy g;
  std::vector<int32_t> order(R);
  for (int32_t t = 0; t < P && !empty; ++t) {
    const int32_t v = t, c = t % R;
    const int32_t* qset = &pl.q_parts[(size_t)t * R];
    const int32_t* kvset = &pl.kv_parts[(size_t)t * R];
    greedy_device(v, qset, kvset, R, causal, g);
    pl.n_steps = std::max(pl.n_steps, greedy ? g.steps : 0);
    int32_t nq = 0, nkv = 0;
    for (int32_t j = 0; j < R; ++j) nq += (g.arr_q[j] >= 0 && qset[j] != v);
    for (int32_t i = 0; i < R; ++i) nkv += (g.arr_kv[i] >= 0 && kvset[i] != v);
    const int32_t own_slots = pl.slot_off[v + 1] - pl.slot_off[v];
    pl.recv[(size_t)v * 3 + 0] = nq;
    pl.recv[(size_t)v * 3 + 1] = nkv;
    pl.recv[(size_t)v * 3 + 2] = own_slots - (slot_of[(size_t)v * R + c] >= 0 ? 1 : 0);
    // KV visiting order: arrival order with greedy, ascending partition without
    std::iota(order.begin(), order.end(), 0);
    if (greedy)
      std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        return g.arr_kv[a] < g.arr_kv[b];
      });
    for (int32_t j = 0; j < R; ++j) {
      const int32_t p = qset[j];
      const int32_t slot = slot_of[(size_t)p * R + c];
      if (slot < 0) continue;
      Key key{0, t, p, slot, (int64_t)kv_scratch.size(), 0};
      int32_t done = 0;
      for (int32_t oi = 0; oi < R; ++oi) {
        const int32_t i = order[oi];
        if (!live(p, kvset[i], causal)) continue;
        kv_scratch.push_back(kvset[i]);
        ++key.n_kv;
        done = std::max(done, std::max(g.arr_q[j], g.arr_kv[i]));
      }
      key.step = greedy ? done : 0;
      keys.push_back(key);
    }
  }
  std::stable_sort(keys.begin(), keys.end(), [](const Key& a, const Key& b) {
    return std::tie(a.step, a.t, a.p) < std::tie(b.step, b.t, b.p);
  });

  pl.items.resize((size_t)n * 3);
  pl.item_step.resize(n);
  pl.kv_off.resize((size_t)n + 1);
  pl.kv_list.resize(kv_scratch.size());
  pl.dev_items.resize(n);
  int64_t pos = 0;
  for (int32_t i = 0; i < n; ++i) {
    const Key& k = keys[i];
    pl.items[(size_t)i * 3 + 0] = k.p;
    pl.items[(size_t)i * 3 + 1] = k.t;
    pl.items[(size_t)i * 3 + 2] = k.slot;
    pl.item_step[i] = k.step;
    pl.kv_off[i] = (int32_t)pos;
    std::copy(kv_scratch.begin() + k.kv_begin, kv_scratch.begin() + k.kv_begin + k.n_kv,
              pl.kv_list.begin() + pos);
    pos += k.n_kv;
  }
  pl.kv_off[n] = (int32_t)pos;
  if (pos != pl.n_live) throw std::logic_error("planner: KV entries do not cover the live blocks");
  // The kernels' copy of the work list takes the tiles one after another (row-major over the
  // mesh), each tile's items in that virtual device's greedy order.  The greedy pass fixes the
  // order within each device; how the devices' sequences interleave on one GPU is free, and
  // tile-major keeps a tile's KV set (shared by its items) and its mesh row's Q partitions
  // (shared with the next tile of the row) in L2.
  std::vector<int32_t> launch(n);
  std::iota(launch.begin(), launch.end(), 0);
  std::stable_sort(launch.begin(), launch.end(), [&](int32_t a, int32_t b) {
    return std::tie(keys[a].t, keys[a].step, keys[a].p) < std::tie(keys[b].t, keys[b].step, keys[b].p);
  });
  for (int32_t j = 0; j < n; ++j) {
    const Key& k = keys[launch[j]];
    pl.dev_items[j] = DevItem{k.p, k.slot, pl.kv_off[launch[j]], k.n_kv};
  }
  pl.launch = std::move(launch);
  build_kv_slots(pl);
}

// Ring-Attention's assignment in the same plan form, for comparison through the same kernels:
// device v owns Q partition v and computes its whole row ("Mesh-Attention" tutorial: the 1D
// ring, item (a), and the section on Ring-Attention's bottleneck).  KV partitions reach device v
// in ring order v, v-1, ... (own first, one hop per step); the item completes at the step its
// last live block arrives; items are ordered by (step, device).  Each device receives P - 1 KV
// partitions (a plain ring forwards all of them) and no Q or partial output.
void build_ring_plan(Plan& pl, int64_t S, int32_t P, bool causal) {
  if (P < 1) throw std::invalid_argument("P must be >= 1");
  if (P > 4096) throw std::invalid_argument("P must be <= 4096");
  if (S < 0) throw std::invalid_argument("S must be >= 0");
  if (S % P != 0) throw std::invalid_argument("S must be a multiple of P");
  pl = Plan();
  pl.S = S; pl.P = P; pl.R = 0; pl.L = S / P;
  pl.layout = 1; pl.tile_q = 1; pl.tile_kv = P;
  pl.causal = causal; pl.kvr = false; pl.greedy = true;
  const bool empty = (S == 0);
  pl.q_parts.resize(P);
  pl.kv_parts.resize((size_t)P * P);
  for (int32_t v = 0; v < P; ++v) {
    pl.q_parts[v] = v;
    for (int32_t i = 0; i < P; ++i) pl.kv_parts[(size_t)v * P + i] = ((v - i) % P + P) % P;
  }
  pl.slot_off.resize(P + 1);
  for (int32_t p = 0; p <= P; ++p) pl.slot_off[p] = empty ? 0 : p;
  pl.n_live = empty ? 0 : (causal ? (int64_t)P * (P + 1) / 2 : (int64_t)P * P);
  pl.recv.assign((size_t)P * 3, 0);
  if (empty) {
    build_kv_slots(pl);
    return;
  }
  std::vector<std::pair<int32_t, int32_t>> order;  // (completion step, device)
  order.reserve(P);
  for (int32_t v = 0; v < P; ++v) {
    int32_t done = 0;
    for (int32_t i = 0; i < P; ++i)
      if (live(v, pl.kv_parts[(size_t)v * P + i], causal)) done = i;
    order.push_back({done, v});
    pl.recv[(size_t)v * 3 + 1] = P - 1;
  }
  std::stable_sort(order.begin(), order.end());
  pl.items.resize((size_t)P * 3);
  pl.item_step.resize(P);
  pl.kv_off.resize((size_t)P + 1);
  pl.dev_items.resize(P);
  int64_t pos = 0;
  for (int32_t i = 0; i < P; ++i) {
    const int32_t v = order[i].second;
    pl.items[(size_t)i * 3 + 0] = v;
    pl.items[(size_t)i * 3 + 1] = v;
    pl.items[(size_t)i * 3 + 2] = v;
    pl.item_step[i] = order[i].first;
    pl.kv_off[i] = (int32_t)pos;
    int32_t n = 0;
    for (int32_t j = 0; j < P; ++j) {
      const int32_t k = pl.kv_parts[(size_t)v * P + j];
      if (live(v, k, causal)) { pl.kv_list.push_back(k); ++n; }
    }
    pl.dev_items[i] = DevItem{v, v, (int32_t)pos, n};
    pl.launch.push_back(i);  // ring: the kernels take the items in the public order
    pos += n;
    pl.n_steps = std::max(pl.n_steps, order[i].first);
  }
  pl.kv_off[P] = (int32_t)pos;
  if (pos != pl.n_live) throw std::logic_error("ring planner: KV entries do not cover the live blocks");
  build_kv_slots(pl);
}

// Backward pass: tile t sums dK and dV of each of its KV partitions over its own live Q
// partitions; those partial sums travel back along the mesh column to k's owner, as the
// forward's partial outputs travel along the mesh row.  Slots are grouped by k, tiles ascending.
void build_kv_slots(Plan& pl) {
  const int32_t P = pl.P;
  pl.kv_slot_off.assign((size_t)P + 1, 0);
  pl.kv_items.clear();
  pl.kv_q_off.assign(1, 0);
  pl.kv_q_list.clear();
  pl.dev_kv_items.clear();
  if (pl.S == 0) return;
  // tiles holding each KV partition, ascending (each tile lists a partition at most once)
  std::vector<std::vector<int32_t>> holders((size_t)P);
  for (int32_t t = 0; t < P; ++t)
    for (int32_t i = 0; i < pl.tile_kv; ++i) holders[(size_t)pl.kv_parts[(size_t)t * pl.tile_kv + i]].push_back(t);
  std::vector<int32_t> qs;
  for (int32_t k = 0; k < P; ++k) {
    for (int32_t t : holders[(size_t)k]) {
      qs.clear();
      for (int32_t j = 0; j < pl.tile_q; ++j) {
        const int32_t p = pl.q_parts[(size_t)t * pl.tile_q + j];
        if (live(p, k, pl.causal)) qs.push_back(p);
      }
      if (qs.empty()) continue;
      std::sort(qs.begin(), qs.end());
      const int32_t slot = (int32_t)pl.dev_kv_items.size();
      pl.kv_items.push_back(k);
      pl.kv_items.push_back(t);
      pl.kv_items.push_back(slot);
      pl.dev_kv_items.push_back(DevItem{k, slot, (int32_t)pl.kv_q_list.size(), (int32_t)qs.size()});
      pl.kv_q_list.insert(pl.kv_q_list.end(), qs.begin(), qs.end());
      pl.kv_q_off.push_back((int32_t)pl.kv_q_list.size());
    }
    pl.kv_slot_off[(size_t)k + 1] = (int32_t)pl.dev_kv_items.size();
  }
  if ((int64_t)pl.kv_q_list.size() != pl.n_live)
    throw std::logic_error("planner: KV slots do not cover the live blocks");
}

BwdWorkspaceLayout bwd_workspace_layout(const Plan& pl) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  BwdWorkspaceLayout w{};
  w.slot_off_off = 0;
  w.slot_off_bytes = sizeof(int32_t) * pl.slot_off.size();
  w.items_off = up(w.slot_off_bytes);
  w.items_bytes = sizeof(DevItem) * pl.dev_items.size();
  w.kv_off = w.items_off + up(w.items_bytes);
  w.kv_bytes = sizeof(int32_t) * pl.kv_list.size();
  w.kv_slot_off_off = w.kv_off + up(w.kv_bytes);
  w.kv_slot_off_bytes = sizeof(int32_t) * pl.kv_slot_off.size();
  w.kv_items_off = w.kv_slot_off_off + up(w.kv_slot_off_bytes);
  w.kv_items_bytes = sizeof(DevItem) * pl.dev_kv_items.size();
  w.q_list_off = w.kv_items_off + up(w.kv_items_bytes);
  w.q_list_bytes = sizeof(int32_t) * pl.kv_q_list.size();
  w.counter_off = w.q_list_off + up(w.q_list_bytes);
  w.total = w.counter_off + 512;
  return w;
}

WorkspaceLayout workspace_layout(const Plan& pl) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  WorkspaceLayout w{};
  w.slot_off_bytes = sizeof(int32_t) * pl.slot_off.size();
  w.items_off = up(w.slot_off_bytes);
  w.items_bytes = sizeof(DevItem) * pl.dev_items.size();
  w.kv_off = w.items_off + up(w.items_bytes);
  w.kv_bytes = sizeof(int32_t) * pl.kv_list.size();
  w.counter_off = w.kv_off + up(w.kv_bytes);
  w.total = w.counter_off + 256;
  return w;
}

}  // namespace mesh
