"""The C ABI from C itself: a C99 program that includes only include/mesh_attn.h and links the
shared library compiles warning-free under -std=c99 -pedantic, runs the host-only calls
(planner, sizes, status strings, argument checks) and finds the plan sizes the planner oracle
gives (P = 16 causal with KVR: 58 partial slots, each device receiving R - 1 = 3 Q, KV and
partial-O partitions; the ring plan: one slot per partition and P - 1 KV partitions)."""
import os
import shutil
import subprocess

import pytest

from oracle import planner as PL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include "mesh_attn.h"

#define CHECK(call) do { int rc_ = (call); if (rc_ != MESH_ATTN_OK) { \
  printf("FAIL %s -> %d (%s)\n", #call, rc_, mesh_attn_last_error()); return 1; } } while (0)

int main(void) {
  mesh_attn_plan* plan = NULL;
  mesh_attn_plan_info info;
  int32_t* items;
  int32_t* order;
  int32_t* counts;
  int32_t* slot_off;
  int32_t i, max_q = 0, max_kv = 0, max_o = 0;
  size_t o_elems = 0, lse_elems = 0, ws = 0;
  int64_t ring_bytes = 0;

  CHECK(mesh_attn_plan_create(16384, 16, 1, 1, 1, &plan));
  CHECK(mesh_attn_plan_get_info(plan, &info));
  printf("mesh P=%d R=%d L=%lld slots=%d live=%lld\n", (int)info.P, (int)info.R, (long long)info.L,
         (int)info.n_slots, (long long)info.n_live_blocks);
  items = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)info.n_slots);
  order = (int32_t*)malloc(sizeof(int32_t) * (size_t)info.n_slots);
  counts = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)info.P);
  slot_off = (int32_t*)malloc(sizeof(int32_t) * ((size_t)info.P + 1));
  CHECK(mesh_attn_plan_order(plan, items, NULL, NULL, NULL));
  CHECK(mesh_attn_plan_launch_order(plan, order));
  CHECK(mesh_attn_plan_slots(plan, slot_off));
  CHECK(mesh_attn_plan_volumes(plan, 16, 16, 128, MESH_ATTN_BF16, counts, NULL, &ring_bytes));
  for (i = 0; i < info.P; ++i) {
    if (counts[3 * i] > max_q) max_q = counts[3 * i];
    if (counts[3 * i + 1] > max_kv) max_kv = counts[3 * i + 1];
    if (counts[3 * i + 2] > max_o) max_o = counts[3 * i + 2];
  }
  printf("recv max q=%d kv=%d o=%d ring_bytes=%lld slots_total=%d\n", (int)max_q, (int)max_kv,
         (int)max_o, (long long)ring_bytes, (int)slot_off[info.P]);
  CHECK(mesh_attn_partials_size(plan, 1, 16, 128, &o_elems, &lse_elems));
  CHECK(mesh_attn_workspace_size(plan, &ws));
  printf("partials o=%llu lse=%llu workspace=%llu\n", (unsigned long long)o_elems,
         (unsigned long long)lse_elems, (unsigned long long)ws);
  CHECK(mesh_attn_plan_destroy(plan));
  plan = NULL;

  CHECK(mesh_attn_plan_create_ring(4096, 8, 1, &plan));
  CHECK(mesh_attn_plan_get_info(plan, &info));
  printf("ring P=%d slots=%d layout=%d tile_kv=%d\n", (int)info.P, (int)info.n_slots, (int)info.layout,
         (int)info.tile_kv);
  CHECK(mesh_attn_plan_destroy(plan));

  /* argument checks come back as status codes, with a message */
  plan = NULL;
  i = mesh_attn_plan_create(1000, 16, 1, 1, 1, &plan); /* S % P != 0 */
  printf("bad S rc=%d ok=%d msg=%s\n", i, i == MESH_ATTN_ERR_INVALID_ARG, mesh_attn_last_error());
  printf("status string: %s\n", mesh_attn_status_string(MESH_ATTN_OK));
  free(items);
  free(order);
  free(counts);
  free(slot_off);
  return 0;
}
"""


def test_c_program_uses_the_abi(lib, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi_check.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(lib.LIB_PATH)
    libname = os.path.basename(lib.LIB_PATH)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), os.path.join(libdir, libname), f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    out = dict()
    for line in run.stdout.splitlines():
        key, _, rest = line.partition(" ")
        out[key] = rest
    ref = PL.make_plan(16384, 16, True, True, True)
    assert f"slots={len(ref.items)}" in out["mesh"]
    assert "P=16 R=4 L=1024" in out["mesh"]
    assert f"live={16 * 17 // 2}" in out["mesh"]  # causal: the blocks (p, k) with k <= p
    assert "max q=3 kv=3 o=3" in out["recv"]
    assert f"slots_total={len(ref.items)}" in out["recv"]
    assert "ring_bytes=" + str(15 * 2 * 1024 * 16 * 128 * 2) in out["recv"]
    assert f"o={16 * len(ref.items) * 1024 * 128} lse={16 * len(ref.items) * 1024}" in out["partials"]
    assert "P=8 slots=8 layout=1 tile_kv=8" in out["ring"]
    assert "ok=1" in out["bad"]
