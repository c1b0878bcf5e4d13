"""The C-ABI library on the host: it loads, exports every declared entry point, validates
arguments before touching a GPU, and plans work (pure host logic). No kernel runs here."""

import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_63_gb300 import lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:const char \*|pa_status_t |int32_t )(pa_[a-z_]+)\(", text,
                                 re.M)))


def test_header_declares_binding_exports():
    assert declared_entry_points() == sorted(lib.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib.load()
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (pa_[a-z_]+)$", out, re.M))
    for name in declared_entry_points():
        assert name in exported, name
        assert hasattr(lib.load(), name)


def test_header_compiles_as_c_and_a_c_program_links(tmp_path):
    """A C99 program includes the header alone, links the library and plans a problem on the
    host (no device needed for planning)."""
    lib.load()
    src = tmp_path / "use.c"
    src.write_text(r'''
#include <stdio.h>
#include "pagedattn.h"
int main(void) {
  pa_problem_t p = {4, 32, 8, 128, 16, 256, 1024, PA_LAYOUT_TOKEN_MAJOR};
  pa_plan_t plan;
  pa_status_t st = pa_plan(&p, NULL, 152, &plan);
  if (st != PA_OK) { printf("%s\n", pa_status_string(st)); return 1; }
  size_t ws = 0;
  st = pa_workspace_size(&p, NULL, &ws);
  printf("%d %d %d %d\n", (int)st, plan.warps_per_cta, plan.stages, pa_version() > 0);
  return 0;
}
''')
    exe = tmp_path / "use"
    build_dir = os.path.dirname(lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                    os.path.join(ROOT, "include"), str(src), "-L", build_dir, "-lpagedattn",
                    "-Wl,-rpath," + build_dir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    st, warps, stages, ver = map(int, r.stdout.split())
    assert warps == 8 and stages >= 1 and ver == 1
    assert st in (0, 6)  # the workspace size needs the device's SM count: none here


def test_version_and_status_strings():
    assert lib.pa_version() >= 100
    assert lib.pa_status_string(0) == "ok"
    assert "workspace" in lib.pa_status_string(4)
    assert lib.pa_status_string(99) == "unknown status"


def P(**kw):
    base = dict(batch=4, query_heads=32, kv_heads=8, head_dim=128, page_size=16,
                max_pages_per_sequence=256, num_physical_pages=1024)
    base.update(kw)
    return lib.problem(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(query_heads=30), 1),
    (dict(kv_heads=0), 1),
    (dict(batch=-1), 1),
    (dict(head_dim=96), 2),
    (dict(head_dim=512), 2),
    (dict(page_size=12), 2),
    (dict(page_size=4), 2),
    (dict(page_size=512), 2),
    (dict(num_physical_pages=1 << 27), 2),
    (dict(max_pages_per_sequence=0), 1),
    (dict(cache_layout=2), 1),
    (dict(cache_layout=1, num_physical_pages=1 << 27, page_size=8, kv_heads=16), 2),
])
def test_plan_rejects_bad_problems(kw, status):
    assert lib.status_of(lib.pa_plan, P(**kw)) == status


def test_plan_rejects_bad_options():
    assert lib.status_of(lib.pa_plan, P(), lib.options(schedule=7)) == 1
    assert lib.status_of(lib.pa_plan, P(), lib.options(stages=99)) == 1
    assert lib.status_of(lib.pa_plan, P(), lib.options(test_flags=2)) == 1
    assert lib.status_of(lib.pa_plan, P(), lib.options(tile_tokens=-1)) == 1
    assert lib.status_of(lib.pa_plan, P(), None, 0) == 1


def test_plan_groups_and_units():
    pl = lib.pa_plan(P(query_heads=24, kv_heads=4, head_dim=256, page_size=64))
    assert pl["heads_per_unit"] == 6 and pl["units"] == 4 * 4
    pl = lib.pa_plan(P(query_heads=96, kv_heads=8))  # g = 12 -> two units of 6 heads per K/V head
    assert pl["heads_per_unit"] == 6 and pl["units"] == 4 * 8 * 2
    pl = lib.pa_plan(P(query_heads=8, kv_heads=8))
    assert pl["heads_per_unit"] == 1


def test_plan_shared_memory_fits_and_tiles():
    for hd in (64, 128, 256):
        for math in ("simt", "mma"):
            pl = lib.pa_plan(P(head_dim=hd, query_heads=64, kv_heads=8), lib.options(math=math))
            assert pl["smem_bytes"] <= 232448
            assert pl["tile_tokens"] == (32 if hd == 64 else 16)
            assert 1 <= pl["warps_per_cta"] <= 8 and pl["stages"] >= 1


def test_plan_keeps_eight_warps_with_up_to_24_kb_in_flight():
    """The default ring: 24 KB of K/V per warp (three 8 KB stages) where eight warps still
    fit, else 16 KB; never fewer than eight warps per CTA for these shapes."""
    for hd, stages in ((64, 3), (128, 3), (256, 1)):
        pl = lib.pa_plan(P(head_dim=hd, query_heads=32, kv_heads=8), lib.options(math="mma"))
        assert pl["warps_per_cta"] == 8
        assert pl["stages"] == stages
        assert 16384 <= pl["stages"] * pl["tile_tokens"] * hd * 4 <= 24576


def test_plan_heuristic():
    # long contexts on few units: balanced split-K with one full wave of workers
    pl = lib.pa_plan(P(batch=4, query_heads=24, kv_heads=4, head_dim=256, page_size=64,
                       max_pages_per_sequence=1563, num_physical_pages=6252), sm_count=152)
    assert pl["schedule"] == 2 and pl["workers"] == 152 * pl["warps_per_cta"]
    assert pl["workspace_bytes"] > 0
    # many short units: one worker per unit, no workspace
    pl = lib.pa_plan(P(batch=4096, max_pages_per_sequence=32, num_physical_pages=4096 * 32))
    assert pl["schedule"] == 1 and pl["workspace_bytes"] == 0 and pl["workers"] == 4096 * 8
    # forced options are honoured
    pl = lib.pa_plan(P(), lib.options(schedule="balanced", workers=7, combine="kernel"))
    assert (pl["schedule"], pl["combine"]) == (2, 2)
    assert pl["workers"] % pl["group"] == 0 and 7 <= pl["workers"] < 7 + pl["group"]
    # many workers per unit: the separate combine kernel; few: the fused merge
    pl = lib.pa_plan(P(batch=4, query_heads=24, kv_heads=4, head_dim=256, page_size=64,
                       max_pages_per_sequence=1563, num_physical_pages=6252))
    assert pl["combine"] == 2
    assert lib.pa_plan(P(batch=256, query_heads=64, kv_heads=8))["combine"] == 1
    assert lib.pa_plan(P(batch=32, query_heads=32, kv_heads=8))["combine"] == 2


def test_workspace_bytes_cover_slots():
    pl = lib.pa_plan(P(), lib.options(schedule="balanced", workers=100))
    units = pl["units"]
    need = (units + 100) * 8 * (128 + 2) * 4 + units * 4
    assert pl["workspace_bytes"] >= need


def test_decode_validates_before_touching_a_gpu():
    """Bad arguments are refused with a status; valid ones fail only at device lookup."""
    prob = P()
    good = 1 << 20  # a fake, 16-byte aligned address that is never dereferenced
    args = [good, good, good, good, good, 0.1, good]
    assert lib.status_of(lib.pa_decode, prob, *args) in (5, 6)  # no device here
    bad = list(args)
    bad[0] = None
    assert lib.status_of(lib.pa_decode, prob, *bad) == 1
    bad = list(args)
    bad[1] = good + 8
    assert lib.status_of(lib.pa_decode, prob, *bad) == 3
    bad = list(args)
    bad[5] = float("nan")
    assert lib.status_of(lib.pa_decode, prob, *bad) == 1
    assert lib.status_of(lib.pa_decode, P(head_dim=80), *args) == 2
    assert lib.status_of(lib.pa_decode_ex, prob, *args, lib.options(schedule=9)) == 1
    assert lib.status_of(lib.pa_split_kv_partial, prob, *args[:6], 0, good, good, good) == 1
    assert lib.status_of(lib.pa_split_kv_combine, prob, 0, good, good, good, good) == 1
    assert lib.status_of(lib.pa_decode, lib.problem(0, 4, 2, 64, 16, 8, 16), *args) == 0


def test_prefill_validates_before_touching_a_gpu():
    """pa_prefill refuses bad arguments with a status before any device work; valid ones fail
    only at device lookup here."""
    prob = P()
    good = 1 << 20
    # query, query_start, total_tokens, max_query_len, k, v, bt, ctx, scale, out
    args = [good, good, 100, 50, good, good, good, good, 0.1, good]
    assert lib.status_of(lib.pa_prefill, prob, *args) in (5, 6)
    for i, bad_value, status in [(0, None, 1), (1, None, 1), (2, -1, 1), (3, -1, 1),
                                 (8, float("inf"), 1), (0, good + 8, 3), (9, good + 4, 3),
                                 (1, good + 2, 3)]:
        bad = list(args)
        bad[i] = bad_value
        assert lib.status_of(lib.pa_prefill, prob, *bad) == status, (i, bad_value)
    assert lib.status_of(lib.pa_prefill, P(head_dim=80), *args) == 2
    assert lib.status_of(lib.pa_prefill, prob, *args, lib.options(stages=2)) == 1
    # nothing to do is not an error
    assert lib.status_of(lib.pa_prefill, lib.problem(0, 4, 2, 64, 16, 8, 16), *args) == 0
    zero_tokens = list(args)
    zero_tokens[2] = 0
    assert lib.status_of(lib.pa_prefill, prob, *zero_tokens) == 0


def test_schedule_arithmetic(tmp_path):
    """The balanced schedule's tile split (internal.h): every tile of every unit belongs to
    exactly one worker, worker_of inverts worker_start, and slots are unique per
    (unit, worker) pair and below units + workers."""
    src = tmp_path / "sched.cpp"
    src.write_text(r'''
#include <cstdio>
#include <cstdlib>
#include <set>
#include <vector>
#include "internal.h"
using namespace pa;
int main() {
  srand(7);
  for (int trial = 0; trial < 400; ++trial) {
    // G warps per worker serve G consecutive units; units = group units * G
    int batch = 1 + rand() % 40, G = 1 << (rand() % 3), upg = 1 + rand() % 5, T = (rand() % 2) ? 16 : 32;
    int ups = upg * G;
    int workers = 1 + rand() % 700;
    std::vector<int> ctx(batch);
    for (auto &c : ctx) c = (rand() % 4 == 0) ? 0 : 1 + rand() % 3000;
    long long total = 0;
    std::vector<long long> u0, u1;  // tile range of each group unit
    for (int b = 0; b < batch; ++b)
      for (int u = 0; u < upg; ++u) {
        u0.push_back(total);
        total += tiles_of(ctx[b], T);
        u1.push_back(total);
      }
    if (total == 0) continue;
    if (workers > total) workers = (int)total;  // the kernel caps workers at the tile count
    std::vector<int> owner(total, -1);
    for (long long c = 0; c < workers; ++c) {
      if (worker_start(c + 1, total, workers) <= worker_start(c, total, workers)) {
        printf("empty range\n"); return 1; }
      for (long long x = worker_start(c, total, workers); x < worker_start(c + 1, total, workers); ++x) {
        if (owner[x] != -1) { printf("tile %lld owned twice\n", x); return 1; }
        owner[x] = (int)c;
      }
    }
    for (long long x = 0; x < total; ++x) {
      if (owner[x] < 0) { printf("tile %lld unowned\n", x); return 1; }
      if (worker_of(x, total, workers) != owner[x]) { printf("worker_of wrong\n"); return 1; }
    }
    std::set<long long> slots;
    const long long units = (long long)u0.size() * G;
    for (size_t gu = 0; gu < u0.size(); ++gu) {
      if (u0[gu] == u1[gu]) continue;
      long long c0 = worker_of(u0[gu], total, workers), c1 = worker_of(u1[gu] - 1, total, workers);
      for (long long c = c0; c <= c1; ++c) {
        // every worker from the first to the last holds tiles of this group unit
        if (worker_start(c, total, workers) >= u1[gu] || worker_start(c + 1, total, workers) <= u0[gu]) {
          printf("gap in contributors\n"); return 1; }
        for (int m = 0; m < G; ++m) {
          long long s = slot_of((long long)gu * G + m, c, G);
          if (!slots.insert(s).second || s >= units + (long long)workers * G) {
            printf("slot clash\n"); return 1; }
        }
      }
    }
  }
  // warps per (unit, head) pair of the separate combine: at most ~8 contributors per warp
  const long long wp[][3] = {{256, 1216, 1}, {16, 1216, 8}, {96, 1056, 2}, {96, 1824, 4},
                             {96, 672, 1}, {96, 768, 2}, {1, 0, 1}, {0, 5, 1}, {4, 100000, 8}};
  for (const auto &c : wp)
    if (combine_warps_per_pair(c[0], c[1]) != c[2]) {
      printf("warps per pair %lld %lld\n", c[0], c[1]); return 1; }
  printf("ok\n");
  return 0;
}
''')
    exe = tmp_path / "sched"
    csrc = os.path.join(ROOT, "paged_kv_cache_63_gb300", "csrc")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", csrc, "-I", os.path.join(ROOT, "include"),
                    "-I", "/usr/local/cuda/include", str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout
