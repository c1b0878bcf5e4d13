"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Small cases span several K/V tiles with ragged tails, every head-group shape the library
handles (g = 1, 2, 3, 4, 6, 8, 12), page sizes 8..256 and empty contexts; every case runs
through both arithmetic variants and every schedule. Full-size workloads run in the
benchmark's launch configuration (pa_decode's plan) and are compared on every output element."""

import numpy as np
import pytest

from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_workload
from tests.gpu_util import assert_close, run, to_device

pytestmark = pytest.mark.gpu


def _cases():
    return {
        "tiny": lambda: make_workload("tiny"),
        "mid_small": lambda: make_workload(
            "gqa4_mid", context_lengths=[1, 15, 16, 17, 31, 32, 33, 100, 513, 1000, 2049, 4096]),
        "mha_small": lambda: make_workload("mha", context_lengths=[2048, 1, 7, 300]),
        "long_small": lambda: make_workload("long_gqa6", context_lengths=[5000, 100, 64, 65]),
        "ragged_small": lambda: make_workload("ragged", batch=24),
        "g12": lambda: make_workload("gqa4_mid", query_heads=24, kv_heads=2,
                                     context_lengths=[50, 700, 33]),
        "g3_hd64_ps8": lambda: make_workload("tiny", query_heads=6, kv_heads=2, page_size=8,
                                             context_lengths=[9, 40, 333]),
        "ps256": lambda: make_workload("gqa4_mid", page_size=256,
                                       context_lengths=[1, 255, 256, 257, 1000]),
        "empty_ctx": lambda: make_workload("tiny", context_lengths=[0, 40, 0, 3]),
        "g8_hd256": lambda: make_workload("long_gqa6", query_heads=32, kv_heads=4,
                                          context_lengths=[700, 2]),
    }


CASES = _cases()
_cache = {}


def case(name):
    if name not in _cache:
        import oracle

        w = CASES[name]()
        _cache[name] = (w, oracle.decode(w))
    return _cache[name]


OPTS = {
    "mma-single": dict(math="mma", schedule="single"),
    "mma-balanced": dict(math="mma", schedule="balanced"),
    "mma-balanced-w7": dict(math="mma", schedule="balanced", workers=7),
    "mma-balanced-kernel": dict(math="mma", schedule="balanced", combine="kernel", workers=13),
    "simt-single": dict(math="simt", schedule="single"),
    "simt-balanced": dict(math="simt", schedule="balanced"),
    "simt-balanced-w7": dict(math="simt", schedule="balanced", workers=7),
    "simt-balanced-kernel": dict(math="simt", schedule="balanced", combine="kernel", workers=13),
}


@pytest.mark.parametrize("opt", sorted(OPTS))
@pytest.mark.parametrize("name", sorted(CASES))
def test_small_parity(name, opt):
    w, ref = case(name)
    got = run(w, opts=lib.options(**OPTS[opt]))
    assert_close(got, ref, f"{name}/{opt}")
    zero = w.context_lengths == 0
    assert not got[zero].any()


@pytest.mark.parametrize("name", sorted(CASES))
def test_default_entry_point(name):
    w, ref = case(name)
    assert_close(run(w), ref, name)


def test_stage_and_warp_options():
    w, ref = case("mid_small")
    for stages, warps in ((1, 1), (2, 3), (5, 2), (8, 1), (3, 4)):
        got = run(w, opts=lib.options(stages=stages, warps_per_cta=warps))
        assert_close(got, ref, f"stages={stages} warps={warps}")
    # a pipeline that does not fit in shared memory is refused, not launched
    assert lib.status_of(run, w, None, lib.options(stages=8, warps_per_cta=8)) == 2


def warps_per_pair(units, workers):
    """The library's choice of warps per (unit, head) pair in the separate combine kernel:
    enough that each warp walks at most about 8 of the 1 + workers / units contributors."""
    avg = 1 + workers // max(units, 1)
    w = 1
    while w < 8 and avg > 8 * w:
        w *= 2
    return w


@pytest.mark.parametrize("avg", [5, 12, 20, 40])
@pytest.mark.parametrize("name", ["mid_small", "long_small", "g3_hd64_ps8", "g12", "empty_ctx"])
def test_combine_kernel_warps_per_pair(name, avg):
    """The separate combine kernel with 1, 2, 4 and 8 warps per (unit, head) pair: worker
    counts chosen so units have about 5, 12, 20 and 40 contributors."""
    w, ref = case(name)
    units = lib.pa_plan(lib.problem_of(w))["units"]
    o = lib.options(math="mma", schedule="balanced", combine="kernel", workers=units * (avg - 1))
    pl = lib.pa_plan(lib.problem_of(w), o)
    assert pl["combine"] == 2
    assert warps_per_pair(pl["units"], pl["workers"]) == {5: 1, 12: 2, 20: 4, 40: 8}[avg]
    got = run(w, opts=o)
    assert_close(got, ref, f"{name}/avg{avg}")
    assert not got[w.context_lengths == 0].any()
    assert np.array_equal(got, run(w, opts=o))


FULL = ["tiny", "gqa4_mid", "mha", "long_gqa6", "ragged"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name):
    """Full-size workload in the benchmark's launch configuration (pa_decode's plan): every
    element of [batch][query_heads][head_dim] against the oracle."""
    import oracle

    w = make_workload(name)
    d = to_device(w)
    got = run(w, d)
    assert_close(got, oracle.decode(w), name)
    # a second call gives the same bits
    assert np.array_equal(got, run(w, d))
    # sequences of length 1 return their single V row exactly
    g = w.query_heads // w.kv_heads
    for b in np.nonzero(w.context_lengths == 1)[0]:
        page = w.block_tables[b, 0]
        for h in range(w.query_heads):
            v = w.value_cache[page, 0, h // g].astype(np.float32)
            assert np.array_equal(got[b, h], v)


HD128 = ["mid_small", "mha_small", "ragged_small", "g12", "ps256"]


@pytest.mark.parametrize("opt", ["mma-single", "mma-balanced", "simt-balanced-kernel"])
@pytest.mark.parametrize("name", HD128)
def test_tile16_parity(name, opt):
    """head_dim 128 with 16-token tiles (the other instantiated tile size)."""
    w, ref = case(name)
    got = run(w, opts=lib.options(tile_tokens=16, **OPTS[opt]))
    assert_close(got, ref, f"{name}/{opt}/t16")
    assert lib.status_of(lib.pa_plan, lib.problem_of(make_workload("long_gqa6")),
                         lib.options(tile_tokens=32)) == 2


@pytest.mark.parametrize("opt", ["mma-single", "mma-balanced", "mma-balanced-kernel", "simt-balanced-w7"])
@pytest.mark.parametrize("name", ["tiny", "mid_small", "long_small", "ragged_small", "g12",
                                  "g3_hd64_ps8", "empty_ctx"])
def test_head_major_parity(name, opt):
    """The [page][kv_head][slot][head_dim] cache layout (the oracle gives the same result for
    both layouts, exactly)."""
    from paged_kv_cache_63_gb300.workloads import to_head_major

    w, ref = case(name)
    assert_close(run(to_head_major(w), opts=lib.options(**OPTS[opt])), ref, f"{name}/{opt}/hm")


@pytest.mark.parametrize("name", ["gqa4_mid", "mha"])
def test_head_major_full_size_every_element(name):
    import oracle
    from paged_kv_cache_63_gb300.workloads import to_head_major

    w = to_head_major(make_workload(name))
    assert_close(run(w), oracle.decode(w), name)
