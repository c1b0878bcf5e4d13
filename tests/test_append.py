"""pa_append_kv (the cache write before a decode step) against the oracle: the caches after
the append must be identical bit for bit, in both cache layouts."""

import dataclasses

import numpy as np
import pytest

from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_workload, to_head_major
from tests.gpu_util import assert_close, run, to_device, torch

pytestmark = pytest.mark.gpu


def room_for_one_more(w):
    """The same workload with a free page mapped wherever a sequence's next token starts a
    new page (so every sequence can append one token)."""
    bt = w.block_tables.copy()
    extra = 0
    for b in range(w.batch):
        t = int(w.context_lengths[b])
        lp = t // w.page_size
        if lp < w.max_pages_per_sequence and bt[b, lp] < 0:
            bt[b, lp] = w.num_physical_pages + extra
            extra += 1
    pad = ((0, extra), (0, 0), (0, 0), (0, 0))
    k = np.pad(w.key_cache, pad)
    v = np.pad(w.value_cache, pad)
    return dataclasses.replace(w, block_tables=bt, key_cache=k, value_cache=v,
                               num_physical_pages=w.num_physical_pages + extra)


def new_rows(w, seed=17):
    rng = np.random.default_rng(seed)
    shape = (w.batch, w.kv_heads, w.head_dim)
    return (rng.standard_normal(shape).astype(np.float16),
            rng.standard_normal(shape).astype(np.float16))


def gpu_append(w, nk, nv):
    t = torch()
    d = to_device(w)
    lib.pa_append_kv(lib.problem_of(w), t.from_numpy(nk).cuda(), t.from_numpy(nv).cuda(), d["bt"],
                     d["ctx"], d["k"], d["v"])
    t.cuda.synchronize()
    return d["k"].cpu().numpy(), d["v"].cpu().numpy(), lib.pa_get_device_error()


CASES = {
    "tiny": lambda: make_workload("tiny"),
    "mid": lambda: make_workload("gqa4_mid", batch=12),
    "long": lambda: make_workload("long_gqa6", context_lengths=[4000, 63, 64, 1]),
    "ragged": lambda: make_workload("ragged", batch=40),
    "ps8": lambda: make_workload("tiny", page_size=8, context_lengths=[0, 7, 8, 9]),
}


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("name", sorted(CASES))
def test_append_bit_exact(name, layout):
    import oracle

    w = room_for_one_more(CASES[name]())
    if layout:
        w = to_head_major(w)
    nk, nv = new_rows(w)
    ek, ev, eflags = oracle.append_kv(w, nk, nv)
    k, v, flags = gpu_append(w, nk, nv)
    assert flags == 0 and eflags == 0
    assert np.array_equal(k.view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(v.view(np.uint16), ev.view(np.uint16))


def test_append_flags_and_skips_bad_sequences():
    import oracle

    w = room_for_one_more(make_workload("gqa4_mid", batch=6))
    ctx = w.context_lengths.copy()
    ctx[1] = w.max_pages_per_sequence * w.page_size  # no room in the table
    ctx[2] = -4
    bt = w.block_tables.copy()
    t3 = int(ctx[3])
    bt[3, t3 // w.page_size] = w.num_physical_pages + 9  # outside the pool
    w = dataclasses.replace(w, context_lengths=ctx, block_tables=bt)
    nk, nv = new_rows(w)
    ek, ev, eflags = oracle.append_kv(w, nk, nv)
    k, v, flags = gpu_append(w, nk, nv)
    assert flags & lib.PA_DEVERR_CONTEXT and flags & lib.PA_DEVERR_PAGE_ID
    assert eflags == 3
    assert np.array_equal(k.view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(v.view(np.uint16), ev.view(np.uint16))


@pytest.mark.parametrize("layout", [0, 1])
def test_append_then_decode(layout):
    """A decode step as a serving loop runs it: append the new token's K/V, then decode with
    every length one longer -- against the oracle doing the same."""
    import oracle

    t = torch()
    w = room_for_one_more(make_workload("ragged", batch=24))
    if layout:
        w = to_head_major(w)
    nk, nv = new_rows(w, seed=5)
    ek, ev, _ = oracle.append_kv(w, nk, nv)
    w1 = dataclasses.replace(w, key_cache=ek, value_cache=ev, context_lengths=w.context_lengths + 1)
    ref = oracle.decode(w1)
    d = to_device(w)
    prob = lib.problem_of(w)
    lib.pa_append_kv(prob, t.from_numpy(nk).cuda(), t.from_numpy(nv).cuda(), d["bt"], d["ctx"],
                     d["k"], d["v"])
    d["ctx"] += 1
    lib.pa_decode(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"])
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    assert_close(d["out"].cpu().numpy(), ref, "append+decode")
