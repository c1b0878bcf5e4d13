"""Invariants the GPU results must satisfy exactly, independent of the oracle: relabelling
physical pages (and remapping the block table to match) changes no output bit; a context of
one token returns that token's V row exactly; a constant V returns the constant. Covered for
the decode step (default plan) and the multi-token kernel."""

import dataclasses

import numpy as np
import pytest

from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_prefill, make_workload
from tests.gpu_util import ATOL, RTOL, run, torch

pytestmark = pytest.mark.gpu


def relabel_pages(w, seed=5):
    """The same logical cache with physical page p moved to perm[p]."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(w.num_physical_pages).astype(np.int32)
    k = np.empty_like(w.key_cache)
    v = np.empty_like(w.value_cache)
    k[perm] = w.key_cache
    v[perm] = w.value_cache
    bt = np.where(w.block_tables >= 0, perm[np.clip(w.block_tables, 0, None)], -1).astype(np.int32)
    return dataclasses.replace(w, key_cache=k, value_cache=v, block_tables=bt)


def prefill_out(p):
    t = torch()
    w = p.cache
    d = [t.from_numpy(x).cuda() for x in (p.query, p.query_start, w.key_cache, w.value_cache,
                                          w.block_tables, w.context_lengths)]
    out = t.full((p.total, w.query_heads, w.head_dim), float("nan"), dtype=t.float32,
                 device="cuda")
    lib.pa_prefill(lib.problem_of(w), d[0], d[1], p.total, p.max_query_len(), d[2], d[3], d[4],
                   d[5], w.scale, out)
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("name", ["gqa4_mid", "ragged", "long_gqa6"])
def test_decode_page_relabelling_is_bitwise_invariant(name):
    kw = dict(gqa4_mid=dict(batch=12), ragged=dict(batch=40),
              long_gqa6=dict(context_lengths=[3000, 17, 700, 1]))[name]
    w = make_workload(name, **kw)
    assert np.array_equal(run(w), run(relabel_pages(w)))


def test_prefill_page_relabelling_is_bitwise_invariant():
    p = make_prefill("prefill_chunked", context_lengths=[300, 77, 513, 129],
                     new_tokens=[300, 10, 200, 129], max_pages_per_sequence=64)
    q = dataclasses.replace(p, cache=relabel_pages(p.cache))
    assert np.array_equal(prefill_out(p), prefill_out(q))


@pytest.mark.parametrize("name", ["tiny", "gqa4_mid", "long_gqa6"])
def test_decode_context_one_returns_the_v_row(name):
    w = make_workload(name, context_lengths=[1] * 6, max_pages_per_sequence=2)
    out = run(w)
    g = w.query_heads // w.kv_heads
    for b in range(w.batch):
        page = int(w.block_tables[b, 0])
        for h in range(w.query_heads):
            assert np.array_equal(out[b, h], w.value_cache[page, 0, h // g].astype(np.float32))


def test_prefill_first_token_of_a_prompt_returns_its_v_row():
    p = make_prefill("prefill_chunked", context_lengths=[90, 300, 33],
                     new_tokens=[90, 300, 33], max_pages_per_sequence=32)
    out = prefill_out(p)
    w = p.cache
    g = w.query_heads // w.kv_heads
    for b in range(w.batch):
        page = int(w.block_tables[b, 0])
        for h in range(w.query_heads):
            assert np.array_equal(out[int(p.query_start[b]), h],
                                  w.value_cache[page, 0, h // g].astype(np.float32))


def test_constant_v_returns_the_constant():
    w = make_workload("gqa4_mid", batch=8)
    w = dataclasses.replace(w, value_cache=np.full_like(w.value_cache, np.float16(0.375)))
    out = run(w)
    assert np.abs(out - 0.375).max() <= ATOL + RTOL * 0.375
    p = make_prefill("prefill_chunked", context_lengths=[300, 77], new_tokens=[300, 10],
                     max_pages_per_sequence=32)
    p = dataclasses.replace(p, cache=dataclasses.replace(
        p.cache, value_cache=np.full_like(p.cache.value_cache, np.float16(-1.25))))
    got = prefill_out(p)
    assert np.abs(got + 1.25).max() <= ATOL + RTOL * 1.25
