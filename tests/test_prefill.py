"""pa_prefill (causal multi-token attention on the tcgen05 tensor cores) against the fp64
oracle: every element of small cases that span several query and key tiles with ragged
tails, every element of the full-size workloads, both cache layouts, and the edge and error
cases (sequences without new tokens, one new token, page sizes below and above the key tile,
a grid taller than needed, bad offsets, bad pages, an expired wait)."""

import dataclasses

import numpy as np
import pytest

import oracle
from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_prefill, to_head_major
from tests.gpu_util import assert_close, torch

pytestmark = pytest.mark.gpu


def gpu_prefill(p, max_query_len=None, extra_rows=0, opts=None, query_start=None,
                check_errors=True):
    """Run pa_prefill; output rows past the new tokens stay NaN (they must be untouched)."""
    t = torch()
    w = p.cache
    qs = p.query_start if query_start is None else query_start
    total = p.total + extra_rows
    q = np.zeros((total, w.query_heads, w.head_dim), dtype=np.float16)
    q[:p.total] = p.query
    d_q = t.from_numpy(q).cuda()
    d_qs = t.from_numpy(np.ascontiguousarray(qs, dtype=np.int32)).cuda()
    d_k = t.from_numpy(w.key_cache).cuda()
    d_v = t.from_numpy(w.value_cache).cuda()
    d_bt = t.from_numpy(w.block_tables).cuda()
    d_ctx = t.from_numpy(w.context_lengths).cuda()
    out = t.full((total, w.query_heads, w.head_dim), float("nan"), dtype=t.float32, device="cuda")
    mq = p.max_query_len() if max_query_len is None else max_query_len
    lib.pa_prefill(lib.problem_of(w), d_q, d_qs, total, mq, d_k, d_v, d_bt, d_ctx, w.scale, out,
                   opts)
    t.cuda.synchronize()
    flags = lib.pa_get_device_error()
    if check_errors:
        assert flags == 0, f"device error flags {flags}"
    return out.cpu().numpy(), flags


def with_layout(p, layout):
    return dataclasses.replace(p, cache=to_head_major(p.cache)) if layout else p


CASES = {
    # hd 64, g 2 (32 tokens per query tile), one fresh prompt and one chunk on a prefix
    "tiny": lambda: make_prefill("prefill_tiny"),
    # hd 128, g 4: ragged new-token counts, empty and single-token sequences, prefixes
    "gqa4_ragged": lambda: make_prefill(
        "prefill_chunked", context_lengths=[300, 77, 513, 1, 129, 1000],
        new_tokens=[300, 10, 200, 1, 0, 129], max_pages_per_sequence=64),
    # hd 128, g 1 (128 tokens per query tile)
    "mha": lambda: make_prefill("prefill_mha", context_lengths=[257, 140]),
    # hd 256, g 6 (21 tokens, 126 of 128 rows), page 64, 64-token key tiles
    "hd256_g6": lambda: make_prefill(
        "prefill_chunked", context_lengths=[700, 65, 128], new_tokens=[700, 65, 30],
        query_heads=24, kv_heads=4, head_dim=256, page_size=64, k_scale=0.5,
        max_pages_per_sequence=16),
    # page size 8: sixteen boxes per key tile
    "ps8": lambda: make_prefill("prefill_chunked", context_lengths=[200, 33],
                                new_tokens=[150, 33], page_size=8, max_pages_per_sequence=32),
    # page size 256: one box covers two key tiles' worth of page
    "ps256": lambda: make_prefill("prefill_chunked", context_lengths=[600, 300],
                                  new_tokens=[200, 300], page_size=256,
                                  max_pages_per_sequence=4, spare_pages=2),
    # g 6 with head_dim 128 (21 tokens, 126 of 128 rows; g does not divide a warp's 32 rows,
    # so every row is stored directly)
    "g6_hd128": lambda: make_prefill("prefill_chunked", context_lengths=[300, 50],
                                     new_tokens=[300, 50], query_heads=48, kv_heads=8,
                                     max_pages_per_sequence=32),
    # g 8 (16 tokens per query tile), hd 128
    "g8": lambda: make_prefill("prefill_chunked", context_lengths=[180, 40],
                               new_tokens=[180, 17], query_heads=64, kv_heads=8,
                               max_pages_per_sequence=16),
}


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name, layout):
    p = with_layout(CASES[name](), layout)
    got, _ = gpu_prefill(p)
    ref = oracle.prefill(p.cache, p.query, p.query_start)
    assert_close(got, ref, f"{name}/layout{layout}")


def test_prefill_grid_taller_than_needed_and_untouched_rows():
    """max_query_len above every n_b adds query tiles that exit at once; rows past the last
    new token are never written."""
    p = CASES["gqa4_ragged"]()
    got, _ = gpu_prefill(p, max_query_len=p.max_query_len() + 300, extra_rows=5)
    assert np.isnan(got[p.total:]).all()
    assert_close(got[:p.total], oracle.prefill(p.cache, p.query, p.query_start), "tall grid")


@pytest.mark.parametrize("head_dim", [128, 256])  # the two-tile and the single-tile kernel
def test_prefill_rescale_path(head_dim):
    """Keys that grow along the sequence push each row's running maximum up by far more than
    2^8 after the first key tile, so O is rescaled in TMEM many times, and full key tiles whose
    exponents were first taken with the old maximum are taken again."""
    extra = dict(query_heads=24, kv_heads=4, head_dim=256, page_size=64) if head_dim == 256 else {}
    p = make_prefill("prefill_chunked", context_lengths=[900, 520], new_tokens=[900, 300],
                     max_pages_per_sequence=64, **extra)
    w = p.cache
    k = w.key_cache.astype(np.float32)
    for b in range(w.batch):
        for tok in range(int(w.context_lengths[b])):
            page, slot = int(w.block_tables[b, tok // w.page_size]), tok % w.page_size
            k[page, slot] *= 1.0 + tok / 64.0
    k = np.clip(k, -60000, 60000).astype(np.float16)
    p = dataclasses.replace(p, cache=dataclasses.replace(w, key_cache=k))
    got, _ = gpu_prefill(p)
    assert_close(got, oracle.prefill(p.cache, p.query, p.query_start), "rescale")


@pytest.mark.parametrize("scale", [0.0, -0.07])
def test_prefill_zero_and_negative_scale(scale):
    """A zero scale averages V over the visible keys; a negative one flips the softmax (the
    row maximum then comes from the smallest raw score)."""
    p = CASES["gqa4_ragged"]()
    p = dataclasses.replace(p, cache=dataclasses.replace(p.cache, scale=scale))
    got, _ = gpu_prefill(p)
    assert_close(got, oracle.prefill(p.cache, p.query, p.query_start, scale=scale),
                 f"scale {scale}")


def test_prefill_one_token_matches_decode():
    """One new token per sequence gives the decode step's result (both through the GPU)."""
    from tests.gpu_util import run
    from paged_kv_cache_63_gb300.workloads import make_workload, Prefill

    w = make_workload("gqa4_mid", batch=6)
    p = Prefill(cache=w, query=w.query.copy(),
                query_start=np.arange(w.batch + 1, dtype=np.int32))
    got, _ = gpu_prefill(p)
    dec = run(w)
    assert_close(got, oracle.prefill(w, p.query, p.query_start), "one token")
    assert np.abs(got - dec).max() < 4e-3


@pytest.mark.parametrize("name", ["prefill_gqa4", "prefill_chunked", "prefill_mha",
                                  "prefill_gqa6_hd256"])
def test_prefill_full_size_every_element(name):
    p = make_prefill(name)
    got, _ = gpu_prefill(p)
    assert_close(got, oracle.prefill(p.cache, p.query, p.query_start), name)


@pytest.mark.parametrize("name,ctx", [("prefill_gqa4", [2048] * 2),          # 512 work items
                                      ("prefill_gqa6_hd256", [4096])])       # 784 work items
def test_prefill_resident_ctas_are_bitwise_deterministic(name, ctx):
    """More work items than SMs: resident CTAs take over the items of CTAs that have not
    started, in whatever order they ask, so which CTA computes which item changes from call
    to call; an item's arithmetic does not depend on it, so every call gives the same bits."""
    p = make_prefill(name, context_lengths=ctx)
    outs = [gpu_prefill(p)[0] for _ in range(3)]
    assert np.isfinite(outs[0]).all()
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


@pytest.mark.parametrize("name", ["tiny", "hd256_g6"])  # the two-tile and the single-tile kernel
def test_prefill_bad_offsets_flagged(name):
    p = CASES[name]()
    qs = p.query_start.copy()
    qs[1] = qs[2] + 1  # decreasing offsets
    _, flags = gpu_prefill(p, query_start=qs, check_errors=False)
    assert flags & lib.PA_DEVERR_QUERY_START
    # the device is still usable
    got, _ = gpu_prefill(p)
    assert_close(got, oracle.prefill(p.cache, p.query, p.query_start), "after bad offsets")


@pytest.mark.parametrize("name", ["tiny", "hd256_g6"])
def test_prefill_bad_page_flagged(name):
    p = CASES[name]()
    bt = p.cache.block_tables.copy()
    bt[0, 1] = p.cache.num_physical_pages + 3  # a page every sequence-0 query reads
    bad = dataclasses.replace(p, cache=dataclasses.replace(p.cache, block_tables=bt))
    _, flags = gpu_prefill(bad, check_errors=False)
    assert flags & lib.PA_DEVERR_PAGE_ID


@pytest.mark.parametrize("name", ["tiny", "hd256_g6"])
def test_prefill_expired_wait_reports_timeout(name):
    """A wait that runs out raises PA_DEVERR_TIMEOUT; the kernel drains and frees its tensor
    memory, so the next call on the same device is correct."""
    p = CASES[name]()
    opts = lib.options(test_flags=lib.PA_TEST_EXPIRE_WAITS)
    _, flags = gpu_prefill(p, opts=opts, check_errors=False)
    assert flags & lib.PA_DEVERR_TIMEOUT
    got, _ = gpu_prefill(p)
    assert_close(got, oracle.prefill(p.cache, p.query, p.query_start), "after timeout")


def test_prefill_rejects_bad_arguments():
    """Argument checks run on the host before any launch (1 = invalid argument, 3 = misaligned)."""
    t = torch()
    p = CASES["tiny"]()
    w = p.cache
    prob = lib.problem_of(w)
    buf = t.zeros(1 << 16, dtype=t.float32, device="cuda")
    qs = t.from_numpy(p.query_start).cuda()
    ok_args = (buf, qs, p.total, 37, buf, buf, qs, qs, w.scale, buf)
    assert lib.status_of(lib.pa_prefill, prob, *ok_args[:2], -1, *ok_args[3:]) == 1
    assert lib.status_of(lib.pa_prefill, prob, *ok_args[:3], -1, *ok_args[4:]) == 1
    assert lib.status_of(lib.pa_prefill, prob, *ok_args[:8], float("nan"), buf) == 1
    assert lib.status_of(lib.pa_prefill, prob, buf[1:], *ok_args[1:]) == 3
    assert lib.status_of(lib.pa_prefill, prob, *ok_args, lib.options(workers=3)) == 1
