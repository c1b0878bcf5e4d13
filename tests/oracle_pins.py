"""Pins that tie the fp64 oracle to facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the oracle
disagrees with an independent fact: the pages' printed block-table sketch, closed forms,
invariants of softmax attention, a brute-force evaluation written separately in plain
Python (``math.fsum``), and numpy's own binary16 widening. ``tests/test_oracle.py``
runs them against the oracle; ``tests/test_oracle_mutants.py`` runs them against
deliberately broken copies of the oracle to show each plausible mistake is caught.

The method ("[TIL] Optimizing paged attention", sections "Paged Attention",
"Data Layout" and "Baseline"): for sequence b and query head h,
kv = h // (query_heads // kv_heads); token t lives at physical page
block_tables[b][t // page_size], slot t % page_size; s_t = scale * q . K_t;
out = sum_t softmax(s)_t V_t.
"""

from __future__ import annotations

import dataclasses
import json
import math
import os
from fractions import Fraction

import numpy as np

from paged_kv_cache_63_gb300.workloads import Workload, make_workload, to_head_major

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers (no oracle code)
def _kv_row(cache: np.ndarray, layout: int, page: int, slot: int, kv: int) -> np.ndarray:
    """One head's row of a cache in either layout (0: [page][slot][kv]; 1: [page][kv][slot])."""
    return cache[page, kv, slot] if layout == 1 else cache[page, slot, kv]


def brute_force_row(w: Workload, b: int, h: int, scale=None):
    """Softmax attention of one (b, h) in plain Python with exactly rounded sums."""
    g = w.query_heads // w.kv_heads
    lay = getattr(w, "cache_layout", 0)
    kv = h // g
    n = int(w.context_lengths[b])
    sc = float(w.scale if scale is None else scale)
    q = [float(x) for x in w.query[b, h]]
    rows = []
    for t in range(n):
        page = int(w.block_tables[b, t // w.page_size])
        rows.append((page, t % w.page_size))
    s = [sc * math.fsum(q[d] * float(_kv_row(w.key_cache, lay, p, sl, kv)[d])
                        for d in range(w.head_dim)) for p, sl in rows]
    if n == 0:
        return [0.0] * w.head_dim, s
    m = max(s)
    wts = [math.exp(x - m) for x in s]
    L = math.fsum(wts)
    out = [math.fsum(wts[t] * float(_kv_row(w.value_cache, lay, p, sl, kv)[d])
                     for t, (p, sl) in enumerate(rows)) / L for d in range(w.head_dim)]
    return out, s


def gather_v(w: Workload, b: int, h: int) -> np.ndarray:
    """The V rows one (b, h) attends to, gathered with numpy fancy indexing, as fp64."""
    g = w.query_heads // w.kv_heads
    n = int(w.context_lengths[b])
    t = np.arange(n)
    pages = w.block_tables[b, t // w.page_size]
    if getattr(w, "cache_layout", 0) == 1:
        return w.value_cache[pages, h // g, t % w.page_size].astype(np.float64)
    return w.value_cache[pages, t % w.page_size, h // g].astype(np.float64)


def replace(w: Workload, **kw) -> Workload:
    return dataclasses.replace(w, **kw)


def small(name="tiny", seed=11, **kw) -> Workload:
    return make_workload(name, seed=seed, **kw)


def load_golden(fname: str):
    with open(os.path.join(GOLDEN, fname)) as f:
        return json.load(f)


def _close(a, b, atol=1e-12, rtol=1e-12):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    assert np.all(np.isfinite(a)), "non-finite values"
    assert np.all(err <= bound), f"max err {float(err.max()):.3e}"


# ---------------------------------------------------------------- pins
def pin_half_widening(o):
    """binary16 -> fp64 matches numpy's conversion for all 65536 bit patterns."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    # spot-check through the oracle one pattern at a time (every 7th, plus the edges)
    idx = sorted(set(range(0, 1 << 16, 7)) | {0, 1, 0x3FF, 0x400, 0x3C00, 0x7BFF, 0x7C00,
                                                0x7C01, 0x8000, 0x8001, 0xFBFF, 0xFC00, 0xFFFF})
    for i in idx:
        got = o.half_to_double(i)
        if math.isnan(ref[i]):
            assert math.isnan(got), hex(i)
        else:
            assert got == ref[i], (hex(i), got, ref[i])


def pin_brute_force(o):
    """Oracle == plain-Python brute force on the tiny workload and a GQA-4 slice."""
    for w in (make_workload("tiny"),
              small("gqa4_mid", seed=5, context_lengths=[1, 17, 40], max_pages_per_sequence=4,
                    spare_pages=2, head_dim=64)):
        out = o.decode(w)
        for b in range(w.batch):
            for h in range(w.query_heads):
                ref, _ = brute_force_row(w, b, h)
                _close(out[b, h], ref)


def pin_context_one(o):
    """A context of one token returns that token's V row exactly."""
    w = small(context_lengths=[1, 1, 1])
    out = o.decode(w)
    for b in range(w.batch):
        for h in range(w.query_heads):
            assert np.array_equal(out[b, h], gather_v(w, b, h)[0])


def pin_constant_v(o):
    """V constant over tokens returns that constant."""
    w = small(context_lengths=[5, 33, 64])
    v = np.full_like(w.value_cache, np.float16(-1.25))
    out = o.decode(replace(w, value_cache=v))
    _close(out, np.full(out.shape, -1.25), atol=1e-14)


def pin_sum_to_one(o):
    """Weights sum to one: V = 1 returns 1."""
    w = small(context_lengths=[3, 50])
    out = o.decode(replace(w, value_cache=np.ones_like(w.value_cache)))
    _close(out, np.ones(out.shape), atol=1e-14)


def pin_identical_keys(o):
    """Identical keys give equal weights: the output is the mean of the gathered V rows."""
    w = small(context_lengths=[7, 48, 100])
    k = np.broadcast_to(w.key_cache[:1, :1], w.key_cache.shape).copy()
    w2 = replace(w, key_cache=k)
    out = o.decode(w2)
    for b in range(w.batch):
        for h in range(w.query_heads):
            _close(out[b, h], gather_v(w2, b, h).mean(axis=0))


def pin_scale_zero(o):
    """scale = 0 gives equal weights: the mean of V."""
    w = small(context_lengths=[9, 31])
    out = o.decode(w, scale=0.0)
    for b in range(w.batch):
        for h in range(w.query_heads):
            _close(out[b, h], gather_v(w, b, h).mean(axis=0))


def _golden_workload(d, poison_nan: bool):
    from paged_kv_cache_63_gb300.workloads import SPECS

    B, qh, kvh, hd = d["batch"], d["query_heads"], d["kv_heads"], d["head_dim"]
    ps, np_ = d["page_size"], d["num_physical_pages"]
    if "key" in d:
        k = np.asarray(d["key"], dtype=np.float16)
        v = np.asarray(d["value"], dtype=np.float16)
        q = np.asarray(d["query"], dtype=np.float16)
    else:
        k = np.zeros((np_, ps, kvh, hd), dtype=np.float16)
        v = np.full((np_, ps, kvh, hd), np.nan if poison_nan else 0.0, dtype=np.float16)
        bt = np.asarray(d["block_tables"])
        ctx = d["context_lengths"]
        for b in range(B):
            for t in range(ctx[b]):
                p, s = bt[b, t // ps], t % ps
                v[p, s, :, 0] = p
                v[p, s, :, 1] = s
        q = np.ones((B, qh, hd), dtype=np.float16)
    return Workload(spec=SPECS["tiny"], batch=B, query_heads=qh, kv_heads=kvh, head_dim=hd,
                    page_size=ps, max_pages_per_sequence=d["max_pages_per_sequence"],
                    num_physical_pages=np_, scale=float(d["scale"]), query=q, key_cache=k,
                    value_cache=v, block_tables=np.asarray(d["block_tables"], dtype=np.int32),
                    context_lengths=np.asarray(d["context_lengths"], dtype=np.int32))


def golden_expected(d):
    return np.array([[float(Fraction(x)) if isinstance(x, str) else float(x) for x in row]
                     for row in d["expected"]])


def pin_golden_block_table(o):
    """The pages' block-table sketch: gathers exactly the listed pages and slots."""
    d = load_golden("block_table_sketch.json")
    w = _golden_workload(d, poison_nan=True)
    out = o.decode(w)[:, 0, :]
    _close(out, golden_expected(d), atol=1e-13)


def pin_golden_two_tokens(o):
    """Two tokens: closed form sigma(s0 - s1) v0 + sigma(s1 - s0) v1."""
    d = load_golden("two_token_closed_form.json")
    w = _golden_workload(d, poison_nan=False)
    out = o.decode(w)[:, 0, :]
    _close(out, golden_expected(d), atol=1e-15)
    e = math.e
    _close(out[0], [1 / (1 + e), e / (1 + e)], atol=1e-15)


def pin_two_tokens_random(o):
    """Two tokens with random values against the closed form computed here."""
    w = small(context_lengths=[2, 2])
    out = o.decode(w)
    for b in range(w.batch):
        for h in range(w.query_heads):
            _, s = brute_force_row(w, b, h)
            v = gather_v(w, b, h)
            sig = 1.0 / (1.0 + math.exp(s[1] - s[0]))
            _close(out[b, h], sig * v[0] + (1 - sig) * v[1])


def pin_page_permutation(o):
    """Relabelling physical pages (moving them and rewriting the table) changes nothing."""
    w = small(context_lengths=[19, 77, 128], spare_pages=5)
    rng = np.random.default_rng(123)
    pi = rng.permutation(w.num_physical_pages)
    k = np.empty_like(w.key_cache)
    v = np.empty_like(w.value_cache)
    k[pi] = w.key_cache
    v[pi] = w.value_cache
    bt = np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out = o.decode(w)
    out2 = o.decode(replace(w, key_cache=k, value_cache=v, block_tables=bt))
    assert np.array_equal(out, out2)


def pin_gqa_is_mha_replicated(o):
    """GQA equals MHA whose K/V heads are the group's K/V head repeated (contiguous groups)."""
    w = small("tiny", context_lengths=[13, 70])
    g = w.query_heads // w.kv_heads
    k = np.repeat(w.key_cache, g, axis=2)
    v = np.repeat(w.value_cache, g, axis=2)
    w2 = replace(w, kv_heads=w.query_heads, key_cache=k, value_cache=v)
    assert np.array_equal(o.decode(w), o.decode(w2))


def pin_partial_combine(o):
    """Merging per-range states reproduces the full result, for any split incl. empty ones."""
    w = small(context_lengths=[90, 1, 64])
    full = o.decode(w)
    for b in range(w.batch):
        n = int(w.context_lengths[b])
        for h in range(w.query_heads):
            r = b * w.query_heads + h
            for cuts in ([0, n], [0, 0, n], [0, n // 3, n // 2, n], [0, 16, 16, 32, n, n]):
                cuts = [min(c, n) for c in cuts]
                st = [o.partial(w, r, a, c) for a, c in zip(cuts[:-1], cuts[1:])]
                m = [x[0] for x in st]
                l = [x[1] for x in st]
                acc = np.stack([x[2] for x in st])
                _close(o.combine(m, l, acc), full[b, h])


def pin_partial_state(o):
    """A range's state: m = max score, l = sum exp(s - m), acc / l = weighted mean of V."""
    w = small(context_lengths=[45, 80])
    for b in range(w.batch):
        for h in range(w.query_heads):
            r = b * w.query_heads + h
            _, s = brute_force_row(w, b, h)
            v = gather_v(w, b, h)
            for t0, t1 in ((0, len(s)), (3, 29), (10, 11)):
                m, l, acc = o.partial(w, r, t0, t1)
                ss = s[t0:t1]
                assert m == max(ss) or abs(m - max(ss)) <= 1e-13 * max(1.0, abs(m))
                wts = [math.exp(x - max(ss)) for x in ss]
                _close(l, math.fsum(wts))
                _close(acc, (np.asarray(wts)[:, None] * v[t0:t1]).sum(axis=0))
            m, l, acc = o.partial(w, r, 5, 5)
            assert m == -math.inf and l == 0.0 and not acc.any()


def pin_poison_unread(o):
    """Unreferenced pages and slots past the context are never read (NaN stays out)."""
    w = small(context_lengths=[21, 50, 3], spare_pages=4)
    clean = o.decode(w)
    k = w.key_cache.copy()
    v = w.value_cache.copy()
    used = np.zeros(k.shape[:2], dtype=bool)
    for b in range(w.batch):
        for t in range(int(w.context_lengths[b])):
            used[w.block_tables[b, t // w.page_size], t % w.page_size] = True
    k[~used] = np.float16(np.nan)
    v[~used] = np.float16(np.inf)
    out = o.decode(replace(w, key_cache=k, value_cache=v))
    assert np.array_equal(out, clean)


def pin_zero_context(o):
    """A context of length 0 yields zeros (empty sum); other rows are unaffected."""
    w = small(context_lengths=[0, 12])
    out = o.decode(w)
    assert not out[0].any()
    for h in range(w.query_heads):
        ref, _ = brute_force_row(w, 1, h)
        _close(out[1, h], ref)


def pin_rejects_bad_indices(o):
    """A page id outside the pool or a context past the table is refused, not read."""
    w = small(context_lengths=[20, 20])
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_physical_pages
    try:
        o.decode(replace(w, block_tables=bt))
    except ValueError:
        pass
    else:
        raise AssertionError("bad page id accepted")
    ctx = w.context_lengths.copy()
    ctx[0] = w.max_pages_per_sequence * w.page_size + 1
    try:
        o.decode(replace(w, context_lengths=ctx))
    except ValueError:
        pass
    else:
        raise AssertionError("over-long context accepted")


def pin_row_subset(o):
    """Computing listed rows gives the same values as the full call."""
    w = small(context_lengths=[30, 60, 90])
    full = o.decode(w).reshape(-1, w.head_dim)
    rows = [0, 5, 11, 7]
    assert np.array_equal(o.decode(w, rows=rows), full[rows])


def pin_head_major_layout(o):
    """The [page][kv_head][slot][head_dim] layout gives exactly the same results as the
    pages' [page][slot][kv_head][head_dim] layout, and matches brute force."""
    for w in (make_workload("tiny"), small("gqa4_mid", seed=8, context_lengths=[33, 1, 70],
                                           head_dim=64, spare_pages=3)):
        hm = to_head_major(w)
        assert hm.key_cache.shape == (w.num_physical_pages, w.kv_heads, w.page_size, w.head_dim)
        a = o.decode(w)
        b = o.decode(hm)
        assert np.array_equal(a, b)
        for bb in range(w.batch):
            for h in range(0, w.query_heads, 3):
                ref, _ = brute_force_row(hm, bb, h)
                _close(b[bb, h], ref)


def _new_rows(w, seed=3):
    rng = np.random.default_rng(seed)
    shape = (w.batch, w.kv_heads, w.head_dim)
    return (rng.standard_normal(shape).astype(np.float16),
            rng.standard_normal(shape).astype(np.float16))


def pin_append_places_row(o):
    """Append writes sequence b's new rows at page block_tables[b][t / ps], slot t % ps
    (t = its length) in either layout, and changes nothing else."""
    for layout in (0, 1):
        w = small("tiny", context_lengths=[5, 16, 31], spare_pages=2)
        w = replace(w, block_tables=w.block_tables.copy())
        # sequence 1 fills its page exactly: its next token needs a fresh page
        w.block_tables[1, 1] = w.num_physical_pages - 1
        if layout:
            w = to_head_major(w)
        nk, nv = _new_rows(w)
        k, v, flags = o.append_kv(w, nk, nv)
        assert flags == 0
        ek = w.key_cache.copy()
        ev = w.value_cache.copy()
        for b in range(w.batch):
            t = int(w.context_lengths[b])
            page, slot = int(w.block_tables[b, t // w.page_size]), t % w.page_size
            for kv in range(w.kv_heads):
                if layout:
                    ek[page, kv, slot] = nk[b, kv]
                    ev[page, kv, slot] = nv[b, kv]
                else:
                    ek[page, slot, kv] = nk[b, kv]
                    ev[page, slot, kv] = nv[b, kv]
        assert np.array_equal(k.view(np.uint16), ek.view(np.uint16))
        assert np.array_equal(v.view(np.uint16), ev.view(np.uint16))


def pin_append_then_decode(o):
    """Decoding with length t + 1 after appending equals brute force over the extended
    sequence (the appended row is the last token)."""
    w = small("tiny", context_lengths=[7, 40])
    nk, nv = _new_rows(w, seed=9)
    k, v, _ = o.append_kv(w, nk, nv)
    w2 = replace(w, key_cache=k, value_cache=v, context_lengths=w.context_lengths + 1)
    out = o.decode(w2)
    for b in range(w.batch):
        for h in range(w.query_heads):
            ref, _ = brute_force_row(w2, b, h)
            _close(out[b, h], ref)
            # the appended token's row is what brute force read last
            g = w.query_heads // w.kv_heads
            assert np.array_equal(gather_v(w2, b, h)[-1], nv[b, h // g].astype(np.float64))


def pin_append_golden_sketch(o):
    """The pages' block-table sketch: stream 3 (5 tokens, pages 16 17 18, page size 2) appends
    its 6th token at page 18, slot 1; a full stream (6 tokens, 3 of 8 pages) needs its 4th
    table entry, a placeholder, so it is refused, not written."""
    d = load_golden("block_table_sketch.json")
    w = _golden_workload(d, poison_nan=False)
    nk = np.full((w.batch, w.kv_heads, w.head_dim), 7.0, dtype=np.float16)
    nv = np.full((w.batch, w.kv_heads, w.head_dim), -3.0, dtype=np.float16)
    k, v, flags = o.append_kv(w, nk, nv)
    assert flags == 1  # streams 1 and 2 hit the placeholder entry -1
    assert (v[18, 1, 0] == -3.0).all() and (k[18, 1, 0] == 7.0).all()
    changed = np.argwhere((v.view(np.uint16) != w.value_cache.view(np.uint16)).any(axis=(2, 3)))
    assert [tuple(x) for x in changed] == [(18, 1)]


def pin_append_rejects_bad_indices(o):
    """A length at the table's capacity or a page outside the pool is skipped and flagged."""
    w = small("tiny", context_lengths=[3, 9])
    ctx = w.context_lengths.copy()
    ctx[0] = w.max_pages_per_sequence * w.page_size
    nk, nv = _new_rows(w)
    k, v, flags = o.append_kv(replace(w, context_lengths=ctx), nk, nv)
    assert flags & 2
    bt = w.block_tables.copy()
    bt[1, 0] = w.num_physical_pages
    k2, v2, flags2 = o.append_kv(replace(w, block_tables=bt), nk, nv)
    assert flags2 & 1


# ---------------------------------------------------------------- multi-token (prefill) pins
def _prefill_small(seed=21, new_tokens=(5, 40, 0, 17), ctx=(5, 70, 9, 17)):
    from paged_kv_cache_63_gb300.workloads import make_prefill
    return make_prefill("prefill_chunked", seed=seed, new_tokens=list(new_tokens),
                        context_lengths=list(ctx), max_pages_per_sequence=6, spare_pages=3,
                        head_dim=64)


def pin_prefill_one_token_is_decode(o):
    """One new token per sequence is exactly the decode step (same query, whole context)."""
    w = small("gqa4_mid", seed=7, context_lengths=[1, 17, 40], max_pages_per_sequence=4,
              head_dim=64)
    qs = np.arange(w.batch + 1, dtype=np.int32)
    got = o.prefill(w, w.query, qs)
    assert np.array_equal(got, o.decode(w))


def pin_prefill_brute_force(o):
    """Every (new token, head) row equals brute force over tokens 0..position, the position
    being context_length - new_tokens + j for the j-th new token."""
    p = _prefill_small()
    w = p.cache
    out = o.prefill(w, p.query, p.query_start)
    for b in range(w.batch):
        n = int(p.query_start[b + 1] - p.query_start[b])
        for j in range(n):
            i = int(p.query_start[b]) + j
            pos = int(w.context_lengths[b]) - n + j
            q = w.query.copy()
            q[b] = p.query[i]
            ctx = w.context_lengths.copy()
            ctx[b] = pos + 1
            wb = replace(w, query=q, context_lengths=ctx)
            for h in range(w.query_heads):
                ref, _ = brute_force_row(wb, b, h)
                _close(out[i, h], ref)


def pin_prefill_first_token_sees_itself(o):
    """In a fresh prompt (every token new) the first token attends only to itself, so its
    output is exactly its own V row (softmax over one score is 1)."""
    p = _prefill_small(seed=23, new_tokens=(5, 70, 9, 17))
    w = p.cache
    out = o.prefill(w, p.query, p.query_start)
    g = w.query_heads // w.kv_heads
    for b in range(w.batch):
        page = int(w.block_tables[b, 0])
        for h in range(w.query_heads):
            v0 = w.value_cache[page, 0, h // g].astype(np.float64)
            assert np.array_equal(out[int(p.query_start[b]), h], v0)


def pin_prefill_causal(o):
    """Changing the K and V of each sequence's last token changes only the last new token's
    rows; every earlier token's output is bit-for-bit unchanged."""
    p = _prefill_small(seed=25)
    w = p.cache
    base = o.prefill(w, p.query, p.query_start)
    k = w.key_cache.copy()
    v = w.value_cache.copy()
    last_rows = []
    for b in range(w.batch):
        n = int(p.query_start[b + 1] - p.query_start[b])
        t = int(w.context_lengths[b]) - 1
        if n == 0:
            continue
        page, slot = int(w.block_tables[b, t // w.page_size]), t % w.page_size
        k[page, slot] = np.float16(3.0)
        v[page, slot] = np.float16(-5.0)
        last_rows.append(int(p.query_start[b + 1]) - 1)
    got = o.prefill(replace(w, key_cache=k, value_cache=v), p.query, p.query_start)
    keep = np.ones(p.total, dtype=bool)
    keep[last_rows] = False
    assert np.array_equal(got[keep], base[keep])
    assert all(not np.array_equal(got[r], base[r]) for r in last_rows)


def pin_prefill_rejects_bad_starts(o):
    """More new tokens than context, or a start offset that is not 0, is refused."""
    p = _prefill_small(seed=27)
    w = p.cache
    qs = p.query_start.copy()
    qs[1:] += 1  # sequence 0 now claims ctx + 1 new tokens
    try:
        o.prefill(w, np.zeros((int(qs[-1]), w.query_heads, w.head_dim), np.float16), qs)
    except ValueError:
        pass
    else:
        raise AssertionError("accepted more new tokens than context")
    qs2 = p.query_start + 1
    try:
        o.prefill(w, np.zeros((int(qs2[-1]), w.query_heads, w.head_dim), np.float16), qs2)
    except ValueError:
        pass
    else:
        raise AssertionError("accepted query_start[0] != 0")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
