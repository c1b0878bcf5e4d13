"""Seeded synthetic inputs for paged decode attention and its multi-token variant.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can consume its
output without sharing any of the method's code.

Layouts follow "[TIL] Optimizing paged attention" (retepy.com), section
"Data Layout" and the block-table sketch in section "Baseline":

* ``query``           fp16 ``[batch][query_heads][head_dim]`` (one token per sequence)
* ``key_cache``       fp16 ``[num_physical_pages][page_size][kv_heads][head_dim]``
* ``value_cache``     same layout as ``key_cache``
  (``to_head_major`` gives the alternative ``[page][kv_heads][page_size][head_dim]``)
* ``block_tables``    int32 ``[batch][max_pages_per_sequence]``; entries past
  ``ceil(context_length / page_size)`` are placeholders, filled with -1 here
* ``context_lengths`` int32 ``[batch]``

Random draws (numpy PCG64 via ``default_rng``), in this order: context lengths
(if random), the physical-page permutation, then q, the K pool and the V pool as
float32 standard normals (K multiplied by ``k_scale`` first), each rounded to
fp16 with round-to-nearest-even. Large pools are drawn in fixed-size chunks from
the same generator, which yields the same stream as one big draw.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

# Chunk of float32 normals drawn at a time when filling a large pool.
_CHUNK = 1 << 24


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and distribution recipe of one workload."""

    name: str
    batch: int
    query_heads: int
    kv_heads: int
    head_dim: int
    page_size: int
    max_pages_per_sequence: int
    seed: int
    # context-length recipe: ("fixed", [lens]) | ("uniform", lo, hi) |
    # ("lognormal", mu, sigma, lo, hi, n_ones)
    ctx: tuple
    # how physical pages are assigned: "tiny16" (16-page pool, seeded
    # permutation) or "shuffled" (pool sized to the total need, permuted)
    pages: str = "shuffled"
    k_scale: float = 1.0


# The five workloads of this library's test and benchmark plan.
SPECS: Dict[str, Spec] = {
    "tiny": Spec("tiny", batch=2, query_heads=4, kv_heads=2, head_dim=64, page_size=16,
                 max_pages_per_sequence=8, seed=0, ctx=("fixed", [37, 100]), pages="tiny16"),
    "gqa4_mid": Spec("gqa4_mid", batch=32, query_heads=32, kv_heads=8, head_dim=128,
                     page_size=16, max_pages_per_sequence=256, seed=1,
                     ctx=("uniform", 512, 4096)),
    "mha": Spec("mha", batch=64, query_heads=32, kv_heads=32, head_dim=128, page_size=16,
                max_pages_per_sequence=128, seed=2, ctx=("fixed", [2048] * 64)),
    "long_gqa6": Spec("long_gqa6", batch=4, query_heads=24, kv_heads=4, head_dim=256,
                      page_size=64, max_pages_per_sequence=1563, seed=3,
                      ctx=("fixed", [100000] * 4), k_scale=0.5),
    "ragged": Spec("ragged", batch=256, query_heads=64, kv_heads=8, head_dim=128,
                   page_size=32, max_pages_per_sequence=1024, seed=4,
                   ctx=("lognormal", 7.0, 1.2, 1, 32768, 4)),
}


@dataclasses.dataclass
class Workload:
    """One decode step's inputs (host numpy arrays)."""

    spec: Spec
    batch: int
    query_heads: int
    kv_heads: int
    head_dim: int
    page_size: int
    max_pages_per_sequence: int
    num_physical_pages: int
    scale: float
    query: np.ndarray
    key_cache: np.ndarray
    value_cache: np.ndarray
    block_tables: np.ndarray
    context_lengths: np.ndarray
    cache_layout: int = 0  # 0: [page][slot][kv_head][dim]; 1: [page][kv_head][slot][dim]

    @property
    def name(self) -> str:
        return self.spec.name

    def dims(self) -> dict:
        return dict(batch=self.batch, query_heads=self.query_heads, kv_heads=self.kv_heads,
                    head_dim=self.head_dim, page_size=self.page_size,
                    max_pages_per_sequence=self.max_pages_per_sequence,
                    num_physical_pages=self.num_physical_pages)

    def kv_bytes(self) -> int:
        """Bytes of K and V that one decode step must read (each once)."""
        return int(self.context_lengths.astype(np.int64).clip(min=0).sum()) * \
            self.kv_heads * self.head_dim * 2 * 2


def to_head_major(w: Workload) -> Workload:
    """The same workload with both caches re-laid out as [page][kv_head][slot][head_dim]."""
    if w.cache_layout == 1:
        return w
    k = np.ascontiguousarray(w.key_cache.transpose(0, 2, 1, 3))
    v = np.ascontiguousarray(w.value_cache.transpose(0, 2, 1, 3))
    return dataclasses.replace(w, key_cache=k, value_cache=v, cache_layout=1)


def _draw_fp16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    flat = out.reshape(-1)
    n = flat.size
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        flat[lo:hi] = x.astype(np.float16)
    return out


def _context_lengths(spec: Spec, rng: np.random.Generator, batch: int) -> np.ndarray:
    kind = spec.ctx[0]
    if kind == "fixed":
        lens = list(spec.ctx[1])
        if len(lens) != batch:
            lens = [lens[i % len(lens)] for i in range(batch)]
        return np.asarray(lens, dtype=np.int32)
    if kind == "uniform":
        lo, hi = spec.ctx[1], spec.ctx[2]
        return rng.integers(lo, hi + 1, size=batch).astype(np.int32)
    if kind == "lognormal":
        mu, sigma, lo, hi, n_ones = spec.ctx[1:]
        x = np.clip(np.rint(rng.lognormal(mu, sigma, size=batch)), lo, hi).astype(np.int32)
        ones = rng.choice(batch, size=min(n_ones, batch), replace=False)
        x[ones] = 1
        return x
    raise ValueError(f"unknown context recipe {kind!r}")


# Multi-token (prefill) workloads: the cache workload they extend and how many of each
# sequence's tokens are new. ("all",) makes every token new (a fresh prompt);
# ("last", n) makes the last min(n, ctx) tokens new (a prompt chunk appended to a
# cached prefix).
PREFILL_SPECS: Dict[str, tuple] = {
    "prefill_tiny": ("tiny", dict(), ("fixed", [37, 20])),
    "prefill_gqa4": ("gqa4_mid", dict(batch=8, context_lengths=[2048] * 8), ("all",)),
    "prefill_chunked": ("gqa4_mid", dict(batch=16), ("last", 512)),
    "prefill_mha": ("mha", dict(batch=8, context_lengths=[2048] * 8), ("all",)),
    # head_dim 256 (the single-tile kernel): two fresh 4096-token prompts, 24/4 heads, page 64
    "prefill_gqa6_hd256": ("long_gqa6", dict(batch=2, context_lengths=[4096] * 2), ("all",)),
}


@dataclasses.dataclass
class Prefill:
    """A paged cache that already holds every sequence's tokens, plus the queries of the
    last ``n_b`` tokens of sequence b: ``query`` fp16 ``[total][query_heads][head_dim]``,
    rows ``query_start[b] .. query_start[b + 1]`` belong to sequence b."""

    cache: Workload
    query: np.ndarray
    query_start: np.ndarray

    @property
    def new_tokens(self) -> np.ndarray:
        return np.diff(self.query_start).astype(np.int32)

    @property
    def total(self) -> int:
        return int(self.query_start[-1])

    def max_query_len(self) -> int:
        return int(self.new_tokens.max()) if self.cache.batch else 0

    def causal_pairs(self) -> int:
        """Number of (query token, attended token) pairs, per query head."""
        ctx = self.cache.context_lengths.astype(np.int64)
        n = self.new_tokens.astype(np.int64)
        # new token j of sequence b attends to ctx - n + j + 1 tokens
        return int((n * (ctx - n) + n * (n + 1) // 2).sum())


def make_prefill(name: str, seed: Optional[int] = None, *, new_tokens=None, **cache_kw) -> Prefill:
    """Build one seeded multi-token workload. ``new_tokens`` (one count per sequence) and
    ``cache_kw`` (passed to ``make_workload``) reshape it for tests. The queries are drawn
    after the cache, from a generator seeded with ``seed + 1000``."""
    base, kw, recipe = PREFILL_SPECS[name]
    kw = dict(kw)
    kw.update(cache_kw)
    w = make_workload(base, seed=seed, **kw)
    ctx = w.context_lengths.astype(np.int64)
    if new_tokens is not None:
        n = np.asarray(new_tokens, dtype=np.int64).reshape(-1)
    elif recipe[0] == "all":
        n = ctx.copy()
    elif recipe[0] == "last":
        n = np.minimum(ctx, recipe[1])
    elif recipe[0] == "fixed":
        n = np.asarray(recipe[1], dtype=np.int64)
    else:
        raise ValueError(f"unknown new-token recipe {recipe[0]!r}")
    if n.size != w.batch or (n < 0).any() or (n > ctx).any():
        raise ValueError("new-token counts must be one per sequence, within [0, context length]")
    qs = np.zeros(w.batch + 1, dtype=np.int32)
    qs[1:] = np.cumsum(n)
    rng = np.random.default_rng((w.spec.seed if seed is None else seed) + 1000)
    q = _draw_fp16(rng, (int(qs[-1]), w.query_heads, w.head_dim))
    return Prefill(cache=w, query=q, query_start=qs)


def make_workload(name: str, seed: Optional[int] = None, *, batch: Optional[int] = None,
                  context_lengths=None, max_pages_per_sequence: Optional[int] = None,
                  spare_pages: int = 0, **override) -> Workload:
    """Build one seeded workload.

    ``batch``, ``context_lengths`` and ``max_pages_per_sequence`` shrink or reshape a
    workload for tests that must finish on the oracle in seconds; ``spare_pages``
    adds unreferenced physical pages to the pool; other keyword arguments override
    fields of the spec (e.g. ``page_size=64``).
    """
    spec = SPECS[name]
    if override:
        spec = dataclasses.replace(spec, **override)
    seed = spec.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    b = spec.batch if batch is None else batch
    hd, ps, kvh, qh = spec.head_dim, spec.page_size, spec.kv_heads, spec.query_heads

    if context_lengths is not None:
        ctx = np.asarray(context_lengths, dtype=np.int32).reshape(-1)
        b = ctx.size
    else:
        ctx = _context_lengths(spec, rng, b)
    need = [max(0, -(-int(c) // ps)) for c in ctx]
    maxp = spec.max_pages_per_sequence if max_pages_per_sequence is None else max_pages_per_sequence
    maxp = max(maxp, max(need) if need else 1, 1)

    if spec.pages == "tiny16" and context_lengths is None and batch is None:
        pool = 16
    else:
        pool = sum(need) + spare_pages
    pool = max(pool, 1)
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.full((b, maxp), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[off:off + n]
        off += n

    q = _draw_fp16(rng, (b, qh, hd))
    k = _draw_fp16(rng, (pool, ps, kvh, hd), spec.k_scale)
    v = _draw_fp16(rng, (pool, ps, kvh, hd))
    return Workload(spec=spec, batch=b, query_heads=qh, kv_heads=kvh, head_dim=hd,
                    page_size=ps, max_pages_per_sequence=maxp, num_physical_pages=pool,
                    scale=1.0 / math.sqrt(hd), query=q, key_cache=k, value_cache=v,
                    block_tables=bt, context_lengths=ctx)
