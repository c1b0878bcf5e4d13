"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check the pins catch
each one: a wrong GQA mapping, a dropped scale, a wrong slot/page/row index, a
transposed cache layout, a missing normalisation, a sign error, a broken log-sum-exp
merge and a wrong binary16 decoding. The real ``oracle.c`` is never modified."""

import os
import subprocess

import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "oracle.c")

MUTANTS = {
    "gqa_interleaved": ("int kv = h / g;", "int kv = h % p->kv_heads;"),
    "scale_dropped": ("s[t - t0] = scale * acc;", "s[t - t0] = acc;"),
    "scale_divides": ("s[t - t0] = scale * acc;", "s[t - t0] = acc / (scale == 0 ? 1 : scale);"),
    "slot_off_by_one": ("int slot = t % p->page_size;", "int slot = (t + 1) % p->page_size;"),
    "logical_page_mod": ("int lp = t / p->page_size;", "int lp = t % p->max_pages;"),
    "bt_row_stride": ("int page = bt[(int64_t)b * p->max_pages + lp];",
                      "int page = bt[(int64_t)b * p->page_size + lp];"),
    "layout_kv_before_slot": (
        "return ((page * p->page_size + slot) * (int64_t)p->kv_heads + kv) * p->head_dim;",
        "return ((page * p->kv_heads + kv) * (int64_t)p->page_size + slot) * p->head_dim;"),
    "query_transposed": ("return attend(p, q + row * p->head_dim,",
                         "return attend(p, q + ((int64_t)h * p->batch + b) * p->head_dim,"),
    "no_normalisation": ("for (int d = 0; d < hd; ++d) out[d] /= l;", ""),
    "exp_sign": ("double w = exp(s[t] - m);", "double w = exp(m - s[t]);"),
    "context_short": ("b, h, ctx[b], scale, out);", "b, h, ctx[b] > 0 ? ctx[b] - 1 : 0, scale, out);"),
    "merge_alpha_sign": ("double alpha = (M == -INFINITY) ? 0.0 : exp(M - Mn);",
                         "double alpha = (M == -INFINITY) ? 0.0 : exp(Mn - M);"),
    "merge_no_skip": ("if (l[i] == 0.0) continue;", ""),
    "merge_beta_missing": ("L = alpha * L + beta * l[i];", "L = alpha * L + l[i];"),
    "half_bias": ("v = ldexp((double)(f + 1024), e - 25);", "v = ldexp((double)(f + 1024), e - 24);"),
    "half_subnormal": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -14);"),
    "head_major_swapped": (
        "if (p->layout == 1) return ((page * p->kv_heads + kv) * (int64_t)p->page_size + slot) * p->head_dim;",
        "if (p->layout == 1) return ((page * p->page_size + slot) * (int64_t)p->kv_heads + kv) * p->head_dim;"),
    "append_slot_off": ("int64_t dst = cache_row(&p, page, t % page_size, kv);",
                        "int64_t dst = cache_row(&p, page, (t + 1) % page_size, kv);"),
    "append_src_transposed": ("int64_t src = ((int64_t)b * kv_heads + kv) * head_dim;",
                              "int64_t src = ((int64_t)kv * batch + b) * head_dim;"),
    "prefill_excludes_self": ("rc = attend(&p, query + r * head_dim, key_cache, value_cache, block_tables, b, h, pos + 1,",
                              "rc = attend(&p, query + r * head_dim, key_cache, value_cache, block_tables, b, h, pos,"),
    "prefill_no_prefix": ("int pos = context_lengths[b] - nb + (qi - query_start[b]);",
                          "int pos = qi - query_start[b];"),
    "prefill_sequence_lookup": ("while (query_start[b + 1] <= qi) ++b;",
                                "while (query_start[b + 1] < qi) ++b;"),
    "prefill_query_head0": ("rc = attend(&p, query + r * head_dim,",
                            "rc = attend(&p, query + (int64_t)qi * query_heads * head_dim,"),
    "value_from_key": ("const uint16_t *vrow = value + cache_row", "const uint16_t *vrow = key + cache_row"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    import oracle

    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = tmp_path / "mut.c"
    path.write_text(mutated)
    so = str(tmp_path / "libmut.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(path),
                    "-o", so, "-lm"], check=True, capture_output=True)
    o = oracle.Oracle(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
