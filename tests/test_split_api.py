"""The fixed-split entry points (the pages' "V4" split-K partial and log-sum-exp merge)
against the oracle's per-range states and merge, through the C ABI."""

import math

import numpy as np
import pytest

from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_workload
from tests.gpu_util import assert_close, to_device, torch

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)


def split_range(w, b, s, ns):
    """Token range of split s of sequence b: ceil(pages / ns) pages per split."""
    ctx = int(w.context_lengths[b])
    pages = -(-ctx // w.page_size)
    pps = -(-pages // ns)
    p0 = min(s * pps, pages)
    p1 = min(p0 + pps, pages)
    return p0 * w.page_size, min(p1 * w.page_size, ctx)


def partial_gpu(w, ns, math_="auto"):
    t = torch()
    d = to_device(w)
    shape = (w.batch, ns, w.query_heads)
    pm = t.full(shape, float("nan"), dtype=t.float32, device="cuda")
    pl = t.full(shape, float("nan"), dtype=t.float32, device="cuda")
    po = t.full(shape + (w.head_dim,), float("nan"), dtype=t.float32, device="cuda")
    lib.pa_split_kv_partial(lib.problem_of(w), d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale,
                            ns, pm, pl, po, math=math_)
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    return d, pm, pl, po


WORKLOADS = {
    "mid": lambda: make_workload("gqa4_mid", context_lengths=[1, 16, 17, 300, 1000, 0]),
    "long": lambda: make_workload("long_gqa6", context_lengths=[3000, 64, 1]),
    "tiny": lambda: make_workload("tiny"),
}


@pytest.mark.parametrize("math_", ["simt", "mma"])
@pytest.mark.parametrize("ns", [1, 2, 3, 7, "max"])
@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_partial_states_and_combine(name, ns, math_):
    """Splits 1, 2, 3, 7 and the most there can be (one page per split for the longest
    sequence, so shorter ones end in empty splits)."""
    import oracle

    w = WORKLOADS[name]()
    if ns == "max":
        ns = max(1, int((-(-w.context_lengths.astype(np.int64) // w.page_size)).max()))
    d, pm, pl, po = partial_gpu(w, ns, math_)
    pm, pl, po = pm.cpu().numpy(), pl.cpu().numpy(), po.cpu().numpy()
    for b in range(w.batch):
        for s in range(ns):
            t0, t1 = split_range(w, b, s, ns)
            for h in range(w.query_heads):
                m, l, acc = oracle.partial(w, b * w.query_heads + h, t0, t1)
                if t1 <= t0:
                    assert pm[b, s, h] == -np.inf and pl[b, s, h] == 0 and not po[b, s, h].any()
                    continue
                # base-2 maximum, and the convention-free log of the total weight
                assert abs(pm[b, s, h] - m * LOG2E) <= 1e-3 + 1e-3 * abs(m * LOG2E)
                lg = math.log2(pl[b, s, h]) + pm[b, s, h]
                assert abs(lg - (math.log(l) + m) * LOG2E) <= 2e-3
                assert_close(po[b, s, h] / pl[b, s, h], acc / l, f"{name} b={b} s={s} h={h}")
    out = torch().full((w.batch, w.query_heads, w.head_dim), float("nan"), device="cuda")
    t = torch()
    lib.pa_split_kv_combine(lib.problem_of(w), ns, t.from_numpy(pm).cuda(),
                            t.from_numpy(pl).cuda(), t.from_numpy(po).cuda(), out)
    t.cuda.synchronize()
    assert_close(out.cpu().numpy(), oracle.decode(w), f"{name} combined")


def test_combine_kernel_on_oracle_states():
    """The combine kernel alone, fed the oracle's states (rounded to fp32, base 2)."""
    import oracle

    t = torch()
    w = make_workload("gqa4_mid", context_lengths=[40, 999, 5, 0])
    ns = 4
    shape = (w.batch, ns, w.query_heads)
    pm = np.zeros(shape, np.float32)
    pl = np.zeros(shape, np.float32)
    po = np.zeros(shape + (w.head_dim,), np.float32)
    ref = np.zeros((w.batch, w.query_heads, w.head_dim))
    for b in range(w.batch):
        for h in range(w.query_heads):
            ms, ls, accs = [], [], []
            for s in range(ns):
                t0, t1 = split_range(w, b, s, ns)
                m, l, acc = oracle.partial(w, b * w.query_heads + h, t0, t1)
                pm[b, s, h] = m * LOG2E if l > 0 else -np.inf
                pl[b, s, h] = l
                po[b, s, h] = acc
                ms.append(m)
                ls.append(l)
                accs.append(acc)
            ref[b, h] = oracle.combine(ms, ls, np.stack(accs))
    out = t.full((w.batch, w.query_heads, w.head_dim), float("nan"), device="cuda")
    lib.pa_split_kv_combine(lib.problem_of(w), ns, t.from_numpy(pm).cuda(),
                            t.from_numpy(pl).cuda(), t.from_numpy(po).cuda(), out)
    t.cuda.synchronize()
    got = out.cpu().numpy()
    assert_close(got, ref, "combine")
    assert not got[3].any()
