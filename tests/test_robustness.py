"""Index exactness, determinism, device-side error flags and workspace handling on the GPU.

Index exactness is shown without a sanitizer: pages no sequence references, slots past a
context inside its last page and block-table placeholders are filled with NaN/Inf/-1,
and the output must equal the clean run bit for bit."""

import numpy as np
import pytest

from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_workload
from tests.gpu_util import assert_close, run, to_device, torch
from tests.test_parity import OPTS

pytestmark = pytest.mark.gpu


def poisoned(w):
    k = w.key_cache.copy()
    v = w.value_cache.copy()
    used = np.zeros(k.shape[:2], dtype=bool)
    for b in range(w.batch):
        n = int(w.context_lengths[b])
        t = np.arange(n)
        used[w.block_tables[b, t // w.page_size], t % w.page_size] = True
    k[~used] = np.float16(np.nan)
    v[~used] = np.float16(np.inf)
    v[~used & (np.arange(k.shape[1])[None, :] % 2 == 0)] = np.float16(np.nan)
    import dataclasses

    return dataclasses.replace(w, key_cache=k, value_cache=v)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("opt", sorted(OPTS))
def test_poisoned_slots_are_never_read(opt, layout):
    from paged_kv_cache_63_gb300.workloads import to_head_major

    w = make_workload("gqa4_mid", context_lengths=[5, 17, 33, 250, 0, 1], spare_pages=3)
    bad = poisoned(w)
    if layout:
        w, bad = to_head_major(w), to_head_major(bad)
    clean = run(w, opts=lib.options(**OPTS[opt]))
    dirty = run(bad, opts=lib.options(**OPTS[opt]))
    assert np.isfinite(dirty).all()
    assert np.array_equal(clean, dirty)


@pytest.mark.parametrize("name", ["mid", "ragged"])
def test_deterministic(name):
    w = (make_workload("gqa4_mid", batch=8) if name == "mid" else make_workload("ragged", batch=40))
    d = to_device(w)
    first = run(w, d)
    for _ in range(4):
        assert np.array_equal(run(w, d), first)


def test_bad_page_id_is_flagged_not_read():
    w = make_workload("tiny")
    bt = w.block_tables.copy()
    bt[1, 2] = w.num_physical_pages + 5  # needed by sequence 1 (100 tokens, 7 pages)
    import dataclasses

    run(dataclasses.replace(w, block_tables=bt), check_errors=False)
    assert lib.pa_get_device_error() & lib.PA_DEVERR_PAGE_ID
    bt[1, 2] = -7
    run(dataclasses.replace(w, block_tables=bt), check_errors=False)
    assert lib.pa_get_device_error() & lib.PA_DEVERR_PAGE_ID
    # the flag is cleared by reading it
    run(w)


def test_bad_context_is_clamped_and_flagged():
    import dataclasses

    import oracle

    w = make_workload("tiny")
    ctx = w.context_lengths.copy()
    ctx[0] = -3
    ctx[1] = w.max_pages_per_sequence * w.page_size + 50
    got = run(dataclasses.replace(w, context_lengths=ctx), check_errors=False)
    assert lib.pa_get_device_error() & lib.PA_DEVERR_CONTEXT
    assert not got[0].any()
    # sequence 1 is clamped to the table's capacity: all 8 listed entries must be valid
    bt = w.block_tables.copy()
    bt[1, 7] = w.block_tables[0, 0]
    clamped = dataclasses.replace(w, context_lengths=np.array([0, 128], np.int32), block_tables=bt)
    ref = oracle.decode(clamped)
    got = run(dataclasses.replace(clamped, context_lengths=ctx), check_errors=False)
    assert lib.pa_get_device_error() & lib.PA_DEVERR_CONTEXT
    assert_close(got, ref, "clamped")


def test_batch_zero_is_a_no_op():
    t = torch()
    x = t.zeros(16, dtype=t.float16, device="cuda")
    o = t.zeros(16, dtype=t.float32, device="cuda")
    i = t.zeros(4, dtype=t.int32, device="cuda")
    lib.pa_decode(lib.problem(0, 4, 2, 64, 16, 8, 16), x, x, x, i, i, 0.1, o)
    t.cuda.synchronize()


def test_workspace_errors_and_reuse():
    t = torch()
    w = make_workload("gqa4_mid", batch=6)
    d = to_device(w)
    prob = lib.problem_of(w)
    opts = lib.options(schedule="balanced")
    n = lib.pa_workspace_size(prob, opts)
    assert n > 0
    args = (prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"], opts)
    assert lib.status_of(lib.pa_decode_ex, *args, None, 0) == 4
    ws = t.empty(n + 512, dtype=t.uint8, device="cuda")
    assert lib.status_of(lib.pa_decode_ex, *args, ws, n - 1) == 4
    assert lib.status_of(lib.pa_decode_ex, *args, ws.data_ptr() + 16, n) == 3
    lib.pa_workspace_init(ws, n)
    outs = []
    for _ in range(3):  # reused as it is: nothing in it needs resetting between calls
        lib.pa_decode_ex(*args, ws, n)
        t.cuda.synchronize()
        outs.append(d["out"].cpu().numpy().copy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    import oracle

    assert_close(outs[0], oracle.decode(w), "workspace reuse")


def test_side_stream():
    import oracle

    t = torch()
    w = make_workload("ragged", batch=12)
    d = to_device(w)
    s = t.cuda.Stream()
    with t.cuda.stream(s):
        lib.pa_decode(lib.problem_of(w), d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale,
                      d["out"], stream=s)
    s.synchronize()
    assert_close(d["out"].cpu().numpy(), oracle.decode(w), "side stream")


def test_workspace_follows_shape_changes():
    """One workspace (library-owned, and one caller buffer) across problems whose unit
    counts grow and shrink, with the caller buffer's calls alternating between the fused
    merge and the combine kernel and between two start addresses 256 bytes apart (so each
    call's flags lie over states and flags that other calls wrote): a flag left by an
    earlier call must never pass for one of this call's."""
    import oracle

    t = torch()
    seq = [make_workload("ragged", batch=100), make_workload("gqa4_mid", batch=3),
           make_workload("ragged", batch=120), make_workload("long_gqa6", context_lengths=[3000, 500]),
           make_workload("ragged", batch=90), make_workload("tiny"),
           make_workload("long_gqa6", context_lengths=[900]), make_workload("ragged", batch=130)]
    refs = [oracle.decode(w) for w in seq]
    for w, ref in zip(seq, refs):  # library-owned workspace (pa_decode), the plan's merge
        assert_close(run(w), ref, f"pa_decode {w.name} b={w.batch}")
    combos = [lib.options(schedule="balanced", combine=c) for c in ("fused", "kernel")]
    n = max(lib.pa_workspace_size(lib.problem_of(w), o) for w in seq for o in combos)
    ws = t.empty(n + 256, dtype=t.uint8, device="cuda")
    lib.pa_workspace_init(ws, n + 256)
    for i, (w, ref) in enumerate(zip(seq, refs)):
        d = to_device(w)
        lib.pa_decode_ex(lib.problem_of(w), d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale,
                         d["out"], combos[i % 2], ws.data_ptr() + 256 * ((i // 2) % 2), n)
        t.cuda.synchronize()
        assert_close(d["out"].cpu().numpy(), ref, f"pa_decode_ex {w.name} b={w.batch}")


def test_expired_wait_is_reported_and_device_stays_usable():
    """Failure detection without a fault: under PA_TEST_EXPIRE_WAITS each warp's first tile
    waits for bytes that never come; the bounded wait gives up (about a second), the call
    raises PA_DEVERR_TIMEOUT, and the next call on the same device and workspace (no
    re-initialisation) is correct."""
    import oracle

    t = torch()
    w = make_workload("gqa4_mid", batch=4)
    d = to_device(w)
    prob = lib.problem_of(w)
    bad = lib.options(test_flags=lib.PA_TEST_EXPIRE_WAITS)
    n = lib.pa_workspace_size(prob, bad)
    ws = t.empty(max(n, 256), dtype=t.uint8, device="cuda")
    lib.pa_workspace_init(ws, n)
    lib.pa_decode_ex(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"], bad,
                     ws, n)
    t.cuda.synchronize()
    assert lib.pa_get_device_error() & lib.PA_DEVERR_TIMEOUT
    assert lib.pa_get_device_error() == 0  # reading clears it
    lib.pa_decode_ex(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"],
                     lib.options(), ws, n)
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    assert_close(d["out"].cpu().numpy(), oracle.decode(w), "after an expired wait")


@pytest.mark.parametrize("case", ["forced_96_workers", "default_plan"])
def test_expired_wait_in_fused_merge_then_correct_calls(case):
    """With more units than workers each shared unit is merged inside the decode kernel by
    the worker holding its first tiles, once the others have published their states (a flag
    per state holding the call's number). Under PA_TEST_EXPIRE_WAITS every warp gives up on
    its first tile, so no state is published and no merge runs; the next call on the same
    workspace -- without pa_workspace_init and before the error word is read -- is correct,
    and so is the one after reading the error word."""
    import oracle

    t = torch()
    forced = case == "forced_96_workers"
    w = make_workload("ragged", batch=48 if forced else 160)
    d = to_device(w)
    prob = lib.problem_of(w)
    kw = dict(schedule="balanced", combine="fused", workers=96) if forced else {}
    pl = lib.pa_plan(prob, lib.options(**kw),
                     t.cuda.get_device_properties(0).multi_processor_count)
    assert pl["combine"] == 1 and pl["units"] > pl["workers"]
    ref = oracle.decode(w)
    bad = lib.options(test_flags=lib.PA_TEST_EXPIRE_WAITS, **kw)
    good = lib.options(**kw)
    n = lib.pa_workspace_size(prob, good)
    ws = t.empty(n, dtype=t.uint8, device="cuda")
    lib.pa_workspace_init(ws, n)
    args = (prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"])
    lib.pa_decode_ex(*args, good, ws, n)  # every shared unit merged once
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    assert_close(d["out"].cpu().numpy(), ref, "before")
    lib.pa_decode_ex(*args, bad, ws, n)
    t.cuda.synchronize()
    d["out"].fill_(float("nan"))
    lib.pa_decode_ex(*args, good, ws, n)
    t.cuda.synchronize()
    assert lib.pa_get_device_error() & lib.PA_DEVERR_TIMEOUT  # the earlier call's flag
    assert_close(d["out"].cpu().numpy(), ref, "next call, error word not yet read")
    d["out"].fill_(float("nan"))
    lib.pa_decode_ex(*args, good, ws, n)
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    assert_close(d["out"].cpu().numpy(), ref, "after the error word was read")
