"""pa_decode_noalloc: decoding for callers that may not allocate device memory.

Such callers exist in serving engines that hand all free HBM to their K/V page pool at
start-up and forbid allocations while decoding (a cudaMalloc there would also stall the
whole device); code embedded in them is given tensors but no allocator. This entry point
takes its split-K scratch from a fixed array inside the library instead.

The file is named so that pytest collects it after every other test file."""

import numpy as np
import pytest

from paged_kv_cache_63_gb300 import lib
from paged_kv_cache_63_gb300.workloads import make_workload
from tests.gpu_util import assert_close, to_device, torch

pytestmark = pytest.mark.gpu

# (workload, overrides, merge the default plan picks: 1 = fused in the decode kernel, 2 =
# separate combine kernel). The fused merge is the path whose flags live in the scratch.
WORKLOADS = {
    "gqa4_mid": ("gqa4_mid", dict(), 2),
    "ragged_b64": ("ragged", dict(batch=64), 2),
    "ragged_b160": ("ragged", dict(batch=160), 1),
    "long_gqa6_short": ("long_gqa6", dict(context_lengths=[20000, 3000, 77, 1]), 2),
    "tiny": ("tiny", dict(), 2),
}


@pytest.mark.parametrize("key", sorted(WORKLOADS))
def test_noalloc_matches_pa_decode_on_two_calls_in_a_row(key):
    """Two pa_decode_noalloc calls in a row give pa_decode's bits exactly (same plan, same
    kernels, deterministic) and match the oracle within the library's tolerance."""
    import oracle

    t = torch()
    name, kw, merge = WORKLOADS[key]
    w = make_workload(name, **kw)
    prob = lib.problem_of(w)
    sm = t.cuda.get_device_properties(t.cuda.current_device()).multi_processor_count
    plan = lib.pa_plan(prob, None, sm)
    # the heuristic picks split-K here, so the fixed scratch is really used
    assert plan["schedule"] == 2 and plan["combine"] == merge
    assert 0 < plan["workspace_bytes"] <= lib.PA_NOALLOC_SCRATCH_BYTES
    d = to_device(w)
    lib.pa_decode(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"])
    t.cuda.synchronize()
    assert lib.pa_get_device_error() == 0
    want = d["out"].cpu().numpy()
    ref = oracle.decode(w)
    for call in range(2):
        out = t.full_like(d["out"], float("nan"))
        lib.pa_decode_noalloc(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, out)
        t.cuda.synchronize()
        assert lib.pa_get_device_error() == 0
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert np.array_equal(got, want), f"{key} call {call}: differs from pa_decode"
        assert_close(got, ref, f"{key} call {call}")


def test_noalloc_refuses_plans_larger_than_its_scratch():
    t = torch()
    # 32768 (sequence, K/V head) units of head_dim 256 need far more than 16 MiB of
    # per-range softmax state; the call must refuse before launching anything
    prob = lib.problem(4096, 64, 8, 256, 16, 4096, 1 << 16)
    assert lib.pa_plan(prob)["workspace_bytes"] > lib.PA_NOALLOC_SCRATCH_BYTES
    x = t.zeros(64, dtype=t.float16, device="cuda")
    i = t.zeros(64, dtype=t.int32, device="cuda")
    o = t.zeros(64, dtype=t.float32, device="cuda")
    assert lib.status_of(lib.pa_decode_noalloc, prob, x, x, x, i, i, 0.0625, o) == 4
