"""Helpers for the GPU tests: move a workload to the device, run libpagedattn through its
C ABI, and compare with the oracle at the library's tolerance."""

from __future__ import annotations

import numpy as np

# Per-element bound |gpu - oracle| <= ATOL + RTOL * |oracle| (fp32 online softmax with
# ex2.approx, fp16 probabilities in the tensor-core path, against exact fp64).
ATOL = 2e-3
RTOL = 2e-3


def torch():
    import torch as t

    return t


def to_device(w) -> dict:
    t = torch()
    return dict(q=t.from_numpy(w.query).cuda(), k=t.from_numpy(w.key_cache).cuda(),
                v=t.from_numpy(w.value_cache).cuda(), bt=t.from_numpy(w.block_tables).cuda(),
                ctx=t.from_numpy(w.context_lengths).cuda(),
                out=t.full((w.batch, w.query_heads, w.head_dim), float("nan"),
                           dtype=t.float32, device="cuda"))


def run(w, d=None, opts=None, check_errors=True) -> np.ndarray:
    """Run pa_decode (opts None) or pa_decode_ex with a fresh zeroed workspace."""
    from paged_kv_cache_63_gb300 import lib

    t = torch()
    d = d or to_device(w)
    prob = lib.problem_of(w)
    if opts is None:
        lib.pa_decode(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"])
    else:
        n = lib.pa_workspace_size(prob, opts)
        ws = t.empty(max(n, 256), dtype=t.uint8, device="cuda")
        lib.pa_workspace_init(ws, n)
        lib.pa_decode_ex(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"], opts,
                         ws if n else None, n)
    t.cuda.synchronize()
    if check_errors:
        flags = lib.pa_get_device_error()
        assert flags == 0, f"device error flags {flags}"
    return d["out"].cpu().numpy()


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(int(np.argmax(err - bound)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r} want {ref[i]!r}")
