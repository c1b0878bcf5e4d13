"""The oracle against its pins (CPU only)."""

import numpy as np
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle_mod, pin):
    pin(oracle_mod.Oracle())


def test_half_widening_exhaustive(oracle_mod):
    """Every binary16 pattern, through the oracle's decoder, against numpy."""
    o = oracle_mod.Oracle()
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_oracle_threads_agree(oracle_mod):
    """Thread count does not change results (rows are independent)."""
    from paged_kv_cache_63_gb300.workloads import make_workload

    w = make_workload("ragged", batch=8, max_pages_per_sequence=64,
                      context_lengths=[1, 300, 77, 1024, 5, 33, 2048, 64])
    a = oracle_mod.decode(w, threads=1)
    b = oracle_mod.decode(w, threads=0)
    assert np.array_equal(a, b)
