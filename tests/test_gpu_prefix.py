"""GPU parity for prefix caching: requests that share system prompts point at
the same physical blocks; only uncached positions are written (cached ones get
slot -1), and decode through the shared tables matches the oracle."""
import numpy as np
import pytest

from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL, gpu_step, host_values, max_abs_err, oracle_decode, oracle_step, sample_pairs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", ["row", "split"])
def test_prefix_cached_step_matches_oracle(layout):
    wl = inputs.workload("prefix", small=True)
    dev, host = host_values(wl, "cpu", layout=layout)
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev)
    np.testing.assert_array_equal(g["host_slots"], r["slots"])
    assert np.array_equal(inputs.to_numpy_elems(g["k_cache"]), r["k_cache"])
    assert np.array_equal(inputs.to_numpy_elems(g["v_cache"]), r["v_cache"])
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


def test_prefix_cached_full_size_sampled():
    wl = inputs.workload("prefix")
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev)
    assert (g["host_slots"] == -1).sum() == 144000  # 9000 cached blocks of 16 positions
    np.testing.assert_array_equal(g["host_slots"], r["slots"])
    assert np.array_equal(inputs.to_numpy_elems(g["k_cache"]), r["k_cache"])
    assert np.array_equal(inputs.to_numpy_elems(g["v_cache"]), r["v_cache"])
    pairs = sample_pairs(wl, 64)
    assert max_abs_err(g["out"], oracle_decode(wl, host, r, pairs=pairs), pairs) <= TOL["bf16"]
