"""The CPU oracle against its pins (hand-worked example, closed forms, invariants,
library routines, brute force).  CPU only."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_thread_count_does_not_change_results(lib):
    import numpy as np
    from workloads import CONFIGS, prefill
    d = prefill(CONFIGS["tiny128"])
    rows = np.arange(0, 128, 5)
    oracle.set_threads(1, lib)
    a = oracle.indexer_scores(d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"], rows, lib)
    oracle.set_threads(4, lib)
    b = oracle.indexer_scores(d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"], rows, lib)
    oracle.set_threads(0, lib)
    np.testing.assert_array_equal(a, b)
