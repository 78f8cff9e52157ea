"""The complete-parity checker (tests/full_parity.py) on the CPU: it passes the oracle's own
results and catches a single wrong pool byte, a wrong output element and a non-finite output."""
import numpy as np
import pytest

import full_parity
import workloads as W
from oracle import attention


@pytest.fixture(scope="module")
def case():
    w = W.make_workload("harness", batch=3, q_len=2, n_heads=8, n_kv_heads=2, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=5, seq_lens=[40, 300, 1030], shared_prefix=32, permute_pages=True,
                        extra_pages=2)
    rng = np.random.default_rng(0)
    fills = [rng.integers(0, 256, (w.num_pages, w.n_kv_heads, s), dtype=np.uint8)
             for s in (17 * 128, 12 * 128)]
    kp, vp = attention.build_pools(w, fill=fills)
    out = attention.reference(w).astype(np.float16)
    return w, out, kp, vp, fills


def test_passes_the_oracles_own_results(case):
    w, out, kp, vp, fills = case
    s = full_parity.check(w, out, kp, vp, *fills, pages_per_piece=7)
    assert s["rows"] == w.batch * w.q_len * w.n_heads
    assert s["max_err"] <= 1e-3


def test_catches_one_pool_byte(case):
    w, out, kp, vp, fills = case
    bad = vp.copy()
    bad[w.num_pages - 1, 1, 5] ^= 1           # a page no row was written to: it must keep the fill bytes
    with pytest.raises(AssertionError, match="V pool differs at 1 bytes"):
        full_parity.check(w, out, kp, bad, *fills, pages_per_piece=7)


def test_catches_one_output_element(case):
    w, out, kp, vp, fills = case
    bad = out.copy()
    bad[2, 1, 7, 100] += np.float16(0.01)
    with pytest.raises(AssertionError, match="max"):
        full_parity.check(w, bad)
    bad[2, 1, 7, 100] = np.float16(np.inf)
    with pytest.raises(AssertionError, match="non-finite"):
        full_parity.check(w, bad)


def test_ring_workload():
    # sliding window over ring page tables: the harness reads each sequence's rows through its ring
    w = W.make_window_workload("harness_ring", batch=2, q_len=2, n_heads=8, n_kv_heads=2, head_dim=128,
                               k_fmt="q8_0", v_fmt="q4_0", seed=9, seq_lens=[70, 400], window=100,
                               permute_pages=True, extra_pages=1)
    kp, vp = attention.build_pools(w)
    out = attention.reference(w).astype(np.float16)
    s = full_parity.check(w, out, kp, vp, pages_per_piece=3)
    assert s["rows"] == w.batch * w.q_len * w.n_heads
    bad = out.copy()
    bad[1, 0, 3, 5] += np.float16(0.01)
    with pytest.raises(AssertionError, match="max"):
        full_parity.check(w, bad, kp, vp, pages_per_piece=3)
