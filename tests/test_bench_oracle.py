"""bench.py's oracle leg computes the whole step: its (sequence, KV head) pieces, run in a spawn
pool over memory-mapped arrays, add up to the oracle's own attention over the same workload."""
import numpy as np
import pytest

import bench
import workloads as W
from oracle import attention


@pytest.mark.parametrize("name", ["tiny", "mtp_verify"])
def test_oracle_step_pieces_are_the_oracle(name):
    st = bench.OracleStep(name, workers=2)
    try:
        sums = {(b, kh): st.pool.submit(bench._oracle_step_piece, st.spec, b, kh).result() for b, kh in st.pieces}
        assert st.run() > 0
    finally:
        st.close()
    w = W.WORKLOADS[name]()
    ref = attention.reference(w)
    G = w.n_heads // w.n_kv_heads
    assert len(sums) == w.batch * w.n_kv_heads
    for (b, kh), s in sums.items():
        assert np.isclose(s, ref[b, :, kh * G:(kh + 1) * G].sum(), rtol=1e-12, atol=1e-9)
    d = st.describe("test")
    assert d["kind"] == "oracle" and d["cores"] == min(2, len(st.pieces)) and d["host_cpus"] >= 1


def test_both_arms_print_the_same_config():
    w = W.tiny()
    assert bench.workload_config(w) == bench.workload_config(W.tiny())
    assert "parallelism" not in bench.workload_config(w)
