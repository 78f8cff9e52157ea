"""The bounded-wait path of the split kernel, driven on the GPU without a fault.

Every pipeline wait of the library is bounded; past the bound the kernel flags
MEMRA_DEVERR_TIMEOUT, waits (bounded) for the copies it issued itself, and
returns.  The test hook of memra_testing.h makes one wait certain to run out:
the first CTA's first page expects 16 bytes more than its copies deliver, and
the page waits give up after a few milliseconds.  Nothing is left in flight
(the short page's copies have landed; only its phase never completes), so the
next call on the same process must be exact again.
"""
import time

import numpy as np
import pytest

import workloads as W
from oracle import attention

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def memra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_block_memra_gb300 import _build
    _build.build()
    import decode_attention_block_memra_gb300 as m
    m.lib()
    return m


def test_a_wait_that_runs_out_is_flagged_and_the_next_call_is_exact(memra):
    from decode_attention_block_memra_gb300.runner import upload
    w = W.random_case(71, batch=2, q_len=1, n_heads=16, n_kv_heads=2, head_dim=128, ctx=(1500, 3000))
    dw = upload(w, fill_seed=3)
    dw.step()                                         # the step's rows are appended
    assert memra.read_status(dw.cache) == 0
    pools = (dw.cache.k_pool.clone(), dw.cache.v_pool.clone())
    ref = attention.reference(w)

    t0 = time.monotonic()
    memra.testing_decode_attn_short_page(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out,
                                         dw.workspace, page_wait_ns=2_000_000, sm_scale=w.sm_scale)
    flags = memra.read_status(dw.cache)              # synchronizes: the call has returned
    elapsed = time.monotonic() - t0
    assert flags & memra.DEVERR_TIMEOUT, f"flags 0x{flags:x}"
    assert elapsed < 30.0
    assert torch.equal(pools[0], dw.cache.k_pool) and torch.equal(pools[1], dw.cache.v_pool)

    # the same process, the same buffers: a normal call is exact and flags nothing
    dw.out.fill_(float("nan"))
    memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace, w.sm_scale)
    assert memra.read_status(dw.cache) == 0
    err = np.abs(dw.out.cpu().numpy().astype(np.float64) - ref).max()
    assert err <= 2e-3, err


def test_the_hook_rejects_limits_outside_its_range(memra):
    from decode_attention_block_memra_gb300.runner import upload
    w = W.random_case(72, batch=1, q_len=1, n_heads=8, n_kv_heads=2, head_dim=128, ctx=(40, 80))
    dw = upload(w)
    for bad in (0, 2_000_000_000):
        with pytest.raises(memra.MemraError) as e:
            memra.testing_decode_attn_short_page(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                                                 dw.out, dw.workspace, page_wait_ns=bad)
        assert e.value.status == 1
    assert memra.read_status(dw.cache) == 0
