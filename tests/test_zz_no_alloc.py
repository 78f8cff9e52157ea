"""The no-allocation decode entry point matches the workspace entry point.

memra_decode_attn_noalloc serves callers that cannot allocate device memory
(code running inside a custom allocator or memory pool, plugins handed only
their inputs and outputs, paths that forbid allocation after start-up).  It
keeps the split-K partials in a fixed library-owned device array instead of a
caller workspace.  This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads as W

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


def _outputs(memra, w):
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    memra.kv_append(dw.cache, dw.step_k, dw.step_v, dw.step_slots)
    memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace, w.sm_scale)
    want = dw.out.clone()
    got = []
    for _ in range(2):                       # two calls in a row share the fixed array
        dw.out.fill_(float("nan"))
        memra.decode_attn_noalloc(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, w.sm_scale)
        got.append(dw.out.clone())
    assert memra.read_status(dw.cache) == 0
    return want, got


@pytest.mark.parametrize("case", ["multi_split", "verify"])
def test_noalloc_matches_workspace_entry_point(memra, case):
    if case == "multi_split":
        w = W.random_case(61, batch=3, q_len=1, n_heads=16, n_kv_heads=2, head_dim=128, ctx=(1500, 4000))
    else:
        w = W.random_case(62, batch=2, q_len=4, n_heads=32, n_kv_heads=4, head_dim=128, ctx=(2000, 3500))
    want, got = _outputs(memra, w)
    # the same kernels on the same inputs: the bytes must match the workspace call's exactly
    for g in got:
        assert torch.isfinite(g.float()).all()
        assert torch.equal(g.view(torch.int16), want.view(torch.int16))


def test_noalloc_rejects_sizes_beyond_the_array(memra):
    w = W.random_case(63, batch=1, q_len=1, n_heads=8, n_kv_heads=2, head_dim=128, ctx=(40, 80))
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    limit = memra.NOALLOC_SCRATCH_BYTES
    # a max_seq_len whose partials need more than the fixed array
    too_long = 1 << 24
    assert memra.decode_attn_workspace_bytes(1, 1, 8, 128, too_long) > limit
    with pytest.raises(memra.MemraError) as e:
        memra.decode_attn_noalloc(dw.cache, dw.q, dw.page_table, dw.seq_lens, too_long, dw.out, w.sm_scale)
    assert e.value.status == 3
    rc = memra.lib().memra_decode_attn_noalloc(dw.cache.ref, dw.q.data_ptr(), dw.page_table.data_ptr(),
                                               dw.page_table.shape[1], dw.seq_lens.data_ptr(), too_long, 1, 1, 8,
                                               2, 128, ctypes.c_float(0.1), dw.out.data_ptr(), None)
    assert rc == 3
