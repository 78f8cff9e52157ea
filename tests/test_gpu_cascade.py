"""GPU parity of the cascade (shared-prefix) decode through the C ABI.

The cascade calls compute the same attention as the plain calls: the oracle
is the same fp64 definition over the page tables.  The prefix pass runs on
the tcgen05 tensor cores with the rows of every sequence in one tile, so on
top of parity the tests check that a row's bytes do not depend on the rest of
the batch (subsets and permutations of the sequences), and that bad tables
are flagged, not faulted.
"""
import ctypes

import numpy as np
import pytest

import full_parity
import workloads as W
from oracle import attention

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3
ALL_PAIRS = [(k, v) for k in ("q8_0", "fp8", "nvfp4") for v in ("q5_1", "q4_0", "fp8", "nvfp4")]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_block_memra_gb300 import _build
    _build.build()
    import decode_attention_block_memra_gb300 as memra
    memra.lib()


def run(w, **kw):
    from decode_attention_block_memra_gb300.runner import run_workload
    return run_workload(w, fill_seed=1, cascade=True, **kw)


def assert_close(w, out, ref, tol=TOL):
    got = out.astype(np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref).max()
    assert err <= tol, f"max |gpu - oracle| = {err:.3e} > {tol}"
    return err


def small(kf="q8_0", vf="q5_1", D=128, q_len=1, seed=31, prefix=1024, seq_lens=(1100, 1300, 1031, 2100, 1025),
          n_heads=16, n_kv_heads=2):
    return W.make_workload("cascade", batch=len(seq_lens), q_len=q_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                           head_dim=D, k_fmt=kf, v_fmt=vf, seed=seed, seq_lens=list(seq_lens),
                           shared_prefix=prefix)


@pytest.mark.parametrize("kf,vf", ALL_PAIRS)
@pytest.mark.parametrize("D", [128, 256])
def test_cascade_formats(kf, vf, D):
    # suffixes of 76, 276, 7, 1076 (two splits) and 1 tokens over 1,024 shared ones
    w = small(kf, vf, D)
    res = run(w)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))


@pytest.mark.parametrize("q_len", [1, 4])
def test_cascade_fused_step_pools_and_rows(q_len):
    # prefix 1,040 = 16 chunks of 64 and one of 16 tokens; the step's rows are stored by the split kernel
    w = small(q_len=q_len, prefix=1040, seq_lens=(1100, 1044, 2090, 1300), seed=32)
    res = run(w, fused=True, want_pools=True)
    assert res.flags == 0
    kp, vp = attention.build_pools(w, fill=(res.initial_k_pool, res.initial_v_pool))
    assert np.array_equal(kp, res.k_pool) and np.array_equal(vp, res.v_pool)
    assert_close(w, res.out, attention.reference(w))


def test_cascade_several_row_tiles():
    # 20 sequences x q_len 2 x group 8 = 320 rows per KV head: tiles of 128, 128 and 64
    lens = [600 + 37 * i for i in range(20)]
    w = small(q_len=2, prefix=528, seq_lens=lens, seed=33)
    res = run(w)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))


@pytest.mark.parametrize("D", [128, 256])
def test_cascade_group_and_heads(D):
    # group 4 (2 KV heads of 4 query heads), 16 KV heads at head_dim 256
    w = small(D=D, n_heads=8 if D == 128 else 16, n_kv_heads=2 if D == 128 else 16, q_len=3, prefix=272,
              seq_lens=(300, 290, 1500), seed=34)
    res = run(w)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))


@pytest.mark.parametrize("fused", [False, True])
def test_cascade_full_size_shared_prefix(fused):
    # every output row and (fused: the step's rows stored by the cascade call) every pool byte
    w = W.shared_prefix()
    res = run(w, fused=fused, want_pools=True)
    assert res.flags == 0
    full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)


def _device_case(w):
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w, fill_seed=1)
    dw.step()                      # the step's rows are appended (plain path), output discarded
    torch.cuda.synchronize()
    return dw


def _cascade_out(dw, idx):
    import decode_attention_block_memra_gb300 as memra
    w = dw.w
    idx = torch.as_tensor(idx, dtype=torch.long, device=dw.q.device)
    q = dw.q[idx].contiguous()
    pt = dw.page_table[idx].contiguous()
    sl = dw.seq_lens[idx].contiguous()
    B = len(idx)
    out = torch.empty_like(q)
    ws = torch.empty(max(1, memra.decode_attn_cascade_workspace_bytes(B, w.q_len, w.n_heads, w.head_dim,
                                                                      w.max_seq_len, w.shared_prefix)),
                     dtype=torch.uint8, device=q.device)
    memra.decode_attn_cascade(dw.cache, q, pt, sl, w.max_seq_len, w.shared_prefix, out, ws, w.sm_scale)
    assert memra.read_status(dw.cache) == 0
    return out.cpu().numpy()


def test_cascade_rows_do_not_depend_on_the_batch():
    lens = [700 + 53 * i for i in range(18)]
    w = small(q_len=1, prefix=640, seq_lens=lens, seed=35)        # 144 rows: two tiles
    dw = _device_case(w)
    full = _cascade_out(dw, list(range(18)))
    assert_close(w, full, attention.reference(w))
    sub = [16, 3, 9]
    part = _cascade_out(dw, sub)
    assert np.array_equal(part.view(np.uint16), full[sub].view(np.uint16))
    perm = list(np.random.default_rng(0).permutation(18))
    assert np.array_equal(_cascade_out(dw, perm).view(np.uint16), full[perm].view(np.uint16))
    again = _cascade_out(dw, list(range(18)))
    assert np.array_equal(again.view(np.uint16), full.view(np.uint16))


def test_cascade_bad_tables_are_flagged_not_faulted():
    import decode_attention_block_memra_gb300 as memra
    w = small(prefix=512, seq_lens=(700, 800, 900), seed=36)
    dw = _device_case(w)
    ws = torch.empty(memra.decode_attn_cascade_workspace_bytes(w.batch, 1, w.n_heads, w.head_dim, w.max_seq_len, 512),
                     dtype=torch.uint8, device=dw.q.device)
    out = torch.empty_like(dw.q)
    # a sequence whose table leaves the shared prefix
    pt = dw.page_table.clone()
    pt[1, 3] = pt[1, 40]
    memra.decode_attn_cascade(dw.cache, dw.q, pt, dw.seq_lens, w.max_seq_len, 512, out, ws, w.sm_scale)
    assert memra.read_status(dw.cache) & memra.DEVERR_PREFIX
    # a prefix page outside the pool
    pt = dw.page_table.clone()
    pt[:, 5] = w.num_pages + 7
    memra.decode_attn_cascade(dw.cache, dw.q, pt, dw.seq_lens, w.max_seq_len, 512, out, ws, w.sm_scale)
    assert memra.read_status(dw.cache) & memra.DEVERR_BAD_PAGE
    # a sequence shorter than the prefix plus its new token
    sl = dw.seq_lens.clone()
    sl[2] = 500
    memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, sl, w.max_seq_len, 512, out, ws, w.sm_scale)
    assert memra.read_status(dw.cache) & memra.DEVERR_BAD_SEQ_LEN
    # the good call still matches afterwards
    memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, 512, out, ws, w.sm_scale)
    assert memra.read_status(dw.cache) == 0
    assert_close(w, out.cpu().numpy(), attention.reference(w))


def test_cascade_host_validation():
    import decode_attention_block_memra_gb300 as memra
    w = small(prefix=512, seq_lens=(700, 800), seed=37)
    dw = _device_case(w)
    L = memra.lib()
    ws = torch.empty(memra.decode_attn_cascade_workspace_bytes(w.batch, 1, w.n_heads, w.head_dim, w.max_seq_len, 512),
                     dtype=torch.uint8, device=dw.q.device)
    out = torch.empty_like(dw.q)

    def call(prefix, wsb=None, max_seq_len=None):
        return L.memra_decode_attn_cascade(dw.cache.ref, dw.q.data_ptr(), dw.page_table.data_ptr(),
                                           int(dw.page_table.shape[1]), dw.seq_lens.data_ptr(),
                                           max_seq_len or w.max_seq_len, prefix, w.batch, 1, w.n_heads, w.n_kv_heads,
                                           w.head_dim, ctypes.c_float(w.sm_scale), ws.data_ptr(),
                                           ws.numel() if wsb is None else wsb, out.data_ptr(), None)
    assert call(500) == 1                       # not a multiple of 16
    assert call(-16) == 1
    assert call(800) == 1                       # above max_seq_len - q_len
    assert call(512, wsb=1000) == 3
    assert call(512) == 0
    assert memra.read_status(dw.cache) == 0
    assert call(0) == 0                         # the plain call
    assert memra.read_status(dw.cache) == 0


@pytest.mark.parametrize("case", ["one_page_prefix", "ten_row_tiles", "d256_ragged"])
def test_cascade_edges(case):
    if case == "one_page_prefix":          # one chunk: one prefix CTA per KV head
        w = small(prefix=16, seq_lens=(17, 40, 300), seed=38)
    elif case == "ten_row_tiles":          # 40 sequences x q_len 4 x group 8 = 1,280 rows per KV head
        lens = [400 + 29 * i for i in range(40)]
        w = small(q_len=4, prefix=384, seq_lens=lens, seed=39)
    else:                                  # head_dim 256, own keys from 1 to 2,000 tokens, verify rows
        w = small(D=256, q_len=2, prefix=832, seq_lens=(834, 1000, 2832, 900), seed=40, kf="fp8", vf="q4_0")
    res = run(w, fused=True)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))


@pytest.mark.parametrize("D,n_kv_heads,prefix,q_len", [(128, 1, 40960, 2), (256, 2, 16384, 1)])
def test_cascade_ctas_loop_over_chunks(D, n_kv_heads, prefix, q_len):
    # more chunks than one wave of CTAs per KV head: each prefix CTA loops over several
    w = small(D=D, n_heads=8 * n_kv_heads, n_kv_heads=n_kv_heads, q_len=q_len, prefix=prefix,
              seq_lens=(prefix + 40, prefix + 700, prefix + 1500), seed=41)
    res = run(w, fused=True)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))


def test_cascade_rescales_the_accumulator():
    # keys of one prefix chunk 8x larger: the row maxima jump by far more than the lazy margin.  With
    # 640 chunks over 152 CTA slots a CTA takes 5 chunks, so chunk 301 (tokens 19,264 .. 19,327; prefix
    # rows are stored in token order) is the second of its CTA, which rescales O in tensor memory
    w = small(n_heads=8, n_kv_heads=1, prefix=40960, seq_lens=(41000, 41600), seed=42)
    k = w.k_rows.astype(np.float32)
    k[19264:19328] *= 8.0
    w.k_rows = k.astype(np.float16)
    res = run(w)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))


def test_cascade_full_size_long_shared_prefix():
    w = W.shared_prefix_long()
    res = run(w, fused=True, want_pools=True)
    assert res.flags == 0
    full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)


@pytest.mark.parametrize("kf,vf", [("q8_0", "q5_1"), ("q8_0", "q4_0")])
def test_cascade_tiny_block_scales(kf, vf):
    # K and V scaled by 1e-3: block scales near 2^-16, below 2^-13, where the staged hi + lo fp16 pair
    # loses the residual's last bits to fp16 subnormals (at most 2^-24 off a value).  The scores are
    # scaled up again through q so the softmax is not uniform
    w = small(kf, vf, prefix=1024, seq_lens=(1100, 1500, 1030), seed=43)
    w.k_rows = (w.k_rows.astype(np.float32) * 1e-3).astype(np.float16)
    w.v_rows = (w.v_rows.astype(np.float32) * 1e-3).astype(np.float16)
    w.q = np.clip(w.q.astype(np.float32) * 1e3, -60000, 60000).astype(np.float16)
    ref = attention.reference(w)
    res = run(w)
    assert res.flags == 0
    # the outputs are ~1e-3 in size: hold them to 2e-3 relative to that scale (x 8 for the largest values)
    assert_close(w, res.out, ref, tol=2e-3 * 1e-3 * 8)


def test_cascade_large_queries():
    # the own-key split pass shares the plain kernel's q8_0 bias correction: large queries there too
    w = small(prefix=1024, seq_lens=(1100, 1500, 1030), seed=44)
    w.q = np.clip(w.q.astype(np.float32) * 1e3, -60000, 60000).astype(np.float16)
    w.k_rows = (w.k_rows.astype(np.float32) * 1e-3).astype(np.float16)
    res = run(w)
    assert res.flags == 0
    assert_close(w, res.out, attention.reference(w))
