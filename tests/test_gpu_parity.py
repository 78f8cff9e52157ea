"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Quantized blocks must match the oracle bit for bit; attention outputs within
max |gpu - oracle| <= 2e-3.  That bound covers the fp16 rounding of the output
(2^-11 |o|, below 1e-3 for |o| < 2) plus the fp16 rounding of the softmax
weights before the P.V product and float32 accumulation; the K and V codes
enter the products exactly.  The pools start as seeded random bytes, so slots
that were never written hold garbage the kernels must ignore.
"""
from types import SimpleNamespace

import numpy as np
import pytest

import full_parity
import workloads as W
from oracle import attention, layout, quant

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3
C = 1280        # MEMRA_SPLIT_TOKENS: the smallest split (tests below place lengths around it)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_block_memra_gb300 import _build
    _build.build()
    import decode_attention_block_memra_gb300 as memra
    memra.lib()
    assert memra.SPLIT_TOKENS == C


def run(w, fill_seed=1, want_pools=True):
    from decode_attention_block_memra_gb300.runner import run_workload
    return run_workload(w, fill_seed=fill_seed, want_pools=want_pools)


def assert_pools_exact(w, res, cache=None):
    kp, vp = attention.build_pools(w, cache=cache, fill=(res.initial_k_pool, res.initial_v_pool))
    for name, want, got in (("K", kp, res.k_pool), ("V", vp, res.v_pool)):
        if not np.array_equal(want, got):
            bad = np.argwhere(want != got)
            raise AssertionError(f"{name} pool differs at {len(bad)} bytes, first (page, head, byte) {bad[:5].tolist()}")


def assert_out_close(w, res, ref, tol=TOL):
    mask = ~np.isnan(ref[..., 0])
    got = res.out.astype(np.float64)[mask]
    want = ref[mask]
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - want).max()
    assert err <= tol, f"max |gpu - oracle| = {err:.3e} > {tol}"
    return err


# ------------------------------------------------------------ small cases ---

def test_tiny_workload():
    w = W.tiny()
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


FORMAT_PAIRS = [("q8_0", "q5_1"), ("q8_0", "q4_0"), ("q8_0", "fp8"), ("fp8", "q5_1"), ("fp8", "q4_0"),
                ("fp8", "fp8")]


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kf,vf", FORMAT_PAIRS)
def test_formats_ragged(kf, vf, D):
    # 3 sequences, contexts spanning 1..3 splits with ragged tails, shuffled pages, GQA group 8
    w = W.random_case(1000 + D + 7 * FORMAT_PAIRS.index((kf, vf)), batch=3, q_len=1, n_heads=16, n_kv_heads=2,
                      head_dim=D, k_fmt=kf, v_fmt=vf, ctx=(5, 2600))
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("q_len,n_heads,n_kv_heads,D", [
    (4, 32, 4, 128),     # MTP verify shape: 32 query rows per KV head (two row groups)
    (2, 8, 2, 128),      # 8 rows
    (3, 8, 2, 128),      # 12 rows: padded row group
    (8, 64, 8, 128),     # 64 rows per KV head: four row groups
    (1, 4, 4, 128),      # no grouping
    (1, 12, 4, 256),     # group 3
    (4, 16, 2, 256),     # 32 rows at D 256
    (5, 4, 1, 256),      # 20 rows at D 256
])
def test_query_shapes(q_len, n_heads, n_kv_heads, D):
    w = W.random_case(77 + q_len * 13 + n_heads + D, batch=2, q_len=q_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                      head_dim=D, ctx=(q_len, 2200))
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 511, 512, 513, 1024, C - 1, C, C + 1, 2 * C + 1])
def test_context_edges(T):
    w = W.make_workload(f"edge{T}", batch=1, q_len=1, n_heads=8, n_kv_heads=1, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=T, seq_lens=[T], permute_pages=True, extra_pages=2)
    res = run(w)
    assert res.flags == 0
    ref = attention.reference(w)
    assert_out_close(w, res, ref)
    if T == 1:
        # one visible key: the output is the dequantized V row (up to the fp16 output rounding)
        cache = attention.quantize_cache(w)
        v_hat = quant.dequantize_rows(cache["v"][0])[0]
        for h in range(8):
            assert np.abs(res.out[0, 0, h].astype(np.float64) - v_hat).max() <= np.abs(v_hat).max() * 2 ** -11 + 1e-7


def test_causal_verify_rows_start_mid_page():
    # q_len 6 with the new rows crossing a page and a split boundary
    w = W.make_workload("verify_cross", batch=2, q_len=6, n_heads=8, n_kv_heads=2, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=3, seq_lens=[C + 3, C + 6])
    res = run(w)
    assert res.flags == 0
    assert_out_close(w, res, attention.reference(w))


def test_shared_prefix_small():
    w = W.make_workload("sp", batch=5, q_len=1, n_heads=16, n_kv_heads=2, head_dim=128, k_fmt="q8_0", v_fmt="q5_1",
                        seed=8, seq_lens=[1100, 1300, 1031, 2100, 1025], shared_prefix=1024)
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


def test_zero_query_and_constant_blocks():
    # q = 0 -> uniform weights: the output is the mean of the visible V^ rows
    w = W.random_case(5, batch=2, q_len=1, n_heads=8, n_kv_heads=2, ctx=(100, 1500))
    w.q[:] = 0
    w.v_rows[::3] = np.float16(0.75)          # flat blocks: q5_1 d = 0, x^ = m
    w.k_rows[1::4] = np.float16(0.0)          # zero blocks: q8_0 d = 0
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    ref = attention.reference(w)
    assert_out_close(w, res, ref)


def test_empty_batch_and_empty_sequence():
    import decode_attention_block_memra_gb300 as memra
    w = W.random_case(9, batch=2, q_len=1, n_heads=8, n_kv_heads=2, ctx=(40, 300))
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    # batch 0: a no-op that touches nothing
    memra.decode_attn(dw.cache, dw.q[:0], dw.page_table[:0], dw.seq_lens[:0], 0, dw.out[:0], dw.workspace)
    # a sequence of length 0 gives zeros
    dw.seq_lens[1] = 0
    dw.out.fill_(7)
    memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace, w.sm_scale)
    flags = memra.read_status(dw.cache)
    assert flags == memra.DEVERR_BAD_SEQ_LEN      # 0 < q_len is reported
    assert torch.all(dw.out[1] == 0)


def test_rows_without_keys_are_zeros_without_a_combine():
    # contexts of at most 1,024 tokens fit one split, so the call launches no combine: a sequence
    # shorter than q_len leaves its first rows without a visible key, and the split pass writes zeros
    import decode_attention_block_memra_gb300 as memra
    w = W.random_case(12, batch=2, q_len=4, n_heads=8, n_kv_heads=2, ctx=(300, 600))
    assert w.max_seq_len <= memra.SPLIT_TOKENS
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    dw.step()                                 # the step's rows are appended
    assert memra.read_status(dw.cache) == 0
    ref = attention.reference(w)
    dw.seq_lens[0] = 2                        # rows 0 and 1 sit before position 0
    dw.out.fill_(7)
    memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace, w.sm_scale)
    assert memra.read_status(dw.cache) == memra.DEVERR_BAD_SEQ_LEN
    out = dw.out.cpu().numpy().astype(np.float64)
    assert (out[0, :2] == 0).all()
    assert np.isfinite(out[0, 2:]).all() and not (out[0, 2:] == 7).any()
    assert np.abs(out[1] - ref[1]).max() <= TOL


def test_bad_page_and_slot_are_flagged_not_faulted():
    import decode_attention_block_memra_gb300 as memra
    w = W.random_case(11, batch=2, q_len=1, n_heads=8, n_kv_heads=2, ctx=(300, 900))
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    dw.page_table[0, 3] = w.num_pages + 5         # outside the pool
    dw.page_table[1, 0] = -2
    memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace, w.sm_scale)
    assert memra.read_status(dw.cache) & memra.DEVERR_BAD_PAGE
    assert torch.isfinite(dw.out.float()).all()
    slots = dw.step_slots.clone()
    slots[0] = w.num_pages * 16 + 1
    slots[1] = -1                                  # padding: skipped silently
    before = dw.cache.k_pool.clone()
    memra.kv_append(dw.cache, dw.step_k, dw.step_v, slots)
    assert memra.read_status(dw.cache) == memra.DEVERR_BAD_SLOT
    assert torch.equal(before, dw.cache.k_pool)    # neither row was written


def test_host_validation_errors():
    import decode_attention_block_memra_gb300 as memra
    w = W.random_case(12, batch=1, q_len=1, n_heads=8, n_kv_heads=2, ctx=(30, 60))
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    with pytest.raises(memra.MemraError) as e:
        memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace[:0])
    assert e.value.status == 3
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(memra.MemraError):
        memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, 5000, dw.out, small_ws)
    q3 = torch.zeros((1, 1, 6, 128), dtype=torch.float16, device="cuda")    # 6 heads over 2 KV heads? fine; 7 is not
    q7 = torch.zeros((1, 1, 7, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(memra.MemraError) as e:
        memra.decode_attn(dw.cache, q7, dw.page_table, dw.seq_lens, w.max_seq_len, torch.empty_like(q7), dw.workspace)
    assert e.value.status == 1
    del q3


# ------------------------------------------------------ self-consistency ----

def test_batch_invariance_and_determinism():
    """A sequence's output bytes do not depend on the batch around it or on the run."""
    w = W.random_case(31, batch=4, q_len=1, n_heads=32, n_kv_heads=4, ctx=(500, 3500))
    full = run(w, want_pools=False)
    again = run(w, want_pools=False)
    assert np.array_equal(full.out.view(np.uint16), again.out.view(np.uint16))
    for b in (0, 2):
        solo = W.make_workload("solo", batch=1, q_len=1, n_heads=32, n_kv_heads=4, head_dim=128, k_fmt="q8_0",
                               v_fmt="q5_1", seed=0, seq_lens=[int(w.seq_lens[b])])
        rows = attention.sequence_rows(w, b)
        solo.q[:] = w.q[b:b + 1]
        solo.k_rows[:] = w.k_rows[rows]
        solo.v_rows[:] = w.v_rows[rows]
        r1 = run(solo, want_pools=False)
        assert np.array_equal(r1.out[0].view(np.uint16), full.out[b].view(np.uint16))


# ------------------------------------------------------ full-size workloads --
# Every output row and every pool byte of the five workloads at their full
# sizes, against the oracle spread over the host's cores (tests/full_parity.py).

def check_everything(w, res):
    s = full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)
    assert s["rows"] == w.batch * w.q_len * w.n_heads
    return s


@pytest.mark.parametrize("name", ["tiny", "shared_prefix", "long_context", "mtp_verify"])
def test_full_size_workloads(name):
    w = W.WORKLOADS[name]()
    res = run(w)
    assert res.flags == 0
    check_everything(w, res)


@pytest.fixture(scope="module")
def sweep_base():
    return W.format_sweep("c")


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_format_sweep_full_size(sweep_base, variant):
    kf, vf = W.SWEEP_FORMATS[variant]
    w = sweep_base.with_formats(kf, vf)
    res = run(w)
    assert res.flags == 0
    check_everything(w, res)


def _adversarial_rows(rng, n, D):
    """fp16 rows whose 32-element blocks sit on rounding ties, subnormals and huge ranges."""
    rows = rng.standard_normal((n, D))
    for r in range(n):
        for b in range(D // 32):
            kind = (r * 7 + b) % 8
            blk = rows[r, 32 * b:32 * b + 32]
            if kind == 0:       # q8_0 ties at d = 1
                blk[:] = np.concatenate([[127.0], np.arange(31) - 15.5])
            elif kind == 1:     # q4_0 ties at d = 1
                blk[:] = np.concatenate([[7.0], (np.arange(31) % 15) - 7.5])
            elif kind == 2:     # q5_1 ties at d = 1, m = -1
                blk[:] = np.concatenate([[-1.0, 30.0], np.arange(30) - 0.5])
            elif kind == 3:     # huge range: x - m is not exact in float32
                blk[:] = rng.standard_normal(32) * 1e-4
                blk[0], blk[1] = 60000.0, -61000.0
            elif kind == 4:     # fp16 subnormals only
                blk[:] = rng.integers(-1023, 1024, 32) * 2.0 ** -24
            elif kind == 5:     # flat subnormal block (d rounds far below max/7)
                blk[:] = -2.0 ** -20
            elif kind == 6:
                blk[:] = rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 3)
    rows = rows.astype(np.float16)
    rng.shuffle(rows)
    return rows


@pytest.mark.parametrize("kf,vf", [("q8_0", "q5_1"), ("q8_0", "q4_0")])
def test_adversarial_blocks_bit_exact(kf, vf):
    """Quantize-append is bit-exact on rounding ties, subnormal scales and extreme ranges."""
    w = W.random_case(404, batch=2, q_len=1, n_heads=8, n_kv_heads=2, head_dim=128, k_fmt=kf, v_fmt=vf,
                      ctx=(300, 700))
    rng = np.random.default_rng(5)
    n = w.k_rows.shape[0] * w.n_kv_heads
    w.k_rows[:] = _adversarial_rows(rng, n, 128).reshape(w.k_rows.shape)
    w.v_rows[:] = _adversarial_rows(rng, n, 128).reshape(w.v_rows.shape)
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert np.isfinite(res.out.astype(np.float32)).all()


def test_long_sequence_with_wide_splits():
    """A long sequence over many KV heads gets splits wider than 1,024 tokens (one wave per head)."""
    w = W.make_workload("wide_splits", batch=2, q_len=2, n_heads=16, n_kv_heads=8, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=17, seq_lens=[100003, 57000], permute_pages=True)
    res = run(w, want_pools=False)
    assert res.flags == 0
    assert_out_close(w, res, attention.reference(w))


# ------------------------------------------- fused append + attention step --
# memra_decode_step stores the step's rows from inside the split kernel.  Its
# pools must match the oracle's bit for bit and its outputs the two-call path
# (memra_kv_append + memra_decode_attn) byte for byte: both read the same
# quantized bytes through the same arithmetic.

def run_fused(w, fill_seed=1, want_pools=True):
    from decode_attention_block_memra_gb300.runner import run_workload
    return run_workload(w, fill_seed=fill_seed, want_pools=want_pools, fused=True)


def assert_fused_matches(w, want_pools=True):
    res = run_fused(w, want_pools=want_pools)
    assert res.flags == 0
    if want_pools:
        assert_pools_exact(w, res)
    two_call = run(w, want_pools=False)
    assert np.array_equal(res.out.view(np.uint16), two_call.out.view(np.uint16)), "fused and two-call outputs differ"
    return res


def test_fused_step_tiny():
    w = W.tiny()
    res = assert_fused_matches(w)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kf,vf", FORMAT_PAIRS)
def test_fused_step_formats(kf, vf, D):
    w = W.random_case(2000 + D + 7 * FORMAT_PAIRS.index((kf, vf)), batch=3, q_len=2, n_heads=16, n_kv_heads=2,
                      head_dim=D, k_fmt=kf, v_fmt=vf, ctx=(5, 2600))
    res = assert_fused_matches(w)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("q_len,n_heads,n_kv_heads,D,seq_lens", [
    (1, 8, 1, 128, [1]),                  # the only key is the new one
    (1, 8, 1, 128, [17, 16, C + 1]),      # new row opens a page / closes a page / opens a split
    (4, 32, 4, 128, [C + 2, C + 6, 4]),   # verify rows cross the smallest split's boundary; whole sequence new
    (6, 8, 2, 128, [8000, 1027]),         # new rows deep in a long split (beyond the first ring fill)
    (8, 64, 8, 128, [700, 2049]),         # 64 rows per KV head
    (4, 16, 2, 256, [33, 1100]),          # D 256: 32 lanes per stored row
])
def test_fused_step_positions(q_len, n_heads, n_kv_heads, D, seq_lens):
    w = W.make_workload("fused_pos", batch=len(seq_lens), q_len=q_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                        head_dim=D, k_fmt="q8_0", v_fmt="q5_1", seed=sum(seq_lens) + q_len, seq_lens=seq_lens,
                        permute_pages=True, extra_pages=3)
    res = assert_fused_matches(w)
    assert_out_close(w, res, attention.reference(w))


def test_fused_step_shared_prefix():
    w = W.make_workload("sp_fused", batch=4, q_len=2, n_heads=16, n_kv_heads=2, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=21, seq_lens=[1100, 1026, 2100, 1040], shared_prefix=1024)
    res = assert_fused_matches(w)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("kf,vf", [("q8_0", "q5_1"), ("q8_0", "q4_0")])
def test_fused_step_adversarial_rows(kf, vf):
    """The fused store is bit-exact on rounding ties, subnormal scales and extreme ranges."""
    w = W.random_case(505, batch=4, q_len=8, n_heads=16, n_kv_heads=2, head_dim=128, k_fmt=kf, v_fmt=vf,
                      ctx=(8, 700))
    rng = np.random.default_rng(6)
    n = w.step_rows.size * w.n_kv_heads
    w.k_rows[w.step_rows] = _adversarial_rows(rng, n, 128).reshape(w.step_rows.size, w.n_kv_heads, 128)
    w.v_rows[w.step_rows] = _adversarial_rows(rng, n, 128).reshape(w.step_rows.size, w.n_kv_heads, 128)
    res = run_fused(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert np.isfinite(res.out.astype(np.float32)).all()


@pytest.mark.parametrize("name", ["long_context", "mtp_verify"])
def test_fused_step_full_size(name):
    w = W.WORKLOADS[name]()
    res = run_fused(w)
    assert res.flags == 0
    check_everything(w, res)


def test_fused_step_bad_page_and_validation():
    import decode_attention_block_memra_gb300 as memra
    w = W.random_case(13, batch=2, q_len=2, n_heads=8, n_kv_heads=2, ctx=(300, 900))
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w, fill_seed=4)
    T0 = int(w.seq_lens[0])
    dw.page_table[0, (T0 - 1) // 16] = w.num_pages + 5      # the page of sequence 0's last new row
    before = dw.cache.k_pool.clone()
    B, Q = w.batch, w.q_len
    k_new = dw.step_k.view(B, Q, w.n_kv_heads, w.head_dim)
    v_new = dw.step_v.view(B, Q, w.n_kv_heads, w.head_dim)
    memra.decode_step(dw.cache, k_new, v_new, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace,
                      w.sm_scale)
    assert memra.read_status(dw.cache) & memra.DEVERR_BAD_PAGE
    assert torch.isfinite(dw.out.float()).all()
    # only rows of the step were stored: every changed byte lies in a page that holds a step row
    changed = (before != dw.cache.k_pool).view(w.num_pages, -1).any(dim=1).nonzero().flatten().cpu().numpy()
    step_pages = set((w.slots[w.step_rows] // 16).tolist())
    assert set(changed.tolist()) <= step_pages
    with pytest.raises(memra.MemraError) as e:                 # misaligned rows
        memra.decode_step(dw.cache, k_new.view(-1)[1:], v_new, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                          dw.out, dw.workspace, w.sm_scale)
    assert e.value.status == 1
    with pytest.raises(memra.MemraError) as e:                 # max_seq_len below q_len
        memra.decode_step(dw.cache, k_new, v_new, dw.q, dw.page_table, dw.seq_lens, 1, dw.out, dw.workspace,
                          w.sm_scale)
    assert e.value.status == 1


# --------------------------------------------- one numeric class (verify) ---
# A verify row (q_len = K + 1, draft tokens K = 1..8) must carry the same bytes
# as a plain q_len = 1 decode at that position over the same cache: the memra
# README's speculative decode gated byte-identical to plain decode.

def _decode_at_positions(dw, w):
    """Plain q_len = 1 decode of every verify position; returns fp16 [B, Q, Hq, D]."""
    import decode_attention_block_memra_gb300 as memra
    B, Q = w.batch, w.q_len
    outs = []
    for qi in range(Q):
        q1 = dw.q[:, qi:qi + 1].contiguous()
        sl = (dw.seq_lens - (Q - 1 - qi)).to(torch.int32).contiguous()
        o1 = torch.empty_like(q1)
        memra.decode_attn(dw.cache, q1, dw.page_table, sl, w.max_seq_len, o1, dw.workspace, w.sm_scale)
        outs.append(o1)
    assert memra.read_status(dw.cache) == 0
    return torch.cat(outs, dim=1).cpu().numpy()


def _verify_vs_decode(w, fused):
    from decode_attention_block_memra_gb300.runner import upload
    import decode_attention_block_memra_gb300 as memra
    dw = upload(w, fill_seed=2)
    dw.step(fused=fused)
    assert memra.read_status(dw.cache) == 0
    verify = dw.out.cpu().numpy()
    plain = _decode_at_positions(dw, w)
    diff = np.argwhere(verify.view(np.uint16) != plain.view(np.uint16))
    assert diff.size == 0, f"{len(diff)} elements differ, first (b, qi, head, j) {diff[:4].tolist()}"
    return verify


@pytest.mark.parametrize("K", range(1, 9))
def test_verify_rows_equal_plain_decode(K):
    Q = K + 1
    # contexts: ragged, crossing a split boundary inside the verify window,
    # one split, and a sequence made only of new tokens
    seq_lens = [2 * C + 3 + K, C + Q // 2, 300 + K, Q]
    w = W.make_workload(f"verify_k{K}", batch=4, q_len=Q, n_heads=32, n_kv_heads=4, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=40 + K, seq_lens=seq_lens, permute_pages=True, extra_pages=2)
    out = _verify_vs_decode(w, fused=(K % 2 == 0))
    ref = attention.reference(w)
    assert_out_close(w, SimpleNamespace(out=out), ref)


@pytest.mark.parametrize("K,D,kf,vf", [(3, 128, "q8_0", "q5_1"), (8, 128, "fp8", "q4_0"), (5, 256, "q8_0", "fp8")])
def test_verify_rows_equal_plain_decode_across_split_size_step(K, D, kf, vf):
    """The split size C(T) grows by 16 tokens inside the verify window: each row still matches its own decode."""
    Q = K + 1
    n_kv_heads = 32
    S = max(1, torch.cuda.get_device_properties(0).multi_processor_count * 2 // n_kv_heads)
    t_step = S * C + 1                    # first length whose ceil(T / S) passes C (C(T): 1,280 -> 1,296)
    seq_lens = [t_step + Q // 2, t_step + Q - 1]
    w = W.make_workload("verify_cstep", batch=2, q_len=Q, n_heads=n_kv_heads, n_kv_heads=n_kv_heads, head_dim=D,
                        k_fmt=kf, v_fmt=vf, seed=90 + K, seq_lens=seq_lens)
    _verify_vs_decode(w, fused=True)


# ------------------------------------------- sliding window over ring pages --
# memra_decode_attn_window / memra_decode_step_window: the row at position p
# sees keys max(0, p - W + 1) .. p, and each sequence keeps only a ring of pages.

@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kf,vf", FORMAT_PAIRS)
def test_window_formats(kf, vf, D):
    # contexts below, at and far past the window (the ring wraps several times), ragged, shuffled ring pages
    w = W.make_window_workload("win_fmt", batch=4, q_len=1, n_heads=16, n_kv_heads=2, head_dim=D, k_fmt=kf,
                               v_fmt=vf, seed=300 + D + FORMAT_PAIRS.index((kf, vf)),
                               seq_lens=[37, 300, 1111, 2900], window=300, permute_pages=True, extra_pages=3)
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("window,q_len,seq_lens", [
    (1, 1, [1, 17, 500]),            # each row sees only itself
    (16, 4, [16, 20, 333]),          # window of one page
    (1000, 4, [999, 1000, 1001, 5000]),
    (1500, 2, [4097, 2050]),         # splits of a window range (C = 1,280), window start mid-page
    (4096, 8, [262144]),             # an SWA layer of a 262,144-token session: a 258-page ring
])
def test_window_shapes(window, q_len, seq_lens):
    w = W.make_window_workload("win", batch=len(seq_lens), q_len=q_len, n_heads=32, n_kv_heads=4, head_dim=128,
                               k_fmt="q8_0", v_fmt="q5_1", seed=window + q_len, seq_lens=seq_lens, window=window,
                               permute_pages=True, extra_pages=2)
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


@pytest.mark.parametrize("K", [1, 3, 8])
def test_window_verify_rows_equal_plain_decode(K):
    Q = K + 1
    w = W.make_window_workload(f"win_verify{K}", batch=3, q_len=Q, n_heads=32, n_kv_heads=4, head_dim=128,
                               k_fmt="q8_0", v_fmt="q5_1", seed=70 + K, seq_lens=[3000 + K, C + 6, Q], window=C + 1,
                               permute_pages=True)
    from decode_attention_block_memra_gb300.runner import upload
    import decode_attention_block_memra_gb300 as memra
    dw = upload(w, fill_seed=3)
    dw.step(fused=True)
    assert memra.read_status(dw.cache) == 0
    verify = dw.out.cpu().numpy()
    for qi in range(Q):
        q1 = dw.q[:, qi:qi + 1].contiguous()
        sl = (dw.seq_lens - (Q - 1 - qi)).to(torch.int32).contiguous()
        o1 = torch.empty_like(q1)
        memra.decode_attn(dw.cache, q1, dw.page_table, sl, w.max_seq_len, o1, dw.workspace, w.sm_scale,
                          window=w.window)
        assert np.array_equal(o1.cpu().numpy()[:, 0].view(np.uint16), verify[:, qi].view(np.uint16)), qi
    assert memra.read_status(dw.cache) == 0
    assert_out_close(w, SimpleNamespace(out=verify), attention.reference(w))


def test_window_fused_step_matches_two_calls():
    w = W.make_window_workload("win_fused", batch=3, q_len=4, n_heads=16, n_kv_heads=2, head_dim=128,
                               k_fmt="q8_0", v_fmt="q5_1", seed=123, seq_lens=[5000, 700, 4], window=700,
                               permute_pages=True, extra_pages=1)
    assert_fused_matches(w)


def test_window_validation():
    import decode_attention_block_memra_gb300 as memra
    w = W.make_window_workload("win_val", batch=1, q_len=2, n_heads=8, n_kv_heads=2, head_dim=128, k_fmt="q8_0",
                               v_fmt="q5_1", seed=5, seq_lens=[100], window=40)
    from decode_attention_block_memra_gb300.runner import upload
    dw = upload(w)
    with pytest.raises(memra.MemraError) as e:           # the ring cannot hold a 100-token window
        memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace,
                          w.sm_scale, window=100)
    assert e.value.status == 1
    with pytest.raises(memra.MemraError) as e:           # negative window
        memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace,
                          w.sm_scale, window=-3)
    assert e.value.status == 1


# ------------------------------------------------------- NVFP4 KV (kf4 arm) --

NVFP4_PAIRS = [("nvfp4", "nvfp4"), ("q8_0", "nvfp4"), ("nvfp4", "q5_1"), ("fp8", "nvfp4"), ("nvfp4", "fp8"),
               ("nvfp4", "q4_0")]


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kf,vf", NVFP4_PAIRS)
def test_nvfp4_formats(kf, vf, D):
    w = W.random_case(4000 + D + 7 * NVFP4_PAIRS.index((kf, vf)), batch=3, q_len=2, n_heads=16, n_kv_heads=2,
                      head_dim=D, k_fmt=kf, v_fmt=vf, ctx=(5, 2600))
    res = run(w)
    assert res.flags == 0
    assert_pools_exact(w, res)
    assert_out_close(w, res, attention.reference(w))


def test_nvfp4_fused_step_and_adversarial_blocks():
    w = W.random_case(4100, batch=4, q_len=8, n_heads=16, n_kv_heads=2, head_dim=128, k_fmt="nvfp4",
                      v_fmt="nvfp4", ctx=(8, 700))
    rng = np.random.default_rng(7)
    n = w.step_rows.size * w.n_kv_heads
    w.k_rows[w.step_rows] = _adversarial_rows(rng, n, 128).reshape(w.step_rows.size, w.n_kv_heads, 128)
    w.v_rows[w.step_rows] = _adversarial_rows(rng, n, 128).reshape(w.step_rows.size, w.n_kv_heads, 128)
    w.k_scale, w.v_scale = W._fp8_scales(w)
    res = assert_fused_matches(w)
    assert np.isfinite(res.out.astype(np.float32)).all()


def test_nvfp4_full_size_long_context():
    w = W.WORKLOADS["long_context"]().with_formats("nvfp4", "nvfp4")
    res = run(w)
    assert res.flags == 0
    check_everything(w, res)


# -------------------------------------------- numeric class across formats --

@pytest.mark.parametrize("kf,vf,D", [("fp8", "q4_0", 128), ("nvfp4", "nvfp4", 128), ("q8_0", "fp8", 256)])
def test_verify_rows_equal_plain_decode_other_formats(kf, vf, D):
    w = W.make_workload("verify_fmt", batch=3, q_len=4, n_heads=16, n_kv_heads=2, head_dim=D, k_fmt=kf, v_fmt=vf,
                        seed=77 + D, seq_lens=[2 * C + 3, C + 2, 300], permute_pages=True, extra_pages=1)
    out = _verify_vs_decode(w, fused=True)
    assert_out_close(w, SimpleNamespace(out=out), attention.reference(w))


@pytest.mark.parametrize("kf,vf", [("nvfp4", "q5_1"), ("fp8", "fp8")])
def test_window_fused_step_d256(kf, vf):
    w = W.make_window_workload("win_d256", batch=3, q_len=3, n_heads=8, n_kv_heads=2, head_dim=256, k_fmt=kf,
                               v_fmt=vf, seed=515, seq_lens=[3000, 513, 3], window=512, permute_pages=True)
    res = assert_fused_matches(w)
    assert_out_close(w, res, attention.reference(w))


# -------------------------------------- every fp16 value through the append --

def _all_fp16_finite():
    """Every finite fp16 value, as float16 (positive and negative, both zeros)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16)
    return v[np.isfinite(v)]


def _sweep_rows(fmt, rng):
    """Rows of 128 (4 blocks of 32) in which every finite fp16 value appears inside a block whose
    scale it does not exceed, for about 60 block scales from subnormal to 65,504."""
    allv = _all_fp16_finite().astype(np.float64)
    amaxes = np.unique(np.concatenate([[2.0 ** -24, 2.0 ** -20, 6.1e-5, 65504.0, 127.0, 7.0, 1.0, 0.5],
                                       2.0 ** rng.uniform(-14, 15.9, 52)]).astype(np.float16)).astype(np.float64)
    blocks = []
    for a in amaxes:
        if fmt == "q5_1":
            lo, hi = -a, a / 3
            vals = allv[(allv >= lo) & (allv <= hi)]
            head = [lo, hi]
        else:
            vals = allv[np.abs(allv) <= a]
            head = [a]
        n = 32 - len(head)
        pad = (-len(vals)) % n
        vals = np.concatenate([vals, np.zeros(pad)]).reshape(-1, n)
        blk = np.concatenate([np.tile(head, (vals.shape[0], 1)), vals], axis=1)
        blocks.append(blk)
    blocks = np.concatenate(blocks)
    rng.shuffle(blocks)
    blocks = np.concatenate([blocks, np.zeros(((-len(blocks)) % 4, 32))])
    return blocks.reshape(-1, 128).astype(np.float16)


@pytest.mark.parametrize("fmt,side", [("q8_0", "k"), ("q4_0", "v"), ("q5_1", "v"), ("fp8", "k"), ("nvfp4", "k"),
                                      ("nvfp4", "v")])
def test_append_every_fp16_value_bit_exact(fmt, side):
    """Quantize-append of every finite fp16 value, against blocks of ~60 scales, matches the oracle byte for byte."""
    import decode_attention_block_memra_gb300 as memra
    rng = np.random.default_rng(11)
    rows = _sweep_rows(fmt, rng)
    n = rows.shape[0]
    n_pages = -(-n // 16)
    other = np.zeros_like(rows)
    k_rows, v_rows = (rows, other) if side == "k" else (other, rows)
    k_fmt = fmt if side == "k" else "q8_0"
    v_fmt = fmt if side == "v" else "q5_1"
    scale = 1.0
    if fmt == "fp8":
        scale = float(np.float32(np.float32(65504.0) / np.float32(448.0)))
    elif fmt == "nvfp4":
        scale = float(np.float32(np.float32(65504.0) / np.float32(2688.0)))
    cache = memra.KVCache(k_fmt, v_fmt, n_pages, 1, 128, k_scale=scale, v_scale=scale, device="cuda")
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    memra.kv_append(cache, torch.from_numpy(k_rows).cuda().view(n, 1, 128), torch.from_numpy(v_rows).cuda().view(n, 1, 128),
                    slots)
    assert memra.read_status(cache) == 0
    pool = (cache.k_pool if side == "k" else cache.v_pool).cpu().numpy().reshape(n_pages, 1, -1)
    fields = quant.quantize_rows(rows, fmt, scale)
    want = np.zeros_like(pool)
    layout.write_rows(want, side, fields, np.arange(n), 0, 128)
    seg = pool.shape[-1]
    written = np.zeros(n_pages * seg, bool)      # bytes of the n rows (the last page may be partly empty)
    offs, _ = layout.row_bytes(side, fields, np.arange(n) % 16, 128)
    written.reshape(n_pages, seg)[np.broadcast_to((np.arange(n) // 16)[:, None], offs.shape), offs] = True
    got = pool.reshape(-1)[written]
    exp = want.reshape(-1)[written]
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"{bad.size} bytes differ"


# --------------------------------------------------- large query magnitudes --
# q8_0 keys enter the MMAs as biased codes, and the bias correction carries
# 1152 * (sum of a 32-element block of q) in fp16: a query whose block sums pass
# ~57 must still give the right scores (the row is scaled by a power of two).

def _large_query_case(seed, kf, vf, D, q_len=1, heads_scaled=None):
    w = W.random_case(seed, batch=3, q_len=q_len, n_heads=16, n_kv_heads=2, head_dim=D, k_fmt=kf, v_fmt=vf,
                      ctx=(q_len + 40, 2600))
    q = w.q.astype(np.float32)
    sel = slice(None) if heads_scaled is None else heads_scaled
    q[:, :, sel, :] *= 1e3                          # |q| up to ~4,500; block sums up to ~30,000
    w.q = q.astype(np.float16)
    w.k_rows = (w.k_rows.astype(np.float32) * 1e-3).astype(np.float16)
    w.k_scale, w.v_scale = W._fp8_scales(w)
    return w


@pytest.mark.parametrize("kf,vf,D", [("q8_0", "q5_1", 128), ("q8_0", "q4_0", 256), ("fp8", "q5_1", 128),
                                     ("nvfp4", "q4_0", 128)])
def test_large_query_magnitudes(kf, vf, D):
    w = _large_query_case(600 + D, kf, vf, D)
    res = run(w)
    assert res.flags == 0
    assert_out_close(w, res, attention.reference(w))


def test_large_and_ordinary_query_rows_in_one_cta():
    # heads 2, 3, 9 scaled up, the others ordinary: each row of an 8-head CTA keeps its own scale
    w = _large_query_case(611, "q8_0", "q5_1", 128, heads_scaled=[2, 3, 9])
    res = run(w)
    assert res.flags == 0
    assert_out_close(w, res, attention.reference(w))


def test_large_query_verify_rows_equal_plain_decode():
    w = _large_query_case(612, "q8_0", "q5_1", 128, q_len=4, heads_scaled=[0, 5, 6, 7, 12])
    out = _verify_vs_decode(w, fused=True)
    assert_out_close(w, SimpleNamespace(out=out), attention.reference(w))


# ----------------------------------------------------- the header's maximums --
# q_len up to MEMRA_MAX_Q_LEN (16: 15 drafts), groups up to MEMRA_MAX_GROUP
# (128 query heads on one KV head), and splits clamped at
# MEMRA_SPLIT_TOKENS_MAX (8,192 tokens) when T / S passes it.

@pytest.mark.parametrize("D", [128, 256])
def test_maximum_q_len(D):
    w = W.make_workload("max_qlen", batch=3, q_len=16, n_heads=16, n_kv_heads=2, head_dim=D, k_fmt="q8_0",
                        v_fmt="q5_1", seed=160 + D, seq_lens=[16, C + 6, 2100], permute_pages=True, extra_pages=2)
    res = run_fused(w)
    assert res.flags == 0
    full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)


def test_maximum_q_len_verify_rows_equal_plain_decode():
    K = 15
    w = W.make_workload("verify_k15", batch=3, q_len=K + 1, n_heads=32, n_kv_heads=4, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=215, seq_lens=[2 * C + 3 + K, C + 8, K + 1], permute_pages=True,
                        extra_pages=2)
    out = _verify_vs_decode(w, fused=True)
    assert_out_close(w, SimpleNamespace(out=out), attention.reference(w))


@pytest.mark.parametrize("q_len", [1, 2])
def test_maximum_group(q_len):
    # 128 query heads on one KV head: 16 CTAs of 8 heads per position and split
    w = W.make_workload("max_group", batch=2, q_len=q_len, n_heads=128, n_kv_heads=1, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=128 + q_len, seq_lens=[q_len + 300, 2500], permute_pages=True)
    res = run_fused(w)
    assert res.flags == 0
    full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)


def test_head_dim_256_splits_above_the_smallest():
    """At head_dim 256 the plan targets three CTAs per SM: a sequence longer than MEMRA_SPLIT_TOKENS x
    (SMs x 3 / KV heads) gets splits wider than the smallest, set by its length (verify rows too)."""
    import decode_attention_block_memra_gb300 as memra
    n_kv = 2
    S = max(1, torch.cuda.get_device_properties(0).multi_processor_count * 3 // n_kv)
    T = S * memra.SPLIT_TOKENS + 40_003                 # -(-T // S) passes the smallest split
    assert -(-T // S) > memra.SPLIT_TOKENS
    w = W.make_workload("d256_wide_splits", batch=1, q_len=2, n_heads=16, n_kv_heads=n_kv, head_dim=256,
                        k_fmt="fp8", v_fmt="q4_0", seed=256, seq_lens=[T], permute_pages=True)
    res = run_fused(w)
    assert res.flags == 0
    full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)


def test_splits_at_the_largest_split_size():
    import decode_attention_block_memra_gb300 as memra
    n_kv = 32
    S = max(1, torch.cuda.get_device_properties(0).multi_processor_count * 2 // n_kv)
    T = 80_000
    assert -(-T // S) > memra.SPLIT_TOKENS and -(-T // S) > 8192     # T / S passes the 8,192-token clamp
    w = W.make_workload("split_cap", batch=1, q_len=2, n_heads=32, n_kv_heads=n_kv, head_dim=128, k_fmt="q8_0",
                        v_fmt="q4_0", seed=8192, seq_lens=[T], permute_pages=True)
    res = run_fused(w)
    assert res.flags == 0
    full_parity.check(w, res.out, res.k_pool, res.v_pool, res.initial_k_pool, res.initial_v_pool, tol=TOL)
