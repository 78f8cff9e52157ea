"""Pins for the oracle's attention on the dequantized paged cache (CPU only)."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention, quant


def brute_force(q, k, v, sm_scale):
    """Explicit loops: one query row, one head, one key at a time."""
    Q, Hq, D = q.shape
    T, Hkv, _ = k.shape
    G = Hq // Hkv
    out = np.zeros((Q, Hq, D))
    for i in range(Q):
        last = T - Q + i
        for h in range(Hq):
            kh = h // G
            scores = []
            for t in range(last + 1):
                s = 0.0
                for j in range(D):
                    s += float(q[i, h, j]) * float(k[t, kh, j])
                scores.append(s * sm_scale)
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            tot = sum(ws)
            for j in range(D):
                acc = 0.0
                for t in range(last + 1):
                    acc += ws[t] * float(v[t, kh, j])
                out[i, h, j] = acc / tot
    return out


@pytest.mark.parametrize("Q,Hq,Hkv,T", [(1, 4, 2, 5), (3, 4, 1, 7), (2, 6, 3, 2)])
def test_matches_brute_force(Q, Hq, Hkv, T):
    rng = np.random.default_rng(Q * 100 + T)
    D = 8
    q = rng.standard_normal((Q, Hq, D))
    k = rng.standard_normal((T, Hkv, D))
    v = rng.standard_normal((T, Hkv, D))
    got = attention.attention_rows(q, k, v, 1 / math.sqrt(D))
    want = brute_force(q, k, v, 1 / math.sqrt(D))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_context_one_returns_the_v_row():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 8, 128)) * 50
    k = rng.standard_normal((1, 2, 128))
    v = rng.standard_normal((1, 2, 128))
    out = attention.attention_rows(q, k, v, 1 / math.sqrt(128))
    for h in range(8):
        assert np.array_equal(out[0, h], v[0, h // 4])


def test_zero_query_averages_visible_rows():
    rng = np.random.default_rng(3)
    T, Q = 37, 4
    k = rng.standard_normal((T, 2, 64))
    v = rng.standard_normal((T, 2, 64))
    out = attention.attention_rows(np.zeros((Q, 4, 64)), k, v, 0.125)
    for i in range(Q):
        for h in range(4):
            np.testing.assert_allclose(out[i, h], v[: T - Q + i + 1, h // 2].mean(axis=0), rtol=0, atol=1e-14)


@pytest.mark.parametrize("Q,G", [(1, 8), (4, 8), (2, 2)])
def test_matches_torch_sdpa_float64(Q, G):
    rng = np.random.default_rng(Q + 10 * G)
    Hkv, D, T = 2, 128, 300
    Hq = Hkv * G
    x = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    k_hat = quant.dequantize_rows(quant.quantize_rows(x, "q8_0"))
    v_hat = quant.dequantize_rows(quant.quantize_rows(rng.standard_normal((T, Hkv, D)).astype(np.float16), "q5_1"))
    q = rng.standard_normal((Q, Hq, D)).astype(np.float16)
    got = attention.attention_rows(q, k_hat, v_hat, 1 / math.sqrt(D))
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)                 # [Hq, Q, D]
    kt = torch.from_numpy(k_hat).permute(1, 0, 2).repeat_interleave(G, dim=0)    # [Hq, T, D]
    vt = torch.from_numpy(v_hat).permute(1, 0, 2).repeat_interleave(G, dim=0)
    mask = torch.arange(T)[None, :] <= (T - Q + torch.arange(Q))[:, None]      # [Q, T]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1 / math.sqrt(D))
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


def test_page_placement_does_not_change_outputs():
    a = W.random_case(21, batch=3, q_len=2, ctx=(20, 90), permute_pages=False, extra_pages=0)
    b = W.random_case(21, batch=3, q_len=2, ctx=(20, 90), permute_pages=True, extra_pages=0)
    assert not np.array_equal(a.page_table, b.page_table)
    assert np.array_equal(attention.reference(a), attention.reference(b))


def test_shared_prefix_pages_are_aliased():
    w = W.make_workload("sp", batch=3, q_len=1, n_heads=4, n_kv_heads=2, head_dim=128, k_fmt="q8_0",
                        v_fmt="q5_1", seed=9, seq_lens=[40, 57, 33], shared_prefix=32)
    assert np.array_equal(w.page_table[0, :2], w.page_table[1, :2]) and np.array_equal(w.page_table[0, :2],
                                                                                         w.page_table[2, :2])
    out = attention.reference(w)
    # sequence b alone, written out without pages, gives the same numbers
    cache = attention.quantize_cache(w)
    for b in range(3):
        rows = attention.sequence_rows(w, b)
        kh = np.stack([quant.dequantize_rows(quant.select_rows(cache["k"][h], rows)) for h in range(2)], 1)
        vh = np.stack([quant.dequantize_rows(quant.select_rows(cache["v"][h], rows)) for h in range(2)], 1)
        np.testing.assert_array_equal(out[b], attention.attention_rows(w.q[b], kh, vh, w.sm_scale))


def test_rows_subset_matches_full():
    w = W.random_case(5, batch=2, q_len=3, n_heads=8, n_kv_heads=2, ctx=(30, 70))
    full = attention.reference(w)
    sub = attention.reference(w, rows=[(1, 2, 5), (0, 0, 0)])
    assert np.array_equal(sub[1, 2, 5], full[1, 2, 5]) and np.array_equal(sub[0, 0, 0], full[0, 0, 0])
    assert np.isnan(sub[1, 0, 0]).all()


def test_workload_recipe():
    w = W.tiny()
    assert w.q.shape == (1, 1, 8, 128) and w.k_rows.shape == (256, 2, 128) and w.num_pages == 16
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 1, 8, 128)).astype(np.float16)
    assert np.array_equal(q, w.q)
    sp = W.make_workload("x", batch=2, q_len=1, n_heads=4, n_kv_heads=1, head_dim=128, k_fmt="fp8", v_fmt="fp8",
                         seed=1, seq_lens=[20, 20])
    assert sp.k_scale == float(np.float32(np.abs(sp.k_rows.astype(np.float32)).max() / np.float32(448)))


# ------------------------------------------------ sliding window (SWA ring) --

def brute_force_window(q, k, v, sm_scale, window):
    """Explicit loops with the window: row i (position T - Q + i) sees keys max(0, pos - window + 1) .. pos."""
    Q, Hq, D = q.shape
    T, Hkv, _ = k.shape
    G = Hq // Hkv
    out = np.zeros((Q, Hq, D))
    for i in range(Q):
        pos = T - Q + i
        keys = [t for t in range(T) if pos - window < t <= pos]
        for h in range(Hq):
            kh = h // G
            scores = [sum(float(q[i, h, j]) * float(k[t, kh, j]) for j in range(D)) * sm_scale for t in keys]
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            for j in range(D):
                out[i, h, j] = sum(wt * float(v[t, kh, j]) for wt, t in zip(ws, keys)) / sum(ws)
    return out


@pytest.mark.parametrize("Q,T,window", [(1, 9, 3), (3, 11, 4), (2, 6, 1), (4, 5, 16)])
def test_window_matches_brute_force(Q, T, window):
    rng = np.random.default_rng(7 * T + window)
    D = 8
    q = rng.standard_normal((Q, 4, D))
    k = rng.standard_normal((T, 2, D))
    v = rng.standard_normal((T, 2, D))
    got = attention.attention_rows(q, k, v, 0.3, window=window)
    np.testing.assert_allclose(got, brute_force_window(q, k, v, 0.3, window), rtol=1e-12, atol=1e-12)


def test_window_of_one_returns_the_own_v_row():
    rng = np.random.default_rng(8)
    T, Q = 30, 3
    q = rng.standard_normal((Q, 4, 64)) * 20
    k = rng.standard_normal((T, 2, 64))
    v = rng.standard_normal((T, 2, 64))
    out = attention.attention_rows(q, k, v, 0.125, window=1)
    for i in range(Q):
        for h in range(4):
            assert np.array_equal(out[i, h], v[T - Q + i, h // 2])


def test_window_zero_query_averages_the_window():
    rng = np.random.default_rng(9)
    T, Q, window = 50, 4, 7
    k = rng.standard_normal((T, 1, 32))
    v = rng.standard_normal((T, 1, 32))
    out = attention.attention_rows(np.zeros((Q, 2, 32)), k, v, 0.2, window=window)
    for i in range(Q):
        pos = T - Q + i
        np.testing.assert_allclose(out[i, 0], v[pos - window + 1: pos + 1, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_window_wider_than_context_is_full_attention():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((3, 4, 16))
    k = rng.standard_normal((20, 2, 16))
    v = rng.standard_normal((20, 2, 16))
    assert np.array_equal(attention.attention_rows(q, k, v, 0.25, window=20),
                          attention.attention_rows(q, k, v, 0.25))


@pytest.mark.parametrize("Q,window", [(1, 100), (4, 37)])
def test_window_matches_torch_sdpa_band_mask(Q, window):
    rng = np.random.default_rng(Q + window)
    Hkv, G, D, T = 2, 4, 64, 300
    Hq = Hkv * G
    k_hat = rng.standard_normal((T, Hkv, D))
    v_hat = rng.standard_normal((T, Hkv, D))
    q = rng.standard_normal((Q, Hq, D))
    got = attention.attention_rows(q, k_hat, v_hat, 1 / math.sqrt(D), window=window)
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k_hat).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = torch.from_numpy(v_hat).permute(1, 0, 2).repeat_interleave(G, dim=0)
    pos = (T - Q + torch.arange(Q))[:, None]
    t = torch.arange(T)[None, :]
    mask = (t <= pos) & (t > pos - window)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1 / math.sqrt(D))
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


def test_ring_workload_reads_the_rows_of_each_position():
    """Through the ring page table, each position's slot holds that position's row (drawn in position order)."""
    w = W.make_window_workload("ring", batch=3, q_len=3, n_heads=4, n_kv_heads=2, head_dim=128, k_fmt="q8_0",
                               v_fmt="q5_1", seed=12, seq_lens=[200, 45, 3], window=40, permute_pages=True,
                               extra_pages=2)
    R = w.page_table.shape[1]
    assert R == W.min_ring_pages(40, 3) == 4
    assert list(w.first_pos) == [(199 // 16 - R + 1) * 16, 0, 0]
    # slots of the resident rows are distinct (a ring never holds two live positions in one slot)
    assert np.unique(w.slots).size == w.slots.size
    base = 0
    for b in range(3):
        rows = attention.sequence_rows(w, b)
        n = int(w.seq_lens[b]) - int(w.first_pos[b])
        assert np.array_equal(rows, np.arange(base, base + n))
        base += n
    # the oracle on the ring equals the plain window attention on rows in position order
    cache = attention.quantize_cache(w)
    out = attention.reference(w, cache=cache)
    base = 0
    for b in range(3):
        n = int(w.seq_lens[b]) - int(w.first_pos[b])
        rows = np.arange(base, base + n)
        kh = np.stack([quant.dequantize_rows(quant.select_rows(cache["k"][h], rows)) for h in range(2)], 1)
        vh = np.stack([quant.dequantize_rows(quant.select_rows(cache["v"][h], rows)) for h in range(2)], 1)
        ref = attention.attention_rows(w.q[b], kh[-min(n, 40 + 2):], vh[-min(n, 40 + 2):], w.sm_scale, window=40,
                                       start=int(w.seq_lens[b]) - min(n, 42))
        np.testing.assert_array_equal(out[b], ref)
        base += n


def test_window_reaching_below_the_rows_given_raises():
    with pytest.raises(ValueError):
        attention.attention_rows(np.zeros((1, 1, 8)), np.zeros((5, 1, 8)), np.zeros((5, 1, 8)), 1.0, window=7,
                                 start=10)
