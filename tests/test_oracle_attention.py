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
