"""Seeded workload generators: determinism, shapes, distributions, cache layout."""
import numpy as np
import pytest

import workloads as W


def test_table_matches_workload_shapes():
    w = W.WORKLOADS
    assert (w[0].batch, w[0].num_q_heads, w[0].num_kv_heads, w[0].context) == (1, 2, 1, 1024)
    assert (w[1].num_q_heads, w[1].num_kv_heads, w[1].context) == (32, 8, 32768)
    assert (w[2].batch, w[2].page_size, w[2].ragged_lo, w[2].ragged_hi) == (16, 64, 4096, 8192)
    assert (w[3].context, w[3].drift) == (196608, True)
    assert (w[4].batch, w[4].num_q_heads, w[4].group, w[4].v_bits) == (64, 40, 5, 9)
    assert (w[5].k_sub, w[5].k_bits, w[5].v_sub, w[5].v_bits) == (8, 12, 8, 12)
    assert [x.k_code_bytes() + x.v_code_bytes() for x in w.values()] == [96, 64, 96, 64, 100, 48]


def test_kv_tokens_deterministic_and_windowed():
    w = W.custom(context=300, num_kv_heads=2, num_q_heads=4)
    a = W.kv_tokens(w, 0, "k")
    assert a.dtype == np.float16 and a.shape == (301, 2, 128)
    assert np.array_equal(a, W.kv_tokens(w, 0, "k"))
    assert np.array_equal(a[37:211], W.kv_tokens(w, 0, "k", 37, 211))
    assert not np.array_equal(a, W.kv_tokens(w, 0, "v"))


def test_kv_tokens_blocks_equal_single_draw(monkeypatch):
    w = W.custom(context=1000, num_kv_heads=2, num_q_heads=2)
    a = W.kv_tokens(w, 0, "v")
    monkeypatch.setattr(W, "_BLOCK_ROWS", 7)
    assert np.array_equal(a, W.kv_tokens(w, 0, "v"))
    assert np.array_equal(a[500:503], W.kv_tokens(w, 0, "v", 500, 503))


def test_outlier_channels_scaled():
    w = W.custom(context=4000, num_kv_heads=2, num_q_heads=2)
    k = W.kv_tokens(w, 0, "k").astype(np.float64)
    ch = W.outlier_channels(w)
    assert ch.shape == (2, 4) and len(set(ch[0])) == 4
    for h in range(2):
        std = k[:, h, :].std(0)
        assert np.all(std[ch[h]] > 15) and np.median(std) < 1.2


def test_drift_range():
    w = W.custom(context=4000, drift=True)
    k = W.kv_tokens(w, 0, "k").astype(np.float64)
    ch = W.outlier_channels(w)[0]
    other = [c for c in range(128) if c not in ch]
    head, tail = k[:500, 0, other].std(), k[-500:, 0, other].std()
    assert 2.4 < tail / head < 3.2


def test_ragged_lengths_and_pages():
    w = W.WORKLOADS[2]
    n = W.seq_lens(w)
    assert n.min() >= 4096 and n.max() <= 8192 and len(set(n.tolist())) > 8
    tab = W.page_table(w)
    used = tab[tab >= 0]
    assert len(used) == W.num_pages(w) and len(set(used.tolist())) == len(used)
    assert not np.array_equal(np.sort(used), used)          # permuted
    for b in range(w.batch):
        assert (tab[b] >= 0).sum() == -(-(n[b] + 1) // 64)


def test_slot_mapping_matches_page_table():
    w = W.WORKLOADS[2]
    tab = W.page_table(w)
    s = W.slot_mapping(w, 3, 60, 70)
    t = np.arange(60, 70)
    assert np.array_equal(s, tab[3][t // 64] * 64 + t % 64)


def test_contiguous_identity_pages():
    w = W.WORKLOADS[1]
    tab = W.page_table(w)
    assert np.array_equal(tab[0], np.arange(tab.shape[1]))
    assert W.num_pages(w) * w.page_size >= w.context + 1


def test_queries_and_calibration_shapes():
    w = W.WORKLOADS[1]
    q = W.queries(w)
    assert q.shape == (1, 32, 128) and q.dtype == np.float16
    kc, vc = W.calibration(W.WORKLOADS[0])
    assert kc.shape == (W.CALIB_TOKENS, 1, 128) and vc.shape == kc.shape


def test_kmeans_init_distinct():
    idx = W.kmeans_init(10000, 512, "v")
    assert len(set(idx.tolist())) == 512 and idx.max() < 10000
