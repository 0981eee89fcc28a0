"""Length-balanced work units vs the oracle.

With two or more sequences the decode kernel lays the (sequence, KV head)
pairs end to end and gives every CTA an equal range of 32-token blocks, so the
blocks of one pair can be spread over several CTAs (at most num_splits of
them) and one CTA can hold pieces of several pairs.  These cases aim at the
edges of that assignment: empty, one-token and clamped sequences, block
boundaries, a long sequence among short ones (the per-CTA range is then set
by the slot count, not by the lengths), many short pairs (many units per CTA)
and grids where most CTAs are idle.  The kernel reads the oracle's own codes,
so the comparison isolates the assignment and the attention arithmetic.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import GpuCache, calib_for, check_outputs, oracle_attention, oracle_encode

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _filled(w, n_max):
    """The oracle's codes for tokens [0, n_max[b]) of every sequence."""
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    refs = []
    for b in range(w.batch):
        n = int(n_max[b])
        r = oracle_encode(w, cal, b, 0, max(n, 1))
        if n > 0:
            gc.write_codes(b, 0, r.kc[:n], r.vc[:n])
        refs.append(r)
    return cal, gc, refs


def _decode(gc, q, lens, max_seq_len, splits):
    seq = torch.from_numpy(np.asarray(lens, dtype=np.int32)).to(gc.device)
    out = gc.vq.decode_attention(gc.layout, torch.from_numpy(q).to(gc.device), gc.lam, gc.ck, gc.cv,
                                 gc.k_pool, gc.v_pool, gc.page_table, seq, max_seq_len,
                                 num_splits=splits, status=gc.status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _check(w, cal, refs, q, got, lens, max_seq_len, label):
    for b in range(w.batch):
        n = min(max(int(lens[b]), 0), max_seq_len)
        if n == 0:
            assert not got[b].any(), (label, b)
            continue
        ref = oracle_attention(w, cal, q[b], refs[b].kc[:n], refs[b].vc[:n])
        check_outputs(got[b:b + 1], ref[None], f"{label} b={b} n={n}")


def _ragged_lens(batch, context, seed):
    """Mixed lengths: empty, one token, block edges (31, 32, 33, 64), full and random."""
    rng = np.random.default_rng(seed)
    edge = [0, 1, 31, 32, 33, 64, context + 1, context, context - 31]
    lens = rng.integers(0, context + 2, size=batch)
    lens[:len(edge)] = edge[:batch]
    return rng.permutation(lens)


@pytest.mark.parametrize("splits", [0, 2, 5, 40])
def test_balanced_ragged_with_empty_and_edge_lengths(splits):
    w = W.custom(name="bal-ragged", batch=37, num_q_heads=8, num_kv_heads=2, context=900, k_sub=2,
                 v_sub=4, page_size=64)
    lens = _ragged_lens(w.batch, w.context, 11)
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    got = _decode(gc, q, lens, w.context + 1, splits)
    assert gc.device_status() == 0
    _check(w, cal, refs, q, got, lens, w.context + 1, f"splits={splits}")


def test_balanced_lengths_clamped_to_max_seq_len():
    """Tokens at or past max_seq_len are ignored; the clamped lengths set the units."""
    w = W.custom(name="bal-clamp", batch=9, num_q_heads=8, num_kv_heads=2, context=900, k_sub=4,
                 v_sub=4, page_size=128)
    lens = np.array([901, 600, 601, 599, 0, 900, 17, 640, 800])
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    for splits in (0, 3):
        got = _decode(gc, q, lens, 600, splits)
        assert gc.device_status() == 0
        _check(w, cal, refs, q, got, lens, 600, f"clamped splits={splits}")


@pytest.mark.parametrize("splits", [2, 3])
def test_balanced_long_sequence_among_short_ones(splits):
    """One 3001-token sequence with three short ones: the per-CTA range is
    ceil(blocks / (splits - 1)), so the long pairs still fit their slots."""
    w = W.custom(name="bal-long", batch=4, num_q_heads=8, num_kv_heads=2, context=3000, k_sub=2,
                 v_sub=4, page_size=256)
    lens = np.array([7, 3001, 0, 45])
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    got = _decode(gc, q, lens, 3001, splits)
    assert gc.device_status() == 0
    _check(w, cal, refs, q, got, lens, 3001, f"long splits={splits}")


def test_balanced_many_short_pairs_per_cta():
    """300 sequences x 2 KV heads of 0-41 tokens: 600 pairs over the grid,
    several whole pairs per CTA."""
    w = W.custom(name="bal-many", batch=300, num_q_heads=4, num_kv_heads=2, context=40, k_sub=4,
                 v_sub=4, page_size=16)
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 42, size=w.batch)
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    got = _decode(gc, q, lens, 41, 0)
    assert gc.device_status() == 0
    _check(w, cal, refs, q, got, lens, 41, "many")


def test_balanced_grid_mostly_idle():
    """Two sequences of one and two tokens: four pairs, most CTAs get no unit."""
    w = W.custom(name="bal-idle", batch=2, num_q_heads=4, num_kv_heads=2, context=8, k_sub=2,
                 v_sub=4, page_size=16)
    lens = np.array([1, 2])
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    for splits in (0, 2):
        got = _decode(gc, q, lens, 2, splits)
        assert gc.device_status() == 0
        _check(w, cal, refs, q, got, lens, 2, f"idle splits={splits}")


def test_balanced_matches_fixed_splits():
    """The same batch with one split (fixed assignment) and with length-balanced
    units agrees to fp32 rounding of the merge."""
    w = W.custom(name="bal-vs-fixed", batch=16, num_q_heads=32, num_kv_heads=8, context=1024,
                 k_sub=2, v_sub=4, page_size=64, ragged=True, ragged_lo=512, ragged_hi=1024,
                 permuted_pages=True)
    lens = W.seq_lens(w) + 1
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    fixed = _decode(gc, q, lens, int(lens.max()), 1)
    bal = _decode(gc, q, lens, int(lens.max()), 0)
    assert gc.device_status() == 0
    assert np.max(np.abs(fixed - bal)) < 1e-3
    _check(w, cal, refs, q, bal, lens, int(lens.max()), "balanced cfg2-reduced")


@pytest.mark.parametrize("splits", [0, 2])
def test_balanced_loose_max_seq_len(splits):
    """max_seq_len far above the real lengths: the per-CTA range comes from the
    batch's own longest sequence, and the outputs still match the oracle."""
    w = W.custom(name="bal-loose", batch=6, num_q_heads=8, num_kv_heads=2, context=900, k_sub=4,
                 v_sub=4, page_size=64)
    lens = np.array([17, 200, 0, 65, 1, 130])
    cal, gc, refs = _filled(w, lens)
    q = W.queries(w)
    got = _decode(gc, q, lens, 901, splits)
    assert gc.device_status() == 0
    _check(w, cal, refs, q, got, lens, 901, f"loose splits={splits}")
