"""Host bound of the length-balanced work assignment (CPU).

When the library reports length-balanced units for a call
(vq_decode_units_balanced == 1), the decode kernel lays the (sequence, KV
head) pairs end to end (each pair's 32-token blocks followed by a 12-block gap
standing for a unit's fixed cost), and CTA c of a grid of one CTA per SM takes
positions [c W, (c + 1) W) with W = max(ceil(total / grid), ceil(longest
pair's blocks / (S - 1))).  The kernel keeps at most 256 units per CTA and S
partial slots per pair.  These tests restate that rule with numpy and check,
on adversarial length mixes, that every shape the library accepts keeps both
limits, that every block of every pair lands in exactly one CTA, and that a
short batch under a loose max_seq_len stays spread over the grid.
"""
import numpy as np
import pytest

import bit_vector_quantized_gb300 as vq

GAP = 12
MAX_UNITS = 256


@pytest.fixture(scope="module")
def lib():
    return vq.lib()


def _assign(lens, hkv, max_seq_len, splits, grid):
    nb = (np.clip(lens, 0, max_seq_len) + 31) // 32
    nb_pair = np.repeat(nb, hkv).astype(np.int64)
    cost = nb_pair + GAP
    q = np.concatenate([[0], np.cumsum(cost)[:-1]])
    ext = np.maximum(nb_pair, 1)
    total = int(cost.sum())
    w = max(-(-total // grid), -(-int(nb_pair.max()) // (splits - 1)))
    c = np.arange(grid, dtype=np.int64)
    x0, x1 = c * w, (c + 1) * w
    pa = np.searchsorted(q + ext, x0, side="right")   # first pair with q + ext > x0
    pb = np.searchsorted(q, x1, side="left") - 1       # last pair with q < x1
    units = np.maximum(pb - pa + 1, 0)
    pieces = (q + ext - 1) // w - q // w + 1
    return units, pieces, q, nb_pair, w


def _mixes(rng, batch, max_seq_len):
    """Length vectors aimed at many units per CTA: all short, one long among
    short ones, empty sequences, alternating long and short, random."""
    yield np.full(batch, 1)
    yield np.concatenate([[max_seq_len], np.ones(batch - 1, dtype=np.int64)])
    yield np.concatenate([[max_seq_len], np.zeros(batch - 1, dtype=np.int64)])
    yield np.where(np.arange(batch) % 2 == 0, max_seq_len, 1)
    yield np.full(batch, max_seq_len)
    yield rng.integers(0, max_seq_len + 1, size=batch)
    yield rng.integers(0, 33, size=batch)


@pytest.mark.parametrize("hkv", [1, 2, 8])
def test_accepted_shapes_keep_the_kernel_limits(lib, hkv):
    rng = np.random.default_rng(5)
    checked = 0
    for batch in (2, 3, 17, 64, 255, 256, 257, 512):
        for max_seq_len in (1, 33, 1000, 16385, 131073, 1 << 20):
            for grid in (152, 148, 7):
                L = vq.make_layout(num_q_heads=hkv * 4, num_kv_heads=hkv)
                for splits in (0, 2, 3):
                    s = splits or vq.vq_default_num_splits(L, batch, max_seq_len, grid)
                    if vq.vq_decode_units_balanced(L, batch, max_seq_len, splits, grid) != 1:
                        continue
                    for lens in _mixes(rng, batch, max_seq_len):
                        units, pieces, _, _, _ = _assign(lens, hkv, max_seq_len, s, grid)
                        assert units.max() <= MAX_UNITS, (batch, max_seq_len, grid, s)
                        assert pieces.max() <= s, (batch, max_seq_len, grid, s)
                        checked += 1
    assert checked > 100


def test_every_block_in_one_cta(lib):
    """The CTA ranges [c W, (c + 1) W) tile the positions, so each block of a
    pair (at position q + i) falls in exactly one CTA, and the pieces of a
    pair are the CTAs from q // W to (q + nb - 1) // W."""
    rng = np.random.default_rng(9)
    for _ in range(50):
        batch = int(rng.integers(2, 40))
        hkv = int(rng.choice([1, 2, 8]))
        max_seq_len = int(rng.integers(1, 5000))
        lens = rng.integers(0, max_seq_len + 1, size=batch)
        s = int(rng.integers(2, 9))
        units, pieces, q, nb, w = _assign(lens, hkv, max_seq_len, s, 152)
        owner = np.concatenate([(q[p] + np.arange(nb[p])) // w for p in range(len(q))])
        assert owner.max(initial=0) < 152
        per_cta = np.bincount(owner, minlength=152)
        assert per_cta.max() <= w                    # no CTA gets more than its range
        assert int(per_cta.sum()) == int(nb.sum())   # every block counted once


def test_loose_max_seq_len_keeps_a_short_batch_spread(lib):
    """256 one-token sequences under max_seq_len 131073: the slot term comes
    from the batch's own longest sequence, so no CTA holds more than a few
    pairs (a term from max_seq_len would put all 256 in one CTA)."""
    L = vq.make_layout(num_q_heads=4, num_kv_heads=1)
    s = vq.vq_default_num_splits(L, 256, 131073, 152)
    assert vq.vq_decode_units_balanced(L, 256, 131073, 0, 152) == 1
    units, pieces, _, _, _ = _assign(np.ones(256, dtype=np.int64), 1, 131073, s, 152)
    assert units.max() <= 3 and pieces.max() == 1
