"""Seeded synthetic workloads for VQ KV-cache decode attention.

This module is shared by the CUDA path (bench, tests) and by the oracle's test
harness.  It holds the workload table and the seeded random draws only: no
smoothing factor, no Hadamard transform, no clustering, no encoding and no
attention arithmetic live here.

Workloads follow the five shapes of the decode-attention study (VecInfer,
"Experimental setup" / "Kernel implementation details"): Llama-3.1-8B and
Qwen2.5-14B layer shapes, 32K and 196K context, batched ragged decode.  The
pages measure on LongBench / GSM8K text; these seeded Gaussian tensors stand in
for those datasets.

Seeds (all through ``numpy.random.SeedSequence`` so every (sequence, tensor)
stream can be regenerated on its own):
  0  test K and V            spawn key (b, 0) for K, (b, 1) for V
  1  calibration K and V     spawn key (0,) for K, (1,) for V, (2,) drift positions
  2  K codebook init         (used by the calibration script)
  3  V codebook init
  4  decode queries
  5  outlier channels
  6  ragged sequence lengths
  7  physical page permutation

Token convention: a workload's context length ``N`` is the number of tokens
already in the cache (the prefill); every decode step appends one more token
(position ``N``) and the query attends over ``N + 1`` tokens.  The K/V streams
therefore hold ``N + 1`` rows per sequence.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

HEAD_DIM = 128
CALIB_TOKENS = 16384          # calibration vectors per KV head
OUTLIERS_PER_HEAD = 4
OUTLIER_SCALE = 20.0
KMEANS_ITERS = 10
_BLOCK_ROWS = 8192


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-attention workload (shapes, code formats, cache layout)."""
    index: int
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    context: int                  # N: cached tokens before the decode step
    k_sub: int                    # d_k, sub-vector length of K codes
    k_bits: int                   # b_k, bits per K code (2**b_k centroids)
    v_sub: int
    v_bits: int
    page_size: int
    ragged: bool = False          # per-sequence N drawn from [ragged_lo, ragged_hi]
    ragged_lo: int = 0
    ragged_hi: int = 0
    permuted_pages: bool = False  # physical pages shuffled (paged cache)
    drift: bool = False           # K channel scale drifts x1 -> x3 over positions
    head_dim: int = HEAD_DIM

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def k_code_bytes(self) -> int:
        """Packed bytes of one token-head's K codes (rounded up to 4)."""
        return _round4(-(-(self.head_dim // self.k_sub) * self.k_bits // 8))

    def v_code_bytes(self) -> int:
        return _round4(-(-(self.head_dim // self.v_sub) * self.v_bits // 8))


def _round4(x: int) -> int:
    return (x + 3) // 4 * 4


WORKLOADS: Dict[int, Workload] = {
    0: Workload(0, "tiny-b1-g2-n1024", batch=1, num_q_heads=2, num_kv_heads=1,
                context=1024, k_sub=2, k_bits=8, v_sub=4, v_bits=8, page_size=256),
    1: Workload(1, "llama3.1-8b-b1-n32768", batch=1, num_q_heads=32, num_kv_heads=8,
                context=32768, k_sub=4, k_bits=8, v_sub=4, v_bits=8, page_size=256),
    2: Workload(2, "ragged-b16-n4096to8192-paged64", batch=16, num_q_heads=32,
                num_kv_heads=8, context=8192, k_sub=2, k_bits=8, v_sub=4, v_bits=8,
                page_size=64, ragged=True, ragged_lo=4096, ragged_hi=8192,
                permuted_pages=True),
    3: Workload(3, "llama3.1-8b-b1-n196608-drift", batch=1, num_q_heads=32,
                num_kv_heads=8, context=196608, k_sub=4, k_bits=8, v_sub=4, v_bits=8,
                page_size=256, drift=True),
    4: Workload(4, "qwen2.5-14b-b64-n16384", batch=64, num_q_heads=40, num_kv_heads=8,
                context=16384, k_sub=2, k_bits=8, v_sub=4, v_bits=9, page_size=256),
    # The pages' 1.5-bit configuration (VecInfer, 实验结果, codebook-size ablation:
    # 2^12 centroids of 8 elements for 1.5 bits) on the 32K Llama layer.
    5: Workload(5, "llama3.1-8b-b1-n32768-1.5bit", batch=1, num_q_heads=32, num_kv_heads=8,
                context=32768, k_sub=8, k_bits=12, v_sub=8, v_bits=12, page_size=256),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(entropy=seed, spawn_key=tuple(key)))


def outlier_channels(w: Workload) -> np.ndarray:
    """int64 [Hkv][4]: the K channels of each KV head that carry outliers (seed 5)."""
    rng = _rng(5)
    return np.stack([np.sort(rng.choice(w.head_dim, OUTLIERS_PER_HEAD, replace=False))
                     for _ in range(w.num_kv_heads)])


def seq_lens(w: Workload) -> np.ndarray:
    """int64 [B]: cached context per sequence before the decode step (seed 6)."""
    if not w.ragged:
        return np.full(w.batch, w.context, dtype=np.int64)
    return _rng(6).integers(w.ragged_lo, w.ragged_hi, endpoint=True, size=w.batch).astype(np.int64)


def _drift(pos: np.ndarray, total: int) -> np.ndarray:
    """Channel-scale drift factor x1 at position 0 to x3 at the last position."""
    return 1.0 + 2.0 * pos / max(total - 1, 1)


def _shape_keys(x: np.ndarray, w: Workload, pos: np.ndarray, total: int) -> np.ndarray:
    """Outlier channels x20, then (drift workloads) the positional drift; fp64 in-place."""
    ch = outlier_channels(w)
    for h in range(w.num_kv_heads):
        x[:, h, ch[h]] *= OUTLIER_SCALE
    if w.drift:
        x *= _drift(pos.astype(np.float64), total)[:, None, None]
    return x


def kv_tokens(w: Workload, b: int, which: str, start: int = 0,
              stop: Optional[int] = None) -> np.ndarray:
    """fp16 [T][Hkv][D] keys ('k') or values ('v') of sequence ``b``, rows start:stop.

    The stream of sequence b has ``seq_lens[b] + 1`` rows (prefill plus the one
    appended decode token).  Rows are N(0,1); keys get the outlier channels and,
    for drift workloads, the positional channel-scale drift, all before the
    fp16 cast (round to nearest even).
    """
    n_rows = int(seq_lens(w)[b]) + 1
    stop = n_rows if stop is None else stop
    assert 0 <= start <= stop <= n_rows
    rng = _rng(0, b, 0 if which == "k" else 1)
    out = np.empty((stop - start, w.num_kv_heads, w.head_dim), dtype=np.float16)
    row = 0
    while row < stop:  # bounded blocks; chunked draws equal one large draw
        n = min(_BLOCK_ROWS, stop - row)
        x = rng.standard_normal((n, w.num_kv_heads, w.head_dim))
        lo, hi = max(row, start), row + n
        if hi > lo:
            x = x[lo - row:]
            if which == "k":
                x = _shape_keys(x, w, np.arange(lo, hi), n_rows)
            out[lo - start:hi - start] = x.astype(np.float16)
        row += n
    return out


def calibration(w: Workload) -> tuple:
    """fp16 (K_cal, V_cal), each [16384][Hkv][D], drawn like the test data (seed 1).

    For drift workloads each calibration row is assigned a position drawn
    uniformly over the sequence, so the calibration set covers the drift range.
    """
    n_rows = w.context + 1
    k = _rng(1, 0).standard_normal((CALIB_TOKENS, w.num_kv_heads, w.head_dim))
    pos = _rng(1, 2).integers(0, n_rows, size=CALIB_TOKENS)
    k = _shape_keys(k, w, pos, n_rows)
    v = _rng(1, 1).standard_normal((CALIB_TOKENS, w.num_kv_heads, w.head_dim))
    return k.astype(np.float16), v.astype(np.float16)


def queries(w: Workload) -> np.ndarray:
    """fp16 [B][Hq][D] decode queries, N(0,1) (seed 4)."""
    return _rng(4).standard_normal((w.batch, w.num_q_heads, w.head_dim)).astype(np.float16)


def pages_per_seq(w: Workload) -> np.ndarray:
    """int64 [B]: pages each sequence needs for its N + 1 tokens."""
    return -(-(seq_lens(w) + 1) // w.page_size)


def page_table(w: Workload) -> np.ndarray:
    """int32 [B][max_pages]: logical page -> physical page (seed 7 permutes them).

    Unused entries are -1.  Contiguous workloads get the identity layout
    (sequence b owns a run of pages).
    """
    pps = pages_per_seq(w)
    total = int(pps.sum())
    phys = np.arange(total, dtype=np.int64)
    if w.permuted_pages:
        phys = _rng(7).permutation(total)
    table = np.full((w.batch, int(pps.max())), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        table[b, :pps[b]] = phys[off:off + pps[b]]
        off += int(pps[b])
    return table


def slot_mapping(w: Workload, b: int, start: int, stop: int) -> np.ndarray:
    """int64 [stop-start]: physical slot (page * P + offset) of tokens start:stop of seq b."""
    t = np.arange(start, stop, dtype=np.int64)
    tab = page_table(w)[b].astype(np.int64)
    return tab[t // w.page_size] * w.page_size + t % w.page_size


def num_pages(w: Workload) -> int:
    return int(pages_per_seq(w).sum())


def kmeans_init(n: int, k: int, which: str) -> np.ndarray:
    """int64 [k]: distinct training rows used as the initial centroids (seed 2 / 3)."""
    return _rng(2 if which == "k" else 3).choice(n, k, replace=False).astype(np.int64)


def custom(index: int = -1, name: str = "custom", **kw) -> Workload:
    """A workload with explicit fields (tests build small and edge-case shapes)."""
    base = dict(batch=1, num_q_heads=2, num_kv_heads=1, context=64, k_sub=2, k_bits=8,
                v_sub=4, v_bits=8, page_size=64)
    base.update(kw)
    return Workload(index, name, **base)


def describe() -> List[str]:
    return [f"{w.index}: {w.name}" for w in WORKLOADS.values()]
