"""GPU parity of vq_dequantize_kv against the oracle's dequantisation.

Codes come from the seeded generator or from the oracle's encode, are packed by
the oracle into the pools, and read back by the kernel.  Values are fp16
centroids copied as they are: bit-exact.  Keys go through the fp32 inverse
transform (seven butterfly stages) and one rounding to fp16, so each element is
within 2^-11 |K^| (the rounding, round-to-nearest) + 1e-6 lambda_max ||K~ row||
(fp32 butterflies: at most 7 * 2^-24 of the row norm after the orthonormal
scaling) + 6e-8 (fp16 subnormal spacing) of the oracle's fp64 value.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from vqcase import Calib, GpuCache, calib_for, compare_codes, oracle_encode

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _random_calib(w, seed):
    """Codebooks and lambda with no training: the kernel reads any values."""
    rng = np.random.default_rng(seed)
    lam = rng.uniform(0.3, 4.0, (w.num_kv_heads, w.head_dim)).astype(np.float32)
    ck = (rng.standard_normal((2 ** w.k_bits, w.k_sub)) * 1.5).astype(np.float16)
    cv = rng.standard_normal((2 ** w.v_bits, w.v_sub)).astype(np.float16)
    return Calib(lam, ck, cv)


def _slots(w, lens):
    return np.concatenate([W.slot_mapping(w, b, 0, int(n)) for b, n in enumerate(lens)])


def _check_keys(got, ref, kt, lam):
    """got fp16 / ref fp64 [T][Hkv][D]; kt the oracle's K~ rows (for the bound)."""
    got = got.astype(np.float64)
    row_norm = np.sqrt((kt ** 2).sum(-1, keepdims=True))
    tol = 2.0 ** -11 * np.abs(ref) + 1e-6 * lam.max(-1)[None, :, None] * row_norm + 6e-8
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} key elements out of bound, worst excess "
                           f"{float((err - tol).max()):.3e} at {np.argwhere(bad)[0].tolist()}")


def _dequant(gc, slots, keys=True, values=True):
    s = torch.from_numpy(slots.astype(np.int64)).to(gc.device)
    k, v = gc.vq.dequantize_kv(gc.layout, s, gc.lam, gc.ck, gc.cv, gc.k_pool, gc.v_pool,
                               keys=keys, values=values, status=gc.status)
    torch.cuda.synchronize()
    return (None if k is None else k.cpu().numpy()), (None if v is None else v.cpu().numpy())


FORMATS = [(4, 8, 4, 8), (2, 8, 4, 9), (2, 8, 2, 8), (1, 4, 8, 12), (8, 12, 1, 3), (4, 5, 2, 7)]


@pytest.mark.parametrize("fmt", FORMATS, ids=lambda f: "k%d.%d-v%d.%d" % f)
def test_dequantize_random_codes(fmt):
    dk, bk, dv, bv = fmt
    w = W.custom(name="dq", batch=3, num_q_heads=6, num_kv_heads=3, context=300, k_sub=dk,
                 k_bits=bk, v_sub=dv, v_bits=bv, page_size=16, ragged=True, ragged_lo=1,
                 ragged_hi=300, permuted_pages=True)
    cal = _random_calib(w, 60 + dk + bv)
    gc = GpuCache(w, cal)
    rng = np.random.default_rng(61 + bk)
    kcs, vcs = [], []
    for b, n in enumerate(gc.lens):
        kc = rng.integers(0, 2 ** bk, (int(n), w.num_kv_heads, 128 // dk)).astype(np.int32)
        vc = rng.integers(0, 2 ** bv, (int(n), w.num_kv_heads, 128 // dv)).astype(np.int32)
        gc.write_codes(b, 0, kc, vc)
        kcs.append(kc)
        vcs.append(vc)
    kc, vc = np.concatenate(kcs), np.concatenate(vcs)
    k, v = _dequant(gc, _slots(w, gc.lens))
    assert gc.device_status() == 0
    ref_k, ref_v = oracle.dequantize_kv(kc, cal.ck, vc, cal.cv, cal.lam.astype(np.float64))
    assert np.array_equal(v.astype(np.float64), ref_v)
    _check_keys(k, ref_k, oracle.dequantize(kc, cal.ck), cal.lam)


def test_dequantize_one_half_only():
    w = W.custom(name="dq1", batch=1, num_q_heads=4, num_kv_heads=2, context=100, k_sub=4,
                 v_sub=4, page_size=16, ragged=False, permuted_pages=True)
    cal = _random_calib(w, 70)
    gc = GpuCache(w, cal)
    rng = np.random.default_rng(71)
    n = int(gc.lens[0])
    kc = rng.integers(0, 256, (n, 2, 32)).astype(np.int32)
    vc = rng.integers(0, 256, (n, 2, 32)).astype(np.int32)
    gc.write_codes(0, 0, kc, vc)
    slots = _slots(w, gc.lens)
    k_only, none_v = _dequant(gc, slots, values=False)
    none_k, v_only = _dequant(gc, slots, keys=False)
    assert none_v is None and none_k is None
    ref_k, ref_v = oracle.dequantize_kv(kc, cal.ck, vc, cal.cv, cal.lam.astype(np.float64))
    assert np.array_equal(v_only.astype(np.float64), ref_v)
    _check_keys(k_only, ref_k, oracle.dequantize(kc, cal.ck), cal.lam)


def test_dequantize_padding_and_bad_slots():
    w = W.custom(name="dq2", batch=1, num_q_heads=4, num_kv_heads=2, context=64, k_sub=4,
                 v_sub=4, page_size=16, ragged=False, permuted_pages=False)
    cal = _random_calib(w, 72)
    gc = GpuCache(w, cal)
    rng = np.random.default_rng(73)
    kc = rng.integers(0, 256, (64, 2, 32)).astype(np.int32)
    vc = rng.integers(0, 256, (64, 2, 32)).astype(np.int32)
    gc.write_codes(0, 0, kc, vc)
    good = W.slot_mapping(w, 0, 5, 8)
    slots = np.array([good[0], -1, good[1], -7, good[2]], np.int64)
    k, v = _dequant(gc, slots)
    assert gc.device_status() == 0
    assert not k[[1, 3]].any() and not v[[1, 3]].any()        # padding: zero rows
    ref_k, ref_v = oracle.dequantize_kv(kc[5:8], cal.ck, vc[5:8], cal.cv, cal.lam.astype(np.float64))
    assert np.array_equal(v[[0, 2, 4]].astype(np.float64), ref_v)
    _check_keys(k[[0, 2, 4]], ref_k, oracle.dequantize(kc[5:8], cal.ck), cal.lam)

    over = np.array([good[0], gc.num_pages * w.page_size + 3], np.int64)
    k, v = _dequant(gc, over)
    assert gc.device_status() == 2                           # VQ_DEV_BAD_SLOT
    assert not k[1].any() and not v[1].any()


def test_dequantize_no_tokens_is_a_no_op():
    w = W.custom(name="dq3", batch=1, num_q_heads=4, num_kv_heads=2, context=16, k_sub=4,
                 v_sub=4, page_size=16, ragged=False)
    gc = GpuCache(w, _random_calib(w, 74))
    k, v = _dequant(gc, np.zeros(0, np.int64))
    assert k.shape == (0, 2, 128) and v.shape == (0, 2, 128)
    assert gc.device_status() == 0


def test_dequantize_full_size_32k_sampled():
    """The 32K Llama layer (every token-head of the cache in one launch), filled
    by the GPU encode; sampled tokens against the oracle's encode + dequantise."""
    w = W.WORKLOADS[1]
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    gc.prefill()
    n = int(gc.lens[0])
    k, v = _dequant(gc, _slots(w, gc.lens))
    assert gc.device_status() == 0
    rng = np.random.default_rng(75)
    for start in sorted(rng.choice(n - 64, 6, replace=False).tolist()) + [n - 64]:
        r = oracle_encode(w, cal, 0, start, start + 64)
        kc, vc = gc.codes(0, start, start + 64)
        log = []
        compare_codes(kc, r.kc, r.kx, cal.ck, w.k_sub, "k", log)
        compare_codes(vc, r.vc, r.vx, cal.cv, w.v_sub, "v", log)
        same = (kc == r.kc).all(-1) & (vc == r.vc).all(-1)       # [64][Hkv] rows without ties
        ref_k, ref_v = oracle.dequantize_kv(r.kc, cal.ck, r.vc, cal.cv, cal.lam.astype(np.float64))
        got_k, got_v = k[start:start + 64], v[start:start + 64]
        assert np.array_equal(got_v[same].astype(np.float64), ref_v[same])
        kt = oracle.dequantize(r.kc, cal.ck)
        _check_keys(np.where(same[..., None], got_k, 0), np.where(same[..., None], ref_k, 0),
                    kt, cal.lam)
