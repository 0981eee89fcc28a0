"""GPU decode attention (vq_decode_attention) vs the oracle.

The decode kernel is fed the oracle's own packed codes (written into the GPU
pools), so the comparison isolates the attention arithmetic; the end-to-end
test runs GPU encode then GPU decode.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import (GpuCache, calib_for, check_outputs, compare_codes, oracle_attention,
                    oracle_encode, skip_end_to_end, write_tie_log)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _oracle_filled(w, heads=None):
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    refs = []
    for b in range(w.batch):
        n = int(gc.lens[b]) + 1
        r = oracle_encode(w, cal, b, 0, n)
        gc.write_codes(b, 0, r.kc, r.vc)
        refs.append(r)
    return cal, gc, refs


def _oracle_out(w, cal, refs, q, lens=None):
    outs = []
    for b in range(w.batch):
        n = refs[b].kc.shape[0] if lens is None else int(lens[b])
        outs.append(oracle_attention(w, cal, q[b], refs[b].kc[:n], refs[b].vc[:n]))
    return np.stack(outs)


# (k_sub, k_bits, v_sub, v_bits): the 2-bit and mixed formats, and the pages'
# 1.5-bit configuration (4096 centroids of 8 elements, 12-bit codes)
DECODE_FORMATS = [(2, 8, 4, 8), (4, 8, 4, 8), (2, 8, 4, 9), (4, 8, 4, 9), (2, 8, 2, 8), (4, 8, 2, 8),
                  (8, 12, 8, 12)]


@pytest.mark.parametrize("group", [1, 2, 4, 5, 8])
@pytest.mark.parametrize("fmt", DECODE_FORMATS, ids=lambda f: "k%d.%d-v%d.%d" % f)
def test_decode_formats_and_groups(fmt, group):
    dk, bk, dv, bv = fmt
    w = W.custom(name="dec", batch=2, num_q_heads=2 * group, num_kv_heads=2, context=700,
                 k_sub=dk, k_bits=bk, v_sub=dv, v_bits=bv, page_size=64, ragged=True,
                 ragged_lo=300, ragged_hi=700)
    cal, gc, refs = _oracle_filled(w)
    q = W.queries(w)
    got = gc.decode(q)
    assert gc.device_status() == 0
    check_outputs(got, _oracle_out(w, cal, refs, q), f"{fmt} G={group}")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_split_invariance(splits):
    w = W.custom(name="split", batch=2, num_q_heads=8, num_kv_heads=2, context=2000,
                 k_sub=4, v_sub=4, page_size=128)
    cal, gc, refs = _oracle_filled(w)
    q = W.queries(w)
    ref = _oracle_out(w, cal, refs, q)
    got = gc.decode(q, num_splits=splits)
    check_outputs(got, ref, f"splits={splits}")
    base = gc.decode(q, num_splits=1)
    assert np.max(np.abs(got - base)) < 1e-3


@pytest.mark.parametrize("n", [1, 2, 15, 16, 17, 31, 33, 129])
def test_short_and_tile_boundary_lengths(n):
    w = W.custom(name="short", batch=1, num_q_heads=4, num_kv_heads=1, context=n - 1,
                 k_sub=2, v_sub=4, page_size=16)
    cal, gc, refs = _oracle_filled(w)
    q = W.queries(w)
    check_outputs(gc.decode(q), _oracle_out(w, cal, refs, q), f"n={n}")
    check_outputs(gc.decode(q, num_splits=4), _oracle_out(w, cal, refs, q), f"n={n} s=4")


def test_zero_length_gives_zero_and_lens_clamped():
    w = W.custom(name="zero", batch=3, num_q_heads=4, num_kv_heads=2, context=90, page_size=32)
    cal, gc, refs = _oracle_filled(w)
    q = W.queries(w)
    lens = np.array([0, 50, 91])
    got = gc.decode(q, lens=lens)
    assert not got[0].any()
    check_outputs(got[1:], _oracle_out(w, cal, refs, q, lens)[1:], "lens")


def test_softmax_scale_override():
    w = W.custom(name="scale", batch=1, num_q_heads=4, num_kv_heads=2, context=300, page_size=64)
    cal, gc, refs = _oracle_filled(w)
    q = W.queries(w)
    got = gc.decode(q, softmax_scale=0.02)
    import oracle
    ref = np.stack([oracle.decode_attention(q[0], cal.lam.astype(np.float64), refs[0].kc, cal.ck,
                                            refs[0].vc, cal.cv, scale=0.02)])
    check_outputs(got, ref, "scale")


def test_bad_page_reports_status():
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="badpage", batch=1, num_q_heads=2, num_kv_heads=1, context=100, page_size=32)
    cal, gc, refs = _oracle_filled(w)
    gc.page_table[0, 1] = gc.num_pages + 5
    got = gc.decode(W.queries(w))
    assert gc.device_status() == vq.VQ_DEV_BAD_PAGE
    assert np.all(np.isfinite(got))


def test_end_to_end_tiny_workload():
    w = W.WORKLOADS[0]
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    q = W.queries(w)
    got = gc.decode(q)
    ref_seq = oracle_encode(w, cal, 0, 0, w.context + 1)
    log = []
    kc, vc = gc.codes(0, 0, w.context + 1)
    ties = compare_codes(kc, ref_seq.kc, ref_seq.kx, cal.ck, w.k_sub, "cfg0/k", log)
    ties += compare_codes(vc, ref_seq.vc, ref_seq.vx, cal.cv, w.v_sub, "cfg0/v", log)
    write_tie_log("cfg0_e2e", log)
    ref = oracle_attention(w, cal, q[0], ref_seq.kc, ref_seq.vc)[None]
    if ties == 0:
        check_outputs(got, ref, "cfg0 end-to-end")
    else:
        skip_end_to_end("cfg0", ties)
    # the kernel on the oracle's codes, same launch
    gc.write_codes(0, 0, ref_seq.kc, ref_seq.vc)
    check_outputs(gc.decode(q), ref, "cfg0 oracle codes")


def test_ragged_paged_workload_reduced():
    """Workload 2's layout (64-token permuted pages, ragged lengths) at 1/8 length."""
    w = W.custom(name="cfg2-reduced", batch=16, num_q_heads=32, num_kv_heads=8, context=1024,
                 k_sub=2, v_sub=4, page_size=64, ragged=True, ragged_lo=512, ragged_hi=1024,
                 permuted_pages=True)
    cal, gc, refs = _oracle_filled(w)
    q = W.queries(w)
    check_outputs(gc.decode(q), _oracle_out(w, cal, refs, q), "cfg2-reduced")
