"""GPU parity of the pages' alternative score and P.V methods (vq_decode_partial_method).

VQ_METHOD_LUT takes the scores from a per-query lookup table of q~ x K-codebook
products summed over the K codes (VecInfer, 内核实现细节 - 融合内核, Algorithm
1); VQ_METHOD_BINS computes P.V by accumulating p into per-code bins and
multiplying by the V codebook once per work unit (CommVQ, 降低计算复杂度,
Softmax(A) S_V C_V).  Both must agree with the fp64 oracle within the stated
tolerance (max-abs 2e-3, mean-abs 2e-4) on the oracle's own codes, and with
the gather method the library uses everywhere else.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import (GpuCache, calib_for, check_outputs, oracle_attention, oracle_encode,
                    stored_calib)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

METHODS = {"lut": 1, "bins": 2}


def _filled(w, cal=None):
    """A cache holding the oracle's codes of every token, and the oracle's results."""
    cal = cal or calib_for(w)
    gc = GpuCache(w, cal)
    lens = gc.lens + 1
    refs = []
    for b in range(w.batch):
        r = oracle_encode(w, cal, b, 0, int(lens[b]))
        gc.write_codes(b, 0, r.kc, r.vc)
        refs.append(r)
    return cal, gc, refs, lens


def _run(vq, gc, q, lens, method, splits=0):
    seq = torch.from_numpy(lens.astype(np.int32)).cuda()
    out = vq.decode_attention_method(gc.layout, torch.from_numpy(q).cuda(), gc.lam, gc.ck, gc.cv,
                                     gc.k_pool, gc.v_pool, gc.page_table, seq, int(lens.max()),
                                     method, num_splits=splits, status=gc.status)
    torch.cuda.synchronize()
    assert gc.device_status() == 0
    return out.float().cpu().numpy()


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("group", [1, 2, 4])
@pytest.mark.parametrize("method", sorted(METHODS))
def test_method_against_oracle(method, group, splits):
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="method", batch=3, num_q_heads=2 * group, num_kv_heads=2, context=900,
                 k_sub=4, v_sub=4, page_size=64, ragged=True, ragged_lo=300, ragged_hi=900,
                 permuted_pages=True)
    cal, gc, refs, lens = _filled(w)
    q = W.queries(w)
    got = _run(vq, gc, q, lens, METHODS[method], splits)
    ref = np.stack([oracle_attention(w, cal, q[b], refs[b].kc, refs[b].vc) for b in range(w.batch)])
    check_outputs(got, ref, f"{method} G={group} splits={splits}")
    gather = gc.decode(q, lens=lens, num_splits=splits)
    check_outputs(got, gather.astype(np.float64), f"{method} vs gather")


@pytest.mark.parametrize("method", sorted(METHODS))
def test_method_edge_lengths(method):
    # lengths 1, 15, 16, 17, 33 and 0 (a zero row), one split and several
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="method-edge", batch=6, num_q_heads=8, num_kv_heads=2, context=64,
                 k_sub=4, v_sub=4, page_size=16, permuted_pages=True)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    lens = np.array([1, 15, 16, 17, 33, 0])
    refs = []
    for b in range(w.batch):
        r = oracle_encode(w, cal, b, 0, max(int(lens[b]), 1))
        if lens[b] > 0:
            gc.write_codes(b, 0, r.kc, r.vc)
        refs.append(r)
    q = W.queries(w)
    for splits in (1, 2):
        got = _run(vq, gc, q, lens, METHODS[method], splits)
        for b in range(w.batch):
            if lens[b] == 0:
                assert not got[b].any()
            else:
                ref = oracle_attention(w, cal, q[b], refs[b].kc, refs[b].vc)
                check_outputs(got[b], ref, f"{method} len {lens[b]} splits {splits}")


@pytest.mark.parametrize("method", sorted(METHODS))
def test_method_full_size_llama_32k(method):
    """The 32K workload at full size, the launch bench.py times for the method
    comparison: one sampled KV head on the oracle's codes against the oracle,
    and every head against the gather method."""
    import bit_vector_quantized_gb300 as vq
    w = W.WORKLOADS[1]
    cal = stored_calib(1)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    lens = gc.lens + 1
    h = 5
    G = w.num_q_heads // w.num_kv_heads
    r = oracle_encode(w, cal, 0, 0, int(lens[0]), heads=[h])
    gc.write_codes(0, 0, r.kc, r.vc, heads=[h])
    q = W.queries(w)
    got = _run(vq, gc, q, lens, METHODS[method])
    ref = oracle_attention(w, cal, q[0, h * G:(h + 1) * G], r.kc, r.vc, heads=[h])
    check_outputs(got[0, h * G:(h + 1) * G], ref, f"{method} cfg1 kv-head {h}")
    check_outputs(got, gc.decode(q, lens=lens).astype(np.float64), f"{method} cfg1 vs gather")


def test_method_rejects_other_layouts():
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="method-k2", batch=1, num_q_heads=4, num_kv_heads=1, context=64, k_sub=2,
                 v_sub=4, page_size=64)
    gc = GpuCache(w, calib_for(w))
    q = W.queries(w)
    with pytest.raises(vq.VQError) as e:
        _run(vq, gc, q, gc.lens + 1, METHODS["lut"])
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED
