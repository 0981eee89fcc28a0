"""GPU encode (vq_encode_kv) vs the oracle: codes bit-exact except logged ties."""
import numpy as np
import pytest

import workloads as W
from vqcase import GpuCache, calib_for, compare_codes, oracle_encode, write_tie_log

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _check_seq(gc, w, cal, b, start, stop, name, log):
    got_k, got_v = gc.codes(b, start, stop)
    ref = oracle_encode(w, cal, b, start, stop)
    n = compare_codes(got_k, ref.kc, ref.kx, cal.ck, w.k_sub, f"{name}/k/b{b}", log)
    n += compare_codes(got_v, ref.vc, ref.vx, cal.cv, w.v_sub, f"{name}/v/b{b}", log)
    return n


FORMATS = [  # (k_sub, k_bits, v_sub, v_bits)
    (2, 8, 4, 8), (4, 8, 4, 8), (2, 8, 4, 9), (4, 8, 2, 8),
    (1, 4, 8, 10), (8, 12, 1, 3), (4, 9, 2, 1), (2, 6, 4, 5), (8, 12, 8, 12),
]


@pytest.mark.parametrize("fmt", FORMATS, ids=lambda f: "k%d.%d-v%d.%d" % f)
def test_encode_formats_small(fmt):
    dk, bk, dv, bv = fmt
    w = W.custom(name="enc-" + "-".join(map(str, fmt)), batch=2, num_q_heads=6, num_kv_heads=3,
                 context=181, k_sub=dk, k_bits=bk, v_sub=dv, v_bits=bv, page_size=32)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    assert gc.device_status() == 0
    log = []
    for b in range(w.batch):
        _check_seq(gc, w, cal, b, 0, int(gc.lens[b]) + 1, w.name, log)
    write_tie_log(w.name, log)


def test_encode_tiny_workload_full():
    w = W.WORKLOADS[0]
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    assert gc.device_status() == 0
    log = []
    _check_seq(gc, w, cal, 0, 0, w.context + 1, "cfg0", log)
    write_tie_log("cfg0_encode", log)


def test_encode_paged_permuted_slots():
    w = W.custom(name="enc-paged", batch=3, num_q_heads=4, num_kv_heads=2, context=150,
                 page_size=16, permuted_pages=True, ragged=True, ragged_lo=40, ragged_hi=150)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    log = []
    for b in range(w.batch):
        _check_seq(gc, w, cal, b, 0, int(gc.lens[b]) + 1, w.name, log)
    # rows of pages no sequence owns stay zero
    used = set(gc.page_table_np[gc.page_table_np >= 0].tolist())
    assert len(used) == gc.num_pages


def test_append_path_equals_prefill_path():
    """The few-token path (codebook scan split over 8 warps) gives the same codes."""
    w = W.custom(name="enc-append", batch=4, num_q_heads=8, num_kv_heads=4, context=8,
                 k_sub=4, v_sub=4, v_bits=9, page_size=16)
    cal = calib_for(w)
    a = GpuCache(w, cal)
    for t in range(w.context + 1):          # one token per call: the split path
        for b in range(w.batch):
            a.encode(b, t, t + 1)
    bcache = GpuCache(w, cal)
    for b in range(w.batch):                 # whole sequences
        bcache.encode(b, 0, w.context + 1)
    torch.cuda.synchronize()
    assert torch.equal(a.k_pool, bcache.k_pool) and torch.equal(a.v_pool, bcache.v_pool)
    log = []
    for b in range(w.batch):
        _check_seq(a, w, cal, b, 0, w.context + 1, w.name, log)


def test_negative_slot_skips_and_bad_slot_reports():
    w = W.custom(name="enc-slots", context=31, page_size=16)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    import bit_vector_quantized_gb300 as vq
    k = torch.from_numpy(W.kv_tokens(w, 0, "k", 0, 3)).cuda()
    v = torch.from_numpy(W.kv_tokens(w, 0, "v", 0, 3)).cuda()
    slots = torch.tensor([-1, 5, gc.num_pages * w.page_size + 3], dtype=torch.int64, device="cuda")
    vq.encode_kv(gc.layout, k, v, slots, gc.lam, gc.ck, gc.cv, gc.k_pool, gc.v_pool, status=gc.status)
    assert gc.device_status() == vq.VQ_DEV_BAD_SLOT
    kp = gc.k_pool.cpu().numpy()
    written = np.argwhere(kp.reshape(-1, gc.krow).any(axis=1)).ravel()
    assert written.tolist() == [5]          # only slot 5 (page 0, head 0, offset 5)
