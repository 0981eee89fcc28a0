"""vq_decode_attention_static: decode attention for callers that cannot allocate.

Some callers of this library cannot give it a workspace: code running where a
device allocation is not allowed or would synchronise the device, embedders
whose memory belongs to an allocator they cannot call, plug-ins handed only the
tensors of one call.  vq_decode_attention_static keeps the split partials in a
fixed device array inside the library instead.  These tests call it through
the C ABI and check it against vq_decode_attention with a caller workspace
(bit for bit: the same kernels run with the same split count) and against the
oracle, on two calls in a row with different queries (the array keeps the
previous call's contents, which must not leak into the next result).  The file is named so
that pytest collects it last.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import GpuCache, calib_for, check_outputs, oracle_attention, oracle_encode

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _static(vq, gc, q, lens, num_splits=0):
    out = torch.empty((q.shape[0], gc.w.num_q_heads, 128), dtype=torch.float16, device="cuda")
    seq = torch.from_numpy(lens.astype(np.int32)).cuda()
    qd = torch.from_numpy(q).cuda()
    vq.vq_decode_attention_static(gc.layout, q.shape[0], qd.data_ptr(), gc.lam.data_ptr(),
                                  gc.ck.data_ptr(), gc.cv.data_ptr(), gc.k_pool.data_ptr(),
                                  gc.v_pool.data_ptr(), gc.num_pages, gc.page_table.data_ptr(),
                                  gc.page_table.shape[1], seq.data_ptr(), int(lens.max()), 0.0,
                                  num_splits, out.data_ptr(), gc.status.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_static_scratch_matches_workspace_path_twice():
    """Same kernels, same split count: the result must be bit-identical to the
    workspace path, on two calls in a row with different queries (a stale
    partial or a wrong offset in the array would show), and within the stated
    tolerance of the oracle."""
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="static", batch=3, num_q_heads=8, num_kv_heads=2, context=900, k_sub=2,
                 v_sub=4, page_size=64, ragged=True, ragged_lo=300, ragged_hi=900,
                 permuted_pages=True)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    lens = gc.lens + 1
    refs = [oracle_encode(w, cal, b, 0, int(lens[b])) for b in range(w.batch)]
    for b in range(w.batch):                      # the oracle's codes in the pools
        gc.write_codes(b, 0, refs[b].kc, refs[b].vc)
    rng = np.random.default_rng(99)
    for call in range(2):
        q = W.queries(w) if call == 0 else rng.standard_normal((w.batch, w.num_q_heads, 128)).astype(np.float16)
        ref = gc.decode(q, lens=lens)                 # caller workspace path
        got = _static(vq, gc, q, lens)                # static scratch path
        assert np.array_equal(got, ref), (call, float(np.abs(got - ref).max()))
        orc = np.stack([oracle_attention(w, cal, q[b], refs[b].kc, refs[b].vc) for b in range(w.batch)])
        check_outputs(got, orc, f"static scratch call {call} vs oracle")
    assert gc.device_status() == 0


def test_static_scratch_lowers_the_default_split_count_to_fit():
    """With num_splits <= 0 the library's split choice is lowered until the
    partials fit the array.  Batch 64 x 64 query heads over 8 KV heads at 4K
    context takes 2 splits (length-balanced units) on a 152-SM GB300, just
    over 4 MiB of partials; the call runs at 1 split, bit-identical to the
    workspace path at that count.  Seeded random codes stand in for a filled
    cache (the result is only compared between the two paths)."""
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="static-big", batch=64, num_q_heads=64, num_kv_heads=8, context=4096,
                 k_sub=4, v_sub=4, page_size=256)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    rng = np.random.default_rng(7)
    gc.k_pool.copy_(torch.from_numpy(rng.integers(0, 256, gc.k_pool.shape, dtype=np.uint8)))
    gc.v_pool.copy_(torch.from_numpy(rng.integers(0, 256, gc.v_pool.shape, dtype=np.uint8)))
    lens = gc.lens + 1
    ml = int(lens.max())
    cap = vq.vq_static_scratch_bytes()
    auto = vq.vq_default_num_splits(gc.layout, w.batch, ml)
    fit = max(s for s in range(1, auto + 1)
              if vq.vq_decode_workspace_bytes(gc.layout, w.batch, ml, s) <= cap)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert vq.vq_decode_workspace_bytes(gc.layout, w.batch, ml, auto) > cap and fit < auto
    q = W.queries(w)
    got = _static(vq, gc, q, lens)
    ref = gc.decode(q, lens=lens, num_splits=fit)
    assert np.array_equal(got, ref)
    assert gc.device_status() == 0


def test_static_scratch_rejects_oversized_requests():
    import bit_vector_quantized_gb300 as vq
    L = vq.make_layout(num_q_heads=40, num_kv_heads=8, k_sub=2, v_bits=9)
    need = vq.vq_decode_workspace_bytes(L, 64, 16385, 8)
    assert need > vq.vq_static_scratch_bytes()
    out = torch.empty((64, 40, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(vq.VQError) as e:
        vq.vq_decode_attention_static(L, 64, 16, 16, 16, 16, 16, 16, 1, 16, 1, 16, 16385, 0.0, 8,
                                      out.data_ptr())
    assert e.value.status == vq.VQ_ERR_WORKSPACE and "static scratch" in str(e.value)
