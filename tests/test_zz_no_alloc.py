"""vq_decode_attention_static: decode attention for callers that cannot allocate.

Some callers of this library cannot give it a workspace: code running where a
device allocation is not allowed or would synchronise the device, embedders
whose memory belongs to an allocator they cannot call, plug-ins handed only the
tensors of one call.  vq_decode_attention_static keeps the split partials in a
fixed device array inside the library instead.  These tests call it through
the C ABI and check it against vq_decode_attention with a caller workspace, on
two calls in a row with different queries (the array keeps the previous call's
contents, which must not leak into the next result).  The file is named so
that pytest collects it last.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import MAX_ABS, MEAN_ABS, GpuCache, calib_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _static(vq, gc, q, lens):
    out = torch.empty((q.shape[0], gc.w.num_q_heads, 128), dtype=torch.float16, device="cuda")
    seq = torch.from_numpy(lens.astype(np.int32)).cuda()
    qd = torch.from_numpy(q).cuda()
    vq.vq_decode_attention_static(gc.layout, q.shape[0], qd.data_ptr(), gc.lam.data_ptr(),
                                  gc.ck.data_ptr(), gc.cv.data_ptr(), gc.k_pool.data_ptr(),
                                  gc.v_pool.data_ptr(), gc.num_pages, gc.page_table.data_ptr(),
                                  gc.page_table.shape[1], seq.data_ptr(), int(lens.max()), 0.0, 0,
                                  out.data_ptr(), gc.status.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_static_scratch_matches_workspace_path_twice():
    import bit_vector_quantized_gb300 as vq
    w = W.custom(name="static", batch=3, num_q_heads=8, num_kv_heads=2, context=900, k_sub=2,
                 v_sub=4, page_size=64, ragged=True, ragged_lo=300, ragged_hi=900,
                 permuted_pages=True)
    gc = GpuCache(w, calib_for(w))
    gc.prefill()
    gc.append()
    lens = gc.lens + 1
    rng = np.random.default_rng(99)
    for call in range(2):
        q = W.queries(w) if call == 0 else rng.standard_normal((w.batch, w.num_q_heads, 128)).astype(np.float16)
        ref = gc.decode(q, lens=lens)                 # caller workspace path
        got = _static(vq, gc, q, lens)                # static scratch path
        err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (call, err.max(), err.mean())
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
