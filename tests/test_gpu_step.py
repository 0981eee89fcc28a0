"""GPU parity of vq_decode_step (append + decode attention in one call).

The call appends each sequence's new token (its codes go to the row of position
seq_lens - 1 through the page table) and attends over the cache.  It must write
exactly the rows vq_encode_kv writes, return exactly what vq_encode_kv +
vq_decode_attention return with the same split count, and agree with the oracle
within the stated tolerance.
"""
import numpy as np
import pytest

import workloads as W
from test_gpu_decode import DECODE_FORMATS
from vqcase import GpuCache, calib_for, check_outputs, oracle_attention, oracle_encode

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _workload(fmt, group, batch=3, context=700):
    dk, bk, dv, bv = fmt
    return W.custom(name="step", batch=batch, num_q_heads=2 * group, num_kv_heads=2,
                    context=context, k_sub=dk, k_bits=bk, v_sub=dv, v_bits=bv, page_size=64,
                    ragged=True, ragged_lo=300, ragged_hi=context, permuted_pages=True)


def _pair(w):
    cal = calib_for(w)
    a, b = GpuCache(w, cal), GpuCache(w, cal)
    a.prefill()
    b.prefill()
    return cal, a, b


@pytest.mark.parametrize("group", [1, 4, 5, 8])
@pytest.mark.parametrize("fmt", DECODE_FORMATS, ids=lambda f: "k%d.%d-v%d.%d" % f)
def test_step_equals_append_then_attention(fmt, group):
    w = _workload(fmt, group)
    _, a, b = _pair(w)
    q = W.queries(w)
    a.append()
    ref = a.decode(q, num_splits=3)
    got = b.step(q, num_splits=3)
    assert a.device_status() == 0 and b.device_status() == 0
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert np.array_equal(got, ref)


def test_step_default_splits_against_oracle_two_steps():
    w = _workload((4, 8, 4, 8), 4, batch=4, context=900)
    cal = calib_for(w)
    a = GpuCache(w, cal)
    for bb in range(w.batch):                             # cache tokens [0, N - 1)
        a.encode(bb, 0, int(a.lens[bb]) - 1)
    rng = np.random.default_rng(11)
    for extra in (0, 1):                                  # append token N - 1, then token N
        lens = a.lens + extra
        q = rng.standard_normal((w.batch, w.num_q_heads, 128)).astype(np.float16)
        got = a.step(q, lens=lens)
        assert a.device_status() == 0
        for bb in range(w.batch):
            n = int(lens[bb])
            r = oracle_encode(w, cal, bb, 0, n)
            kc, vc = a.codes(bb, n - 1, n)
            assert np.array_equal(kc, r.kc[-1:]) and np.array_equal(vc, r.vc[-1:])
            ref = oracle_attention(w, cal, q[bb], r.kc, r.vc)
            check_outputs(got[bb], ref, f"step {extra} seq {bb}")


@pytest.mark.parametrize("splits", [1, 2, 17])
def test_step_split_counts(splits):
    w = _workload((2, 8, 4, 9), 5)
    _, a, b = _pair(w)
    q = W.queries(w)
    a.append()
    ref = a.decode(q, num_splits=splits)
    got = b.step(q, num_splits=splits)
    assert b.device_status() == 0
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert np.array_equal(got, ref)


def test_step_edge_lengths():
    # attended lengths 0 (nothing appended, zero row), 1 (only the new token), 16, 17, 33
    w = W.custom(name="edge", batch=5, num_q_heads=8, num_kv_heads=2, context=64, k_sub=4,
                 v_sub=4, page_size=16, ragged=False, permuted_pages=True)
    cal = calib_for(w)
    lens = np.array([0, 1, 16, 17, 33])
    a, b = GpuCache(w, cal), GpuCache(w, cal)
    for gc in (a, b):
        for bb in range(w.batch):
            if lens[bb] > 1:
                gc.encode(bb, 0, int(lens[bb]) - 1)
    for bb in range(w.batch):
        if lens[bb] > 0:
            a.encode(bb, int(lens[bb]) - 1, int(lens[bb]))
    q = W.queries(w)
    ref = a.decode(q, lens=lens, num_splits=2)
    got = b.step(q, lens=lens, num_splits=2)
    assert b.device_status() == 0
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert np.array_equal(got, ref)
    assert not got[0].any()


def test_step_bad_page_of_the_new_token_is_reported():
    w = _workload((4, 8, 4, 8), 2, batch=2, context=300)
    _, a, _ = _pair(w)
    n = int(a.lens[1])
    a.page_table[1, n // w.page_size] = a.num_pages + 5     # the new token's page is out of range
    a.step(W.queries(w))
    assert a.device_status() == 1                            # VQ_DEV_BAD_PAGE


def test_step_large_batch():
    # 400 sequences x 2 KV heads: the append is encoded several vectors per warp
    w = W.custom(name="wide", batch=400, num_q_heads=8, num_kv_heads=2, context=40, k_sub=2,
                 k_bits=8, v_sub=4, v_bits=9, page_size=16, ragged=True, ragged_lo=1,
                 ragged_hi=40, permuted_pages=True)
    _, a, b = _pair(w)
    q = W.queries(w)
    a.append()
    ref = a.decode(q)
    got = b.step(q)
    assert a.device_status() == 0 and b.device_status() == 0
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert np.array_equal(got, ref)


def test_step_length_beyond_max_seq_len():
    """A sequence longer than max_seq_len: its new token is stored where
    vq_encode_kv stores it, but, like every token at or past max_seq_len, it is
    not attended."""
    import bit_vector_quantized_gb300 as vq
    w = _workload((4, 8, 4, 8), 4, batch=3, context=700)
    _, a, b = _pair(w)
    lens = a.lens + 1
    ml = int(lens.min())                                     # shorter than the other sequences
    assert (lens > ml).any()
    q = W.queries(w)
    a.append()                                               # every sequence's token lens - 1
    seq = torch.from_numpy(lens.astype(np.int32)).cuda()
    qd = torch.from_numpy(q).cuda()
    ref = vq.decode_attention(a.layout, qd, a.lam, a.ck, a.cv, a.k_pool, a.v_pool, a.page_table, seq,
                              ml, num_splits=3, status=a.status)
    pos = [int(n) - 1 for n in lens]
    kn = torch.from_numpy(np.stack([W.kv_tokens(w, bb, "k", p, p + 1)[0] for bb, p in enumerate(pos)])).cuda()
    vn = torch.from_numpy(np.stack([W.kv_tokens(w, bb, "v", p, p + 1)[0] for bb, p in enumerate(pos)])).cuda()
    got = vq.decode_step(b.layout, qd, kn, vn, b.lam, b.ck, b.cv, b.k_pool, b.v_pool, b.page_table, seq,
                         ml, num_splits=3, status=b.status)
    torch.cuda.synchronize()
    assert a.device_status() == 0 and b.device_status() == 0
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert torch.equal(got, ref)


def test_step_replayed_from_a_cuda_graph():
    # replays of one captured call, over a workspace holding stale bytes, must
    # all give the separate calls' output (the append inside the attention
    # kernel, then the merge of the splits)
    w = _workload((4, 8, 4, 8), 4, batch=3, context=700)
    _, a, b = _pair(w)
    q = W.queries(w)
    a.append()
    ref = a.decode(q, num_splits=5)
    vq, dev = b.vq, b.device
    lens = b.lens + 1
    pos = [int(n) - 1 for n in lens]
    k = np.stack([W.kv_tokens(w, bb, "k", p, p + 1)[0] for bb, p in enumerate(pos)])
    v = np.stack([W.kv_tokens(w, bb, "v", p, p + 1)[0] for bb, p in enumerate(pos)])
    q_d, k_d, v_d = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    seq = torch.from_numpy(lens.astype(np.int32)).to(dev)
    ml = int(lens.max())
    wsb = vq.vq_decode_workspace_bytes(b.layout, w.batch, ml, 5)
    ws = torch.full((wsb,), 0xA5, dtype=torch.uint8, device=dev)  # stale bytes
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float16, device=dev)
    P = lambda t: t.data_ptr()  # noqa: E731

    def call():
        vq.vq_decode_step(b.layout, w.batch, P(q_d), P(k_d), P(v_d), P(b.lam), P(b.ck), P(b.cv),
                          P(b.k_pool), P(b.v_pool), b.num_pages, P(b.page_table),
                          b.page_table.shape[1], P(seq), ml, 0.0, 5, P(out), P(ws), wsb,
                          P(b.status), torch.cuda.current_stream().cuda_stream)

    call()
    torch.cuda.synchronize()
    assert np.array_equal(out.float().cpu().numpy(), ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.float().cpu().numpy(), ref)
    assert b.device_status() == 0
