"""GPU parity of vq_decode_attention_residual (quantized cache + fp16 residual).

Each sequence's N_b + 1 tokens are split into a quantized part (the first
N_b + 1 - R_b tokens, as the oracle's codes written into the pools) and a
full-precision residual (the last R_b tokens, raw fp16).  The GPU result must
match the oracle's one-softmax attention over both parts within max-abs 2e-3 /
mean-abs 2e-4; with every R_b = 0 it must equal vq_decode_attention exactly.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from test_gpu_decode import DECODE_FORMATS
from vqcase import GpuCache, calib_for, check_outputs, oracle_encode, stored_calib

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _workload(fmt, group, batch=3, context=500, hkv=2):
    dk, bk, dv, bv = fmt
    return W.custom(name="res", batch=batch, num_q_heads=hkv * group, num_kv_heads=hkv,
                    context=context, k_sub=dk, k_bits=bk, v_sub=dv, v_bits=bv, page_size=32,
                    ragged=True, ragged_lo=200, ragged_hi=context, permuted_pages=True)


class ResidualCase:
    """Pools holding the oracle's codes of the quantized part; fp16 residual buffers."""

    def __init__(self, w, cal, res_lens, capacity, heads=None):
        self.w, self.cal = w, cal
        self.gc = gc = GpuCache(w, cal)
        B, H, D = w.batch, w.num_kv_heads, w.head_dim
        self.total = gc.lens + 1                      # N_b + 1 tokens per sequence
        self.res_lens = np.asarray(res_lens, np.int32)
        self.nq = (self.total - self.res_lens).astype(np.int32)
        self.heads = heads
        self.codes, self.kr, self.vr = [], [], []
        k_res = np.zeros((B, H, capacity, D), np.float16)
        v_res = np.zeros((B, H, capacity, D), np.float16)
        for b in range(B):
            n, t = int(self.nq[b]), int(self.total[b])
            r = oracle_encode(w, cal, b, 0, n, heads=heads)
            if n > 0:
                gc.write_codes(b, 0, r.kc, r.vc, heads=heads)
            kr = W.kv_tokens(w, b, "k", n, t)
            vr = W.kv_tokens(w, b, "v", n, t)
            k_res[b, :, :t - n] = kr.transpose(1, 0, 2)
            v_res[b, :, :t - n] = vr.transpose(1, 0, 2)
            self.codes.append(r)
            self.kr.append(kr)
            self.vr.append(vr)
        dev = gc.device
        self.k_res = torch.from_numpy(k_res).to(dev)
        self.v_res = torch.from_numpy(v_res).to(dev)

    def run(self, q, num_splits=0):
        gc = self.gc
        dev = gc.device
        out = gc.vq.decode_attention_residual(
            gc.layout, torch.from_numpy(q).to(dev), gc.lam, gc.ck, gc.cv, gc.k_pool, gc.v_pool,
            gc.page_table, torch.from_numpy(self.nq).to(dev), int(self.nq.max()),
            self.k_res, self.v_res, torch.from_numpy(self.res_lens).to(dev),
            num_splits=num_splits, status=gc.status)
        torch.cuda.synchronize()
        return out.float().cpu().numpy()

    def oracle(self, q, b, heads=None):
        """fp64 rows of sequence b (KV heads `heads`, all by default)."""
        w, cal, r = self.w, self.cal, self.codes[b]
        G = w.num_q_heads // w.num_kv_heads
        hs = list(range(w.num_kv_heads)) if heads is None else heads
        rows = np.concatenate([np.arange(h * G, (h + 1) * G) for h in hs])
        return oracle.decode_attention_residual(q[b, rows], cal.lam[hs].astype(np.float64),
                                                r.kc[:, hs] if self.heads is None else r.kc,
                                                cal.ck, r.vc[:, hs] if self.heads is None else r.vc,
                                                cal.cv, self.kr[b][:, hs], self.vr[b][:, hs]), rows


@pytest.mark.parametrize("group", [1, 4, 5, 8])
@pytest.mark.parametrize("fmt", DECODE_FORMATS, ids=lambda f: "k%d.%d-v%d.%d" % f)
def test_residual_against_oracle(fmt, group):
    w = _workload(fmt, group)
    case = ResidualCase(w, calib_for(w), [0, 37, 128], 128)
    q = W.queries(w)
    got = case.run(q, num_splits=3)
    assert case.gc.device_status() == 0
    for b in range(w.batch):
        ref, rows = case.oracle(q, b)
        check_outputs(got[b, rows], ref, f"seq {b} residual {case.res_lens[b]}")


def test_residual_default_splits_and_short_capacity():
    w = _workload((4, 8, 4, 8), 4, batch=4, context=700)
    case = ResidualCase(w, calib_for(w), [1, 16, 17, 5], 17)
    q = W.queries(w)
    got = case.run(q)
    assert case.gc.device_status() == 0
    for b in range(w.batch):
        ref, rows = case.oracle(q, b)
        check_outputs(got[b, rows], ref, f"seq {b}")


def test_residual_window_in_several_chunks():
    # one split: a unit's window slice is the whole window, staged in shared
    # memory 64 tokens at a time (five chunks for 300 tokens, edges 64 / 65)
    w = W.custom(name="res-chunks", batch=3, num_q_heads=8, num_kv_heads=2, context=900, k_sub=4,
                 v_sub=4, page_size=32, ragged=True, ragged_lo=400, ragged_hi=900, permuted_pages=True)
    case = ResidualCase(w, calib_for(w), [300, 65, 64], 300)
    q = W.queries(w)
    got = case.run(q, num_splits=1)
    assert case.gc.device_status() == 0
    for b in range(w.batch):
        ref, rows = case.oracle(q, b)
        check_outputs(got[b, rows], ref, f"seq {b} residual {case.res_lens[b]}")


def test_residual_zero_equals_decode_attention():
    w = _workload((2, 8, 4, 9), 5)
    case = ResidualCase(w, calib_for(w), [0, 0, 0], 64)
    q = W.queries(w)
    got = case.run(q, num_splits=4)
    gc = case.gc
    ref = gc.decode(q, lens=case.nq, num_splits=4)
    assert np.array_equal(got, ref)


def test_residual_only_and_empty_sequences():
    # sequence 0: nothing at all (zero row); 1: only residual; 2: only codes
    w = W.custom(name="res-edge", batch=3, num_q_heads=8, num_kv_heads=2, context=96, k_sub=4,
                 v_sub=4, page_size=16, ragged=False, permuted_pages=True)
    cal = calib_for(w)
    gc = GpuCache(w, cal)
    total = gc.lens + 1
    case = ResidualCase.__new__(ResidualCase)
    case.w, case.cal, case.gc, case.heads = w, cal, gc, None
    case.total = np.array([0, 40, int(total[2])], np.int32)
    case.res_lens = np.array([0, 40, 0], np.int32)
    case.nq = (case.total - case.res_lens).astype(np.int32)
    case.codes, case.kr, case.vr = [], [], []
    k_res = np.zeros((3, 2, 64, 128), np.float16)
    v_res = np.zeros((3, 2, 64, 128), np.float16)
    for b in range(3):
        n, t = int(case.nq[b]), int(case.total[b])
        r = oracle_encode(w, cal, b, 0, n)
        if n > 0:
            gc.write_codes(b, 0, r.kc, r.vc)
        kr, vr = W.kv_tokens(w, b, "k", n, t), W.kv_tokens(w, b, "v", n, t)
        k_res[b, :, :t - n] = kr.transpose(1, 0, 2)
        v_res[b, :, :t - n] = vr.transpose(1, 0, 2)
        case.codes.append(r)
        case.kr.append(kr)
        case.vr.append(vr)
    case.k_res = torch.from_numpy(k_res).to(gc.device)
    case.v_res = torch.from_numpy(v_res).to(gc.device)
    q = W.queries(w)
    got = case.run(q)
    assert gc.device_status() == 0
    assert not got[0].any()
    for b in (1, 2):
        ref, rows = case.oracle(q, b)
        check_outputs(got[b, rows], ref, f"seq {b}")


def test_residual_full_size_32k_sampled():
    """The 32K Llama layer with the pages' residual length of 128: the last 128
    tokens raw, the 32641 before them as the oracle's codes (sampled heads)."""
    w = W.WORKLOADS[1]
    heads = [0, 5]
    case = ResidualCase(w, stored_calib(1), [128], 128, heads=heads)
    q = W.queries(w)
    got = case.run(q)
    assert case.gc.device_status() == 0
    ref, rows = case.oracle(q, 0, heads=heads)
    check_outputs(got[0, rows], ref, "32K + residual 128")
