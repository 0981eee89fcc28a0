"""The C ABI library: loads, exports every declared symbol, host-side logic.

No test here launches a kernel: every call either is pure host arithmetic or
fails argument validation before anything reaches the GPU.
"""
import ctypes
import os
import re

import pytest

import bit_vector_quantized_gb300 as vq

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "vqattn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(vq.LIB_PATH):
        from bit_vector_quantized_gb300 import build
        build.build()
    return vq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vq_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(vq.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert "sm_103a" in vq.vq_version()


@pytest.mark.parametrize("d,sub,bits,expect", [(128, 4, 8, 32), (128, 2, 8, 64), (128, 4, 9, 36),
                                                (128, 8, 12, 24), (128, 1, 1, 16), (128, 3, 8, 0),
                                                (128, 4, 0, 0), (0, 4, 8, 0)])
def test_code_row_bytes(lib, d, sub, bits, expect):
    assert vq.vq_code_row_bytes(d, sub, bits) == expect


def test_check_layout(lib):
    vq.vq_check_layout(vq.make_layout(), True)
    vq.vq_check_layout(vq.make_layout(k_sub=2, v_bits=9, num_q_heads=40), True)
    vq.vq_check_layout(vq.make_layout(k_sub=8, k_bits=12), False)
    cases = [(dict(head_dim=96), vq.VQ_ERR_INVALID_ARG), (dict(head_dim=64), vq.VQ_ERR_UNSUPPORTED),
             (dict(num_q_heads=30), vq.VQ_ERR_INVALID_ARG), (dict(num_q_heads=72), vq.VQ_ERR_UNSUPPORTED),
             (dict(k_sub=3), vq.VQ_ERR_INVALID_ARG), (dict(v_bits=13), vq.VQ_ERR_INVALID_ARG),
             (dict(page_size=40), vq.VQ_ERR_INVALID_ARG)]
    for kw, st in cases:
        with pytest.raises(vq.VQError) as e:
            vq.vq_check_layout(vq.make_layout(**kw), False)
        assert e.value.status == st
    with pytest.raises(vq.VQError) as e:
        vq.vq_check_layout(vq.make_layout(k_sub=8, k_bits=12), True)
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED and "decode" in vq.vq_last_error()


def test_split_heuristic_and_workspace(lib):
    L1 = vq.make_layout()
    assert vq.vq_default_num_splits(L1, 1, 32769, 152) == 19          # 8 heads x 19 = 152 units
    assert vq.vq_default_num_splits(L1, 1, 196609, 152) == 19
    L4 = vq.make_layout(num_q_heads=40, k_sub=2, v_bits=9)
    s4 = vq.vq_default_num_splits(L4, 64, 16385, 152)
    assert 1 <= s4 <= 8
    assert vq.vq_default_num_splits(L1, 1, 0, 152) == 1
    n = vq.vq_decode_workspace_bytes(L1, 1, 32769, 19, 152)
    assert n >= 32 * 19 * (128 + 2) * 4 and n % 256 == 0
    assert vq.vq_decode_workspace_bytes(L1, -1, 10, 0, 152) == 0


def _up256(x):
    return (x + 255) // 256 * 256


def test_length_balanced_split_counts_and_workspace(lib):
    """Two or more sequences get length-balanced units with 1 + ceil(2 SMs /
    pairs) partial slots per (sequence, KV head); the workspace holds the
    partials, then one int32 unit count per pair."""
    L1 = vq.make_layout()                                                  # 8 KV heads
    assert vq.vq_default_num_splits(L1, 16, 8193, 152) == 1 + 3            # 128 pairs
    assert vq.vq_default_num_splits(L1, 2, 32769, 152) == 1 + 19           # 16 pairs
    L4 = vq.make_layout(num_q_heads=40, k_sub=2, v_bits=9)
    assert vq.vq_default_num_splits(L4, 64, 16385, 152) == 2               # 512 pairs
    # more sequences than the balanced assignment takes: the fixed-split heuristic
    s = vq.vq_default_num_splits(L1, 600, 100, 152)
    assert s >= 1
    assert vq.vq_decode_units_balanced(L1, 600, 100, 0, 152) == 0
    assert vq.vq_decode_units_balanced(L1, 16, 8193, 0, 152) == 1
    assert vq.vq_decode_units_balanced(L1, 1, 32769, 0, 152) == 0         # one sequence: fixed splits
    assert vq.vq_decode_units_balanced(L1, 16, 8193, 1, 152) == 0         # one slot per pair
    assert vq.vq_decode_units_balanced(L1, 16, 0, 0, 152) == 0            # nothing to attend
    assert vq.vq_decode_units_balanced(L1, -1, 10, 0, 152) == -1
    # 512 sequences x 8 KV heads of 1M tokens: too many units per CTA for the balanced bound
    assert vq.vq_decode_units_balanced(L1, 512, 1 << 20, 4, 152) == 0
    rows = 3 * 32 * 19
    assert vq.vq_decode_workspace_bytes(L1, 3, 32769, 19, 152) == \
        _up256(rows * 128 * 4) + _up256(rows * 2 * 4) + _up256(3 * 8 * 4)


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation fails first


def test_encode_rejects_bad_arguments(lib):
    L = vq.make_layout()
    args = dict(layout=L, num_tokens=4, k=FAKE, v=FAKE, slot_mapping=FAKE, lambda_=FAKE,
                codebook_k=FAKE, codebook_v=FAKE, k_pool=FAKE, v_pool=FAKE, num_pages=4)
    bad = [dict(num_tokens=-1), dict(k=None, v=None), dict(slot_mapping=None), dict(num_pages=0),
           dict(lambda_=None), dict(codebook_v=None), dict(k=FAKE + 4), dict(v_pool=FAKE + 8),
           dict(layout=vq.make_layout(page_size=8))]
    for kw in bad:
        a = dict(args, **kw)
        with pytest.raises(vq.VQError) as e:
            vq.vq_encode_kv(**a)
        assert e.value.status == vq.VQ_ERR_INVALID_ARG, kw


def test_decode_rejects_bad_arguments(lib):
    L = vq.make_layout()
    args = dict(layout=L, batch=1, q=FAKE, lambda_=FAKE, codebook_k=FAKE, codebook_v=FAKE,
                k_pool=FAKE, v_pool=FAKE, num_pages=4, page_table=FAKE, max_pages_per_seq=4,
                seq_lens=FAKE, max_seq_len=100, softmax_scale=0.0, num_splits=0, out=FAKE,
                workspace=FAKE, workspace_bytes=1 << 30)
    bad = [(dict(batch=-2), vq.VQ_ERR_INVALID_ARG), (dict(q=None), vq.VQ_ERR_INVALID_ARG),
           (dict(out=FAKE + 2), vq.VQ_ERR_INVALID_ARG), (dict(max_seq_len=5000), vq.VQ_ERR_INVALID_ARG),
           (dict(max_pages_per_seq=0), vq.VQ_ERR_INVALID_ARG),
           (dict(softmax_scale=float("nan")), vq.VQ_ERR_INVALID_ARG),
           (dict(num_splits=5000), vq.VQ_ERR_INVALID_ARG),
           (dict(layout=vq.make_layout(v_sub=8)), vq.VQ_ERR_UNSUPPORTED)]
    for kw, st in bad:
        with pytest.raises(vq.VQError) as e:
            vq.vq_decode_attention(**dict(args, **kw))
        assert e.value.status == st, kw


def test_empty_calls_are_noops(lib):
    L = vq.make_layout()
    vq.vq_encode_kv(L, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4)
    vq.vq_decode_attention(L, 0, None, None, None, None, None, None, 1, None, 1, None, 0, 0.0, 0,
                           None, None, 0)


def test_check_layout_one_and_a_half_bit(lib):
    L = vq.make_layout(k_sub=8, k_bits=12, v_sub=8, v_bits=12)
    vq.vq_check_layout(L, True)                      # the pages' 1.5-bit configuration
    assert vq.vq_code_row_bytes(128, 8, 12) == 24
    for kw in (dict(k_sub=8, k_bits=12, v_sub=8, v_bits=8), dict(k_sub=8, k_bits=11, v_sub=8, v_bits=12),
               dict(k_sub=4, k_bits=8, v_sub=8, v_bits=12)):
        with pytest.raises(vq.VQError) as e:
            vq.vq_check_layout(vq.make_layout(**kw), True)
        assert e.value.status == vq.VQ_ERR_UNSUPPORTED, kw


def test_workspace_holds_the_sliced_append_candidates_for_large_codebooks(lib):
    # 12-bit codebooks: the decode step's append leaves 8 slices x 32 lanes x 4
    # (score, index) candidates per new vector and tensor after the partials
    small = vq.make_layout()
    wide = vq.make_layout(k_sub=8, k_bits=12, v_sub=8, v_bits=12)
    n = vq.vq_decode_workspace_bytes(small, 3, 32769, 19, 152)
    w = vq.vq_decode_workspace_bytes(wide, 3, 32769, 19, 152)
    assert w == n + 3 * 8 * 2 * 8 * 32 * 4 * 8


def test_residual_workspace_is_the_split_workspace(lib):
    # the window's tokens join the split partials: no extra partial per row
    L = vq.make_layout()
    n = vq.vq_decode_workspace_bytes(L, 3, 32769, 19, 152)
    r = vq.vq_decode_residual_workspace_bytes(L, 3, 32769, 19, 152)
    assert r == n
    assert vq.vq_decode_residual_workspace_bytes(L, 3, 32769, 0, 152) == \
        vq.vq_decode_residual_workspace_bytes(L, 3, 32769, vq.vq_default_num_splits(L, 3, 32769, 152), 152)
    assert vq.vq_decode_residual_workspace_bytes(L, -1, 10, 0, 152) == 0


def test_residual_rejects_bad_arguments(lib):
    L = vq.make_layout()
    args = dict(layout=L, batch=1, q=FAKE, lambda_=FAKE, codebook_k=FAKE, codebook_v=FAKE,
                k_pool=FAKE, v_pool=FAKE, num_pages=4, page_table=FAKE, max_pages_per_seq=4,
                seq_lens=FAKE, max_seq_len=100, k_res=FAKE, v_res=FAKE, res_lens=FAKE,
                res_capacity=128, softmax_scale=0.0, num_splits=0, out=FAKE, workspace=FAKE,
                workspace_bytes=1 << 30)
    bad = [dict(res_capacity=0), dict(res_capacity=4097), dict(k_res=None), dict(v_res=FAKE + 4),
           dict(res_lens=None), dict(out=None), dict(batch=-1), dict(q=None)]
    for kw in bad:
        with pytest.raises(vq.VQError) as e:
            vq.vq_decode_attention_residual(**dict(args, **kw))
        assert e.value.status == vq.VQ_ERR_INVALID_ARG, kw
    with pytest.raises(vq.VQError) as e:
        vq.vq_decode_attention_residual(**dict(args, layout=vq.make_layout(v_sub=8)))
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED
    vq.vq_decode_attention_residual(**dict(args, batch=0, q=None, k_res=None))  # empty batch: no-op


def test_dequantize_rejects_bad_arguments(lib):
    L = vq.make_layout()
    args = dict(layout=L, num_tokens=4, slot_mapping=FAKE, lambda_=FAKE, codebook_k=FAKE,
                codebook_v=FAKE, k_pool=FAKE, v_pool=FAKE, num_pages=4, k_out=FAKE, v_out=FAKE)
    bad = [dict(num_tokens=-1), dict(k_out=None, v_out=None), dict(slot_mapping=None),
           dict(num_pages=0), dict(lambda_=None), dict(codebook_v=None), dict(k_pool=None),
           dict(k_out=FAKE + 8), dict(layout=vq.make_layout(page_size=8))]
    for kw in bad:
        with pytest.raises(vq.VQError) as e:
            vq.vq_dequantize_kv(**dict(args, **kw))
        assert e.value.status == vq.VQ_ERR_INVALID_ARG, kw
    vq.vq_dequantize_kv(**dict(args, num_tokens=0, k_out=None, v_out=None))  # no tokens: no-op


def test_step_rejects_bad_arguments(lib):
    L = vq.make_layout()
    args = dict(layout=L, batch=1, q=FAKE, k_new=FAKE, v_new=FAKE, lambda_=FAKE, codebook_k=FAKE,
                codebook_v=FAKE, k_pool=FAKE, v_pool=FAKE, num_pages=4, page_table=FAKE,
                max_pages_per_seq=4, seq_lens=FAKE, max_seq_len=100, softmax_scale=0.0,
                num_splits=0, out=FAKE, workspace=FAKE, workspace_bytes=1 << 30)
    for kw in (dict(k_new=None), dict(v_new=FAKE + 2), dict(out=None), dict(batch=-3),
               dict(page_table=None), dict(num_pages=0)):
        with pytest.raises(vq.VQError) as e:
            vq.vq_decode_step(**dict(args, **kw))
        assert e.value.status == vq.VQ_ERR_INVALID_ARG, kw
