"""Python binding of libvqattn.so, the sm_103a VQ KV-cache decode-attention library.

Two layers, both argument marshalling only (every step of the computation runs
in the library's CUDA kernels):

* ``vq_*`` functions mirror the C ABI of include/vqattn.h one to one: they take
  device pointers as Python ints and raise :class:`VQError` on a non-OK status.
* ``encode_kv`` / ``decode_attention`` / ``alloc_pools`` / ``alloc_workspace``
  accept torch tensors (PyTorch supplies device memory and streams), check
  dtypes, shapes and devices, and pass their pointers to the ``vq_*`` calls.

There is no fallback: if libvqattn.so has not been built the first call raises.
Build it with ``python -m bit_vector_quantized_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvqattn.so")

VQ_OK = 0
VQ_ERR_INVALID_ARG = -1
VQ_ERR_UNSUPPORTED = -2
VQ_ERR_WORKSPACE = -3
VQ_ERR_CUDA = -4
STATUS_NAMES = {0: "VQ_OK", -1: "VQ_ERR_INVALID_ARG", -2: "VQ_ERR_UNSUPPORTED",
                -3: "VQ_ERR_WORKSPACE", -4: "VQ_ERR_CUDA"}
VQ_DEV_OK, VQ_DEV_BAD_PAGE, VQ_DEV_BAD_SLOT, VQ_DEV_TIMEOUT, VQ_DEV_BAD_CONFIG = 0, 1, 2, 3, 4

# every symbol include/vqattn.h declares
EXPORTED = ("vq_code_row_bytes", "vq_check_layout", "vq_encode_kv", "vq_decode_workspace_bytes",
            "vq_default_num_splits", "vq_decode_units_balanced", "vq_decode_attention",
            "vq_decode_partial",
            "vq_decode_partial_method", "vq_decode_combine", "vq_decode_step", "vq_dequantize_kv",
            "vq_decode_residual_workspace_bytes", "vq_decode_attention_residual",
            "vq_decode_attention_static", "vq_static_scratch_bytes", "vq_last_error",
            "vq_version")


class VQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class vq_layout(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("k_sub", ctypes.c_int32),
                ("k_bits", ctypes.c_int32), ("v_sub", ctypes.c_int32),
                ("v_bits", ctypes.c_int32), ("page_size", ctypes.c_int32)]

    def __repr__(self):
        return "vq_layout(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


def make_layout(head_dim=128, num_q_heads=32, num_kv_heads=8, k_sub=4, k_bits=8, v_sub=4,
                v_bits=8, page_size=256) -> vq_layout:
    return vq_layout(head_dim, num_q_heads, num_kv_heads, k_sub, k_bits, v_sub, v_bits, page_size)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m bit_vector_quantized_gb300.build` (no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        LP = ctypes.POINTER(vq_layout)
        sig = {
            "vq_code_row_bytes": (SZ, [I32, I32, I32]),
            "vq_check_layout": (I32, [LP, I32]),
            "vq_encode_kv": (I32, [LP, I32, P, P, P, P, P, P, P, P, I64, P, P]),
            "vq_dequantize_kv": (I32, [LP, I32, P, P, P, P, P, P, I64, P, P, P, P]),
            "vq_decode_residual_workspace_bytes": (SZ, [LP, I32, I32, I32, I32]),
            "vq_decode_attention_residual": (I32, [LP, I32, P, P, P, P, P, P, I64, P, I32, P, I32,
                                                   P, P, P, I32, ctypes.c_float, I32, P, P, SZ,
                                                   P, P]),
            "vq_decode_workspace_bytes": (SZ, [LP, I32, I32, I32, I32]),
            "vq_default_num_splits": (I32, [LP, I32, I32, I32]),
            "vq_decode_units_balanced": (I32, [LP, I32, I32, I32, I32]),
            "vq_decode_attention": (I32, [LP, I32, P, P, P, P, P, P, I64, P, I32, P, I32,
                                          ctypes.c_float, I32, P, P, SZ, P, P]),
            "vq_decode_partial": (I32, [LP, I32, P, P, P, P, P, P, I64, P, I32, P, I32,
                                        ctypes.c_float, I32, P, SZ, P, P]),
            "vq_decode_partial_method": (I32, [LP, I32, P, P, P, P, P, P, I64, P, I32, P, I32,
                                               ctypes.c_float, I32, I32, P, SZ, P, P]),
            "vq_decode_combine": (I32, [LP, I32, I32, I32, P, SZ, P, P]),
            "vq_decode_step": (I32, [LP, I32, P, P, P, P, P, P, P, P, I64, P, I32, P, I32,
                                     ctypes.c_float, I32, P, P, SZ, P, P]),
            "vq_decode_attention_static": (I32, [LP, I32, P, P, P, P, P, P, I64, P, I32, P, I32,
                                                 ctypes.c_float, I32, P, P, P]),
            "vq_static_scratch_bytes": (SZ, []),
            "vq_last_error": (ctypes.c_char_p, []),
            "vq_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(st: int) -> None:
    if st != VQ_OK:
        raise VQError(st, lib().vq_last_error().decode())


def _ptr(x) -> Optional[int]:
    return None if x is None or x == 0 else int(x)


# ------------------------------------------------------------- C ABI layer ---

def vq_code_row_bytes(head_dim: int, sub: int, bits: int) -> int:
    return int(lib().vq_code_row_bytes(head_dim, sub, bits))


def vq_check_layout(layout: vq_layout, for_decode: bool = False) -> None:
    _check(lib().vq_check_layout(ctypes.byref(layout), int(for_decode)))


def vq_encode_kv(layout, num_tokens, k, v, slot_mapping, lambda_, codebook_k, codebook_v,
                 k_pool, v_pool, num_pages, status=None, stream=None) -> None:
    _check(lib().vq_encode_kv(ctypes.byref(layout), num_tokens, _ptr(k), _ptr(v),
                              _ptr(slot_mapping), _ptr(lambda_), _ptr(codebook_k),
                              _ptr(codebook_v), _ptr(k_pool), _ptr(v_pool), num_pages,
                              _ptr(status), _ptr(stream)))


def vq_dequantize_kv(layout, num_tokens, slot_mapping, lambda_, codebook_k, codebook_v, k_pool,
                     v_pool, num_pages, k_out, v_out, status=None, stream=None) -> None:
    _check(lib().vq_dequantize_kv(ctypes.byref(layout), num_tokens, _ptr(slot_mapping),
                                  _ptr(lambda_), _ptr(codebook_k), _ptr(codebook_v), _ptr(k_pool),
                                  _ptr(v_pool), num_pages, _ptr(k_out), _ptr(v_out), _ptr(status),
                                  _ptr(stream)))


def vq_decode_residual_workspace_bytes(layout, batch, max_seq_len, num_splits=0, num_sms=0) -> int:
    return int(lib().vq_decode_residual_workspace_bytes(ctypes.byref(layout), batch, max_seq_len,
                                                        num_splits, num_sms))


def vq_decode_attention_residual(layout, batch, q, lambda_, codebook_k, codebook_v, k_pool,
                                 v_pool, num_pages, page_table, max_pages_per_seq, seq_lens,
                                 max_seq_len, k_res, v_res, res_lens, res_capacity, softmax_scale,
                                 num_splits, out, workspace, workspace_bytes, status=None,
                                 stream=None) -> None:
    _check(lib().vq_decode_attention_residual(
        ctypes.byref(layout), batch, _ptr(q), _ptr(lambda_), _ptr(codebook_k), _ptr(codebook_v),
        _ptr(k_pool), _ptr(v_pool), num_pages, _ptr(page_table), max_pages_per_seq,
        _ptr(seq_lens), max_seq_len, _ptr(k_res), _ptr(v_res), _ptr(res_lens), res_capacity,
        float(softmax_scale), num_splits, _ptr(out), _ptr(workspace), workspace_bytes,
        _ptr(status), _ptr(stream)))


def vq_decode_workspace_bytes(layout, batch, max_seq_len, num_splits=0, num_sms=0) -> int:
    return int(lib().vq_decode_workspace_bytes(ctypes.byref(layout), batch, max_seq_len,
                                               num_splits, num_sms))


def vq_default_num_splits(layout, batch, max_seq_len, num_sms=0) -> int:
    return int(lib().vq_default_num_splits(ctypes.byref(layout), batch, max_seq_len, num_sms))


def vq_decode_units_balanced(layout, batch, max_seq_len, num_splits=0, num_sms=0) -> int:
    return int(lib().vq_decode_units_balanced(ctypes.byref(layout), batch, max_seq_len,
                                              num_splits, num_sms))


def vq_decode_attention(layout, batch, q, lambda_, codebook_k, codebook_v, k_pool, v_pool,
                        num_pages, page_table, max_pages_per_seq, seq_lens, max_seq_len,
                        softmax_scale, num_splits, out, workspace, workspace_bytes,
                        status=None, stream=None) -> None:
    _check(lib().vq_decode_attention(ctypes.byref(layout), batch, _ptr(q), _ptr(lambda_),
                                     _ptr(codebook_k), _ptr(codebook_v), _ptr(k_pool),
                                     _ptr(v_pool), num_pages, _ptr(page_table), max_pages_per_seq,
                                     _ptr(seq_lens), max_seq_len, float(softmax_scale),
                                     num_splits, _ptr(out), _ptr(workspace), workspace_bytes,
                                     _ptr(status), _ptr(stream)))


def vq_decode_partial(layout, batch, q, lambda_, codebook_k, codebook_v, k_pool, v_pool,
                      num_pages, page_table, max_pages_per_seq, seq_lens, max_seq_len,
                      softmax_scale, num_splits, workspace, workspace_bytes, status=None,
                      stream=None) -> None:
    _check(lib().vq_decode_partial(ctypes.byref(layout), batch, _ptr(q), _ptr(lambda_),
                                   _ptr(codebook_k), _ptr(codebook_v), _ptr(k_pool), _ptr(v_pool),
                                   num_pages, _ptr(page_table), max_pages_per_seq, _ptr(seq_lens),
                                   max_seq_len, float(softmax_scale), num_splits, _ptr(workspace),
                                   workspace_bytes, _ptr(status), _ptr(stream)))


VQ_METHOD_GATHER, VQ_METHOD_LUT, VQ_METHOD_BINS = 0, 1, 2


def vq_decode_partial_method(layout, batch, q, lambda_, codebook_k, codebook_v, k_pool, v_pool,
                             num_pages, page_table, max_pages_per_seq, seq_lens, max_seq_len,
                             softmax_scale, num_splits, method, workspace, workspace_bytes,
                             status=None, stream=None) -> None:
    _check(lib().vq_decode_partial_method(
        ctypes.byref(layout), batch, _ptr(q), _ptr(lambda_), _ptr(codebook_k), _ptr(codebook_v),
        _ptr(k_pool), _ptr(v_pool), num_pages, _ptr(page_table), max_pages_per_seq, _ptr(seq_lens),
        max_seq_len, float(softmax_scale), num_splits, method, _ptr(workspace), workspace_bytes,
        _ptr(status), _ptr(stream)))


def vq_decode_combine(layout, batch, max_seq_len, num_splits, workspace, workspace_bytes, out,
                      stream=None) -> None:
    _check(lib().vq_decode_combine(ctypes.byref(layout), batch, max_seq_len, num_splits,
                                   _ptr(workspace), workspace_bytes, _ptr(out), _ptr(stream)))


def vq_decode_step(layout, batch, q, k_new, v_new, lambda_, codebook_k, codebook_v, k_pool,
                   v_pool, num_pages, page_table, max_pages_per_seq, seq_lens, max_seq_len,
                   softmax_scale, num_splits, out, workspace, workspace_bytes, status=None,
                   stream=None) -> None:
    """Append the new token of every sequence (position seq_lens - 1), then decode attention."""
    _check(lib().vq_decode_step(ctypes.byref(layout), batch, _ptr(q), _ptr(k_new), _ptr(v_new),
                                _ptr(lambda_), _ptr(codebook_k), _ptr(codebook_v), _ptr(k_pool),
                                _ptr(v_pool), num_pages, _ptr(page_table), max_pages_per_seq,
                                _ptr(seq_lens), max_seq_len, float(softmax_scale), num_splits,
                                _ptr(out), _ptr(workspace), workspace_bytes, _ptr(status),
                                _ptr(stream)))


def vq_decode_attention_static(layout, batch, q, lambda_, codebook_k, codebook_v, k_pool, v_pool,
                               num_pages, page_table, max_pages_per_seq, seq_lens, max_seq_len,
                               softmax_scale, num_splits, out, status=None, stream=None) -> None:
    """vq_decode_attention for callers that cannot allocate: no workspace argument;
    the split partials live in the library's fixed device array (see the header)."""
    _check(lib().vq_decode_attention_static(ctypes.byref(layout), batch, _ptr(q), _ptr(lambda_),
                                            _ptr(codebook_k), _ptr(codebook_v), _ptr(k_pool),
                                            _ptr(v_pool), num_pages, _ptr(page_table),
                                            max_pages_per_seq, _ptr(seq_lens), max_seq_len,
                                            float(softmax_scale), num_splits, _ptr(out),
                                            _ptr(status), _ptr(stream)))


def vq_static_scratch_bytes() -> int:
    return int(lib().vq_static_scratch_bytes())


def vq_last_error() -> str:
    return lib().vq_last_error().decode()


def vq_version() -> str:
    return lib().vq_version().decode()


# ------------------------------------------------------------ torch layer ---

def _torch():
    import torch
    return torch


def _dev_ptr(t, dtype, name, shape=None):
    torch = _torch()
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def row_bytes(layout: vq_layout) -> Tuple[int, int]:
    return (vq_code_row_bytes(layout.head_dim, layout.k_sub, layout.k_bits),
            vq_code_row_bytes(layout.head_dim, layout.v_sub, layout.v_bits))


def alloc_pools(layout: vq_layout, num_pages: int, device="cuda", zero: bool = False):
    """(k_pool, v_pool) uint8 tensors [num_pages][Hkv][P][row_bytes]."""
    torch = _torch()
    kr, vr = row_bytes(layout)
    mk = torch.zeros if zero else torch.empty
    shape = (num_pages, layout.num_kv_heads, layout.page_size)
    return (mk(shape + (kr,), dtype=torch.uint8, device=device),
            mk(shape + (vr,), dtype=torch.uint8, device=device))


def alloc_workspace(layout: vq_layout, batch: int, max_seq_len: int, num_splits: int = 0,
                    device="cuda"):
    torch = _torch()
    n = vq_decode_workspace_bytes(layout, batch, max_seq_len, num_splits)
    if n == 0 and batch > 0:
        raise VQError(VQ_ERR_INVALID_ARG, "cannot size the workspace")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def encode_kv(layout: vq_layout, k, v, slot_mapping, lambda_, codebook_k, codebook_v,
              k_pool, v_pool, status=None, stream=None) -> None:
    """Encode fp16 keys/values [T][Hkv][D] into the pools at slot_mapping (int64 [T])."""
    torch = _torch()
    ref = k if k is not None else v
    T = ref.shape[0]
    D, H = layout.head_dim, layout.num_kv_heads
    vq_encode_kv(layout, T,
                 _dev_ptr(k, torch.float16, "k", (T, H, D)),
                 _dev_ptr(v, torch.float16, "v", (T, H, D)),
                 _dev_ptr(slot_mapping, torch.int64, "slot_mapping", (T,)),
                 _dev_ptr(lambda_, torch.float32, "lambda", (H, D)) if k is not None else None,
                 _dev_ptr(codebook_k, torch.float16, "codebook_k",
                          (1 << layout.k_bits, layout.k_sub)) if k is not None else None,
                 _dev_ptr(codebook_v, torch.float16, "codebook_v",
                          (1 << layout.v_bits, layout.v_sub)) if v is not None else None,
                 _dev_ptr(k_pool, torch.uint8, "k_pool") if k is not None else None,
                 _dev_ptr(v_pool, torch.uint8, "v_pool") if v is not None else None,
                 (k_pool if k is not None else v_pool).shape[0],
                 _dev_ptr(status, torch.int32, "status", (1,)), _stream(stream))


def dequantize_kv(layout: vq_layout, slot_mapping, lambda_, codebook_k, codebook_v, k_pool,
                  v_pool, keys: bool = True, values: bool = True, k_out=None, v_out=None,
                  status=None, stream=None):
    """(K^, V^) fp16 [T][Hkv][D] read back from the pools at slot_mapping (int64 [T]);
    keys in the original space.  A half not asked for is returned as None."""
    torch = _torch()
    T = slot_mapping.shape[0]
    D, H = layout.head_dim, layout.num_kv_heads
    dev = slot_mapping.device
    if keys and k_out is None:
        k_out = torch.empty((T, H, D), dtype=torch.float16, device=dev)
    if values and v_out is None:
        v_out = torch.empty((T, H, D), dtype=torch.float16, device=dev)
    k_out, v_out = (k_out if keys else None), (v_out if values else None)
    vq_dequantize_kv(layout, T, _dev_ptr(slot_mapping, torch.int64, "slot_mapping", (T,)),
                     _dev_ptr(lambda_, torch.float32, "lambda", (H, D)) if keys else None,
                     _dev_ptr(codebook_k, torch.float16, "codebook_k",
                              (1 << layout.k_bits, layout.k_sub)) if keys else None,
                     _dev_ptr(codebook_v, torch.float16, "codebook_v",
                              (1 << layout.v_bits, layout.v_sub)) if values else None,
                     _dev_ptr(k_pool, torch.uint8, "k_pool") if keys else None,
                     _dev_ptr(v_pool, torch.uint8, "v_pool") if values else None,
                     (k_pool if keys else v_pool).shape[0],
                     _dev_ptr(k_out, torch.float16, "k_out", (T, H, D)) if keys else None,
                     _dev_ptr(v_out, torch.float16, "v_out", (T, H, D)) if values else None,
                     _dev_ptr(status, torch.int32, "status", (1,)), _stream(stream))
    return k_out, v_out


def decode_attention(layout: vq_layout, q, lambda_, codebook_k, codebook_v, k_pool, v_pool,
                     page_table, seq_lens, max_seq_len: int, out=None, workspace=None,
                     softmax_scale: float = 0.0, num_splits: int = 0, status=None,
                     stream=None):
    """fp16 [B][Hq][D] attention of queries q [B][Hq][D] over the quantized pools."""
    torch = _torch()
    B = q.shape[0]
    D = layout.head_dim
    if out is None:
        out = torch.empty((B, layout.num_q_heads, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(layout, B, max_seq_len, num_splits, q.device)
    vq_decode_attention(layout, B,
                        _dev_ptr(q, torch.float16, "q", (B, layout.num_q_heads, D)),
                        _dev_ptr(lambda_, torch.float32, "lambda", (layout.num_kv_heads, D)),
                        _dev_ptr(codebook_k, torch.float16, "codebook_k",
                                 (1 << layout.k_bits, layout.k_sub)),
                        _dev_ptr(codebook_v, torch.float16, "codebook_v",
                                 (1 << layout.v_bits, layout.v_sub)),
                        _dev_ptr(k_pool, torch.uint8, "k_pool"),
                        _dev_ptr(v_pool, torch.uint8, "v_pool"), k_pool.shape[0],
                        _dev_ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                        _dev_ptr(seq_lens, torch.int32, "seq_lens", (B,)), max_seq_len,
                        softmax_scale, num_splits,
                        _dev_ptr(out, torch.float16, "out", (B, layout.num_q_heads, D)),
                        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                        _dev_ptr(status, torch.int32, "status", (1,)), _stream(stream))
    return out


def decode_attention_method(layout: vq_layout, q, lambda_, codebook_k, codebook_v, k_pool,
                            v_pool, page_table, seq_lens, max_seq_len: int, method: int,
                            out=None, workspace=None, softmax_scale: float = 0.0,
                            num_splits: int = 0, status=None, stream=None):
    """decode_attention with an explicit score / P.V method (vq_decode_partial_method,
    then vq_decode_combine)."""
    torch = _torch()
    B = q.shape[0]
    D = layout.head_dim
    if out is None:
        out = torch.empty((B, layout.num_q_heads, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(layout, B, max_seq_len, num_splits, q.device)
    st = _stream(stream)
    vq_decode_partial_method(layout, B,
                             _dev_ptr(q, torch.float16, "q", (B, layout.num_q_heads, D)),
                             _dev_ptr(lambda_, torch.float32, "lambda", (layout.num_kv_heads, D)),
                             _dev_ptr(codebook_k, torch.float16, "codebook_k",
                                      (1 << layout.k_bits, layout.k_sub)),
                             _dev_ptr(codebook_v, torch.float16, "codebook_v",
                                      (1 << layout.v_bits, layout.v_sub)),
                             _dev_ptr(k_pool, torch.uint8, "k_pool"),
                             _dev_ptr(v_pool, torch.uint8, "v_pool"), k_pool.shape[0],
                             _dev_ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                             _dev_ptr(seq_lens, torch.int32, "seq_lens", (B,)), max_seq_len,
                             softmax_scale, num_splits, method,
                             _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                             _dev_ptr(status, torch.int32, "status", (1,)), st)
    vq_decode_combine(layout, B, max_seq_len, num_splits,
                      _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                      _dev_ptr(out, torch.float16, "out", (B, layout.num_q_heads, D)), st)
    return out


def decode_attention_residual(layout: vq_layout, q, lambda_, codebook_k, codebook_v, k_pool,
                              v_pool, page_table, seq_lens, max_seq_len: int, k_res, v_res,
                              res_lens, out=None, workspace=None, softmax_scale: float = 0.0,
                              num_splits: int = 0, status=None, stream=None):
    """fp16 [B][Hq][D] attention of q over the quantized pools (seq_lens tokens)
    plus the full-precision residual k_res / v_res [B][Hkv][capacity][D]
    (res_lens tokens), one softmax."""
    torch = _torch()
    B = q.shape[0]
    D, H = layout.head_dim, layout.num_kv_heads
    cap = k_res.shape[2]
    if out is None:
        out = torch.empty((B, layout.num_q_heads, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        n = vq_decode_residual_workspace_bytes(layout, B, max_seq_len, num_splits)
        if n == 0 and B > 0:
            raise VQError(VQ_ERR_INVALID_ARG, "cannot size the workspace")
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    vq_decode_attention_residual(
        layout, B, _dev_ptr(q, torch.float16, "q", (B, layout.num_q_heads, D)),
        _dev_ptr(lambda_, torch.float32, "lambda", (H, D)),
        _dev_ptr(codebook_k, torch.float16, "codebook_k", (1 << layout.k_bits, layout.k_sub)),
        _dev_ptr(codebook_v, torch.float16, "codebook_v", (1 << layout.v_bits, layout.v_sub)),
        _dev_ptr(k_pool, torch.uint8, "k_pool"), _dev_ptr(v_pool, torch.uint8, "v_pool"),
        k_pool.shape[0], _dev_ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
        _dev_ptr(seq_lens, torch.int32, "seq_lens", (B,)), max_seq_len,
        _dev_ptr(k_res, torch.float16, "k_res", (B, H, cap, D)),
        _dev_ptr(v_res, torch.float16, "v_res", (B, H, cap, D)),
        _dev_ptr(res_lens, torch.int32, "res_lens", (B,)), cap, softmax_scale, num_splits,
        _dev_ptr(out, torch.float16, "out", (B, layout.num_q_heads, D)),
        _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev_ptr(status, torch.int32, "status", (1,)), _stream(stream))
    return out


def decode_step(layout: vq_layout, q, k_new, v_new, lambda_, codebook_k, codebook_v, k_pool,
                v_pool, page_table, seq_lens, max_seq_len: int, out=None, workspace=None,
                softmax_scale: float = 0.0, num_splits: int = 0, status=None, stream=None):
    """One decode step: append k_new / v_new [B][Hkv][D] as token seq_lens - 1 of each
    sequence, then fp16 [B][Hq][D] attention of q [B][Hq][D] over seq_lens tokens."""
    torch = _torch()
    B = q.shape[0]
    D, H = layout.head_dim, layout.num_kv_heads
    if out is None:
        out = torch.empty((B, layout.num_q_heads, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        n = vq_decode_workspace_bytes(layout, B, max_seq_len, num_splits)
        if n == 0 and B > 0:
            raise VQError(VQ_ERR_INVALID_ARG, "cannot size the workspace")
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    vq_decode_step(layout, B,
                   _dev_ptr(q, torch.float16, "q", (B, layout.num_q_heads, D)),
                   _dev_ptr(k_new, torch.float16, "k_new", (B, H, D)),
                   _dev_ptr(v_new, torch.float16, "v_new", (B, H, D)),
                   _dev_ptr(lambda_, torch.float32, "lambda", (H, D)),
                   _dev_ptr(codebook_k, torch.float16, "codebook_k", (1 << layout.k_bits, layout.k_sub)),
                   _dev_ptr(codebook_v, torch.float16, "codebook_v", (1 << layout.v_bits, layout.v_sub)),
                   _dev_ptr(k_pool, torch.uint8, "k_pool"),
                   _dev_ptr(v_pool, torch.uint8, "v_pool"), k_pool.shape[0],
                   _dev_ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                   _dev_ptr(seq_lens, torch.int32, "seq_lens", (B,)), max_seq_len,
                   softmax_scale, num_splits,
                   _dev_ptr(out, torch.float16, "out", (B, layout.num_q_heads, D)),
                   _dev_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                   _dev_ptr(status, torch.int32, "status", (1,)), _stream(stream))
    return out
