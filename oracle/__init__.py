"""ctypes wrapper around the fp64 C oracle (``vq_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never imports this
package.  The wrapper only marshals arrays; all arithmetic is in the C file,
which cites the VecInfer page section by section.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vq_oracle.c")
_LIB = os.path.join(_HERE, "libvq_oracle.so")
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (in-tree); returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
        sig = {
            "vqo_num_threads": (I, []),
            "vqo_set_num_threads": (None, [I]),
            "vqo_hadamard": (I, [I, P]),
            "vqo_smoothing_lambda": (None, [L, I, I, P, P]),
            "vqo_transform_keys": (None, [L, I, I, P, P, P, P]),
            "vqo_transform_query": (None, [I, P, P, P, P]),
            "vqo_vq_assign": (None, [L, I, I, P, P, P, P, P, P]),
            "vqo_kmeans": (None, [L, I, I, P, P, I, P, P]),
            "vqo_pack": (I, [L, I, I, P, I, P]),
            "vqo_unpack": (None, [L, I, I, P, I, P]),
            "vqo_dequantize": (None, [L, I, I, P, P, P]),
            "vqo_inverse_transform_keys": (None, [L, I, I, P, P, P, P]),
            "vqo_decode_attention": (None, [L, I, I, I, P, P, P, I, P, P, I, P, P, D, P]),
            "vqo_attention_fp": (None, [L, I, I, I, P, P, P, D, P]),
            "vqo_decode_attention_residual": (None, [L, L, I, I, I, P, P, P, I, P, P, I, P, P,
                                                      P, P, D, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _p(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def num_threads() -> int:
    return lib().vqo_num_threads()


def set_num_threads(n: int) -> None:
    lib().vqo_set_num_threads(int(n))


def hadamard(D: int) -> np.ndarray:
    H = np.zeros((D, D), dtype=np.float64)
    if lib().vqo_hadamard(D, _p(H)) != 0:
        raise ValueError(f"D={D} is not a power of two")
    return H


def smoothing_lambda(k_cal: np.ndarray) -> np.ndarray:
    """fp64 [Hkv][D] from calibration keys [T][Hkv][D]."""
    k = _f64(k_cal)
    T, Hkv, D = k.shape
    lam = np.zeros((Hkv, D))
    lib().vqo_smoothing_lambda(T, Hkv, D, _p(k), _p(lam))
    return lam


def transform_keys(k: np.ndarray, lam: np.ndarray) -> np.ndarray:
    """fp64 K~ = K diag(lam)^-1 H for keys [T][Hkv][D]."""
    k = _f64(k)
    T, Hkv, D = k.shape
    lam, H = _f64(lam), hadamard(D)
    out = np.zeros_like(k)
    lib().vqo_transform_keys(T, Hkv, D, _p(k), _p(lam), _p(H), _p(out))
    return out


def transform_query(q: np.ndarray, lam: np.ndarray) -> np.ndarray:
    q, lam = _f64(q), _f64(lam)
    D = q.shape[-1]
    H = hadamard(D)
    out = np.zeros(D)
    lib().vqo_transform_query(D, _p(q), _p(lam), _p(H), _p(out))
    return out


def vq_assign(x: np.ndarray, C: np.ndarray):
    """Nearest centroid of each row of x [n][d] in C [k][d].

    Returns (codes int32 [n], best fp64 [n], second fp64 [n], second_idx int32 [n]).
    """
    x, C = _f64(x), _f64(C)
    n, d = x.shape
    k = C.shape[0]
    codes = np.zeros(n, np.int32)
    best, second = np.zeros(n), np.zeros(n)
    sidx = np.zeros(n, np.int32)
    lib().vqo_vq_assign(n, d, k, _p(x), _p(C), _p(codes), _p(best), _p(second), _p(sidx))
    return codes, best, second, sidx


def kmeans(x: np.ndarray, init_idx: np.ndarray, iters: int) -> Tuple[np.ndarray, np.ndarray]:
    """Lloyd K-means; returns (centroids fp64 [k][d], objective fp64 [iters + 1])."""
    x = _f64(x)
    n, d = x.shape
    init = np.ascontiguousarray(init_idx, dtype=np.int64)
    k = init.shape[0]
    C = np.zeros((k, d))
    obj = np.zeros(iters + 1)
    lib().vqo_kmeans(n, d, k, _p(x), _p(init), iters, _p(C), _p(obj))
    return C, obj


def row_bytes(S: int, b: int) -> int:
    """Packed bytes per row of S codes of b bits, rounded up to a multiple of 4."""
    return (-(-S * b // 8) + 3) // 4 * 4


def pack(codes: np.ndarray, b: int, nbytes: Optional[int] = None) -> np.ndarray:
    """uint8 [..][nbytes] from int codes [..][S] (LSB-first bit stream per row)."""
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    S = codes.shape[-1]
    n = codes.size // S if S else 0
    nbytes = row_bytes(S, b) if nbytes is None else nbytes
    out = np.zeros(codes.shape[:-1] + (nbytes,), np.uint8)
    if lib().vqo_pack(n, S, b, _p(codes), nbytes, _p(out)) != 0:
        raise ValueError("codes do not fit the row")
    return out


def unpack(packed: np.ndarray, S: int, b: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    nbytes = packed.shape[-1]
    n = packed.size // nbytes if nbytes else 0
    out = np.zeros(packed.shape[:-1] + (S,), np.int32)
    lib().vqo_unpack(n, S, b, _p(packed), nbytes, _p(out))
    return out


def encode_keys(k: np.ndarray, lam: np.ndarray, Ck: np.ndarray, d: int):
    """Transform keys [T][Hkv][D] and assign every d-long sub-vector to C_k.

    Returns (codes int32 [T][Hkv][D/d], k~ fp64 [T][Hkv][D], best, second) with
    the distance arrays shaped like the codes.
    """
    kt = transform_keys(k, lam)
    T, Hkv, D = kt.shape
    codes, best, second, _ = vq_assign(kt.reshape(-1, d), Ck)
    shp = (T, Hkv, D // d)
    return codes.reshape(shp), kt, best.reshape(shp), second.reshape(shp)


def encode_values(v: np.ndarray, Cv: np.ndarray, d: int):
    """Assign every d-long sub-vector of raw values [T][Hkv][D] to C_v."""
    x = _f64(v)
    T, Hkv, D = x.shape
    codes, best, second, _ = vq_assign(x.reshape(-1, d), Cv)
    shp = (T, Hkv, D // d)
    return codes.reshape(shp), x, best.reshape(shp), second.reshape(shp)


def dequantize(codes: np.ndarray, C: np.ndarray) -> np.ndarray:
    """fp64 [..][S * d]: the centroids named by codes [..][S], concatenated."""
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    C = _f64(C)
    S, d = codes.shape[-1], C.shape[1]
    n = codes.size // S if S else 0
    out = np.zeros(codes.shape[:-1] + (S * d,))
    lib().vqo_dequantize(n, S, d, _p(codes), _p(C), _p(out))
    return out


def inverse_transform_keys(kt: np.ndarray, lam: np.ndarray) -> np.ndarray:
    """fp64 K = K~ H diag(lam) for transformed keys [T][Hkv][D]."""
    kt = _f64(kt)
    T, Hkv, D = kt.shape
    lam, H = _f64(lam), hadamard(D)
    out = np.zeros_like(kt)
    lib().vqo_inverse_transform_keys(T, Hkv, D, _p(kt), _p(lam), _p(H), _p(out))
    return out


def dequantize_kv(k_codes: np.ndarray, Ck: np.ndarray, v_codes: np.ndarray, Cv: np.ndarray,
                  lam: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 (K^, V^) [T][Hkv][D] in the original key and value spaces from codes
    [T][Hkv][S]: K^ = VQ^-1(K~_q) H diag(lam), V^ = VQ^-1(V_q)."""
    return inverse_transform_keys(dequantize(k_codes, Ck), lam), dequantize(v_codes, Cv)


def decode_attention(q: np.ndarray, lam: np.ndarray, k_codes: np.ndarray, Ck: np.ndarray,
                     v_codes: np.ndarray, Cv: np.ndarray, scale: Optional[float] = None
                     ) -> np.ndarray:
    """fp64 [Hq][D]: attention of one sequence's queries [Hq][D] over its codes.

    k_codes [N][Hkv][D/dk], v_codes [N][Hkv][D/dv]; scale defaults to 1/sqrt(D).
    """
    q, lam, Ck, Cv = _f64(q), _f64(lam), _f64(Ck), _f64(Cv)
    Hq, D = q.shape
    kc = np.ascontiguousarray(k_codes, dtype=np.int32)
    vc = np.ascontiguousarray(v_codes, dtype=np.int32)
    N, Hkv, _ = kc.shape
    dk, dv = Ck.shape[1], Cv.shape[1]
    H = hadamard(D)
    out = np.zeros((Hq, D))
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    lib().vqo_decode_attention(N, Hq, Hkv, D, _p(q), _p(lam), _p(H), dk, _p(kc), _p(Ck),
                               dv, _p(vc), _p(Cv), scale, _p(out))
    return out


def decode_attention_residual(q: np.ndarray, lam: np.ndarray, k_codes: np.ndarray,
                              Ck: np.ndarray, v_codes: np.ndarray, Cv: np.ndarray,
                              k_res: np.ndarray, v_res: np.ndarray,
                              scale: Optional[float] = None) -> np.ndarray:
    """fp64 [Hq][D]: one sequence's attention over its codes [N][Hkv][S] and its
    full-precision residual tokens k_res, v_res [R][Hkv][D], one softmax."""
    q, lam, Ck, Cv = _f64(q), _f64(lam), _f64(Ck), _f64(Cv)
    kr, vr = _f64(k_res), _f64(v_res)
    Hq, D = q.shape
    kc = np.ascontiguousarray(k_codes, dtype=np.int32)
    vc = np.ascontiguousarray(v_codes, dtype=np.int32)
    N, Hkv, _ = kc.shape
    R = kr.shape[0]
    dk, dv = Ck.shape[1], Cv.shape[1]
    H = hadamard(D)
    out = np.zeros((Hq, D))
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    lib().vqo_decode_attention_residual(N, R, Hq, Hkv, D, _p(q), _p(lam), _p(H), dk, _p(kc),
                                        _p(Ck), dv, _p(vc), _p(Cv), _p(kr), _p(vr), scale,
                                        _p(out))
    return out


def attention_fp(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                 scale: Optional[float] = None) -> np.ndarray:
    """fp64 [Hq][D]: unquantized softmax attention over K, V [N][Hkv][D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Hq, D = q.shape
    N, Hkv, _ = k.shape
    out = np.zeros((Hq, D))
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    lib().vqo_attention_fp(N, Hq, Hkv, D, _p(q), _p(k), _p(v), scale, _p(out))
    return out
