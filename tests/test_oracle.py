"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, a library routine,
a hand-computed fixture under tests/golden/, an invariant the VecInfer page
states, or brute force on tiny inputs.  Chosen so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails at least one test.
"""
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        rows.setdefault(key, []).append([float(v) for v in vals])
    return rows


# ---------------------------------------------------------------- Hadamard ---

@pytest.mark.parametrize("D", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_closed_form_and_orthogonality(D):
    """Recursion == Sylvester closed form (-1)^popcount(i&j)/sqrt(D); H H^T = I."""
    H = oracle.hadamard(D)
    i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
    pop = np.vectorize(lambda x: bin(x).count("1"))(i & j)
    closed = (-1.0) ** pop / np.sqrt(D)
    assert np.max(np.abs(H - closed)) < 1e-15
    assert np.max(np.abs(H @ H.T - np.eye(D))) < 1e-12
    assert np.allclose(np.abs(H), 1 / np.sqrt(D), rtol=0, atol=1e-15)


@pytest.mark.parametrize("D", [2, 8, 128])
def test_hadamard_matches_scipy(D):
    """scipy's Sylvester construction (+-1 entries) scaled by 1/sqrt(D)."""
    assert np.max(np.abs(oracle.hadamard(D) - scipy.linalg.hadamard(D) / np.sqrt(D))) < 1e-15


def test_hadamard_golden_h4():
    rows = np.array([[float(v) for v in line.split()]
                     for line in open(os.path.join(GOLDEN, "hadamard_h4.txt"))
                     if line.strip() and not line.startswith("#")])
    assert np.max(np.abs(oracle.hadamard(4) * 2 - rows)) < 1e-15


def test_hadamard_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        oracle.hadamard(12)


def _fwht(x):
    """Textbook in-place fast Walsh-Hadamard butterflies (natural order), / sqrt(n)."""
    x = np.array(x, dtype=np.float64)
    n = x.shape[-1]
    h = 1
    while h < n:
        for i in range(0, n, 2 * h):
            a = x[..., i:i + h].copy()
            b = x[..., i + h:i + 2 * h].copy()
            x[..., i:i + h] = a + b
            x[..., i + h:i + 2 * h] = a - b
        h *= 2
    return x / np.sqrt(n)


def test_dense_transform_equals_fast_wht():
    rng = np.random.default_rng(10)
    k = rng.standard_normal((7, 3, 128))
    lam = rng.uniform(0.5, 4.0, (3, 128))
    kt = oracle.transform_keys(k, lam)
    assert np.max(np.abs(kt - _fwht(k / lam[None]))) < 1e-12


# ------------------------------------------------------ transforms, scores ---

def test_golden_key_transform():
    f = _fixture("attention_d2.txt")
    kt = oracle.transform_keys(np.array(f["k"]).reshape(1, 1, 2), np.array(f["lambda_k"]))
    assert np.max(np.abs(kt.reshape(2) - np.array(f["ktilde"][0]))) < 1e-15


def test_score_invariance_unquantized():
    """(q diag(lam) H)(K diag(lam)^-1 H)^T / sqrt(D) == q K^T / sqrt(D) to 1e-9."""
    rng = np.random.default_rng(11)
    D, T = 128, 64
    k = rng.standard_normal((T, 1, D))
    k[:, 0, [3, 77]] *= 20.0
    lam = np.sqrt(np.abs(k).max(axis=0))
    q = rng.standard_normal(D)
    qt = oracle.transform_query(q, lam[0])
    kt = oracle.transform_keys(k, lam)
    s_t = kt[:, 0, :] @ qt / np.sqrt(D)
    s = k[:, 0, :] @ q / np.sqrt(D)
    assert np.max(np.abs(s_t - s)) < 1e-9


def test_transform_preserves_norm():
    """Lemma 1 setting: H is orthogonal, so ||K~_row|| == ||K_row / lam||."""
    rng = np.random.default_rng(12)
    k = rng.standard_normal((16, 2, 128)) * 5
    lam = rng.uniform(0.3, 3, (2, 128))
    kt = oracle.transform_keys(k, lam)
    assert np.allclose(np.linalg.norm(kt, axis=-1), np.linalg.norm(k / lam[None], axis=-1),
                       rtol=1e-13, atol=0)


def test_transform_gaussianizes_outliers():
    """Lemma 1: outlier channels are spread; per-entry variance ~ ||K_i||^2 / D."""
    rng = np.random.default_rng(13)
    D = 128
    k = rng.standard_normal((4096, 1, D))
    k[:, 0, 5] *= 20.0
    kt = oracle.transform_keys(k, np.ones((1, D)))
    assert np.abs(kt).max() < 0.5 * np.abs(k).max()
    pred = (k[:, 0, :] ** 2).sum(1).mean() / D
    assert abs(kt.var() / pred - 1) < 0.05


def test_smoothing_lambda_hand_example():
    """lambda_i = sqrt(max_t |K[t, i]|): K = [[1,-4],[-9,2]] -> [3, 2]."""
    k = np.array([[[1.0, -4.0]], [[-9.0, 2.0]]])
    assert np.array_equal(oracle.smoothing_lambda(k), np.array([[3.0, 2.0]]))


def test_smoothing_lambda_per_head():
    k = np.zeros((3, 2, 4))
    k[1, 0, :] = [16, -25, 0.25, 1]
    k[2, 1, :] = [-4, 9, 100, 0]
    lam = oracle.smoothing_lambda(k)
    assert np.array_equal(lam, np.array([[4, 5, 0.5, 1], [2, 3, 10, 0]]))


# ------------------------------------------------------------ VQ argmin ---

def test_vq_assign_brute_force_tiny():
    """All inputs on a small integer grid (exact distances, exhaustive ties)."""
    grid = np.array([[a, b] for a in range(-2, 3) for b in range(-2, 3)], dtype=np.float64)
    rng = np.random.default_rng(14)
    for k in (1, 2, 3, 4, 7, 16):
        C = rng.integers(-2, 3, size=(k, 2)).astype(np.float64)
        codes, best, second, sidx = oracle.vq_assign(grid, C)
        for v, x in enumerate(grid):
            d = [float(((x - c) ** 2).sum()) for c in C]
            jstar = min(range(k), key=lambda j: (d[j], j))   # first index of the minimum
            assert codes[v] == jstar
            assert best[v] == d[jstar]
            rest = sorted((d[j], j) for j in range(k) if j != jstar)
            if rest:
                assert second[v] == rest[0][0]
                assert sidx[v] == rest[0][1]
            else:
                assert second[v] == np.inf and sidx[v] == -1


def test_vq_assign_duplicate_centroids_pick_lowest():
    C = np.array([[1.0, 1.0], [0.0, 0.0], [0.0, 0.0], [1.0, 1.0]])
    x = np.array([[0.0, 0.0], [1.0, 1.0], [0.5, 0.5]])
    codes, best, second, _ = oracle.vq_assign(x, C)
    assert list(codes) == [1, 0, 0]
    assert best[2] == second[2] == 0.5


def test_vq_assign_matches_expanded_numpy_argmin():
    """Random sub-vectors, d = 4: oracle vs numpy's first-minimum argmin."""
    rng = np.random.default_rng(15)
    x = rng.standard_normal((500, 4))
    C = rng.standard_normal((64, 4))
    codes, best, _, _ = oracle.vq_assign(x, C)
    dd = ((x[:, None, :] - C[None]) ** 2).sum(-1)
    assert np.array_equal(codes, dd.argmin(1))
    assert np.allclose(best, dd.min(1), rtol=1e-15, atol=0)


# ----------------------------------------------------------- packing ---

def test_pack_golden_9bit():
    f = _fixture("pack9.txt")
    for codes, expect in zip(f["codes"], f["bytes"]):
        codes = np.array(codes, np.int32)[None]
        got = oracle.pack(codes, 9)[0]
        assert list(got) == [int(b) for b in expect]
        assert list(oracle.unpack(got[None], codes.shape[1], 9)[0]) == list(codes[0])


@pytest.mark.parametrize("S,b", [(64, 8), (32, 8), (32, 9), (16, 12), (128, 1), (11, 5), (32, 2)])
def test_pack_matches_numpy_packbits(S, b):
    rng = np.random.default_rng(16)
    codes = rng.integers(0, 2 ** b, size=(9, S)).astype(np.int32)
    got = oracle.pack(codes, b)
    bits = ((codes[:, :, None] >> np.arange(b)) & 1).astype(np.uint8).reshape(9, S * b)
    ref = np.packbits(bits, axis=1, bitorder="little")
    assert got.shape[1] == (-(-S * b // 8) + 3) // 4 * 4
    assert np.array_equal(got[:, :ref.shape[1]], ref)
    assert not got[:, ref.shape[1]:].any()
    assert np.array_equal(oracle.unpack(got, S, b), codes)


def test_pack_8bit_is_bytes():
    codes = np.arange(64, dtype=np.int32)[None] * 3 % 256
    assert np.array_equal(oracle.pack(codes, 8)[0], codes[0].astype(np.uint8))


def test_storage_accounting():
    """Index bytes per vector = (d_h / d) * (b / 8) (VecInfer, 向量量化原理)."""
    assert oracle.row_bytes(128 // 4, 8) == 32      # 2 bits/element
    assert oracle.row_bytes(128 // 2, 8) == 64      # 4 bits/element
    assert oracle.row_bytes(128 // 4, 9) == 36      # 2.25 bits/element, 9-bit codes
    assert oracle.row_bytes(128 // 8, 12) == 24     # 1.5 bits/element


# --------------------------------------------------------- attention ---

def test_decode_attention_golden_d2():
    f = _fixture("attention_d2.txt")
    q = np.array(f["q"][0]).reshape(1, 2)
    lam = np.array(f["lambda"][0]).reshape(1, 2)
    Ck = np.array(f["ck"][0]).reshape(2, 2)
    Cv = np.array(f["cv"][0]).reshape(2, 2)
    kc = np.array(f["kcodes"][0], np.int32).reshape(2, 1, 1)
    vc = np.array(f["vcodes"][0], np.int32).reshape(2, 1, 1)
    out = oracle.decode_attention(q, lam, kc, Ck, vc, Cv)
    assert np.max(np.abs(out[0] - np.array(f["out"][0]))) < 1e-14


def test_attention_fp_matches_scipy_softmax():
    rng = np.random.default_rng(17)
    N, Hq, Hkv, D = 50, 4, 2, 16
    q = rng.standard_normal((Hq, D))
    k = rng.standard_normal((N, Hkv, D)) * 3
    v = rng.standard_normal((N, Hkv, D))
    out = oracle.attention_fp(q, k, v)
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        p = scipy.special.softmax(k[:, kvh] @ q[h] / np.sqrt(D))
        assert np.max(np.abs(out[h] - p @ v[:, kvh])) < 1e-13


def _exact_codebook_case(rng, N, Hq, Hkv, D, dk, dv, kk, kv):
    """Caches built from codebook rows: K = K~ H^T diag(lam), V = concat C_v rows."""
    Ck = rng.standard_normal((kk, dk)) * 2
    Cv = rng.standard_normal((kv, dv))
    kc = rng.integers(0, kk, size=(N, Hkv, D // dk)).astype(np.int32)
    vc = rng.integers(0, kv, size=(N, Hkv, D // dv)).astype(np.int32)
    lam = rng.uniform(0.5, 3.0, (Hkv, D))
    kt = Ck[kc].reshape(N, Hkv, D)
    H = scipy.linalg.hadamard(D) / np.sqrt(D)
    k = (kt @ H.T) * lam[None]
    v = Cv[vc].reshape(N, Hkv, D)
    q = rng.standard_normal((Hq, D))
    return q, k, v, lam, Ck, Cv, kc, vc


@pytest.mark.parametrize("dk,dv", [(2, 4), (4, 4), (1, 2), (8, 8)])
def test_exact_codebook_encode_and_attention(dk, dv):
    """A codebook holding every sub-vector: codes recovered exactly and quantized
    attention equals full-precision attention (spec pin)."""
    rng = np.random.default_rng(18 + dk)
    N, Hq, Hkv, D = 37, 6, 2, 128
    q, k, v, lam, Ck, Cv, kc, vc = _exact_codebook_case(rng, N, Hq, Hkv, D, dk, dv, 32, 16)
    got_kc, _, kbest, _ = oracle.encode_keys(k, lam, Ck, dk)
    got_vc, _, vbest, _ = oracle.encode_values(v, Cv, dv)
    assert np.array_equal(got_kc, kc) and np.array_equal(got_vc, vc)
    assert kbest.max() < 1e-20 and vbest.max() == 0
    out_q = oracle.decode_attention(q, lam, kc, Ck, vc, Cv)
    out_fp = oracle.attention_fp(q, k, v)
    assert np.max(np.abs(out_q - out_fp)) < 1e-12


# ---------------------------------------------------------- dequantisation ---

def test_dequantize_golden_d2():
    f = _fixture("dequant_d2.txt")
    Ck = np.array(f["ck"][0]).reshape(2, 2)
    Cv = np.array(f["cv"][0]).reshape(2, 2)
    kc = np.array(f["kcode"][0], np.int32).reshape(1, 1, 1)
    vc = np.array(f["vcode"][0], np.int32).reshape(1, 1, 1)
    lam = np.array(f["lambda"][0]).reshape(1, 2)
    k, v = oracle.dequantize_kv(kc, Ck, vc, Cv, lam)
    assert np.max(np.abs(k[0, 0] - np.array(f["k"][0]))) < 1e-15
    assert np.array_equal(v[0, 0], np.array(f["v"][0]))


@pytest.mark.parametrize("dk,dv", [(2, 4), (4, 4), (1, 2), (8, 8)])
def test_dequantize_kv_recovers_codebook_built_cache(dk, dv):
    """Caches built from codebook rows with scipy's Hadamard come back exactly."""
    rng = np.random.default_rng(40 + dk)
    _, k, v, lam, Ck, Cv, kc, vc = _exact_codebook_case(rng, 29, 4, 3, 128, dk, dv, 64, 32)
    got_k, got_v = oracle.dequantize_kv(kc, Ck, vc, Cv, lam)
    assert np.max(np.abs(got_k - k)) < 1e-12 * np.abs(k).max()
    assert np.array_equal(got_v, v)


def test_inverse_key_transform_round_trip():
    rng = np.random.default_rng(44)
    k = rng.standard_normal((40, 2, 128))
    k[:, :, 7] *= 20.0                                    # an outlier channel
    lam = oracle.smoothing_lambda(k)
    back = oracle.inverse_transform_keys(oracle.transform_keys(k, lam), lam)
    assert np.max(np.abs(back - k)) < 1e-12 * np.abs(k).max()


def test_attention_over_dequantized_cache_equals_decode_attention():
    """Dense attention of the raw query over (K^, V^) gives the quantized
    attention over the codes: q K^T = q~ VQ^-1(K~_q)^T (score rewriting)."""
    rng = np.random.default_rng(45)
    N, Hq, Hkv, D = 31, 6, 2, 128
    Ck, Cv = rng.standard_normal((64, 4)), rng.standard_normal((32, 2))
    kc = rng.integers(0, 64, (N, Hkv, D // 4)).astype(np.int32)
    vc = rng.integers(0, 32, (N, Hkv, D // 2)).astype(np.int32)
    lam = rng.uniform(0.3, 4.0, (Hkv, D))
    q = rng.standard_normal((Hq, D))
    k, v = oracle.dequantize_kv(kc, Ck, vc, Cv, lam)
    out_fp = oracle.attention_fp(q, k, v)
    out_q = oracle.decode_attention(q, lam, kc, Ck, vc, Cv)
    assert np.max(np.abs(out_fp - out_q)) < 1e-12


# ---------------------------------------------------- full-precision residual ---

def test_residual_attention_golden_d2():
    f = _fixture("attention_residual_d2.txt")
    q = np.array(f["q"][0]).reshape(1, 2)
    lam = np.array(f["lambda"][0]).reshape(1, 2)
    Ck = np.array(f["ck"][0]).reshape(2, 2)
    Cv = np.array(f["cv"][0]).reshape(2, 2)
    kc = np.array(f["kcode"][0], np.int32).reshape(1, 1, 1)
    vc = np.array(f["vcode"][0], np.int32).reshape(1, 1, 1)
    kr = np.array(f["kres"][0]).reshape(1, 1, 2)
    vr = np.array(f["vres"][0]).reshape(1, 1, 2)
    out = oracle.decode_attention_residual(q, lam, kc, Ck, vc, Cv, kr, vr)
    assert np.max(np.abs(out[0] - np.array(f["out"][0]))) < 1e-14


def test_residual_attention_reduces_to_its_parts():
    """No residual: the quantized attention; no codes: textbook attention."""
    rng = np.random.default_rng(50)
    N, R, Hq, Hkv, D = 27, 9, 6, 2, 128
    Ck, Cv = rng.standard_normal((64, 4)), rng.standard_normal((32, 2))
    kc = rng.integers(0, 64, (N, Hkv, 32)).astype(np.int32)
    vc = rng.integers(0, 32, (N, Hkv, 64)).astype(np.int32)
    lam = rng.uniform(0.3, 4.0, (Hkv, D))
    q = rng.standard_normal((Hq, D))
    kr, vr = rng.standard_normal((R, Hkv, D)) * 2, rng.standard_normal((R, Hkv, D))
    none_r = oracle.decode_attention_residual(q, lam, kc, Ck, vc, Cv, kr[:0], vr[:0])
    assert np.max(np.abs(none_r - oracle.decode_attention(q, lam, kc, Ck, vc, Cv))) < 1e-13
    none_q = oracle.decode_attention_residual(q, lam, kc[:0], Ck, vc[:0], Cv, kr, vr)
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        p = scipy.special.softmax(kr[:, kvh] @ q[h] / np.sqrt(D))
        assert np.max(np.abs(none_q[h] - p @ vr[:, kvh])) < 1e-13
    empty = oracle.decode_attention_residual(q, lam, kc[:0], Ck, vc[:0], Cv, kr[:0], vr[:0])
    assert not empty.any()


def test_residual_attention_equals_full_attention_over_the_joined_cache():
    """A cache built from codebook rows, its last R tokens given raw instead of
    as codes: the same result as full-precision attention over all tokens."""
    rng = np.random.default_rng(51)
    N, R, Hq, Hkv, D = 40, 12, 8, 2, 128
    q, k, v, lam, Ck, Cv, kc, vc = _exact_codebook_case(rng, N, Hq, Hkv, D, 4, 4, 32, 16)
    out = oracle.decode_attention_residual(q, lam, kc[:N - R], Ck, vc[:N - R], Cv, k[N - R:], v[N - R:])
    full = np.zeros((Hq, D))
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        p = scipy.special.softmax(k[:, kvh] @ q[h] / np.sqrt(D))
        full[h] = p @ v[:, kvh]
    assert np.max(np.abs(out - full)) < 1e-12


def test_attention_single_token_returns_decoded_value():
    rng = np.random.default_rng(19)
    D = 128
    Ck, Cv = rng.standard_normal((16, 2)), rng.standard_normal((8, 4))
    kc = rng.integers(0, 16, (1, 1, 64)).astype(np.int32)
    vc = rng.integers(0, 8, (1, 1, 32)).astype(np.int32)
    out = oracle.decode_attention(rng.standard_normal((3, D)), np.ones((1, D)), kc, Ck, vc, Cv)
    assert np.max(np.abs(out - Cv[vc[0, 0]].reshape(D)[None])) < 1e-15


def test_attention_equal_scores_is_mean_of_values():
    rng = np.random.default_rng(20)
    D, N = 128, 23
    Ck, Cv = rng.standard_normal((16, 2)), rng.standard_normal((8, 4))
    kc = rng.integers(0, 16, (N, 1, 64)).astype(np.int32)
    vc = rng.integers(0, 8, (N, 1, 32)).astype(np.int32)
    out = oracle.decode_attention(np.zeros((2, D)), np.ones((1, D)), kc, Ck, vc, Cv)
    assert np.max(np.abs(out - Cv[vc[:, 0]].reshape(N, D).mean(0)[None])) < 1e-14


def test_attention_single_centroid():
    rng = np.random.default_rng(21)
    D, N = 128, 40
    k = rng.standard_normal((N, 1, D)).astype(np.float16)
    v = rng.standard_normal((N, 1, D)).astype(np.float16)
    Ck, Cv = rng.standard_normal((1, 2)), rng.standard_normal((1, 4))
    kc, *_ = oracle.encode_keys(k, np.ones((1, D)), Ck, 2)
    vc, *_ = oracle.encode_values(v, Cv, 4)
    assert not kc.any() and not vc.any()
    out = oracle.decode_attention(rng.standard_normal((2, D)), np.ones((1, D)), kc, Ck, vc, Cv)
    assert np.max(np.abs(out - np.tile(Cv[0], 32)[None])) < 1e-15


def test_attention_empty_context_is_zero():
    out = oracle.decode_attention(np.ones((2, 128)), np.ones((1, 128)),
                                  np.zeros((0, 1, 64), np.int32), np.ones((4, 2)),
                                  np.zeros((0, 1, 32), np.int32), np.ones((4, 4)))
    assert not out.any()


def test_attention_scale_and_gqa_mapping():
    """Query head h reads KV head h // G; a custom scale multiplies the scores."""
    rng = np.random.default_rng(22)
    N, Hq, Hkv, D = 30, 6, 3, 128
    q, k, v, lam, Ck, Cv, kc, vc = _exact_codebook_case(rng, N, Hq, Hkv, D, 4, 4, 16, 16)
    out = oracle.decode_attention(q, lam, kc, Ck, vc, Cv, scale=0.37)
    for h in range(Hq):
        kvh = h // 2
        p = scipy.special.softmax(0.37 * (k[:, kvh] @ q[h]))
        assert np.max(np.abs(out[h] - p @ v[:, kvh])) < 1e-11


# -------------------------------------------------------------- K-means ---

def test_kmeans_objective_non_increasing():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((3000, 4))
    init = rng.choice(3000, 32, replace=False)
    C, obj = oracle.kmeans(x, init, 10)
    assert np.all(np.diff(obj) <= 1e-9 * obj[0])
    assert obj[-1] < obj[0]
    # the reported final objective is the distortion of the returned centroids
    _, best, _, _ = oracle.vq_assign(x, C)
    assert abs(best.sum() - obj[-1]) <= 1e-9 * obj[-1]


def test_kmeans_recovers_separated_blobs():
    rng = np.random.default_rng(24)
    centers = np.array([[10.0, 0], [-10, 0], [0, 10], [0, -10]])
    lab = rng.integers(0, 4, 4000)
    x = centers[lab] + 0.1 * rng.standard_normal((4000, 2))
    init = np.array([np.flatnonzero(lab == j)[0] for j in range(4)])
    C, _ = oracle.kmeans(x, init, 5)
    for j in range(4):
        assert np.max(np.abs(C[j] - x[lab == j].mean(0))) < 1e-12


def test_kmeans_empty_cluster_keeps_centroid():
    """Centroids 0 and 2 start on the same point; ties go to index 0, so after one
    iteration cluster 2 is empty and keeps its start value."""
    x = np.array([[0.0], [0.1], [10.0], [10.1]])
    C, _ = oracle.kmeans(x, np.array([0, 2, 0]), 1)
    assert C[2, 0] == 0.0
    assert abs(C[0, 0] - 0.05) < 1e-15 and abs(C[1, 0] - 10.05) < 1e-15


def test_kmeans_thread_count_independent():
    rng = np.random.default_rng(25)
    x = rng.standard_normal((20000, 2))
    init = rng.choice(20000, 64, replace=False)
    n0 = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        C1, o1 = oracle.kmeans(x, init, 4)
        oracle.set_num_threads(max(n0, 3))
        C2, o2 = oracle.kmeans(x, init, 4)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(C1, C2) and np.array_equal(o1, o2)
