/*
 * vq_oracle.c -- plain, slow, fp64 CPU oracle for VQ KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant with the CUDA library, and nothing in the product path
 * calls it.
 *
 * Every function follows a definition on the VecInfer page (papercache.org
 * summary of "VecInfer: Efficient LLM Inference With Low-Bit KV Cache via
 * Outlier-Suppressed Vector Quantization"), cited per function as
 * "VecInfer, <section>".  Arithmetic is IEEE fp64 throughout, written as the
 * definitions read: dense matrix-vector products, full distance scans, a
 * single-pass softmax.  No blocking, fusion or reordering.
 *
 * Thread parallelism (OpenMP) is only ever over independent outer items
 * (vectors, heads); every reduction is summed in a fixed order, so results do
 * not depend on the thread count.  Build with -ffp-contract=off so that the
 * results are the same on every host architecture.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int vqo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void vqo_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Walsh-Hadamard matrix H_D by its recursion (VecInfer, 方法细节 /
 * "异常值抑制的向量量化"): H_1 = [1], H_{2^k} = (1/sqrt 2) [[H, H], [H, -H]].
 * Row-major D x D.  Returns -1 when D is not a power of two.
 */
int vqo_hadamard(int D, double *H) {
  if (D < 1 || (D & (D - 1))) return -1;
  H[0] = 1.0;
  const double r = 1.0 / sqrt(2.0);
  for (int n = 1; n < D; n *= 2) {
    /* build the 2n x 2n matrix in place from the n x n block in the top-left
       corner (row stride D); fill the other three blocks first, then scale */
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) {
        double h = H[(long)i * D + j];
        H[(long)i * D + j + n] = h;
        H[(long)(i + n) * D + j] = h;
        H[(long)(i + n) * D + j + n] = -h;
      }
    for (int i = 0; i < 2 * n; ++i)
      for (int j = 0; j < 2 * n; ++j) H[(long)i * D + j] *= r;
  }
  return 0;
}

/*
 * Smoothing factors (VecInfer, 方法细节 / "异常值抑制的向量量化"):
 * lambda_i = sqrt(max_t |K[t, i]|) per channel i, computed offline from the
 * calibration keys, separately for each KV head.
 * K: [T][Hkv][D], lam: [Hkv][D].
 */
void vqo_smoothing_lambda(long T, int Hkv, int D, const double *K, double *lam) {
  for (int h = 0; h < Hkv; ++h)
    for (int i = 0; i < D; ++i) {
      double m = 0.0;
      for (long t = 0; t < T; ++t) {
        double a = fabs(K[(t * Hkv + h) * D + i]);
        if (a > m) m = a;
      }
      lam[h * D + i] = sqrt(m);
    }
}

/*
 * Key transform (VecInfer, 方法细节 / "Hadamard引理与注意力分数重写"):
 * K~ = K diag(lambda)^-1 H_D, as a dense row-vector times matrix product.
 * K, Kt: [T][Hkv][D]; lam: [Hkv][D]; H: [D][D].
 */
void vqo_transform_keys(long T, int Hkv, int D, const double *K, const double *lam,
                        const double *H, double *Kt) {
#pragma omp parallel for schedule(static)
  for (long th = 0; th < T * Hkv; ++th) {
    const int h = (int)(th % Hkv);
    const double *k = K + th * D;
    double *o = Kt + th * D;
    double *x = (double *)malloc(sizeof(double) * D);
    for (int l = 0; l < D; ++l) x[l] = k[l] / lam[h * D + l];
    for (int j = 0; j < D; ++j) {
      double s = 0.0;
      for (int l = 0; l < D; ++l) s += x[l] * H[(long)l * D + j];
      o[j] = s;
    }
    free(x);
  }
}

/*
 * Query transform (same section): q~ = q diag(lambda) H_D, one query vector.
 */
void vqo_transform_query(int D, const double *q, const double *lam, const double *H,
                         double *qt) {
  for (int j = 0; j < D; ++j) {
    double s = 0.0;
    for (int l = 0; l < D; ++l) s += (q[l] * lam[l]) * H[(long)l * D + j];
    qt[j] = s;
  }
}

static double sqdist(int d, const double *x, const double *c) {
  double s = 0.0;
  for (int e = 0; e < d; ++e) {
    double t = x[e] - c[e];
    s += t * t;
  }
  return s;
}

/*
 * Nearest-centroid assignment (VecInfer, 背景知识 / "向量量化原理"):
 * j* = argmin_j ||x - C_j||^2 over all 2^b centroids, scanned in index order;
 * an exact tie keeps the lower index.  Also reports the best and runner-up
 * distances and the runner-up index, used to adjudicate near-ties.
 * X: [n][d]; C: [k][d]; outputs [n] (best/second/second_idx may be NULL).
 */
void vqo_vq_assign(long n, int d, int k, const double *X, const double *C,
                   int32_t *codes, double *best, double *second, int32_t *second_idx) {
#pragma omp parallel for schedule(static)
  for (long v = 0; v < n; ++v) {
    const double *x = X + v * d;
    double b1 = INFINITY, b2 = INFINITY;
    int32_t j1 = 0, j2 = -1;
    for (int j = 0; j < k; ++j) {
      double s = sqdist(d, x, C + (long)j * d);
      if (s < b1) {          /* new best: the old best becomes the runner-up */
        b2 = b1; j2 = (j == 0) ? -1 : j1;
        b1 = s; j1 = j;
      } else if (s < b2) {   /* includes an exact tie with the best */
        b2 = s; j2 = j;
      }
    }
    codes[v] = j1;
    if (best) best[v] = b1;
    if (second) second[v] = b2;
    if (second_idx) second_idx[v] = j2;
  }
}

/*
 * Lloyd's K-means for the offline codebooks (VecInfer, 方法细节 / "注意力机制中的
 * 向量量化KV缓存": codebooks are pre-trained with K-Means on pre-sampled
 * vectors).  Starts from the rows X[init_idx[j]]; each iteration assigns every
 * vector to its nearest centroid (lowest index on ties) and moves each centroid
 * to the mean of its members; an empty cluster keeps its previous centroid.
 * objective[it] (it = 0..iters) is the sum of squared distances of the
 * assignment made at the start of iteration it (it = iters: after the last
 * update).  Member sums are accumulated per fixed block of 4096 vectors and the
 * blocks are added in order, so the result is independent of the thread count.
 */
void vqo_kmeans(long n, int d, int k, const double *X, const int64_t *init_idx, int iters,
                double *C, double *objective) {
  const long BLK = 4096;
  const long nblk = (n + BLK - 1) / BLK;
  int32_t *a = (int32_t *)malloc(sizeof(int32_t) * n);
  double *bd = (double *)malloc(sizeof(double) * n);
  double *psum = (double *)malloc(sizeof(double) * nblk * k * d);
  long *pcnt = (long *)malloc(sizeof(long) * nblk * k);
  double *pobj = (double *)malloc(sizeof(double) * nblk);
  for (int j = 0; j < k; ++j)
    for (int e = 0; e < d; ++e) C[(long)j * d + e] = X[init_idx[j] * d + e];
  for (int it = 0; it <= iters; ++it) {
    vqo_vq_assign(n, d, k, X, C, a, bd, NULL, NULL);
#pragma omp parallel for schedule(static)
    for (long bl = 0; bl < nblk; ++bl) {
      double *s = psum + bl * k * d;
      long *c = pcnt + bl * k;
      memset(s, 0, sizeof(double) * k * d);
      memset(c, 0, sizeof(long) * k);
      double o = 0.0;
      for (long v = bl * BLK; v < n && v < (bl + 1) * BLK; ++v) {
        for (int e = 0; e < d; ++e) s[(long)a[v] * d + e] += X[v * d + e];
        c[a[v]] += 1;
        o += bd[v];
      }
      pobj[bl] = o;
    }
    double obj = 0.0;
    for (long bl = 0; bl < nblk; ++bl) obj += pobj[bl];
    objective[it] = obj;
    if (it == iters) break;
    for (int j = 0; j < k; ++j) {
      long cnt = 0;
      for (long bl = 0; bl < nblk; ++bl) cnt += pcnt[bl * k + j];
      if (cnt == 0) continue; /* empty cluster: keep the previous centroid */
      for (int e = 0; e < d; ++e) {
        double s = 0.0;
        for (long bl = 0; bl < nblk; ++bl) s += psum[(bl * k + j) * d + e];
        C[(long)j * d + e] = s / (double)cnt;
      }
    }
  }
  free(a); free(bd); free(psum); free(pcnt); free(pobj);
}

/*
 * Index packing (VecInfer, 背景知识 / "向量量化原理": each sub-vector index is
 * stored as a b-bit value and the indices of a vector form its compressed
 * representation).  Code i of a row occupies bits [i*b, (i+1)*b) of the row's
 * byte string, least significant bit first; bit m of the string is bit (m % 8)
 * of byte m / 8.  Unused trailing bits and bytes are zero.
 * codes: [n][S]; out: [n][row_bytes].  Returns -1 if the codes do not fit.
 */
int vqo_pack(long n, int S, int b, const int32_t *codes, int row_bytes, uint8_t *out) {
  if ((long)S * b > 8L * row_bytes) return -1;
  memset(out, 0, (size_t)n * row_bytes);
  for (long v = 0; v < n; ++v)
    for (int i = 0; i < S; ++i) {
      uint32_t c = (uint32_t)codes[v * S + i];
      for (int m = 0; m < b; ++m) {
        long bit = (long)i * b + m;
        if ((c >> m) & 1u) out[v * row_bytes + bit / 8] |= (uint8_t)(1u << (bit % 8));
      }
    }
  return 0;
}

void vqo_unpack(long n, int S, int b, const uint8_t *in, int row_bytes, int32_t *codes) {
  for (long v = 0; v < n; ++v)
    for (int i = 0; i < S; ++i) {
      uint32_t c = 0;
      for (int m = 0; m < b; ++m) {
        long bit = (long)i * b + m;
        c |= (uint32_t)((in[v * row_bytes + bit / 8] >> (bit % 8)) & 1u) << m;
      }
      codes[v * S + i] = (int32_t)c;
    }
}

/*
 * Dequantisation VQ^-1 (VecInfer, 背景知识 "向量量化原理" and 方法细节 /
 * "注意力机制中的向量量化KV缓存"): a vector is stored as the indices of its
 * sub-vectors' nearest centroids, and read back as the concatenation of those
 * centroids.  codes: [n][S]; C: [2^b][d]; out: [n][S * d].
 */
void vqo_dequantize(long n, int S, int d, const int32_t *codes, const double *C, double *out) {
  for (long v = 0; v < n; ++v)
    for (int i = 0; i < S; ++i) {
      const double *c = C + (long)codes[v * S + i] * d;
      for (int e = 0; e < d; ++e) out[(v * S + i) * d + e] = c[e];
    }
}

/*
 * Inverse of the key transform (VecInfer, 方法细节 / "Hadamard引理与注意力分数重写"
 * defines K~ = K diag(lambda)^-1 H_D).  H_D is symmetric and orthonormal
 * (H_D H_D = I), so K = K~ H_D diag(lambda): a dense row-vector times matrix
 * product, then a per-channel multiply.  Kt, K: [T][Hkv][D]; lam: [Hkv][D].
 */
void vqo_inverse_transform_keys(long T, int Hkv, int D, const double *Kt, const double *lam,
                                const double *H, double *K) {
#pragma omp parallel for schedule(static)
  for (long th = 0; th < T * Hkv; ++th) {
    const int h = (int)(th % Hkv);
    const double *x = Kt + th * D;
    double *o = K + th * D;
    for (int j = 0; j < D; ++j) {
      double s = 0.0;
      for (int l = 0; l < D; ++l) s += x[l] * H[(long)l * D + j];
      o[j] = s * lam[h * D + j];
    }
  }
}

/*
 * Decode attention over vector-quantized caches for one sequence (VecInfer,
 * 方法细节 / "注意力机制中的向量量化KV缓存"):
 *   s = q~ VQ^-1(K~_q, C_k)^T * scale,  p = softmax(s),  o = p VQ^-1(V_q, C_v)
 * with q~ = q diag(lambda) H_D.  VQ^-1 replaces every index by its centroid and
 * concatenates the sub-vectors.  Query head h reads KV head h / (Hq / Hkv).
 * The softmax subtracts the maximum score and normalises once at the end.
 *   q: [Hq][D]; lam: [Hkv][D]; H: [D][D]
 *   kc: [N][Hkv][D/dk]; vc: [N][Hkv][D/dv]; Ck: [2^bk][dk]; Cv: [2^bv][dv]
 *   out: [Hq][D].  N == 0 gives a zero output.
 */
void vqo_decode_attention(long N, int Hq, int Hkv, int D, const double *q, const double *lam,
                          const double *H, int dk, const int32_t *kc, const double *Ck,
                          int dv, const int32_t *vc, const double *Cv, double scale,
                          double *out) {
  const int G = Hq / Hkv, Sk = D / dk, Sv = D / dv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < Hq; ++h) {
    const int kvh = h / G;
    double *qt = (double *)malloc(sizeof(double) * D);
    double *kh = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * (N > 0 ? N : 1));
    double *o = out + (long)h * D;
    vqo_transform_query(D, q + (long)h * D, lam + (long)kvh * D, H, qt);
    double m = -INFINITY;
    for (long t = 0; t < N; ++t) {
      const int32_t *c = kc + (t * Hkv + kvh) * Sk;
      for (int i = 0; i < Sk; ++i)
        for (int e = 0; e < dk; ++e) kh[i * dk + e] = Ck[(long)c[i] * dk + e];
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += qt[j] * kh[j];
      s[t] = acc * scale;
      if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int j = 0; j < D; ++j) o[j] = 0.0;
    for (long t = 0; t < N; ++t) {
      double p = exp(s[t] - m);
      l += p;
      const int32_t *c = vc + (t * Hkv + kvh) * Sv;
      for (int i = 0; i < Sv; ++i)
        for (int e = 0; e < dv; ++e) o[i * dv + e] += p * Cv[(long)c[i] * dv + e];
    }
    if (N > 0)
      for (int j = 0; j < D; ++j) o[j] /= l;
    free(qt); free(kh); free(s);
  }
}

/*
 * Decode attention over a quantized cache plus a full-precision residual
 * (VecInfer, 实验结果 / 实验设置: every method keeps a residual of the most
 * recent tokens, 128, unquantized).  One softmax runs over the N quantized
 * tokens and the R residual tokens together:
 *   quantized token t:  s_t = q~ VQ^-1(K~_q)_t^T * scale, value VQ^-1(V_q)_t
 *                       (q~ = q diag(lambda) H_D, as vqo_decode_attention)
 *   residual token r:   s_r = q Kr_r^T * scale, value Vr_r (raw fp16 inputs)
 *   o = sum_t p_t value_t,  p = softmax over all N + R scores.
 *   kr, vr: [R][Hkv][D]; the other arguments as vqo_decode_attention.
 * N + R == 0 gives a zero output.
 */
void vqo_decode_attention_residual(long N, long R, int Hq, int Hkv, int D, const double *q,
                                   const double *lam, const double *H, int dk, const int32_t *kc,
                                   const double *Ck, int dv, const int32_t *vc, const double *Cv,
                                   const double *kr, const double *vr, double scale, double *out) {
  const int G = Hq / Hkv, Sk = D / dk, Sv = D / dv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < Hq; ++h) {
    const int kvh = h / G;
    const double *qh = q + (long)h * D;
    double *qt = (double *)malloc(sizeof(double) * D);
    double *kh = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * (N + R > 0 ? N + R : 1));
    double *o = out + (long)h * D;
    vqo_transform_query(D, qh, lam + (long)kvh * D, H, qt);
    for (long t = 0; t < N; ++t) {  /* quantized tokens: transformed query, decoded key */
      const int32_t *c = kc + (t * Hkv + kvh) * Sk;
      for (int i = 0; i < Sk; ++i)
        for (int e = 0; e < dk; ++e) kh[i * dk + e] = Ck[(long)c[i] * dk + e];
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += qt[j] * kh[j];
      s[t] = acc * scale;
    }
    for (long r = 0; r < R; ++r) {  /* residual tokens: raw query and key */
      const double *k = kr + (r * Hkv + kvh) * D;
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += qh[j] * k[j];
      s[N + r] = acc * scale;
    }
    double m = -INFINITY;
    for (long t = 0; t < N + R; ++t)
      if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int j = 0; j < D; ++j) o[j] = 0.0;
    for (long t = 0; t < N + R; ++t) {
      const double p = exp(s[t] - m);
      l += p;
      if (t < N) {
        const int32_t *c = vc + (t * Hkv + kvh) * Sv;
        for (int i = 0; i < Sv; ++i)
          for (int e = 0; e < dv; ++e) o[i * dv + e] += p * Cv[(long)c[i] * dv + e];
      } else {
        const double *v = vr + ((t - N) * Hkv + kvh) * D;
        for (int j = 0; j < D; ++j) o[j] += p * v[j];
      }
    }
    if (N + R > 0)
      for (int j = 0; j < D; ++j) o[j] /= l;
    free(qt); free(kh); free(s);
  }
}

/*
 * Full-precision decode attention (VecInfer, 背景知识 / "KV缓存与注意力机制"):
 * s = q K^T * scale, p = softmax(s), o = p V, on unquantized K and V.
 * K, V: [N][Hkv][D]; q, out: [Hq][D].
 */
void vqo_attention_fp(long N, int Hq, int Hkv, int D, const double *q, const double *K,
                      const double *V, double scale, double *out) {
  const int G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < Hq; ++h) {
    const int kvh = h / G;
    double *s = (double *)malloc(sizeof(double) * (N > 0 ? N : 1));
    double *o = out + (long)h * D;
    double m = -INFINITY;
    for (long t = 0; t < N; ++t) {
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += q[(long)h * D + j] * K[(t * Hkv + kvh) * D + j];
      s[t] = acc * scale;
      if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int j = 0; j < D; ++j) o[j] = 0.0;
    for (long t = 0; t < N; ++t) {
      double p = exp(s[t] - m);
      l += p;
      for (int j = 0; j < D; ++j) o[j] += p * V[(t * Hkv + kvh) * D + j];
    }
    if (N > 0)
      for (int j = 0; j < D; ++j) o[j] /= l;
    free(s);
  }
}
