// vq_encode.cu -- K/V encode kernel (cache fill) for sm_103a.
//
// VecInfer, section 方法细节: keys are smoothed and Hadamard transformed,
// k~ = k diag(lambda)^-1 H_D ("异常值抑制的向量量化"), then keys and raw values are
// vector-quantized with the offline codebooks and the indices appended to the
// cache ("注意力机制中的向量量化KV缓存").  Nearest centroid as in section
// 背景知识 "向量量化原理": j* = argmin_j ||x_i - C_j||^2 per sub-vector.
//
// One warp owns one token-head vector (128 fp16 values, 4 per lane).  The key
// transform runs in fp32 registers: divide by lambda, 7 butterfly stages
// (2 in registers, 5 by shuffle), scale by 1/sqrt(128).  Each lane then owns
// the sub-vectors covering its 4 elements and scans the codebook, which the
// CTA keeps in shared memory as (-2 c_j, ||c_j||^2) in fp32: the score
// ||c_j||^2 - 2 x.c_j orders centroids exactly as ||x - c_j||^2 does.  The
// lanes read one or two centroids at once (shared-memory broadcasts), so the
// scan is bound by the FP32 pipe.  For d = 8 the two lanes that share a
// sub-vector each form its whole dot product and take alternate centroids;
// for d <= 4, four centroids per iteration keep several FMA chains in flight.
// Many vectors with d = 2 or 4 (a prefill) go four to a warp, sharing every
// centroid load.  With few tokens (a decode-step append) the scan of one
// vector is split over `split` warps that each take a slice of the codebook,
// and the slices are merged keeping the lowest index on ties.  A large
// codebook (the 1.5-bit format's 4096 centroids of 8) is also split over
// several CTAs per vector, each preparing and scanning its own part of the
// table; a one-warp merge kernel combines their candidates in order.
// Finally the warp packs the codes into the LSB-first bit stream of the row
// (one 32-bit word per lane) and stores it into the token's paged slot.
#include "vq_device.cuh"
#include "vq_kernels.h"

namespace vqk {
namespace {

constexpr int kEncWarps = 8;

template <int D>
struct Scan {
  static constexpr int kSub = D <= 4 ? 4 / D : 1;  // sub-vectors per lane
};

// Scans centroids [j0, j1) for the lane's sub-vectors; strict '<' keeps the
// lowest index among equal scores.
template <int D>
__device__ __forceinline__ void scan_centroids(const float (&x)[4], const float* cmul,
                                               const float* cnorm, int j0, int j1, int lane,
                                               float (&best)[4], int (&idx)[4]) {
  constexpr int NS = Scan<D>::kSub;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    best[s] = INFINITY;
    idx[s] = 0x7fffffff;
  }
  // d = 8 and d = 4: four centroids per iteration, their scores formed
  // independently (each with the same operations as one at a time), then
  // compared in index order, so the result is that of the plain loop.
  if constexpr (D == 8) {
    // Lanes 2i and 2i+1 hold elements 0..3 and 4..7 of sub-vector i.  Each
    // takes the whole sub-vector (its partner's half by shuffle) and scans
    // every other centroid, lane 2i the even ones, lane 2i+1 the odd ones; the
    // score is ||c||^2 + (lo + hi) with lo, hi the dot products of the two
    // halves, and the pair keeps the lower score (lower index on a tie).
    const int par = lane & 1;
    float xa[4], xb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], 1);
      xa[e] = par ? o : x[e];
      xb[e] = par ? x[e] : o;
    }
    auto score = [&](int j) {
      const float4 c0 = *reinterpret_cast<const float4*>(cmul + j * 8);
      const float4 c1 = *reinterpret_cast<const float4*>(cmul + j * 8 + 4);
      float lo = xa[0] * c0.x;
      lo = fmaf(xa[1], c0.y, lo);
      lo = fmaf(xa[2], c0.z, lo);
      lo = fmaf(xa[3], c0.w, lo);
      float hi = xb[0] * c1.x;
      hi = fmaf(xb[1], c1.y, hi);
      hi = fmaf(xb[2], c1.z, hi);
      hi = fmaf(xb[3], c1.w, hi);
      return cnorm[j] + (lo + hi);
    };
    int j = j0 + ((j0 & 1) != par ? 1 : 0);  // this lane's first centroid of its parity
    for (; j + 6 < j1; j += 8) {
      float sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) sc[u] = score(j + 2 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (sc[u] < best[0]) {
          best[0] = sc[u];
          idx[0] = j + 2 * u;
        }
    }
    for (; j < j1; j += 2) {
      const float sv = score(j);
      if (sv < best[0]) {
        best[0] = sv;
        idx[0] = j;
      }
    }
    const float ob = __shfl_xor_sync(0xffffffffu, best[0], 1);
    const int oi = __shfl_xor_sync(0xffffffffu, idx[0], 1);
    if (ob < best[0] || (ob == best[0] && oi < idx[0])) {
      best[0] = ob;
      idx[0] = oi;
    }
  } else if constexpr (D == 4) {
    auto score = [&](int j) {
      const float4 c = *reinterpret_cast<const float4*>(cmul + j * 4);
      float s = cnorm[j];
      s = fmaf(x[0], c.x, s);
      s = fmaf(x[1], c.y, s);
      s = fmaf(x[2], c.z, s);
      return fmaf(x[3], c.w, s);
    };
    int j = j0;
    for (; j + 4 <= j1; j += 4) {
      float sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) sc[u] = score(j + u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (sc[u] < best[0]) {
          best[0] = sc[u];
          idx[0] = j + u;
        }
    }
    for (; j < j1; ++j) {
      const float s = score(j);
      if (s < best[0]) {
        best[0] = s;
        idx[0] = j;
      }
    }
  } else if constexpr (D == 2) {
    for (int j = j0; j < j1; ++j) {
      const float2 c = *reinterpret_cast<const float2*>(cmul + j * 2);
      const float n = cnorm[j];
      const float s0 = fmaf(x[1], c.y, fmaf(x[0], c.x, n));
      const float s1 = fmaf(x[3], c.y, fmaf(x[2], c.x, n));
      if (s0 < best[0]) {
        best[0] = s0;
        idx[0] = j;
      }
      if (s1 < best[1]) {
        best[1] = s1;
        idx[1] = j;
      }
    }
  } else {  // D == 1
    for (int j = j0; j < j1; ++j) {
      const float c = cmul[j];
      const float n = cnorm[j];
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const float v = fmaf(x[s], c, n);
        if (v < best[s]) {
          best[s] = v;
          idx[s] = j;
        }
      }
    }
  }
}

// Slot of token t: from slot_mapping, or (decode-step append, no slot mapping)
// position seq_lens[t] - 1 of sequence t through its page table.  -1: nothing to
// store (padding, or an empty sequence); -2: the page-table entry is invalid.
__device__ __forceinline__ long long token_slot(const EncodeParams& p, long long t) {
  if (p.slots) return __ldg(p.slots + t);
  const int len = __ldg(p.seq_lens + t);
  if (len <= 0) return -1;
  const int pos = len - 1, pi = pos / p.page_size;
  const int page = pi < p.max_pages ? __ldg(p.page_table + t * p.max_pages + pi) : -1;
  if (page < 0 || static_cast<long long>(page) * p.page_size >= p.num_slots) return -2;
  return static_cast<long long>(page) * p.page_size + pos % p.page_size;
}

// One warp's vector: its location and the values loaded before the codebook
// barrier, so that every global load of the CTA is in flight at once.
struct VecIn {
  bool active;
  long long t;
  int h;
  uint2 raw;        // 4 fp16 elements of the lane
  float4 lam;       // smoothing factors of those elements (keys)
  long long slot;
};

__device__ __forceinline__ VecIn load_vector(const EncodeParams& p, int which) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = warp / p.split;
  const long long bx = p.slices > 1 ? blockIdx.x / p.slices : blockIdx.x;
  const long long th = bx * (kEncWarps / p.split) + group;
  VecIn in;
  in.active = th < static_cast<long long>(p.num_tokens) * p.hkv;
  in.t = in.active ? th / p.hkv : 0;
  in.h = in.active ? static_cast<int>(th % p.hkv) : 0;
  in.raw = make_uint2(0, 0);
  in.lam = make_float4(1.f, 1.f, 1.f, 1.f);
  in.slot = -1;
  if (in.active) {
    in.raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.src[which]) +
                                                  (in.t * p.hkv + in.h) * kHeadDim) +
                   lane);
    if (which == 0) in.lam = __ldg(reinterpret_cast<const float4*>(p.lambda + in.h * kHeadDim) + lane);
    in.slot = token_slot(p, in.t);
  }
  return in;
}

// Packs one vector's codes and stores the row.  Lane w assembles 32-bit word w
// of the row from the codes that overlap bits [32w, 32w + 32) of the LSB-first
// stream; idx[s] is the code of the lane's s-th sub-vector.  Every lane of the
// warp must call it (shuffles); `active` false stores nothing.
template <int D>
__device__ __forceinline__ void pack_store(const EncodeParams& p, int which, const int (&idx)[4],
                                           bool active, int h, long long slot) {
  constexpr int NS = Scan<D>::kSub;
  const int lane = threadIdx.x & 31;
  const int bits = p.bits[which];
  const int S = kHeadDim / D;
  const int row_words = p.row_bytes[which] / 4;
  pdl_wait();  // the pool may be read by the previous kernel: store only after it
  const int i_lo = (32 * lane) / bits;
  const int kmax = 32 / bits + 2;
  uint32_t word = 0;
  for (int k = 0; k < kmax; ++k) {
    const int i = i_lo + k;
    int own, reg;
    if constexpr (D == 8) {
      own = 2 * i;
      reg = 0;
    } else {
      own = i / NS;
      reg = i % NS;
    }
    own = own > 31 ? 31 : own;
    uint32_t v = 0;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const uint32_t tv = __shfl_sync(0xffffffffu, static_cast<uint32_t>(idx[s]), own);
      if (s == reg) v = tv;
    }
    if (i < S) {
      const int pos = i * bits - 32 * lane;
      if (pos < 32 && pos > -bits)
        word |= static_cast<uint32_t>((static_cast<uint64_t>(v) << (pos + 32)) >> 32);
    }
  }
  if (!active || lane >= row_words) return;
  if (slot == -2) {  // the appended token's page is out of range
    if (lane == 0) report(p.status, kDevBadPage);
    return;
  }
  if (slot < 0) return;  // padding token
  if (slot >= p.num_slots) {
    if (lane == 0) report(p.status, kDevBadSlot);
    return;
  }
  const long long page = slot / p.page_size, off = slot % p.page_size;
  uint8_t* row = p.pool[which] +
                 ((page * p.hkv + h) * p.page_size + off) * static_cast<long long>(p.row_bytes[which]);
  reinterpret_cast<uint32_t*>(row)[lane] = word;
}

template <int D>
__device__ void encode_vector(const EncodeParams& p, int which, const VecIn& in, const float* cmul,
                              const float* cnorm, float* red_best, int* red_idx, int cs0, int cs1) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = p.split;
  const int wing = warp % split;
  const bool active = in.active;
  const int h = in.h;

  float x[4];
  {
    const __half2 lo = *reinterpret_cast<const __half2*>(&in.raw.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&in.raw.y);
    x[0] = __low2float(lo);
    x[1] = __high2float(lo);
    x[2] = __low2float(hi);
    x[3] = __high2float(hi);
  }
  if (which == 0) {  // keys: smoothing then Walsh-Hadamard
    x[0] = x[0] / in.lam.x;
    x[1] = x[1] / in.lam.y;
    x[2] = x[2] / in.lam.z;
    x[3] = x[3] / in.lam.w;
    fwht128_warp(x, lane);
    const float r = 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] *= r;
  }

  // the warp's slice of the CTA's centroids [cs0, cs1)
  const int j0 = cs0 + static_cast<int>((static_cast<long long>(wing) * (cs1 - cs0)) / split);
  const int j1 = cs0 + static_cast<int>((static_cast<long long>(wing + 1) * (cs1 - cs0)) / split);
  float best[4];
  int idx[4];
  scan_centroids<D>(x, cmul, cnorm, j0, j1, lane, best, idx);

  if (split > 1) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      red_best[(warp * 32 + lane) * 4 + s] = best[s];
      red_idx[(warp * 32 + lane) * 4 + s] = idx[s];
    }
    __syncthreads();
    if (wing == 0) {
      for (int w = 1; w < split; ++w)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float b2 = red_best[((warp + w) * 32 + lane) * 4 + s];
          if (b2 < best[s]) {  // later slices hold higher indices: strict '<'
            best[s] = b2;
            idx[s] = red_idx[((warp + w) * 32 + lane) * 4 + s];
          }
        }
    }
  }
  if (wing != 0) return;
  if (p.slices > 1) {  // this CTA's candidates; the merge kernel stores the row
    if (!active) return;
    const long long v = in.t * p.hkv + h;
    int2* c = p.cand + ((v * 2 + which) * p.slices + blockIdx.x % p.slices) * 32 * 4 + lane * 4;
#pragma unroll
    for (int s = 0; s < 4; ++s) c[s] = make_int2(__float_as_int(best[s]), idx[s]);
    return;
  }
  pack_store<D>(p, which, idx, active, h, in.slot);
}

// Merge of a sliced append (slices > 1): the warp of (vector, tensor) reads the
// slices' candidates in slice order, which cover increasing index ranges, so a
// strict '<' keeps the lowest index among equal scores, then packs and stores
// the row.
__global__ void __launch_bounds__(32) vq_encode_merge_kernel(const EncodeParams p) {
  const int lane = threadIdx.x;
  const long long v = blockIdx.x;
  const int which = blockIdx.y + p.which_base;
  pdl_trigger();
  const long long t = v / p.hkv;
  const int h = static_cast<int>(v % p.hkv);
  const long long slot = token_slot(p, t);
  pdl_wait();  // the candidates are written by the previous kernel
  float best[4];
  int idx[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    best[s] = INFINITY;
    idx[s] = 0x7fffffff;
  }
  const int2* c = p.cand + (v * 2 + which) * p.slices * 32 * 4 + lane * 4;
  for (int sl = 0; sl < p.slices; ++sl) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int2 e = __ldcg(c + sl * 32 * 4 + s);
      if (__int_as_float(e.x) < best[s]) {
        best[s] = __int_as_float(e.x);
        idx[s] = e.y;
      }
    }
  }
  switch (p.sub[which]) {
    case 1: pack_store<1>(p, which, idx, true, h, slot); break;
    case 2: pack_store<2>(p, which, idx, true, h, slot); break;
    case 4: pack_store<4>(p, which, idx, true, h, slot); break;
    default: pack_store<8>(p, which, idx, true, h, slot); break;
  }
}

// Cache fill of many vectors (prefill): each warp encodes NV consecutive
// token-head vectors and reads every centroid once for all of them, so the
// shared-memory loads are amortised and the NV argmin chains run side by side.
// The score of each (vector, sub-vector, centroid) is computed exactly as in
// scan_centroids, so the codes are the same.  Sub-vector lengths 2 and 4.
template <int D, int NV>
__device__ void encode_multi(const EncodeParams& p, int which, const float* cmul, const float* cnorm) {
  static_assert(D == 2 || D == 4, "multi-vector scan");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long nvec = static_cast<long long>(p.num_tokens) * p.hkv;
  const long long base = (static_cast<long long>(blockIdx.x) * kEncWarps + warp) * NV;
  uint2 raw[NV];
  float4 lam[NV];
  bool act[NV];
  int hh[NV];
  long long slot[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {  // every global load of the warp in flight before the barrier
    const long long th = base + v;
    act[v] = th < nvec;
    const long long t = act[v] ? th / p.hkv : 0;
    hh[v] = act[v] ? static_cast<int>(th % p.hkv) : 0;
    raw[v] = make_uint2(0, 0);
    lam[v] = make_float4(1.f, 1.f, 1.f, 1.f);
    slot[v] = -1;
    if (act[v]) {
      raw[v] = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.src[which]) +
                                                    (t * p.hkv + hh[v]) * kHeadDim) + lane);
      if (which == 0) lam[v] = __ldg(reinterpret_cast<const float4*>(p.lambda + hh[v] * kHeadDim) + lane);
      slot[v] = token_slot(p, t);
    }
  }
  __syncthreads();  // the codebook table is ready
  float x[NV][4];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const __half2 lo = *reinterpret_cast<const __half2*>(&raw[v].x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&raw[v].y);
    x[v][0] = __low2float(lo);
    x[v][1] = __high2float(lo);
    x[v][2] = __low2float(hi);
    x[v][3] = __high2float(hi);
    if (which == 0) {  // keys: smoothing then Walsh-Hadamard
      x[v][0] = x[v][0] / lam[v].x;
      x[v][1] = x[v][1] / lam[v].y;
      x[v][2] = x[v][2] / lam[v].z;
      x[v][3] = x[v][3] / lam[v].w;
      fwht128_warp(x[v], lane);
      const float r = 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[v][e] *= r;
    }
  }
  float best[NV][2];
  int idx[NV][4];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    best[v][0] = best[v][1] = INFINITY;
    idx[v][0] = idx[v][1] = idx[v][2] = idx[v][3] = 0x7fffffff;
  }
  const int ncent = 1 << p.bits[which];
#pragma unroll 2
  for (int j = 0; j < ncent; ++j) {
    const float n = cnorm[j];
    if constexpr (D == 4) {
      const float4 c = *reinterpret_cast<const float4*>(cmul + j * 4);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float sc = n;
        sc = fmaf(x[v][0], c.x, sc);
        sc = fmaf(x[v][1], c.y, sc);
        sc = fmaf(x[v][2], c.z, sc);
        sc = fmaf(x[v][3], c.w, sc);
        if (sc < best[v][0]) {
          best[v][0] = sc;
          idx[v][0] = j;
        }
      }
    } else {
      const float2 c = *reinterpret_cast<const float2*>(cmul + j * 2);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float s0 = fmaf(x[v][1], c.y, fmaf(x[v][0], c.x, n));
        const float s1 = fmaf(x[v][3], c.y, fmaf(x[v][2], c.x, n));
        if (s0 < best[v][0]) {
          best[v][0] = s0;
          idx[v][0] = j;
        }
        if (s1 < best[v][1]) {
          best[v][1] = s1;
          idx[v][1] = j;
        }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) pack_store<D>(p, which, idx[v], act[v], hh[v], slot[v]);
}

// Centroid j (d fp16 elements, d in {1, 2, 4, 8}) with one load.
__device__ __forceinline__ void load_centroid(const __half* cb, int j, int d, __half (&c)[8]) {
  if (d == 8) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(cb) + j);
    memcpy(c, &u, 16);
  } else if (d == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(cb) + j);
    memcpy(c, &u, 8);
  } else if (d == 2) {
    const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(cb) + j);
    memcpy(c, &u, 4);
  } else {
    c[0] = __ldg(cb + j);
  }
}

__global__ void __launch_bounds__(kEncWarps * 32) vq_encode_kernel(const EncodeParams p) {
  extern __shared__ __align__(16) float enc_smem[];
  const int which = blockIdx.y + p.which_base;
  const int d = p.sub[which];
  const int ncent = 1 << p.bits[which];
  float* cmul = enc_smem;                 // [ncent][d]: -2 c_j
  float* cnorm = cmul + ncent * d;        // [ncent]: ||c_j||^2
  float* red_best = cnorm + ((ncent + 3) & ~3);
  int* red_idx = reinterpret_cast<int*>(red_best + kEncWarps * 32 * 4);
  pdl_trigger();
  // the vector's loads go out first, so they overlap the codebook loads below
  VecIn in{};
  if (p.vec_per_warp != kMultiVec) in = load_vector(p, which);
  // the codebook table: each thread loads four centroids (one vector load
  // each) before it uses any, so a large codebook costs a few L2 round trips
  const __half* cb = static_cast<const __half*>(p.cb[which]);
  // the CTA's centroids: all of them, or its slice of a sliced append
  const int sl = p.slices > 1 ? static_cast<int>(blockIdx.x % p.slices) : 0;
  const int cs0 = p.slices > 1 ? static_cast<int>((static_cast<long long>(sl) * ncent) / p.slices) : 0;
  const int cs1 = p.slices > 1 ? static_cast<int>((static_cast<long long>(sl + 1) * ncent) / p.slices) : ncent;
  constexpr int kPrepBatch = 4;
  for (int j0 = cs0 + static_cast<int>(threadIdx.x); j0 < cs1; j0 += kPrepBatch * blockDim.x) {
    __half c[kPrepBatch][8];
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const int j = j0 + u * static_cast<int>(blockDim.x);
      if (j < cs1) load_centroid(cb, j, d, c[u]);
    }
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const int j = j0 + u * static_cast<int>(blockDim.x);
      if (j >= cs1) break;
      float n = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e >= d) break;
        const float v = __half2float(c[u][e]);
        cmul[j * d + e] = -2.f * v;
        n = fmaf(v, v, n);
      }
      cnorm[j] = n;
    }
  }
  if (p.vec_per_warp == kMultiVec) {  // prefill: several vectors per warp (sub-vector length 2 or 4)
    if (d == 4) encode_multi<4, kMultiVec>(p, which, cmul, cnorm);
    else encode_multi<2, kMultiVec>(p, which, cmul, cnorm);
    return;
  }
  __syncthreads();
  switch (d) {
    case 1: encode_vector<1>(p, which, in, cmul, cnorm, red_best, red_idx, cs0, cs1); break;
    case 2: encode_vector<2>(p, which, in, cmul, cnorm, red_best, red_idx, cs0, cs1); break;
    case 4: encode_vector<4>(p, which, in, cmul, cnorm, red_best, red_idx, cs0, cs1); break;
    default: encode_vector<8>(p, which, in, cmul, cnorm, red_best, red_idx, cs0, cs1); break;
  }
}

}  // namespace

size_t encode_smem_bytes(int sub, int bits) {
  const size_t ncent = size_t(1) << bits;
  return (ncent * sub + ((ncent + 3) & ~size_t(3))) * 4 + size_t(kEncWarps) * 32 * 4 * 8;
}

cudaError_t launch_encode(const EncodeParams& p, int grid_x, int grid_y, size_t smem,
                          cudaStream_t stream, bool overlap) {
  static SmemOptIn opt_in;
  cudaError_t e = ensure_smem(vq_encode_kernel, smem, opt_in);
  if (e != cudaSuccess) return e;
  e = launch_pdl(vq_encode_kernel, dim3(grid_x, grid_y), dim3(kEncWarps * 32), smem, stream, p, overlap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_encode_merge(const EncodeParams& p, int vectors, int grid_y, cudaStream_t stream) {
  if (vectors == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(vq_encode_merge_kernel, dim3(vectors, grid_y), dim3(32), 0, stream, p, true);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace vqk
