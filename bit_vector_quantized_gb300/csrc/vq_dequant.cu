// vq_dequant.cu -- dequantisation of cached keys and values for sm_103a.
//
// VecInfer, section 方法细节: the cache holds codes of the transformed keys
// K~ = K diag(lambda)^-1 H_D ("Hadamard引理与注意力分数重写") and of the raw
// values; reading a vector back replaces every code by its centroid and
// concatenates the sub-vectors ("注意力机制中的向量量化KV缓存").  Since H_D is
// symmetric and orthonormal, the key in the original space is
// K^ = VQ^-1(K~_q) H_D diag(lambda).  This is the dequantisation step of an
// unfused pipeline (dequantise, then dense attention), which the VecInfer page
// compares its fused kernel against (实验结果, 图5).
//
// One warp owns one token: all its KV heads, keys and values.  Lane l produces
// elements 4l .. 4l+3 of each vector.  Heads go in groups of four: the lane
// first loads the code words of all eight vectors of the group (one
// independent load each, so the HBM latency is paid once per group, not once
// per vector), then their centroids, then for keys runs the unnormalised
// Walsh-Hadamard butterflies across the warp (2 stages in registers, 5 by
// shuffle), scales by 1/sqrt(128) and multiplies by lambda.  Every vector goes
// out as one 8-byte store per lane, 256 contiguous bytes per warp.  The kernel
// is bound by the fp16 output it writes.
#include "vq_device.cuh"
#include "vq_kernels.h"

namespace vqk {
namespace {

constexpr int kDqWarps = 8;
constexpr int kHeadGroup = 4;

// A lane's codes (at most four, at most 48 bits) sit inside the three 32-bit
// words starting at word (first bit) / 32: their bit offset in that window is
// below 32, so the last bit is below 32 + 48.  Code i of the row (bits
// [i*b, (i+1)*b) of the LSB-first stream) from the window starting at word wi.
__device__ __forceinline__ uint32_t window_code(const uint32_t (&win)[3], int wi, int i, int b) {
  const int pos = i * b - 32 * wi;  // 0 .. 75
  const uint32_t x = pos < 32 ? __funnelshift_r(win[0], win[1], pos) : __funnelshift_r(win[1], win[2], pos - 32);
  return x & ((1u << b) - 1u);
}

// Loads the centroid values of this lane's four elements of one vector.
__device__ __forceinline__ void centroids(const __half* cb, int d, const uint32_t (&c)[4], int lane,
                                          float (&x)[4]) {
  if (d == 8) {  // half of one centroid
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(cb + c[0] * 8 + 4 * (lane & 1)));
    const __half2 lo = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&u.y);
    x[0] = __low2float(lo);
    x[1] = __high2float(lo);
    x[2] = __low2float(hi);
    x[3] = __high2float(hi);
  } else if (d == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(cb + c[0] * 4));
    const __half2 lo = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&u.y);
    x[0] = __low2float(lo);
    x[1] = __high2float(lo);
    x[2] = __low2float(hi);
    x[3] = __high2float(hi);
  } else if (d == 2) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __half2 v = __ldg(reinterpret_cast<const __half2*>(cb + c[k] * 2));
      x[2 * k] = __low2float(v);
      x[2 * k + 1] = __high2float(v);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = __half2float(__ldg(cb + c[k]));
  }
}

// Unnormalised Walsh-Hadamard butterflies of one 128-vector held 4 per lane
// (element 4l + e in x[e] of lane l): 2 stages in registers, 5 by shuffle.
// Each shuffle stage is one FMA per element: the lower partner keeps x + y,
// the upper one y - x = fma(-1, x, y), both exact up to the one rounding.
__device__ __forceinline__ void butterflies(float (&x)[4], int lane) {
  const float a0 = x[0] + x[1], a1 = x[0] - x[1];
  const float a2 = x[2] + x[3], a3 = x[2] - x[3];
  x[0] = a0 + a2;
  x[2] = a0 - a2;
  x[1] = a1 + a3;
  x[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float sg = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = fmaf(sg, x[e], __shfl_xor_sync(0xffffffffu, x[e], m));
  }
}

// DK, BK, DV, BV: the formats at compile time (0: read them from the params).
template <int DK, int BK, int DV, int BV>
__global__ void __launch_bounds__(kDqWarps * 32, 4) vq_dequant_kernel(const DequantParams p) {
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>(blockIdx.x) * kDqWarps + (threadIdx.x >> 5);
  if (t >= p.num_tokens) return;  // whole warps leave together
  const long long slot = __ldg(p.slots + t);
  const bool valid = slot >= 0 && slot < p.num_slots;
  if (slot >= p.num_slots && lane == 0) report(p.status, kDevBadSlot);
  const long long page = valid ? slot / p.page_size : 0;
  const int off = valid ? static_cast<int>(slot - page * p.page_size) : 0;
  const int w0 = p.which_base, w1 = p.which_last;

  // per tensor: sub-vector length, bits, row bytes, this lane's first code
  // and code count (d <= 4: 4/d whole sub-vectors; d = 8: half of one), and
  // its window: first word and the number of words holding its codes
  int d[2], b[2], rb[2], c0[2], nc[2], wi[2], nw[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    d[w] = w ? (DV ? DV : p.v_sub) : (DK ? DK : p.k_sub);
    b[w] = w ? (BV ? BV : p.v_bits) : (BK ? BK : p.k_bits);
    rb[w] = w ? (DV ? ((kHeadDim / DV) * BV + 31) / 32 * 4 : p.v_row)
              : (DK ? ((kHeadDim / DK) * BK + 31) / 32 * 4 : p.k_row);
    nc[w] = d[w] >= 4 ? 1 : 4 / d[w];
    c0[w] = d[w] == 8 ? lane >> 1 : lane * nc[w];
    wi[w] = (c0[w] * b[w]) >> 5;
    nw[w] = (((c0[w] + nc[w]) * b[w] - 1) >> 5) - wi[w] + 1;  // 1 .. 3
  }

  for (int h0 = 0; h0 < p.hkv; h0 += kHeadGroup) {
    // 1. code words of every vector of the group, all loads in flight at once
    uint32_t win[2][kHeadGroup][3];
#pragma unroll
    for (int w = 0; w < 2; ++w)
#pragma unroll
      for (int j = 0; j < kHeadGroup; ++j) {
        const bool on = valid && w >= w0 && w <= w1 && h0 + j < p.hkv;
        const uint8_t* pool = w ? p.v_pool : p.k_pool;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(
            pool + ((page * p.hkv + h0 + j) * p.page_size + off) * rb[w]) + wi[w];
#pragma unroll
        for (int k = 0; k < 3; ++k) win[w][j][k] = (on && k < nw[w]) ? __ldg(row + k) : 0u;
      }
    // 2. centroids, 3. the key transform, 4. one 8-byte store per lane and vector
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      if (w < w0 || w > w1) continue;
      const __half* cb = static_cast<const __half*>(w ? p.cb_v : p.cb_k);
      __half* out = static_cast<__half*>(w ? p.out_v : p.out_k);
      float x[kHeadGroup][4];
#pragma unroll
      for (int j = 0; j < kHeadGroup; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[j][e] = 0.f;
        if (valid && h0 + j < p.hkv) {
          uint32_t c[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) c[k] = k < nc[w] ? window_code(win[w][j], wi[w], c0[w] + k, b[w]) : 0u;
          centroids(cb, d[w], c, lane, x[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < kHeadGroup; ++j) {
        const int h = h0 + j;
        if (h >= p.hkv) break;  // uniform over the warp
        if (w == 0) {  // K^ = K~ H_D diag(lambda)
          butterflies(x[j], lane);
          const float4 lam = __ldg(reinterpret_cast<const float4*>(p.lambda + h * kHeadDim) + lane);
          constexpr float kInvSqrtD = 0.08838834764831845f;  // 1 / sqrt(128)
          x[j][0] *= kInvSqrtD * lam.x;
          x[j][1] *= kInvSqrtD * lam.y;
          x[j][2] *= kInvSqrtD * lam.z;
          x[j][3] *= kInvSqrtD * lam.w;
        }
        const __half2 lo = __floats2half2_rn(x[j][0], x[j][1]);
        const __half2 hi = __floats2half2_rn(x[j][2], x[j][3]);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
        reinterpret_cast<uint2*>(out + (static_cast<long long>(t) * p.hkv + h) * kHeadDim)[lane] = o;
      }
    }
  }
}

}  // namespace

cudaError_t launch_dequant(const DequantParams& p, int grid_x, cudaStream_t stream) {
  // the decode formats at compile time; any other format reads them at run time
  auto kern = vq_dequant_kernel<0, 0, 0, 0>;
  const bool k8 = p.k_bits == 8 && (p.k_sub == 2 || p.k_sub == 4);
  if (k8 && p.v_sub == 4 && p.v_bits == 8)
    kern = p.k_sub == 4 ? vq_dequant_kernel<4, 8, 4, 8> : vq_dequant_kernel<2, 8, 4, 8>;
  else if (k8 && p.v_sub == 4 && p.v_bits == 9)
    kern = p.k_sub == 4 ? vq_dequant_kernel<4, 8, 4, 9> : vq_dequant_kernel<2, 8, 4, 9>;
  else if (k8 && p.v_sub == 2 && p.v_bits == 8)
    kern = p.k_sub == 4 ? vq_dequant_kernel<4, 8, 2, 8> : vq_dequant_kernel<2, 8, 2, 8>;
  kern<<<grid_x, kDqWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

int dequant_tokens_per_cta() { return kDqWarps; }

}  // namespace vqk
