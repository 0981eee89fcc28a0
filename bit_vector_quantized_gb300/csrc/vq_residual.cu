// vq_residual.cu -- attention partials over a full-precision residual window
// (sm_103a).
//
// VecInfer keeps the most recent tokens unquantized (实验结果 / 实验设置: a
// residual length of 128 for every method).  Their scores use the raw query
// and keys, s = q k^T * scale, and they join the quantized tokens in one
// softmax.  This kernel turns the residual tokens of each (sequence, KV head)
// into one more split partial (m, l, o) in the log2 domain of the split
// kernel (m: the maximum of s * log2(e); l = sum 2^(s log2 e - m);
// o = sum 2^(s log2 e - m) v), which the split combine merges with the others.
//
// One CTA of 256 threads (8 warps) per (sequence, KV head) serves its G query
// heads.  Every global load is issued in batches of 16 independent loads per
// thread, so a 128-token window costs about one HBM round trip per phase:
//   1. scores: warp w takes tokens w, w + 8, ...; a lane holds 4 elements of
//      the key and of every query head, and a shuffle reduction gives the G
//      scores (log2 domain) into shared memory;
//   2. per head (one warp each): the maximum, the exponentials (in place) and
//      their sum;
//   3. output: warp w accumulates, for tokens w, w + 8, ..., lane l's four
//      elements 4l .. 4l+3 of every head's sum of p v; the 8 token groups are
//      added in shared memory.
// It runs before the split kernel (programmatic dependent launch) and its
// few CTAs overlap that kernel's prologue.
#include "vq_device.cuh"
#include "vq_kernels.h"

namespace vqk {
namespace {

constexpr int kResWarps = 8;
constexpr int kResThreads = kResWarps * 32;
constexpr int kMaxGroup = 8;
constexpr int kBatch = 16;  // independent loads in flight per thread

__global__ void __launch_bounds__(kResThreads) vq_residual_kernel(const ResidualParams p) {
  // dynamic shared memory: scores / probabilities [G][capacity], then the
  // output partials of the token groups [kResWarps][G][128]
  extern __shared__ __align__(16) float res_smem[];
  __shared__ float2 ml_s[kMaxGroup];
  pdl_trigger();
  const int b = static_cast<int>(blockIdx.x) / p.hkv, kvh = static_cast<int>(blockIdx.x) % p.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  int R = __ldg(p.res_lens + b);
  R = R < 0 ? 0 : (R > p.capacity ? p.capacity : R);
  const long long head = static_cast<long long>(b) * p.hkv + kvh;
  const uint2* kr = reinterpret_cast<const uint2*>(static_cast<const __half*>(p.k_res) + head * p.capacity * kHeadDim);
  const uint2* vr = reinterpret_cast<const uint2*>(static_cast<const __half*>(p.v_res) + head * p.capacity * kHeadDim);
  float* s = res_smem;
  float* part = res_smem + ((G * p.capacity + 3) & ~3);  // 16-byte aligned for float4 stores

  auto unpack = [](uint2 u, float (&f)[4]) {
    const __half2 lo = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&u.y);
    f[0] = __low2float(lo);
    f[1] = __high2float(lo);
    f[2] = __low2float(hi);
    f[3] = __high2float(hi);
  };

  // 1. scores, log2 domain: lane holds elements 4 lane .. 4 lane + 3
  float qv[kMaxGroup][4];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    qv[g][0] = qv[g][1] = qv[g][2] = qv[g][3] = 0.f;
    if (g < G) {
      float f[4];
      unpack(__ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.q) +
                                                 (static_cast<long long>(b) * p.hq + kvh * G + g) * kHeadDim) + lane), f);
#pragma unroll
      for (int e = 0; e < 4; ++e) qv[g][e] = f[e] * p.scale_log2;
    }
  }
  for (int t0 = warp; t0 < R; t0 += kResWarps * kBatch) {
    uint2 u[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = t0 + i * kResWarps;
      u[i] = t < R ? __ldg(kr + static_cast<long long>(t) * (kHeadDim / 4) + lane) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = t0 + i * kResWarps;
      if (t >= R) break;  // uniform over the warp
      float k[4];
      unpack(u[i], k);
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g >= G) break;
        float a = qv[g][0] * k[0];
        a = fmaf(qv[g][1], k[1], a);
        a = fmaf(qv[g][2], k[2], a);
        a = fmaf(qv[g][3], k[3], a);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
        if (lane == 0) s[g * p.capacity + t] = a;
      }
    }
  }
  __syncthreads();

  // 2. per head: maximum, exponentials (in place) and their sum
  for (int g = warp; g < G; g += kResWarps) {
    float m = -INFINITY;
    for (int t = lane; t < R; t += 32) m = fmaxf(m, s[g * p.capacity + t]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int t = lane; t < R; t += 32) {
      const float e = fast_exp2(s[g * p.capacity + t] - m);
      s[g * p.capacity + t] = e;
      l += e;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) ml_s[g] = make_float2(m, l);  // R == 0: (-inf, 0)
  }
  __syncthreads();

  // 3. token group `warp`: lane's four elements of every head's sum of p v
  float acc[kMaxGroup][4];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0.f;
  for (int t0 = warp; t0 < R; t0 += kResWarps * kBatch) {
    uint2 u[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = t0 + i * kResWarps;
      u[i] = t < R ? __ldg(vr + static_cast<long long>(t) * (kHeadDim / 4) + lane) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = t0 + i * kResWarps;
      if (t >= R) break;
      float v[4];
      unpack(u[i], v);
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g >= G) break;
        const float pr = s[g * p.capacity + t];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = fmaf(pr, v[e], acc[g][e]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g >= G) break;
    reinterpret_cast<float4*>(part + (warp * G + g) * kHeadDim)[lane] =
        make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
  }
  __syncthreads();
  pdl_wait();  // the partials may be read by the previous kernel: write only after it
  for (int o = tid; o < G * kHeadDim; o += kResThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kResWarps; ++w) sum += part[w * G * kHeadDim + o];
    const int g = o / kHeadDim, d = o % kHeadDim;
    const long long row = static_cast<long long>(b) * p.hq + kvh * G + g;
    p.res_o[row * kHeadDim + d] = sum;
    if (d == 0) p.res_ml[row] = ml_s[g];
  }
}

}  // namespace

size_t residual_smem_bytes(int group, int capacity) {
  return ((static_cast<size_t>(group) * capacity + 3) / 4 * 4 +
          static_cast<size_t>(kResWarps) * group * kHeadDim) * sizeof(float);
}

cudaError_t launch_residual(const ResidualParams& p, int grid, cudaStream_t stream, bool overlap) {
  const size_t smem = residual_smem_bytes(p.group, p.capacity);
  static SmemOptIn opt_in;
  cudaError_t e = ensure_smem(vq_residual_kernel, smem, opt_in);
  if (e != cudaSuccess) return e;
  e = launch_pdl(vq_residual_kernel, dim3(grid), dim3(kResThreads), smem, stream, p, overlap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace vqk
