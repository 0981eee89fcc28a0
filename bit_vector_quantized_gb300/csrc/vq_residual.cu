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
// One CTA of 128 threads per (sequence, KV head) serves its G query heads:
//   1. each warp takes every fourth token; a lane holds 4 elements of the key
//      and of every query head, and a shuffle reduction gives the G scores;
//   2. each warp takes query heads warp, warp + 4: the maximum, the
//      exponentials and their sum over the tokens;
//   3. thread d accumulates element d of every head's output over the tokens
//      (one coalesced 256-byte row of V per token).
// The work is a few hundred thousand FMAs per CTA at the residual length of
// 128; it runs before the split kernel and is hidden behind that kernel's
// prologue.
#include "vq_device.cuh"
#include "vq_kernels.h"

namespace vqk {
namespace {

constexpr int kResThreads = 128;
constexpr int kMaxGroup = 8;

__global__ void __launch_bounds__(kResThreads) vq_residual_kernel(const ResidualParams p) {
  extern __shared__ __align__(16) float res_smem[];  // [G][capacity] scores, then p
  __shared__ float2 ml_s[kMaxGroup];
  pdl_trigger();
  const int b = static_cast<int>(blockIdx.x) / p.hkv, kvh = static_cast<int>(blockIdx.x) % p.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  int R = __ldg(p.res_lens + b);
  R = R < 0 ? 0 : (R > p.capacity ? p.capacity : R);
  const long long head = static_cast<long long>(b) * p.hkv + kvh;
  const __half* kr = static_cast<const __half*>(p.k_res) + head * p.capacity * kHeadDim;
  const __half* vr = static_cast<const __half*>(p.v_res) + head * p.capacity * kHeadDim;
  float* s = res_smem;

  // 1. scores, log2 domain: lane holds elements 4 lane .. 4 lane + 3
  float qv[kMaxGroup][4];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    qv[g][0] = qv[g][1] = qv[g][2] = qv[g][3] = 0.f;
    if (g < G) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.q) +
                                                           (static_cast<long long>(b) * p.hq + kvh * G + g) * kHeadDim) + lane);
      const __half2 lo = *reinterpret_cast<const __half2*>(&u.x);
      const __half2 hi = *reinterpret_cast<const __half2*>(&u.y);
      qv[g][0] = __low2float(lo) * p.scale_log2;
      qv[g][1] = __high2float(lo) * p.scale_log2;
      qv[g][2] = __low2float(hi) * p.scale_log2;
      qv[g][3] = __high2float(hi) * p.scale_log2;
    }
  }
  for (int t = warp; t < R; t += kResThreads / 32) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(kr + static_cast<long long>(t) * kHeadDim) + lane);
    const __half2 lo = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&u.y);
    const float k0 = __low2float(lo), k1 = __high2float(lo), k2 = __low2float(hi), k3 = __high2float(hi);
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g >= G) break;
      float a = qv[g][0] * k0;
      a = fmaf(qv[g][1], k1, a);
      a = fmaf(qv[g][2], k2, a);
      a = fmaf(qv[g][3], k3, a);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
      if (lane == 0) s[g * p.capacity + t] = a;
    }
  }
  __syncthreads();

  // 2. per head: maximum, exponentials (in place) and their sum
  for (int g = warp; g < G; g += kResThreads / 32) {
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

  // 3. thread d: element d of every head's sum of p v
  float acc[kMaxGroup];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) acc[g] = 0.f;
  for (int t = 0; t < R; ++t) {
    const float v = __half2float(vr[static_cast<long long>(t) * kHeadDim + tid]);
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g)
      if (g < G) acc[g] = fmaf(s[g * p.capacity + t], v, acc[g]);
  }
  pdl_wait();  // the partials may be read by the previous kernel: write only after it
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g >= G) break;
    const long long row = static_cast<long long>(b) * p.hq + kvh * G + g;
    p.res_o[row * kHeadDim + tid] = acc[g];
    if (tid == 0) p.res_ml[row] = ml_s[g];
  }
}

}  // namespace

size_t residual_smem_bytes(int group, int capacity) {
  return static_cast<size_t>(group) * capacity * sizeof(float);
}

cudaError_t launch_residual(const ResidualParams& p, int grid, cudaStream_t stream) {
  const size_t smem = residual_smem_bytes(p.group, p.capacity);
  static size_t configured = 0;
  if (smem > 48 * 1024 && smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(vq_residual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaError_t e = launch_pdl(vq_residual_kernel, dim3(grid), dim3(kResThreads), smem, stream, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace vqk
