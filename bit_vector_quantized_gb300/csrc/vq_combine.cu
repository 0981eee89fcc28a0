// vq_combine.cu -- merge of the split-attention partials (sm_103a).
//
// The decode attention splits each sequence across CTAs (VecInfer, section
// 方法细节 "细粒度分块计算": a (batch, heads, splits) decomposition); every split
// leaves a partial (m_s, l_s, o_s) in the log2 domain, and the merge is the
// running-max / running-sum recurrence of the online softmax (相关工作 -
// FlashAttention) applied across splits.
#include "vq_device.cuh"
#include "vq_kernels.h"

namespace vqk {
namespace {

// Merge of the split partials: o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// Each thread (one output element) loads all of its (m, l) pairs and partial
// outputs of a chunk of up to 32 splits before using any (one round trip to
// L2, bypassing L1: the partials were written by the previous kernel), then
// merges them; chunks after the first rescale the running sums.  With at most
// kC splits the sums are formed in split order from the global maximum.  With
// length-balanced units a row's pair has cnt <= splits partials (slots
// 0 .. cnt-1); the other slots are loaded with them but left out.
template <int kC, bool kCounted>
__global__ void __launch_bounds__(kHeadDim) vq_combine_kernel(const CombineParams p) {
  const int row = blockIdx.x, d = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  const float2* ml = p.ws_ml + static_cast<long long>(row) * p.splits;
  const float* o = p.ws_o + static_cast<long long>(row) * p.splits * kHeadDim + d;
  const int cnt = kCounted ? __ldcg(p.cnt + row / p.group) : p.splits;
  float M = -INFINITY, acc = 0.f, l = 0.f;
  for (int s0 = 0; s0 < p.splits; s0 += kC) {
    float2 v[kC];
    float ov[kC];
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      const int sp = s0 + i;
      v[i] = make_float2(-INFINITY, 0.f);
      ov[i] = 0.f;
      if (sp < p.splits) {
        v[i] = __ldcg(ml + sp);
        ov[i] = __ldcg(o + static_cast<long long>(sp) * kHeadDim);
      }
    }
    if constexpr (kCounted) {
#pragma unroll
      for (int i = 0; i < kC; ++i) {
        if (s0 + i >= cnt) {
          v[i] = make_float2(-INFINITY, 0.f);
          ov[i] = 0.f;
        }
      }
    }
    float Mc = M;
#pragma unroll
    for (int i = 0; i < kC; ++i) Mc = fmaxf(Mc, v[i].x);
    if (Mc == -INFINITY) continue;
    const float a = fast_exp2(M - Mc);  // 0 while nothing is accumulated yet
    acc *= a;
    l *= a;
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      const float f = fast_exp2(v[i].x - Mc);
      acc = fmaf(f, ov[i], acc);
      l = fmaf(f, v[i].y, l);
    }
    M = Mc;
  }
  const float res = l > 0.f ? acc / l : 0.f;
  static_cast<__half*>(p.out)[static_cast<long long>(row) * kHeadDim + d] = __float2half_rn(res);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool overlap) {
  if (p.rows == 0) return cudaSuccess;
  // chunk of partials loaded at once: the smallest of 4, 8, 16, 32 that holds them all
  const int terms = p.splits;
  auto kern = p.cnt ? (terms <= 4 ? vq_combine_kernel<4, true> : terms <= 8 ? vq_combine_kernel<8, true>
                       : terms <= 16 ? vq_combine_kernel<16, true> : vq_combine_kernel<32, true>)
                    : (terms <= 4 ? vq_combine_kernel<4, false> : terms <= 8 ? vq_combine_kernel<8, false>
                       : terms <= 16 ? vq_combine_kernel<16, false> : vq_combine_kernel<32, false>);
  cudaError_t e = launch_pdl(kern, dim3(p.rows), dim3(kHeadDim), 0, stream, p, overlap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace vqk
