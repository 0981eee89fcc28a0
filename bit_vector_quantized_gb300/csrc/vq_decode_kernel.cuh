// vq_decode_kernel.cuh -- split-K fused decode attention over vector-quantized
// KV codes (sm_103a).  vq_decode.cu instantiates it for fixed splits and
// vq_decode_balanced.cu for length-balanced units (two translation units,
// compiled in parallel); the split partials are merged by vq_combine.cu.
//
// What is computed (VecInfer, section 方法细节 "注意力机制中的向量量化KV缓存"):
//   q~ = q diag(lambda) H_D,  s = q~ VQ^-1(K~_q, C_k)^T * scale,
//   p = softmax(s),  o = p VQ^-1(V_q, C_v),
// one decode query per sequence, query head h reading KV head h / G.  The
// softmax is evaluated online over tiles with the running-max / running-sum
// recurrence of the FlashAttention appendix ("相关工作 - FlashAttention"); the
// sequence is split across CTAs (VecInfer, "细粒度分块计算": a (batch, heads,
// splits) decomposition) and the split partials are merged by a second kernel
// with the same recurrence.
//
// How it maps to GB300:
//   * Work unit = a run of 32-token blocks of one (sequence, KV head).  A
//     persistent grid of at most one CTA per SM walks its units.  A CTA has NW
//     consumer warps (12 for G <= 4, 8 for G > 4) and 4 producer warps, and
//     serves all G query heads of the unit's KV head, so every code byte is
//     read from HBM once.  Fixed splits (kBal false): split s of every pair
//     covers the same blocks of max_seq_len, clipped to the sequence's length,
//     and units go round-robin over the grid.  Length-balanced units (kBal,
//     batches of two or more sequences): the pairs' blocks are laid end to end
//     and each CTA takes an equal range of them (balance_units), so ragged
//     lengths and pair counts that are not a multiple of the grid leave no
//     CTA with more than its share.
//   * Pipeline stages of NW x 16 tokens (their K rows, then their V rows)
//     stream HBM -> shared memory with the TMA bulk-copy engine (cp.async.bulk,
//     completion on the stage slot's "full" mbarrier) into a ring of `nstage`
//     slots, released by the consumers through "empty" mbarriers (VecInfer,
//     "异步流水线执行": asynchronous prefetch of the next blocks).  Producer warp
//     w issues stages w, w + 4, ...: each lane copies one piece (at most 4 KB,
//     never crossing a page) after looking up its page 4 stages ahead, so
//     several warps keep enough bytes in flight.
//   * Consumer warp w takes the w-th 16-token chunk of every stage.
//     Dequantisation is a gather of fp16 centroids straight into warp-mma
//     operand registers.  Codebooks stay resident in shared memory, replicated
//     16x (8-byte centroids) or 32x (4-byte centroids); lane L reads copy L % 16
//     (L), which places every lane's gather in its own bank pair (bank): gathers
//     are free of bank conflicts whatever the codes.  The 1.5-bit format (4096
//     centroids of 8 elements) cannot be replicated and uses a half-major table.
//   * Both contractions run on the tensor pipe with m16n8k16 fp16 mma, fp32
//     accumulation.  Scores: s^T[16 tok x 8] = K^[16 tok x 128] q~^T; values:
//     o^T[128 x 8] += V^^T[128 x 16 tok] P^T[16 tok x 8].  q~ is split into
//     fp16 hi + lo parts, so the scores keep about fp32 accuracy: with G <= 4
//     the hi and lo parts occupy the otherwise empty columns 2g and 2g+1 of the
//     8-wide operand (no extra mma); with 4 < G <= 8 hi and lo take one mma
//     each.  Centroids are exact fp16 values; p (at most 2^8 with the lazy
//     running maximum) is rounded to fp16 once.
//   * The K and V feature dimensions are permuted consistently (a dot product
//     and an output row set do not depend on the order) so that each lane's
//     operand registers are exactly one centroid gather: the lane with
//     (lane % 4) = c holds dims 32c + 4k .. 32c + 4k + 3 of k-step k for K, and
//     the lane with lane / 4 = r accumulates output dims 16r .. 16r + 15 for V.
//   * Each stage's scores and the previous stage's P.V form one basic block, so
//     the two mma chains, their gathers and the softmax bookkeeping overlap.
//   * Compile-time variants of the same kernel:
//       - kAppend (the decode step in one launch): the producer warps encode
//         the new token of each (sequence, KV head) whose split the CTA owns,
//         with the encode kernel's arithmetic, while their first copies are
//         in flight, store the packed rows and fence them for the copy
//         engine; the stage holding the token is copied after that.
//       - kMethod: the pages' other score and P.V forms (a per-query lookup
//         table of q~ x C_k for the scores; P.V through per-code bins), for
//         measurement against the gather form.
//       - kResidual: every unit also merges its share of a full-precision
//         window of recent tokens (prefetched with cp.async while its stages
//         stream) into its own online softmax.
//   * Every mbarrier wait is bounded (%globaltimer); on a timeout the CTA
//     raises an abort flag, drains its copies in flight and reports
//     VQ_DEV_TIMEOUT.  Launch ordering follows pdl_wait in vq_device.cuh.
#pragma once

#include <type_traits>

#include "vq_device.cuh"
#include "vq_kernels.h"

namespace vqk {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLazyLog2 = 8.f;  // running-max slack of the online softmax (log2 units)

// The dynamic shared memory of the split kernel; the codebook table sits at
// its start (offset 0), so a gather is one load at (code << 8) | lane byte.
extern __shared__ __align__(128) uint8_t g_smem[];

__device__ __forceinline__ uint2 tab64(uint32_t off) {
  return *reinterpret_cast<const uint2*>(g_smem + off);
}
__device__ __forceinline__ uint32_t tab32(uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(g_smem + off);
}
__device__ __forceinline__ uint4 tab128(uint32_t off) {
  return *reinterpret_cast<const uint4*>(g_smem + off);
}
// Table offset of the 8-bit code in byte i of w: byte 1 of the result is the
// code (the 256-byte row), byte 0 the lane's byte inside the row (lw < 256).
__device__ __forceinline__ uint32_t row_addr(uint32_t w, uint32_t lw, int i) {
  return __byte_perm(w, lw, 0x5504 | (i << 4));
}

// The same with 128-byte table rows (one tensor per table, the table-based
// methods): (code << 7) | lane byte.
__device__ __forceinline__ uint32_t row7_addr(uint32_t w, uint32_t lw, int i) {
  return (__byte_perm(w, 0u, 0x4440 | i) << 7) | lw;
}

// K codes of one token for the lane's 8 (dk = 4) or 16 (dk = 2) sub-vectors.
template <int DK>
struct KCodes;
template <>
struct KCodes<4> {
  uint2 w;
  __device__ __forceinline__ void load(const uint8_t* row, int c) {
    w = *reinterpret_cast<const uint2*>(row + 8 * c);
  }
  __device__ __forceinline__ uint32_t off(int i, uint32_t lw) const {
    return row_addr(i < 4 ? w.x : w.y, lw, i & 3);
  }
  __device__ __forceinline__ uint32_t off7(int i, uint32_t lw) const {
    return row7_addr(i < 4 ? w.x : w.y, lw, i & 3);
  }
  __device__ __forceinline__ uint32_t code(int i) const {  // code of sub-vector 8c + i
    return __byte_perm(i < 4 ? w.x : w.y, 0u, 0x4440 | (i & 3));
  }
};
template <>
struct KCodes<2> {
  uint4 w;
  __device__ __forceinline__ void load(const uint8_t* row, int c) {
    w = *reinterpret_cast<const uint4*>(row + 16 * c);
  }
  __device__ __forceinline__ uint32_t off(int i, uint32_t lw) const {
    const uint32_t v = i < 4 ? w.x : i < 8 ? w.y : i < 12 ? w.z : w.w;
    return row_addr(v, lw, i & 3);
  }
};

// V codes of one token for the lane's sub-vectors: dv = 4 -> sub-vectors
// 4r .. 4r+3 (8- or 9-bit codes), dv = 2 -> sub-vectors 8r .. 8r+7 (8-bit).
template <int DV, int BV>
struct VCodes;
template <>
struct VCodes<4, 8> {
  uint32_t w;
  __device__ __forceinline__ void load(const uint8_t* row, int r) {
    w = *reinterpret_cast<const uint32_t*>(row + 4 * r);
  }
  __device__ __forceinline__ uint32_t off(int i, uint32_t lw) const { return row_addr(w, lw, i); }
  __device__ __forceinline__ uint32_t off7(int i, uint32_t lw) const { return row7_addr(w, lw, i); }
};
template <>
struct VCodes<4, 9> {
  uint32_t a, b;  // the lane's 36-bit code group: bits 0..31 in a, 32..35 in b
  __device__ __forceinline__ void load(const uint8_t* row, int r) {
    // codes 4r .. 4r+3 sit at bits 36r .. 36r+35: words r and r+1, shift 4r
    const uint32_t lo = *reinterpret_cast<const uint32_t*>(row + 4 * r);
    const uint32_t hi = *reinterpret_cast<const uint32_t*>(row + 4 * r + 4);
    a = __funnelshift_r(lo, hi, 4 * r);
    b = hi >> (4 * r);
  }
  __device__ __forceinline__ uint32_t off(int i, uint32_t lw) const {
    // code i = group bits 9i .. 9i+8, moved to bits 8..16 (the table row)
    const uint32_t x = i == 0 ? a << 8 : i == 1 ? a >> 1 : i == 2 ? a >> 10 : __funnelshift_r(a, b, 19);
    return (x & 0x1ff00u) | lw;
  }
};
template <>
struct VCodes<2, 8> {
  uint2 w;
  __device__ __forceinline__ void load(const uint8_t* row, int r) {
    w = *reinterpret_cast<const uint2*>(row + 8 * r);
  }
  __device__ __forceinline__ uint32_t off(int i, uint32_t lw) const {
    return row_addr(i < 4 ? w.x : w.y, lw, i & 3);
  }
};

// d = 8, 12-bit codes (the pages' 1.5-bit configuration): the table is not
// replicated (two 64 KiB tables, K at 0 and V at 64 KiB, one 16-byte row of
// fp16 elements per code).  A lane reads a whole centroid with one 16-byte
// load, which serves two k-steps (K) or two output steps (V): a quarter-warp
// phase of 8 random rows meets fewer bank conflicts than the half-warp phase
// of two 8-byte loads.
__device__ __forceinline__ uint32_t row16(uint32_t code, uint32_t lw) { return (code << 4) | lw; }
template <>
struct KCodes<8> {
  uint32_t a, b;  // the lane's 48-bit code group (sub-vectors 4c .. 4c+3), from bit 0
  __device__ __forceinline__ void load(const uint8_t* row, int c) {
    // codes 4c .. 4c+3 sit at bits 48c .. 48c+47: words w0, w0+1, shift 0 or 16
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(row);
    const int w0 = (48 * c) >> 5;
    const uint32_t lo = rw[w0], hi = rw[w0 + 1];
    const uint32_t sh = (48 * c) & 31;
    a = __funnelshift_r(lo, hi, sh);
    b = hi >> sh;
  }
  // sub-vector 4c + j (0..3): k-steps 2j (elements 0..3) and 2j + 1 (4..7)
  __device__ __forceinline__ uint32_t off16(int j, uint32_t lw) const {
    const uint32_t code = j == 0 ? (a & 0xfffu) : j == 1 ? ((a >> 12) & 0xfffu)
                        : j == 2 ? (__funnelshift_r(a, b, 24) & 0xfffu) : ((b >> 4) & 0xfffu);
    return row16(code, lw);
  }
};
template <>
struct VCodes<8, 12> {
  uint32_t x;  // the lane's 24-bit code pair (sub-vectors 2r, 2r+1), from bit 0
  __device__ __forceinline__ void load(const uint8_t* row, int r) {
    // codes 2r, 2r+1 sit at bits 24r .. 24r+23 of the 24-byte row; the next
    // word is needed only when they cross a word boundary (never for r = 7)
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(row);
    const int w0 = (24 * r) >> 5;
    const uint32_t sh = (24 * r) & 31;
    const uint32_t lo = rw[w0];
    const uint32_t hi = sh > 8 ? rw[w0 + 1] : 0u;
    x = __funnelshift_r(lo, hi, sh);
  }
  // sub-vector 2r + m (m = 0, 1): output steps 2m (elements 0..3) and 2m + 1 (4..7)
  __device__ __forceinline__ uint32_t off16(int m, uint32_t lw) const {
    return row16(m ? ((x >> 12) & 0xfffu) : (x & 0xfffu), lw);
  }
};

struct UnitId {
  int b, kvh, s;
};

// A CTA's length-balanced units (shared-memory ints): the first unit's pair
// (b * Hkv + kvh), the unit count, the first unit's partial slot and first
// 32-token block, the last unit's end block and its pair's unit count.
// Unit k is pair first + k: only the first unit can start inside its pair
// and only the last can end inside it.
enum BalanceInfo : int { kBalPair = 0, kBalUnits, kBalSlot0, kBalBlock0, kBalBlockEnd, kBalCountLast };

// Unit k of this CTA (kBal: length-balanced units, bal their range).
// Fixed splits: unit u of the grid goes to CTA u % grid and is (split,
// sequence, KV head) with the split index varying slowest, so the CTAs each
// get a mix of splits and with them an even share of the decode-step appends
// (the unit holding a sequence's last token encodes it).  Measured against
// the split-fastest order: ~5 % faster on the long-context shapes, ~3 %
// slower at batch 64 with two splits; an order chosen at run time cost more
// than either (the kernel's instruction count rose 15 %).
template <bool kBal>
__device__ __forceinline__ UnitId unit_id(const DecodeParams& p, const int* bal, int k) {
  UnitId id;
  if constexpr (kBal) {
    const int pr = bal[kBalPair] + k;
    id.b = pr / p.hkv;
    id.kvh = pr - id.b * p.hkv;
    id.s = k == 0 ? bal[kBalSlot0] : 0;
    return id;
  } else {
    const int u = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int pairs = p.batch * p.hkv;
    id.s = u / pairs;
    const int bk = u - id.s * pairs;
    id.kvh = bk % p.hkv;
    id.b = bk / p.hkv;
    return id;
  }
}

// Barrier among the NP producer warps only (id 2).
template <int NP>
__device__ __forceinline__ void producer_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(NP * 32) : "memory");
}

// Barrier among the NW consumer warps only (id 1; the producer warps run ahead).
template <int NW>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

// First 32-token block of split s: split s covers blocks
// [s q + min(s, r), (s + 1) q + min(s + 1, r)) of the max_seq_len / 32 blocks
// (q, r: their quotient and remainder by the split count).
__device__ __forceinline__ int split_first_block(const DecodeParams& p, int s) {
  return s * p.split_q + min(s, p.split_r);
}

// Pipeline stages of one work unit.  A unit covers 32-token blocks of its
// (sequence, KV head) pair, clipped to the sequence length; stage j holds its
// tokens [t0, tend) with t0 = t_begin + kStageTok j.  s is the unit's partial
// slot and cnt the number of units of its pair; t_lim is the end of its
// blocks clipped to max_seq_len only.
struct UnitStages {
  int b, kvh, s, cnt, t_begin, t_end, t_lim, count;
};

template <int kStageTok, bool kBal>
__device__ __forceinline__ UnitStages unit_stages(const DecodeParams& p, const int* bal, int k, int len) {
  UnitStages u;
  int blk0, blk1;
  if constexpr (kBal) {
    const int pr = bal[kBalPair] + k;
    u.b = pr / p.hkv;
    u.kvh = pr - u.b * p.hkv;
    const int nb = (len + kUnitTok - 1) / kUnitTok;
    const bool first = k == 0, last = k == bal[kBalUnits] - 1;
    blk0 = first ? min(bal[kBalBlock0], nb) : 0;
    blk1 = last ? min(bal[kBalBlockEnd], nb) : nb;
    u.s = first ? bal[kBalSlot0] : 0;
    u.cnt = last ? bal[kBalCountLast] : u.s + 1;
  } else {
    const UnitId id = unit_id<false>(p, bal, k);
    u.b = id.b;
    u.kvh = id.kvh;
    u.s = id.s;
    u.cnt = p.splits;
    blk0 = split_first_block(p, id.s);
    blk1 = blk0 + p.split_q + (id.s < p.split_r ? 1 : 0);
  }
  u.t_begin = blk0 * kUnitTok;
  u.t_end = min(blk1 * kUnitTok, len);
  u.t_lim = min(blk1 * kUnitTok, p.max_seq_len);
  u.count = u.t_end > u.t_begin ? (u.t_end - u.t_begin + kStageTok - 1) / kStageTok : 0;
  return u;
}

// Decode-step append inside the attention kernel: the new token of (b, kvh)
// is token raw_len - 1 (raw_len = seq_lens[b], unclamped).  The unit whose
// blocks hold that position encodes and stores it, and so does the pair's
// last unit when the position is at or past max_seq_len (stored, not
// attended).
__device__ __forceinline__ bool append_owned(const DecodeParams& p, const UnitStages& u, int raw_len) {
  if (raw_len < 1) return false;
  const int pos = raw_len - 1;
  return (pos >= u.t_begin && pos < u.t_lim) || (u.s == u.cnt - 1 && pos >= p.max_seq_len);
}

// True when the appended token is attended in unit u: a stage of the unit
// then copies its rows, which must be in the pools first.
__device__ __forceinline__ bool append_attended(const DecodeParams& p, int t_begin, int t_end, int raw_len) {
  const int pos = raw_len - 1;
  return raw_len >= 1 && raw_len <= p.max_seq_len && pos >= t_begin && pos < t_end;
}

// The CTA's length-balanced units (one warp; lens: the batch's raw lengths
// in shared memory, pre: room for batch + 1 prefix sums).  Pair (b, kvh) sits
// at position Q = pre[b] + kvh (nb_b + gap) and occupies max(nb_b, 1)
// positions from there (nb_b: its 32-token blocks); CTA c takes the pairs
// that meet [c W, (c + 1) W), W = max(ceil(total / grid), ceil(max_b nb_b /
// (splits - 1))): the second term keeps every pair within `splits` CTAs, and
// taking the batch's own longest sequence (not max_seq_len) keeps a short
// batch spread over the grid when max_seq_len is a loose bound.
__device__ __forceinline__ void balance_units(const DecodeParams& p, const int* lens, int* pre, int* bal,
                                              int lane) {
  auto blocks = [&](int b) {
    const int len = min(max(lens[b], 0), p.max_seq_len);
    return (len + kUnitTok - 1) / kUnitTok;
  };
  const int B = p.batch, per = (B + 31) / 32;
  const int b_lo = min(lane * per, B), b_hi = min(b_lo + per, B);
  int sum = 0, nb_max = 0;
  for (int b = b_lo; b < b_hi; ++b) {
    const int nb = blocks(b);
    sum += p.hkv * (nb + kBalanceGap);
    nb_max = max(nb_max, nb);
  }
  nb_max = __reduce_max_sync(kFull, nb_max);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  int run = incl - sum;
  for (int b = b_lo; b < b_hi; ++b) {
    pre[b] = run;
    run += p.hkv * (blocks(b) + kBalanceGap);
  }
  __syncwarp();
  const long long total = __shfl_sync(kFull, incl, 31);
  const long long grid = gridDim.x, c = blockIdx.x;
  const long long W = max((total + grid - 1) / grid, static_cast<long long>((nb_max + p.splits - 2) / (p.splits - 1)));
  const long long x0 = c * W, x1 = x0 + W;
  const int pairs = B * p.hkv;
  auto pos = [&](int pr) -> long long {
    const int b = pr / p.hkv;
    return pre[b] + static_cast<long long>(pr - b * p.hkv) * (blocks(b) + kBalanceGap);
  };
  auto extent = [&](int pr) { return max(blocks(pr / p.hkv), 1); };
  // the first pair in [0, pairs) for which `pred` holds (pairs: none); pred
  // is monotone.  Each round the 32 lanes probe evenly spaced pairs.
  auto first_true = [&](auto pred) {
    int lo = 0, hi = pairs;
    while (lo < hi) {
      const int step = (hi - lo + 31) / 32;
      const int i = lo + lane * step;
      const unsigned m = __ballot_sync(kFull, i >= hi || pred(i));
      if (m == 0u) {
        lo += 31 * step + 1;
      } else {
        const int f = __ffs(m) - 1;
        const int nhi = min(lo + f * step, hi);
        lo = f == 0 ? lo : lo + (f - 1) * step + 1;
        hi = nhi;
      }
    }
    return lo;
  };
  const int pa = first_true([&](int pr) { return pos(pr) + extent(pr) > x0; });
  const int pb = first_true([&](int pr) { return pos(pr) >= x1; }) - 1;
  if (lane == 0) {
    int n = pb >= pa ? pb - pa + 1 : 0;
    if (n > kMaxUnitsPerCta) {  // the host never launches such a grid
      report(p.status, kDevBadConfig);
      n = 0;
    }
    bal[kBalPair] = pa;
    bal[kBalUnits] = n;
    if (n > 0) {
      const long long qa = pos(pa), qb = pos(pb);
      bal[kBalSlot0] = static_cast<int>(c - qa / W);
      bal[kBalBlock0] = static_cast<int>(min(max(x0 - qa, 0LL), static_cast<long long>(blocks(pa / p.hkv))));
      bal[kBalBlockEnd] = static_cast<int>(min(max(x1 - qb, 0LL), static_cast<long long>(blocks(pb / p.hkv))));
      bal[kBalCountLast] = static_cast<int>((qb + extent(pb) - 1) / W - qb / W + 1);
    }
  }
}

// Packed code-row bytes of a format: (128 / d) codes of b bits, rounded up to 4 bytes.
template <int D, int B>
struct RowBytes {
  static constexpr int value = (((kHeadDim / D) * B + 7) / 8 + 3) / 4 * 4;
};

// log2 of the tokens of one bulk-copy piece: the largest 16 * 2^i that
// divides the page size with at most 4 KB of rows, so a piece never crosses
// a page.
__device__ __forceinline__ int piece_log2(int page_size, int row) {
  int t = kChunk;
  while (t * 2 <= page_size && page_size % (t * 2) == 0 && t * 2 * row <= 4096) t *= 2;
  return __ffs(t) - 1;
}

// A producer lane's piece of a stage: lanes 0..15 take the K pieces, lanes
// 16..31 the V pieces, piece i of a tensor being the i-th piece-grid cell the
// stage touches.  Its first token depends only on the stage's first token, so
// its page can be looked up before the sequence length is known.
__device__ __forceinline__ int piece_lo(int t0, int lane, int l2) {
  return max(t0, ((t0 >> l2) + (lane & 15)) << l2);
}

// ---- decode-step append inside the attention kernel ---------------------------
// Nearest centroid over [j0, j1) for the lane's sub-vectors of a 128-vector
// held 4 elements per lane (d = 4: sub-vector `lane`; d = 2: sub-vectors
// 2 lane and 2 lane + 1).  The score ||c||^2 - 2 x.c is formed as the encode
// kernel forms it (the same fused multiply-adds, in the same order, on the same
// fp32 -2 c and ||c||^2 values), and a strict '<' in index order keeps the
// lowest index among equal scores, so the codes are those of vq_encode_kv.
// cm: the fp32 -2 c table [code][D]; cn: ||c||^2 [code].
template <int D>
__device__ __forceinline__ void append_scan(const float (&x)[4], const float* cm, const float* cn,
                                            int j0, int j1, float (&best)[2], int (&idx)[2]) {
  static_assert(D == 2 || D == 4, "sub-vector length 2 or 4");
  best[0] = best[1] = INFINITY;
  idx[0] = idx[1] = 0x7fffffff;
  // the scan runs beside the streaming consumer warps, whose gathers keep the
  // shared-memory pipe busy: the loads of kU centroids go out before any use
  constexpr int kU = 8;
  auto group = [&](int j, int u_n) {
    float c[kU][D], n[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (u >= u_n) break;
      if constexpr (D == 4) {
        const float4 v = reinterpret_cast<const float4*>(cm)[j + u];
        c[u][0] = v.x; c[u][1] = v.y; c[u][2] = v.z; c[u][3] = v.w;
      } else {
        const float2 v = reinterpret_cast<const float2*>(cm)[j + u];
        c[u][0] = v.x; c[u][1] = v.y;
      }
      n[u] = cn[j + u];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (u >= u_n) break;
      if constexpr (D == 4) {
        float sc = fmaf(x[0], c[u][0], n[u]);
        sc = fmaf(x[1], c[u][1], sc);
        sc = fmaf(x[2], c[u][2], sc);
        sc = fmaf(x[3], c[u][3], sc);
        if (sc < best[0]) {
          best[0] = sc;
          idx[0] = j + u;
        }
      } else {
        const float s0 = fmaf(x[1], c[u][1], fmaf(x[0], c[u][0], n[u]));
        const float s1 = fmaf(x[3], c[u][1], fmaf(x[2], c[u][0], n[u]));
        if (s0 < best[0]) {
          best[0] = s0;
          idx[0] = j + u;
        }
        if (s1 < best[1]) {
          best[1] = s1;
          idx[1] = j + u;
        }
      }
    }
  };
  int j = j0;
  for (; j + kU <= j1; j += kU) group(j, kU);
  for (; j < j1; ++j) group(j, 1);
}

// ||c_j||^2 and -2 c_j in fp32 for the fused append's scan, as the encode
// kernel forms them: the norm a chain of fused multiply-adds in element
// order, -2 c exact.  w holds the fp16 centroid (its first D elements).
template <int D>
__device__ __forceinline__ void append_tables(uint2 w, int j, float* cn, float* cm) {
  const __half2 h01 = *reinterpret_cast<const __half2*>(&w.x);
  const __half2 h23 = *reinterpret_cast<const __half2*>(&w.y);
  const float v[4] = {__low2float(h01), __high2float(h01), D == 4 ? __low2float(h23) : 0.f,
                      D == 4 ? __high2float(h23) : 0.f};
  float n = 0.f;
#pragma unroll
  for (int e = 0; e < D; ++e) n = fmaf(v[e], v[e], n);
  cn[j] = n;
  if constexpr (D == 4)
    reinterpret_cast<float4*>(cm)[j] = make_float4(-2.f * v[0], -2.f * v[1], -2.f * v[2], -2.f * v[3]);
  else
    reinterpret_cast<float2*>(cm)[j] = make_float2(-2.f * v[0], -2.f * v[1]);
}

// Merges the warps' argmin slices of one tensor, held as (score bits, index)
// pairs [warp][lane][NS]: slices cover increasing index ranges, so a strict
// '<' in warp order keeps the lowest index among equal scores.
template <int NS>
__device__ __forceinline__ void merge_slices(const int2* scr, int nw, int lane, int (&idx)[2]) {
  float best[2] = {INFINITY, INFINITY};
  idx[0] = idx[1] = 0x7fffffff;
  for (int w = 0; w < nw; ++w)
#pragma unroll
    for (int t = 0; t < NS; ++t) {
      const int2 e = scr[(w * 32 + lane) * NS + t];
      if (__int_as_float(e.x) < best[t]) {
        best[t] = __int_as_float(e.x);
        idx[t] = e.y;
      }
    }
}

// Word `lane` of a packed code row: code i (sub-vector i, held in register
// i % NS of lane i / NS) occupies bits [i BITS, (i + 1) BITS) of the LSB-first
// stream.  Every lane of the warp must call it (shuffles).
template <int NS, int BITS>
__device__ __forceinline__ uint32_t pack_row_word(const int (&idx)[2], int lane) {
  constexpr int S = 32 * NS;  // codes in the row
  const int i_lo = (32 * lane) / BITS;
  uint32_t word = 0;
#pragma unroll
  for (int k = 0; k < 32 / BITS + 2; ++k) {
    const int i = i_lo + k;
    const int own = min(i / NS, 31);
    uint32_t v = __shfl_sync(kFull, static_cast<uint32_t>(idx[0]), own);
    if constexpr (NS == 2) {
      const uint32_t v1 = __shfl_sync(kFull, static_cast<uint32_t>(idx[1]), own);
      v = (i & 1) ? v1 : v;
    }
    const int pos = i * BITS - 32 * lane;
    if (i < S && pos < 32 && pos > -BITS)
      word |= static_cast<uint32_t>((static_cast<uint64_t>(v) << (pos + 32)) >> 32);
  }
  return word;
}

template <int DK, int BK, int DV, int BV, int NG, int NW, bool kAppend, int kMethod, bool kResidual, bool kBal>
__global__ void __launch_bounds__((NW + kProducerWarps) * 32, 1) vq_decode_split_kernel(const DecodeParams p) {
  static_assert(BK == 8 || (DK == 8 && BK == 12 && DV == 8 && BV == 12),
                "K codes are byte-aligned, or the 1.5-bit format (d = 8, 12-bit codes)");
  constexpr bool kWide = DK == 8;            // 1.5-bit format: 32-byte table rows, no replicas
  static_assert(NG == 4 || NG == 8, "query heads per pass");
  constexpr int NGL = NG == 4 ? 1 : 2;       // heads owned by one lane
  constexpr int NP = kProducerWarps;
  constexpr int kStageTok = NW * kChunk;     // tokens per pipeline stage (one chunk per consumer warp)
  constexpr int KROW = RowBytes<DK, BK>::value, VROW = RowBytes<DV, BV>::value;
  constexpr int kStageBytes = kStageTok * (KROW + VROW);
  constexpr int kConsumerThreads = NW * 32;
  uint8_t* const smem = g_smem;
  const int G = p.group;
  const int NS = p.nstage;
  static_assert(kMethod == kMethodGather ||
                    (DK == 4 && BK == 8 && DV == 4 && BV == 8 && NG == 4 && NW == 12 && !kAppend),
                "the table-based methods are built for d = 4, 8-bit codes, G <= 4");
  constexpr bool kLut = kMethod == kMethodLut, kBins = kMethod == kMethodBins;
  static_assert(!kResidual || (kMethod == kMethodGather && !kAppend), "the residual window runs alone");
  const DecodeSmem L = decode_smem(BK, BV, G, KROW, VROW, NS, NW, kStageTok,
                                   kAppend && !kWide ? append_enc_bytes(BK, BV, DK, DV) : 0, kMethod,
                                   kResidual ? p.res_tok : 0);
  float* qt = reinterpret_cast<float*>(smem + L.qt);
  // the LUT method's merge buffer shares the LUT (built again for every unit)
  float* merge = reinterpret_cast<float*>(smem + (kLut ? L.aux : L.merge));
  float2* mlbuf = reinterpret_cast<float2*>(smem + L.ml);
  int* ulen_c = reinterpret_cast<int*>(smem + L.units);  // unit lengths, consumers' copy
  int* ulen_p = ulen_c + kMaxUnitsPerCta;                  // producers' copy
  int* ures_c = ulen_p + kMaxUnitsPerCta;                  // residual window lengths (kResidual)
  int4* meta = reinterpret_cast<int4*>(smem + L.meta);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* empty = full + NS;
  float* const enc_kn = reinterpret_cast<float*>(smem + L.enc);  // fused append: ||c||^2 tables
  float* const enc_vn = enc_kn + (1 << BK);
  float* const enc_km = enc_vn + (1 << BV);                          // -2 c tables (fp32)
  float* const enc_vm = enc_km + (1 << BK) * DK;
  int2* const enc_scr = reinterpret_cast<int2*>(enc_vm + (1 << BV) * DV);  // [NP][32][4] argmin scratch
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flag);
  int* const bal = reinterpret_cast<int*>(smem + L.flag) + 4;  // length-balanced range (BalanceInfo)
  uint8_t* stages = smem + L.stage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  // units of this CTA (length-balanced: known once the batch's lengths are in)
  int n_units = kBal ? 0
                           : (p.num_units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                 static_cast<int>(gridDim.x);
  auto clamp_len = [&](int len) { return len < 0 ? 0 : (len > p.max_seq_len ? p.max_seq_len : len); };
  // the slot hand-off needs NS >= NP; the rows must be the format's (the host never launches otherwise)
  if (NS < NP || NS > kMaxStages || p.k_row != KROW || p.v_row != VROW) {
    pdl_wait();
    if (tid == 0) report(p.status, kDevBadConfig);
    return;
  }

  // ---- every global load of the prologue goes out first -----------------------
  // The loads of one round trip: codebooks, the first unit's query and lambda,
  // the units' sequence lengths and the first page of each producer lane's
  // first piece.  Only inputs of the call are read here (none of them is
  // written by the previous kernel of the call).
  constexpr int kNK = kWide ? 1 : ((1 << BK) + kConsumerThreads - 1) / kConsumerThreads;
  constexpr int kNV = kWide ? 1 : ((1 << BV) + kConsumerThreads - 1) / kConsumerThreads;
  constexpr int kNB = kNK > kNV ? kNK : kNV;
  uint2 cbk_r[kNB], cbv_r[kNB];  // centroid tid + i * kConsumerThreads (i < kNK, kNV)
  uint2 q_r = make_uint2(0, 0);
  float4 lam_r = make_float4(0.f, 0.f, 0.f, 0.f);
  int len_r[2] = {0, 0};
  int page_r = -1, lk = 0, lv = 0;
  auto load_q = [&](int k) {  // query and lambda of unit k (consumer warps < G)
    if (warp < G && k < n_units) {
      const UnitId id = unit_id<kBal>(p, bal, k);
      q_r = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.q) +
                                               (static_cast<long long>(id.b) * p.hq + id.kvh * G + warp) * kHeadDim) +
                  lane);
      lam_r = __ldg(reinterpret_cast<const float4*>(p.lambda + id.kvh * kHeadDim) + lane);
    }
  };
  if (warp < NW) {
#pragma unroll
    for (int i = 0; i < kNK; ++i) {
      const int j = tid + i * kConsumerThreads;
      if (!kWide && j < (1 << BK)) {
        if constexpr (DK == 4) cbk_r[i] = __ldg(reinterpret_cast<const uint2*>(p.cb_k) + j);
        else cbk_r[i].x = __ldg(reinterpret_cast<const uint32_t*>(p.cb_k) + j);
      }
    }
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int j = tid + i * kConsumerThreads;
      if (!kWide && j < (1 << BV)) {
        if constexpr (DV == 4) cbv_r[i] = __ldg(reinterpret_cast<const uint2*>(p.cb_v) + j);
        else cbv_r[i].x = __ldg(reinterpret_cast<const uint32_t*>(p.cb_v) + j);
      }
    }
    if (tid < n_units) {
      const int b = unit_id<kBal>(p, bal, tid).b;
      len_r[0] = __ldg(p.seq_lens + b);
      if constexpr (kResidual) len_r[1] = __ldg(p.res_lens + b);
    }
    load_q(0);
  } else {
    const int ptid = tid - NW * 32, pw = warp - NW;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int k = ptid + i * NP * 32;
      if (k < n_units) len_r[i] = __ldg(p.seq_lens + unit_id<kBal>(p, bal, k).b);
    }
    lk = piece_log2(p.page_size, KROW);
    lv = piece_log2(p.page_size, VROW);
    if (n_units > 0) {  // this lane's piece of stage pw of the first unit, at full length
      const UnitId id = unit_id<kBal>(p, bal, 0);
      const int t0 = split_first_block(p, id.s) * kUnitTok + pw * kStageTok;
      const int pi = piece_lo(t0, lane, lane < 16 ? lk : lv) / p.page_size;
      if (pi < p.max_pages) page_r = __ldg(p.page_table + static_cast<long long>(id.b) * p.max_pages + pi);
    }
  }
  if constexpr (kBal) {  // the batch's lengths, in the pipeline slots (no copy has been issued yet)
    int* lens = reinterpret_cast<int*>(stages);
    for (int b = tid; b < p.batch; b += blockDim.x) {
      lens[b] = __ldg(p.seq_lens + b);
      if constexpr (kResidual) lens[p.batch + b] = __ldg(p.res_lens + b);
    }
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, NW);
    }
    mbar_init_fence();
    *abort_flag = 0;
  }
  __syncthreads();  // barriers initialised; producers and consumers now run independently
  if constexpr (kBal) {
    // Length-balanced units: one warp finds this CTA's range, then every
    // thread takes its units' lengths as the fixed-split prologue does.
    const int* lens = reinterpret_cast<const int*>(stages);
    if (warp == 0) balance_units(p, lens, reinterpret_cast<int*>(stages) + 2 * p.batch, bal, lane);
    __syncthreads();
    n_units = bal[kBalUnits];
    const int pa = bal[kBalPair];
    if (warp < NW) {
      if (tid < n_units) {
        const int b = (pa + tid) / p.hkv;
        len_r[0] = lens[b];
        if constexpr (kResidual) len_r[1] = lens[p.batch + b];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = tid - NW * 32 + i * NP * 32;
        if (k < n_units) len_r[i] = lens[(pa + k) / p.hkv];
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before the copies reuse the slots
    __syncthreads();
    load_q(0);
  }

  if (warp >= NW) {
    // =========================== producer warps ==============================
    // Producer warp pw = warp - NW owns stages n = pw, pw + NP, pw + 2 NP, ...
    // (numbered over the CTA's units); stage n goes to slot n % NS.  Lane i
    // copies piece i & 15 of the K (i < 16) or V (i >= 16) rows as one bulk
    // copy after lane 0 has armed the slot's full barrier with the byte count.
    // A warp issuing bulk copies stalls while the copy engine accepts them, so
    // several producer warps together keep enough bytes in flight to reach
    // HBM bandwidth.  The page of a lane's next piece is looked up right after
    // its current issue, so the lookup overlaps the wait for the next slot.
    const int pw = warp - NW, ptid = tid - NW * 32;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int k = ptid + i * NP * 32;
      if (k < n_units) ulen_p[k] = len_r[i];  // raw: the append needs the unclamped length
    }
    producer_sync<NP>();
    const int P = p.page_size;
    const int l2 = lane < 16 ? lk : lv;
    const int row = lane < 16 ? KROW : VROW;
    struct It {  // stage iterator over (unit k, stage j), skipping empty units
      int k, j;
      UnitStages u;
    };
    auto it_seek = [&](It& it) {
      while (it.k < n_units && it.j >= it.u.count) {
        ++it.k;
        it.j = 0;
        if (it.k < n_units) it.u = unit_stages<kStageTok, kBal>(p, bal, it.k, clamp_len(ulen_p[it.k]));
      }
    };
    auto skip = [&](It& it) {  // advance by NP stages
#pragma unroll 1
      for (int i = 0; i < NP && it.k < n_units; ++i) {
        ++it.j;
        it_seek(it);
      }
    };
    auto lookup = [&](const It& it) -> int {  // page of this lane's piece of stage `it`
      if (it.k >= n_units) return -1;
      const int pi = piece_lo(it.u.t_begin + it.j * kStageTok, lane, l2) / P;
      return pi < p.max_pages ? __ldg(p.page_table + static_cast<long long>(it.u.b) * p.max_pages + pi) : -1;
    };
    auto issue = [&](const UnitStages& su, int sj, int page, int n) {
      const int slot = n % NS;
      const int t0 = su.t_begin + sj * kStageTok;
      const int tend = min(t0 + kStageTok, su.t_end);
      const int tend16 = (tend + kChunk - 1) & ~(kChunk - 1);
      const int t_lo = piece_lo(t0, lane, l2);
      const int t_hi = min(tend16, ((t0 >> l2) + (lane & 15) + 1) << l2);
      const bool has = t_lo < t_hi;
      const bool ok = has && page >= 0 && page < p.num_pages;
      if (has && !ok) report(p.status, kDevBadPage);
      const uint32_t bytes = ok ? static_cast<uint32_t>(t_hi - t_lo) * row : 0u;
      uint32_t mask = 0;  // 16-token chunks with data (from the K pieces)
      if (ok && lane < 16) {
        const int c0 = (t_lo - t0) / kChunk, c1 = (t_hi - t0) / kChunk;
        mask = ((1u << c1) - 1u) & ~((1u << c0) - 1u);
      }
      const uint32_t total = __reduce_add_sync(kFull, bytes);
      const uint32_t vmask = __reduce_or_sync(kFull, mask);
      if (lane == 0) {
        meta[slot] = make_int4(t0, tend, static_cast<int>(vmask), 0);
        if (total) mbar_arrive_expect_tx(full + slot, total);
        else mbar_arrive(full + slot);
      }
      __syncwarp();
      if (ok) {
        uint8_t* dst = stages + static_cast<size_t>(slot) * kStageBytes +
                       (lane < 16 ? 0 : kStageTok * KROW) + (t_lo - t0) * row;
        const uint8_t* pool = lane < 16 ? p.k_pool : p.v_pool;
        const long long row0 = (static_cast<long long>(page) * p.hkv + su.kvh) * P + (t_lo % P);
        bulk_copy_g2s(dst, pool + row0 * row, (t_hi - t_lo) * row, full + slot);
      }
    };
    It cur;
    cur.k = 0;
    cur.j = 0;
    if (n_units > 0) cur.u = unit_stages<kStageTok, kBal>(p, bal, 0, clamp_len(ulen_p[0]));
    it_seek(cur);
#pragma unroll 1
    for (int i = 0; i < pw && cur.k < n_units; ++i) {
      ++cur.j;
      it_seek(cur);
    }
    // Fused append: the producer warps encode the new token of every unit
    // the CTA owns one for (append_owned), once the first ring of stages is
    // on its way (or before the stage holding such a token, whichever comes
    // first).  Each warp scans a slice of each codebook with the encode
    // kernel's score arithmetic; warps 0 and 1 merge the slices in index order
    // (lowest index on ties), pack the K and V rows and store them into the
    // pools through the page table, fencing the stores for the copy engine.
    // The stage holding an attended new token is issued only after this.
    // The 1.5-bit format's codebooks are too large to scan here: the encode
    // kernel launched before this one scans each new vector over several CTAs
    // and leaves their candidates (app_cand); warps 0 and 1 merge them in
    // slice order (lowest index on ties), then pack and store the rows.
    auto encode_phase = [&]() {
      if constexpr (kAppend && kWide) {
        asm volatile("bar.sync 4, %0;" ::"n"((NW + NP) * 32) : "memory");
        for (int k = 0; k < n_units && pw < 2; ++k) {
          const int raw = ulen_p[k];
          const UnitStages id = unit_stages<kStageTok, kBal>(p, bal, k, clamp_len(raw));
          if (!append_owned(p, id, raw)) continue;
          const int pos = raw - 1;
          const int pi = pos / P;
          const int pg = pi < p.max_pages ? __ldg(p.page_table + static_cast<long long>(id.b) * p.max_pages + pi) : -1;
          // lane i < 16 takes sub-vector i, whose candidate the encode kernel's lane 2i holds
          const long long v = static_cast<long long>(id.b) * p.hkv + id.kvh;
          int idx[2] = {0, 0};
          if (lane < 16) {
            const int2* cand = p.app_cand + (v * 2 + pw) * p.app_slices * 32 * 4 + (2 * lane) * 4;
            float best = INFINITY;
            int bi = 0x7fffffff;
            for (int sl = 0; sl < p.app_slices; ++sl) {
              const int2 e = __ldcg(cand + sl * 32 * 4);
              if (__int_as_float(e.x) < best) {
                best = __int_as_float(e.x);
                bi = e.y;
              }
            }
            idx[0] = bi;
          }
          const uint32_t word = pack_row_word<1, BK>(idx, lane);  // codes 16 .. 31 fall past the row
          const int rb = pw == 0 ? KROW : VROW;
          const bool okp = pg >= 0 && pg < p.num_pages;
          if (!okp && lane == 0 && pw == 0) report(p.status, kDevBadPage);
          if (okp && lane < rb / 4) {
            uint8_t* pool = pw == 0 ? p.k_pool_w : p.v_pool_w;
            const long long r0 = (static_cast<long long>(pg) * p.hkv + id.kvh) * P + pos % P;
            reinterpret_cast<uint32_t*>(pool + r0 * rb)[lane] = word;
            fence_proxy_async_global();
          }
        }
        producer_sync<NP>();  // every new row is stored and fenced before its stage is copied
      } else if constexpr (kAppend) {
        asm volatile("bar.sync 4, %0;" ::"n"((NW + NP) * 32) : "memory");  // the consumers' table and norms
        constexpr int NSK = DK == 2 ? 2 : 1, NSV = DV == 2 ? 2 : 1;
        for (int k = 0; k < n_units; ++k) {
          const int raw = ulen_p[k];
          const UnitStages id = unit_stages<kStageTok, kBal>(p, bal, k, clamp_len(raw));
          if (!append_owned(p, id, raw)) continue;
          const int pos = raw - 1;
          const long long vrow = (static_cast<long long>(id.b) * p.hkv + id.kvh) * kHeadDim;
          const uint2 rk = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.k_new) + vrow) + lane);
          const uint2 rv = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.v_new) + vrow) + lane);
          const float4 lam = __ldg(reinterpret_cast<const float4*>(p.lambda + id.kvh * kHeadDim) + lane);
          const int pi = pos / P;
          const int pg = pi < p.max_pages ? __ldg(p.page_table + static_cast<long long>(id.b) * p.max_pages + pi) : -1;
          float xk[4], xv[4];
          {
            const __half2 k01 = *reinterpret_cast<const __half2*>(&rk.x), k23 = *reinterpret_cast<const __half2*>(&rk.y);
            const __half2 v01 = *reinterpret_cast<const __half2*>(&rv.x), v23 = *reinterpret_cast<const __half2*>(&rv.y);
            xk[0] = __low2float(k01) / lam.x;  // keys: smoothing, Walsh-Hadamard, 1/sqrt(128)
            xk[1] = __high2float(k01) / lam.y;
            xk[2] = __low2float(k23) / lam.z;
            xk[3] = __high2float(k23) / lam.w;
            xv[0] = __low2float(v01);
            xv[1] = __high2float(v01);
            xv[2] = __low2float(v23);
            xv[3] = __high2float(v23);
          }
          fwht128_warp(xk, lane);
          const float rs = 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
          for (int e = 0; e < 4; ++e) xk[e] *= rs;
          float bk[2], bv[2];
          int ik[2], iv[2];
          append_scan<DK>(xk, enc_km, enc_kn, (pw << BK) / NP, ((pw + 1) << BK) / NP, bk, ik);
          append_scan<DV>(xv, enc_vm, enc_vn, (pw << BV) / NP, ((pw + 1) << BV) / NP, bv, iv);
          producer_sync<NP>();  // the previous token's scratch has been read
          int2* scr_k = enc_scr;
          int2* scr_v = enc_scr + NP * 32 * NSK;
#pragma unroll
          for (int t = 0; t < NSK; ++t) scr_k[(pw * 32 + lane) * NSK + t] = make_int2(__float_as_int(bk[t]), ik[t]);
#pragma unroll
          for (int t = 0; t < NSV; ++t) scr_v[(pw * 32 + lane) * NSV + t] = make_int2(__float_as_int(bv[t]), iv[t]);
          producer_sync<NP>();
          if (pw < 2) {  // warp 0 merges and stores K, warp 1 V
            int idx[2];
            if (pw == 0) merge_slices<NSK>(scr_k, NP, lane, idx);
            else merge_slices<NSV>(scr_v, NP, lane, idx);
            const uint32_t word = pw == 0 ? pack_row_word<NSK, BK>(idx, lane) : pack_row_word<NSV, BV>(idx, lane);
            const int rb = pw == 0 ? KROW : VROW;
            const bool okp = pg >= 0 && pg < p.num_pages;
            if (!okp && lane == 0 && pw == 0) report(p.status, kDevBadPage);
            if (okp && lane < rb / 4) {
              uint8_t* pool = pw == 0 ? p.k_pool_w : p.v_pool_w;
              const long long r0 = (static_cast<long long>(pg) * p.hkv + id.kvh) * P + pos % P;
              reinterpret_cast<uint32_t*>(pool + r0 * rb)[lane] = word;
              fence_proxy_async_global();
            }
          }
        }
        producer_sync<NP>();  // every new row is stored and fenced before its stage is copied
      }
    };
    // the page looked up at entry is this stage's unless the first unit was too short
    int page = (!kBal && cur.k == 0 && cur.j == pw) ? page_r : lookup(cur);
    pdl_wait();  // the pools may be written by the previous kernel: copy only after it
    int n = pw;
    bool stop = false, encoded = !kAppend;
    while (cur.k < n_units) {
      if constexpr (kAppend) {
        if (!encoded) {  // before the first slot wait, or before a stage holding a new token
          const int t0 = cur.u.t_begin + cur.j * kStageTok;
          if (n >= NS || append_attended(p, t0, min(t0 + kStageTok, cur.u.t_end), ulen_p[cur.k])) {
            encode_phase();
            encoded = true;
          }
        }
      }
      const int slot = n % NS;
      if (n >= NS) {  // wait until the consumers have released the slot
        const uint32_t par = static_cast<uint32_t>(n / NS - 1) & 1u;
        bool ok = mbar_try_wait(empty + slot, par);
        if (!__all_sync(kFull, ok)) {
          ok = !*abort_flag && mbar_wait_bounded(empty + slot, par, abort_flag, p.timeout_ns);
          if (!__all_sync(kFull, ok)) {
            if (lane == 0 && !*abort_flag) {
              *abort_flag = 1;
              report(p.status, kDevTimeout);
            }
            stop = true;
            break;
          }
        }
      }
      issue(cur.u, cur.j, page, n);
      skip(cur);
      page = lookup(cur);
      n += NP;
    }
    if (!encoded) encode_phase();  // every producer warp takes part once
    __syncthreads();  // every consumer is done
    if (stop && lane == 0) {  // wait (bounded) for this warp's copies still in flight
      for (int i = n - NP; i >= 0 && i >= n - NS - NP; i -= NP) {
        volatile int no_abort = 0;
        mbar_wait_bounded(full + i % NS, static_cast<uint32_t>(i / NS) & 1u, &no_abort,
                          p.timeout_ns);
      }
    }
    return;
  }

  // ============================= consumer warps ==============================
  // Codebook table: row j = 16 copies of 8-byte (32 copies of 4-byte) K
  // centroid j, then the same for V centroid j; the 1.5-bit format's tables
  // are the codebooks as they are (K at 0, V at 64 KiB, see row16).
  if constexpr (kWide) {
    const uint32_t tab = smem_addr(smem + L.tab);
    constexpr int kBatch = 4;  // loads in flight per thread
    for (int j0 = tid; j0 < (1 << BK); j0 += kBatch * kConsumerThreads) {
      uint4 kv[kBatch][2];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i * kConsumerThreads;
        if (j < (1 << BK)) {
          kv[i][0] = __ldg(reinterpret_cast<const uint4*>(p.cb_k) + j);
          kv[i][1] = __ldg(reinterpret_cast<const uint4*>(p.cb_v) + j);
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i * kConsumerThreads;
        if (j < (1 << BK)) {
#pragma unroll
          for (int t = 0; t < 2; ++t)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(tab + t * 65536u + j * 16u),
                         "r"(kv[i][t].x), "r"(kv[i][t].y), "r"(kv[i][t].z), "r"(kv[i][t].w));
        }
      }
    }
  } else {
    // Warp w holds centroids 32 b + lane of blocks b = w, w + NW, ... (loaded
    // at entry).  One store instruction fills 128 contiguous bytes of one or
    // two rows, so no two lanes share a bank: the replicas of centroid row i
    // reach the lanes by shuffle.
    const uint32_t tab = smem_addr(smem + L.tab);
    constexpr int kRow = kMethod == kMethodGather ? kTabRow : kTabRow / 2;
    auto fill = [&](const uint2 (&cb)[kNB], int n_i, int rows, int d, uint32_t half) {
#pragma unroll
      for (int i = 0; i < kNB; ++i) {
        const int block = warp + i * NW;
        if (i >= n_i || block * 32 >= rows) break;
        if (d == 4) {  // two rows per store: lanes 0..15 row 2 t, lanes 16..31 row 2 t + 1
#pragma unroll 4
          for (int t = 0; t < 16; ++t) {
            const int src = 2 * t + (lane >> 4);
            const uint32_t x = __shfl_sync(kFull, cb[i].x, src), y = __shfl_sync(kFull, cb[i].y, src);
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(tab + (block * 32 + src) * kRow + half +
                                                                  (lane & 15) * 8),
                         "r"(x), "r"(y));
          }
        } else {       // one row per store: lane l writes replica l
#pragma unroll 4
          for (int t = 0; t < 32; ++t) {
            const uint32_t x = __shfl_sync(kFull, cb[i].x, t);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(tab + (block * 32 + t) * kRow + half + lane * 4),
                         "r"(x));
          }
        }
      }
    };
    if constexpr (kLut) {         // V only: the scores come from the LUT
      fill(cbv_r, kNV, 1 << BV, DV, 0u);
    } else if constexpr (kBins) {  // K only: P.V goes through the bins
      fill(cbk_r, kNK, 1 << BK, DK, 0u);
      // the fp32 V codebook for the bins' final product, after the bins
      float4* cvf = reinterpret_cast<float4*>(smem + L.aux + kLutBytes);
      if (tid < (1 << BV)) {
        const __half2 h01 = *reinterpret_cast<const __half2*>(&cbv_r[0].x);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&cbv_r[0].y);
        cvf[tid] = make_float4(__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23));
      }
    } else {
      fill(cbk_r, kNK, 1 << BK, DK, 0u);
      fill(cbv_r, kNV, 1 << BV, DV, 128u);
    }
  }
  if (tid < n_units) {
    ulen_c[tid] = len_r[0];  // raw: the append needs the unclamped length
    if constexpr (kResidual) ures_c[tid] = min(max(len_r[1], 0), p.res_capacity);
  }

  // Fused append: ||c||^2 and -2 c of every centroid in fp32, computed as the
  // encode kernel computes them (the norm a chain of fused multiply-adds in
  // element order; -2 c exact).
  if constexpr (kAppend && !kWide) {
#pragma unroll
    for (int i = 0; i < kNK; ++i) {
      const int j = tid + i * kConsumerThreads;
      if (j < (1 << BK)) append_tables<DK>(cbk_r[i], j, enc_kn, enc_km);
    }
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int j = tid + i * kConsumerThreads;
      if (j < (1 << BV)) append_tables<DV>(cbv_r[i], j, enc_vn, enc_vm);
    }
  }
  if constexpr (kAppend) {
    // the tables and the norms (none for the 1.5-bit format) are what the
    // producers' encode reads
    asm volatile("bar.arrive 4, %0;" ::"n"((NW + NP) * 32) : "memory");
  }
  // q~ = q diag(lambda) H_D * scale * log2(e), split into fp16 hi + lo parts
  // and stored in the score mma's B-operand order: table [head][hi, lo][c][16
  // words], words 2kk, 2kk+1 = dims 32c + 4kk + {0, 1} and {2, 3} (lane l of
  // the head's warp holds dims 4l .. 4l+3, i.e. c = l / 8, kk = l % 8).  Heads
  // G .. NG-1 are zeros.  The consumers then read their operands with a few
  // 16-byte loads.
  auto transform_query = [&](int k) {
    if (warp < NG) {
      uint32_t h01 = 0u, l01 = 0u, h23 = 0u, l23 = 0u;
      if (warp < G) {
        const __half2 lo = *reinterpret_cast<const __half2*>(&q_r.x);
        const __half2 hi = *reinterpret_cast<const __half2*>(&q_r.y);
        float x[4] = {__low2float(lo) * lam_r.x, __high2float(lo) * lam_r.y,
                      __low2float(hi) * lam_r.z, __high2float(hi) * lam_r.w};
        fwht128_warp(x, lane);
        if constexpr (kLut) {  // fp32 q~ [head][128] for the LUT
          reinterpret_cast<float4*>(qt + warp * kHeadDim)[lane] =
              make_float4(x[0] * p.qscale, x[1] * p.qscale, x[2] * p.qscale, x[3] * p.qscale);
        }
        split_half2(x[0] * p.qscale, x[1] * p.qscale, h01, l01);
        split_half2(x[2] * p.qscale, x[3] * p.qscale, h23, l23);
        load_q(k + 1);  // prefetch the next unit's query
      } else if constexpr (kLut) {
        reinterpret_cast<float4*>(qt + warp * kHeadDim)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if constexpr (!kLut) {
        uint32_t* qf = reinterpret_cast<uint32_t*>(qt) + (warp * 2 * 4 + (lane >> 3)) * 16 + 2 * (lane & 7);
        *reinterpret_cast<uint2*>(qf) = make_uint2(h01, h23);
        *reinterpret_cast<uint2*>(qf + 4 * 16) = make_uint2(l01, l23);
      }
    }
  };
  transform_query(0);
  consumer_sync<NW>();  // codebook table, unit lengths and the first unit's q~ visible

  const int r = lane >> 2, c = lane & 3;
  // the lane's byte inside a table row: its replica of the K (bytes 0..127)
  // or V (bytes 128..255) centroid, one bank pair (8-byte) or bank (4-byte) per lane
  const uint32_t lwk = kWide ? 0u : DK == 4 ? (lane & 15) * 8 : lane * 4;
  const uint32_t lwv = kWide ? 65536u : (kLut ? 0u : 128u) + (DV == 4 ? (lane & 15) * 8 : lane * 4);
  uint32_t qa[8][2];  // score B operands: NG == 4: columns (2g: hi, 2g+1: lo); NG == 8: hi
  uint32_t qb[8][2];  // NG == 8: lo
  float O[8][4];      // output accumulators (NG == 4 uses O[0..3])
  float m_run[NGL], l_run[NGL] = {};

  // ---- code registers -------------------------------------------------------
  // K: tokens r and r+8 of the warp's chunk.  V (G <= 4): tokens c, c+4, c+8,
  // c+12; V (G > 4): tokens 2c, 2c+1, 2c+8, 2c+9, and with 32-byte rows lanes
  // c >= 2 read each pair swapped so that every load hits 32 different banks
  // (the PRMT selectors undo the swap).
  constexpr bool kSwap = NG == 8 && DV == 4 && BV == 8;
  const int sw = (kSwap && c >= 2) ? 1 : 0;
  const uint32_t sel_lo = sw ? 0x1054u : 0x5410u, sel_hi = sw ? 0x3276u : 0x7632u;
  // P operand placement (G <= 4): lane (r, c) puts p into half r & 1 of its
  // B registers; selectors taking the low / high half of a packed pair
  const uint32_t sel_p_lo = (r & 1) ? 0x1044u : 0x4410u, sel_p_hi = (r & 1) ? 0x3244u : 0x4432u;
  KCodes<DK> kc[2];          // current stage
  VCodes<DV, BV> vc[4];      // current stage
  VCodes<DV, BV> pvc[4];     // previous stage, P.V pending
  uint32_t pb[2][2] = {{0u, 0u}, {0u, 0u}};  // previous stage's P operands [k-step or token pair][reg]

  // lane-constant byte offsets of the lane's code rows inside a stage
  const int koff0 = (warp * kChunk + r) * KROW, koff1 = koff0 + 8 * KROW;
  const int voff = kStageTok * KROW + warp * kChunk * VROW;
  const int voff0 = voff;  // the warp's V rows (bins method: whole rows of tokens r and r+8)
  auto load_codes = [&](const uint8_t* st) {
    kc[0].load(st + koff0, c);
    kc[1].load(st + koff1, c);
    const uint8_t* sv = st + voff;
    if constexpr (NG == 4) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) vc[jj].load(sv + (c + 4 * jj) * VROW, r);
    } else {
      const uint8_t* vr0 = sv + (2 * c) * VROW;
      vc[0].load(vr0 + sw * VROW, r);
      vc[1].load(vr0 + (1 - sw) * VROW, r);
      vc[2].load(vr0 + (8 + sw) * VROW, r);
      vc[3].load(vr0 + (9 - sw) * VROW, r);
    }
  };

  // P.V of the previous stage's chunk, output step q (0..3 for G <= 4).
  //  G <= 4: the mma reduction index runs over (token t', element e) with
  //    k = 2 t' + e, so one gathered fp16 pair of a centroid is one operand
  //    register; the output column (2g + e') selects element e' of head g.
  //    Output rows r, r+8 of step q are the element pairs 0 and 1 (dv = 4) or
  //    sub-vectors 8r + 2q, 8r + 2q + 1 (dv = 2); lane (r, c) accumulates dims
  //    16r + 4q .. 16r + 4q + 3 of head c.
  //  G > 4: reduction over 16 tokens, A = V^T built with PRMT (pairs of tokens).
  // gather offsets: 256-byte table rows, or 128-byte rows for the table-based methods
  auto vgoff = [&](const VCodes<DV, BV>& v, int i) -> uint32_t {
    if constexpr (kWide) return 0u;  // the 1.5-bit format gathers whole centroids (off16)
    else if constexpr (kLut) return v.off7(i, lwv);
    else return v.off(i, lwv);
  };
  auto kgoff = [&](const KCodes<DK>& kcd, int i) -> uint32_t {
    if constexpr (kWide) return 0u;
    else if constexpr (kBins) return kcd.off7(i, lwk);
    else return kcd.off(i, lwk);
  };
  uint4 vw[4];  // 1.5-bit format: the whole centroids of the current output-step pair
  auto pv_step = [&](int q) {
    if constexpr (kWide) {
      if ((q & 1) == 0) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) vw[jj] = tab128(pvc[jj].off16(q >> 1, lwv));
      }
      uint2 W[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) W[jj] = (q & 1) ? make_uint2(vw[jj].z, vw[jj].w) : make_uint2(vw[jj].x, vw[jj].y);
      if constexpr (NG == 4) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)  // tokens 8ks + c and 8ks + c + 4
          mma16816(O[q], W[2 * ks].x, W[2 * ks].y, W[2 * ks + 1].x, W[2 * ks + 1].y, pb[ks][0], pb[ks][1]);
      } else {
        mma16816(O[2 * q], __byte_perm(W[0].x, W[1].x, sel_lo), __byte_perm(W[0].x, W[1].x, sel_hi),
                 __byte_perm(W[2].x, W[3].x, sel_lo), __byte_perm(W[2].x, W[3].x, sel_hi), pb[0][0],
                 pb[0][1]);
        mma16816(O[2 * q + 1], __byte_perm(W[0].y, W[1].y, sel_lo), __byte_perm(W[0].y, W[1].y, sel_hi),
                 __byte_perm(W[2].y, W[3].y, sel_lo), __byte_perm(W[2].y, W[3].y, sel_hi), pb[0][0],
                 pb[0][1]);
      }
    } else if constexpr (NG == 4) {
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {  // tokens 8ks + c and 8ks + c + 4
        uint32_t a0, a1, a2, a3;
        if constexpr (DV >= 4) {
          const uint2 w0 = tab64(vgoff(pvc[2 * ks], q));
          const uint2 w1 = tab64(vgoff(pvc[2 * ks + 1], q));
          a0 = w0.x; a1 = w0.y; a2 = w1.x; a3 = w1.y;
        } else {
          a0 = tab32(pvc[2 * ks].off(2 * q, lwv));
          a1 = tab32(pvc[2 * ks].off(2 * q + 1, lwv));
          a2 = tab32(pvc[2 * ks + 1].off(2 * q, lwv));
          a3 = tab32(pvc[2 * ks + 1].off(2 * q + 1, lwv));
        }
        mma16816(O[q], a0, a1, a2, a3, pb[ks][0], pb[ks][1]);
      }
    } else {
      if constexpr (DV >= 4) {  // q = output step pair (2q, 2q+1)
        uint2 W[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) W[jj] = tab64(pvc[jj].off(q, lwv));
        mma16816(O[2 * q], __byte_perm(W[0].x, W[1].x, sel_lo), __byte_perm(W[0].x, W[1].x, sel_hi),
                 __byte_perm(W[2].x, W[3].x, sel_lo), __byte_perm(W[2].x, W[3].x, sel_hi), pb[0][0],
                 pb[0][1]);
        mma16816(O[2 * q + 1], __byte_perm(W[0].y, W[1].y, sel_lo), __byte_perm(W[0].y, W[1].y, sel_hi),
                 __byte_perm(W[2].y, W[3].y, sel_lo), __byte_perm(W[2].y, W[3].y, sel_hi), pb[0][0],
                 pb[0][1]);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t W[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) W[jj] = tab32(pvc[jj].off(2 * q + h, lwv));
          mma16816(O[2 * q + h], __byte_perm(W[0], W[1], 0x5410), __byte_perm(W[0], W[1], 0x7632),
                   __byte_perm(W[2], W[3], 0x5410), __byte_perm(W[2], W[3], 0x7632), pb[0][0],
                   pb[0][1]);
        }
      }
    }
  };

  // One basic block: scores of the current chunk and P.V of the previous
  // chunk, two independent streams the scheduler interleaves.
  auto fused = [&](float (&sc)[4], bool with_qk) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    uint4 kw0, kw1;  // 1.5-bit format: whole centroids of tokens r and r+8 for k-steps 2j, 2j+1
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (with_qk) {
        uint32_t a0, a1, a2, a3;
        if constexpr (kWide) {
          if ((kk & 1) == 0) {
            kw0 = tab128(kc[0].off16(kk >> 1, lwk));
            kw1 = tab128(kc[1].off16(kk >> 1, lwk));
          }
          a0 = (kk & 1) ? kw0.z : kw0.x;
          a1 = (kk & 1) ? kw1.z : kw1.x;
          a2 = (kk & 1) ? kw0.w : kw0.y;
          a3 = (kk & 1) ? kw1.w : kw1.y;
        } else if constexpr (DK >= 4) {
          const uint2 g0 = tab64(kgoff(kc[0], kk));
          const uint2 g1 = tab64(kgoff(kc[1], kk));
          a0 = g0.x; a1 = g1.x; a2 = g0.y; a3 = g1.y;
        } else {
          a0 = tab32(kc[0].off(2 * kk, lwk));
          a1 = tab32(kc[1].off(2 * kk, lwk));
          a2 = tab32(kc[0].off(2 * kk + 1, lwk));
          a3 = tab32(kc[1].off(2 * kk + 1, lwk));
        }
        mma16816(acc, a0, a1, a2, a3, qa[kk][0], qa[kk][1]);
        if constexpr (NG == 8) mma16816(acc2, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      if constexpr (!kBins) {
        if ((kk & 1) == 0) pv_step(kk >> 1);
      }
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sc[jj] = NG == 8 ? acc[jj] + acc2[jj] : acc[jj];
  };

  // LUT method: scores of the warp's chunk from the per-query table
  // LUT[i][j][g] = q~_g[4i .. 4i+3] . C_k[j] (fp32, [subspace][code][head]):
  // lane (r, c) sums subspaces 8c .. 8c+7 of tokens r and r+8 for every head,
  // the four lanes of a row add their sums by shuffle, and the lane keeps head
  // c, the score layout the softmax takes (hi part = score, lo part = 0).  The
  // previous chunk's P.V runs in the same block, as in `fused`.
  auto fused_lut = [&](float (&sc)[4], bool with_qk) {
   if constexpr (kLut) {
    const float4* lut = reinterpret_cast<const float4*>(smem + L.aux) + 8 * c * 256;
    float a[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (with_qk) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float4 e = lut[kk * 256 + kc[t].code(kk)];
          a[t][0] += e.x;
          a[t][1] += e.y;
          a[t][2] += e.z;
          a[t][3] += e.w;
        }
      }
      if ((kk & 1) == 0) pv_step(kk >> 1);
    }
    if (with_qk) {
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          a[t][g] += __shfl_xor_sync(kFull, a[t][g], 1);
          a[t][g] += __shfl_xor_sync(kFull, a[t][g], 2);
        }
      sc[0] = c == 0 ? a[0][0] : c == 1 ? a[0][1] : c == 2 ? a[0][2] : a[0][3];
      sc[2] = c == 0 ? a[1][0] : c == 1 ? a[1][1] : c == 2 ? a[1][2] : a[1][3];
      sc[1] = sc[3] = 0.f;
    }
   }
  };

  // LUT method: the table of the unit's q~ (built after q~ is visible).
  auto build_lut = [&]() {
    if constexpr (kLut) {
      float4* lut = reinterpret_cast<float4*>(smem + L.aux);
      const float4* q4 = reinterpret_cast<const float4*>(qt);  // fp32 q~ [head][128]
      for (int e = tid; e < 32 * 256; e += kConsumerThreads) {
        const int i = e >> 8, j = e & 255;
        const uint2 cw = __ldg(reinterpret_cast<const uint2*>(p.cb_k) + j);
        const __half2 c01 = *reinterpret_cast<const __half2*>(&cw.x), c23 = *reinterpret_cast<const __half2*>(&cw.y);
        const float c0 = __low2float(c01), c1 = __high2float(c01), c2 = __low2float(c23), c3 = __high2float(c23);
        float v[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 qg = q4[g * (kHeadDim / 4) + i];
          v[g] = fmaf(qg.w, c3, fmaf(qg.z, c2, fmaf(qg.y, c1, qg.x * c0)));
        }
        lut[e] = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
  };

  // Bins method: p of every (token, subspace) is added into bins[i][code][head]
  // (fp32, shared by the consumer warps); at the end of the unit o_g[4i + e] =
  // sum_j bins[i][j][g] C_v[j][e].  The warps share one reference maximum per
  // head, so each stage first agrees on the stage's maximum (a consumer
  // barrier) and, when it grew by more than kLazyLog2, rescales the bins.
  float mref = -INFINITY;  // bins method: this lane's head (c) reference
  auto bins_update = [&](const float (&sc)[4], const uint4 (&vr)[2][2], int tok0, int lim, bool live,
                         int par) {
    if constexpr (kBins) {
      float* bins = reinterpret_cast<float*>(smem + L.aux);
      float* smax = reinterpret_cast<float*>(mlbuf);  // [2][NW][4]: the stage maxima per warp and head
      float s0 = sc[0] + sc[1], s1 = sc[2] + sc[3];   // head c, tokens r and r+8
      if (!live || tok0 + kChunk > lim) {
        const int lim_n = live ? lim : 0;
        s0 = tok0 + r < lim_n ? s0 : -INFINITY;
        s1 = tok0 + r + 8 < lim_n ? s1 : -INFINITY;
      }
      float mx = fmaxf(s0, s1);
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
      if (r == 0) smax[(par * NW + warp) * 4 + c] = mx;
      consumer_sync<NW>();
      float M = mref;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, smax[(par * NW + w) * 4 + c]);
      // every warp reads the same maxima, so the decision is the same in all of them
      if (__any_sync(kFull, M > mref + kLazyLog2)) {
        const bool grows = M > mref + kLazyLog2;
        const float alpha = !grows ? 1.f : mref == -INFINITY ? 0.f : fast_exp2(mref - M);
        float al[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) al[g] = __shfl_sync(kFull, alpha, g);  // lane g holds head g
        float4* b4 = reinterpret_cast<float4*>(bins);
        for (int e = tid; e < 32 * 256; e += kConsumerThreads) {
          float4 b = b4[e];
          b.x *= al[0];
          b.y *= al[1];
          b.z *= al[2];
          b.w *= al[3];
          b4[e] = b;
        }
        l_run[0] *= alpha;
        if (grows) mref = M;
        consumer_sync<NW>();  // the bins are at the new reference before any warp adds to them
      }
      const float mr = mref == -INFINITY ? 0.f : mref;
      const float p0 = fast_exp2(s0 - mr), p1 = fast_exp2(s1 - mr);
      l_run[0] += p0 + p1;
      const uint32_t base = smem_addr(bins) + 4u * c;  // + ((i * 256 + code) * 4) * 4
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float pt = t ? p1 : p0;
        if (pt != 0.f) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t w = (i < 16) ? (i < 8 ? (i < 4 ? vr[t][0].x : vr[t][0].y) : (i < 12 ? vr[t][0].z : vr[t][0].w))
                                        : (i < 24 ? (i < 20 ? vr[t][1].x : vr[t][1].y) : (i < 28 ? vr[t][1].z : vr[t][1].w));
            const uint32_t code = __byte_perm(w, 0u, 0x4440 | (i & 3));
            asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(base + i * 4096u + (code << 4)), "f"(pt) : "memory");
          }
        }
      }
    }
  };

  // Online softmax (log2 domain) over the current chunk: updates m and l,
  // rescales O, and leaves the chunk's P operands (fp16) in pb.  Tokens at or
  // past `lim` get p = 0, and all of them when `live` is false.
  auto softmax = [&](const float (&sc)[4], int tok0, int lim, bool live) {
    float s[NGL][2];
    if constexpr (NG == 4) {  // columns 2c (hi) + 2c+1 (lo) of head c
      s[0][0] = sc[0] + sc[1];
      s[0][1] = sc[2] + sc[3];
    } else {                  // columns 2c, 2c+1 = heads 2c, 2c+1
      s[0][0] = sc[0];
      s[1][0] = sc[1];
      s[0][1] = sc[2];
      s[1][1] = sc[3];
    }
    if (!live || tok0 + kChunk > lim) {  // warp-uniform: a chunk at the end of the unit, or no data
      const int lim_n = live ? lim : 0;
      const bool v0 = tok0 + r < lim_n, v1 = tok0 + r + 8 < lim_n;
#pragma unroll
      for (int gi = 0; gi < NGL; ++gi) {
        s[gi][0] = v0 ? s[gi][0] : -INFINITY;
        s[gi][1] = v1 ? s[gi][1] : -INFINITY;
      }
    }
    // Lazy running max: m_run moves only when a score exceeds it by more than
    // kLazyLog2, so p = 2^(s - m_run) <= 2^kLazyLog2 stays far inside fp16 and
    // fp32 range, and most chunks skip the warp max reduction and the rescale
    // of O and l.  Any common reference gives the same normalised result.
    float lmax[NGL];
    bool grow = false;
#pragma unroll
    for (int gi = 0; gi < NGL; ++gi) {
      lmax[gi] = fmaxf(s[gi][0], s[gi][1]);
      grow = grow || lmax[gi] > m_run[gi] + kLazyLog2;
    }
    if (__any_sync(kFull, grow)) {
      float alpha[NGL];
#pragma unroll
      for (int gi = 0; gi < NGL; ++gi) {
        float mx = lmax[gi];
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float mnew = fmaxf(m_run[gi], mx);
        alpha[gi] = mnew == -INFINITY ? 1.f : fast_exp2(m_run[gi] - mnew);  // 0 from -inf
        l_run[gi] *= alpha[gi];
        m_run[gi] = mnew;
      }
      if constexpr (NG == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) O[i][jj] *= alpha[0];
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          O[i][0] *= alpha[0]; O[i][2] *= alpha[0];
          O[i][1] *= alpha[NGL - 1]; O[i][3] *= alpha[NGL - 1];
        }
      }
    }
#pragma unroll
    for (int gi = 0; gi < NGL; ++gi) {
      const float mref = m_run[gi] == -INFINITY ? 0.f : m_run[gi];
      s[gi][0] = fast_exp2(s[gi][0] - mref);
      s[gi][1] = fast_exp2(s[gi][1] - mref);
      l_run[gi] += s[gi][0] + s[gi][1];
    }
    if constexpr (NG == 4) {
      // B[k = 2t' + e][col = 2g + e'] = p[t'][g] * (e == e'): lane (r, c) needs
      // p of head r/2 for tokens c, c+4 (k-step 0) and c+8, c+12 (k-step 1).
      // Lane (r', c') holds p of head c' for tokens r' and r'+8: packed into one
      // fp16 pair, two shuffles fetch the pairs of tokens (c, c+8) and (c+4,
      // c+12), and each operand register takes one half, placed in half r & 1.
      const uint32_t mine = pack_half2(__float2half_rn(s[0][0]), __float2half_rn(s[0][1]));
      const uint32_t x = __shfl_sync(kFull, mine, 4 * c + (r >> 1));
      const uint32_t y = __shfl_sync(kFull, mine, 4 * (c + 4) + (r >> 1));
      pb[0][0] = __byte_perm(x, 0u, sel_p_lo);
      pb[0][1] = __byte_perm(y, 0u, sel_p_lo);
      pb[1][0] = __byte_perm(x, 0u, sel_p_hi);
      pb[1][1] = __byte_perm(y, 0u, sel_p_hi);
    } else {
      // P^T operand: transpose the fp16 pairs (head 2c, 2c+1) of each 8-token block
#pragma unroll
      for (int t = 0; t < 2; ++t)
        pb[0][t] = movmatrix_trans(pack_half2(__float2half_rn(s[0][t]), __float2half_rn(s[NGL - 1][t])));
    }
  };

  // Copies window tokens [t0, t0 + n) of the unit's (sequence, KV head) to
  // the window area of shared memory (K rows at 0, V rows at res_tok * 256,
  // then the raw queries when with_q), 16 bytes per cp.async.
  auto res_issue = [&](const UnitStages& u, int t0, int n, bool with_q) {
    if constexpr (kResidual) {
      const long long head = static_cast<long long>(u.b) * p.hkv + u.kvh;
      const uint8_t* kr = static_cast<const uint8_t*>(p.k_res) + (head * p.res_capacity + t0) * (kHeadDim * 2);
      const uint8_t* vr = static_cast<const uint8_t*>(p.v_res) + (head * p.res_capacity + t0) * (kHeadDim * 2);
      const uint8_t* qr = static_cast<const uint8_t*>(p.q) + (static_cast<long long>(u.b) * p.hq + u.kvh * G) * (kHeadDim * 2);
      const int nk = n * 16;  // 16-byte pieces of the K (then V) rows
      const int total = 2 * nk + (with_q ? G * 16 : 0);
      for (int i = tid; i < total; i += kConsumerThreads) {
        const uint8_t* src = i < nk ? kr + i * 16 : i < 2 * nk ? vr + (i - nk) * 16 : qr + (i - 2 * nk) * 16;
        const int off = i < nk ? i * 16 : i < 2 * nk ? p.res_tok * 256 + (i - nk) * 16 : 2 * p.res_tok * 256 + (i - 2 * nk) * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem + L.res + off)), "l"(src)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  };

  // The unit's window slice (see the unit loop) joins the warp's online
  // softmax: warp w takes slice tokens w, w + NW, ...; every lane forms the G
  // dot products from its four elements and a butterfly reduction, then lane
  // (r, c) updates its heads' running maximum, sum and output elements.
  auto residual_merge = [&](int t0, int n, const UnitStages& u) {
    if constexpr (kResidual) {
      const int T = p.res_tok;
      asm volatile("cp.async.wait_all;" ::: "memory");
      consumer_sync<NW>();  // every thread's copies are visible
      const uint8_t* rs = smem + L.res;
      auto unpack = [](uint2 w, float (&f)[4]) {
        const __half2 lo = *reinterpret_cast<const __half2*>(&w.x), hi = *reinterpret_cast<const __half2*>(&w.y);
        f[0] = __low2float(lo);
        f[1] = __high2float(lo);
        f[2] = __low2float(hi);
        f[3] = __high2float(hi);
      };
      float qv[NG][4];
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (g < G) unpack(reinterpret_cast<const uint2*>(rs + 2 * T * 256 + g * 256)[lane], qv[g]);
        else qv[g][0] = qv[g][1] = qv[g][2] = qv[g][3] = 0.f;
      }
      // one window token: its G scores (the reductions side by side; heads
      // >= G have q = 0 and get -inf), then the lane's heads' softmax state
      // and outputs
      auto token = [&](const uint8_t* kr, const uint8_t* vr) {
        float kf[4];
        unpack(reinterpret_cast<const uint2*>(kr)[lane], kf);
        float sg[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          sg[g] = qv[g][0] * kf[0];
          sg[g] = fmaf(qv[g][1], kf[1], sg[g]);
          sg[g] = fmaf(qv[g][2], kf[2], sg[g]);
          sg[g] = fmaf(qv[g][3], kf[3], sg[g]);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
          for (int g = 0; g < NG; ++g) sg[g] += __shfl_xor_sync(kFull, sg[g], o);
#pragma unroll
        for (int g = 0; g < NG; ++g) sg[g] = g < G ? sg[g] * p.res_scale_log2 : -INFINITY;
        float s[NGL];
#pragma unroll
        for (int gi = 0; gi < NGL; ++gi) {
          const int hd = NG == 4 ? c : 2 * c + gi;  // the lane's head(s)
          float v = sg[0];
#pragma unroll
          for (int g = 1; g < NG; ++g) v = hd == g ? sg[g] : v;
          s[gi] = v;
        }
        bool grow = false;
#pragma unroll
        for (int gi = 0; gi < NGL; ++gi) grow = grow || s[gi] > m_run[gi] + kLazyLog2;
        if (__any_sync(kFull, grow)) {
          float alpha[NGL];
#pragma unroll
          for (int gi = 0; gi < NGL; ++gi) {
            const float mnew = fmaxf(m_run[gi], s[gi]);
            alpha[gi] = mnew == -INFINITY ? 1.f : fast_exp2(m_run[gi] - mnew);
            l_run[gi] *= alpha[gi];
            m_run[gi] = mnew;
          }
          if constexpr (NG == 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) O[q][jj] *= alpha[0];
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              O[q][0] *= alpha[0]; O[q][2] *= alpha[0];
              O[q][1] *= alpha[NGL - 1]; O[q][3] *= alpha[NGL - 1];
            }
          }
        }
        float pr[NGL];
#pragma unroll
        for (int gi = 0; gi < NGL; ++gi) {
          pr[gi] = fast_exp2(s[gi] - (m_run[gi] == -INFINITY ? 0.f : m_run[gi]));
          if (r == 0) l_run[gi] += pr[gi];  // the warp's sum adds the 8 lanes of a head once
        }
        // value elements 16 r .. 16 r + 15: the lane's output rows
        const uint4 w0 = reinterpret_cast<const uint4*>(vr + 32 * r)[0];
        const uint4 w1 = reinterpret_cast<const uint4*>(vr + 32 * r)[1];
        float vf[4][4];
        unpack(make_uint2(w0.x, w0.y), vf[0]);
        unpack(make_uint2(w0.z, w0.w), vf[1]);
        unpack(make_uint2(w1.x, w1.y), vf[2]);
        unpack(make_uint2(w1.z, w1.w), vf[3]);
        if constexpr (NG == 4) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) O[q][jj] = fmaf(pr[0], vf[q][jj], O[q][jj]);
        } else {
          // head 2c + gi: element 16r + 4i + {0, 1, 2, 3} sits in O[2i][gi],
          // O[2i][2 + gi], O[2i + 1][gi], O[2i + 1][2 + gi]
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
            for (int gi = 0; gi < NGL; ++gi) {
              O[2 * i4][gi] = fmaf(pr[gi], vf[i4][0], O[2 * i4][gi]);
              O[2 * i4][2 + gi] = fmaf(pr[gi], vf[i4][1], O[2 * i4][2 + gi]);
              O[2 * i4 + 1][gi] = fmaf(pr[gi], vf[i4][2], O[2 * i4 + 1][gi]);
              O[2 * i4 + 1][2 + gi] = fmaf(pr[gi], vf[i4][3], O[2 * i4 + 1][2 + gi]);
            }
        }
      };
      // chunks of T tokens; the first was copied at unit start
      for (int c0 = 0; c0 < n; c0 += T) {
        if (c0 > 0) {
          consumer_sync<NW>();  // every warp is done with the previous chunk
          res_issue(u, t0 + c0, min(n - c0, T), false);
          asm volatile("cp.async.wait_all;" ::: "memory");
          consumer_sync<NW>();
        }
        for (int i = warp; i < min(n - c0, T); i += NW) token(rs + i * 256, rs + T * 256 + i * 256);
      }
    }
  };

  int slot = 0;          // slot of the next stage (stages run in the producers' order)
  uint32_t phase = 0u;   // parity of the slot's current fill
  for (int k = 0; k < n_units; ++k) {
    const UnitStages u = unit_stages<kStageTok, kBal>(p, bal, k, clamp_len(ulen_c[k]));
    if (k > 0) consumer_sync<NW>();  // previous unit's merge buffers and q~ are free
    // Full-precision residual window (VecInfer, 实验结果 / 实验设置: the most
    // recent tokens stay unquantized): unit s of the cnt units of a
    // (sequence, KV head) takes window tokens [s R / cnt, (s + 1) R / cnt) and merges
    // them into its own online softmax after its stages, with s = q . k *
    // scale * log2(e) from the raw query and key (the log2 domain of q~'s
    // scores).  The slice's first res_tok rows and the raw queries are copied
    // to shared memory with cp.async here, while the stages stream.
    int res_t0 = 0, res_n = 0;
    if constexpr (kResidual) {
      const int R = ures_c[k];
      res_t0 = u.s * R / u.cnt;
      res_n = (u.s + 1) * R / u.cnt - res_t0;
      res_issue(u, res_t0, min(res_n, p.res_tok), true);
    }
    if (k > 0) {
      transform_query(k);
      consumer_sync<NW>();
    }
    // B operands of the score mma: k-step kk, rows {2c, 2c+1, 2c+8, 2c+9} hold
    // dims 32c + 4kk + {0, 1, 2, 3}; column = r (G <= 4: head r / 2, hi part
    // for even r, lo for odd r; G > 4: head r, hi in qa and lo in qb).
    if constexpr (kLut) {
      build_lut();
      consumer_sync<NW>();  // the unit's LUT is complete
    } else {
      const uint4* qf = reinterpret_cast<const uint4*>(qt);
      if constexpr (NG == 4) {
        const int blk = ((r >> 1) * 2 + (r & 1)) * 4 + c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 wv = qf[blk * 4 + i];
          qa[2 * i][0] = wv.x;
          qa[2 * i][1] = wv.y;
          qa[2 * i + 1][0] = wv.z;
          qa[2 * i + 1][1] = wv.w;
        }
      } else {
        const int bh = (r * 2) * 4 + c, bl = (r * 2 + 1) * 4 + c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 wh = qf[bh * 4 + i], wl = qf[bl * 4 + i];
          qa[2 * i][0] = wh.x;
          qa[2 * i][1] = wh.y;
          qa[2 * i + 1][0] = wh.z;
          qa[2 * i + 1][1] = wh.w;
          qb[2 * i][0] = wl.x;
          qb[2 * i][1] = wl.y;
          qb[2 * i + 1][0] = wl.z;
          qb[2 * i + 1][1] = wl.w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) O[i][jj] = 0.f;
#pragma unroll
    for (int gi = 0; gi < NGL; ++gi) {
      m_run[gi] = -INFINITY;
      l_run[gi] = 0.f;
    }
    if constexpr (kBins) {  // empty bins at no reference
      float4* b4 = reinterpret_cast<float4*>(smem + L.aux);
      for (int e = tid; e < 32 * 256; e += kConsumerThreads) b4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      mref = -INFINITY;
      consumer_sync<NW>();
    }
    if (k == 0) pdl_wait();  // partials are written only after the previous kernel completes
    pb[0][0] = pb[0][1] = pb[1][0] = pb[1][1] = 0u;  // nothing pending yet
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) pvc[jj] = VCodes<DV, BV>{};

    for (int j = 0; j < u.count; ++j) {
      bool ok = mbar_try_wait(full + slot, phase);
      if (!__all_sync(kFull, ok)) {  // slow path: bounded wait
        ok = !*abort_flag && mbar_wait_bounded(full + slot, phase, abort_flag, p.timeout_ns);
        ok = __all_sync(kFull, ok);
        if (!ok && lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          report(p.status, kDevTimeout);
        }
      }
      const int4 m = meta[slot];
      const int tok0 = m.x + warp * kChunk;      // first token of the warp's chunk
      const bool live = ok && ((static_cast<uint32_t>(m.z) >> warp) & 1u) && tok0 < m.y;
      if constexpr (kBins) {
        const uint8_t* st = stages + slot * kStageBytes;
        kc[0].load(st + koff0, c);
        kc[1].load(st + koff1, c);
        uint4 vr[2][2];  // V rows of tokens r and r+8 (32 codes each)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint4* row = reinterpret_cast<const uint4*>(st + voff0 + (r + 8 * t) * VROW);
          vr[t][0] = row[0];
          vr[t][1] = row[1];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        if (++slot == NS) {
          slot = 0;
          phase ^= 1u;
        }
        float sc[4];
        fused(sc, true);                         // scores only
        bins_update(sc, vr, tok0, m.y, live, j & 1);
      } else {
        load_codes(stages + slot * kStageBytes);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);  // codes are in registers: the slot may be refilled
        if (++slot == NS) {
          slot = 0;
          phase ^= 1u;
        }
        float sc[4];
        if constexpr (kLut) fused_lut(sc, true);
        else fused(sc, true);                      // scores now, P.V of the previous stage
        softmax(sc, tok0, m.y, live);              // tokens past the end and invalid pages: p = 0
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) pvc[jj] = vc[jj];
      }
    }
    if constexpr (!kBins) {  // P.V of the unit's last stage
      float sc[4];
      if constexpr (kLut) fused_lut(sc, false);
      else fused(sc, false);
    }
    if constexpr (kResidual) {
      residual_merge(res_t0, res_n, u);
      consumer_sync<NW>();  // the window slice (in the merge buffer) has been read
    }

    // ---- merge the consumer warps of this unit, write the split partial ------
#pragma unroll
    for (int gi = 0; gi < NGL; ++gi) {
      l_run[gi] += __shfl_xor_sync(kFull, l_run[gi], 4);
      l_run[gi] += __shfl_xor_sync(kFull, l_run[gi], 8);
      l_run[gi] += __shfl_xor_sync(kFull, l_run[gi], 16);
    }
    if constexpr (kBins) {
      // every stage's additions are in; the stage-maximum buffer holds the sums next
      consumer_sync<NW>();
      float* lsum = reinterpret_cast<float*>(mlbuf);  // [NW][4]
      if (r == 0) lsum[warp * 4 + c] = l_run[0];
      consumer_sync<NW>();
      // o_g[4i + e] = sum_j bins[i][j][g] C_v[j][e]: warp w takes subspaces w, w + NW, ...;
      // lane l the codes l, l + 32, ..., then a shuffle reduction
      const float4* b4 = reinterpret_cast<const float4*>(smem + L.aux);
      const float4* cvf = reinterpret_cast<const float4*>(smem + L.aux + kLutBytes);
      for (int i = warp; i < 32; i += NW) {
        float acc[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[g][e] = 0.f;
#pragma unroll
        for (int m8 = 0; m8 < 8; ++m8) {
          const int j = lane + 32 * m8;
          const float4 b = b4[i * 256 + j], cv = cvf[j];
          const float bg[4] = {b.x, b.y, b.z, b.w}, ce[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[g][e] = fmaf(bg[g], ce[e], acc[g][e]);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) acc[g][e] += __shfl_xor_sync(kFull, acc[g][e], sh);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (lane == g && g < G) {
            const long long row = (static_cast<long long>(u.b) * p.hq + u.kvh * G + g) * p.splits + u.s;
            reinterpret_cast<float4*>(p.ws_o + row * kHeadDim)[i] =
                make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
          }
      }
      if (warp == 0 && lane < G) {  // lane g (row 0, column g) holds head g's reference
        float l = 0.f;
        for (int w = 0; w < NW; ++w) l += lsum[w * 4 + lane];
        const long long row = (static_cast<long long>(u.b) * p.hq + u.kvh * G + lane) * p.splits + u.s;
        p.ws_ml[row] = make_float2(mref, mref == -INFINITY ? 0.f : l);
      }
      if (kBal && tid == 0 && u.s == 0) p.ws_cnt[static_cast<long long>(u.b) * p.hkv + u.kvh] = u.cnt;
      continue;  // the next unit starts with a consumer barrier
    }
    if constexpr (kLut) consumer_sync<NW>();  // the merge buffer is the LUT: every warp is done with it
    if constexpr (NG == 4) {
      if (c < G) {
        float4* mo = reinterpret_cast<float4*>(merge + (warp * G + c) * kHeadDim + 16 * r);
#pragma unroll
        for (int i = 0; i < 4; ++i) mo[i] = make_float4(O[i][0], O[i][1], O[i][2], O[i][3]);
        if (r == 0) mlbuf[warp * G + c] = make_float2(m_run[0], l_run[0]);
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < NGL; ++gi) {
        const int g = 2 * c + gi;
        if (g < G) {
          float4* mo = reinterpret_cast<float4*>(merge + (warp * G + g) * kHeadDim + 16 * r);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mo[i] = make_float4(O[2 * i][gi], O[2 * i][2 + gi], O[2 * i + 1][gi], O[2 * i + 1][2 + gi]);
          if (r == 0) mlbuf[warp * G + g] = make_float2(m_run[gi], l_run[gi]);
        }
      }
    }
    consumer_sync<NW>();
    // one thread per 4 output dims of a head: o = sum_w 2^(m_w - M) o_w, l likewise
    for (int i = tid; i < G * (kHeadDim / 4); i += kConsumerThreads) {
      const int g = i / (kHeadDim / 4), d4 = i % (kHeadDim / 4);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, mlbuf[w * G + g].x);
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float l = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float2 ml = mlbuf[w * G + g];
          const float f = fast_exp2(ml.x - M);
          const float4 v = reinterpret_cast<const float4*>(merge + (w * G + g) * kHeadDim)[d4];
          o.x = fmaf(f, v.x, o.x);
          o.y = fmaf(f, v.y, o.y);
          o.z = fmaf(f, v.z, o.z);
          o.w = fmaf(f, v.w, o.w);
          l = fmaf(f, ml.y, l);
        }
      }
      const long long row = (static_cast<long long>(u.b) * p.hq + u.kvh * G + g) * p.splits + u.s;
      reinterpret_cast<float4*>(p.ws_o + row * kHeadDim)[d4] = o;
      if (d4 == 0) p.ws_ml[row] = make_float2(M, l);
    }
    // the pair's unit count, for the combine (length-balanced units)
    if (kBal && tid == 0 && u.s == 0) p.ws_cnt[static_cast<long long>(u.b) * p.hkv + u.kvh] = u.cnt;
  }
  __syncthreads();  // matches the producers' final barrier
}

template <bool kBal, int DK, int BK, int DV, int BV, int NG, int NW, bool kAppend,
          int kMethod = kMethodGather, bool kResidual = false>
cudaError_t launch_split(const DecodeParams& p, int grid, size_t smem, cudaStream_t stream,
                         bool overlap) {
  auto kern = vq_decode_split_kernel<DK, BK, DV, BV, NG, NW, kAppend, kMethod, kResidual, kBal>;
  static SmemOptIn opt_in;
  cudaError_t e = ensure_smem(kern, smem, opt_in);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid), dim3((NW + kProducerWarps) * 32), smem, stream, p, overlap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool kBal, int DK, int BK, int DV, int BV>
cudaError_t launch_formats(const DecodeParams& p, int grid, size_t smem, cudaStream_t stream,
                           bool ov, int method) {
  const bool wide = p.group > 4;
  if (method != kMethodGather) {  // the table-based methods: d = 4, 8-bit codes, G <= 4, 12 warps
    if constexpr (DK == 4 && BK == 8 && DV == 4 && BV == 8) {
      if (!wide && p.warps == 12 && !p.append) {
        if (method == kMethodLut) return launch_split<kBal, 4, 8, 4, 8, 4, 12, false, kMethodLut>(p, grid, smem, stream, ov);
        if (method == kMethodBins) return launch_split<kBal, 4, 8, 4, 8, 4, 12, false, kMethodBins>(p, grid, smem, stream, ov);
      }
    }
    return cudaErrorInvalidValue;
  }
  if (p.residual) {  // attention with the residual window inside: the default shapes only
    if (p.warps == 12 && !wide)
      return launch_split<kBal, DK, BK, DV, BV, 4, 12, false, kMethodGather, true>(p, grid, smem, stream, ov);
    if (p.warps == 8)
      return wide ? launch_split<kBal, DK, BK, DV, BV, 8, 8, false, kMethodGather, true>(p, grid, smem, stream, ov)
                  : launch_split<kBal, DK, BK, DV, BV, 4, 8, false, kMethodGather, true>(p, grid, smem, stream, ov);
    return cudaErrorInvalidValue;
  }
  if (p.append) {  // the decode step with the append inside: the default shapes only
    if constexpr ((BK <= 9 && BV <= 9) || (DK == 8 && BK == 12)) {
      if (p.warps == 12 && !wide) return launch_split<kBal, DK, BK, DV, BV, 4, 12, true>(p, grid, smem, stream, ov);
      if (p.warps == 8)
        return wide ? launch_split<kBal, DK, BK, DV, BV, 8, 8, true>(p, grid, smem, stream, ov)
                    : launch_split<kBal, DK, BK, DV, BV, 4, 8, true>(p, grid, smem, stream, ov);
    }
    return cudaErrorInvalidValue;
  }
  if (p.warps == 12)
    return wide ? launch_split<kBal, DK, BK, DV, BV, 8, 12, false>(p, grid, smem, stream, ov)
                : launch_split<kBal, DK, BK, DV, BV, 4, 12, false>(p, grid, smem, stream, ov);
  if (p.warps == 8)
    return wide ? launch_split<kBal, DK, BK, DV, BV, 8, 8, false>(p, grid, smem, stream, ov)
                : launch_split<kBal, DK, BK, DV, BV, 4, 8, false>(p, grid, smem, stream, ov);
  return cudaErrorInvalidValue;
}

// The format dispatch of one instantiation family (kBal: length-balanced units).
template <bool kBal>
cudaError_t dispatch_decode(const DecodeParams& p, int k_sub, int k_bits, int v_sub, int v_bits,
                            int grid, size_t smem, cudaStream_t stream, bool overlap, int method) {
#define VQ_CASE(DK, BK, DV, BV) \
  if (k_sub == DK && k_bits == BK && v_sub == DV && v_bits == BV) \
    return launch_formats<kBal, DK, BK, DV, BV>(p, grid, smem, stream, overlap, method);
  VQ_CASE(2, 8, 4, 8)
  VQ_CASE(4, 8, 4, 8)
  VQ_CASE(2, 8, 4, 9)
  VQ_CASE(4, 8, 4, 9)
  VQ_CASE(2, 8, 2, 8)
  VQ_CASE(4, 8, 2, 8)
  VQ_CASE(8, 12, 8, 12)
#undef VQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace vqk
