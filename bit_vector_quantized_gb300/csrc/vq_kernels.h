// vq_kernels.h -- host-visible parameter blocks and launch entry points of the
// sm_103a kernels (internal to the library; the public ABI is include/vqattn.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace vqk {

struct EncodeParams {
  const void* src[2];    // fp16 [T][Hkv][128]: 0 = keys, 1 = values
  const void* cb[2];     // fp16 codebooks [2^bits][sub]
  uint8_t* pool[2];      // [num_pages][Hkv][P][row_bytes]
  int sub[2];
  int bits[2];
  int row_bytes[2];
  const float* lambda;   // fp32 [Hkv][128]
  const int64_t* slots;  // [T]
  int32_t* status;
  long long num_slots;   // num_pages * P
  int num_tokens;
  int hkv;
  int page_size;
  int split;             // warps per token-head: 1, 2, 4 or 8
  int which_base;        // blockIdx.y + which_base selects keys (0) or values (1)
  int vec_per_warp;      // 1, or kMultiVec (prefill with sub-vector lengths 2 / 4; split == 1)
  // A decode-step append with a large codebook can be spread over `slices`
  // CTAs per vector: CTA c scans centroids [c N / slices, (c + 1) N / slices)
  // and leaves its argmin candidates in `cand`; the merge kernel then merges
  // the slices in order (lowest index on ties) and stores the row.
  int slices;            // 1: each CTA stores its vectors' rows itself
  int2* cand;            // [vectors][2 tensors][slices][32 lanes][4] (score bits, index)
  // Decode-step append (slots == NULL): token t is the new token of sequence t,
  // stored at position seq_lens[t] - 1 through the page table.
  const int32_t* page_table;  // [T][max_pages]
  const int32_t* seq_lens;    // [T]
  int max_pages;
};

constexpr int kMultiVec = 4;  // vectors per warp of the prefill encode

struct DecodeParams {
  const void* q;              // fp16 [B][Hq][128]
  const float* lambda;        // fp32 [Hkv][128]
  const void* cb_k;           // fp16 [2^bk][dk]
  const void* cb_v;           // fp16 [2^bv][dv]
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* page_table;  // [B][max_pages]
  const int32_t* seq_lens;    // [B]
  float* ws_o;                // [B][Hq][S][128] unnormalised split outputs
  float2* ws_ml;              // [B][Hq][S] (running max in log2 units, row sum)
  int32_t* status;
  long long num_pages;
  unsigned long long timeout_ns;
  int batch, hq, hkv, group;
  int page_size, max_pages, max_seq_len;
  int splits, num_units;
  int split_q, split_r;       // ceil(max_seq_len / 32) = split_q * splits + split_r
  // Length-balanced units (balanced != 0, batches of two or more sequences):
  // the (sequence, KV head) pairs are laid end to end, each as its 32-token
  // blocks followed by kBalanceGap positions standing for a unit's fixed
  // cost, and CTA c takes positions [c W, (c + 1) W) with
  // W = max(ceil(total / grid), ceil(longest pair's blocks / (splits - 1))).
  // The blocks of a pair that fall in one CTA form a unit; the pair's j-th
  // unit writes partial slot j, and its first writes the pair's unit count
  // to ws_cnt.  The second term of W keeps the units of a pair within
  // `splits` slots.
  int balanced;
  int* ws_cnt;                // [B][Hkv] units per pair (balanced)
  int k_row, v_row;
  int nstage;
  int warps;                  // consumer warps (DecodeShape)
  float qscale;               // softmax scale * log2(e) / sqrt(128)
  // Decode-step append inside the attention kernel (append != 0): the new
  // token of every sequence, position seq_lens[b] - 1, is encoded by the CTA
  // whose unit holds that position and written to the pools through the
  // page table, and its codes join the attention directly.
  int append;
  const void* k_new;          // fp16 [B][Hkv][128]
  const void* v_new;
  uint8_t* k_pool_w;          // the pools, written (k_pool / v_pool as writable pointers)
  uint8_t* v_pool_w;
  // the 1.5-bit format: the encode kernel's sliced-scan candidates
  // [vectors][2 tensors][app_slices][32 lanes][4] (score bits, index)
  const int2* app_cand;
  int app_slices;
  // Full-precision residual window inside the attention kernel (residual != 0):
  // the unit of split s of each (sequence, KV head) merges window tokens
  // [s R / S, (s + 1) R / S) into its own partial.
  int residual;
  const void* k_res;          // fp16 [B][Hkv][res_capacity][128]
  const void* v_res;
  const int32_t* res_lens;    // [B], clamped to [0, res_capacity]
  int res_capacity;
  int res_tok;                // window tokens staged in shared memory at a time
  float res_scale_log2;       // softmax scale * log2(e) (raw q . k)
};

struct DequantParams {
  const uint8_t* k_pool;      // code pools [num_pages][Hkv][P][row bytes]
  const uint8_t* v_pool;
  const void* cb_k;           // fp16 [2^bits][sub]
  const void* cb_v;
  void* out_k;                // fp16 [T][Hkv][128]
  void* out_v;
  int k_sub, k_bits, k_row, v_sub, v_bits, v_row;
  const float* lambda;        // fp32 [Hkv][128]
  const int64_t* slots;       // [T]
  int32_t* status;
  long long num_slots;        // num_pages * P
  int num_tokens, hkv, page_size;
  int which_base, which_last;  // tensors produced: keys (0) and / or values (1)
};

struct CombineParams {
  const float* ws_o;
  const float2* ws_ml;
  void* out;                  // fp16 [B][Hq][128]
  int rows;                   // B * Hq
  int splits;
  const int* cnt;             // [B][Hkv] partials per pair (length-balanced units), or NULL: `splits`
  int group;                  // Hq / Hkv (row / group = pair)
};


constexpr int kProducerWarps = 4;  // TMA-issuing warps (one in four stages each)
constexpr int kMaxUnitsPerCta = 256;
constexpr int kUnitTok = 32;       // split boundaries are multiples of this many tokens
constexpr int kBalanceGap = 12;    // a unit's fixed cost in 32-token blocks (length-balanced units)
constexpr int kBalanceMaxBatch = 512;  // sequences, at most, for length-balanced units

constexpr int kMaxResTok = 64;     // residual window tokens staged in shared memory at a time, at most
constexpr int kMaxStages = 16;     // pipeline slots of the split kernel, at most

// Consumer shape: `warps` consumer warps, each taking one 16-token mma chunk
// of every pipeline stage (a stage holds warps * 16 tokens).
struct DecodeShape {
  int warps;
  __host__ __device__ int stage_tok() const { return warps * 16; }
};

// Shared-memory carve-up of the split attention kernel (bytes, 128-aligned);
// `warps` is the number of consumer warps.  The codebook table comes first (at
// offset 0 of the dynamic shared memory): row j is 256 bytes, the replicas of K
// centroid j in bytes 0..127 and those of V centroid j in bytes 128..255, so a
// gather address is (code << 8) | lane byte.  The 1.5-bit format (4096
// centroids of 8 elements) has no replicas: 32 bytes per centroid index, laid
// out half-major ([tensor][half][code] x 8 bytes).
struct DecodeSmem {
  int tab, qt, merge, ml, units, meta, bar, flag, enc, aux, res, stage, total;
};



// Score and P.V methods of the split kernel (the pages' alternatives):
//   kMethodGather: scores and P.V from centroid gathers on the tensor cores;
//   kMethodLut:    scores from a per-query, per-subspace lookup table
//                  q~_i . C_k[j] summed over the K codes, P.V by gather;
//   kMethodBins:   scores by gather, P.V by accumulating p into per-code bins,
//                  multiplied by the V codebook at the end of each unit.
// The table-based methods exist for d = 4, 8-bit K and V codes, G <= 4.
enum DecodeMethod : int { kMethodGather = 0, kMethodLut = 1, kMethodBins = 2 };

constexpr int kLutBytes = 32 * 256 * 4 * 4;  // [subspace][code][head] fp32: the LUT or the bins

constexpr int kTabRow = 256;      // bytes per codebook table row (replicated centroids)
constexpr int kTabRowWide = 32;   // 1.5-bit format (12-bit codes): K and V centroid, no replicas

__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }

// Bytes of the fused append's encode tables: per tensor ||c_j||^2 (fp32,
// 2^bits), then -2 c_j in fp32 (2^bits x sub, K then V), then the producer
// warps' argmin scratch ([4 warps][32 lanes][up to 2 + 2 sub-vectors] x
// (score, index)).
__host__ __device__ inline int append_enc_bytes(int k_bits, int v_bits, int k_sub, int v_sub) {
  return ((1 << k_bits) + (1 << v_bits)) * 4 + ((1 << k_bits) * k_sub + (1 << v_bits) * v_sub) * 4 +
         4 * 32 * 4 * 8;
}

// append_enc: the fused append's table and scratch bytes (0: no append)
// method: a DecodeMethod; the table-based ones keep only the gathered
// tensor's centroids in the replicated table (128-byte rows), the LUT or the
// bins in `aux` (the LUT method's merge buffer shares it), and the bins
// method's fp32 V codebook after them.
__host__ __device__ inline DecodeSmem decode_smem(int k_bits, int v_bits, int group, int k_row,
                                                  int v_row, int nstage, int warps, int stage_tok,
                                                  int append_enc = 0, int method = 0, int res_tok = 0) {
  DecodeSmem s;
  int o = 0;
  const int rows = 1 << (k_bits > v_bits ? k_bits : v_bits);
  s.tab = o; o = align128(o + rows * (k_bits == 12 ? kTabRowWide : method ? kTabRow / 2 : kTabRow));
  s.qt = o; o = align128(o + (group > 4 ? 8 : 4) * 128 * 4);  // q~ operand table, 4 or 8 heads
  // the merge buffer also holds a unit's residual window tokens (res_tok of
  // them at a time: K and V rows, then the raw queries)
  const int merge = method ? 0 : warps * group * 128 * 4;
  const int res = res_tok ? 2 * res_tok * 256 + 8 * 256 : 0;
  s.merge = o; o = align128(o + (merge > res ? merge : res));
  s.ml = o; o = align128(o + warps * (group > 4 ? 8 : 4) * 8);
  s.units = o; o = align128(o + 3 * kMaxUnitsPerCta * 4);  // lengths (consumers, producers), window lengths
  s.meta = o; o = align128(o + nstage * 16);
  s.bar = o; o = align128(o + (nstage * 2 + 1) * 8);  // full and empty per slot, then the append's
  s.flag = o; o = align128(o + 64);  // abort flag, then the CTA's length-balanced unit range
  s.enc = o; o = align128(o + append_enc);
  s.aux = o; o = align128(o + (method ? kLutBytes : 0) + (method == 2 ? (1 << v_bits) * 4 * 4 : 0));
  s.res = s.merge;
  s.stage = o; o = align128(o + nstage * stage_tok * (k_row + v_row));
  s.total = o;
  return s;
}

// Launches `kern`.  With `overlap` the launch carries programmatic stream
// serialization: the kernel may start while the previous kernel in the stream
// still runs, once that kernel has signalled pdl_trigger (see pdl_wait in
// vq_device.cuh).  Without it the kernel starts after all earlier work in the
// stream has completed.  The first kernel of every public call is launched
// without `overlap`, so nothing a caller's kernel writes can be read early;
// only the later kernels of the same call overlap their predecessor, whose
// early start already followed the completion of everything before the call.
template <typename Params>
inline cudaError_t launch_pdl(void (*kern)(Params), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, const Params& p, bool overlap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

constexpr int kMaxDevices = 64;

// The dynamic shared-memory size one kernel has been opted in to, per device
// (cudaFuncSetAttribute acts on the current device only).
struct SmemOptIn {
  std::mutex mu;
  std::atomic<size_t> bytes[kMaxDevices] = {};
};

// Raises `kern`'s dynamic shared-memory limit on the current device to at
// least `smem` bytes and prefers the largest shared-memory carveout, once per
// device and size.  Thread-safe.
template <typename K>
inline cudaError_t ensure_smem(K kern, size_t smem, SmemOptIn& st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (smem <= st.bytes[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(st.mu);
  if (smem <= st.bytes[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) st.bytes[dev].store(smem, std::memory_order_release);
  return e;
}

// Launchers (return the cudaError_t of the launch).
cudaError_t launch_encode(const EncodeParams& p, int grid_x, int grid_y, size_t smem,
                          cudaStream_t stream, bool overlap);
size_t encode_smem_bytes(int sub, int bits);
// The merge of a sliced append's candidates: one warp per (vector, tensor).
cudaError_t launch_encode_merge(const EncodeParams& p, int vectors, int grid_y, cudaStream_t stream);
constexpr int kAppendSlices = 8;  // CTAs per vector for appends with 1024 or more centroids

// Returns cudaErrorInvalidValue when no kernel is compiled for the formats.
// launch_decode takes either assignment (p.balanced); launch_decode_balanced
// is its length-balanced half.
cudaError_t launch_decode(const DecodeParams& p, int k_sub, int k_bits, int v_sub, int v_bits,
                          int grid, size_t smem, cudaStream_t stream, bool overlap,
                          int method = kMethodGather);
cudaError_t launch_decode_balanced(const DecodeParams& p, int k_sub, int k_bits, int v_sub, int v_bits,
                                   int grid, size_t smem, cudaStream_t stream, bool overlap, int method);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool overlap);
cudaError_t launch_dequant(const DequantParams& p, int grid_x, cudaStream_t stream);
int dequant_tokens_per_cta();

}  // namespace vqk
