/*
 * vqattn.h -- C ABI of the GB300 (sm_103a) VQ KV-cache decode-attention library.
 *
 * The method is VecInfer's ("VecInfer: Efficient LLM Inference With Low-Bit KV
 * Cache via Outlier-Suppressed Vector Quantization", papercache.org summary):
 *   - keys are smoothed per channel and Walsh-Hadamard transformed,
 *     K~ = K diag(lambda)^-1 H_D  (section 方法细节, "异常值抑制的向量量化");
 *   - transformed keys and raw values are vector-quantized: every d-long
 *     sub-vector is replaced by the b-bit index of its nearest codebook
 *     centroid (section 背景知识, "向量量化原理");
 *   - a decode query is transformed to q~ = q diag(lambda) H_D and attends
 *     directly over the codes:  s = q~ VQ^-1(K~_q)^T * scale, p = softmax(s),
 *     o = p VQ^-1(V_q)  (section 方法细节, "注意力机制中的向量量化KV缓存").
 *
 * Conventions shared by every call:
 *   - All tensor arguments are DEVICE pointers to caller-owned memory unless a
 *     parameter says "host".  The library never allocates or frees memory.
 *   - Every call is asynchronous and ordered on the CUDA stream `stream`
 *     (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *     No call synchronises the device.
 *   - The first kernel of every call starts after all earlier work on
 *     `stream` has completed, as with any plain launch, so the call sees
 *     everything the caller wrote before it.  Later kernels of the same call
 *     (the attention kernel after the append of vq_decode_step, the merge
 *     after the attention kernel) are launched with programmatic stream
 *     serialization: each may start while its predecessor in the call runs,
 *     reading only the call's inputs early, and reads what its predecessor
 *     writes only after that kernel has completed.  A caller's kernel
 *     launched after a call with programmatic serialization must wait
 *     (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads
 *     the call's outputs, as the CUDA programming model requires.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns a negative vq_status and launches nothing.
 *     vq_last_error() then describes the failure (thread-local string).
 *   - Device-detected failures (an out-of-range page or slot index, a
 *     pipeline wait that timed out) never fault the GPU: the kernel skips the
 *     access and stores a nonzero vq_device_status code into `*status` (first
 *     error wins) when `status` is non-NULL.  The caller zeroes the word and
 *     reads it after synchronising.
 *   - fp16 means IEEE binary16, fp32 IEEE binary32, all little-endian, rows
 *     contiguous (C order).  Device buffers must be 16-byte aligned.
 *
 * Cache layout ("pool"): one pool for K codes and one for V codes, each
 *   [num_pages][num_kv_heads][page_size][row_bytes]  bytes,
 * where row_bytes = vq_code_row_bytes(head_dim, sub, bits).  Token t of a
 * sequence lives in logical page t / page_size at offset t % page_size; the
 * page table maps logical pages to physical pages.  A row holds the
 * head_dim / sub codes of one token-head as a bit stream: code i occupies bits
 * [i*bits, (i+1)*bits), least significant bit first (bit m of the stream is bit
 * m % 8 of byte m / 8); trailing bits are zero.
 */
#ifndef VQATTN_H
#define VQATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vq_status {
  VQ_OK = 0,
  VQ_ERR_INVALID_ARG = -1,   /* null pointer, bad shape, misaligned buffer ... */
  VQ_ERR_UNSUPPORTED = -2,   /* valid but not implemented (e.g. head_dim != 128) */
  VQ_ERR_WORKSPACE = -3,     /* workspace smaller than vq_decode_workspace_bytes() */
  VQ_ERR_CUDA = -4           /* a CUDA runtime call or launch failed */
} vq_status;

/* Codes a kernel stores into the optional device status word. */
typedef enum vq_device_status {
  VQ_DEV_OK = 0,
  VQ_DEV_BAD_PAGE = 1,       /* page_table entry outside [0, num_pages): page skipped */
  VQ_DEV_BAD_SLOT = 2,       /* slot_mapping entry >= num_pages * page_size: token skipped */
  VQ_DEV_TIMEOUT = 3,        /* an asynchronous-copy wait exceeded its time limit */
  VQ_DEV_BAD_CONFIG = 4      /* launch parameters the kernel cannot honour: it did nothing
                                (not reachable through this ABI's validated calls) */
} vq_device_status;

/*
 * Shape of one attention layer's quantized KV cache (host struct, read during
 * the call only).
 *   head_dim      D; a power of two.  This build implements D = 128.
 *   num_q_heads   Hq; query head h reads KV head h / (Hq / Hkv).
 *   num_kv_heads  Hkv; Hq % Hkv == 0 and Hq / Hkv <= 8.
 *   k_sub,k_bits  d_k, b_k: K sub-vector length and bits per code (2^b_k
 *                 centroids).  d_k divides D.
 *   v_sub,v_bits  d_v, b_v: the same for V.
 *   page_size     tokens per page, a multiple of 16.
 */
typedef struct vq_layout {
  int32_t head_dim;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t k_sub;
  int32_t k_bits;
  int32_t v_sub;
  int32_t v_bits;
  int32_t page_size;
} vq_layout;

/*
 * Bytes of one packed code row: ceil((head_dim / sub) * bits / 8) rounded up
 * to a multiple of 4.  Index storage follows VecInfer, section 背景知识,
 * "向量量化原理": (d_h / d) * (b / 8) bytes of indices per vector.
 * Returns 0 for an invalid combination.
 */
size_t vq_code_row_bytes(int32_t head_dim, int32_t sub, int32_t bits);

/*
 * Checks a layout against what this build implements.  VQ_OK, or
 * VQ_ERR_INVALID_ARG / VQ_ERR_UNSUPPORTED with vq_last_error() set.
 * Encode supports sub in {1, 2, 4, 8} and bits in 1..12; decode attention
 * supports (k_sub, k_bits) in {(2, 8), (4, 8)} with (v_sub, v_bits) in
 * {(2, 8), (4, 8), (4, 9)}, and the 1.5-bit format (8, 12) with (8, 12)
 * (VecInfer, 实验结果, codebook-size ablation: 2^12 centroids of 8 elements).
 */
vq_status vq_check_layout(const vq_layout* layout, int32_t for_decode);

/*
 * Encode K/V tokens into the code pools (the cache fill of VecInfer, section
 * 方法细节 "注意力机制中的向量量化KV缓存": prefill encodes every token, decode
 * encodes each new token and appends its codes).
 *   For each token t and KV head h:
 *     k~ = (k[t][h] / lambda[h]) H_D      (fp32 arithmetic, fast WHT)
 *     K code i = argmin_j ||k~_i - C_k[j]||^2, V code i likewise on raw v
 *     (lowest index on an exact tie), packed into row
 *     pool[slot / P][h][slot % P] with slot = slot_mapping[t].
 *   k, v          fp16 [num_tokens][Hkv][D].  Either may be NULL (that half is
 *                 not encoded), not both.
 *   slot_mapping  int64 [num_tokens].  A negative slot skips the token; a slot
 *                 >= num_pages * P skips it and reports VQ_DEV_BAD_SLOT.
 *   lambda        fp32 [Hkv][D] smoothing factors (lambda, not 1/lambda),
 *                 all > 0.  Required when k is non-NULL.
 *   codebook_k    fp16 [2^k_bits][k_sub]; codebook_v fp16 [2^v_bits][v_sub].
 *   k_pool,v_pool pools as described above, num_pages pages each.
 *   status        optional device int32 status word.
 * num_tokens == 0 is a no-op returning VQ_OK.
 */
vq_status vq_encode_kv(const vq_layout* layout, int32_t num_tokens,
                       const void* k, const void* v, const int64_t* slot_mapping,
                       const float* lambda, const void* codebook_k, const void* codebook_v,
                       void* k_pool, void* v_pool, int64_t num_pages,
                       int32_t* status, void* stream);

/*
 * Dequantise cached tokens back to fp16 keys and values in their original
 * spaces: the inverse of vq_encode_kv up to the quantisation error (VecInfer,
 * section 方法细节: a vector is read back as the concatenation of the
 * centroids its codes name, "注意力机制中的向量量化KV缓存"; keys were coded as
 * K~ = K diag(lambda)^-1 H_D, "Hadamard引理与注意力分数重写", and H_D is
 * symmetric and orthonormal).  This is the first half of an unfused pipeline
 * (dequantise, then dense attention), the baseline the VecInfer page compares
 * its fused kernel against (实验结果, 图5).
 *   For each token t and KV head h, with slot = slot_mapping[t]:
 *     k_out[t][h] = VQ^-1(K code row) H_D diag(lambda[h])  (fp32, rounded to fp16)
 *     v_out[t][h] = VQ^-1(V code row)                       (exact fp16 centroids)
 *   k_out, v_out  fp16 [num_tokens][Hkv][D], written in full.  Either may be
 *                 NULL (that half is not produced), not both.
 *   slot_mapping  int64 [num_tokens].  A negative slot gives zero rows; a slot
 *                 >= num_pages * P gives zero rows and reports VQ_DEV_BAD_SLOT.
 *   lambda        fp32 [Hkv][D]; required when k_out is non-NULL.
 *   codebooks, pools, num_pages, status: as in vq_encode_kv (the pools are
 *                 only read).
 * Supports every format vq_encode_kv supports.  Launched without programmatic
 * overlap: it starts after the previous work on `stream` has completed.
 * num_tokens == 0 is a no-op returning VQ_OK.
 */
vq_status vq_dequantize_kv(const vq_layout* layout, int32_t num_tokens,
                           const int64_t* slot_mapping, const float* lambda,
                           const void* codebook_k, const void* codebook_v, const void* k_pool,
                           const void* v_pool, int64_t num_pages, void* k_out, void* v_out,
                           int32_t* status, void* stream);

/*
 * Workspace bytes vq_decode_attention (and vq_decode_step) needs for `batch`
 * sequences split `num_splits` ways (num_splits <= 0: the value
 * vq_default_num_splits picks): the split partials, one int32 per
 * (sequence, KV head) for the partial count of length-balanced units, and
 * for codebooks of 1024 centroids or more (10- to 12-bit codes) also the
 * candidates of vq_decode_step's append, which spreads each new vector's
 * codebook scan over several CTAs.  Pure host arithmetic.  Returns 0 for
 * invalid arguments.
 */
size_t vq_decode_workspace_bytes(const vq_layout* layout, int32_t batch,
                                 int32_t max_seq_len, int32_t num_splits, int32_t num_sms);

/*
 * Split-K factor the library picks for a batch (num_sms <= 0: query the
 * current device).  One sequence: the number of splits per (sequence, KV
 * head) that balances work units over num_sms SMs.  Two or more sequences
 * (up to 512): 1 + ceil(2 num_sms / (batch * Hkv)) partial slots per
 * (sequence, KV head) for length-balanced units, where every SM gets an
 * equal share of the batch's 32-token blocks whatever the lengths (the
 * fixed-split count when that assignment's bounds do not hold).  Returns
 * >= 1, or 0 on error.
 */
int32_t vq_default_num_splits(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                              int32_t num_sms);

/*
 * How the decode kernels divide the work of `batch` sequences for these
 * arguments (num_splits <= 0: vq_default_num_splits' choice; num_sms <= 0:
 * the current device): 1 for length-balanced units (the batch's 32-token
 * blocks divided evenly over the SMs; a (sequence, KV head) then has between
 * 1 and num_splits partials), 0 for fixed splits (num_splits ranges of
 * max_seq_len per sequence).  Pure host arithmetic.  Returns -1 for invalid
 * arguments.
 */
int32_t vq_decode_units_balanced(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                                 int32_t num_splits, int32_t num_sms);

/*
 * Decode attention for one query token per sequence over the quantized cache
 * (VecInfer, section 方法细节 "注意力机制中的向量量化KV缓存"; split-K with an
 * online-softmax merge as in the FlashAttention recurrence of the appendix
 * "相关工作 - FlashAttention").
 *   q            fp16 [batch][Hq][D] decode queries (untransformed).
 *   lambda       fp32 [Hkv][D] smoothing factors used when the keys were encoded.
 *   codebook_k/v fp16 codebooks used when the caches were encoded.
 *   k_pool/v_pool the pools (num_pages pages each).
 *   page_table   int32 [batch][max_pages_per_seq]: logical -> physical page.
 *   seq_lens     int32 [batch]: tokens each query attends to (cached plus
 *                appended); 0 gives a zero output row.
 *   max_seq_len  host upper bound of seq_lens, used to size the split grid;
 *                tokens beyond it are ignored.  With one sequence (fixed
 *                splits) the split boundaries are fractions of it, so a tight
 *                bound spreads the work best; with two or more the kernel
 *                divides the batch's actual blocks.
 *   softmax_scale multiplies the scores; 0 selects 1/sqrt(D).
 *   num_splits   partials per (sequence, KV head); <= 0 selects the
 *                library's choice.  With one sequence (or num_splits 1) each
 *                sequence is cut into num_splits ranges of max_seq_len;
 *                with two or more, the batch's blocks are divided evenly
 *                over the SMs and a (sequence, KV head) meets at most
 *                num_splits of them.  Results do not depend on it beyond
 *                fp32 rounding.
 *   out          fp16 [batch][Hq][D] attention output.
 *   workspace    device scratch of at least vq_decode_workspace_bytes(...)
 *                bytes (fp32 partial results of the splits); 256-byte aligned.
 *   status       optional device int32 status word.
 * Two kernels are launched on `stream`: the split attention kernel and the
 * split-combine kernel.
 */
vq_status vq_decode_attention(const vq_layout* layout, int32_t batch, const void* q,
                              const float* lambda, const void* codebook_k,
                              const void* codebook_v, const void* k_pool, const void* v_pool,
                              int64_t num_pages, const int32_t* page_table,
                              int32_t max_pages_per_seq, const int32_t* seq_lens,
                              int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                              void* out, void* workspace, size_t workspace_bytes,
                              int32_t* status, void* stream);

/*
 * The two halves of vq_decode_attention, for callers that schedule them
 * separately (for example to overlap the combine with other work):
 *   vq_decode_partial  takes the arguments of vq_decode_attention except `out`
 *                      and launches only the split attention kernel, which
 *                      writes one (max, sum, unnormalised output) partial per
 *                      (sequence, query head, split) into the workspace;
 *   vq_decode_combine  launches only the merge of those partials into `out`
 *                      (fp16 [batch][Hq][D]).
 * Both must be called with the same layout, batch, max_seq_len, num_splits and
 * workspace, on the same device and stream order; num_splits <= 0 resolves to
 * the same value in both calls.
 */
vq_status vq_decode_partial(const vq_layout* layout, int32_t batch, const void* q,
                            const float* lambda, const void* codebook_k, const void* codebook_v,
                            const void* k_pool, const void* v_pool, int64_t num_pages,
                            const int32_t* page_table, int32_t max_pages_per_seq,
                            const int32_t* seq_lens, int32_t max_seq_len, float softmax_scale,
                            int32_t num_splits, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream);

vq_status vq_decode_combine(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                            int32_t num_splits, const void* workspace, size_t workspace_bytes,
                            void* out, void* stream);

/*
 * Score and P.V methods of the split attention kernel.  The pages name two
 * ways for each half of the attention over codes (VecInfer, 内核实现细节 -
 * 融合内核, Algorithm 1: a lookup table of query x K-codebook products summed
 * over the codes; CommVQ, 降低计算复杂度: Softmax(A) S_V C_V, i.e. P.V by
 * accumulating p into per-code bins and multiplying by the V codebook once):
 *   VQ_METHOD_GATHER  scores and P.V from in-register centroid gathers on the
 *                     tensor cores (what every other call uses);
 *   VQ_METHOD_LUT     scores from the table LUT[i][j] = q~_i . C_k[j] (fp32,
 *                     built per work unit), P.V by gather;
 *   VQ_METHOD_BINS    scores by gather, P.V through fp32 bins[i][j] += p,
 *                     o_i = sum_j bins[i][j] C_v[j] at the end of each unit.
 */
typedef enum vq_decode_method {
  VQ_METHOD_GATHER = 0,
  VQ_METHOD_LUT = 1,
  VQ_METHOD_BINS = 2
} vq_decode_method;

/*
 * vq_decode_partial with an explicit method (above), for measuring the
 * methods against each other; vq_decode_combine then merges the partials as
 * usual.  The results agree with every method's within fp32 rounding (the
 * bins method adds in an order that varies from run to run).  The table-based
 * methods are built for k_sub = v_sub = 4 with 8-bit codes and
 * num_q_heads / num_kv_heads <= 4; other layouts return VQ_ERR_UNSUPPORTED.
 * The bins method keeps one reference maximum per head for the whole work
 * unit, agreed between the warps at every pipeline stage.
 */
vq_status vq_decode_partial_method(const vq_layout* layout, int32_t batch, const void* q,
                                   const float* lambda, const void* codebook_k,
                                   const void* codebook_v, const void* k_pool, const void* v_pool,
                                   int64_t num_pages, const int32_t* page_table,
                                   int32_t max_pages_per_seq, const int32_t* seq_lens,
                                   int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                                   int32_t method, void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream);

/*
 * One decode step: append each sequence's new token to the cache, then decode
 * attention over the cache with the new token included (VecInfer, section
 * 方法细节 "注意力机制中的向量量化KV缓存": during decoding the new key and value
 * are encoded and appended, then the query attends over the quantized cache).
 * Exactly the results of vq_encode_kv of the new tokens followed by
 * vq_decode_attention with the same split count, without a slot mapping: the
 * slots come from the page table.  Two ways, chosen by the library and equal
 * bit for bit:
 *   - with at most one sequence-KV-head pair per SM, the attention kernel
 *     itself appends each new token (the producer warps of the CTA whose
 *     split holds it encode it while their first copies are in flight, and
 *     store the codes; the stage that holds the token is copied only after
 *     the store), then the merge: two kernels (the fused append of HACK's
 *     decode kernel and of VecInfer's 注意力机制中的向量量化KV缓存, where the new
 *     code joins the cached ones).  For the 1.5-bit format (4096 centroids)
 *     a kernel first scans each new vector's codebooks over several CTAs and
 *     leaves their candidates in the workspace, which the attention kernel's
 *     producers merge: three kernels;
 *   - otherwise three kernels: the append encode, the split attention (it
 *     starts while the append runs, prepares its tables, and waits for the
 *     append before it reads the pools) and the merge; with 10- to 12-bit
 *     codes the append is two kernels (each new vector's codebook scan split
 *     over several CTAs whose candidates sit in the workspace, then their
 *     merge and the store).
 *   k_new, v_new fp16 [batch][Hkv][D]: the new token of every sequence.  It is
 *                token seq_lens[b] - 1 of sequence b and goes to slot
 *                page_table[b][t / P] * P + t % P of the pools
 *                (t = seq_lens[b] - 1).  seq_lens[b] == 0 appends nothing and
 *                gives a zero output row.  An out-of-range page for the new
 *                token reports VQ_DEV_BAD_PAGE; it is neither stored nor
 *                attended.
 *   k_pool, v_pool are written (the new rows) as well as read.
 *   workspace    at least vq_decode_workspace_bytes(layout, batch,
 *                max_seq_len, num_splits, 0) bytes, 256-byte aligned; no
 *                initialisation needed.
 * All other arguments, the split choice for num_splits <= 0 and the errors are
 * those of vq_decode_attention.
 */
vq_status vq_decode_step(const vq_layout* layout, int32_t batch, const void* q, const void* k_new,
                         const void* v_new, const float* lambda, const void* codebook_k,
                         const void* codebook_v, void* k_pool, void* v_pool, int64_t num_pages,
                         const int32_t* page_table, int32_t max_pages_per_seq,
                         const int32_t* seq_lens, int32_t max_seq_len, float softmax_scale,
                         int32_t num_splits, void* out, void* workspace, size_t workspace_bytes,
                         int32_t* status, void* stream);

/*
 * Decode attention over a quantized cache plus a full-precision residual
 * window of the most recent tokens (VecInfer, section 实验结果 / 实验设置:
 * every method keeps a residual of 128 unquantized tokens).  The quantized
 * tokens score as in vq_decode_attention (s = q~ VQ^-1(K~_q)^T * scale); a
 * residual token scores with the raw query and key, s = q k^T * scale, and
 * both join one softmax: o = softmax(s) [VQ^-1(V_q); V_res].
 *   seq_lens      int32 [batch]: quantized tokens of each sequence (as in
 *                 vq_decode_attention; 0 is allowed).
 *   k_res, v_res  fp16 [batch][Hkv][res_capacity][D]: the residual tokens of
 *                 sequence b and KV head h are rows 0 .. res_lens[b] - 1 of
 *                 [b][h] (their order does not matter).
 *   res_lens      int32 [batch], clamped to [0, res_capacity].
 *   res_capacity  1 .. 4096.
 *   workspace     at least vq_decode_residual_workspace_bytes(layout, batch,
 *                 max_seq_len, num_splits, 0) bytes (the same as
 *                 vq_decode_workspace_bytes: the window joins the split
 *                 partials), 256-byte aligned; no initialisation needed.
 * Two kernels on `stream`: the split attention over the codes, in which the
 * work unit of split s of each (sequence, KV head) also merges window tokens
 * [s R / S, (s + 1) R / S) (R = res_lens[b], S splits) into its own partial
 * with the same online softmax, and the merge of the splits.  Moving tokens
 * from the residual into
 * the cache (vq_encode_kv) is the caller's policy.  Other arguments and errors
 * as in vq_decode_attention.  A sequence with no token at all gives a zero
 * row.
 */
size_t vq_decode_residual_workspace_bytes(const vq_layout* layout, int32_t batch,
                                          int32_t max_seq_len, int32_t num_splits,
                                          int32_t num_sms);

vq_status vq_decode_attention_residual(const vq_layout* layout, int32_t batch, const void* q,
                                       const float* lambda, const void* codebook_k,
                                       const void* codebook_v, const void* k_pool,
                                       const void* v_pool, int64_t num_pages,
                                       const int32_t* page_table, int32_t max_pages_per_seq,
                                       const int32_t* seq_lens, int32_t max_seq_len,
                                       const void* k_res, const void* v_res,
                                       const int32_t* res_lens, int32_t res_capacity,
                                       float softmax_scale, int32_t num_splits, void* out,
                                       void* workspace, size_t workspace_bytes, int32_t* status,
                                       void* stream);

/*
 * Decode attention for callers that cannot allocate device memory.
 *
 * No counterpart on the VecInfer pages: this is a deployment variant of
 * vq_decode_attention.  Some callers cannot hand the library a workspace:
 * code running where device allocation is not allowed (or would synchronise
 * the device), embedders whose memory belongs to an allocator they cannot
 * call, and plug-ins that receive only the tensors of one call.  This entry
 * point takes the same arguments as vq_decode_attention minus the workspace
 * and keeps the split partials in a fixed device array inside the library
 * instead, so it allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library call).
 *   - The array holds vq_static_scratch_bytes() bytes (4 MiB) on every GPU
 *     that loads the library, until the process exits.  With num_splits <= 0
 *     the library's split choice is lowered until the partials fit; a request
 *     that does not fit even so (or an explicit num_splits whose
 *     vq_decode_workspace_bytes() exceeds the array) returns
 *     VQ_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks the array's device address up with
 *     cudaGetSymbolAddress (once per device and CUDA context, for the device
 *     that is current); make that first call before any stream capture, and
 *     again after a cudaDeviceReset.
 *   - All calls on a device share the one array, which keeps the contents of
 *     the last call.  Nothing in it has to start at zero: the split kernel
 *     writes every partial the combine reads.  Calls whose kernels overlap on
 *     the GPU (different streams without ordering, or several host threads)
 *     race on the array and give wrong results; serialise them.
 * Arguments, validation and outputs are those of vq_decode_attention.
 */
vq_status vq_decode_attention_static(const vq_layout* layout, int32_t batch, const void* q,
                                     const float* lambda, const void* codebook_k,
                                     const void* codebook_v, const void* k_pool,
                                     const void* v_pool, int64_t num_pages,
                                     const int32_t* page_table, int32_t max_pages_per_seq,
                                     const int32_t* seq_lens, int32_t max_seq_len,
                                     float softmax_scale, int32_t num_splits, void* out,
                                     int32_t* status, void* stream);

/* Bytes of the fixed device array vq_decode_attention_static uses. */
size_t vq_static_scratch_bytes(void);

/* Human-readable description of the last non-OK status on this host thread. */
const char* vq_last_error(void);

/* Library version string, e.g. "vqattn 0.1.0 sm_103a". */
const char* vq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VQATTN_H */
