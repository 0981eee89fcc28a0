// vq_api.cu -- the extern "C" boundary (include/vqattn.h): argument checks,
// launch-shape choice and kernel launches.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/vqattn.h"
#include "vq_kernels.h"

namespace {

thread_local std::string g_last_error;

vq_status fail(vq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

vq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(VQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Device attributes the launch choices need, read once per device.
struct DeviceAttrs {
  std::atomic<int> sms[vqk::kMaxDevices] = {};
  std::atomic<int> smem_optin[vqk::kMaxDevices] = {};
};
DeviceAttrs g_attrs;

int device_attr(std::atomic<int>* cache, cudaDeviceAttr attr) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= vqk::kMaxDevices) return 0;
  n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, attr, dev) != cudaSuccess) return 0;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

int device_sms() { return device_attr(g_attrs.sms, cudaDevAttrMultiProcessorCount); }

int device_smem_optin() {
  return device_attr(g_attrs.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin);
}

bool decode_formats_supported(const vq_layout& L) {
  const bool k_ok = (L.k_sub == 2 || L.k_sub == 4) && L.k_bits == 8;
  const bool v_ok = (L.v_sub == 4 && (L.v_bits == 8 || L.v_bits == 9)) ||
                    (L.v_sub == 2 && L.v_bits == 8);
  const bool wide = L.k_sub == 8 && L.k_bits == 12 && L.v_sub == 8 && L.v_bits == 12;
  return (k_ok && v_ok) || wide;
}

constexpr int kMaxSplits = 4096;
constexpr int kMaxResidual = 4096;  // residual window capacity (tokens)

// Largest value the length-balanced kernel's slot term of W,
// ceil(longest pair's blocks / (splits - 1)), can take: the pairs' blocks
// are at most ceil(max_seq_len / 32).
int balance_wmin(int max_seq_len, int splits) {
  const int nsl = (max_seq_len + vqk::kUnitTok - 1) / vqk::kUnitTok;
  return (nsl + splits - 2) / (splits - 1);
}

// Length-balanced units (decode kernel, DecodeParams::balanced) for batches
// of two or more sequences: the grid (one CTA per SM) splits the pairs' blocks
// evenly whatever the lengths.  Needs two or more partial slots per pair and
// at most kMaxUnitsPerCta units per CTA, which holds with at most that many
// pairs or with a per-CTA range W <= (kMaxUnitsPerCta - 2) (1 + kBalanceGap)
// (pairs after a CTA's first start inside its range, 1 + kBalanceGap
// positions apart at least); the kernel's W is at most the bound taken here
// from max_seq_len.
bool balanced_units(const vq_layout& L, int batch, int max_seq_len, int splits, int sms) {
  if (batch < 2 || batch > vqk::kBalanceMaxBatch || splits < 2 || sms <= 0 || max_seq_len < 1) return false;
  const long long pairs = static_cast<long long>(batch) * L.num_kv_heads;
  const long long nsl = (static_cast<long long>(max_seq_len) + vqk::kUnitTok - 1) / vqk::kUnitTok;
  const long long total = pairs * (nsl + vqk::kBalanceGap);  // the largest total the kernel can see
  if (total >= (1LL << 30)) return false;
  const long long w = std::max<long long>((total + sms - 1) / sms, balance_wmin(max_seq_len, splits));
  return pairs <= vqk::kMaxUnitsPerCta ||
         w <= static_cast<long long>(vqk::kMaxUnitsPerCta - 2) * (1 + vqk::kBalanceGap);
}

// Split count.  Batches of two or more sequences: length-balanced units with
// 1 + ceil(2 SMs / pairs) slots per pair (a pair may be twice the average
// length before the slot term, rather than the total, sets the CTA range).
// Otherwise the count minimising an estimate of the persistent grid's
// makespan: waves(units) * (tokens per unit + fixed per-unit cost).
int pick_splits(const vq_layout& L, int batch, int max_seq_len, int sms) {
  const long long pairs = static_cast<long long>(batch) * L.num_kv_heads;
  const long long chunks = (static_cast<long long>(max_seq_len) + 15) / 16;
  if (pairs <= 0 || chunks <= 0 || sms <= 0) return 1;
  if (batch >= 2) {
    const int sb = static_cast<int>(std::min<long long>(1 + (2LL * sms + pairs - 1) / pairs, kMaxSplits));
    if (balanced_units(L, batch, max_seq_len, sb, sms)) return sb;
  }
  const double kUnitOverhead = 384.0;  // tokens-equivalent per unit (q~, merge, pipeline fill)
  int best = 1;
  double best_cost = 1e300;
  const long long smax = std::min<long long>(kMaxSplits, chunks);
  for (long long s = 1; s <= smax; ++s) {
    const long long units = pairs * s;
    if ((units + sms - 1) / sms > vqk::kMaxUnitsPerCta) break;
    const double waves = static_cast<double>((units + sms - 1) / sms);
    const double per_unit = std::ceil(static_cast<double>(chunks) / s) * 16.0 + kUnitOverhead;
    const double cost = waves * per_unit + 8.0 * s;  // combine reads grow with s
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = static_cast<int>(s);
    }
  }
  return best;
}

// Codebooks of 1024 centroids or more: the decode step's append is spread
// over kAppendSlices CTAs per vector.
bool sliced_append(const vq_layout& L) { return L.k_bits >= 10 || L.v_bits >= 10; }

struct WsLayout {
  size_t o_off, ml_off, cnt_off, cand_off, total;
};

// Split partials, the units per (sequence, KV head) of length-balanced
// units, then (large codebooks) the sliced append's candidates.
WsLayout ws_layout(const vq_layout& L, int batch, int splits) {
  WsLayout w;
  const size_t rows = static_cast<size_t>(batch) * L.num_q_heads * splits;
  w.o_off = 0;
  w.ml_off = (rows * L.head_dim * sizeof(float) + 255) & ~size_t(255);
  w.cnt_off = w.ml_off + ((rows * 2 * sizeof(float) + 255) & ~size_t(255));
  w.cand_off = w.cnt_off + ((static_cast<size_t>(batch) * L.num_kv_heads * sizeof(int) + 255) & ~size_t(255));
  const size_t cand = sliced_append(L) ? static_cast<size_t>(batch) * L.num_kv_heads * 2 *
                                             vqk::kAppendSlices * 32 * 4 * sizeof(int2)
                                       : 0;
  w.total = w.cand_off + cand;
  return w;
}

vq_status check_layout_impl(const vq_layout* L, int for_decode) {
  if (!L) return fail(VQ_ERR_INVALID_ARG, "layout is NULL");
  if (!is_pow2(L->head_dim)) return fail(VQ_ERR_INVALID_ARG, "head_dim %d is not a power of two", L->head_dim);
  if (L->head_dim != 128)
    return fail(VQ_ERR_UNSUPPORTED, "head_dim %d: this build implements head_dim 128", L->head_dim);
  if (L->num_q_heads < 1 || L->num_kv_heads < 1 || L->num_q_heads % L->num_kv_heads)
    return fail(VQ_ERR_INVALID_ARG, "num_q_heads %d must be a positive multiple of num_kv_heads %d",
                L->num_q_heads, L->num_kv_heads);
  if (L->num_q_heads / L->num_kv_heads > 8)
    return fail(VQ_ERR_UNSUPPORTED, "query group %d > 8", L->num_q_heads / L->num_kv_heads);
  const int subs[2] = {L->k_sub, L->v_sub}, bits[2] = {L->k_bits, L->v_bits};
  for (int i = 0; i < 2; ++i) {
    if (!(subs[i] == 1 || subs[i] == 2 || subs[i] == 4 || subs[i] == 8))
      return fail(VQ_ERR_INVALID_ARG, "%s_sub %d not in {1, 2, 4, 8}", i ? "v" : "k", subs[i]);
    if (bits[i] < 1 || bits[i] > 12)
      return fail(VQ_ERR_INVALID_ARG, "%s_bits %d not in 1..12", i ? "v" : "k", bits[i]);
  }
  if (L->page_size < 16 || L->page_size % 16)
    return fail(VQ_ERR_INVALID_ARG, "page_size %d must be a positive multiple of 16", L->page_size);
  if (for_decode && !decode_formats_supported(*L))
    return fail(VQ_ERR_UNSUPPORTED,
                "decode attention implements (k_sub,k_bits) in {(2,8),(4,8)} with (v_sub,v_bits) "
                "in {(2,8),(4,8),(4,9)}, and (8,12) with (8,12); got (%d,%d) and (%d,%d)",
                L->k_sub, L->k_bits, L->v_sub, L->v_bits);
  return VQ_OK;
}

}  // namespace

extern "C" {

size_t vq_code_row_bytes(int32_t head_dim, int32_t sub, int32_t bits) {
  if (head_dim <= 0 || sub <= 0 || head_dim % sub || bits < 1 || bits > 16) return 0;
  const size_t n = static_cast<size_t>(head_dim / sub) * bits;
  return ((n + 7) / 8 + 3) / 4 * 4;
}

vq_status vq_check_layout(const vq_layout* layout, int32_t for_decode) {
  return check_layout_impl(layout, for_decode);
}

// Launches the encode of num_tokens tokens: the caller has set the sources,
// codebooks, pools, lambda, the slot source and the status word; the launch
// shape follows from the number of vectors.
vq_status launch_encode_impl(const vq_layout& L, vqk::EncodeParams& p, int32_t num_tokens,
                             bool has_k, bool has_v, void* stream, const char* what,
                             bool overlap, int2* cand = nullptr, bool merge_kernel = true) {
  p.sub[0] = L.k_sub;
  p.sub[1] = L.v_sub;
  p.bits[0] = L.k_bits;
  p.bits[1] = L.v_bits;
  p.row_bytes[0] = static_cast<int>(vq_code_row_bytes(L.head_dim, L.k_sub, L.k_bits));
  p.row_bytes[1] = static_cast<int>(vq_code_row_bytes(L.head_dim, L.v_sub, L.v_bits));
  p.num_tokens = num_tokens;
  p.hkv = L.num_kv_heads;
  p.page_size = L.page_size;
  const long long vectors = static_cast<long long>(num_tokens) * L.num_kv_heads;
  const int sms = device_sms();
  // few vectors (a decode-step append): spread each codebook scan over 8 warps
  p.split = vectors * 2 < static_cast<long long>(sms > 0 ? sms : 148) * 8 ? 8 : 1;
  // many vectors with sub-vector lengths 2 / 4: several vectors per warp
  const bool multi_ok = (!has_k || L.k_sub == 2 || L.k_sub == 4) && (!has_v || L.v_sub == 2 || L.v_sub == 4);
  p.vec_per_warp = (p.split == 1 && multi_ok) ? vqk::kMultiVec : 1;
  const int per_cta = 8 * p.vec_per_warp / p.split;
  // a few vectors of a large codebook (with candidate space): several CTAs each
  p.slices = (cand && p.split > 1 && sliced_append(L)) ? vqk::kAppendSlices : 1;
  p.cand = cand;
  const long long grid_x = (vectors + per_cta - 1) / per_cta * p.slices;
  if (grid_x > 0x7fffffffLL) return fail(VQ_ERR_INVALID_ARG, "too many tokens (%d)", num_tokens);
  p.which_base = has_k ? 0 : 1;
  const int grid_y = (has_k && has_v) ? 2 : 1;
  size_t smem = 0;
  if (has_k) smem = std::max(smem, vqk::encode_smem_bytes(L.k_sub, L.k_bits));
  if (has_v) smem = std::max(smem, vqk::encode_smem_bytes(L.v_sub, L.v_bits));
  const int optin = device_smem_optin();
  if (optin > 0 && smem > static_cast<size_t>(optin))
    return fail(VQ_ERR_UNSUPPORTED, "encode needs %zu bytes of shared memory, device has %d", smem, optin);
  cudaError_t e = vqk::launch_encode(p, static_cast<int>(grid_x), grid_y, smem,
                                     static_cast<cudaStream_t>(stream), overlap);
  if (e != cudaSuccess) return cuda_fail(e, what);
  if (p.slices > 1 && merge_kernel) {
    e = vqk::launch_encode_merge(p, static_cast<int>(vectors), grid_y, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, what);
  }
  return VQ_OK;
}

vq_status vq_encode_kv(const vq_layout* layout, int32_t num_tokens, const void* k, const void* v,
                       const int64_t* slot_mapping, const float* lambda, const void* codebook_k,
                       const void* codebook_v, void* k_pool, void* v_pool, int64_t num_pages,
                       int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 0);
  if (st != VQ_OK) return st;
  const vq_layout& L = *layout;
  if (num_tokens < 0) return fail(VQ_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (!k && !v) return fail(VQ_ERR_INVALID_ARG, "k and v are both NULL");
  if (!slot_mapping) return fail(VQ_ERR_INVALID_ARG, "slot_mapping is NULL");
  if (num_pages < 1) return fail(VQ_ERR_INVALID_ARG, "num_pages %lld < 1", (long long)num_pages);
  if (k && (!lambda || !codebook_k || !k_pool))
    return fail(VQ_ERR_INVALID_ARG, "k given but lambda, codebook_k or k_pool is NULL");
  if (v && (!codebook_v || !v_pool))
    return fail(VQ_ERR_INVALID_ARG, "v given but codebook_v or v_pool is NULL");
  const void* ptrs[] = {k, v, lambda, codebook_k, codebook_v, k_pool, v_pool, slot_mapping};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return fail(VQ_ERR_INVALID_ARG, "device buffer %p is not 16-byte aligned", ptr);
  if (num_tokens == 0) return VQ_OK;

  vqk::EncodeParams p{};
  p.src[0] = k;
  p.src[1] = v;
  p.cb[0] = codebook_k;
  p.cb[1] = codebook_v;
  p.pool[0] = static_cast<uint8_t*>(k_pool);
  p.pool[1] = static_cast<uint8_t*>(v_pool);
  p.lambda = lambda;
  p.slots = slot_mapping;
  p.status = status;
  p.num_slots = static_cast<long long>(num_pages) * L.page_size;
  return launch_encode_impl(L, p, num_tokens, k != nullptr, v != nullptr, stream,
                            "vq_encode_kv launch", false);
}

vq_status vq_dequantize_kv(const vq_layout* layout, int32_t num_tokens,
                           const int64_t* slot_mapping, const float* lambda,
                           const void* codebook_k, const void* codebook_v, const void* k_pool,
                           const void* v_pool, int64_t num_pages, void* k_out, void* v_out,
                           int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 0);
  if (st != VQ_OK) return st;
  const vq_layout& L = *layout;
  if (num_tokens < 0) return fail(VQ_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return VQ_OK;  // empty tensors may come with NULL pointers
  if (!k_out && !v_out) return fail(VQ_ERR_INVALID_ARG, "k_out and v_out are both NULL");
  if (!slot_mapping) return fail(VQ_ERR_INVALID_ARG, "slot_mapping is NULL");
  if (num_pages < 1) return fail(VQ_ERR_INVALID_ARG, "num_pages %lld < 1", (long long)num_pages);
  if (k_out && (!lambda || !codebook_k || !k_pool))
    return fail(VQ_ERR_INVALID_ARG, "k_out given but lambda, codebook_k or k_pool is NULL");
  if (v_out && (!codebook_v || !v_pool))
    return fail(VQ_ERR_INVALID_ARG, "v_out given but codebook_v or v_pool is NULL");
  const void* ptrs[] = {k_out, v_out, lambda, codebook_k, codebook_v, k_pool, v_pool, slot_mapping};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return fail(VQ_ERR_INVALID_ARG, "device buffer %p is not 16-byte aligned", ptr);

  vqk::DequantParams p{};
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.cb_k = codebook_k;
  p.cb_v = codebook_v;
  p.out_k = k_out;
  p.out_v = v_out;
  p.k_sub = L.k_sub;
  p.k_bits = L.k_bits;
  p.k_row = static_cast<int>(vq_code_row_bytes(L.head_dim, L.k_sub, L.k_bits));
  p.v_sub = L.v_sub;
  p.v_bits = L.v_bits;
  p.v_row = static_cast<int>(vq_code_row_bytes(L.head_dim, L.v_sub, L.v_bits));
  p.lambda = lambda;
  p.slots = slot_mapping;
  p.status = status;
  p.num_slots = static_cast<long long>(num_pages) * L.page_size;
  p.num_tokens = num_tokens;
  p.hkv = L.num_kv_heads;
  p.page_size = L.page_size;
  p.which_base = k_out ? 0 : 1;
  p.which_last = v_out ? 1 : 0;
  const int per_cta = vqk::dequant_tokens_per_cta();
  const int grid_x = (num_tokens + per_cta - 1) / per_cta;
  cudaError_t e = vqk::launch_dequant(p, grid_x, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "vq_dequantize_kv launch");
  return VQ_OK;
}

int32_t vq_default_num_splits(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                              int32_t num_sms) {
  if (!layout || batch < 0 || max_seq_len < 0 || layout->num_kv_heads < 1) return 0;
  const int sms = num_sms > 0 ? num_sms : device_sms();
  if (sms <= 0) return 0;
  return pick_splits(*layout, batch, max_seq_len, sms);
}

int32_t vq_decode_units_balanced(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                                 int32_t num_splits, int32_t num_sms) {
  if (!layout || batch < 0 || max_seq_len < 0 || layout->num_kv_heads < 1) return -1;
  if (num_splits > kMaxSplits) return -1;
  const int sms = num_sms > 0 ? num_sms : device_sms();
  if (sms <= 0) return -1;
  const int splits = num_splits > 0 ? num_splits : pick_splits(*layout, batch, max_seq_len, sms);
  return balanced_units(*layout, batch, max_seq_len, splits, sms) ? 1 : 0;
}

size_t vq_decode_workspace_bytes(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                                 int32_t num_splits, int32_t num_sms) {
  if (!layout || batch < 0 || max_seq_len < 0 || layout->num_q_heads < 1) return 0;
  int splits = num_splits;
  if (splits <= 0) splits = vq_default_num_splits(layout, batch, max_seq_len, num_sms);
  if (splits <= 0 || splits > kMaxSplits) return 0;
  return ws_layout(*layout, batch, splits).total;
}

}  // extern "C"

namespace {

// Validates the decode arguments and fills the split kernel's parameters.
vq_status prepare_decode(const vq_layout* layout, int32_t batch, const void* q, const float* lambda,
                         const void* codebook_k, const void* codebook_v, const void* k_pool,
                         const void* v_pool, int64_t num_pages, const int32_t* page_table,
                         int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                         float softmax_scale, int32_t num_splits, const void* workspace,
                         size_t workspace_bytes, int32_t* status, vqk::DecodeParams& p,
                         int& grid, size_t& smem, bool* append = nullptr,
                         int method = vqk::kMethodGather, int res_capacity = 0) {
  const vq_layout& L = *layout;
  const void* ptrs[] = {q, lambda, codebook_k, codebook_v, k_pool, v_pool, page_table, seq_lens, workspace};
  const char* names[] = {"q", "lambda", "codebook_k", "codebook_v", "k_pool", "v_pool",
                         "page_table", "seq_lens", "workspace"};
  for (int i = 0; i < 9; ++i) {
    if (!ptrs[i]) return fail(VQ_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return fail(VQ_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  if (num_pages < 1) return fail(VQ_ERR_INVALID_ARG, "num_pages %lld < 1", (long long)num_pages);
  if (max_pages_per_seq < 1) return fail(VQ_ERR_INVALID_ARG, "max_pages_per_seq %d < 1", max_pages_per_seq);
  if (max_seq_len < 0) return fail(VQ_ERR_INVALID_ARG, "max_seq_len %d < 0", max_seq_len);
  if (static_cast<long long>(max_seq_len) > static_cast<long long>(max_pages_per_seq) * L.page_size)
    return fail(VQ_ERR_INVALID_ARG, "max_seq_len %d exceeds max_pages_per_seq * page_size", max_seq_len);
  if (!std::isfinite(softmax_scale)) return fail(VQ_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (num_splits > kMaxSplits) return fail(VQ_ERR_INVALID_ARG, "num_splits %d > %d", num_splits, kMaxSplits);

  const int sms = device_sms();
  if (sms <= 0) return fail(VQ_ERR_CUDA, "no CUDA device");
  const int splits = num_splits > 0 ? num_splits : pick_splits(L, batch, max_seq_len, sms);
  const WsLayout ws = ws_layout(L, batch, splits);
  if (workspace_bytes < ws.total)
    return fail(VQ_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, ws.total);
  const long long units = static_cast<long long>(batch) * L.num_kv_heads * splits;
  if (units > 0x7fffffffLL) return fail(VQ_ERR_INVALID_ARG, "too many work units");
  const bool balanced = balanced_units(L, batch, max_seq_len, splits, sms);
  long long g = std::min<long long>(units, sms);
  g = std::max<long long>(g, (units + vqk::kMaxUnitsPerCta - 1) / vqk::kMaxUnitsPerCta);
  grid = static_cast<int>(balanced ? sms : g);

  p = vqk::DecodeParams{};
  p.q = q;
  p.lambda = lambda;
  p.cb_k = codebook_k;
  p.cb_v = codebook_v;
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  uint8_t* wsb = static_cast<uint8_t*>(const_cast<void*>(workspace));
  p.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  p.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  p.status = status;
  p.num_pages = num_pages;
  p.timeout_ns = 2000000000ULL;
  p.batch = batch;
  p.hq = L.num_q_heads;
  p.hkv = L.num_kv_heads;
  p.group = L.num_q_heads / L.num_kv_heads;
  p.page_size = L.page_size;
  p.max_pages = max_pages_per_seq;
  p.max_seq_len = max_seq_len;
  p.splits = splits;
  p.num_units = static_cast<int>(units);
  const int nsl = (max_seq_len + vqk::kUnitTok - 1) / vqk::kUnitTok;
  p.split_q = nsl / splits;
  p.split_r = nsl % splits;
  p.balanced = balanced ? 1 : 0;
  p.ws_cnt = balanced ? reinterpret_cast<int*>(wsb + ws.cnt_off) : nullptr;
  p.k_row = static_cast<int>(vq_code_row_bytes(L.head_dim, L.k_sub, L.k_bits));
  p.v_row = static_cast<int>(vq_code_row_bytes(L.head_dim, L.v_sub, L.v_bits));
  const float scale = softmax_scale == 0.f ? 1.f / std::sqrt(static_cast<float>(L.head_dim)) : softmax_scale;
  p.qscale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 / std::sqrt(128.0));
  // residual window: a unit's slice is at most ceil(capacity / splits)
  // tokens (length-balanced units: the whole window), staged in shared
  // memory up to kMaxResTok at a time
  const int res_slice = balanced ? res_capacity : (res_capacity + splits - 1) / splits;
  const int res_tok = res_capacity > 0 ? std::min(res_slice, vqk::kMaxResTok) : 0;
  p.res_tok = res_tok;

  const int optin = device_smem_optin();
  // Pipeline stages: the most (up to kMaxStages) that fit, and never fewer
  // than the producer warps.  A producer waits for its slot to be released by
  // the parity of the slot's "empty" barrier, which tells adjacent phases
  // apart only; with at least as many stages as producer warps, the
  // producer's own previous stage guarantees the barrier is at most one phase
  // behind.
  bool with_append = false;
  auto stages_for = [&](const vqk::DecodeShape& sh, size_t& bytes) {
    int ns = vqk::kMaxStages;
    for (; ns >= vqk::kProducerWarps; --ns) {
      bytes = vqk::decode_smem(L.k_bits, L.v_bits, p.group, p.k_row, p.v_row, ns, sh.warps,
                               sh.stage_tok(),
                               with_append && !sliced_append(L)
                                   ? vqk::append_enc_bytes(L.k_bits, L.v_bits, L.k_sub, L.v_sub) : 0,
                               method, res_tok)
                  .total;
      if (optin <= 0 || bytes <= static_cast<size_t>(optin)) return ns;
    }
    return 0;
  };
  // Consumer shape: 12 warps for G <= 4, 8 warps for G > 4 (register
  // budget), and 8 wherever 12 leaves room for fewer than kProducerWarps
  // stages; VQ_DECODE_SHAPE=8x1|12x1 selects a shape explicitly (a tuning
  // switch for profiling; an explicit shape that does not fit is an error).
  // (the 1.5-bit format: 8, its whole-centroid gathers need the registers)
  vqk::DecodeShape shape = (p.group > 4 || L.k_bits == 12) ? vqk::DecodeShape{8} : vqk::DecodeShape{12};
  bool explicit_shape = false;
  if (const char* env = std::getenv("VQ_DECODE_SHAPE")) {
    if (std::strcmp(env, "8x1") == 0) shape = vqk::DecodeShape{8}, explicit_shape = true;
    if (std::strcmp(env, "12x1") == 0) shape = vqk::DecodeShape{12}, explicit_shape = true;
  }
  if (method != vqk::kMethodGather) {
    if (!(L.k_sub == 4 && L.k_bits == 8 && L.v_sub == 4 && L.v_bits == 8 && p.group <= 4))
      return fail(VQ_ERR_UNSUPPORTED,
                  "the LUT and bins methods are built for k_sub = v_sub = 4, 8-bit codes and "
                  "num_q_heads / num_kv_heads <= 4");
    shape = vqk::DecodeShape{12};
    explicit_shape = true;
  }
  int nstage = stages_for(shape, smem);
  if (nstage == 0 && !explicit_shape && shape.warps != 8) {
    shape = vqk::DecodeShape{8};
    nstage = stages_for(shape, smem);
  }
  if (nstage == 0)
    return fail(VQ_ERR_UNSUPPORTED,
                "decode pipeline does not fit: %d consumer warps need %zu bytes of shared memory "
                "for %d stages",
                shape.warps, smem, vqk::kProducerWarps);
  // The decode-step append inside the attention kernel needs a little more
  // shared memory; it runs only with the same consumer shape (so the results
  // equal the separate append and attention bit for bit) and enough stages.
  if (append && *append) {
    with_append = true;
    size_t bytes_app = 0;
    const int ns_app = stages_for(shape, bytes_app);
    if (ns_app >= vqk::kProducerWarps) {
      nstage = ns_app;
      smem = bytes_app;
    } else {
      *append = false;
    }
  }
  p.warps = shape.warps;
  p.nstage = nstage;
  return VQ_OK;
}

// CTAs of the decode step's append encode: one warp per (sequence, KV head)
// vector, 8 per CTA, keys and values.
vq_status launch_partial(const vq_layout& L, const vqk::DecodeParams& p, int grid, size_t smem,
                         void* stream, bool overlap, int method = vqk::kMethodGather) {
  cudaError_t e = vqk::launch_decode(p, L.k_sub, L.k_bits, L.v_sub, L.v_bits, grid, smem,
                                     static_cast<cudaStream_t>(stream), overlap, method);
  if (e != cudaSuccess) return cuda_fail(e, "decode split kernel");
  return VQ_OK;
}

vq_status combine_impl(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                       int32_t num_splits, const void* workspace, size_t workspace_bytes,
                       void* out, void* stream, bool overlap) {
  const vq_layout& L = *layout;
  if (!workspace || !out) return fail(VQ_ERR_INVALID_ARG, "workspace or out is NULL");
  if (!aligned16(workspace) || !aligned16(out))
    return fail(VQ_ERR_INVALID_ARG, "workspace or out is not 16-byte aligned");
  if (num_splits > kMaxSplits) return fail(VQ_ERR_INVALID_ARG, "num_splits %d > %d", num_splits, kMaxSplits);
  int splits = num_splits;
  int sms = 0;
  if (splits <= 0 || batch >= 2) {  // the split choice, or whether the units were length-balanced
    sms = device_sms();
    if (sms <= 0) return fail(VQ_ERR_CUDA, "no CUDA device");
  }
  if (splits <= 0) splits = pick_splits(L, batch, max_seq_len, sms);
  const WsLayout ws = ws_layout(L, batch, splits);
  if (workspace_bytes < ws.total)
    return fail(VQ_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, ws.total);
  vqk::CombineParams cp{};
  const uint8_t* wsb = static_cast<const uint8_t*>(workspace);
  cp.ws_o = reinterpret_cast<const float*>(wsb + ws.o_off);
  cp.ws_ml = reinterpret_cast<const float2*>(wsb + ws.ml_off);
  cp.out = out;
  cp.rows = batch * L.num_q_heads;
  cp.splits = splits;
  cp.cnt = balanced_units(L, batch, max_seq_len, splits, sms) ? reinterpret_cast<const int*>(wsb + ws.cnt_off)
                                                               : nullptr;
  cp.group = L.num_q_heads / L.num_kv_heads;
  cudaError_t e = vqk::launch_combine(cp, static_cast<cudaStream_t>(stream), overlap);
  if (e != cudaSuccess) return cuda_fail(e, "decode combine kernel");
  return VQ_OK;
}

}  // namespace

extern "C" {

vq_status vq_decode_partial(const vq_layout* layout, int32_t batch, const void* q,
                            const float* lambda, const void* codebook_k, const void* codebook_v,
                            const void* k_pool, const void* v_pool, int64_t num_pages,
                            const int32_t* page_table, int32_t max_pages_per_seq,
                            const int32_t* seq_lens, int32_t max_seq_len, float softmax_scale,
                            int32_t num_splits, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  if (batch < 0) return fail(VQ_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (batch == 0) return VQ_OK;
  vqk::DecodeParams p;
  int grid = 0;
  size_t smem = 0;
  st = prepare_decode(layout, batch, q, lambda, codebook_k, codebook_v, k_pool, v_pool, num_pages,
                      page_table, max_pages_per_seq, seq_lens, max_seq_len, softmax_scale,
                      num_splits, workspace, workspace_bytes, status, p, grid, smem);
  if (st != VQ_OK) return st;
  return launch_partial(*layout, p, grid, smem, stream, false);
}

vq_status vq_decode_partial_method(const vq_layout* layout, int32_t batch, const void* q,
                                   const float* lambda, const void* codebook_k,
                                   const void* codebook_v, const void* k_pool, const void* v_pool,
                                   int64_t num_pages, const int32_t* page_table,
                                   int32_t max_pages_per_seq, const int32_t* seq_lens,
                                   int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                                   int32_t method, void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  if (method < VQ_METHOD_GATHER || method > VQ_METHOD_BINS)
    return fail(VQ_ERR_INVALID_ARG, "method %d is not a vq_decode_method", method);
  if (batch < 0) return fail(VQ_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (batch == 0) return VQ_OK;
  vqk::DecodeParams p;
  int grid = 0;
  size_t smem = 0;
  st = prepare_decode(layout, batch, q, lambda, codebook_k, codebook_v, k_pool, v_pool, num_pages,
                      page_table, max_pages_per_seq, seq_lens, max_seq_len, softmax_scale,
                      num_splits, workspace, workspace_bytes, status, p, grid, smem, nullptr, method);
  if (st != VQ_OK) return st;
  return launch_partial(*layout, p, grid, smem, stream, false, method);
}

vq_status vq_decode_combine(const vq_layout* layout, int32_t batch, int32_t max_seq_len,
                            int32_t num_splits, const void* workspace, size_t workspace_bytes,
                            void* out, void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  if (batch < 0 || max_seq_len < 0) return fail(VQ_ERR_INVALID_ARG, "batch or max_seq_len < 0");
  if (batch == 0) return VQ_OK;
  return combine_impl(layout, batch, max_seq_len, num_splits, workspace, workspace_bytes, out, stream,
                      false);
}

vq_status vq_decode_step(const vq_layout* layout, int32_t batch, const void* q, const void* k_new,
                         const void* v_new, const float* lambda, const void* codebook_k,
                         const void* codebook_v, void* k_pool, void* v_pool, int64_t num_pages,
                         const int32_t* page_table, int32_t max_pages_per_seq,
                         const int32_t* seq_lens, int32_t max_seq_len, float softmax_scale,
                         int32_t num_splits, void* out, void* workspace, size_t workspace_bytes,
                         int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  const vq_layout& L = *layout;
  if (batch < 0) return fail(VQ_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (batch == 0) return VQ_OK;
  const void* ptrs[] = {k_new, v_new, out};
  const char* names[] = {"k_new", "v_new", "out"};
  for (int i = 0; i < 3; ++i) {
    if (!ptrs[i]) return fail(VQ_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return fail(VQ_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  vqk::DecodeParams p;
  int grid = 0;
  size_t smem = 0;
  // With at most one (sequence, KV head) pair per SM the new tokens are
  // appended inside the attention kernel: the producer warps of the CTA whose
  // split holds a new token encode it while their first copies are in flight
  // (codes of at most 9 bits), or merge the candidates that the encode
  // kernel's sliced scan left in the workspace (the 1.5-bit format, whose
  // 4096-centroid scan needs more than one CTA).  With more pairs than SMs the
  // separate append kernel spreads the appends over the GPU sooner (measured:
  // 32K, ragged batch-16 and 196K steps faster fused, batch 64 no faster).
  const int sms_now = device_sms();
  const bool wide = sliced_append(L);
  const bool wide_ok = L.k_sub == 8 && L.k_bits == 12 && L.v_sub == 8 && L.v_bits == 12;
  bool fused = ((L.k_bits <= 9 && L.v_bits <= 9) || wide_ok) &&
               static_cast<long long>(batch) * L.num_kv_heads <= (sms_now > 0 ? sms_now : 0);
  st = prepare_decode(layout, batch, q, lambda, codebook_k, codebook_v, k_pool, v_pool, num_pages,
                      page_table, max_pages_per_seq, seq_lens, max_seq_len, softmax_scale,
                      num_splits, workspace, workspace_bytes, status, p, grid, smem, &fused);
  if (st != VQ_OK) return st;

  vqk::EncodeParams ep{};
  ep.src[0] = k_new;
  ep.src[1] = v_new;
  ep.cb[0] = codebook_k;
  ep.cb[1] = codebook_v;
  ep.pool[0] = static_cast<uint8_t*>(k_pool);
  ep.pool[1] = static_cast<uint8_t*>(v_pool);
  ep.lambda = lambda;
  ep.slots = nullptr;
  ep.page_table = page_table;
  ep.seq_lens = seq_lens;
  ep.max_pages = max_pages_per_seq;
  ep.status = status;
  ep.num_slots = static_cast<long long>(num_pages) * L.page_size;
  // a large codebook's append goes over several CTAs per vector, its
  // candidates in the workspace after the split partials
  const WsLayout wsl = ws_layout(L, batch, p.splits);
  int2* cand = wide ? reinterpret_cast<int2*>(static_cast<uint8_t*>(workspace) + wsl.cand_off) : nullptr;

  if (fused) {
    p.append = 1;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_pool_w = static_cast<uint8_t*>(k_pool);
    p.v_pool_w = static_cast<uint8_t*>(v_pool);
    bool overlap = false;
    if (wide) {  // the sliced scan first; the attention kernel merges its candidates
      st = launch_encode_impl(L, ep, batch, true, true, stream, "vq_decode_step append scan", false, cand,
                              false);
      if (st != VQ_OK) return st;
      if (ep.slices <= 1) return fail(VQ_ERR_UNSUPPORTED, "vq_decode_step: the append scan was not sliced");
      p.app_cand = cand;
      p.app_slices = ep.slices;
      overlap = true;
    }
    st = launch_partial(L, p, grid, smem, stream, overlap);
    if (st != VQ_OK) return st;
    return combine_impl(layout, batch, max_seq_len, p.splits, workspace, workspace_bytes, out, stream,
                        true);
  }

  // 1. append: token seq_lens[b] - 1 of every sequence, slot from the page table
  st = launch_encode_impl(L, ep, batch, true, true, stream, "vq_decode_step append encode", false, cand);
  if (st != VQ_OK) return st;
  // 2. split attention (its copies wait for the append), 3. merge of the splits
  st = launch_partial(L, p, grid, smem, stream, true);
  if (st != VQ_OK) return st;
  return combine_impl(layout, batch, max_seq_len, p.splits, workspace, workspace_bytes, out, stream,
                      true);
}

vq_status vq_decode_attention(const vq_layout* layout, int32_t batch, const void* q,
                              const float* lambda, const void* codebook_k, const void* codebook_v,
                              const void* k_pool, const void* v_pool, int64_t num_pages,
                              const int32_t* page_table, int32_t max_pages_per_seq,
                              const int32_t* seq_lens, int32_t max_seq_len, float softmax_scale,
                              int32_t num_splits, void* out, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  if (batch < 0) return fail(VQ_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (batch == 0) return VQ_OK;
  if (!out) return fail(VQ_ERR_INVALID_ARG, "out is NULL");
  if (!aligned16(out)) return fail(VQ_ERR_INVALID_ARG, "out is not 16-byte aligned");
  vqk::DecodeParams p;
  int grid = 0;
  size_t smem = 0;
  st = prepare_decode(layout, batch, q, lambda, codebook_k, codebook_v, k_pool, v_pool, num_pages,
                      page_table, max_pages_per_seq, seq_lens, max_seq_len, softmax_scale,
                      num_splits, workspace, workspace_bytes, status, p, grid, smem);
  if (st != VQ_OK) return st;
  st = launch_partial(*layout, p, grid, smem, stream, false);
  if (st != VQ_OK) return st;
  return combine_impl(layout, batch, max_seq_len, p.splits, workspace, workspace_bytes, out, stream,
                      true);
}

}  // extern "C"

// ---- decode attention without a caller workspace ----------------------------
// Some callers cannot allocate device memory at the point where they run
// attention: code that executes inside a region where allocation is forbidden
// or would synchronise the device, embedders whose memory is owned by a
// foreign allocator they cannot call, or plug-ins that are handed only the
// tensors of one call.  For them the split partials live in this fixed,
// file-scope device array instead of a workspace.  Every GPU that loads the
// library holds the array until the process exits.
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // the context the address belongs to (0: not looked up)
  void* ptr;
};
ScratchAddr g_scratch[vqk::kMaxDevices] = {};

// Identity of the current context, so that an address looked up in a context
// that has since been destroyed (cudaDeviceReset) is looked up again.  The
// driver entry points come through the runtime, so no driver library is linked.
unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, nullptr) ==
        cudaSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, nullptr) ==
        cudaSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 1;
  return id + 1;  // never 0
}

// Device address of the array in the current context (a host-side name of a
// __device__ variable is not a device address); looked up once per device and
// context.
vq_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= vqk::kMaxDevices) return fail(VQ_ERR_UNSUPPORTED, "device %d out of range", dev);
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch[dev].ctx_id != ctx || !g_scratch[dev].ptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_scratch[dev].ptr = ptr;
    g_scratch[dev].ctx_id = ctx;
  }
  *out = g_scratch[dev].ptr;
  return VQ_OK;
}

}  // namespace

extern "C" {

vq_status vq_decode_attention_static(const vq_layout* layout, int32_t batch, const void* q,
                                     const float* lambda, const void* codebook_k,
                                     const void* codebook_v, const void* k_pool,
                                     const void* v_pool, int64_t num_pages,
                                     const int32_t* page_table, int32_t max_pages_per_seq,
                                     const int32_t* seq_lens, int32_t max_seq_len,
                                     float softmax_scale, int32_t num_splits, void* out,
                                     int32_t* status, void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  if (batch < 0) return fail(VQ_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (batch == 0) return VQ_OK;
  if (!out) return fail(VQ_ERR_INVALID_ARG, "out is NULL");
  if (!aligned16(out)) return fail(VQ_ERR_INVALID_ARG, "out is not 16-byte aligned");
  if (max_seq_len < 0) return fail(VQ_ERR_INVALID_ARG, "max_seq_len %d < 0", max_seq_len);
  if (num_splits > kMaxSplits) return fail(VQ_ERR_INVALID_ARG, "num_splits %d > %d", num_splits, kMaxSplits);
  int splits = num_splits;
  if (splits <= 0) {
    // the library's split choice, lowered until the partials fit the array
    const int sms = device_sms();
    if (sms <= 0) return fail(VQ_ERR_CUDA, "no CUDA device");
    splits = pick_splits(*layout, batch, max_seq_len, sms);
    while (splits > 1 && ws_layout(*layout, batch, splits).total > kStaticScratchBytes) --splits;
  }
  const size_t need = ws_layout(*layout, batch, splits).total;
  if (need > kStaticScratchBytes)
    return fail(VQ_ERR_WORKSPACE,
                "batch %d x %d query heads x %d splits needs %zu bytes of split scratch; the static "
                "scratch holds %zu bytes (use vq_decode_attention with a workspace, or fewer splits)",
                batch, layout->num_q_heads, splits, need, kStaticScratchBytes);
  void* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != VQ_OK) return st;
  // The split kernel writes every partial it later merges, so nothing in the
  // scratch has to start at zero; stale contents of an earlier call are never read.
  vqk::DecodeParams p;
  int grid = 0;
  size_t smem = 0;
  st = prepare_decode(layout, batch, q, lambda, codebook_k, codebook_v, k_pool, v_pool, num_pages,
                      page_table, max_pages_per_seq, seq_lens, max_seq_len, softmax_scale, splits,
                      scratch, kStaticScratchBytes, status, p, grid, smem);
  if (st != VQ_OK) return st;
  st = launch_partial(*layout, p, grid, smem, stream, false);
  if (st != VQ_OK) return st;
  return combine_impl(layout, batch, max_seq_len, splits, scratch, kStaticScratchBytes, out, stream,
                      true);
}

size_t vq_static_scratch_bytes(void) { return kStaticScratchBytes; }

const char* vq_last_error(void) { return g_last_error.c_str(); }

const char* vq_version(void) { return "vqattn 0.1.0 sm_103a"; }

size_t vq_decode_residual_workspace_bytes(const vq_layout* layout, int32_t batch,
                                          int32_t max_seq_len, int32_t num_splits,
                                          int32_t num_sms) {
  if (!layout || batch < 0 || max_seq_len < 0 || layout->num_q_heads < 1) return 0;
  int splits = num_splits;
  if (splits <= 0) splits = vq_default_num_splits(layout, batch, max_seq_len, num_sms);
  if (splits <= 0 || splits > kMaxSplits) return 0;
  return ws_layout(*layout, batch, splits).total;
}

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
                                       void* stream) {
  vq_status st = check_layout_impl(layout, 1);
  if (st != VQ_OK) return st;
  const vq_layout& L = *layout;
  if (batch < 0) return fail(VQ_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (batch == 0) return VQ_OK;
  if (res_capacity < 1 || res_capacity > kMaxResidual)
    return fail(VQ_ERR_INVALID_ARG, "res_capacity %d not in 1..%d", res_capacity, kMaxResidual);
  const void* ptrs[] = {out, k_res, v_res, res_lens};
  const char* names[] = {"out", "k_res", "v_res", "res_lens"};
  for (int i = 0; i < 4; ++i) {
    if (!ptrs[i]) return fail(VQ_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return fail(VQ_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  vqk::DecodeParams p;
  int grid = 0;
  size_t smem = 0;
  st = prepare_decode(layout, batch, q, lambda, codebook_k, codebook_v, k_pool, v_pool, num_pages,
                      page_table, max_pages_per_seq, seq_lens, max_seq_len, softmax_scale,
                      num_splits, workspace, workspace_bytes, status, p, grid, smem, nullptr,
                      vqk::kMethodGather, res_capacity);
  if (st != VQ_OK) return st;

  // 1. split attention over the codes, every unit merging its slice of the
  // residual window into its own partial, 2. merge of the splits
  p.residual = 1;
  p.k_res = k_res;
  p.v_res = v_res;
  p.res_lens = res_lens;
  p.res_capacity = res_capacity;
  const float scale = softmax_scale == 0.f ? 1.f / std::sqrt(static_cast<float>(L.head_dim)) : softmax_scale;
  p.res_scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  st = launch_partial(L, p, grid, smem, stream, false);
  if (st != VQ_OK) return st;
  return combine_impl(layout, batch, max_seq_len, p.splits, workspace, workspace_bytes, out, stream,
                      true);
}

}  // extern "C"
