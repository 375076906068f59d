// api.cu -- the C interface: host-side argument checks, TMA tensor-map
// encoding and kernel launches. Every check runs before any CUDA call, so a
// rejected call touches neither the device nor the stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/gqa.h"
#include "launch.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn load_encode_fn() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    return nullptr;
  }
  return reinterpret_cast<EncodeTiledFn>(p);
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = load_encode_fn();  // thread-safe one-time init
  return fn;
}

// Tensor map with the 128-byte swizzle; dims/strides innermost first,
// strides in bytes for dims 1..rank-1. Out-of-range boxes read zeros (loads)
// or are skipped (stores).
bool encode_sw128(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16(CUtensorMap* m, int rank, const void* base, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box) {
  return encode_sw128(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

// Heads / group-size rules shared by prefill and decode.
bool heads_ok(int h_q, int g, int d) {
  if (h_q < 1 || g < 1 || h_q % g != 0) return false;
  const int G = h_q / g;
  if (!pow2(G) || G > 128) return false;
  return d == 64 || d == 128;
}

constexpr long long kMaxElems = 1LL << 40;

struct DecodeLayout {
  int split_len, n_split;
  size_t part_o_bytes, part_lse_off, counter_off, total;
};

DecodeLayout decode_layout(int B, int h_q, int g, int d, int S_max) {
  DecodeLayout l{};
  l.split_len = gqa::decode_split_len(B, h_q, g, S_max);
  l.n_split = (S_max + l.split_len - 1) / l.split_len;
  const size_t rows = static_cast<size_t>(B) * h_q * l.n_split * gqa::kDecodeSlices;
  l.part_o_bytes = rows * d * sizeof(float);
  l.part_lse_off = (l.part_o_bytes + 255) & ~static_cast<size_t>(255);
  l.counter_off = (l.part_lse_off + rows * sizeof(float) + 255) & ~static_cast<size_t>(255);
  l.total = l.counter_off + 16;
  return l;
}

bool decode_shape_ok(int B, int h_q, int g, int d, int S_max) {
  if (B < 1 || B > 65535 || S_max < 1 || !heads_ok(h_q, g, d)) return false;
  const long long G = h_q / g;
  if (static_cast<long long>(B) * g * S_max * d >= kMaxElems) return false;
  // work items (64-token stages at the finest split) index an int
  if (static_cast<long long>(B) * g * ((G + 31) / 32) * (S_max / 64 + 1) >= (1LL << 31))
    return false;
  return true;
}

// Pages of 16 .. 65536 tokens (a power of two); the logical capacity
// page_size * max_blocks must fit an int.
bool paged_ok(int page_size, int max_blocks) {
  return page_size >= 16 && page_size <= 65536 && pow2(page_size) && max_blocks >= 1 &&
         static_cast<long long>(page_size) * max_blocks < (1LL << 31);
}

int decode_common(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* seq_lens, const int32_t* block_table, int page_size,
                  int num_pages, int max_blocks, void* o, int o_dtype, float* lse, int B,
                  int h_q, int g, int d, int S_max, float scale, int window,
                  const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                  int32_t* status_dev, void* stream);

}  // namespace

extern "C" {

const char* gqa_status_string(int status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_NULL: return "GQA_ERR_NULL: a required pointer is NULL";
    case GQA_ERR_SHAPE: return "GQA_ERR_SHAPE: size out of range or inconsistent";
    case GQA_ERR_ALIGN: return "GQA_ERR_ALIGN: pointer not 16-byte aligned";
    case GQA_ERR_WORKSPACE: return "GQA_ERR_WORKSPACE: workspace missing or too small";
    case GQA_ERR_CACHE_FULL: return "GQA_ERR_CACHE_FULL: appended rows did not fit";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA: a CUDA call or launch failed";
    case GQA_ERR_TIMEOUT: return "GQA_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case GQA_ERR_BAD_LENGTH: return "GQA_ERR_BAD_LENGTH: a sequence length was out of range";
    case GQA_ERR_SCRATCH_LIMIT:
      return "GQA_ERR_SCRATCH_LIMIT: sizes need more than the built-in decode scratch";
    case GQA_ERR_BAD_PAGE: return "GQA_ERR_BAD_PAGE: a block-table entry in use was outside the pool";
    default: return "GQA_ERR_UNKNOWN";
  }
}

int gqa_version(void) { return 100; }

}  // extern "C"

namespace {

// Shared by the prefill entry points. K/V come either in the projection
// layout [B, Lk, g, d] (kv_lens == nullptr, Lk == Lq) or from a cache
// [B, g, S_max, d] with per-sequence key counts kv_lens (then kv_extent is
// S_max and the queries are the last Lq keys of every sequence).
int prefill_common(const void* q, const void* k, const void* v, const int32_t* kv_lens, void* o,
                   int o_dtype, float* lse, int B, int Lq, int kv_extent, int h_q, int g, int d,
                   float scale, int causal, int window, const float* alibi, int32_t* status_dev,
                   void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return GQA_ERR_NULL;
  if (B < 1 || B > 65535 || Lq < 1 || kv_extent < 1 || !heads_ok(h_q, g, d) || g > 65535)
    return GQA_ERR_SHAPE;
  if (o_dtype != GQA_OUT_F32 && o_dtype != GQA_OUT_BF16) return GQA_ERR_SHAPE;
  if (!scale_ok(scale)) return GQA_ERR_SHAPE;
  if (window < 0 || (window > 0 && !causal)) return GQA_ERR_SHAPE;
  if (static_cast<long long>(B) * Lq * h_q * d >= kMaxElems) return GQA_ERR_SHAPE;
  if (static_cast<long long>(B) * g * kv_extent * d >= kMaxElems) return GQA_ERR_SHAPE;
  {
    // work units (pairs of 128-row query tiles x K/V heads x batch) index an int
    const long long pm2 = 2LL * (gqa::kPrefillBM / (h_q / g));
    if ((Lq + pm2 - 1) / pm2 * g * B >= (1LL << 31)) return GQA_ERR_SHAPE;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return GQA_ERR_ALIGN;
  if (lse != nullptr && !aligned4(lse)) return GQA_ERR_ALIGN;
  if (alibi != nullptr && !aligned4(alibi)) return GQA_ERR_ALIGN;
  if (kv_lens != nullptr && !aligned4(kv_lens)) return GQA_ERR_ALIGN;
  if (status_dev != nullptr && !aligned4(status_dev)) return GQA_ERR_ALIGN;

  const int G = h_q / g;
  gqa::PrefillArgs a{};
  const cuuint64_t e = 2;  // bytes per bf16
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h_q),
                                static_cast<cuuint64_t>(Lq), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {d * e, static_cast<cuuint64_t>(h_q) * d * e,
                                   static_cast<cuuint64_t>(Lq) * h_q * d * e};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G),
                               static_cast<cuuint32_t>(gqa::kPrefillBM / G), 1};
    if (!encode_bf16(&a.tm_q, 4, q, dims, strides, box)) return GQA_ERR_CUDA;
    // the output has the query layout; a box is one 128-byte column chunk of
    // the 32 rows (positions x heads of the group) one warp stores
    const cuuint64_t oe = o_dtype == GQA_OUT_F32 ? 4 : 2;
    const cuuint64_t ostrides[3] = {d * oe, static_cast<cuuint64_t>(h_q) * d * oe,
                                    static_cast<cuuint64_t>(Lq) * h_q * d * oe};
    const cuuint32_t obox[4] = {static_cast<cuuint32_t>(128 / oe),
                                static_cast<cuuint32_t>(G < 32 ? G : 32),
                                static_cast<cuuint32_t>(G < 32 ? 32 / G : 1), 1};
    if (!encode_sw128(&a.tm_o, o_dtype == GQA_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      4, o, dims, ostrides, obox))
      return GQA_ERR_CUDA;
  }
  if (kv_lens == nullptr) {
    // [B, Lk, g, d]: 4-D map {d, g, Lk, B}, a box is 128 keys of one head
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g),
                                static_cast<cuuint64_t>(kv_extent), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {d * e, static_cast<cuuint64_t>(g) * d * e,
                                   static_cast<cuuint64_t>(kv_extent) * g * d * e};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(gqa::kPrefillBN), 1};
    if (!encode_bf16(&a.tm_k, 4, k, dims, strides, box)) return GQA_ERR_CUDA;
    if (!encode_bf16(&a.tm_v, 4, v, dims, strides, box)) return GQA_ERR_CUDA;
  } else {
    // cache [B, g, S_max, d]: 3-D map {d, S_max, B*g} (as in decode)
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(kv_extent),
                                static_cast<cuuint64_t>(B) * g};
    const cuuint64_t strides[2] = {d * e, static_cast<cuuint64_t>(kv_extent) * d * e};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(gqa::kPrefillBN), 1};
    if (!encode_bf16(&a.tm_k, 3, k, dims, strides, box)) return GQA_ERR_CUDA;
    if (!encode_bf16(&a.tm_v, 3, v, dims, strides, box)) return GQA_ERR_CUDA;
  }
  a.o_dtype = o_dtype;
  a.lse = lse;
  a.B = B;
  a.Lq = Lq;
  a.Lk = kv_lens == nullptr ? kv_extent : 0;
  a.S_max = kv_extent;
  a.h_q = h_q;
  a.g = g;
  a.d = d;
  a.G = G;
  a.G_log2 = log2i(G);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal != 0;
  a.kv_lens = kv_lens;
  a.window = window;
  a.alibi = alibi;
  a.status = status_dev;
  return gqa::launch_prefill(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GQA_OK
                                                                                    : GQA_ERR_CUDA;
}

}  // namespace

extern "C" {

int gqa_prefill_fwd(const void* q, const void* k, const void* v, void* o, int o_dtype,
                    float* lse, int B, int L, int h_q, int g, int d, float scale, int causal,
                    int32_t* status_dev, void* stream) {
  return prefill_common(q, k, v, nullptr, o, o_dtype, lse, B, L, L, h_q, g, d, scale, causal, 0,
                        nullptr, status_dev, stream);
}

int gqa_prefill_fwd_ex(const void* q, const void* k, const void* v, void* o, int o_dtype,
                       float* lse, int B, int L, int h_q, int g, int d, float scale, int causal,
                       int window, const float* alibi_slopes, int32_t* status_dev,
                       void* stream) {
  return prefill_common(q, k, v, nullptr, o, o_dtype, lse, B, L, L, h_q, g, d, scale, causal,
                        window, alibi_slopes, status_dev, stream);
}

int gqa_prefill_kvcache_fwd(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B,
                            int T, int h_q, int g, int d, int S_max, float scale, int window,
                            const float* alibi_slopes, int32_t* status_dev, void* stream) {
  if (seq_lens == nullptr) return GQA_ERR_NULL;
  if (T > S_max) return GQA_ERR_SHAPE;
  return prefill_common(q, k_cache, v_cache, seq_lens, o, o_dtype, lse, B, T, S_max, h_q, g, d,
                        scale, 1, window, alibi_slopes, status_dev, stream);
}

size_t gqa_decode_workspace_bytes(int B, int h_q, int g, int d, int S_max) {
  if (!decode_shape_ok(B, h_q, g, d, S_max)) return 0;
  return decode_layout(B, h_q, g, d, S_max).total;
}

int gqa_decode_fwd(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B, int h_q,
                   int g, int d, int S_max, float scale, void* workspace, size_t workspace_bytes,
                   int32_t* status_dev, void* stream) {
  return gqa_decode_fwd_ex(q, k_cache, v_cache, seq_lens, o, o_dtype, lse, B, h_q, g, d, S_max,
                           scale, 0, nullptr, workspace, workspace_bytes, status_dev, stream);
}

int gqa_decode_fwd_ex(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B, int h_q,
                      int g, int d, int S_max, float scale, int window,
                      const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                      int32_t* status_dev, void* stream) {
  return decode_common(q, k_cache, v_cache, seq_lens, nullptr, 0, 0, 0, o, o_dtype, lse, B, h_q,
                       g, d, S_max, scale, window, alibi_slopes, workspace, workspace_bytes,
                       status_dev, stream);
}

size_t gqa_decode_paged_workspace_bytes(int B, int h_q, int g, int d, int page_size,
                                        int max_blocks) {
  if (!paged_ok(page_size, max_blocks)) return 0;
  return gqa_decode_workspace_bytes(B, h_q, g, d, page_size * max_blocks);
}

int gqa_decode_paged_fwd(const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_table, const int32_t* seq_lens, void* o,
                         int o_dtype, float* lse, int B, int h_q, int g, int d, int page_size,
                         int num_pages, int max_blocks, float scale, int window,
                         const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, void* stream) {
  if (block_table == nullptr) return GQA_ERR_NULL;
  if (!paged_ok(page_size, max_blocks) || num_pages < 1 ||
      static_cast<long long>(num_pages) * g * page_size * d >= kMaxElems ||
      static_cast<long long>(num_pages) * g >= (1LL << 31))
    return GQA_ERR_SHAPE;
  if (!aligned4(block_table)) return GQA_ERR_ALIGN;
  return decode_common(q, k_pool, v_pool, seq_lens, block_table, page_size, num_pages,
                       max_blocks, o, o_dtype, lse, B, h_q, g, d, page_size * max_blocks, scale,
                       window, alibi_slopes, workspace, workspace_bytes, status_dev, stream);
}

}  // extern "C"

namespace {

int decode_common(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* seq_lens, const int32_t* block_table, int page_size,
                  int num_pages, int max_blocks, void* o, int o_dtype, float* lse, int B,
                  int h_q, int g, int d, int S_max, float scale, int window,
                  const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                  int32_t* status_dev, void* stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr ||
      o == nullptr)
    return GQA_ERR_NULL;
  if (!decode_shape_ok(B, h_q, g, d, S_max)) return GQA_ERR_SHAPE;
  if (o_dtype != GQA_OUT_F32 && o_dtype != GQA_OUT_BF16) return GQA_ERR_SHAPE;
  if (!scale_ok(scale) || window < 0) return GQA_ERR_SHAPE;
  if (alibi_slopes != nullptr && !aligned4(alibi_slopes)) return GQA_ERR_ALIGN;
  const DecodeLayout lay = decode_layout(B, h_q, g, d, S_max);
  if (workspace == nullptr || workspace_bytes < lay.total) return GQA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(workspace) || !aligned4(seq_lens))
    return GQA_ERR_ALIGN;
  if (lse != nullptr && !aligned4(lse)) return GQA_ERR_ALIGN;
  if (status_dev != nullptr && !aligned4(status_dev)) return GQA_ERR_ALIGN;

  gqa::DecodeArgs a{};
  const cuuint64_t e = 2;
  if (block_table == nullptr) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(S_max),
                                static_cast<cuuint64_t>(B) * g};
    const cuuint64_t strides[2] = {d * e, static_cast<cuuint64_t>(S_max) * d * e};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(gqa::kDecodeStage), 1};
    if (!encode_bf16(&a.tm_k, 3, k_cache, dims, strides, box)) return GQA_ERR_CUDA;
    if (!encode_bf16(&a.tm_v, 3, v_cache, dims, strides, box)) return GQA_ERR_CUDA;
  } else {
    // pool [num_pages, g, page_size, d]: map {d, page_size, num_pages * g}; a box
    // is one page's rows, at most one 64-token stage
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(page_size),
                                static_cast<cuuint64_t>(num_pages) * g};
    const cuuint64_t strides[2] = {d * e, static_cast<cuuint64_t>(page_size) * d * e};
    const cuuint32_t rows = static_cast<cuuint32_t>(
        page_size < gqa::kDecodeStage ? page_size : gqa::kDecodeStage);
    const cuuint32_t box[3] = {64, rows, 1};
    if (!encode_bf16(&a.tm_k, 3, k_cache, dims, strides, box)) return GQA_ERR_CUDA;
    if (!encode_bf16(&a.tm_v, 3, v_cache, dims, strides, box)) return GQA_ERR_CUDA;
  }
  a.block_table = block_table;
  a.page_log2 = block_table == nullptr ? 0 : log2i(page_size);
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.q = q;
  a.seq_lens = seq_lens;
  a.o = o;
  a.o_dtype = o_dtype;
  a.lse = lse;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + lay.part_lse_off);
  a.item_counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + lay.counter_off);
  a.B = B;
  a.h_q = h_q;
  a.g = g;
  a.d = d;
  a.G = h_q / g;
  a.S_max = S_max;
  a.split_len = lay.split_len;
  a.n_split = lay.n_split;
  if (window > 0) {
    // A window reads at most W' + 63 rows per sequence (W' = min(W, S_max);
    // the 63 covers its first row sitting anywhere inside a 64-row stage).
    // The split length follows the same rule as for a cache of that many
    // rows, so a short window is not cut into needlessly small items; if that
    // needed more splits than the workspace holds, the window's rows are
    // spread over the workspace's n_split splits instead.
    const long long w = window < S_max ? window : S_max;
    const long long rows = w + gqa::kDecodeStage - 1;
    long long l = gqa::decode_split_len(B, h_q, g, static_cast<int>(rows));
    if ((rows + l - 1) / l > lay.n_split) {
      l = (rows + lay.n_split - 1) / lay.n_split;
      l = (l + gqa::kDecodeStage - 1) / gqa::kDecodeStage * gqa::kDecodeStage;
    }
    a.split_len = static_cast<int>(l);
  }
  a.scale_log2 = scale * 1.4426950408889634f;
  a.window = window;
  a.alibi = alibi_slopes;
  a.status = status_dev;
  return gqa::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GQA_OK
                                                                                   : GQA_ERR_CUDA;
}

}  // namespace

extern "C" {

int kv_cache_append_paged(void* k_pool, void* v_pool, const int32_t* block_table,
                          int32_t* seq_lens, const void* k_new, const void* v_new, int B, int g,
                          int d, int page_size, int num_pages, int max_blocks, int T,
                          int32_t* status_dev, void* stream) {
  if (k_pool == nullptr || v_pool == nullptr || block_table == nullptr || seq_lens == nullptr ||
      k_new == nullptr || v_new == nullptr)
    return GQA_ERR_NULL;
  if (B < 1 || g < 1 || (d != 64 && d != 128) || T < 0 || num_pages < 1 ||
      !paged_ok(page_size, max_blocks))
    return GQA_ERR_SHAPE;
  if (static_cast<long long>(num_pages) * g * page_size * d >= kMaxElems ||
      static_cast<long long>(B) * T * g * d >= kMaxElems ||
      static_cast<long long>(B) * max_blocks >= (1LL << 31))
    return GQA_ERR_SHAPE;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned4(seq_lens) || !aligned4(block_table))
    return GQA_ERR_ALIGN;
  if (status_dev != nullptr && !aligned4(status_dev)) return GQA_ERR_ALIGN;
  if (T == 0) return GQA_OK;
  return gqa::launch_append_paged(k_pool, v_pool, block_table, seq_lens, k_new, v_new, B, g, d,
                                  log2i(page_size), num_pages, max_blocks, T, status_dev,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Checks shared by the two RoPE appends; `cap` is the logical capacity.
int rope_append_check(const void* k_new, const void* v_new, const void* q, void* q_out,
                      const float* rope_cos, const float* rope_sin, int rope_n_pos, int B,
                      int h_q, int g, int d, int T, long long cap) {
  if (k_new == nullptr || v_new == nullptr || rope_cos == nullptr || rope_sin == nullptr)
    return GQA_ERR_NULL;
  if ((q == nullptr) != (q_out == nullptr)) return GQA_ERR_NULL;
  if (B < 1 || g < 1 || (d != 64 && d != 128) || T < 0) return GQA_ERR_SHAPE;
  if (q != nullptr && !heads_ok(h_q, g, d)) return GQA_ERR_SHAPE;
  // every stored row's position must have a table row
  if (rope_n_pos < cap || static_cast<long long>(rope_n_pos) * d >= kMaxElems)
    return GQA_ERR_SHAPE;
  const long long qn = q != nullptr ? static_cast<long long>(B) * T * h_q * d : 0;
  if (static_cast<long long>(B) * T * g * d >= kMaxElems || qn >= kMaxElems) return GQA_ERR_SHAPE;
  if (q != nullptr && q != q_out) {
    // the rotated queries go in place or to a buffer that does not overlap q
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(q), b0 = reinterpret_cast<uintptr_t>(q_out);
    const uintptr_t n = static_cast<uintptr_t>(qn) * 2;
    if (a0 < b0 + n && b0 < a0 + n) return GQA_ERR_SHAPE;
  }
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(rope_cos) || !aligned16(rope_sin))
    return GQA_ERR_ALIGN;
  if (q != nullptr && (!aligned16(q) || !aligned16(q_out))) return GQA_ERR_ALIGN;
  return GQA_OK;
}

int rope_append_launch(gqa::RopeAppendArgs& a, void* stream) {
  if (a.T == 0) return GQA_OK;
  return gqa::launch_append_rope(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

}  // namespace

extern "C" {

int kv_cache_append_rope(void* k_cache, void* v_cache, int32_t* seq_lens, const void* k_new,
                         const void* v_new, const void* q, void* q_out, const float* rope_cos,
                         const float* rope_sin, int rope_n_pos, int B, int h_q, int g, int d,
                         int S_max, int T, int32_t* status_dev, void* stream) {
  if (k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr) return GQA_ERR_NULL;
  if (S_max < 1) return GQA_ERR_SHAPE;
  int rc = rope_append_check(k_new, v_new, q, q_out, rope_cos, rope_sin, rope_n_pos, B, h_q, g,
                             d, T, S_max);
  if (rc != GQA_OK) return rc;
  if (static_cast<long long>(B) * g * S_max * d >= kMaxElems) return GQA_ERR_SHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned4(seq_lens)) return GQA_ERR_ALIGN;
  if (status_dev != nullptr && !aligned4(status_dev)) return GQA_ERR_ALIGN;
  gqa::RopeAppendArgs a{};
  a.k_dst = k_cache;
  a.v_dst = v_cache;
  a.table = nullptr;
  a.S_max = S_max;
  a.seq_lens = seq_lens;
  a.k_new = k_new;
  a.v_new = v_new;
  a.q = q;
  a.q_out = q_out;
  a.cos = rope_cos;
  a.sin = rope_sin;
  a.B = B;
  a.T = T;
  a.h_q = q != nullptr ? h_q : 0;
  a.g = g;
  a.d = d;
  a.status = status_dev;
  return rope_append_launch(a, stream);
}

int kv_cache_append_paged_rope(void* k_pool, void* v_pool, const int32_t* block_table,
                               int32_t* seq_lens, const void* k_new, const void* v_new,
                               const void* q, void* q_out, const float* rope_cos,
                               const float* rope_sin, int rope_n_pos, int B, int h_q, int g,
                               int d, int page_size, int num_pages, int max_blocks, int T,
                               int32_t* status_dev, void* stream) {
  if (k_pool == nullptr || v_pool == nullptr || block_table == nullptr || seq_lens == nullptr)
    return GQA_ERR_NULL;
  if (num_pages < 1 || !paged_ok(page_size, max_blocks)) return GQA_ERR_SHAPE;
  int rc = rope_append_check(k_new, v_new, q, q_out, rope_cos, rope_sin, rope_n_pos, B, h_q, g,
                             d, T, static_cast<long long>(page_size) * max_blocks);
  if (rc != GQA_OK) return rc;
  if (static_cast<long long>(num_pages) * g * page_size * d >= kMaxElems ||
      static_cast<long long>(B) * max_blocks >= (1LL << 31))
    return GQA_ERR_SHAPE;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned4(seq_lens) || !aligned4(block_table))
    return GQA_ERR_ALIGN;
  if (status_dev != nullptr && !aligned4(status_dev)) return GQA_ERR_ALIGN;
  gqa::RopeAppendArgs a{};
  a.k_dst = k_pool;
  a.v_dst = v_pool;
  a.table = block_table;
  a.page_log2 = log2i(page_size);
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.k_new = k_new;
  a.v_new = v_new;
  a.q = q;
  a.q_out = q_out;
  a.cos = rope_cos;
  a.sin = rope_sin;
  a.B = B;
  a.T = T;
  a.h_q = q != nullptr ? h_q : 0;
  a.g = g;
  a.d = d;
  a.status = status_dev;
  return rope_append_launch(a, stream);
}

int gqa_selftest_bounded_wait(int32_t* status_dev, int limit_us, void* stream) {
  if (status_dev == nullptr) return GQA_ERR_NULL;
  if (limit_us < 1 || limit_us > 2000000) return GQA_ERR_SHAPE;
  if (!aligned4(status_dev)) return GQA_ERR_ALIGN;
  return gqa::launch_bounded_wait_selftest(status_dev, static_cast<long long>(limit_us) * 1000,
                                           static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

int kv_cache_append(void* k_cache, void* v_cache, int32_t* seq_lens, const void* k_new,
                    const void* v_new, int B, int g, int d, int S_max, int T,
                    int32_t* status_dev, void* stream) {
  if (k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr || k_new == nullptr ||
      v_new == nullptr)
    return GQA_ERR_NULL;
  if (B < 1 || g < 1 || (d != 64 && d != 128) || S_max < 1 || T < 0) return GQA_ERR_SHAPE;
  if (static_cast<long long>(B) * g * S_max * d >= kMaxElems ||
      static_cast<long long>(B) * T * g * d >= kMaxElems)
    return GQA_ERR_SHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned4(seq_lens))
    return GQA_ERR_ALIGN;
  if (status_dev != nullptr && !aligned4(status_dev)) return GQA_ERR_ALIGN;
  if (T == 0) return GQA_OK;
  return gqa::launch_append(k_cache, v_cache, seq_lens, k_new, v_new, B, g, d, S_max, T,
                            status_dev, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

}  // extern "C"
