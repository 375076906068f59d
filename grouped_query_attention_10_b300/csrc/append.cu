// append.cu -- KV-cache append: copy T new K/V tokens per sequence into rows
// seq_lens[b] .. seq_lens[b]+T-1 of every K/V head of a [B, g, S_max, d]
// cache, then advance the lengths. This is the cache concatenation along the
// sequence axis of the "What is Grouped-Query Attention" explainer
// (ijyty.com), section 3.2; only g heads are stored, never h_q.
#include <cuda_bf16.h>

#include "../../include/gqa.h"
#include "launch.h"
#include "ptx.cuh"

namespace gqa {

// One thread per 16-byte chunk of one (b, t, kv head) row of K and of V.
// Reads of k_new/v_new are fully coalesced; writes are contiguous per row.
__global__ void __launch_bounds__(256) kv_append_rows_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    const int32_t* __restrict__ seq_lens, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, int B, int g, int chunks, int S_max, int T,
    int32_t* status) {
  const long long total = static_cast<long long>(B) * T * g * chunks;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % chunks);
    long long r = idx / chunks;
    const int h = static_cast<int>(r % g);
    r /= g;
    const int t = static_cast<int>(r % T);
    const int b = static_cast<int>(r / T);
    const int len = seq_lens[b];
    if (len < 0 || len > S_max) {
      if (t == 0 && h == 0 && c == 0) record_status(status, GQA_ERR_BAD_LENGTH);
      continue;
    }
    const int pos = len + t;
    if (pos >= S_max) {
      if (h == 0 && c == 0) record_status(status, GQA_ERR_CACHE_FULL);
      continue;
    }
    const size_t src = idx;  // [B, T, g, chunks] is the iteration order itself
    const size_t dst =
        ((static_cast<size_t>(b) * g + h) * S_max + static_cast<size_t>(pos)) * chunks + c;
    k_cache[dst] = k_new[src];
    v_cache[dst] = v_new[src];
  }
}

// Advance every valid length by T, saturating at S_max. Runs after the row
// copy (same stream), so no row-copy thread can observe the new length.
__global__ void kv_append_lens_kernel(int32_t* seq_lens, int B, int S_max, int T) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int len = seq_lens[b];
  if (len < 0 || len > S_max) return;  // flagged by the row kernel, left as is
  const long long n = static_cast<long long>(len) + T;
  seq_lens[b] = static_cast<int32_t>(n < S_max ? n : S_max);
}

// Paged cache: row pos of sequence b lives in row pos % page_size of page
// block_table[b][pos / page_size] of a [num_pages, g, page_size, d] pool.
__global__ void __launch_bounds__(256) kv_append_paged_rows_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ table,
    const int32_t* __restrict__ seq_lens, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, int B, int g, int chunks, int page_log2, int num_pages,
    int max_blocks, int T, int32_t* status) {
  const long long total = static_cast<long long>(B) * T * g * chunks;
  const int cap = max_blocks << page_log2;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % chunks);
    long long r = idx / chunks;
    const int h = static_cast<int>(r % g);
    r /= g;
    const int t = static_cast<int>(r % T);
    const int b = static_cast<int>(r / T);
    const int len = seq_lens[b];
    if (len < 0 || len > cap) {
      if (t == 0 && h == 0 && c == 0) record_status(status, GQA_ERR_BAD_LENGTH);
      continue;
    }
    const int pos = len + t;
    if (pos >= cap) {
      if (h == 0 && c == 0) record_status(status, GQA_ERR_CACHE_FULL);
      continue;
    }
    const int page = table[static_cast<size_t>(b) * max_blocks + (pos >> page_log2)];
    if (page < 0 || page >= num_pages) {
      if (h == 0 && c == 0) record_status(status, GQA_ERR_BAD_PAGE);
      continue;
    }
    const size_t dst = ((static_cast<size_t>(page) * g + h) << page_log2 |
                        static_cast<size_t>(pos & ((1 << page_log2) - 1))) * chunks + c;
    k_pool[dst] = k_new[idx];
    v_pool[dst] = v_new[idx];
  }
}

cudaError_t launch_append_paged(void* k_pool, void* v_pool, const int32_t* block_table,
                                int32_t* seq_lens, const void* k_new, const void* v_new, int B,
                                int g, int d, int page_log2, int num_pages, int max_blocks, int T,
                                int32_t* status, cudaStream_t s) {
  const int chunks = d / 8;
  const long long total = static_cast<long long>(B) * T * g * chunks;
  long long blocks = (total + 255) / 256;
  if (blocks > 148LL * 32) blocks = 148LL * 32;
  if (blocks < 1) blocks = 1;
  kv_append_paged_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_table, seq_lens,
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, g, chunks, page_log2,
      num_pages, max_blocks, T, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kv_append_lens_kernel<<<(B + 127) / 128, 128, 0, s>>>(seq_lens, B, max_blocks << page_log2, T);
  return cudaGetLastError();
}

cudaError_t launch_append(void* k_cache, void* v_cache, int32_t* seq_lens, const void* k_new,
                          const void* v_new, int B, int g, int d, int S_max, int T,
                          int32_t* status, cudaStream_t s) {
  const int chunks = d / 8;
  const long long total = static_cast<long long>(B) * T * g * chunks;
  long long blocks = (total + 255) / 256;
  if (blocks > 148LL * 32) blocks = 148LL * 32;  // grid-stride beyond 32 CTAs per SM
  if (blocks < 1) blocks = 1;
  kv_append_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), seq_lens,
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, g, chunks, S_max, T,
      status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kv_append_lens_kernel<<<(B + 127) / 128, 128, 0, s>>>(seq_lens, B, S_max, T);
  return cudaGetLastError();
}

}  // namespace gqa
