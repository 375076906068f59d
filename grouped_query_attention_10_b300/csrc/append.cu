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
