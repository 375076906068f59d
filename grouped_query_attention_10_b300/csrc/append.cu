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

// Splits a flat chunk index of the [B, T, g, chunks] new-token layout into
// (b, t, h, c). Idx is 32-bit when the whole range fits (two 32-bit divisions
// per chunk, instead of 64-bit ones that made the copy instruction bound).
template <typename Idx>
__device__ __forceinline__ void split_chunk(Idx idx, int T, int g, int chunk_log2, int& b, int& t,
                                            int& h, int& c) {
  const Idx per_tok = static_cast<Idx>(g) << chunk_log2;  // chunks of one token (all heads)
  const Idx tok = idx / per_tok;
  const int i = static_cast<int>(idx - tok * per_tok);
  h = i >> chunk_log2;
  c = i & ((1 << chunk_log2) - 1);
  const Idx bb = tok / static_cast<Idx>(T);
  b = static_cast<int>(bb);
  t = static_cast<int>(tok - bb * static_cast<Idx>(T));
}

// End of a row-copy CTA: every length its threads read has been read, so the
// length update (a programmatic dependent launch) may start once all CTAs
// have passed this point; it need not wait for the copies to land.
__device__ __forceinline__ void lengths_read() {
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One thread per 16-byte chunk of one (b, t, kv head) row of K and of V.
// Reads of k_new/v_new are fully coalesced; writes are contiguous per row.
template <typename Idx>
__global__ void __launch_bounds__(256) kv_append_rows_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    const int32_t* __restrict__ seq_lens, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, int B, int g, int chunk_log2, int S_max, int T,
    int32_t* status) {
  const int chunks = 1 << chunk_log2;
  const Idx total = static_cast<Idx>(B) * T * g * chunks;
  for (Idx idx = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<Idx>(gridDim.x) * blockDim.x) {
    int b, t, h, c;
    split_chunk<Idx>(idx, T, g, chunk_log2, b, t, h, c);
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
  lengths_read();
}

// Advance every valid length by T, saturating at S_max. After the K/V row
// copies it is launched as a programmatic dependent: it starts once every
// row-copy CTA has read its lengths (lengths_read), so no row-copy thread can
// observe the new length, and writes the lengths while the row stores may
// still be in flight. It then waits (griddepcontrol.wait) for the row copy to
// complete before it exits: work queued after the append is ordered after
// this kernel, and so after the copy as well. After the RoPE append it runs
// in plain stream order (the wait is then a no-op).
__global__ void kv_append_lens_kernel(int32_t* seq_lens, int B, int S_max, int T) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int len = seq_lens[b];
    if (len >= 0 && len <= S_max) {  // a bad length is flagged by the row kernel, left as is
      const long long n = static_cast<long long>(len) + T;
      seq_lens[b] = static_cast<int32_t>(n < S_max ? n : S_max);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

static cudaError_t launch_lens_update(int32_t* seq_lens, int B, int cap, int T, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((B + 127) / 128));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_append_lens_kernel, seq_lens, B, cap, T);
}

// Paged cache: row pos of sequence b lives in row pos % page_size of page
// block_table[b][pos / page_size] of a [num_pages, g, page_size, d] pool.
template <typename Idx>
__global__ void __launch_bounds__(256) kv_append_paged_rows_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ table,
    const int32_t* __restrict__ seq_lens, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, int B, int g, int chunk_log2, int page_log2, int num_pages,
    int max_blocks, int T, int32_t* status) {
  const int chunks = 1 << chunk_log2;
  const Idx total = static_cast<Idx>(B) * T * g * chunks;
  const int cap = max_blocks << page_log2;
  for (Idx idx = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<Idx>(gridDim.x) * blockDim.x) {
    int b, t, h, c;
    split_chunk<Idx>(idx, T, g, chunk_log2, b, t, h, c);
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
  lengths_read();
}

cudaError_t launch_append_paged(void* k_pool, void* v_pool, const int32_t* block_table,
                                int32_t* seq_lens, const void* k_new, const void* v_new, int B,
                                int g, int d, int page_log2, int num_pages, int max_blocks, int T,
                                int32_t* status, cudaStream_t s) {
  const int chunk_log2 = d == 64 ? 3 : 4;  // 16-byte chunks per row: 8 or 16
  const long long total = static_cast<long long>(B) * T * g << chunk_log2;
  long long blocks = (total + 255) / 256;
  if (blocks > 148LL * 32) blocks = 148LL * 32;
  if (blocks < 1) blocks = 1;
  if (total + 148LL * 32 * 256 < (1LL << 31))
    kv_append_paged_rows_kernel<uint32_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_table, seq_lens,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, g, chunk_log2,
        page_log2, num_pages, max_blocks, T, status);
  else
    kv_append_paged_rows_kernel<uint64_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_table, seq_lens,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, g, chunk_log2,
        page_log2, num_pages, max_blocks, T, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lens_update(seq_lens, B, max_blocks << page_log2, T, s);
}

// ---------------------------------------------------------------------------
// RoPE append: one launch rotates the new tokens' query rows (into q_out) and
// key rows (into the cache) and copies their value rows, at the position each
// token takes in the cache (seq_lens[b] + t). The rotation is the RoPE code of
// the jsqmd.com attention survey, chapter 1: pair (x[2i], x[2i+1]) is turned
// by the angle of table row `pos`, the turned even parts fill the first half
// of the output row and the turned odd parts the second half. Arithmetic is
// binary32 with every product, sum and difference rounded (no contraction),
// as the survey's code evaluates bf16 rows times fp32 tables; the stored
// value is rounded to bf16.
//
// One thread per (row, u): input chunks 2u and 2u+1 (16 elements = 8 pairs)
// give output chunks u and u + d/16 of a rotated row; a value row is copied
// as chunks 2u and 2u+1. The loop is uniform per warp and every lane reads
// before any lane writes (a row never spans two warps), so q_out may be q.
// One pair: w holds input elements 2i (low half) and 2i+1 (high half).
__device__ __forceinline__ void rope_pair(uint32_t w, float c, float s, float* first,
                                          float* second) {
  const float e = __uint_as_float(w << 16);
  const float o = __uint_as_float(w & 0xffff0000u);
  *first = __fsub_rn(__fmul_rn(e, c), __fmul_rn(o, s));
  *second = __fadd_rn(__fmul_rn(e, s), __fmul_rn(o, c));
}

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Idx: 32-bit when the whole index range fits (cheap divisions), else 64-bit.
template <bool PAGED, typename Idx>
__global__ void __launch_bounds__(256) kv_append_rope_kernel(const RopeAppendArgs a) {
  const int half_log2 = a.d == 64 ? 2 : 3;  // threads per row: d / 16
  const int half = 1 << half_log2;
  const int chunks = a.d / 8;  // 16-byte chunks per row
  const int rows_bt = a.h_q + 2 * a.g;  // query, key and value rows of one token
  const Idx total = static_cast<Idx>(a.B) * a.T * rows_bt * half;
  const int cap = PAGED ? (a.max_blocks << a.page_log2) : a.S_max;
  const int lane = threadIdx.x & 31;
  const Idx stride = static_cast<Idx>(gridDim.x) * blockDim.x;
  const float4* cos4 = reinterpret_cast<const float4*>(a.cos);
  const float4* sin4 = reinterpret_cast<const float4*>(a.sin);
  for (Idx base = static_cast<Idx>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const Idx idx = base + lane;
    bool act = idx < total;
    uint4 out0 = make_uint4(0u, 0u, 0u, 0u), out1 = out0;
    uint4* dst0 = nullptr;
    uint4* dst1 = nullptr;
    if (act) {
      const int u = static_cast<int>(idx & (half - 1));
      const Idx r = idx >> half_log2;
      const Idx bt = r / static_cast<Idx>(rows_bt);
      const int row = static_cast<int>(r - bt * static_cast<Idx>(rows_bt));
      const Idx bq = bt / static_cast<Idx>(a.T);
      const int t = static_cast<int>(bt - bq * static_cast<Idx>(a.T));
      const int b = static_cast<int>(bq);
      const int len = a.seq_lens[b];
      int pos = 0;
      if (len < 0 || len > cap) {
        if (t == 0 && row == 0 && u == 0) record_status(a.status, GQA_ERR_BAD_LENGTH);
        act = false;
      } else {
        pos = len + t;
        if (pos >= cap) {
          if (row == 0 && u == 0) record_status(a.status, GQA_ERR_CACHE_FULL);
          act = false;
        }
      }
      const uint4* src = nullptr;
      uint4* drow = nullptr;
      bool rotate = true;
      if (act) {
        if (row < a.h_q) {
          const size_t off = (static_cast<size_t>(bt) * a.h_q + row) * chunks;
          src = static_cast<const uint4*>(a.q) + off;
          drow = static_cast<uint4*>(a.q_out) + off;
        } else {
          int h = row - a.h_q;
          const bool value = h >= a.g;
          if (value) h -= a.g;
          rotate = !value;
          src = static_cast<const uint4*>(value ? a.v_new : a.k_new) +
                (static_cast<size_t>(bt) * a.g + h) * chunks;
          size_t dst_row;
          if (PAGED) {
            const int page = a.table[static_cast<size_t>(b) * a.max_blocks + (pos >> a.page_log2)];
            if (page < 0 || page >= a.num_pages) {
              if (u == 0) record_status(a.status, GQA_ERR_BAD_PAGE);
              act = false;
            }
            dst_row = (static_cast<size_t>(page) * a.g + h) << a.page_log2 |
                      static_cast<size_t>(pos & ((1 << a.page_log2) - 1));
          } else {
            dst_row = (static_cast<size_t>(b) * a.g + h) * a.S_max + static_cast<size_t>(pos);
          }
          drow = static_cast<uint4*>(value ? a.v_dst : a.k_dst) + dst_row * chunks;
        }
      }
      if (act) {
        const uint4 x0 = src[2 * u];
        const uint4 x1 = src[2 * u + 1];
        if (rotate) {
          const size_t trow = static_cast<size_t>(pos) * (a.d / 8);  // float4s per table row
          const float4 c0 = cos4[trow + 2 * u], c1 = cos4[trow + 2 * u + 1];
          const float4 s0 = sin4[trow + 2 * u], s1 = sin4[trow + 2 * u + 1];
          const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          float f[8], g2[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) rope_pair(w[j], cv[j], sv[j], &f[j], &g2[j]);
          out0 = make_uint4(pack_bf16_rn(f[0], f[1]), pack_bf16_rn(f[2], f[3]),
                            pack_bf16_rn(f[4], f[5]), pack_bf16_rn(f[6], f[7]));
          out1 = make_uint4(pack_bf16_rn(g2[0], g2[1]), pack_bf16_rn(g2[2], g2[3]),
                            pack_bf16_rn(g2[4], g2[5]), pack_bf16_rn(g2[6], g2[7]));
          dst0 = drow + u;
          dst1 = drow + u + half;
        } else {
          out0 = x0;
          out1 = x1;
          dst0 = drow + 2 * u;
          dst1 = drow + 2 * u + 1;
        }
      }
    }
    __syncwarp();  // every lane has read its row chunks (q_out may alias q)
    if (act) {
      *dst0 = out0;
      *dst1 = out1;
    }
  }
}

cudaError_t launch_append_rope(const RopeAppendArgs& a, cudaStream_t s) {
  const long long total = static_cast<long long>(a.B) * a.T * (a.h_q + 2 * a.g) * (a.d / 16);
  long long blocks = (total + 255) / 256;
  if (blocks > 148LL * 16) blocks = 148LL * 16;  // grid-stride beyond 16 CTAs per SM
  if (blocks < 1) blocks = 1;
  const bool paged = a.table != nullptr;
  const bool narrow = total + 148LL * 16 * 256 < (1LL << 31);
  if (paged && narrow)
    kv_append_rope_kernel<true, uint32_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  else if (paged)
    kv_append_rope_kernel<true, uint64_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  else if (narrow)
    kv_append_rope_kernel<false, uint32_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  else
    kv_append_rope_kernel<false, uint64_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int cap = paged ? (a.max_blocks << a.page_log2) : a.S_max;
  // stream order here: as a programmatic dependent the update measured ~4 %
  // slower for this kernel (while it gains ~3 % after the plain row copies)
  kv_append_lens_kernel<<<(a.B + 127) / 128, 128, 0, s>>>(a.seq_lens, a.B, cap, a.T);
  return cudaGetLastError();
}

cudaError_t launch_append(void* k_cache, void* v_cache, int32_t* seq_lens, const void* k_new,
                          const void* v_new, int B, int g, int d, int S_max, int T,
                          int32_t* status, cudaStream_t s) {
  const int chunk_log2 = d == 64 ? 3 : 4;  // 16-byte chunks per row: 8 or 16
  const long long total = static_cast<long long>(B) * T * g << chunk_log2;
  long long blocks = (total + 255) / 256;
  if (blocks > 148LL * 32) blocks = 148LL * 32;  // grid-stride beyond 32 CTAs per SM
  if (blocks < 1) blocks = 1;
  // 32-bit indices whenever the range (plus one grid stride) fits
  if (total + 148LL * 32 * 256 < (1LL << 31))
    kv_append_rows_kernel<uint32_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), seq_lens,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, g, chunk_log2,
        S_max, T, status);
  else
    kv_append_rows_kernel<uint64_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), seq_lens,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), B, g, chunk_log2,
        S_max, T, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lens_update(seq_lens, B, S_max, T, s);
}

}  // namespace gqa
