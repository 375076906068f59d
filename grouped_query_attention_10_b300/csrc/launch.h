// launch.h -- host-side launchers shared between the kernel files and the
// C interface (api.cu). Arguments are already validated when these run.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

namespace gqa {

// Devices a process may drive through this library (ordinals 0 .. 63).
constexpr int kMaxDevices = 64;

// One-time set-up that must happen on every device the library launches on
// (a kernel's dynamic shared-memory opt-in is a per-device attribute). Safe to
// call from several host threads; a set-up that failed is tried again on the
// next call.
struct DeviceOnce {
  std::mutex mu;
  std::atomic<bool> done[kMaxDevices] = {};
};

template <typename F>
cudaError_t run_once_per_device(DeviceOnce& once, F setup) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (once.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(once.mu);
  if (once.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess) once.done[dev].store(true, std::memory_order_release);
  return e;
}

// Streaming multiprocessors of the current device (looked up once per device).
inline int device_sm_count() {
  static std::atomic<int> count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 148;
  count[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Rows of one prefill query tile (TMEM lanes) and keys per K/V tile.
constexpr int kPrefillBM = 128;
constexpr int kPrefillBN = 128;

// Tokens per decode pipeline stage.
constexpr int kDecodeStage = 64;
// Most partial results the decode split pass writes per (query head, split):
// one per consumer warp's slice of the split's tokens.
constexpr int kDecodeSlices = 4;

struct PrefillArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // K/V maps are {d, g, keys, B} in either K/V layout
  CUtensorMap tm_o;  // output, 128-byte-wide column chunks (32 fp32 or 64 bf16)
  int o_dtype;
  float* lse;
  int B, Lq, Lk, S_max, h_q, g, d, G, G_log2;
  float scale_log2;  // softmax scale * log2(e)
  int causal;
  const int32_t* kv_lens;  // per-sequence key counts (K/V from a cache), or nullptr
  int window;              // sliding window (causal only), 0: none
  const float* alibi;      // per-query-head ALiBi slopes, or nullptr
  int32_t* status;
};

struct DecodeArgs {
  CUtensorMap tm_k, tm_v;
  const void* q;
  const int32_t* seq_lens;
  void* o;
  int o_dtype;
  float* lse;
  float* part_o;    // [B, h_q, n_split * slices, d]
  float* part_lse;  // [B, h_q, n_split * slices] (log2 units of the scaled scores)
  int* item_counter; // work-item counter of the split pass (zeroed before each launch)
  int B, h_q, g, d, G, S_max, split_len, n_split;
  float scale_log2;
  int window;          // sliding window (the last `window` rows), 0: none
  const float* alibi;  // per-query-head ALiBi slopes, or nullptr
  // paged cache (block_table != nullptr): K/V maps are {d, page_size, num_pages*g}
  const int32_t* block_table;  // [B, max_blocks] physical page of each logical block
  int page_log2, num_pages, max_blocks;
  int32_t* status;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_append(void* k_cache, void* v_cache, int32_t* seq_lens, const void* k_new,
                          const void* v_new, int B, int g, int d, int S_max, int T,
                          int32_t* status, cudaStream_t s);
// Paged variant: rows go through block_table [B, max_blocks] into a pool
// [num_pages, g, 1 << page_log2, d].
cudaError_t launch_append_paged(void* k_pool, void* v_pool, const int32_t* block_table,
                                int32_t* seq_lens, const void* k_new, const void* v_new, int B,
                                int g, int d, int page_log2, int num_pages, int max_blocks, int T,
                                int32_t* status, cudaStream_t s);

// Split length (tokens per split-KV CTA) used for these decode sizes.
int decode_split_len(int B, int h_q, int g, int S_max);

// RoPE append (contiguous cache when table == nullptr, else paged pool).
struct RopeAppendArgs {
  void* k_dst;                // [B, g, S_max, d] cache or [num_pages, g, page_size, d] pool
  void* v_dst;
  const int32_t* table;       // [B, max_blocks] page ids, or nullptr
  int page_log2, num_pages, max_blocks;
  int S_max;
  int32_t* seq_lens;
  const void* k_new;          // [B, T, g, d]
  const void* v_new;
  const void* q;              // [B, T, h_q, d] or nullptr (then h_q = 0)
  void* q_out;
  const float* cos;           // [n_pos, d / 2]
  const float* sin;
  int B, T, h_q, g, d;
  int32_t* status;
};
cudaError_t launch_append_rope(const RopeAppendArgs& a, cudaStream_t s);

cudaError_t launch_bounded_wait_selftest(int32_t* status, long long limit_ns, cudaStream_t s);

}  // namespace gqa
