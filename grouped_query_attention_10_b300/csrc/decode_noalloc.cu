// decode_noalloc.cu -- one-token decode for callers that cannot allocate.
//
// gqa_decode_fwd needs a caller-provided device workspace for its split-KV
// partial results. Some callers have no way to provide one: plugin hosts
// that hand a library only its input and output buffers while their own
// memory planner owns every other allocation, and serving loops that must
// not call cudaMalloc after start-up (it can synchronise the device and
// stall every stream). gqa_decode_fwd_noalloc serves them from a fixed
// scratch array that lives in this library's device image instead.
//
// The array is a file-scope __device__ variable: each GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits. In host
// code its name is only a host-side stand-in, never a device address, so the
// address is looked up with cudaGetSymbolAddress once per device (on the
// first call made while that device is current) and then reused.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/gqa.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return GQA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GQA_OK;
}

}  // namespace

extern "C" {

size_t gqa_decode_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int gqa_decode_fwd_noalloc(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B,
                           int h_q, int g, int d, int S_max, float scale, int32_t* status_dev,
                           void* stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr ||
      o == nullptr)
    return GQA_ERR_NULL;
  const size_t need = gqa_decode_workspace_bytes(B, h_q, g, d, S_max);
  if (need == 0) return GQA_ERR_SHAPE;
  if (need > kNoAllocScratchBytes) return GQA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != GQA_OK) return rc;
  return gqa_decode_fwd(q, k_cache, v_cache, seq_lens, o, o_dtype, lse, B, h_q, g, d, S_max,
                        scale, scratch, kNoAllocScratchBytes, status_dev, stream);
}

}  // extern "C"
