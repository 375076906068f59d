// decode.cu -- one-token GQA decode over a [B, g, S_max, d] bf16 KV cache.
//
// The decode step of the "What is Grouped-Query Attention" explainer
// (ijyty.com), section 2.1: the new token's query attends over every cached
// K/V row. Design (split-KV, the split attention forward sketched in the
// "Qwen, DeepSeek and LLaMA3 attention survey" (jsqmd.com), chapter 5):
//
//  * pass 1 (decode_split_kernel): one CTA per (split, kv head, sequence).
//    It streams its split of the K and V rows through a TMA-fed shared-memory
//    ring (128-byte swizzle, so ldmatrix reads are bank-conflict free) and
//    serves ALL G = h_q/g query heads of the group from the same bytes: the G
//    query rows are stacked as the M side of m16n8k16 tensor-core MMAs. Each
//    K/V byte is read from HBM once per K/V head, never once per query head.
//    The CTA writes its normalised partial output and its log2 sum-exp.
//  * pass 2 (decode_combine_kernel): log-sum-exp combine of the partials.
#include <cuda_bf16.h>

#include "../../include/gqa.h"
#include "launch.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kStages = 2;     // ring depth (stages of kDecodeStage tokens)
constexpr int kThreads = 128;  // 4 warps

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// c += a * b for one m16n8k16 tile, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside one
// [rows x 128 B] box written by TMA with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace

// D: head dim (64 or 128). MT: m16 tiles of stacked query rows (G <= 16*MT).
template <int D, int MT>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ seq_lens,
    float* __restrict__ part_o, float* __restrict__ part_lse, int h_q, int g, int G,
    int n_hslice, int S_max, int split_len, int n_split, float scale_log2, int32_t* status) {
  constexpr int kBoxBytes = kDecodeStage * 128;       // 64 rows x 128 B
  constexpr int kCB = D / 64;                         // 64-wide column blocks
  constexpr int kStageBytes = 2 * kCB * kBoxBytes;    // K + V
  constexpr int kNSlices = 4 / MT;                    // warps sharing one m-tile
  constexpr int kSubPerWarp = (kDecodeStage / 16) / kNSlices;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ int abort_flag;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y / n_hslice;
  const int hs = blockIdx.y % n_hslice;  // 32-row slice of the group (G > 32 only)
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  int len = seq_lens[b];
  if (len < 0 || len > S_max) {
    if (tid == 0 && split == 0 && kvh == 0) record_status(status, GQA_ERR_BAD_LENGTH);
    len = len < 0 ? 0 : S_max;
  }
  const int s0 = split * split_len;
  if (s0 >= len) return;  // the combine pass ignores splits past the length
  const int s1 = min(len, s0 + split_len);
  const int n_st = (s1 - s0 + kDecodeStage - 1) / kDecodeStage;
  const int zrow = b * g + kvh;

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(&full_bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue_stage = [&](int st) {
    const int slot = st % kStages;
    uint8_t* base = smem + slot * kStageBytes;
    const int y = s0 + st * kDecodeStage;
    mbar_arrive_expect_tx(&full_bar[slot], kStageBytes);
#pragma unroll
    for (int cb = 0; cb < kCB; ++cb) {
      tma_load_3d(base + cb * kBoxBytes, &tm_k, &full_bar[slot], cb * 64, y, zrow);
      tma_load_3d(base + (kCB + cb) * kBoxBytes, &tm_v, &full_bar[slot], cb * 64, y, zrow);
    }
  };
  if (tid == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    for (int st = 0; st < kStages && st < n_st; ++st) issue_stage(st);
  }

  // ---- this warp's stacked query rows as m16n8k16 A fragments
  const int mt = warp % MT;
  const int slice = warp / MT;
  const int gr = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // fragment column pair
  const int row0 = mt * 16 + gr;
  const int row1 = row0 + 8;
  const size_t head0 = static_cast<size_t>(b) * h_q + static_cast<size_t>(kvh) * G + hs * 32;
  const int Gs = min(G - hs * 32, 16 * MT);  // stacked rows served by this CTA
  const __nv_bfloat16* qg = q + head0 * D;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int c = kk * 16 + tq * 2;
    qa[kk][0] = row0 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row0 * D + c) : 0u;
    qa[kk][1] = row1 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row1 * D + c) : 0u;
    qa[kk][2] = row0 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row0 * D + c + 8) : 0u;
    qa[kk][3] = row1 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row1 * D + c + 8) : 0u;
  }

  float o_acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};

  const uint32_t smem_base = smem_u32(smem);
  bool ok = true;
  for (int st = 0; st < n_st && ok; ++st) {
    const int slot = st % kStages;
    // every thread waits; the vote keeps `ok` uniform across the CTA so the
    // barriers below are never reached by only part of it
    ok = __syncthreads_and(mbar_wait(&full_bar[slot], (st / kStages) & 1, &abort_flag) ? 1 : 0);
    const int tok0 = s0 + st * kDecodeStage;
    const int valid = s1 - tok0;  // rows of this stage that are real
    const uint32_t kbase = smem_base + slot * kStageBytes;
    const uint32_t vbase = kbase + kCB * kBoxBytes;
    if (ok && valid < kDecodeStage) {
      // rows past the sequence may hold anything (even NaN); 0 * NaN would
      // poison P.V, so zero those V rows before any warp reads them
      uint8_t* vrows = smem + slot * kStageBytes + kCB * kBoxBytes;
      for (int i = tid; i < (kDecodeStage - valid) * kCB * 8; i += kThreads) {
        const int r = valid + i / (kCB * 8);
        const int cb = (i / 8) % kCB;
        const int ch = i % 8;
        *reinterpret_cast<uint4*>(vrows + cb * kBoxBytes + r * 128 + ch * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }
    if (ok) {
#pragma unroll
      for (int sbi = 0; sbi < kSubPerWarp; ++sbi) {
        const int r0 = (slice + sbi * kNSlices) * 16;  // first row of this 16-token block
        float s[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        // S = Q K^T over d
        {
          const int mi = lane >> 3;
          const int ri = lane & 7;
          const int tok = r0 + (mi >> 1) * 8 + ri;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int chunk = (kk * 2 + (mi & 1)) & 7;
            const uint32_t addr = kbase + (kk >> 2) * kBoxBytes + sw128(tok, chunk);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma16816(s[0], qa[kk], b0, b1);
            mma16816(s[1], qa[kk], b2, b3);
          }
        }
        // mask, scale to log2 units, online softmax for rows row0 / row1
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = r0 + j * 8 + tq * 2 + (e & 1);
            const float x = tok < valid ? s[j][e] * scale_log2 : -INFINITY;
            s[j][e] = x;
            mx[e >> 1] = fmaxf(mx[e >> 1], x);
          }
        }
        float alpha[2], m_use[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          const float m_new = fmaxf(m_r[h], mx[h]);
          // all-masked so far: keep everything at zero weight
          m_use[h] = m_new == -INFINITY ? 0.f : m_new;
          alpha[h] = ex2_approx(m_r[h] - m_use[h]);
          m_r[h] = m_new;
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p = ex2_approx(s[j][e] - m_use[e >> 1]);
            s[j][e] = p;
            rs[e >> 1] += p;
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 1);
          rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 2);
          l_r[h] = l_r[h] * alpha[h] + rs[h];
        }
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          o_acc[i][0] *= alpha[0];
          o_acc[i][1] *= alpha[0];
          o_acc[i][2] *= alpha[1];
          o_acc[i][3] *= alpha[1];
        }
        // P (bf16) as the A fragment of O += P V
        uint32_t pa[4];
        pa[0] = pack_bf16x2(s[0][0], s[0][1]);
        pa[1] = pack_bf16x2(s[0][2], s[0][3]);
        pa[2] = pack_bf16x2(s[1][0], s[1][1]);
        pa[3] = pack_bf16x2(s[1][2], s[1][3]);
        {
          const int mi = lane >> 3;
          const int ri = lane & 7;
          const int tok = r0 + (mi & 1) * 8 + ri;
#pragma unroll
          for (int np = 0; np < D / 16; ++np) {
            const int cg = np * 2 + (mi >> 1);
            const uint32_t addr = vbase + (cg >> 3) * kBoxBytes + sw128(tok, cg & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            mma16816(o_acc[np * 2], pa, b0, b1);
            mma16816(o_acc[np * 2 + 1], pa, b2, b3);
          }
        }
      }
    }
    __syncthreads();  // every warp is done with this slot
    if (tid == 0 && ok && !abort_flag && st + kStages < n_st) issue_stage(st + kStages);
  }

  if (!ok) {
    // drain TMA copies still in flight into the ring before leaving
    if (tid == 0) {
      for (int st = 0; st < n_st && st < kStages; ++st) {
        const int last = st + ((n_st - 1 - st) / kStages) * kStages;
        mbar_drain(&full_bar[last % kStages], (last / kStages) & 1);
      }
      record_status(status, GQA_ERR_TIMEOUT);
    }
    return;
  }

  // ---- merge the warps that share an m-tile, write this split's partial
  float* wm = reinterpret_cast<float*>(smem);            // [4][16]
  float* wl = wm + 4 * 16;                                // [4][16]
  float* wo = wl + 4 * 16;                                // [4][16][D]
  if (tq == 0) {
    wm[warp * 16 + gr] = m_r[0];
    wm[warp * 16 + gr + 8] = m_r[1];
    wl[warp * 16 + gr] = l_r[0];
    wl[warp * 16 + gr + 8] = l_r[1];
  }
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + tq * 2;
    wo[(warp * 16 + gr) * D + col] = o_acc[i][0];
    wo[(warp * 16 + gr) * D + col + 1] = o_acc[i][1];
    wo[(warp * 16 + gr + 8) * D + col] = o_acc[i][2];
    wo[(warp * 16 + gr + 8) * D + col + 1] = o_acc[i][3];
  }
  __syncthreads();
  for (int idx = tid; idx < Gs * D; idx += kThreads) {
    const int row = idx / D;
    const int col = idx % D;
    const int m_t = row >> 4;
    const int r = row & 15;
    float mc = -INFINITY;
#pragma unroll
    for (int sl = 0; sl < kNSlices; ++sl) mc = fmaxf(mc, wm[(sl * MT + m_t) * 16 + r]);
    float lc = 0.f, oc = 0.f;
#pragma unroll
    for (int sl = 0; sl < kNSlices; ++sl) {
      const int w = sl * MT + m_t;
      const float ms = wm[w * 16 + r];
      const float f = ms == -INFINITY ? 0.f : ex2_approx(ms - mc);
      lc += f * wl[w * 16 + r];
      oc += f * wo[(w * 16 + r) * D + col];
    }
    const size_t ps = (head0 + row) * n_split + split;
    part_o[ps * D + col] = oc / lc;
    if (col == 0) part_lse[ps] = mc + __log2f(lc);
  }
}

// One CTA per (sequence, query head): merge the splits that hold data.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int32_t* __restrict__ seq_lens, void* __restrict__ o, int o_dtype,
    float* __restrict__ lse_out, int h_q, int S_max, int split_len, int n_split) {
  const int bh = blockIdx.x;
  const int b = bh / h_q;
  const int col = threadIdx.x;
  int len = seq_lens[b];
  len = len < 0 ? 0 : (len > S_max ? S_max : len);
  const int n = (len + split_len - 1) / split_len;
  float out = 0.f;
  float lse_nat = -INFINITY;
  if (n > 0) {
    const float* pl = part_lse + static_cast<size_t>(bh) * n_split;
    float m = -INFINITY;
    for (int s = 0; s < n; ++s) m = fmaxf(m, pl[s]);
    float den = 0.f, num = 0.f;
    const float* po = part_o + static_cast<size_t>(bh) * n_split * D + col;
    for (int s = 0; s < n; ++s) {
      const float w = ex2_approx(pl[s] - m);
      den += w;
      num += w * po[static_cast<size_t>(s) * D];
    }
    out = num / den;
    lse_nat = (m + __log2f(den)) * 0.69314718055994531f;
  }
  if (o_dtype == GQA_OUT_F32) {
    static_cast<float*>(o)[static_cast<size_t>(bh) * D + col] = out;
  } else {
    static_cast<__nv_bfloat16*>(o)[static_cast<size_t>(bh) * D + col] = __float2bfloat16_rn(out);
  }
  if (lse_out != nullptr && col == 0) lse_out[bh] = lse_nat;
}

int decode_split_len(int B, int g, int S_max) {
  // Enough CTAs for several waves over 148 SMs while keeping each split long
  // enough that the partial-output traffic stays small next to the K/V bytes.
  const long long pairs = static_cast<long long>(B) * g;
  int split = 1024;
  while (split > kDecodeStage &&
         pairs * ((S_max + split - 1) / split) < 148LL * 8) {
    split /= 2;
  }
  return split;
}

template <int D, int MT>
static cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  constexpr int kSmem = kStages * 2 * (D / 64) * kDecodeStage * 128 + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_hslice = (a.G + 31) / 32;
  dim3 grid(a.n_split, a.g * n_hslice, a.B);
  decode_split_kernel<D, MT><<<grid, kThreads, kSmem, s>>>(
      a.tm_k, a.tm_v, static_cast<const __nv_bfloat16*>(a.q), a.seq_lens, a.part_o, a.part_lse,
      a.h_q, a.g, a.G, n_hslice, a.S_max, a.split_len, a.n_split, a.scale_log2, a.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D><<<a.B * a.h_q, D, 0, s>>>(a.part_o, a.part_lse, a.seq_lens, a.o,
                                                     a.o_dtype, a.lse, a.h_q, a.S_max,
                                                     a.split_len, a.n_split);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  // Groups larger than 32 query heads run as 32-row slices (grid.y), each
  // re-reading the split; no workload here has G > 32.
  const int mt = (a.G + 15) / 16;
  if (a.d == 64) return mt <= 1 ? launch_decode_t<64, 1>(a, s) : launch_decode_t<64, 2>(a, s);
  return mt <= 1 ? launch_decode_t<128, 1>(a, s) : launch_decode_t<128, 2>(a, s);
}

}  // namespace gqa
