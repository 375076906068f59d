// prefill.cu -- GQA prefill forward on tcgen05 tensor cores with TMEM
// accumulators (sm_103a).
//
// Computes, per (batch, query head h, query row i),
//   O = softmax_j(scale * Q_i . K_j) V_j,  K/V head = h / G,  G = h_q / g,
// over all keys or over j <= i (causal): the GroupedQueryAttention forward of
// "Modern LLM architecture (1): GQA and RMSNorm" (zeeklog.com), section 2.3,
// without the repeat_interleave: K/V tiles are loaded once and shared by the
// whole group. The score matrix never leaves the chip (the on-chip softmax
// the ijyty.com explainer credits to FlashAttention, section 4.3).
//
// Work unit: one CTA per (pair of query tiles, K/V head, batch). A query tile
// holds 128 rows = (128 / G) consecutive positions x the G query heads of one
// K/V group, stacked position-major (the G heads of one position are
// contiguous in the [B, L, h_q, d] input, so one 4-D TMA box fetches a tile).
// The two tiles cover consecutive positions and share every K/V tile the CTA
// loads, so each K/V byte brought into shared memory serves 2 x 128 rows of
// all G heads of the group.
//
// Warp roles (384 threads):
//   warp 0        TMA producer: both query tiles once, then K and V tiles
//                 through shared-memory rings
//   warp 1        TMEM allocator + tcgen05.mma issuer (the warp walks the
//                 schedule, one elected lane issues)
//   warps 4..7    softmax of query tile 0 (warp w owns TMEM lanes 32*(w%4)..)
//   warps 8..11   softmax of query tile 1
// TMEM (512 columns): S_t = scores of tile t (128 columns), O_t = output
// accumulator of tile t (d columns). The softmax writes P_t (bf16, two per
// 32-bit column) over the first 64 columns of S_t and the P.V product reads
// it from there (A operand in TMEM), so P never touches shared memory.
//
// MMA issue order per K/V tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1). One
// thread issues every MMA, and tcgen05 MMAs from one thread execute in order,
// so S_t(j+1) overwrites S_t/P_t only after PV_t(j) has read P_t, and the
// commit that announces S_t(j+1) also covers PV_t(j): when the softmax sees
// S_t(j+1), O_t is final for keys < (j+1)*128 and may be rescaled in place.
// While the softmax of one tile runs, the tensor core works on the other.
//
// The online softmax keeps a running row max in log2 units and rescales O
// lazily: only when some row's max grew by more than 2^8 (exact either way,
// because O and the row sum always share the same reference max).
#include <cuda_bf16.h>

#include "../../include/gqa.h"
#include "launch.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int BM = kPrefillBM;
constexpr int BN = kPrefillBN;
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct PrefillCfg {
  static constexpr int KS = D == 128 ? 2 : 4;  // K ring depth
  static constexpr int VS = KS;                 // V ring depth
  static constexpr uint32_t kQTile = BM * D * 2;
  static constexpr uint32_t kKVStage = BN * D * 2;
  static constexpr uint32_t kOffK = 2 * kQTile;
  static constexpr uint32_t kOffV = kOffK + KS * kKVStage;
  static constexpr uint32_t kSmem = kOffV + VS * kKVStage + 1024;  // + alignment slack
};

// Row max of one 128-key score tile in TMEM (three-input max, four chains).
// With MASK, columns e > nvis (relative to the tile) are ignored.
template <bool MASK>
__device__ __forceinline__ float tile_row_max(uint32_t t_s, int nvis) {
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t r[64];
    tmem_ld32(t_s + h * 64, r);
    tmem_ld32(t_s + h * 64 + 32, r + 32);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float a = __uint_as_float(r[2 * e]);
      float b = __uint_as_float(r[2 * e + 1]);
      if (MASK) {
        if (h * 64 + 2 * e > nvis) a = -INFINITY;
        if (h * 64 + 2 * e + 1 > nvis) b = -INFINITY;
      }
      mx4[e & 3] = max3f(mx4[e & 3], a, b);
    }
  }
  return max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
}

// P = 2^(s * scale_log2 - m) for one 128-key tile, written as bf16 pairs over
// the first 64 TMEM columns of the tile; returns the row sum of P (fp32).
// Scale-and-shift and the running sum use packed two-lane fp32 ops.
template <bool MASK>
__device__ __forceinline__ float tile_exp_to_p(uint32_t t_s, int nvis, float scale_log2,
                                               float m) {
  const uint64_t c2 = f32x2(scale_log2, scale_log2);
  const uint64_t nm2 = f32x2(-m, -m);
  uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t r[64];
    tmem_ld32(t_s + h * 64, r);
    tmem_ld32(t_s + h * 64 + 32, r + 32);
    tmem_ld_wait();
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float xa, xb;
      split_f32x2(ffma_x2(u32x2(r[2 * e], r[2 * e + 1]), c2, nm2), xa, xb);
      float pa = ex2_approx(xa);
      float pb = ex2_approx(xb);
      if (MASK) {
        if (h * 64 + 2 * e > nvis) pa = 0.f;
        if (h * 64 + 2 * e + 1 > nvis) pb = 0.f;
      }
      sum2[e & 1] = fadd_x2(sum2[e & 1], f32x2(pa, pb));
      w[e] = pack_bf16x2(pa, pb);
    }
    tmem_st32(t_s + h * 32, w);  // P columns [32h, 32h+32) hold keys [64h, 64h+64)
  }
  float a0, a1, b0, b1;
  split_f32x2(sum2[0], a0, a1);
  split_f32x2(sum2[1], b0, b1);
  return (a0 + a1) + (b0 + b1);
}

}  // namespace

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o, int o_dtype,
    float* __restrict__ lse, int L, int h_q, int G, int G_log2, float scale_log2, int n_ctiles,
    int32_t* status) {
  using C = PrefillCfg<D>;
  constexpr int KS = C::KS;
  constexpr int VS = C::VS;
  constexpr uint32_t kTmCols = 512;
  constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, false);  // Q (K-major) x K (K-major)
  constexpr uint32_t kIdescO = idesc_bf16_f32(BM, D, true);    // P (TMEM) x V (MN-major)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bar_q;
  __shared__ __align__(8) uint64_t bar_kf[KS];
  __shared__ __align__(8) uint64_t bar_ke[KS];
  __shared__ __align__(8) uint64_t bar_vf[VS];
  __shared__ __align__(8) uint64_t bar_ve[VS];
  __shared__ __align__(8) uint64_t bar_s[2];  // S_t(j) in TMEM (and PV_t(j-1) retired)
  __shared__ __align__(8) uint64_t bar_p[2];  // P_t(j) written to TMEM, O_t rescaled
  __shared__ __align__(8) uint64_t bar_o[2];  // PV_t(j) retired
  __shared__ __align__(8) uint64_t bar_fin;   // every MMA retired
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ct = CAUSAL ? (n_ctiles - 1 - static_cast<int>(blockIdx.x)) : blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int PM = BM >> G_log2;  // positions per query tile
  const int p0 = ct * 2 * PM;
  // K/V tiles each query tile needs (0 for a tile that lies wholly past L)
  const int n_kv0 = (CAUSAL ? min(L, p0 + PM) + BN - 1 : L + BN - 1) / BN;
  const int n_kv1 =
      p0 + PM < L ? (CAUSAL ? min(L, p0 + 2 * PM) + BN - 1 : L + BN - 1) / BN : 0;
  const int n_kv = max(n_kv0, n_kv1);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    for (int i = 0; i < KS; ++i) {
      mbar_init(&bar_kf[i], 1);
      mbar_init(&bar_ke[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&bar_vf[i], 1);
      mbar_init(&bar_ve[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 128);
      mbar_init(&bar_o[t], 1);
    }
    mbar_init(&bar_fin, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const int n_qt = n_kv1 > 0 ? 2 : 1;
      mbar_arrive_expect_tx(&bar_q, n_qt * C::kQTile);
      for (int t = 0; t < n_qt; ++t) {
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_4d(smem + t * C::kQTile + cb * (BM * 128), &tm_q, &bar_q, cb * 64, kvh * G,
                      p0 + t * PM, b);
      }
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ks = j % KS;
        if (j >= KS) ok = mbar_wait(&bar_ke[ks], ((j / KS) - 1) & 1, &abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_kf[ks], C::kKVStage);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_4d(smem + C::kOffK + ks * C::kKVStage + cb * (BN * 128), &tm_k, &bar_kf[ks],
                      cb * 64, kvh, j * BN, b);
        issued_k = j + 1;
        const int vs = j % VS;
        if (j >= VS) ok = mbar_wait(&bar_ve[vs], ((j / VS) - 1) & 1, &abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_vf[vs], C::kKVStage);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_4d(smem + C::kOffV + vs * C::kKVStage + cb * (BN * 128), &tm_v, &bar_vf[vs],
                      cb * 64, kvh, j * BN, b);
        issued_v = j + 1;
      }
      // every issued copy must have landed before the CTA may exit
      mbar_drain(&bar_q, 0);
      for (int s = 0; s < KS && s < issued_k; ++s) {
        const int last = s + ((issued_k - 1 - s) / KS) * KS;
        mbar_drain(&bar_kf[s], (last / KS) & 1);
      }
      for (int s = 0; s < VS && s < issued_v; ++s) {
        const int last = s + ((issued_v - 1 - s) / VS) * VS;
        mbar_drain(&bar_vf[s], (last / VS) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the schedule (so it stays converged and keeps the
    // descriptors in uniform registers); one elected lane issues the MMAs.
    const bool leader = elect_one();
    const uint32_t sQ = smem_u32(smem);
    // descriptor bases; a k-step only moves the 14-bit start-address field
    const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sQ + C::kOffK, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sQ + C::kOffV, BN * 128, 1024);
    // byte offset (>> 4) of k-step kk inside a K-major 128-byte-swizzled tile
    auto kmaj = [](int kk) -> uint64_t {
      return static_cast<uint64_t>(((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4);
    };
    auto issue_s = [&](int t, int ks) {
      const uint32_t d_s = tmem + static_cast<uint32_t>(t) * BN;
      const uint64_t aq = dq0 + ((t * C::kQTile) >> 4);
      const uint64_t bk = dk0 + ((ks * C::kKVStage) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_ss(d_s, aq + kmaj(kk), bk + kmaj(kk), kIdescS, kk > 0 ? 1u : 0u);
      mma_commit(&bar_s[t]);
    };
    auto issue_pv = [&](int t, int vs, bool first) {
      const uint32_t p_t = tmem + static_cast<uint32_t>(t) * BN;  // P_t over S_t
      const uint32_t o_t = tmem + 2 * BN + static_cast<uint32_t>(t) * D;
      // V tile [BN keys x D], D contiguous: MN-major B operand; LBO = distance
      // between the 64-wide column blocks of D; a k-step is 16 rows of 128 B
      const uint64_t bv = dv0 + ((vs * C::kKVStage) >> 4);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)
        mma_bf16_ts(o_t, p_t + kk * 8, bv + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                    kIdescO, (!first || kk > 0) ? 1u : 0u);
      mma_commit(&bar_o[t]);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag));
    };

    bool ok = wait_all(&bar_q, 0) && wait_all(&bar_kf[0], 0);
    if (ok) {
      tc_fence_after();
      if (leader) {
        issue_s(0, 0);
        if (n_kv1 > 0) issue_s(1, 0);
        mma_commit(&bar_ke[0]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const int vs = j % VS;
      const int nx = j + 1;
      const int ks = nx % KS;
      ok = wait_all(&bar_vf[vs], (j / VS) & 1);
      if (ok && nx < n_kv) ok = wait_all(&bar_kf[ks], (nx / KS) & 1);
      for (int t = 0; ok && t < 2; ++t) {
        const int n_t = t == 0 ? n_kv0 : n_kv1;
        if (j >= n_t) continue;
        ok = wait_all(&bar_p[t], j & 1);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
          issue_pv(t, vs, j == 0);
          if (nx < n_t) issue_s(t, ks);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) {
        mma_commit(&bar_ve[vs]);
        if (nx < n_kv) mma_commit(&bar_ke[ks]);
      }
      __syncwarp();
    }
    // every MMA must have retired before TMEM is released
    if (leader) {
      mma_commit(&bar_fin);
      mbar_drain(&bar_fin, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;        // TMEM lane quadrant
    const int row = wq * 32 + lane;
    const int pt = p0 + t * PM;
    const int pos = pt + (row >> G_log2);
    const int head = kvh * G + (row & (G - 1));
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + static_cast<uint32_t>(t) * BN;
    const uint32_t t_o = tmem + lane_base + 2 * BN + static_cast<uint32_t>(t) * D;
    const int n_my = t == 0 ? n_kv0 : n_kv1;
    // last key this row may see
    const int last_key = CAUSAL ? min(L - 1, pos) : L - 1;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s, possibly stale by < 2^8
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_my; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[t], j & 1, &abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int key0 = j * BN;
      const bool need_mask = (key0 + BN > L) || (CAUSAL && key0 + BN - 1 > pt);
      const int nvis = last_key - key0;  // tile columns e <= nvis are visible
      const float mx = need_mask ? tile_row_max<true>(t_s, nvis) : tile_row_max<false>(t_s, nvis);
      const float m_new = fmaxf(m_run, mx * scale_log2);
      if (__any_sync(0xffffffffu, m_new > m_run + kRescaleThreshold)) {
        // the whole warp adopts its new maxima (tcgen05.ld/st are warp-wide)
        const float alpha = m_run == -INFINITY ? 0.f : ex2_approx(m_run - m_new);
        if (j > 0) {
          // O_t holds keys < j*128 and no MMA writes it until P_t(j) is ready
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(t_o + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(t_o + c * 32, r);
          }
        }
        l_run *= alpha;
        m_run = m_new;
      }
      // P = 2^(s * scale * log2(e) - m_run) as bf16 pairs over S_t
      l_run += need_mask ? tile_exp_to_p<true>(t_s, nvis, scale_log2, m_run)
                         : tile_exp_to_p<false>(t_s, nvis, scale_log2, m_run);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_p[t]);
    }
    if (ok && n_my > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[t], (n_my - 1) & 1, &abort_flag));
    if (ok && n_my > 0) {
      tc_fence_after();
      const bool store = pos < L;
      const float inv_l = 1.f / l_run;
      const size_t orow = (static_cast<size_t>(b) * L + pos) * h_q + head;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_o + c * 32, r);
        tmem_ld_wait();
        if (store) {
          if (o_dtype == GQA_OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(o) + orow * D + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv_l,
                                   __uint_as_float(r[4 * e + 1]) * inv_l,
                                   __uint_as_float(r[4 * e + 2]) * inv_l,
                                   __uint_as_float(r[4 * e + 3]) * inv_l);
          } else {
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + orow * D + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint32_t wv[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float lo = __uint_as_float(r[8 * e + 2 * q]) * inv_l;
                const float hi = __uint_as_float(r[8 * e + 2 * q + 1]) * inv_l;
                __nv_bfloat162 v2 = __floats2bfloat162_rn(lo, hi);
                wv[q] = *reinterpret_cast<uint32_t*>(&v2);
              }
              dst[e] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
        }
      }
      if (lse != nullptr && store)
        lse[(static_cast<size_t>(b) * h_q + head) * L + pos] =
            (m_run + __log2f(l_run)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
  if (threadIdx.x == 0 && abort_flag) record_status(status, GQA_ERR_TIMEOUT);
}

template <int D, bool CAUSAL>
static cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t s) {
  constexpr uint32_t kSmem = PrefillCfg<D>::kSmem;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, CAUSAL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int PM = BM / a.G;
  const int n_ctiles = (a.L + 2 * PM - 1) / (2 * PM);
  dim3 grid(n_ctiles, a.g, a.B);
  prefill_kernel<D, CAUSAL><<<grid, kThreads, kSmem, s>>>(
      a.tm_q, a.tm_k, a.tm_v, a.o, a.o_dtype, a.lse, a.L, a.h_q, a.G, a.G_log2, a.scale_log2,
      n_ctiles, a.status);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  if (a.d == 64)
    return a.causal ? launch_prefill_t<64, true>(a, s) : launch_prefill_t<64, false>(a, s);
  return a.causal ? launch_prefill_t<128, true>(a, s) : launch_prefill_t<128, false>(a, s);
}

}  // namespace gqa
