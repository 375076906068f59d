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
// Work unit: one CTA per (query tile, K/V head, batch). A query tile holds
// 128 rows = (128 / G) consecutive positions x the G query heads of one K/V
// group, stacked position-major (the G heads of one position are contiguous
// in the [B, L, h_q, d] input, so a single 4-D TMA box fetches the tile).
// Every K/V tile the CTA loads therefore serves all G heads of the group.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q once, then K and V tiles through smem rings
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 4..7  softmax: warp w owns TMEM lanes 32*(w-4) .. +31 = tile rows
// Per K/V tile j: S_j = Q K_j^T (M=128, N=128, K=d) into one of two TMEM
// score buffers, so S_{j+1} is computed while the softmax works on S_j; the
// softmax writes P_j (bf16) into a 128-byte-swizzled smem tile and the MMA
// warp accumulates O += P_j V_j (M=128, N=d, K=128) into TMEM. The online
// softmax keeps a running row max in log2 units and rescales O lazily: only
// when some row's max grew by more than 2^8 (exact either way, because O and
// the row sum always share the same reference max).
#include <cuda_bf16.h>

#include "../../include/gqa.h"
#include "launch.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int BM = kPrefillBM;
constexpr int BN = kPrefillBN;
constexpr int kThreads = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct PrefillCfg {
  static constexpr int KS = D == 128 ? 2 : 3;  // K ring depth
  static constexpr int VS = KS;                 // V ring depth
  static constexpr uint32_t kQBytes = BM * D * 2;
  static constexpr uint32_t kKVStage = BN * D * 2;
  static constexpr uint32_t kPBytes = BM * BN * 2;
  static constexpr uint32_t kOffK = kQBytes;
  static constexpr uint32_t kOffV = kOffK + KS * kKVStage;
  static constexpr uint32_t kOffP = kOffV + VS * kKVStage;
  static constexpr uint32_t kSmem = kOffP + kPBytes + 1024;  // + alignment slack
};

}  // namespace

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o, int o_dtype,
    float* __restrict__ lse, int L, int h_q, int G, int G_log2, float scale_log2, int n_qtiles,
    int32_t* status) {
  using C = PrefillCfg<D>;
  constexpr int KS = C::KS;
  constexpr int VS = C::VS;
  constexpr uint32_t kTmS = 0;      // two score buffers: columns [0,128) and [128,256)
  constexpr uint32_t kTmO = 256;    // O accumulator: columns [256, 256 + D)
  constexpr uint32_t kTmCols = 512;
  constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, false);  // Q (K-major) x K (K-major)
  constexpr uint32_t kIdescO = idesc_bf16_f32(BM, D, true);    // P (K-major) x V (MN-major)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bar_q;
  __shared__ __align__(8) uint64_t bar_kf[KS];
  __shared__ __align__(8) uint64_t bar_ke[KS];
  __shared__ __align__(8) uint64_t bar_vf[VS];
  __shared__ __align__(8) uint64_t bar_ve[VS];
  __shared__ __align__(8) uint64_t bar_sf[2];     // S_j ready in TMEM buffer j&1
  __shared__ __align__(8) uint64_t bar_sfree[2];  // softmax has read TMEM buffer
  __shared__ __align__(8) uint64_t bar_p;         // P_j written to smem
  __shared__ __align__(8) uint64_t bar_o;         // PV_j retired (O updated, P free)
  __shared__ __align__(8) uint64_t bar_fin;       // every MMA retired
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = CAUSAL ? (n_qtiles - 1 - static_cast<int>(blockIdx.x)) : blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int PM = BM >> G_log2;  // positions per query tile
  const int p0 = qt * PM;
  const int kv_end = CAUSAL ? min(L, p0 + PM) : L;
  const int n_kv = (kv_end + BN - 1) / BN;

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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_sf[i], 1);
      mbar_init(&bar_sfree[i], 128);
    }
    mbar_init(&bar_p, 128);
    mbar_init(&bar_o, 1);
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
      mbar_arrive_expect_tx(&bar_q, C::kQBytes);
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb)
        tma_load_4d(smem + cb * (BM * 128), &tm_q, &bar_q, cb * 64, kvh * G, p0, b);
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
    if (lane == 0) {
      const uint32_t sQ = smem_u32(smem);
      const uint32_t sK = sQ + C::kOffK;
      const uint32_t sV = sQ + C::kOffV;
      const uint32_t sP = sQ + C::kOffP;
      bool ok = mbar_wait(&bar_q, 0, &abort_flag);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          const int ks = j % KS;
          ok = mbar_wait(&bar_kf[ks], (j / KS) & 1, &abort_flag);
          if (ok && j >= 2) ok = mbar_wait(&bar_sfree[j & 1], ((j - 2) >> 1) & 1, &abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_s = tmem + kTmS + static_cast<uint32_t>(j & 1) * BN;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad =
                smem_desc_sw128(sQ + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(
                sK + ks * C::kKVStage + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
            mma_bf16_ss(d_s, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bar_sf[j & 1]);
          mma_commit(&bar_ke[ks]);
        }
        if (j >= 1) {
          const int i = j - 1;
          const int vs = i % VS;
          ok = mbar_wait(&bar_p, i & 1, &abort_flag);
          if (ok) ok = mbar_wait(&bar_vf[vs], (i / VS) & 1, &abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad =
                smem_desc_sw128(sP + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
            // V tile [BN keys x D] with D contiguous: MN-major B operand;
            // LBO = distance between 64-wide column blocks of D
            const uint64_t bd =
                smem_desc_sw128(sV + vs * C::kKVStage + kk * (16 * 128), BN * 128, 1024);
            mma_bf16_ss(tmem + kTmO, ad, bd, kIdescO, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bar_o);
          mma_commit(&bar_ve[vs]);
        }
      }
      // every MMA must have retired before TMEM is released
      mma_commit(&bar_fin);
      mbar_drain(&bar_fin, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp - 4;
    const int row = q4 * 32 + lane;
    const int pos = p0 + (row >> G_log2);
    const int head = kvh * G + (row & (G - 1));
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    uint8_t* p_row = smem + C::kOffP + row * 128;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s, possibly stale by < 2^8
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int buf = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_sf[buf], (j >> 1) & 1, &abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(t_lane + kTmS + buf * BN + c * 32, sr + c * 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bar_sfree[buf]);
      float s[BN];
#pragma unroll
      for (int e = 0; e < BN; ++e) s[e] = __uint_as_float(sr[e]);

      const int key0 = j * BN;
      const bool need_mask = (key0 + BN > L) || (CAUSAL && key0 + BN - 1 > p0);
      float mx = -INFINITY;
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int key = key0 + e;
          const bool vis = key < L && (!CAUSAL || key <= pos);
          s[e] = vis ? s[e] : -INFINITY;
          mx = fmaxf(mx, s[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < BN; ++e) mx = fmaxf(mx, s[e]);
      }
      const float m_new = fmaxf(m_run, mx * scale_log2);
      bool waited_o = false;
      if (__any_sync(0xffffffffu, m_new > m_run + kRescaleThreshold)) {
        // the whole warp adopts its new maxima (tcgen05.ld/st are warp-wide)
        const float alpha = (m_run == -INFINITY || m_new == -INFINITY)
                                ? (m_run == -INFINITY ? 0.f : 1.f)
                                : ex2_approx(m_run - m_new);
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_o, (j - 1) & 1, &abort_flag));
          if (!ok) break;
          waited_o = true;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(t_lane + kTmO + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(t_lane + kTmO + c * 32, r);
          }
          tmem_st_wait();
        }
        l_run *= alpha;
        m_run = m_new;
      }
      // P = 2^(s * scale * log2(e) - m_run), packed to bf16 pairs
      uint32_t pk[BN / 2];
      float rsum = 0.f;
#pragma unroll
      for (int e = 0; e < BN / 2; ++e) {
        const float pa = ex2_approx(fmaf(s[2 * e], scale_log2, -m_run));
        const float pb = ex2_approx(fmaf(s[2 * e + 1], scale_log2, -m_run));
        rsum += pa + pb;
        pk[e] = pack_bf16x2(pa, pb);
      }
      l_run += rsum;
      if (j > 0 && !waited_o) {
        // P_{j-1} is still being read by PV_{j-1}
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_o, (j - 1) & 1, &abort_flag));
        if (!ok) break;
      }
#pragma unroll
      for (int c = 0; c < BN / 8; ++c) {
        const int phys = (c & 7) ^ (row & 7);
        *reinterpret_cast<uint4*>(p_row + (c >> 3) * (BM * 128) + phys * 16) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();  // generic-proxy P writes -> tensor-core reads
      tc_fence_before();
      mbar_arrive(&bar_p);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar_o, (n_kv - 1) & 1, &abort_flag));
    if (ok) {
      tc_fence_after();
      const bool store = pos < L;
      const float inv_l = 1.f / l_run;
      const size_t orow = (static_cast<size_t>(b) * L + pos) * h_q + head;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_lane + kTmO + c * 32, r);
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
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const float lo = __uint_as_float(r[8 * e + 2 * t]) * inv_l;
                const float hi = __uint_as_float(r[8 * e + 2 * t + 1]) * inv_l;
                __nv_bfloat162 v2 = __floats2bfloat162_rn(lo, hi);
                w[t] = *reinterpret_cast<uint32_t*>(&v2);
              }
              dst[e] = make_uint4(w[0], w[1], w[2], w[3]);
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
  const int n_qtiles = (a.L + PM - 1) / PM;
  dim3 grid(n_qtiles, a.g, a.B);
  prefill_kernel<D, CAUSAL><<<grid, kThreads, kSmem, s>>>(
      a.tm_q, a.tm_k, a.tm_v, a.o, a.o_dtype, a.lse, a.L, a.h_q, a.G, a.G_log2, a.scale_log2,
      n_qtiles, a.status);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  if (a.d == 64)
    return a.causal ? launch_prefill_t<64, true>(a, s) : launch_prefill_t<64, false>(a, s);
  return a.causal ? launch_prefill_t<128, true>(a, s) : launch_prefill_t<128, false>(a, s);
}

}  // namespace gqa
