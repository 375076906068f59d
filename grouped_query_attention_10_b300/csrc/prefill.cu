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
// Work unit: (pair of query tiles, K/V head, batch). A query tile holds 128
// rows = (128 / G) consecutive positions x the G query heads of one K/V
// group, stacked position-major (the G heads of one position are contiguous
// in the [B, L, h_q, d] input, so one 4-D TMA box fetches a tile). The two
// tiles cover consecutive positions and share every K/V tile the CTA loads,
// so each K/V byte brought into shared memory serves 2 x 128 rows of all G
// heads of the group.
//
// The kernel is persistent: one CTA per SM walks the units u = blockIdx.x,
// blockIdx.x + gridDim.x, ... (causal units ordered longest first). The K/V
// rings, the barrier phases and the TMEM buffers carry over from one unit to
// the next, so the loads and score products of the next unit overlap the
// output epilogue of the current one.
//
// Warp roles (384 threads):
//   warp 0        TMA producer: query tiles, then K and V tiles through
//                 shared-memory rings
//   warp 1        TMEM allocator + tcgen05.mma issuer (d = 64: of query
//                 tile 0; d = 128: of both query tiles, in a fixed order)
//   warp 2        d = 64: tcgen05.mma issuer of query tile 1 (each issuer
//                 warp walks the schedule, one elected lane issues)
//   warps 4..7    softmax + epilogue of query tile 0 (warp w owns TMEM lanes
//                 32*(w%4)..)
//   warps 8..11   softmax + epilogue of query tile 1
// TMEM (512 columns): S_t = scores of tile t (128 columns), O_t = output
// accumulator of tile t (d columns), P_t = probabilities (bf16, two per
// 32-bit column, 64 columns) read by the P.V product as the A operand.
//  * d = 64: P_t has columns of its own. The softmax releases S_t as soon as
//    it has read the scores into registers, so S_t(j+1) = Q K_{j+1}^T runs on
//    the tensor core while the exponentials of tile j are computed.
//  * d = 128: S and O fill TMEM, so P_t overwrites the first 64 columns of
//    S_t and S_t(j+1) is issued after P_t(j).V_j (one thread issues all of
//    tile t's MMAs, and tcgen05 MMAs from one thread execute in order). The
//    softmax hands P_t over in two halves (keys 0..63, then 64..127), so the
//    first half of P_t.V runs while the second half's exponentials are
//    computed.
// While the softmax of one tile runs, the tensor core works on the other.
//
// Every K (V) ring slot is released by a commit issued right after the last
// score (P.V) product that reads it, so the producer can refill it as soon
// as that product retires; with the 2-deep rings of d = 128 a release one
// product later left the next K tile still in flight when its score product
// was due.
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

// Register plan. The kernel is built for 168 registers per thread (the most
// 384 threads may hold on one SM); right after set-up the control warpgroup
// (producer, two MMA issuers, one idle warp) gives registers back and the two
// softmax warpgroups take them, so a softmax thread can hold a whole
// 128-column score row. The launcher refuses to launch unless the built
// kernel uses exactly kRegsLaunch registers, so the increase always finds
// the registers the decrease released.
constexpr int kRegsLaunch = 168;
constexpr int kRegsCtl = 88;
constexpr int kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register plan exceeds the launch pool");
static_assert(kThreads * kRegsLaunch <= 65536, "launch pool exceeds the register file");

// lo += the bf16 in bits 0..15 of w, hi += the bf16 in bits 16..31: each
// widened exactly to fp32 and added with one rounding (mixed-precision add of
// sm_100 and later)
__device__ __forceinline__ void add_bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.bf16 %0, l, %0; "
      "add.rn.f32.bf16 %1, h, %1; }"
      : "+f"(lo), "+f"(hi)
      : "r"(w));
}

template <int D>
struct PrefillCfg {
  static constexpr bool kSepP = D == 64;           // P_t has TMEM columns of its own
  static constexpr int NQ = D == 64 ? 2 : 1;       // query-tile buffers (units in flight)
  static constexpr int KS = D == 128 ? 2 : 3;      // K ring depth
  static constexpr int VS = KS;                    // V ring depth
  static constexpr uint32_t kQTile = BM * D * 2;   // one 128-row query tile
  static constexpr uint32_t kQSlot = 2 * kQTile;   // both query tiles of a unit
  static constexpr uint32_t kKVStage = BN * D * 2;
  static constexpr uint32_t kOffK = NQ * kQSlot;
  static constexpr uint32_t kOffV = kOffK + KS * kKVStage;
  // Output staging, per query tile: 128 rows x kStageChunks 128-byte column
  // chunks (a chunk = 32 fp32 or 64 bf16 columns), written by the softmax
  // threads and stored by TMA (d = 64: the whole tile in one pass). Each warp
  // owns the 32 rows (4 KB of every chunk) of its TMEM lane quadrant and
  // stores them itself.
  static constexpr int kStageChunks = D == 64 ? 2 : 1;
  static constexpr uint32_t kChunkBytes = BM * 128;
  static constexpr uint32_t kStageBytes = kStageChunks * kChunkBytes;
  static constexpr uint32_t kOffStage = kOffV + VS * kKVStage;
  static constexpr uint32_t kSmem = kOffStage + 2 * kStageBytes + 1024;  // + alignment slack
  // TMEM columns
  static constexpr uint32_t kColO = 2 * BN;                   // O_t at kColO + t * D
  static constexpr uint32_t kColP = kSepP ? 2 * BN + 2 * D : 0;
  static constexpr uint32_t kStrideP = kSepP ? BN / 2 : BN;   // P_t at kColP + t * kStrideP
};

// Runtime sizes and options of one launch (kernel parameter, read-only).
struct PrefillParams {
  float* lse;                // [B, h_q, Lq] natural-log sum-exp, or nullptr
  int o_dtype;
  int B, Lq, Lk, S_max;      // Lk: keys per sequence unless kv_lens is given
  int h_q, g, G, G_log2;
  float scale_log2;          // softmax scale * log2(e)
  int n_ctiles, n_units;
  const int32_t* kv_lens;    // per-sequence key counts (K/V read from a cache), or nullptr
  int window;                // sliding window in keys (causal only), 0: none
  const float* alibi;        // per-query-head ALiBi slopes (natural units), or nullptr
  int32_t* status;
};

// One decoded work unit.
struct Unit {
  int b, kvh, p0;  // batch, K/V head, first position of query tile 0
  int Lk, q_off;   // keys of this sequence; query position i sits at key position i + q_off
  int kv0;         // first K/V tile the unit reads (all earlier keys are outside the window)
  int n0, n1;      // K/V tiles from kv0 on seen by query tile 0 / 1 (n1 = 0: tile 1 past Lq)
};

__device__ __forceinline__ Unit decode_unit(int u, const PrefillParams& p, int PM, bool causal,
                                            bool windowed, bool cached) {
  const int n_pairs = p.g * p.B;  // (batch, K/V head) pairs
  int ct, pair;
  if (causal) {
    // longest units first (later query tiles see more keys), dealt to the
    // CTAs in snake order (every other round reversed) so that each CTA's
    // total work comes out nearly equal
    const int G0 = static_cast<int>(gridDim.x);
    const int round = u / G0;
    const bool flip = (round & 1) && (round + 1) * G0 <= p.n_units;  // full rounds only
    const int r = flip ? round * G0 + (G0 - 1 - u % G0) : u;
    ct = p.n_ctiles - 1 - r / n_pairs;
    pair = r % n_pairs;
  } else {
    // consecutive units share the (batch, K/V head), so CTAs that run at the
    // same time read the same K/V tiles and hit in L2
    ct = u % p.n_ctiles;
    pair = u / p.n_ctiles;
  }
  Unit w;
  w.kvh = pair % p.g;
  w.b = pair / p.g;
  w.p0 = ct * 2 * PM;
  w.Lk = p.Lk;
  if (cached) {
    // keys in the cache; the new queries are its last Lq rows
    const int n = p.kv_lens[w.b];
    w.Lk = n < p.Lq ? p.Lq : (n > p.S_max ? p.S_max : n);
  }
  w.q_off = causal ? w.Lk - p.Lq : 0;
  const int lo0 = windowed ? max(0, w.q_off + w.p0 - p.window + 1) : 0;
  w.kv0 = lo0 / BN;
  const int last0 = min(p.Lq, w.p0 + PM) - 1;
  const int hi0 = causal ? min(w.Lk - 1, w.q_off + last0) : w.Lk - 1;
  w.n0 = hi0 / BN - w.kv0 + 1;
  if (w.p0 + PM < p.Lq) {
    const int last1 = min(p.Lq, w.p0 + 2 * PM) - 1;
    const int hi1 = causal ? min(w.Lk - 1, w.q_off + last1) : w.Lk - 1;
    w.n1 = hi1 / BN - w.kv0 + 1;
  } else {
    w.n1 = 0;
  }
  return w;
}

// Drain helper for the abort path: wait (bounded) for the last fill issued
// into every slot of a ring whose fills were numbered 0 .. issued-1.
__device__ __forceinline__ void drain_ring(uint64_t* full, int depth, int issued) {
  for (int s = 0; s < depth && s < issued; ++s) {
    const int last = s + ((issued - 1 - s) / depth) * depth;
    mbar_drain(&full[s], (last / depth) & 1);
  }
}

}  // namespace

// VAR: bit 0 = sliding window, bit 1 = ALiBi bias, bit 2 = K/V read from a
// [B, g, S_max, d] cache with per-sequence key counts (chunked prefill).
template <int D, bool CAUSAL, int VAR>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
    const PrefillParams p) {
  constexpr bool kWindow = (VAR & 1) != 0;
  constexpr bool kAlibi = (VAR & 2) != 0;
  constexpr bool kCache = (VAR & 4) != 0;
  const int g = p.g, G = p.G, G_log2 = p.G_log2, h_q = p.h_q, n_units = p.n_units;
  using C = PrefillCfg<D>;
  constexpr int KS = C::KS;
  constexpr int VS = C::VS;
  constexpr int NQ = C::NQ;
  constexpr bool kSepP = C::kSepP;
  constexpr uint32_t kTmCols = 512;
  constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, false);  // Q (K-major) x K (K-major)
  constexpr uint32_t kIdescO = idesc_bf16_f32(BM, D, true);    // P (TMEM) x V (MN-major)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bar_q[NQ];   // query tiles landed
  __shared__ __align__(8) uint64_t bar_qe[NQ];  // every S MMA of the unit retired
  __shared__ __align__(8) uint64_t bar_kf[KS];
  __shared__ __align__(8) uint64_t bar_ke[KS];
  __shared__ __align__(8) uint64_t bar_vf[VS];
  __shared__ __align__(8) uint64_t bar_ve[VS];
  __shared__ __align__(8) uint64_t bar_s[2];    // S_t in TMEM
  __shared__ __align__(8) uint64_t bar_sf[2];   // S_t read by the softmax (separate-P only)
  __shared__ __align__(8) uint64_t bar_p[2];    // P_t (d = 128: its first half) in TMEM, O_t rescaled
  __shared__ __align__(8) uint64_t bar_p2[2];   // d = 128: second half of P_t in TMEM
  __shared__ __align__(8) uint64_t bar_o[2];    // P_t.V retired
  __shared__ __align__(8) uint64_t bar_fin[2];  // every MMA of issuer t retired
  __shared__ __align__(8) uint64_t bar_turn[4]; // exponential phases, one per SM sub-partition
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  // ALiBi: the column offsets 0 .. BN-1 as floats, read as packed operands
  __shared__ __align__(16) float s_cols[kAlibi ? BN : 4];
  if (kAlibi && threadIdx.x < BN) s_cols[threadIdx.x] = static_cast<float>(threadIdx.x);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int PM = BM >> G_log2;  // positions per query tile

  if (threadIdx.x == 0) {
    abort_flag = 0;
    // empty barriers take one arrival from each MMA issuer (two at d = 64,
    // one issuing for both tiles at d = 128)
    constexpr uint32_t kIssuers = kSepP ? 2 : 1;
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bar_q[i], 1);
      mbar_init(&bar_qe[i], kIssuers);
    }
    for (int i = 0; i < KS; ++i) {
      mbar_init(&bar_kf[i], 1);
      mbar_init(&bar_ke[i], kIssuers);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&bar_vf[i], 1);
      mbar_init(&bar_ve[i], kIssuers);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_sf[t], 128);
      mbar_init(&bar_p[t], 128);
      mbar_init(&bar_p2[t], 128);
      mbar_init(&bar_o[t], 1);
    }
    mbar_init(&bar_fin[0], 1);
    mbar_init(&bar_fin[1], 1);
    for (int q = 0; q < 4; ++q) mbar_init(&bar_turn[q], 32);
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
  if (warp < 4) {
  setmaxnreg_dec<kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      // K/V tiles are re-read by the other units of their (batch, K/V head)
      // pair: keep them in L2; each query tile is read once: stream it
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t stream = l2_policy_evict_first();
      int nu = 0, kc = 0, vc = 0;  // units, K tiles and V tiles issued so far
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++nu) {
        const Unit w = decode_unit(u, p, PM, CAUSAL, kWindow, kCache);
        const int n_kv = max(w.n0, w.n1);
        const int qs = nu % NQ;
        if (nu >= NQ) ok = mbar_wait(&bar_qe[qs], ((nu / NQ) - 1) & 1, &abort_flag);
        if (!ok) break;
        const int n_qt = w.n1 > 0 ? 2 : 1;
        mbar_arrive_expect_tx(&bar_q[qs], n_qt * C::kQTile);
        for (int t = 0; t < n_qt; ++t) {
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb)
            tma_load_4d_hint(smem + qs * C::kQSlot + t * C::kQTile + cb * (BM * 128), &tm_q,
                             &bar_q[qs], cb * 64, w.kvh * G, w.p0 + t * PM, w.b, stream);
        }
        for (int j = 0; j < n_kv && ok; ++j) {
          const int ks = kc % KS;
          if (kc >= KS) ok = mbar_wait(&bar_ke[ks], ((kc / KS) - 1) & 1, &abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_kf[ks], C::kKVStage);
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb) {
            uint8_t* dst = smem + C::kOffK + ks * C::kKVStage + cb * (BN * 128);
            if (kCache)  // 3-D map over the cache
              tma_load_3d_hint(dst, &tm_k, &bar_kf[ks], cb * 64, (w.kv0 + j) * BN,
                               w.b * g + w.kvh, keep);
            else
              tma_load_4d_hint(dst, &tm_k, &bar_kf[ks], cb * 64, w.kvh, (w.kv0 + j) * BN, w.b,
                               keep);
          }
          ++kc;
          const int vs = vc % VS;
          if (vc >= VS) ok = mbar_wait(&bar_ve[vs], ((vc / VS) - 1) & 1, &abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_vf[vs], C::kKVStage);
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb) {
            uint8_t* dst = smem + C::kOffV + vs * C::kKVStage + cb * (BN * 128);
            if (kCache)  // 3-D map over the cache
              tma_load_3d_hint(dst, &tm_v, &bar_vf[vs], cb * 64, (w.kv0 + j) * BN,
                               w.b * g + w.kvh, keep);
            else
              tma_load_4d_hint(dst, &tm_v, &bar_vf[vs], cb * 64, w.kvh, (w.kv0 + j) * BN, w.b,
                               keep);
          }
          ++vc;
        }
        if (!ok) {
          ++nu;  // this unit's query load was issued
          break;
        }
      }
      if (!ok) {
        // every issued copy must have landed before the CTA may exit
        drain_ring(bar_q, NQ, nu);
        drain_ring(bar_kf, KS, kc);
        drain_ring(bar_vf, VS, vc);
      }
    }
  } else if (warp <= 2) {
    // ------------------------------------------------------------ MMA issuers
    // The whole issuing warp walks the schedule (it stays converged and keeps
    // the descriptors in uniform registers); one elected lane issues.
    const bool leader = elect_one();
    const uint32_t sbase = smem_u32(smem);
    // descriptor bases; a k-step only moves the 14-bit start-address field
    const uint64_t dq0 = smem_desc_sw128(sbase, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sbase + C::kOffK, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sbase + C::kOffV, BN * 128, 1024);
    // byte offset (>> 4) of k-step kk inside a K-major 128-byte-swizzled tile
    auto kmaj = [](int kk) -> uint64_t {
      return static_cast<uint64_t>(((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4);
    };
    // S_t = Q_t K^T for query tile t (query slot qs, K ring slot ks)
    auto issue_s = [&](int t, int qs, int ks) {
      const uint64_t aq = dq0 + static_cast<uint64_t>((qs * C::kQSlot + t * C::kQTile) >> 4);
      const uint64_t bk = dk0 + static_cast<uint64_t>((ks * C::kKVStage) >> 4);
      const uint32_t d_s = tmem + static_cast<uint32_t>(t) * BN;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_ss(d_s, aq + kmaj(kk), bk + kmaj(kk), kIdescS, kk > 0 ? 1u : 0u);
      mma_commit(&bar_s[t]);
    };
    // O_t += P_t V over the keys of k-steps [k0, k1) (16 keys each). V tile
    // [BN keys x D], D contiguous: MN-major B operand; LBO = distance between
    // the 64-wide column blocks of D; a k-step is 16 rows of 128 B
    auto issue_pv = [&](int t, int vs, bool first, int k0, int k1) {
      const uint64_t bv = dv0 + static_cast<uint64_t>((vs * C::kKVStage) >> 4);
      const uint32_t p_t = tmem + C::kColP + static_cast<uint32_t>(t) * C::kStrideP;
      const uint32_t o_t = tmem + C::kColO + static_cast<uint32_t>(t) * D;
#pragma unroll
      for (int kk = k0; kk < k1; ++kk)
        mma_bf16_ts(o_t, p_t + kk * 8, bv + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                    kIdescO, (!first || kk > 0) ? 1u : 0u);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag));
    };
    // release (commit) or give up (plain arrive) a slot of an empty barrier
    auto release = [&](uint64_t* bar, bool used) {
      if (leader) {
        if (used)
          mma_commit(bar);
        else
          mbar_arrive(bar);
      }
      __syncwarp();
    };

    if (kSepP) {
      // d = 64: warp 1 + t issues every MMA of query tile t, so the two
      // tiles' chains (S_t -> softmax -> P_t.V) never wait on each other's
      // hand-offs. A K/V ring slot (and the query slot) is released once BOTH
      // issuers are done with it: the empty barriers count two arrivals, a
      // commit from an issuer that used the slot or a plain arrive from one
      // that did not.
      const int t = warp - 1;
      int nu = 0, kb = 0;  // units and K/V tiles (of all units) consumed so far
      int it = 0;          // (unit, K/V tile) steps of this query tile so far
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++nu) {
        const Unit w = decode_unit(u, p, PM, CAUSAL, kWindow, kCache);
        const int n_kv = max(w.n0, w.n1);
        const int n_me = t == 0 ? w.n0 : w.n1;
        const int qs = nu % NQ;
        if (n_me > 0) {
          ok = wait_all(&bar_q[qs], (nu / NQ) & 1);
          if (ok) ok = wait_all(&bar_kf[kb % KS], (kb / KS) & 1);
          // S_t(0) once the softmax has read the previous S_t
          if (ok && it > 0) ok = wait_all(&bar_sf[t], (it - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          if (leader) issue_s(t, qs, kb % KS);
          __syncwarp();
          release(&bar_ke[kb % KS], true);  // K tile 0: its only reader is issued
        }
        // the query slot is free once this tile's last score product retires;
        // a tile without keys gives it back only once it has landed (a plain
        // arrive must never run ahead of the fill it releases)
        if (n_me == 0) {
          ok = wait_all(&bar_q[qs], (nu / NQ) & 1);
          if (!ok) break;
        }
        if (n_me <= 1) release(&bar_qe[qs], n_me == 1);
        for (int j = 0; ok && j < n_kv; ++j) {
          const int kj = kb + j;  // ring index of K/V tile j
          if (j >= n_me) {
            // this query tile sees no keys from tile j on: give the slots
            // back, each only after its fill has landed, so this issuer can
            // never arrive twice on a slot before the other issuer has used it
            ok = wait_all(&bar_kf[kj % KS], (kj / KS) & 1);
            if (!ok) break;
            release(&bar_ke[kj % KS], false);
            ok = wait_all(&bar_vf[kj % VS], (kj / VS) & 1);
            if (!ok) break;
            release(&bar_ve[kj % VS], false);
            continue;
          }
          if (j + 1 < n_me) {
            // S_t(j+1) as soon as the softmax has read S_t(j)
            ok = wait_all(&bar_kf[(kj + 1) % KS], ((kj + 1) / KS) & 1);
            if (ok) ok = wait_all(&bar_sf[t], (it + j) & 1);
            if (!ok) break;
            tc_fence_after();
            if (leader) issue_s(t, qs, (kj + 1) % KS);
            __syncwarp();
            release(&bar_ke[(kj + 1) % KS], true);
            if (j + 2 == n_me) release(&bar_qe[qs], true);
          }
          ok = wait_all(&bar_vf[kj % VS], (kj / VS) & 1);
          if (ok) ok = wait_all(&bar_p[t], (it + j) & 1);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            issue_pv(t, kj % VS, j == 0, 0, BN / 16);
            mma_commit(&bar_o[t]);
          }
          __syncwarp();
          release(&bar_ve[kj % VS], true);
        }
        if (!ok) break;
        kb += n_kv;
        it += n_me;
      }
      // every MMA must have retired before TMEM is released
      if (leader) {
        mma_commit(&bar_fin[t]);
        mbar_drain(&bar_fin[t], 0);
      }
      __syncwarp();
    } else if (warp == 1) {
      // d = 128: P_t(j) lives in S_t, so S_t(j+1) can only follow P_t(j).V_j.
      // One warp issues the MMAs of both query tiles, tile 0's work of a step
      // before tile 1's. The tensor core executes them in that order, so one
      // tile's next scores are ready a whole batch (P.V + S, ~1000 cycles)
      // before the other's and the two softmax warpgroups take turns with the
      // tensor core. (Two issuers let the tensor core interleave the two
      // batches; both tiles' scores then finished together and the softmax
      // warpgroups ran side by side while the tensor core idled.) Each ring
      // slot has one release, a commit issued right after its last reader.
      int nu = 0, kb = 0;       // units and K/V tiles (of all units) consumed so far
      int it0 = 0, it1 = 0;     // (unit, K/V tile) steps of query tile 0 / 1 so far
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++nu) {
        const Unit w = decode_unit(u, p, PM, CAUSAL, kWindow, kCache);
        const int n_kv = max(w.n0, w.n1);  // w.n0 >= 1: tile 0 always sees a key tile
        const int qs = nu % NQ;
        ok = wait_all(&bar_q[qs], (nu / NQ) & 1);
        if (ok) ok = wait_all(&bar_kf[kb % KS], (kb / KS) & 1);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
          issue_s(0, qs, kb % KS);
          if (w.n1 > 0) issue_s(1, qs, kb % KS);
        }
        __syncwarp();
        release(&bar_ke[kb % KS], true);
        if (n_kv == 1) release(&bar_qe[qs], true);
        for (int j = 0; ok && j < n_kv; ++j) {
          const int kj = kb + j;  // ring index of K/V tile j
          ok = wait_all(&bar_vf[kj % VS], (kj / VS) & 1);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int n_t = t == 0 ? w.n0 : w.n1;
            const int ph = ((t == 0 ? it0 : it1) + j) & 1;
            if (!ok || j >= n_t) continue;
            // keys 0..63 as soon as their half of P_t(j) is written
            ok = wait_all(&bar_p[t], ph);
            if (!ok) break;
            tc_fence_after();
            if (leader) issue_pv(t, kj % VS, j == 0, 0, BN / 32);
            __syncwarp();
            ok = wait_all(&bar_p2[t], ph);
            if (ok && j + 1 < n_t) ok = wait_all(&bar_kf[(kj + 1) % KS], ((kj + 1) / KS) & 1);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              issue_pv(t, kj % VS, j == 0, BN / 32, BN / 16);
              mma_commit(&bar_o[t]);
              if (j + 1 < n_t) issue_s(t, qs, (kj + 1) % KS);
            }
            __syncwarp();
          }
          if (!ok) break;
          release(&bar_ve[kj % VS], true);               // both tiles' P.V_j issued
          if (j + 1 < n_kv) release(&bar_ke[(kj + 1) % KS], true);  // both S(j+1) issued
          if (j + 2 == n_kv) release(&bar_qe[qs], true);  // the unit's last S issued
        }
        if (!ok) break;
        kb += n_kv;
        it0 += w.n0;
        it1 += w.n1;
      }
      // every MMA must have retired before TMEM is released
      if (leader) {
        mma_commit(&bar_fin[0]);
        mbar_drain(&bar_fin[0], 0);
      }
      __syncwarp();
    }
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;        // TMEM lane quadrant
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + static_cast<uint32_t>(t) * BN;
    const uint32_t t_o = tmem + lane_base + C::kColO + static_cast<uint32_t>(t) * D;
    const uint32_t t_p = tmem + lane_base + C::kColP + static_cast<uint32_t>(t) * C::kStrideP;
    const float scale_log2 = p.scale_log2;
    const uint64_t c2 = f32x2(scale_log2, scale_log2);
    const uint64_t o_policy = l2_policy_evict_first();  // O is written once: stream it
    int it = 0;      // (unit, K/V tile) steps of this query tile so far
    int npass = 0;   // output staging passes of this query tile so far
    int kturn = 0;   // exponential phases of both tiles in earlier units
    int kvbase = 0;  // K/V tiles of earlier units (ring index of this unit's first tile)
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(u, p, PM, CAUSAL, kWindow, kCache);
      const int n_my = t == 0 ? w.n0 : w.n1;
      const int n_kv = max(w.n0, w.n1);
      if (kCache && threadIdx.x == 128 && w.kvh == 0 && w.p0 == 0) {
        const int n = p.kv_lens[w.b];
        if (n < p.Lq || n > p.S_max) record_status(p.status, GQA_ERR_BAD_LENGTH);
      }
      if (n_my == 0) {
        kturn += w.n0 + w.n1;  // this tile sees no keys in this unit
        kvbase += n_kv;
        continue;
      }
      const int pt = w.p0 + t * PM;
      const int pos = pt + (row >> G_log2);
      const int head = w.kvh * G + (row & (G - 1));
      const int q_abs = w.q_off + pos;  // key position of this row's query
      // keys this row may see: [first_key, last_key]
      const int last_key = CAUSAL ? min(w.Lk - 1, q_abs) : w.Lk - 1;
      const int first_key = kWindow ? q_abs - p.window + 1 : 0;
      // last query row of the tile, for the tile-level mask decisions
      const int q_abs_last = w.q_off + min(p.Lq, pt + PM) - 1;
      // ALiBi: -slope * |q_abs - key| in log2 units of the scaled score
      const float slope_log2 = kAlibi ? p.alibi[head] * 1.4426950408889634f : 0.f;
      float m_run = -INFINITY;  // running max of the log2-unit scores, possibly stale by < 2^8
      float l_run = 0.f;
      for (int j = 0; j < n_my; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[t], (it + j) & 1, &abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t r[BN];
        if (D == 128) {
          tmem_ld128(t_s, r);  // one instruction: measured faster than four x32 loads here
        } else {
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) tmem_ld32(t_s + c * 32, r + c * 32);
        }
        tmem_ld_wait();
        if (kSepP) {
          // S_t may be overwritten by the next score product from here on
          tc_fence_before();
          mbar_arrive(&bar_sf[t]);
        }
        const int key0 = (w.kv0 + j) * BN;
        const bool need_mask = (key0 + BN > w.Lk) || (CAUSAL && key0 + BN - 1 > w.q_off + pt) ||
                               (kWindow && key0 <= q_abs_last - p.window);
        if (kAlibi) {
          // biased log2-unit scores; masked keys become -inf
          if (CAUSAL) {
            // every visible key is at or before the query: the bias of key
            // key0 + e is b0 + slope * e
            const float b0 = -slope_log2 * static_cast<float>(q_abs - key0);
            // two keys per packed op: t = slope * e + b0, x = s * scale + t
            // (the same roundings as one fmaf each)
            const uint64_t sc2 = f32x2(scale_log2, scale_log2);
            const uint64_t sl2 = f32x2(slope_log2, slope_log2);
            const uint64_t b02 = f32x2(b0, b0);
            const float4* cols = reinterpret_cast<const float4*>(s_cols);
#pragma unroll
            for (int e4 = 0; e4 < BN / 4; ++e4) {
              const float4 ev = cols[e4];
              const uint64_t x0 = ffma_x2(u32x2(r[4 * e4], r[4 * e4 + 1]), sc2,
                                          ffma_x2(sl2, f32x2(ev.x, ev.y), b02));
              const uint64_t x1 = ffma_x2(u32x2(r[4 * e4 + 2], r[4 * e4 + 3]), sc2,
                                          ffma_x2(sl2, f32x2(ev.z, ev.w), b02));
              float xa, xb, xc, xd;
              split_f32x2(x0, xa, xb);
              split_f32x2(x1, xc, xd);
              r[4 * e4] = __float_as_uint(xa);
              r[4 * e4 + 1] = __float_as_uint(xb);
              r[4 * e4 + 2] = __float_as_uint(xc);
              r[4 * e4 + 3] = __float_as_uint(xd);
            }
            if (need_mask) {
#pragma unroll
              for (int e = 0; e < BN; ++e) {
                const int key = key0 + e;
                if (key > last_key || key < first_key) r[e] = 0xff800000u;  // -inf
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < BN; ++e) {
              const int key = key0 + e;
              const float bias = -slope_log2 * static_cast<float>(abs(q_abs - key));
              const float x = fmaf(__uint_as_float(r[e]), scale_log2, bias);
              r[e] = __float_as_uint(key > last_key || key < first_key ? -INFINITY : x);
            }
          }
        } else if (need_mask) {
#pragma unroll
          for (int e = 0; e < BN; ++e) {
            const int key = key0 + e;
            if (key > last_key || (kWindow && key < first_key)) r[e] = 0xff800000u;  // -inf
          }
        }
        // row max (three-input max, four independent chains)
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < BN / 2; ++e)
          mx4[e & 3] = max3f(mx4[e & 3], __uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
        const float mx = max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        const float m_new = fmaxf(m_run, kAlibi ? mx : mx * scale_log2);
        const bool rescale = __any_sync(0xffffffffu, m_new > m_run + kRescaleThreshold);
        float alpha = 1.f;
        if (rescale) {
          // the whole warp adopts its new maxima (tcgen05.ld/st are warp-wide)
          alpha = m_run == -INFINITY ? 0.f : ex2_approx(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
        }
        if (j > 0) {
          // P_t(j-1).V_{j-1} has retired: O_t holds keys < j*128 and, with
          // separate P, the P_t columns are free again
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[t], (it + j - 1) & 1, &abort_flag));
          if (!ok) break;
          tc_fence_after();
          if (rescale) {
            // rare (lazy rescale); small chunks keep the score registers live
#pragma unroll 1
            for (int c = 0; c < D / 8; ++c) {
              uint32_t ov[8];
              tmem_ld8(t_o + c * 8, ov);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 8; ++e)
                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tmem_st8(t_o + c * 8, ov);
            }
          }
        }
        if (kCache && key0 + BN > w.Lk) {
          // cache rows past the sequence may hold anything (even NaN) and
          // 0 * NaN would poison P.V: zero them in this V stage (both query
          // tiles may write the same zeros) once the stage has landed, before
          // any part of P_t(j) is handed to the tensor core
          const int vslot = (kvbase + j) % VS;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_vf[vslot], ((kvbase + j) / VS) & 1,
                                                  &abort_flag));
          if (!ok) break;
          uint8_t* vst = smem + C::kOffV + vslot * C::kKVStage;
          const int r_lo = max(0, w.Lk - key0);
          for (int i = threadIdx.x - 128 - 128 * t; i < (BN - r_lo) * (D / 64) * 8; i += 128) {
            const int rr = r_lo + i / ((D / 64) * 8);
            const int cb = (i / 8) % (D / 64);
            *reinterpret_cast<uint4*>(vst + cb * (BN * 128) + rr * 128 + (i % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // visible to the tensor core's reads of V
        }
        // d = 64: the two softmax warps that share an SM sub-partition (warp
        // 4+q of tile 0, warp 8+q of tile 1) take turns on the exponential
        // unit, in the order (step j, tile 0), (step j, tile 1), (step j+1,
        // tile 0)...: one warp's exponentials overlap the other's loads, max
        // and waits instead of both halving each other's throughput. Phase k
        // waits for phase k-1 (of either warp; phase k+1 cannot have started).
        // At d = 128 the two tiles' steps are already staggered by their
        // score products and the turns only add waits.
        const int kt = kturn + min(j, w.n0) + min(j, w.n1) + (t == 1 && j < w.n0 ? 1 : 0);
        if (kSepP && kt > 0) {
          ok = mbar_wait(&bar_turn[wq], (kt - 1) & 1, &abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        // P = 2^(s * scale * log2(e) - m_run) as bf16 pairs, 64 keys at a time;
        // scale-and-shift and the running sum use packed two-lane fp32 ops
        // a row that has seen no key yet keeps m_run = -inf: shift by 0 instead
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        const uint64_t nm2 = f32x2(-m_use, -m_use);
        const uint64_t one2 = f32x2(1.f, 1.f);
        uint64_t sum2[2] = {0ull, 0ull};
        float bsum[4] = {0.f, 0.f, 0.f, 0.f};  // ALiBi: sums of the bf16 weights, four chains
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = hh * 64 + 2 * e;
            float xa, xb;
            split_f32x2(ffma_x2(u32x2(r[c], r[c + 1]), kAlibi ? one2 : c2, nm2), xa, xb);
            const float pa = ex2_approx(xa);
            const float pb = ex2_approx(xb);
            pw[e] = pack_bf16x2(pa, pb);
            if (kAlibi) {
              // ALiBi makes rows peaked (one weight near 1): sum the bf16
              // weights the P.V product really uses, so numerator and
              // denominator round alike
              add_bf16x2_to_f32(pw[e], bsum[(e & 1) * 2], bsum[(e & 1) * 2 + 1]);
            } else {
              sum2[e & 1] = fadd_x2(sum2[e & 1], f32x2(pa, pb));
            }
          }
          tmem_st32(t_p + hh * 32, pw);  // P columns [32hh, 32hh+32) = keys [64hh, 64hh+64)
          if (!kSepP && hh == 0) {
            // d = 128: keys 0..63 of P_t(j) (and the rescaled O_t) go to the
            // tensor core while the second half is computed
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_p[t]);
          }
        }
        if (kSepP) mbar_arrive(&bar_turn[wq]);  // this warp's exponential phase is over
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(kSepP ? &bar_p[t] : &bar_p2[t]);
        if (kAlibi) {
          sum2[0] = f32x2(bsum[0], bsum[1]);
          sum2[1] = f32x2(bsum[2], bsum[3]);
        }
        float a0, a1, b0, b1;
        split_f32x2(sum2[0], a0, a1);
        split_f32x2(sum2[1], b0, b1);
        l_run += (a0 + a1) + (b0 + b1);
      }
      if (!ok) break;
      // epilogue: O_t is final once the last P_t.V retires
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[t], (it + n_my - 1) & 1, &abort_flag));
      if (!ok) break;
      tc_fence_after();
      it += n_my;
      kturn += w.n0 + w.n1;
      kvbase += n_kv;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;  // a row with no key writes zeros
      // O_t / l: staged in shared memory (128-byte swizzle, so the row-per-
      // thread writes spread over all banks) and stored by TMA in 128-byte
      // column chunks; rows past L are dropped by the store itself
      const bool f32 = p.o_dtype == GQA_OUT_F32;
      const int n_chunks = f32 ? D / 32 : D / 64;
      uint8_t* stage = smem + C::kOffStage + t * C::kStageBytes;
      const uint32_t sw = static_cast<uint32_t>(row & 7);
      // this warp's 32 rows start at position pt + (32 wq) / G, head
      // kvh * G + (32 wq) % G; its TMA store box is 32 rows of the tile
      const int r0 = wq * 32;
      const int st_pos = pt + (r0 >> G_log2);
      const int st_head = w.kvh * G + (r0 & (G - 1));
      for (int c0 = 0; c0 < n_chunks; c0 += C::kStageChunks, ++npass) {
        // this pass's accumulator columns, read from TMEM before waiting for
        // the stage (fp32: kStageChunks chunks of 32 columns; bf16: one chunk
        // of 64 columns)
        uint32_t v[64];
        tmem_ld32(t_o + (f32 ? c0 * 32 : c0 * 64), v);
        if (!f32 || C::kStageChunks == 2)
          tmem_ld32(t_o + (f32 ? c0 * 32 + 32 : c0 * 64 + 32), v + 32);
        tmem_ld_wait();
        if (npass > 0) {
          // the warp's previous stores have read its rows of the stage
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
        if (f32) {
#pragma unroll
          for (int cc = 0; cc < C::kStageChunks; ++cc) {
            uint8_t* dst = stage + cc * C::kChunkBytes + row * 128;
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4)
              *reinterpret_cast<float4*>(dst + ((u4 ^ sw) << 4)) =
                  make_float4(__uint_as_float(v[32 * cc + 4 * u4]) * inv_l,
                              __uint_as_float(v[32 * cc + 4 * u4 + 1]) * inv_l,
                              __uint_as_float(v[32 * cc + 4 * u4 + 2]) * inv_l,
                              __uint_as_float(v[32 * cc + 4 * u4 + 3]) * inv_l);
          }
        } else {
          uint8_t* dst = stage + row * 128;
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            uint32_t wv[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2)
              wv[q2] = pack_bf16x2(__uint_as_float(v[8 * u4 + 2 * q2]) * inv_l,
                                   __uint_as_float(v[8 * u4 + 2 * q2 + 1]) * inv_l);
            *reinterpret_cast<uint4*>(dst + ((u4 ^ sw) << 4)) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
        fence_proxy_async_smem();  // the generic-proxy writes become visible to TMA
        __syncwarp();
        if (lane == 0) {
          // a warp whose rows all lie past the sequence stores nothing
          if (st_pos < p.Lq) {
            for (int cc = 0; cc < (f32 ? C::kStageChunks : 1); ++cc)
              tma_store_4d_hint(&tm_o, stage + cc * C::kChunkBytes + r0 * 128,
                                (c0 + cc) * (f32 ? 32 : 64), st_head, st_pos, w.b, o_policy);
          }
          bulk_commit_group();
        }
      }
      if (!ok) break;
      const bool store = pos < p.Lq;
      if (p.lse != nullptr && store)
        p.lse[(static_cast<size_t>(w.b) * h_q + head) * p.Lq + pos] =
            l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
  if (threadIdx.x == 0 && abort_flag) record_status(p.status, GQA_ERR_TIMEOUT);
}

template <int D, bool CAUSAL, int VAR>
static cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t s) {
  constexpr uint32_t kSmem = PrefillCfg<D>::kSmem;
  static DeviceOnce attr_once;
  cudaError_t e = run_once_per_device(attr_once, [] {
    // the register hand-over inside the kernel assumes the launch pool
    cudaFuncAttributes fa{};
    cudaError_t r = cudaFuncGetAttributes(&fa, prefill_kernel<D, CAUSAL, VAR>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidKernelImage;
    return cudaFuncSetAttribute(prefill_kernel<D, CAUSAL, VAR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  const int PM = BM / a.G;
  const int n_ctiles = (a.Lq + 2 * PM - 1) / (2 * PM);
  const long long n_units = static_cast<long long>(n_ctiles) * a.g * a.B;
  const int n_sm = device_sm_count();
  const int grid = static_cast<int>(n_units < n_sm ? n_units : n_sm);
  PrefillParams p{};
  p.lse = a.lse;
  p.o_dtype = a.o_dtype;
  p.B = a.B;
  p.Lq = a.Lq;
  p.Lk = a.Lk;
  p.S_max = a.S_max;
  p.h_q = a.h_q;
  p.g = a.g;
  p.G = a.G;
  p.G_log2 = a.G_log2;
  p.scale_log2 = a.scale_log2;
  p.n_ctiles = n_ctiles;
  p.n_units = static_cast<int>(n_units);
  p.kv_lens = a.kv_lens;
  p.window = a.window;
  p.alibi = a.alibi;
  p.status = a.status;
  prefill_kernel<D, CAUSAL, VAR><<<grid, kThreads, kSmem, s>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o,
                                                              p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t s) {
  const int var =
      (a.window > 0 ? 1 : 0) | (a.alibi != nullptr ? 2 : 0) | (a.kv_lens != nullptr ? 4 : 0);
  if (!a.causal)  // a window or a cache needs causal attention (checked by the caller)
    return var & 2 ? launch_prefill_t<D, false, 2>(a, s) : launch_prefill_t<D, false, 0>(a, s);
  switch (var) {
    case 1: return launch_prefill_t<D, true, 1>(a, s);
    case 2: return launch_prefill_t<D, true, 2>(a, s);
    case 3: return launch_prefill_t<D, true, 3>(a, s);
    case 4: return launch_prefill_t<D, true, 4>(a, s);
    case 5: return launch_prefill_t<D, true, 5>(a, s);
    case 6: return launch_prefill_t<D, true, 6>(a, s);
    case 7: return launch_prefill_t<D, true, 7>(a, s);
    default: return launch_prefill_t<D, true, 0>(a, s);
  }
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_prefill_d<64>(a, s) : launch_prefill_d<128>(a, s);
}

}  // namespace gqa
