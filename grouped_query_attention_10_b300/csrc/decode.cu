// decode.cu -- one-token GQA decode over a [B, g, S_max, d] bf16 KV cache.
//
// The decode step of the "What is Grouped-Query Attention" explainer
// (ijyty.com), section 2.1: the new token's query attends over every cached
// K/V row. Design (split-KV, the split attention forward sketched in the
// "Qwen, DeepSeek and LLaMA3 attention survey" (jsqmd.com), chapter 5):
//
//  * pass 1 (decode_split_kernel): the work items are (split, slice of the
//    group's query heads, K/V head, sequence); persistent CTAs (two per SM)
//    walk them. A producer warp streams each item's K and V rows through a
//    TMA-fed shared-memory ring (128-byte swizzle, so ldmatrix reads are
//    bank-conflict free); the ring carries on from one item to the next.
//    Four consumer warps serve ALL query heads of the group from the same
//    bytes: the heads are stacked as the M side of m16n8k16 tensor-core
//    MMAs, so each K/V byte is read from HBM once per K/V head, never once
//    per query head. Every item ends with its normalised partial output and
//    its log2 sum-exp.
//  * pass 2 (decode_combine_kernel): log-sum-exp combine of the partials,
//    launched as a programmatic dependent of pass 1. When every sequence's
//    rows (or window) fit one split, pass 1 merges the partials of each item
//    itself, right after its consumer warps have written them, and writes the
//    output; pass 2 is not launched.
#include <cuda_bf16.h>

#include "../../include/gqa.h"
#include "launch.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kConsumers = 4;                    // consumer warps
constexpr int kThreads = 32 * (kConsumers + 1);  // + one producer warp
constexpr int kCtasPerSm = 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct DecCfg {
  static constexpr int kStages = D == 128 ? 3 : 6;         // ring depth (96 KB)
  static constexpr int kCB = D / 64;                        // 64-wide column blocks
  static constexpr int kBoxBytes = kDecodeStage * 128;      // 64 rows x 128 B
  static constexpr int kStageBytes = 2 * kCB * kBoxBytes;   // K + V
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kSmem = kRing + 1024;                // + alignment slack
};

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

// lo += the bf16 in bits 0..15 of w, hi += the bf16 in bits 16..31: each
// widened exactly to fp32 and added with one rounding (mixed-precision add of
// sm_100 and later)
__device__ __forceinline__ void add_bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.bf16 %0, l, %0; "
      "add.rn.f32.bf16 %1, h, %1; }"
      : "+f"(lo), "+f"(hi)
      : "r"(w));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside one
// [rows x 128 B] box written by TMA with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// One decoded work item.
struct Item {
  int b, kvh, hs, split;
  int len;           // valid rows of the sequence (the query sits at len - 1)
  int lo;            // first row inside the sliding window (0 without one)
  int s0, s1, n_st;  // token range [s0, s1) and its 64-token stages (0: nothing to do)
};

// Items are numbered split-major (every segment's first split, then every
// segment's second split, ...): items are fetched in that order, so the
// partial and empty splits at the end of short sequences come last and fill
// the tail of the pass.
__device__ __forceinline__ Item decode_item(int u, const int32_t* seq_lens, int g, int n_hslice,
                                            int S_max, int split_len, int n_segs, int window) {
  Item it;
  it.split = u / n_segs;
  const int seg = u % n_segs;
  it.hs = seg % n_hslice;
  const int pair = seg / n_hslice;
  it.kvh = pair % g;
  it.b = pair / g;
  int len = seq_lens[it.b];
  len = len < 0 ? 0 : (len > S_max ? S_max : len);
  it.len = len;
  // With a sliding window only its rows are read: the splits tile the
  // window from the 64-row stage that holds its first row (a window of W
  // rows is spread over all n_split splits, whatever the cache size), and
  // the rows of that stage before the window are masked. Every stage start
  // stays a multiple of 64, so a paged stage never begins inside a page.
  it.lo = window > 0 ? max(0, len - window) : 0;
  it.s0 = (it.lo & ~(kDecodeStage - 1)) + it.split * split_len;
  it.s1 = min(len, it.s0 + split_len);
  it.n_st = it.s0 < it.s1 ? (it.s1 - it.s0 + kDecodeStage - 1) / kDecodeStage : 0;
  return it;
}

}  // namespace

// D: head dim (64 or 128). MT: m16 tiles of stacked query rows (G <= 16*MT).
template <int D, int MT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_split_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ seq_lens,
    float* __restrict__ part_o, float* __restrict__ part_lse, int h_q, int g, int G,
    int n_hslice, int S_max, int split_len, int n_split, int n_items, float scale_log2,
    int window, const float* __restrict__ alibi, const int32_t* __restrict__ block_table,
    int page_log2, int num_pages, int max_blocks, int* __restrict__ item_counter,
    void* __restrict__ o_out, int o_dtype, float* __restrict__ lse_out, int fused,
    int32_t* status) {
  using C = DecCfg<D>;
  constexpr int kStages = C::kStages;
  constexpr int kCB = C::kCB;
  constexpr int kNSlices = kConsumers / MT;                // warps sharing one m-tile
  constexpr int kSubPerWarp = (kDecodeStage / 16) / kNSlices;
  constexpr int kPf = MT == 2 ? 1 : 2;  // shared-memory fragment loads issued this many steps early

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];   // one arrival per consumer warp
  __shared__ int4 tag[kStages];              // item, stage, stages of the item (item < 0: end)
  __shared__ int abort_flag;
  __shared__ __align__(8) uint64_t merge_bar;  // the consumer warps' partials of an item written

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumers);
    }
    mbar_init(&merge_bar, kConsumers);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const int n_segs = n_items / n_split;
      int sc = 0;  // stages issued so far
      bool ok = true;
      // items are fetched from a counter the host zeroes before the launch,
      // so CTAs that drew short items simply fetch more
      for (int u = atomicAdd(item_counter, 1); u < n_items && ok;
           u = atomicAdd(item_counter, 1)) {
        const Item it = decode_item(u, seq_lens, g, n_hslice, S_max, split_len, n_segs, window);
        const int zrow = it.b * g + it.kvh;
        if (fused && it.split == 0) {
          // no combine runs to flag a bad length: flag it here
          const int raw = seq_lens[it.b];
          if ((raw < 0 || raw > S_max) && it.kvh == 0 && it.hs == 0)
            record_status(status, GQA_ERR_BAD_LENGTH);
        }
        if (fused && it.n_st == 0 && it.split == 0) {
          // a sequence with no rows: its output rows are zero, lse -inf
          const size_t h0 = static_cast<size_t>(it.b) * h_q + static_cast<size_t>(it.kvh) * G +
                            it.hs * 32;
          const int gs = min(G - it.hs * 32, 16 * MT);
          for (int r = 0; r < gs; ++r) {
            for (int c = 0; c < D; ++c) {
              if (o_dtype == GQA_OUT_F32)
                static_cast<float*>(o_out)[(h0 + r) * D + c] = 0.f;
              else
                static_cast<__nv_bfloat16*>(o_out)[(h0 + r) * D + c] =
                    __float2bfloat16_rn(0.f);
            }
            if (lse_out != nullptr) lse_out[h0 + r] = -INFINITY;
          }
        }
        for (int st = 0; st < it.n_st; ++st, ++sc) {
          const int slot = sc % kStages;
          if (sc >= kStages) ok = mbar_wait(&empty_bar[slot], ((sc / kStages) - 1) & 1, &abort_flag);
          if (!ok) break;
          tag[slot] = make_int4(u, st, it.n_st, 0);
          uint8_t* base = smem + slot * C::kStageBytes;
          const int y = it.s0 + st * kDecodeStage;
          mbar_arrive_expect_tx(&full_bar[slot], C::kStageBytes);
          if (block_table == nullptr) {
#pragma unroll
            for (int cb = 0; cb < kCB; ++cb) {
              tma_load_3d(base + cb * C::kBoxBytes, &tm_k, &full_bar[slot], cb * 64, y, zrow);
              tma_load_3d(base + (kCB + cb) * C::kBoxBytes, &tm_v, &full_bar[slot], cb * 64, y,
                          zrow);
            }
          } else {
            // paged cache: the stage's 64 rows come from one page or from
            // 64 / page_size consecutive logical blocks; a box lands at its
            // row offset of the stage (a multiple of 16 rows, so the 128-byte
            // swizzle of the whole stage is kept)
            const int rows = min(kDecodeStage, 1 << page_log2);
            for (int sub = 0; sub < kDecodeStage; sub += rows) {
              const int tok = y + sub;
              const int lb = tok >> page_log2;
              int page = lb < max_blocks ? block_table[static_cast<size_t>(it.b) * max_blocks + lb]
                                         : -1;
              if (page < 0 || page >= num_pages) {
                // an entry the sequence uses inside its window must name a
                // page of the pool (pages wholly before the window may be
                // gone); a missing page reads zeros (the load starts out of
                // range)
                if (tok < it.s1 && tok + rows > it.lo) record_status(status, GQA_ERR_BAD_PAGE);
                page = -1;
              }
              const int zr = page < 0 ? -1 : page * g + it.kvh;
              const int yr = tok & ((1 << page_log2) - 1);
#pragma unroll
              for (int cb = 0; cb < kCB; ++cb) {
                tma_load_3d(base + cb * C::kBoxBytes + sub * 128, &tm_k, &full_bar[slot],
                            cb * 64, yr, zr);
                tma_load_3d(base + (kCB + cb) * C::kBoxBytes + sub * 128, &tm_v,
                            &full_bar[slot], cb * 64, yr, zr);
              }
            }
          }
        }
      }
      if (ok) {
        // end marker: a slot with no data and a negative item
        const int slot = sc % kStages;
        if (sc >= kStages) ok = mbar_wait(&empty_bar[slot], ((sc / kStages) - 1) & 1, &abort_flag);
        if (ok) {
          tag[slot] = make_int4(-1, 0, 0, 0);
          mbar_arrive(&full_bar[slot]);
        }
      }
      if (!ok) {
        // every issued copy must land before the CTA may exit
        for (int s = 0; s < kStages && s < sc; ++s) {
          const int last = s + ((sc - 1 - s) / kStages) * kStages;
          mbar_drain(&full_bar[s], (last / kStages) & 1);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int mt = warp % MT;
    const int slice = warp / MT;
    const int gr = lane >> 2;  // fragment row group
    const int tq = lane & 3;   // fragment column pair
    const int row0 = mt * 16 + gr;
    const int row1 = row0 + 8;
    const uint32_t smem_base = smem_u32(smem);
    const int n_segs = n_items / n_split;
    int sc = 0;  // stages consumed so far
    bool ok = true;
    Item it{};
    size_t head0 = 0;
    int Gs = 0;
    int n_merged = 0;  // items merged by this CTA (merge_bar phases)
    uint32_t qa[D / 16][4];
    float o_acc[D / 8][4];
    float m_r[2] = {-INFINITY, -INFINITY};  // running max (log2 units), stale by < 2^8
    float l_r[2] = {0.f, 0.f};
    float slope[2] = {0.f, 0.f};
    while (ok) {
      const int slot = sc % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&full_bar[slot], (sc / kStages) & 1, &abort_flag));
      if (!ok) break;
      const int4 tg = tag[slot];
      if (tg.x < 0) break;  // no more items
      const int st = tg.y;
      if (st == 0) {
        // a new item: its query rows and fresh accumulators
        it = decode_item(tg.x, seq_lens, g, n_hslice, S_max, split_len, n_segs, window);
        head0 = static_cast<size_t>(it.b) * h_q + static_cast<size_t>(it.kvh) * G + it.hs * 32;
        Gs = min(G - it.hs * 32, 16 * MT);  // stacked rows served by this item
        const __nv_bfloat16* qg = q + head0 * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk * 16 + tq * 2;
          qa[kk][0] = row0 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row0 * D + c) : 0u;
          qa[kk][1] = row1 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row1 * D + c) : 0u;
          qa[kk][2] = row0 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row0 * D + c + 8) : 0u;
          qa[kk][3] = row1 < Gs ? *reinterpret_cast<const uint32_t*>(qg + row1 * D + c + 8) : 0u;
        }
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
        m_r[0] = m_r[1] = -INFINITY;
        l_r[0] = l_r[1] = 0.f;
        if (alibi != nullptr) {
          // ALiBi slopes of this lane's two rows, in log2 units of the scaled score
          slope[0] = row0 < Gs ? alibi[head0 - static_cast<size_t>(it.b) * h_q + row0] *
                                     1.4426950408889634f
                               : 0.f;
          slope[1] = row1 < Gs ? alibi[head0 - static_cast<size_t>(it.b) * h_q + row1] *
                                     1.4426950408889634f
                               : 0.f;
        }
      }
      const int tok0 = it.s0 + st * kDecodeStage;
      const int valid = it.s1 - tok0;  // rows of this stage that are real
      const int first = it.lo - tok0;  // rows of this stage before the window
      const uint32_t kbase = smem_base + slot * C::kStageBytes;
      const uint32_t vbase = kbase + kCB * C::kBoxBytes;
      // This warp's 16-token blocks of the stage are processed together (their
      // score products form independent MMA chains), with one max reduction
      // and one rescale decision for all of them (the row sums are kept per
      // thread and reduced once per item).
      int r0[kSubPerWarp];
      bool act[kSubPerWarp];
#pragma unroll
      for (int sb = 0; sb < kSubPerWarp; ++sb) {
        r0[sb] = (slice + sb * kNSlices) * 16;  // first row of the 16-token block
        act[sb] = r0[sb] < valid;               // any real token in it
        if (act[sb] && (r0[sb] + 16 > valid || r0[sb] < first)) {
          // rows past the sequence or before the window may hold anything
          // (even NaN) and 0 * NaN would poison P.V: zero this block's V rows
          // there. Only the warps that read these rows write them, and all
          // write zeros.
          uint8_t* vrows = smem + slot * C::kStageBytes + kCB * C::kBoxBytes;
          for (int i = lane; i < 16 * kCB * 8; i += 32) {
            const int r = r0[sb] + i / (kCB * 8);
            const int cb = (i / 8) % kCB;
            const int ch = i % 8;
            if (r >= valid || r < first)
              *reinterpret_cast<uint4*>(vrows + cb * C::kBoxBytes + r * 128 + ch * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
      }
      if (act[0]) {
        float s[kSubPerWarp][2][4];
#pragma unroll
        for (int sb = 0; sb < kSubPerWarp; ++sb)
#pragma unroll
          for (int j = 0; j < 2; ++j) s[sb][j][0] = s[sb][j][1] = s[sb][j][2] = s[sb][j][3] = 0.f;
        // S = Q K^T over d. The inline-asm loads and MMAs keep their source
        // order, so each step's K fragments are loaded kPf steps ahead of the
        // MMAs that use them.
        {
          const int mi = lane >> 3;
          const int ri = lane & 7;
          uint32_t fb[kPf + 1][kSubPerWarp][4];
          auto kfetch = [&](int kk, int buf) {
            const int chunk = (kk * 2 + (mi & 1)) & 7;
#pragma unroll
            for (int sb = 0; sb < kSubPerWarp; ++sb) {
              if (!act[sb]) continue;
              const int tok = r0[sb] + (mi >> 1) * 8 + ri;
              ldsm_x4(kbase + (kk >> 2) * C::kBoxBytes + sw128(tok, chunk), fb[buf][sb][0],
                      fb[buf][sb][1], fb[buf][sb][2], fb[buf][sb][3]);
            }
          };
#pragma unroll
          for (int kk = 0; kk < kPf; ++kk) kfetch(kk, kk);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk + kPf < D / 16) kfetch(kk + kPf, (kk + kPf) % (kPf + 1));
            const int bf = kk % (kPf + 1);
#pragma unroll
            for (int sb = 0; sb < kSubPerWarp; ++sb) {
              if (!act[sb]) continue;
              mma16816(s[sb][0], qa[kk], fb[bf][sb][0], fb[bf][sb][1]);
              mma16816(s[sb][1], qa[kk], fb[bf][sb][2], fb[bf][sb][3]);
            }
          }
        }
        // mask, scale to log2 units, online softmax for rows row0 / row1.
        // A plain stage (every token of the warp's blocks real, none before the
        // window, no ALiBi) needs no per-score bias or bound: the max is taken
        // over the raw scores and the scale goes into the exponent's FMA.
        float mx[2] = {-INFINITY, -INFINITY};
        bool plain = alibi == nullptr && scale_log2 > 0.f;
#pragma unroll
        for (int sb = 0; sb < kSubPerWarp; ++sb)
          plain = plain && act[sb] && r0[sb] + 16 <= valid && r0[sb] >= first;
        if (plain) {
#pragma unroll
          for (int sb = 0; sb < kSubPerWarp; ++sb)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) mx[e >> 1] = fmaxf(mx[e >> 1], s[sb][j][e]);
          mx[0] *= scale_log2;
          mx[1] *= scale_log2;
        } else {
#pragma unroll
          for (int sb = 0; sb < kSubPerWarp; ++sb)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int tok = r0[sb] + j * 8 + tq * 2 + (e & 1);
                // ALiBi: -slope * (query position - key position)
                const float bias =
                    slope[e >> 1] * static_cast<float>(tok0 + tok - (it.len - 1));
                const float x = act[sb] && tok < valid && tok >= first
                                    ? fmaf(s[sb][j][e], scale_log2, bias)
                                    : -INFINITY;
                s[sb][j][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
              }
        }
        float m_new[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          m_new[h] = fmaxf(m_r[h], mx[h]);
        }
        // lazy rescale: only when some row's max grew by more than 2^8
        if (__any_sync(0xffffffffu, m_new[0] > m_r[0] + kRescaleThreshold ||
                                        m_new[1] > m_r[1] + kRescaleThreshold)) {
          float alpha[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            alpha[h] = m_r[h] == -INFINITY ? 0.f : ex2_approx(m_r[h] - m_new[h]);
            l_r[h] *= alpha[h];
            m_r[h] = m_new[h];
          }
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            o_acc[i][0] *= alpha[0];
            o_acc[i][1] *= alpha[0];
            o_acc[i][2] *= alpha[1];
            o_acc[i][3] *= alpha[1];
          }
        }
        // all-masked so far: keep everything at zero weight
        const float m_use[2] = {m_r[0] == -INFINITY ? 0.f : m_r[0],
                                m_r[1] == -INFINITY ? 0.f : m_r[1]};
        // P in bf16 (the A operand of P.V), rounded once per pair of one row;
        // this thread's share of each row sum adds the same rounded weights,
        // so numerator and denominator round alike (the four shares of a row
        // are added when the item ends)
        const float mul = plain ? scale_log2 : 1.f;
        uint32_t pw[kSubPerWarp][2][2];  // [block][j][row]: two weights of one row
        float rsa[2] = {0.f, 0.f};
        float rsb[2] = {0.f, 0.f};
#pragma unroll
        for (int sb = 0; sb < kSubPerWarp; ++sb)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float e0 = ex2_approx(fmaf(s[sb][j][2 * h], mul, -m_use[h]));
              const float e1 = ex2_approx(fmaf(s[sb][j][2 * h + 1], mul, -m_use[h]));
              pw[sb][j][h] = pack_bf16x2(e0, e1);
              add_bf16x2_to_f32(pw[sb][j][h], rsa[h], rsb[h]);
            }
        l_r[0] += rsa[0] + rsb[0];
        l_r[1] += rsa[1] + rsb[1];
        // O += P V with P (bf16) as the A fragments; V fragments loaded kPf
        // steps (of one 16-column pair) ahead of their MMAs
        {
          const int mi = lane >> 3;
          const int ri = lane & 7;
          constexpr int kSteps = kSubPerWarp * (D / 16);
          uint32_t vf[kPf + 1][4];
          auto vfetch = [&](int i, int buf) {
            const int sb = i / (D / 16);
            const int np = i % (D / 16);
            if (!act[sb]) return;
            const int tok = r0[sb] + (mi & 1) * 8 + ri;
            const int cg = np * 2 + (mi >> 1);
            ldsm_x4_t(vbase + (cg >> 3) * C::kBoxBytes + sw128(tok, cg & 7), vf[buf][0],
                      vf[buf][1], vf[buf][2], vf[buf][3]);
          };
#pragma unroll
          for (int i = 0; i < kPf; ++i) vfetch(i, i);
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            if (i + kPf < kSteps) vfetch(i + kPf, (i + kPf) % (kPf + 1));
            const int sb = i / (D / 16);
            const int np = i % (D / 16);
            if (!act[sb]) continue;
            const uint32_t pa[4] = {pw[sb][0][0], pw[sb][0][1], pw[sb][1][0], pw[sb][1][1]};
            const int bf = i % (kPf + 1);
            mma16816(o_acc[np * 2], pa, vf[bf][0], vf[bf][1]);
            mma16816(o_acc[np * 2 + 1], pa, vf[bf][2], vf[bf][3]);
          }
        }
      }
      // this warp is done with the slot (ldmatrix reads have completed)
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
      ++sc;
      if (st + 1 < tg.z) continue;  // the item goes on in the next stage

      // ---- this warp's partial for its rows and slice of the item's tokens:
      // O / l and log2 sum-exp; a slice that saw no real token writes O = 0,
      // lse = -inf (weight 0 in the combine)
      {
        const int pslot = it.split * kNSlices + slice;  // partial index within the row
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
          l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = h == 0 ? row0 : row1;
          if (row >= Gs) continue;
          const bool any = l_r[h] > 0.f;
          const float inv = any ? 1.f / l_r[h] : 0.f;
          const size_t ps = (head0 + row) * (static_cast<size_t>(n_split) * kNSlices) + pslot;
          float* dst = part_o + ps * D + tq * 2;
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<float2*>(dst + i * 8) =
                make_float2(o_acc[i][2 * h] * inv, o_acc[i][2 * h + 1] * inv);
          if (tq == 0) part_lse[ps] = any ? m_r[h] + __log2f(l_r[h]) : -INFINITY;
        }
      }
      if (fused) {
        // one split per segment: every consumer warp has written its slice's
        // partial of this item; merge them and write the output rows here
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(&merge_bar);
        ok = __all_sync(0xffffffffu, mbar_wait(&merge_bar, n_merged & 1, &abort_flag));
        ++n_merged;
        if (!ok) break;
        constexpr int kCols = D / 4;               // columns per warp
        constexpr int kRowStep = 32 / kCols;       // rows per pass of the warp
        const int c = warp * kCols + lane % kCols;
        const size_t n_part = static_cast<size_t>(n_split) * kNSlices;
        for (int r = lane / kCols; r < Gs; r += kRowStep) {
          const size_t pr = (head0 + r) * n_part + it.split * kNSlices;
          float ls[kNSlices];
          float mx = -INFINITY;
#pragma unroll
          for (int s2 = 0; s2 < kNSlices; ++s2) {
            ls[s2] = part_lse[pr + s2];
            mx = fmaxf(mx, ls[s2]);
          }
          const float mm = mx == -INFINITY ? 0.f : mx;
          float den = 0.f, acc = 0.f;
#pragma unroll
          for (int s2 = 0; s2 < kNSlices; ++s2) {
            const float w = ex2_approx(ls[s2] - mm);
            den += w;
            acc += w * part_o[(pr + s2) * D + c];
          }
          const float out = den > 0.f ? acc / den : 0.f;
          if (o_dtype == GQA_OUT_F32)
            static_cast<float*>(o_out)[(head0 + r) * D + c] = out;
          else
            static_cast<__nv_bfloat16*>(o_out)[(head0 + r) * D + c] = __float2bfloat16_rn(out);
          if (lse_out != nullptr && c == 0)
            lse_out[head0 + r] =
                den > 0.f ? (mm + __log2f(den)) * 0.69314718055994531f : -INFINITY;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && abort_flag) record_status(status, GQA_ERR_TIMEOUT);
  // the combine (launched as a programmatic dependent) may start launching;
  // it waits for this whole grid before it reads a partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA per (sequence, query head): merge the partials that hold data.
// The log2 sum-exps are staged in shared memory (up to kCombineSmem of
// them; longer rows loop over global memory), the weights 2^(lse - max) are
// computed once, and eight thread groups each sum every eighth partial of
// float4 columns, so many partial loads are in flight at once.
constexpr int kCombineThreads = 256;
constexpr int kCombineSmem = 2048;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int32_t* __restrict__ seq_lens, void* __restrict__ o, int o_dtype,
    float* __restrict__ lse_out, int h_q, int S_max, int split_len, int n_split, int n_slices,
    int window, int32_t* status) {
  constexpr int kLanesPerRow = D / 4;                       // threads covering one row
  constexpr int kGroups = kCombineThreads / kLanesPerRow;   // partial groups
  constexpr int kWarps = kCombineThreads / 32;
  __shared__ float red[kWarps];
  __shared__ float wsh[kCombineSmem];
  __shared__ float acc_sh[kGroups][D];
  // launched as a programmatic dependent of the split pass: wait until that
  // grid has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bh = blockIdx.x;
  const int b = bh / h_q;
  const int tid = threadIdx.x;
  int len = seq_lens[b];
  if (len < 0 || len > S_max) {
    if (tid == 0 && (bh % h_q) == 0) record_status(status, GQA_ERR_BAD_LENGTH);
    len = len < 0 ? 0 : S_max;
  }
  // partials of this row: n_slices per split (one per token slice; a slice
  // that saw no token holds lse = -inf and weighs nothing)
  // the splits that saw rows (with a window they start at the window's first
  // 64-row stage); later splits were never written
  const int base = (window > 0 ? max(0, len - window) : 0) & ~(kDecodeStage - 1);
  const int n = (len - base + split_len - 1) / split_len * n_slices;
  const int n_part = n_split * n_slices;
  const float* pl = part_lse + static_cast<size_t>(bh) * n_part;
  const bool staged = n <= kCombineSmem;
  auto lse_at = [&](int s) { return staged ? wsh[s] : pl[s]; };
  // block max of the partial log-sum-exps
  float m = -INFINITY;
  for (int s = tid; s < n; s += kCombineThreads) {
    const float x = pl[s];
    if (staged) wsh[s] = x;
    m = fmaxf(m, x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  // weights (kept in shared memory when staged) and their block sum
  float den = 0.f;
  for (int s = tid; s < n; s += kCombineThreads) {
    const float w = ex2_approx(lse_at(s) - m);
    if (staged) wsh[s] = w;
    den += w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if ((tid & 31) == 0) red[tid >> 5] = den;
  __syncthreads();
  den = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) den += red[w];
  // weighted sum of the partial outputs
  const int grp = tid / kLanesPerRow;
  const int c4 = (tid % kLanesPerRow) * 4;
  const float* po = part_o + static_cast<size_t>(bh) * n_part * D + c4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = grp; s < n; s += kGroups) {
    const float w = staged ? wsh[s] : ex2_approx(pl[s] - m);
    const float4 v = *reinterpret_cast<const float4*>(po + static_cast<size_t>(s) * D);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  *reinterpret_cast<float4*>(&acc_sh[grp][c4]) = acc;
  __syncthreads();
  if (tid < D) {
    float out = 0.f;
    if (n > 0) {
#pragma unroll
      for (int gi = 0; gi < kGroups; ++gi) out += acc_sh[gi][tid];
      out /= den;
    }
    if (o_dtype == GQA_OUT_F32)
      static_cast<float*>(o)[static_cast<size_t>(bh) * D + tid] = out;
    else
      static_cast<__nv_bfloat16*>(o)[static_cast<size_t>(bh) * D + tid] =
          __float2bfloat16_rn(out);
    if (lse_out != nullptr && tid == 0)
      lse_out[bh] = n > 0 ? (m + __log2f(den)) * 0.69314718055994531f : -INFINITY;
  }
}

int decode_split_len(int B, int h_q, int g, int S_max) {
  // The split pass streams the cache from HBM, which all CTAs share: once
  // enough CTAs are streaming, the total time is the cache bytes over the
  // bandwidth plus per-item costs (query load, partial write, and the
  // combine's reads of the partials), so fewer, longer items are better as
  // long as every CTA slot (two per SM of a 148-SM B300) gets one. Choose the
  // fewest splits per segment that give at least 80 % of the slots an item,
  // and cap an item at 2048 tokens so that sequences of very different
  // lengths still even out over the dynamic fetch. Only performance depends
  // on this choice.
  constexpr long long kSlots = 148LL * kCtasPerSm;
  constexpr long long kMaxLen = 2048;
  const long long G = h_q / g;
  const long long segs = static_cast<long long>(B) * g * ((G + 31) / 32);
  const long long want = (kSlots * 4 + 4) / 5;  // 80 % of the slots
  const long long n_split = segs >= want ? 1 : (want + segs - 1) / segs;
  long long l = (static_cast<long long>(S_max) + n_split - 1) / n_split;
  l = (l + kDecodeStage - 1) / kDecodeStage * kDecodeStage;
  if (l > kMaxLen) l = kMaxLen;
  if (l < kDecodeStage) l = kDecodeStage;
  return static_cast<int>(l);
}

template <int D, int MT>
static cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  constexpr int kSmem = DecCfg<D>::kSmem;
  static DeviceOnce attr_once;
  cudaError_t e = run_once_per_device(attr_once, [] {
    return cudaFuncSetAttribute(decode_split_kernel<D, MT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  const int n_hslice = (a.G + 31) / 32;
  const long long n_items = static_cast<long long>(a.B) * a.g * n_hslice * a.n_split;
  const long long slots = static_cast<long long>(device_sm_count()) * kCtasPerSm;
  const int grid = static_cast<int>(n_items < slots ? n_items : slots);
  // every segment's rows (a window: its rows plus up to 63 before it in its
  // first stage) fit one split: the split pass writes the output itself
  const long long w_rows = a.window < a.S_max ? a.window : a.S_max;
  const long long rows_max = a.window > 0 ? w_rows + kDecodeStage - 1 : a.S_max;
  const bool fused = rows_max <= a.split_len;
  // the item counter the persistent CTAs fetch from starts at zero
  e = cudaMemsetAsync(a.item_counter, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  decode_split_kernel<D, MT><<<grid, kThreads, kSmem, s>>>(
      a.tm_k, a.tm_v, static_cast<const __nv_bfloat16*>(a.q), a.seq_lens, a.part_o, a.part_lse,
      a.h_q, a.g, a.G, n_hslice, a.S_max, a.split_len, a.n_split, static_cast<int>(n_items),
      a.scale_log2, a.window, a.alibi, a.block_table, a.page_log2, a.num_pages, a.max_blocks,
      a.item_counter, a.o, a.o_dtype, a.lse, fused ? 1 : 0, a.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (fused) return cudaSuccess;
  // The combine is a programmatic dependent launch: its CTAs are scheduled
  // while the split pass drains and block in griddepcontrol.wait until it
  // has finished, which hides most of the launch gap between the two.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.h_q));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, static_cast<const float*>(a.part_o),
                            static_cast<const float*>(a.part_lse), a.seq_lens, a.o, a.o_dtype,
                            a.lse, a.h_q, a.S_max, a.split_len, a.n_split, kConsumers / MT,
                            a.window, a.status);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  // Groups larger than 32 query heads run as 32-row slices (separate items),
  // each re-reading the split; no workload here has G > 32.
  const int mt = (a.G + 15) / 16;
  if (a.d == 64) return mt <= 1 ? launch_decode_t<64, 1>(a, s) : launch_decode_t<64, 2>(a, s);
  return mt <= 1 ? launch_decode_t<128, 1>(a, s) : launch_decode_t<128, 2>(a, s);
}

}  // namespace gqa
