// fa_fwd_kernel.cuh — exact attention forward on sm_103a (tcgen05 + TMA).
//
// Method: "Hacker News Digest — gpu-computing", section "Алгоритм Flash
// Attention 2" (loop over query tiles; for each key/value tile form
// S = Q K^T * scale, apply the online softmax in place, accumulate S @ V),
// with the running max / denominator of section "v1 — базовая версия",
// item 3, and the FA2 work split of the "flash attention v3 paper" search
// page, third snippet (a thread block owns row blocks of O and walks all
// key/value blocks for them).  The division by the denominator is deferred
// to the epilogue, which gives the same result as the per-tile
// renormalisation the pages print.
//
// One CTA owns two 128-row query tiles (A: rows r0..r0+127, B: the next 128
// rows) of one (batch, query head); both share every K/V block the CTA
// loads.  Warp roles (320 threads):
//   warp 0     MMA issuer (one thread), see below
//   warp 1     TMA producer, see below
//   warps 2-5  softmax of tile A: warp w owns rows 32*(w%4) .. +31 of the
//              tile (its TMEM lane quadrant), one row per thread
//   warps 6-9  softmax of tile B (same lanes, its own TMEM columns)
//              each reads S from TMEM, masks the causal diagonal / ragged
//              tail, keeps the row's reference max m and sum l in the log2
//              domain (scale folded into one FFMA), writes P = exp2(s*c - m)
//              as bf16 into TMEM, rescales its O accumulator in TMEM when m
//              moves, and finally writes O / l and the LSE (each warp stages
//              its 32 rows in the K ring, idle once the last S MMA has run,
//              and one lane writes them with TMA stores).
//   TMA producer: Q_A and Q_B once, then K_j and V_j into two rings of
//              shared-memory stages (128-byte swizzle).
//   MMA issuer (one thread), in the order
//                 PV_A(j-1), S_A(j), PV_B(j-1), S_B(j), PV_A(j), ...
//              so the tensor pipe works on one tile while the other tile's
//              softmax runs.  S = Q K^T has both operands in shared memory
//              (K-major); O += P V takes P from TMEM and V (MN-major) from
//              shared memory.
//
// The reference max m is moved lazily: only when a block's max exceeds it
// by more than kRescaleLog2 (a factor 2^8).  O, l and every later p use the
// same m, so the result is exact either way; the threshold only bounds the
// size of p (<= 2^8) and of l and O (far below fp32 overflow).
//
// TMEM columns (512 allocated): S_A at 0, S_B at 128, O_A at 256, O_B after
// it (D columns each).  At D=128 P overwrites the first 64 columns of its own
// S (packed bf16x2) once the softmax has read S; the next S MMA into that
// region is issued after the P*V MMA that reads it, and tcgen05 MMAs issued
// by one thread execute in order.  At D=64 P has its own columns (384, 448).
// Nothing larger than one 128x128 score tile exists, and only on chip.
#pragma once

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBM = 128;          // query rows per tile (TMEM lanes)
constexpr int kBN = 128;          // keys per K/V block
constexpr int kTilesPerCta = 2;
constexpr int kBoxCols = 64;      // bf16 elements per 128-byte swizzle row
constexpr int kBoxBytes = kBM * kBoxCols * 2;   // one TMA box: 128 x 64 bf16
constexpr int kThreads = 320;
// The MMA and TMA warps come first: the warp schedulers favour older warps,
// and the single MMA-issuing thread must not queue behind the softmax warps.
constexpr int kMmaWarp = 0;
constexpr int kLoadWarp = 1;
constexpr int kSoftmaxWarp0 = 2;
constexpr float kRescaleLog2 = 8.0f;
// K/V bytes of the head groups a causal grid of one-unit CTAs runs
// together (see causal_grid_item): two heads of 32768 keys at head dim 128.
constexpr int64_t kCausalGroupKVBytes = 40ll << 20;
constexpr uint32_t kTmemCols = 512;

// QK8: Q and K are e4m3 (one byte per element) and S = Q K^T runs as
// kind::f8f6f4; V, P and O stay as without it.
template <int D, bool QK8 = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!QK8 || D == 128, "e4m3 Q/K at head dim 128 only");
  static constexpr int kTileBytes = kBM * D * 2;       // 16 KiB or 32 KiB
  static constexpr int kBoxes = D / kBoxCols;          // TMA boxes per tile
  // Q and K tiles: a 128-byte swizzle row holds 64 bf16 or 128 e4m3.
  static constexpr int kQKElemBytes = QK8 ? 1 : 2;
  static constexpr int kQKBoxCols = 128 / kQKElemBytes;
  static constexpr int kQKBoxes = D / kQKBoxCols;
  static constexpr int kQKTileBytes = kBM * D * kQKElemBytes;
  // Ring depths.  V_j is released one MMA group later than K_j (after the
  // second tile's P*V rather than its S), so V gets the deeper ring: both
  // loads are then issued two iterations ahead of their use.
  static constexpr int kKStages = (D == 128) ? (QK8 ? 4 : 2) : 4;
  static constexpr int kVStages = (D == 128) ? 3 : 4;
  // barriers: Q of tile A, K full/empty, V full/empty, S full x2, P full
  // x2, O final, drain, Q of tile B, first half of P x2
  static constexpr int kNumBars =
      1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 1 + 1 + 1 + 2;
  // + tmem slot (8 bytes with padding) + the wait state (24 bytes)
  static constexpr int kBarBytes = 8 * kNumBars + 32;
  static constexpr int kSmemBytes =
      1024 /*alignment slack*/ +
      kQKTileBytes * (kTilesPerCta + kKStages) + kTileBytes * kVStages +
      kBarBytes;
  // TMEM column of tile x's S, O and P.
  __host__ __device__ static constexpr uint32_t col_s(int x) {
    return x ? 128u : 0u;
  }
  __host__ __device__ static constexpr uint32_t col_o(int x) {
    return x ? 256u + D : 256u;
  }
  __host__ __device__ static constexpr uint32_t col_p(int x) {
    return D == 128 ? col_s(x) : (x ? 448u : 384u);
  }
  static constexpr uint32_t kIdescS = QK8 ? idesc_e4m3_f32(kBM, kBN)
                                          : idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
  // fp32 words of one partial slot: O rows [256][D] (unnormalised, relative
  // to the slot's reference max), then m[256] (log2 domain), l[256] (exact
  // row sums) and w[256] (row sums of the bf16 weights).
  static constexpr int64_t kSlotFloats =
      static_cast<int64_t>(kTilesPerCta * kBM) * (D + 3);
};

// The K ring holds the staged output rows of all eight softmax warps
// (32 rows x D bf16 each) once the last S MMA has read it.
template <int D, bool QK8>
constexpr bool k_ring_holds_output() {
  return 8 * 32 * D * 2 <=
         FwdCfg<D, QK8>::kKStages * FwdCfg<D, QK8>::kQKTileBytes;
}
static_assert(k_ring_holds_output<64, false>() &&
                  k_ring_holds_output<128, false>() &&
                  k_ring_holds_output<128, true>(),
              "output staging");

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int Nq, Nkv, Hq, Hkv;
  float scale_log2;   // scale * log2(e)
  int* status;        // device status word (bounded-wait timeouts)
  uint64_t wait_limit_ns;
  // Split-KV: each (batch, head, tile pair) is cut into kv_splits contiguous
  // ranges of K/V blocks, one CTA each.  With kv_splits > 1 the CTAs leave
  // fp32 partials in `work` (see kSlotFloats) for fa_merge_kernel.
  int kv_splits;
  float* work;
  // Stream schedule (fa_fwd_stream.cuh): batch count, K/V blocks per CTA,
  // and the value this launch's CTAs publish their partials under.
  int B;
  int stream_len;
  uint64_t epoch;
};

// S = Q K^T for one tile and one K/V block: D/16 MMAs of 128x128x16.  Both
// operands are K-major with the 128-byte swizzle; stepping K by 16 elements
// moves the start address 32 bytes within a swizzle row, and every 64
// elements to the next TMA box.  Offsets are compile-time constants added to
// the start-address field of prebuilt descriptors.
template <int D, bool QK8>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq,
                                         uint64_t dk, uint32_t idesc) {
  if constexpr (QK8) {
    // e4m3: K = 32 elements (32 bytes) per MMA, D / 32 MMAs in one box
    mma_ss8_w<0>(d_tmem, dq, dk, idesc);
#pragma unroll
    for (int kk = 1; kk < D / 32; ++kk) {
      const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
      mma_ss8_w<1>(d_tmem, dq + off, dk + off, idesc);
    }
  } else {
    mma_ss_w<0>(d_tmem, dq, dk, idesc);
#pragma unroll
    for (int kk = 1; kk < D / 16; ++kk) {
      const uint64_t off = static_cast<uint64_t>(
          ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
      mma_ss_w<1>(d_tmem, dq + off, dk + off, idesc);
    }
  }
}

// O += P V for one tile and one K/V block: 8 MMAs of 128xDx16.  P (bf16x2
// packed, 8 TMEM columns per 16 keys) comes from TMEM; V is MN-major with the
// 128-byte swizzle, 16 keys = 2048 bytes per step.  `acc` is false for the
// first block of a tile (initialises O).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t a_tmem,
                                         uint64_t dv, uint32_t idesc,
                                         bool acc) {
  mma_ts_w(d_tmem, a_tmem, dv, idesc, acc ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < kBN / 16; ++kk)
    mma_ts_wc<1>(d_tmem, a_tmem + kk * 8,
                 dv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc);
}

// The same P*V in two halves of the block's keys: H = 0 the first kBN/2
// keys (4 MMAs, `acc` as in issue_pv), H = 1 the rest (always accumulating).
template <int D, int H>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem,
                                              uint32_t a_tmem, uint64_t dv,
                                              uint32_t idesc, bool acc) {
  constexpr int k0 = H * (kBN / 32);
  if constexpr (H == 0)
    mma_ts_w(d_tmem, a_tmem, dv, idesc, acc ? 1u : 0u);
  else
    mma_ts_wc<1>(d_tmem, a_tmem + k0 * 8,
                 dv + static_cast<uint64_t>(k0 * (2048 >> 4)), idesc);
#pragma unroll
  for (int kk = k0 + 1; kk < k0 + kBN / 32; ++kk)
    mma_ts_wc<1>(d_tmem, a_tmem + kk * 8,
                 dv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc);
}

// Number of K/V blocks a tile starting at query row `row0` visits.
template <bool CAUSAL>
__device__ __forceinline__ int kv_blocks(int row0, int Nkv) {
  const int end = CAUSAL ? min(Nkv, row0 + kBM) : Nkv;
  return (end + kBN - 1) / kBN;
}

// The work unit (unit, head hq, batch b) of this CTA for a causal grid of
// (units, Hq, B) CTAs that start in grid order (x fastest).  With a causal
// mask the units (query-row ranges) differ in length, and one head's units
// longest first, head after head, leave the SMs unevenly loaded at every
// head's end; all units of the call longest first keep every head's K/V in
// use at once.  So the heads go in groups whose K and V (kv_head_bytes per
// KV head) together stay within kCausalGroupKVBytes, and so in L2, and each
// group's units longest first with its heads interleaved: a static list
// the hardware's in-order start deals out.
__device__ __forceinline__ void causal_grid_item(const FwdParams& p,
                                                 int64_t kv_head_bytes,
                                                 int& unit, int& hq, int& b) {
  const int n_units = static_cast<int>(gridDim.x);
  const int G = p.Hq / p.Hkv;
  const int gkv = static_cast<int>(max(
      int64_t{1}, kCausalGroupKVBytes / max(kv_head_bytes, int64_t{1})));
  const int BH = static_cast<int>(gridDim.y * gridDim.z);
  const int gsz = min(BH, gkv * G);
  const int i = static_cast<int>(blockIdx.x) +
                n_units * (static_cast<int>(blockIdx.y) +
                           static_cast<int>(gridDim.y) *
                               static_cast<int>(blockIdx.z));
  const int span = gsz * n_units;                  // items of a full group
  const int g = i / span;
  const int k = i - g * span;
  const int ng = min(gsz, BH - g * gsz);           // heads in this group
  unit = n_units - 1 - k / ng;
  const int bh = g * gsz + k % ng;
  b = bh / p.Hq;
  hq = bh - b * p.Hq;
}

// P = exp2(s * c - m) for the scores I0 .. I1-1 of one row (sr, fp32 bit
// patterns), packed to bf16x2 into pp (word i / 2 for key i), their fp32
// values added pairwise into the four f32x2 sums acc.  With MASK, only the
// first n_vis keys count (the others get p = 0).  The scores are scaled and
// shifted by one f32x2 FMA per pair; exp2 runs on the MUFU.
template <int I0, int I1, bool MASK>
__device__ __forceinline__ void exp_pack_range(const uint32_t* sr, float c,
                                               float m_use, int n_vis,
                                               uint32_t* pp, uint64_t* acc) {
  const uint64_t c2 = f2(c, c);
  const uint64_t nm2 = f2(-m_use, -m_use);
#pragma unroll
  for (int i = I0; i < I1; i += 2) {
    float x0, x1;
    f2_split(fma2(f2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])),
                  c2, nm2),
             x0, x1);
    if (MASK) {
      x0 = (i < n_vis) ? x0 : -INFINITY;
      x1 = (i + 1 < n_vis) ? x1 : -INFINITY;
    }
    const float e0 = ex2_approx(x0);
    const float e1 = ex2_approx(x1);
    acc[(i >> 1) & 3] = add2(acc[(i >> 1) & 3], f2(e0, e1));
    pp[i / 2] = pack_bf16x2(e0, e1);
  }
}

// The row sum of the four f32x2 sums of exp_pack_range.
__device__ __forceinline__ float exp_sum(const uint64_t* acc) {
  float s0, s1;
  f2_split(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), s0, s1);
  return s0 + s1;
}

// exp_pack_range over all N keys of the row; returns the row sum.
template <int N, bool MASK>
__device__ __forceinline__ float exp_pack_row(const uint32_t* sr, float c,
                                              float m_use, int n_vis,
                                              uint32_t* pp) {
  uint64_t acc[4] = {0, 0, 0, 0};
  exp_pack_range<0, N, MASK>(sr, c, m_use, n_vis, pp, acc);
  return exp_sum(acc);
}

// Rescale this row's O accumulator (TMEM at o_addr, D fp32 columns) by
// alpha, for the whole warp when any lane's alpha differs from 1.  S(j)
// complete means every earlier MMA of the issuing thread, including the P*V
// of the previous block, is complete, so O is stable here.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t o_addr, float alpha) {
  if (!__any_sync(0xffffffffu, alpha != 1.f)) return;
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t orr[32];
    tmem_ld32(o_addr + cc * 32, orr);
    tmem_ld_wait();
    reg_fence32(orr);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
    tmem_st32(o_addr + cc * 32, orr);
  }
}

// rescale_o in chunks of 8 columns, for a caller that still holds the
// block's scores in registers.
template <int D>
__device__ __forceinline__ void rescale_o_narrow(uint32_t o_addr,
                                                 float alpha) {
  if (!__any_sync(0xffffffffu, alpha != 1.f)) return;
#pragma unroll 1
  for (int cc = 0; cc < D / 8; ++cc) {
    uint32_t orr[8];
    tmem_ld8(o_addr + cc * 8, orr);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 8; ++i)
      orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
    tmem_st8(o_addr + cc * 8, orr);
  }
}

// exp_pack_row for one block of kBN keys, P written to TMEM in two halves:
// the first half is stored (8 columns at a time, as computed), O rescaled by
// alpha when the reference moved and O already holds earlier blocks
// (`o_live`), and every lane arrives on p_half_bar (count: the tile's
// threads) once those stores are complete, so that the first half's P*V can
// start while the second half is computed; the second half's store is left
// in flight.  Returns the row sum, added in the same order as exp_pack_row.
template <int D, bool MASK>
__device__ __forceinline__ float exp_pack_split(
    const uint32_t* sr, float c, float m_use, int n_vis, uint32_t* pp,
    uint32_t p_addr, uint32_t o_addr, bool o_live, float alpha,
    uint32_t p_half_bar) {
  uint64_t acc[4] = {0, 0, 0, 0};
  // the first half in pieces of 16 keys (8 packed columns), each stored as
  // soon as it is computed
  exp_pack_range<0, 16, MASK>(sr, c, m_use, n_vis, pp, acc);
  tmem_st8(p_addr, pp);
  exp_pack_range<16, 32, MASK>(sr, c, m_use, n_vis, pp, acc);
  tmem_st8(p_addr + 8, pp + 8);
  exp_pack_range<32, 48, MASK>(sr, c, m_use, n_vis, pp, acc);
  tmem_st8(p_addr + 16, pp + 16);
  exp_pack_range<48, 64, MASK>(sr, c, m_use, n_vis, pp, acc);
  tmem_st8(p_addr + 24, pp + 24);
  if (o_live) rescale_o_narrow<D>(o_addr, alpha);
  tmem_st_wait();
  tc_fence_before();
  mbar_arrive(p_half_bar);
  exp_pack_range<kBN / 2, kBN, MASK>(sr, c, m_use, n_vis, pp, acc);
  tmem_st32(p_addr + kBN / 4, pp + kBN / 4);
  return exp_sum(acc);
}

// The bf16 rounding error of a block's largest weight: with s_ext the
// block's extreme score (the one with the largest s * c), the weight is
// exp2(s_ext * c - m_use), computed as exp_pack_row computes it, and the
// result is round_bf16(p) - p.  Zero when the block has no visible key.
//
// Why: P V applies the bf16-rounded weights, so dividing O by the exact
// row sum leaves each weight's rounding (up to 2^-8 of it) in O.  When a
// row's weight concentrates on a few keys (large logits) that is up to
// 2^-8 |V| on top of O's own bf16 rounding; adding each block's largest
// weight's rounding to the divisor makes those terms cancel, while the
// roundings of the many small weights average out.  (On the 32768-key
// large-logit workload this gives the same largest |dO| as summing every
// rounded weight, at a few instructions per block instead of two per key.)
__device__ __forceinline__ float top_rounding(float s_ext, float c,
                                              float m_use) {
  const float p = ex2_approx(fmaf(s_ext, c, -m_use));
  const uint32_t b = pack_bf16x2(p, 0.f);
  return __uint_as_float(b << 16) - p;
}

// One K/V block of the online softmax, for the query row this thread owns
// (TMEM lane = row): reads the block's scores from TMEM at s_addr, takes the
// row's extreme over the visible keys, moves the reference max m_ref (log2
// domain) only when the block exceeds it by more than kRescaleLog2, writes
// P = exp2(s * c - m_ref) as packed bf16 to p_addr, adds the row sums to
// l_run (exact values) and w_run (the bf16 values; see exp_pack_row), and
// rescales O (at o_addr) when the reference moved and O already holds
// earlier blocks (`o_live`).  Returns once its TMEM stores are done and
// fenced; the caller then signals that P is ready.  Keys from col0 on are
// visible up to Nkv and, when CAUSAL, up to the row's own index q_abs.
// Steps: "Hacker News Digest — gpu-computing", section "v1 — базовая
// версия", item 3 (running max and denominator); the lazy rescale is the
// one-pass form of the same recurrence with a stale reference.  INTERIOR:
// no key of the block needs masking here (every key is visible to every row
// of the tile, or the hidden ones already hold the extreme's identity as
// their score, see hide_keys), and no mask code is compiled.  SPLIT_P: P is
// written in two halves of the block's keys, and once the first half (and
// any rescale of O) is stored and fenced the warp arrives on p_half_bar, so
// that its P*V can start while the second half is computed.
template <int D, bool CAUSAL, bool INTERIOR = false, bool SPLIT_P = false>
__device__ __forceinline__ void softmax_block(
    uint32_t s_addr, uint32_t p_addr, uint32_t o_addr, int col0, int my_row0,
    int q_abs, int Nkv, float c, bool neg_scale, bool o_live, float& m_ref,
    float& l_run, float& w_run, uint32_t p_half_bar = 0) {
  uint32_t sr[kBN];
  const bool need_mask =
      !INTERIOR &&
      ((col0 + kBN > Nkv) || (CAUSAL && col0 + kBN - 1 > my_row0));
  // Unmasked blocks take the row's extreme from reducing TMEM loads (one
  // max/min per 32 columns, computed by the load itself).
  float red[kBN / 32];
  if (!need_mask && !neg_scale) {
#pragma unroll
    for (int cc = 0; cc < kBN / 32; ++cc)
      tmem_ld32_max(s_addr + cc * 32, sr + cc * 32, red[cc]);
  } else if (!need_mask) {
#pragma unroll
    for (int cc = 0; cc < kBN / 32; ++cc)
      tmem_ld32_min(s_addr + cc * 32, sr + cc * 32, red[cc]);
  } else {
#pragma unroll
    for (int cc = 0; cc < kBN / 32; ++cc) {
      tmem_ld32(s_addr + cc * 32, sr + cc * 32);
      red[cc] = 0.f;
    }
  }
  tmem_ld_wait();
#pragma unroll
  for (int cc = 0; cc < kBN / 32; ++cc) {
    reg_fence32(sr + cc * 32);
    reg_fence_f(red[cc]);
  }
#define S_(i) __uint_as_float(sr[(i)])

  // ---- row extreme over the visible keys of this block ----
  int n_vis = kBN;   // keys [col0, col0 + n_vis) are visible to this row
  if (need_mask) {
    int lim = Nkv - col0;
    if (CAUSAL) lim = min(lim, q_abs - col0 + 1);
    n_vis = max(0, min(kBN, lim));
  }
  float ext;
  if (!need_mask) {
    ext = neg_scale ? fminf(fminf(red[0], red[1]), fminf(red[2], red[3]))
                    : fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  } else {
    // four independent chains of three-input extremes over the visible
    // keys (the others take the identity)
    const float idn = neg_scale ? INFINITY : -INFINITY;
    float e4[4] = {idn, idn, idn, idn};
#pragma unroll
    for (int i = 0; i < kBN; i += 2) {
      const float v0 = (i < n_vis) ? S_(i) : idn;
      const float v1 = (i + 1 < n_vis) ? S_(i + 1) : idn;
      float& e = e4[(i >> 1) & 3];
      e = neg_scale ? fmin3(e, v0, v1) : fmax3(e, v0, v1);
    }
    ext = neg_scale ? fminf(fminf(e4[0], e4[1]), fminf(e4[2], e4[3]))
                    : fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]));
  }
  const float m_blk = (n_vis > 0) ? ext * c : -INFINITY;
  // Move the reference max only when this block exceeds it by more than
  // the threshold (always on the first visible block).
  const bool move = m_blk > m_ref + kRescaleLog2 ||
                    (m_ref == -INFINITY && m_blk != -INFINITY);
  const float m_new = move ? m_blk : m_ref;
  const float alpha =
      (move && m_ref != -INFINITY) ? ex2_approx(m_ref - m_new) : 1.f;
  const float m_use = (m_new == -INFINITY) ? 0.f : m_new;

  // the divisor of O also takes the rounding of this block's largest weight
  w_run = w_run * alpha + (n_vis > 0 ? top_rounding(ext, c, m_use) : 0.f);

  // ---- P = exp2(s * c - m), packed to bf16, row sums ----
  uint32_t pp[kBN / 2];
  float rsum;
  if constexpr (SPLIT_P) {
    rsum = need_mask
               ? exp_pack_split<D, true>(sr, c, m_use, n_vis, pp, p_addr,
                                         o_addr, o_live, alpha, p_half_bar)
               : exp_pack_split<D, false>(sr, c, m_use, kBN, pp, p_addr,
                                          o_addr, o_live, alpha, p_half_bar);
  } else {
    rsum = need_mask ? exp_pack_row<kBN, true>(sr, c, m_use, n_vis, pp)
                     : exp_pack_row<kBN, false>(sr, c, m_use, kBN, pp);
  }
#undef S_
  l_run = l_run * alpha + rsum;
  w_run += rsum;
  m_ref = m_new;

  if constexpr (!SPLIT_P) {
    // ---- rescale O when the reference max moved ----
    if (o_live) rescale_o<D>(o_addr, alpha);
    tmem_st32(p_addr, pp);
    tmem_st32(p_addr + 32, pp + 32);
  }
  tmem_st_wait();
  tc_fence_before();
}

// Hide the keys n_vis .. kBN-1 of this block from this thread's row: their
// scores in TMEM (the warp's 32 lanes at s_addr, kBN fp32 columns) become
// idn, the identity of the row extreme (-inf, or +inf for a negative scale)
// and a score whose weight exp2(idn * c - m) is 0 for any nonzero scale c.
// The unmasked softmax_block then gives this block the same bits as the
// masked one.  Chunks of 32 keys that every lane of the warp sees are left
// alone, chunks that no lane sees are overwritten whole, and the chunks in
// between are read, masked key by key and written back.  Returns once the
// stores are complete.
__device__ __forceinline__ void hide_keys(uint32_t s_addr, int n_vis,
                                          float idn) {
  const int lo = __reduce_min_sync(0xffffffffu, n_vis);  // all lanes see < lo
  const int hi = __reduce_max_sync(0xffffffffu, n_vis);  // no lane sees >= hi
  const uint32_t idn_b = __float_as_uint(idn);
#pragma unroll 1
  for (int cc = lo >> 5; cc < kBN / 32; ++cc) {
    uint32_t v[32];
    if (cc * 32 >= hi) {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = idn_b;
    } else {
      tmem_ld32(s_addr + cc * 32, v);
      tmem_ld_wait();
      reg_fence32(v);
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (cc * 32 + k >= n_vis) v[k] = idn_b;
    }
    tmem_st32(s_addr + cc * 32, v);
  }
  tmem_st_wait();
}

// Where a warp's finished rows go.  smem == 0: each lane stores its own row
// (one 16-byte store per 8 columns; a warp's store then touches 32 rows).
// Otherwise smem is free, 1024-byte aligned shared memory of 32 * D * 2
// bytes: the 32 rows are staged there as D/64 boxes of 32 rows x 128 bytes in
// the 128-byte swizzle (16-byte chunk k of row r at position k ^ (r & 7), so
// eight lanes' stores hit distinct banks) and one lane writes the boxes with
// TMA stores through `map` (the O tensor, boxes of 64 columns x 32 rows),
// starting at row row0 of slice z, whose rows run to n; rows past n are
// dropped by the TMA unit, and a warp whose rows all lie past n stores
// nothing.
struct OutRows {
  uint32_t smem;
  const CUtensorMap* map;
  int row0, z, n;
};

template <int D>
__device__ __forceinline__ void put_row_chunk(const OutRows& out, int lane,
                                              int cc, const uint32_t* packed,
                                              __nv_bfloat16* orow,
                                              bool in_range) {
  if (out.smem != 0) {
    const uint32_t row = out.smem + (cc >> 1) * (32 * 128) +
                         static_cast<uint32_t>(lane) * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t k = static_cast<uint32_t>((cc & 1) * 4 + i);
      st_shared_v4(row + ((k ^ static_cast<uint32_t>(lane & 7)) << 4),
                   packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                   packed[4 * i + 3]);
    }
  } else if (in_range) {
    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1],
                          packed[4 * i + 2], packed[4 * i + 3]);
  }
}

// After every lane has put all its chunks: write the staged boxes (no-op for
// direct stores).  Returns once the TMA unit has read the shared memory.
template <int D>
__device__ __forceinline__ void flush_rows(const OutRows& out, int lane) {
  if (out.smem == 0) return;
  fence_async_smem();
  __syncwarp();
  if (lane == 0 && out.row0 < out.n) {
#pragma unroll
    for (int box = 0; box < D / 64; ++box)
      tma_store_3d(out.map, out.smem + box * (32 * 128), box * 64, out.row0,
                   out.z);
    tma_store_commit();
    tma_store_wait_read();
  }
  __syncwarp();
}

// The last step for one query row: O (unnormalised, in TMEM at o_addr,
// relative to the reference max m_ref) divided by w_run, the row sum of the
// bf16 weights P V applied, rounded to bf16 and stored (see OutRows; orow is
// the row's address for direct stores); LSE = (m_ref + log2 l_run) ln 2 from
// the exact row sum, at lse_at (skipped when null).  Rows past the end
// (`in_range` false) store nothing.
template <int D>
__device__ __forceinline__ void store_final_row(uint32_t o_addr, float m_ref,
                                                float l_run, float w_run,
                                                __nv_bfloat16* orow,
                                                float* lse_at, bool in_range,
                                                const OutRows& out) {
  const float inv_l = (w_run > 0.f) ? 1.f / w_run : 0.f;
  const int lane = static_cast<int>(threadIdx.x & 31);
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t orr[32];
    tmem_ld32(o_addr + cc * 32, orr);
    tmem_ld_wait();
    reg_fence32(orr);
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l,
                              __uint_as_float(orr[2 * i + 1]) * inv_l);
    put_row_chunk<D>(out, lane, cc, packed, orow, in_range);
  }
  flush_rows<D>(out, lane);
  if (in_range && lse_at != nullptr) {
    const float lse2 = (l_run > 0.f) ? (m_ref + log2f(l_run)) : -INFINITY;
    *lse_at = lse2 * 0.69314718055994530942f;
  }
}

// SPLIT: the grid's z index also carries the K/V range (split-KV) and the
// epilogue writes fp32 partials; without it the code is the plain one-pair-
// per-CTA forward.
template <int D, bool CAUSAL, bool SPLIT, bool QK8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, QK8>;
  constexpr int NK = C::kKStages;
  constexpr int NV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (batch b, query head hq, tile pair) ----
  const int n_pairs = gridDim.x;
  int pair = CAUSAL ? (n_pairs - 1 - static_cast<int>(blockIdx.x))
                    : static_cast<int>(blockIdx.x);
  int hq = blockIdx.y;
  const int splits = SPLIT ? p.kv_splits : 1;
  int b = SPLIT ? static_cast<int>(blockIdx.z) / splits
                : static_cast<int>(blockIdx.z);
  const int split = SPLIT ? static_cast<int>(blockIdx.z) - b * splits : 0;
  if constexpr (CAUSAL && !SPLIT)
    causal_grid_item(p, 4ll * p.Nkv * D, pair, hq, b);   // see there
  const int hk = hq / (p.Hq / p.Hkv);
  const int row0[2] = {pair * (2 * kBM), pair * (2 * kBM) + kBM};
  const bool has_b = row0[1] < p.Nq;
  const int nblk[2] = {kv_blocks<CAUSAL>(row0[0], p.Nkv),
                       has_b ? kv_blocks<CAUSAL>(row0[1], p.Nkv) : 0};
  // This CTA's contiguous range [j0, j1) of the pair's K/V blocks.  A tile
  // visits the prefix [j0, min(j1, nblk)) of it (causal tiles end earlier).
  const int n_pair = max(nblk[0], nblk[1]);
  const int chunk = SPLIT ? (n_pair + splits - 1) / splits : n_pair;
  const int j0 = SPLIT ? min(n_pair, split * chunk) : 0;
  const int n_blocks = SPLIT ? min(n_pair, j0 + chunk) - j0 : n_pair;

  // ---- shared memory carve-up (1024-byte aligned for the swizzle atoms) --
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sQ = base;                          // Q_A, then Q_B
  const uint32_t sK = sQ + kTilesPerCta * C::kQKTileBytes;
  const uint32_t sV = sK + NK * C::kQKTileBytes;
  const uint32_t sBar = sV + NV * C::kTileBytes;
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  const uint32_t bQFull = bar(0);
  constexpr int kB0 = 1 + 2 * NK + 2 * NV;       // first non-ring barrier
  auto bKFull = [&](int s) { return bar(1 + s); };
  auto bKEmpty = [&](int s) { return bar(1 + NK + s); };
  auto bVFull = [&](int s) { return bar(1 + 2 * NK + s); };
  auto bVEmpty = [&](int s) { return bar(1 + 2 * NK + NV + s); };
  auto bSFull = [&](int x) { return bar(kB0 + x); };
  auto bPFull = [&](int x) { return bar(kB0 + 2 + x); };
  const uint32_t bOFinal = bar(kB0 + 4);
  const uint32_t bDrain = bar(kB0 + 5);
  // Q of tile A at bQFull, of tile B here: S_A(first) waits only for Q_A
  const uint32_t bQFullB = bar(kB0 + 6);
  // first half of tile x's P stored (see softmax_block)
  auto bPHalf = [&](int x) { return bar(kB0 + 7 + x); };
  uint8_t* const misc = base_ptr + (sBar - base) + 8 * C::kNumBars;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  WaitState* const wstate = reinterpret_cast<WaitState*>(misc + 8);

  if (threadIdx.x == 0) {
    mbar_init(bQFull, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(bKFull(s), 1);
      mbar_init(bKEmpty(s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bVFull(s), 1);
      mbar_init(bVEmpty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bSFull(x), 1);
      mbar_init(bPFull(x), 4);
      mbar_init(bPHalf(x), 4 * 32);
    }
    mbar_init(bOFinal, 1);
    mbar_init(bDrain, 1);
    mbar_init(bQFullB, 1);
    wstate->abort = 0u;
    wstate->status = p.status;
    wstate->limit_ns = p.wait_limit_ns;
    mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{smem_addr(wstate)};

  if (warp == kLoadWarp) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      const int zq = b * p.Hq + hq;
      const int zk = b * p.Hkv + hk;
      // Order of the first loads: Q_A, K_0, then Q_B, so S_A(0) can start
      // once the first two have landed (at the start every CTA loads from
      // DRAM at once).
      auto load_q = [&](int x, uint32_t qbar) {
        mbar_arrive_expect_tx(qbar, C::kQKTileBytes);
        for (int c = 0; c < C::kQKBoxes; ++c)
          tma_load_3d(sQ + x * C::kQKTileBytes + c * kBoxBytes, &tmQ, qbar,
                      c * C::kQKBoxCols, row0[x], zq, once);
      };
      load_q(0, bQFull);
      bool q_b_issued = false;
      int k_issued = 0, v_issued = 0;
      for (int i = 0; i < n_blocks; ++i) {
        const int j = j0 + i;                    // block index in the pair
        const int sk = i % NK, sv = i % NV;
        if (!mbar_wait(bKEmpty(sk), ((i / NK) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bKFull(sk), C::kQKTileBytes);
        for (int c = 0; c < C::kQKBoxes; ++c)
          tma_load_3d(sK + sk * C::kQKTileBytes + c * kBoxBytes, &tmK,
                      bKFull(sk), c * C::kQKBoxCols, j * kBN, zk, keep);
        k_issued = i + 1;
        if (has_b && !q_b_issued) {
          load_q(1, bQFullB);
          q_b_issued = true;
        }
        if (!mbar_wait(bVEmpty(sv), ((i / NV) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bVFull(sv), C::kTileBytes);
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_3d(sV + sv * C::kTileBytes + c * kBoxBytes, &tmV,
                      bVFull(sv), c * kBoxCols, j * kBN, zk, keep);
        v_issued = i + 1;
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the
      // last load issued into each stage of each ring, and for Q.
      for (int j = (k_issued > NK ? k_issued - NK : 0); j < k_issued; ++j)
        mbar_wait(bKFull(j % NK), (j / NK) & 1, wc, false);
      for (int j = (v_issued > NV ? v_issued - NV : 0); j < v_issued; ++j)
        mbar_wait(bVFull(j % NV), (j / NV) & 1, wc, false);
      mbar_wait(bQFull, 0, wc, false);
      if (q_b_issued) mbar_wait(bQFullB, 0, wc, false);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ==============================
    // The whole warp runs this loop, converged and with warp-uniform values;
    // one elected lane issues each MMA and commit.  Wait outcomes are made
    // warp-uniform before they steer control flow.
    constexpr uint32_t kAll = 0xffffffffu;
    // Descriptors of every operand tile, built once.
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = sdesc_sw128(sV, kBoxBytes, 1024);
    constexpr uint64_t kStep = static_cast<uint64_t>(C::kTileBytes >> 4);
    constexpr uint64_t kQKStep = static_cast<uint64_t>(C::kQKTileBytes >> 4);
    bool ok = __all_sync(kAll, mbar_wait(bQFull, 0, wc));
    // j counts this CTA's blocks (ring position); block j0 + j of the pair
    for (int j = 0; ok && j <= n_blocks; ++j) {
      const int s = j % NK;                  // K stage of block j
      const int sp = (j + NV - 1) % NV;      // V stage of block j-1
      if (j >= 1 &&
          !(ok = __all_sync(kAll, mbar_wait(bVFull(sp), ((j - 1) / NV) & 1,
                                            wc))))
        break;
      if (j < n_blocks &&
          !(ok = __all_sync(kAll, mbar_wait(bKFull(s), (j / NK) & 1, wc))))
        break;
      const uint64_t dKs = dK + static_cast<uint64_t>(s) * kQKStep;
      const uint64_t dVs = dV + static_cast<uint64_t>(sp) * kStep;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        // O_x += P_x(j-1) V_{j-1}, each half of the keys once its half of
        // P is stored
        if (j >= 1 && j0 + j - 1 < nblk[x]) {
          if (!(ok = __all_sync(kAll,
                                mbar_wait(bPHalf(x), (j - 1) & 1, wc))))
            break;
          tc_fence_after();
          issue_pv_half<D, 0>(tmem + C::col_o(x), tmem + C::col_p(x), dVs,
                              C::kIdescPV, j > 1);
          if (!(ok = __all_sync(kAll,
                                mbar_wait(bPFull(x), (j - 1) & 1, wc))))
            break;
          tc_fence_after();
          issue_pv_half<D, 1>(tmem + C::col_o(x), tmem + C::col_p(x), dVs,
                              C::kIdescPV, true);
        }
        // S_x(j) = Q_x K_j^T
        if (j < n_blocks && j0 + j < nblk[x]) {
          if (x == 1 && j == 0 &&
              !(ok = __all_sync(kAll, mbar_wait(bQFullB, 0, wc))))
            break;
          issue_qk<D, QK8>(tmem + C::col_s(x),
                           dQ + static_cast<uint64_t>(x) * kQKStep, dKs,
                           C::kIdescS);
          mma_commit_w(bSFull(x));
        }
      }
      if (!ok) break;
      if (j < n_blocks) mma_commit_w(bKEmpty(s));
      if (j >= 1) mma_commit_w(bVEmpty(sp));
    }
    mma_commit_w(bOFinal);
    // Every MMA this warp issued completes before the CTA tears down.
    mma_commit_w(bDrain);
    mbar_wait(bDrain, 0, wc, false);
  } else {
    // ============================ softmax warps ===========================
    const int x = (warp - kSoftmaxWarp0) >> 2;     // tile A (0) or B (1)
    // blocks of this tile in the CTA's range: [j0, j0 + nb)
    const int nb = max(0, min(j0 + n_blocks, x ? nblk[1] : nblk[0]) - j0);
    const int my_row0 = x ? row0[1] : row0[0];
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    const bool neg_scale = c < 0.f;
    // TMEM lane quadrant of a warp is fixed by warp % 4.
    const int q_abs = my_row0 + (warp & 3) * 32 + lane;
    float m_ref = -INFINITY;   // reference max (log2 domain) of p and l
    float l_run = 0.f;         // sum of exp2(s*c - m_ref) over seen keys
    float w_run = 0.f;         // the same sum of the bf16-rounded values
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      // Warp-uniform outcome: the tcgen05 loads below are .sync.aligned.
      if (!(ok = __all_sync(0xffffffffu,
                            mbar_wait(bSFull(x), j & 1, wc))))
        break;
      tc_fence_after();
      softmax_block<D, CAUSAL, false, true>(
          tmem + lane_off + C::col_s(x), tmem + lane_off + C::col_p(x),
          tmem + lane_off + C::col_o(x), (j0 + j) * kBN, my_row0, q_abs,
          p.Nkv, c, neg_scale, j >= 1, m_ref, l_run, w_run, bPHalf(x));
      __syncwarp();
      if (lane == 0) mbar_arrive(bPFull(x));
    }

    // ---- epilogue ----
    // The merge of split-KV partials may be scheduled from here on; it
    // waits for this whole grid before it reads them.
    if constexpr (SPLIT) grid_dep_launch();
    if constexpr (SPLIT) {
      // Partial of one K/V range: unnormalised O (relative to m_ref), m and
      // l per row, for fa_merge_kernel.  A tile with no block in this range
      // leaves l = 0, m = -inf.
      float* slot = p.work + ((static_cast<int64_t>(b) * p.Hq + hq) *
                                  static_cast<int64_t>(gridDim.x) +
                              pair) * splits * C::kSlotFloats +
                    static_cast<int64_t>(split) * C::kSlotFloats;
      const int prow = q_abs - pair * (2 * kBM);     // row within the pair
      if (ok && nb > 0)
        ok = __all_sync(0xffffffffu, mbar_wait(bOFinal, 0, wc));
      if (ok && nb > 0) {
        tc_fence_after();
        const uint32_t o_addr = tmem + lane_off + C::col_o(x);
        float4* orow = reinterpret_cast<float4*>(slot + prow * D);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          tmem_ld32(o_addr + cc * 32, orr);
          tmem_ld_wait();
          reg_fence32(orr);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            orow[cc * 8 + i] = make_float4(
                __uint_as_float(orr[4 * i]), __uint_as_float(orr[4 * i + 1]),
                __uint_as_float(orr[4 * i + 2]),
                __uint_as_float(orr[4 * i + 3]));
        }
      }
      slot[kTilesPerCta * kBM * D + prow] = nb > 0 ? m_ref : -INFINITY;
      slot[kTilesPerCta * kBM * D + kTilesPerCta * kBM + prow] =
          nb > 0 ? l_run : 0.f;
      slot[kTilesPerCta * kBM * D + 2 * kTilesPerCta * kBM + prow] =
          nb > 0 ? w_run : 0.f;
    } else {
    if (ok && nb > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bOFinal, 0, wc));
    if (ok && nb > 0) {
      tc_fence_after();
      const size_t row_idx =
          (static_cast<size_t>(b) * p.Hq + hq) * static_cast<size_t>(p.Nq) +
          static_cast<size_t>(q_abs);
      // Every MMA is complete and every K tile consumed: the K ring is free
      // shared memory for staging the rows (8 warps x 32 rows x D bf16 fit
      // in it at both head dims).
      const int role = warp - kSoftmaxWarp0;
      const OutRows out{sK + static_cast<uint32_t>(role) * (32u * D * 2u),
                        &tmO, my_row0 + (warp & 3) * 32, b * p.Hq + hq, p.Nq};
      store_final_row<D>(tmem + lane_off + C::col_o(x), m_ref, l_run, w_run,
                         p.o + row_idx * D,
                         p.lse != nullptr ? p.lse + row_idx : nullptr,
                         q_abs < p.Nq, out);
    }
    }
  }

  // ---- teardown: every role is done with TMEM and shared memory ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Split-KV merge: for every query row, combine the partials of its K/V
// ranges.  Range s left O_s (unnormalised, relative to its reference max
// m_s, log2 domain), l_s (exact row sum) and w_s (row sum of the bf16
// weights); with m = max_s m_s
//     l = sum_s l_s 2^(m_s - m),   w = sum_s w_s 2^(m_s - m),
//     O = sum_s O_s 2^(m_s - m) / w,   LSE = (m + log2 l) ln 2,
// the same rescaling the online softmax applies between K/V blocks.  A
// partial slot covers one unit of ROWS query rows (a tile pair of the
// two-tile kernel, a tile of the wide-head kernel): fp32 O [ROWS][D], then
// m [ROWS], l [ROWS], w [ROWS].  One thread per (row, 4 columns).
template <int D>
struct MergeCfg {
  static constexpr int kChunks = D / 4;           // float4 per row
  static constexpr int kRowsPerBlock = (D == 64) ? 16 : (D == 128) ? 8 : 4;
  static constexpr int kThreads = kRowsPerBlock * kChunks;
};

template <int D, int ROWS>
__global__ void __launch_bounds__(MergeCfg<D>::kThreads)
    fa_merge_kernel(const __grid_constant__ FwdParams p) {
  using M = MergeCfg<D>;
  constexpr int64_t kSlot = static_cast<int64_t>(ROWS) * (D + 3);
  const int splits = p.kv_splits;
  constexpr int kBlocksPerUnit = ROWS / M::kRowsPerBlock;
  const int unit = static_cast<int>(blockIdx.x) / kBlocksPerUnit;
  const int prow = (static_cast<int>(blockIdx.x) % kBlocksPerUnit) *
                       M::kRowsPerBlock +
                   static_cast<int>(threadIdx.x) / M::kChunks;
  const int ch = static_cast<int>(threadIdx.x) % M::kChunks;
  const int hq = blockIdx.y, b = blockIdx.z;
  const int q_row = unit * ROWS + prow;
  // Launched while the forward grid runs: wait for it (and its partials).
  grid_dep_wait();
  if (q_row >= p.Nq) return;
  const int n_units = (p.Nq + ROWS - 1) / ROWS;
  const float* base = p.work + ((static_cast<int64_t>(b) * p.Hq + hq) *
                                    n_units + unit) * splits * kSlot;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s)
    m = fmaxf(m, base[s * kSlot + ROWS * D + prow]);
  float l = 0.f, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = 0; s < splits; ++s) {
    const float* slot = base + s * kSlot;
    const float ms = slot[ROWS * D + prow];
    if (ms == -INFINITY) continue;                // range saw no key
    const float w = ex2_approx(ms - m);
    l += slot[ROWS * D + ROWS + prow] * w;
    wsum += slot[ROWS * D + 2 * ROWS + prow] * w;
    const float4 o = reinterpret_cast<const float4*>(slot + prow * D)[ch];
    acc.x += o.x * w;
    acc.y += o.y * w;
    acc.z += o.z * w;
    acc.w += o.w * w;
  }
  const float inv_l = (wsum > 0.f) ? 1.f / wsum : 0.f;
  const size_t row_idx =
      (static_cast<size_t>(b) * p.Hq + hq) * static_cast<size_t>(p.Nq) +
      static_cast<size_t>(q_row);
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv_l, acc.y * inv_l);
  packed.y = pack_bf16x2(acc.z * inv_l, acc.w * inv_l);
  reinterpret_cast<uint2*>(p.o + row_idx * D)[ch] = packed;
  if (ch == 0 && p.lse != nullptr)
    p.lse[row_idx] =
        (l > 0.f ? (m + log2f(l)) : -INFINITY) * 0.69314718055994530942f;
}

}  // namespace fa
