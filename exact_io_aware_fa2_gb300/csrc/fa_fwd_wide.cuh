// fa_fwd_wide.cuh — the attention forward with one query tile per CTA: head
// dims 192 and 256, and causal shapes at head dim 64 (two CTAs per SM).
//
// Same method as fa_fwd_kernel.cuh ("Hacker News Digest — gpu-computing",
// section "Алгоритм Flash Attention 2", with the online softmax of section
// "v1 — базовая версия", item 3, and the division by the denominator
// deferred to the epilogue); wide heads are the "head_dim > 128" direction
// that page's closing notes point to.  Only the schedule differs, because an
// fp32 O of 192 or 256 columns leaves TMEM room for one query tile per CTA:
//
//   TMEM (512 columns): S buffers at 0 and 64 (64 keys each), O at 128
//   (D columns).  P(j) (bf16x2, 32 columns) overwrites the first half of
//   its own S buffer once the softmax has read S(j).
//
// K/V blocks are 64 keys, and the two S buffers let the MMA warp issue
// S(j+1) = Q K_{j+1}^T before P(j) exists:
//
//   tensor pipe:  S(0) S(1) PV(0) S(2) PV(1) S(3) PV(2) ...
//
// so the softmax of block j runs while S(j+1) executes, and the pipe waits
// only when a block's softmax is slower than the next block's S.  S(j+2)
// reuses the buffer of S(j) and P(j); it is issued after PV(j), and MMAs
// issued by one thread execute in order.
//
// Because S(j+1) completes before PV(j) has run, a softmax that must
// rescale O (its reference max moved) first waits for PV(j) on the
// pv_done barrier.  The wait is unambiguous: PV(j+1) cannot run before this
// softmax publishes P(j+1).
//
// At head dim 64 the CTA needs 192 TMEM columns (256 allocated) and about
// 64 KiB of shared memory, so two CTAs share an SM: they keep its tensor
// pipe busy in turn, and one's start-up and epilogue overlap the other's
// work, which pays for causal shapes with many short CTAs.
//
// Warp roles (192 threads): warp 0 MMA issuer (one elected lane), warp 1
// TMA producer, warps 2-5 softmax (warp w owns rows 32*(w%4) .. +31 of the
// tile, one row per thread).
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kWideThreads = 192;
constexpr int kWideMmaWarp = 0;
constexpr int kWideLoadWarp = 1;
constexpr int kWideSoftmaxWarp0 = 2;

template <int D>
struct WideCfg {
  static_assert(D == 64 || D == 192 || D == 256, "one-tile head dim");
  // keys per K/V block: TMEM holds two S buffers of kBN columns and O
  static constexpr int kBN = 64;
  static constexpr int kBoxes = D / kBoxCols;              // 64-column boxes
  static constexpr int kQBoxBytes = kBM * kBoxCols * 2;    // 128 rows: 16 KiB
  static constexpr int kKVBoxBytes = kBN * kBoxCols * 2;   // kBN rows
  static constexpr int kQBytes = kBoxes * kQBoxBytes;
  static constexpr int kKVBytes = kBoxes * kKVBoxBytes;
  // K_{j+1} is needed one step before V_j (S(j+1) is issued before PV(j)),
  // so K gets the deeper ring; 227 KiB of shared memory bounds the total.
  static constexpr int kKStages = 3;
  static constexpr int kVStages = (D == 256) ? 2 : 3;
  // barriers: Q, K full/empty, V full/empty, S full x2, P full x2, PV done,
  // O final, drain
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 3;
  static constexpr int kBarBytes = 8 * kNumBars + 32;  // + tmem slot, waits
  // At D = 64 two CTAs share an SM (TMEM: 2 x 64 S + 64 O columns, 256
  // allocated): padding shared memory past a third of the SM's keeps a
  // third CTA, which would wait for TMEM, from being scheduled beside them.
  static constexpr int kCtasPerSm = (D == 64) ? 2 : 1;
  static constexpr uint32_t kTmemAlloc = (D == 64) ? 256u : 512u;
  static constexpr int kSmemUsed = 1024 + kQBytes +
                                   (kKStages + kVStages) * kKVBytes + kBarBytes;
  static constexpr int kSmemBytes =
      (D == 64 && kSmemUsed < 80 * 1024) ? 80 * 1024 : kSmemUsed;
  static constexpr uint32_t kColO = 2 * kBN;
  // fp32 words of one split-KV partial slot: O rows [128][D] (unnormalised,
  // relative to the slot's reference max), then m[128], l[128] (exact row
  // sums) and w[128] (row sums of the bf16 weights).
  static constexpr int64_t kSlotFloats = static_cast<int64_t>(kBM) * (D + 3);
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
  // the K ring holds the four softmax warps' staged output rows
  static_assert(4 * 32 * D * 2 <= kKStages * kKVBytes, "output staging");
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
};

// S = Q K^T for one block: D/16 MMAs of 128 x kBN x 16, both operands
// K-major with the 128-byte swizzle.  Stepping K by 16 elements moves 32
// bytes within a swizzle row and, every 64 elements, to the next box (16 KiB
// for the 128-row Q box, kBN * 128 bytes for the K box).
template <int D>
__device__ __forceinline__ void wide_issue_qk(uint32_t d_tmem, uint64_t dq,
                                              uint64_t dk, uint32_t idesc) {
  using W = WideCfg<D>;
  mma_ss_w<0>(d_tmem, dq, dk, idesc);
#pragma unroll
  for (int kk = 1; kk < D / 16; ++kk) {
    const uint64_t in_row = static_cast<uint64_t>(((kk & 3) * 32) >> 4);
    const uint64_t qoff =
        in_row + static_cast<uint64_t>(((kk >> 2) * W::kQBoxBytes) >> 4);
    const uint64_t koff =
        in_row + static_cast<uint64_t>(((kk >> 2) * W::kKVBoxBytes) >> 4);
    mma_ss_w<1>(d_tmem, dq + qoff, dk + koff, idesc);
  }
}

// O += P V for one block: kBN/16 MMAs of 128xDx16.  P (bf16x2, 8 TMEM
// columns per 16 keys) comes from TMEM; V is MN-major with the 128-byte
// swizzle (16 keys = 2048 bytes).
template <int D>
__device__ __forceinline__ void wide_issue_pv(uint32_t d_tmem, uint32_t a_tmem,
                                              uint64_t dv, uint32_t idesc,
                                              bool acc) {
  mma_ts_w(d_tmem, a_tmem, dv, idesc, acc ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < WideCfg<D>::kBN / 16; ++kk)
    mma_ts_wc<1>(d_tmem, a_tmem + kk * 8,
                 dv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc);
}

// SPLIT: the grid's z index also carries a K/V range (split-KV); the CTA
// then processes that range of its tile's blocks and leaves fp32 partials
// for fa_merge_kernel<D, 128>.
template <int D, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(kWideThreads, WideCfg<D>::kCtasPerSm)
    fa_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmO,
                       const __grid_constant__ FwdParams p) {
  using W = WideCfg<D>;
  constexpr int BN = W::kBN;
  constexpr int NK = W::kKStages;
  constexpr int NV = W::kVStages;
  constexpr uint32_t kAll = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (batch b, query head hq, 128-row tile) ----
  int tile = CAUSAL ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                    : static_cast<int>(blockIdx.x);
  int hq = blockIdx.y;
  const int splits = SPLIT ? p.kv_splits : 1;
  int b = SPLIT ? static_cast<int>(blockIdx.z) / splits
                : static_cast<int>(blockIdx.z);
  const int split = SPLIT ? static_cast<int>(blockIdx.z) - b * splits : 0;
  if constexpr (CAUSAL && !SPLIT)
    causal_grid_item(p, 4ll * p.Nkv * D, tile, hq, b);   // head groups
  const int hk = hq / (p.Hq / p.Hkv);
  const int row0 = tile * kBM;
  const int kv_end = CAUSAL ? min(p.Nkv, row0 + kBM) : p.Nkv;
  const int nblk_tile = (kv_end + BN - 1) / BN;
  // This CTA's contiguous range [j0, j0 + nblk) of the tile's K/V blocks
  // (all of them without split-KV; possibly none for a short causal tile).
  const int chunk = SPLIT ? (nblk_tile + splits - 1) / splits : nblk_tile;
  const int j0 = SPLIT ? min(nblk_tile, split * chunk) : 0;
  const int nblk = SPLIT ? min(nblk_tile, j0 + chunk) - j0 : nblk_tile;

  // ---- shared memory (1024-byte aligned for the swizzle atoms) ----
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sQ = base;
  const uint32_t sK = sQ + W::kQBytes;
  const uint32_t sV = sK + NK * W::kKVBytes;
  const uint32_t sBar = sV + NV * W::kKVBytes;
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  const uint32_t bQFull = bar(0);
  auto bKFull = [&](int s) { return bar(1 + s); };
  auto bKEmpty = [&](int s) { return bar(1 + NK + s); };
  auto bVFull = [&](int s) { return bar(1 + 2 * NK + s); };
  auto bVEmpty = [&](int s) { return bar(1 + 2 * NK + NV + s); };
  constexpr int kB0 = 1 + 2 * NK + 2 * NV;
  auto bSFull = [&](int u) { return bar(kB0 + u); };
  auto bPFull = [&](int u) { return bar(kB0 + 2 + u); };
  const uint32_t bPVDone = bar(kB0 + 4);
  const uint32_t bOFinal = bar(kB0 + 5);
  const uint32_t bDrain = bar(kB0 + 6);
  uint8_t* const misc = base_ptr + (sBar - base) + 8 * W::kNumBars;
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
    for (int u = 0; u < 2; ++u) {
      mbar_init(bSFull(u), 1);
      mbar_init(bPFull(u), 4);
    }
    mbar_init(bPVDone, 1);
    mbar_init(bOFinal, 1);
    mbar_init(bDrain, 1);
    wstate->abort = 0u;
    wstate->status = p.status;
    wstate->limit_ns = p.wait_limit_ns;
    mbar_init_fence();
  }
  if (warp == kWideMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), W::kTmemAlloc);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{smem_addr(wstate)};

  if (warp == kWideLoadWarp) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      const int zq = b * p.Hq + hq;
      const int zk = b * p.Hkv + hk;
      mbar_arrive_expect_tx(bQFull, W::kQBytes);
      for (int c = 0; c < W::kBoxes; ++c)
        tma_load_3d(sQ + c * W::kQBoxBytes, &tmQ, bQFull, c * kBoxCols, row0,
                    zq, once);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int sk = j % NK, sv = j % NV;
        if (!mbar_wait(bKEmpty(sk), ((j / NK) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bKFull(sk), W::kKVBytes);
        for (int c = 0; c < W::kBoxes; ++c)
          tma_load_3d(sK + sk * W::kKVBytes + c * W::kKVBoxBytes, &tmK,
                      bKFull(sk), c * kBoxCols, (j0 + j) * BN, zk, keep);
        k_issued = j + 1;
        if (!mbar_wait(bVEmpty(sv), ((j / NV) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bVFull(sv), W::kKVBytes);
        for (int c = 0; c < W::kBoxes; ++c)
          tma_load_3d(sV + sv * W::kKVBytes + c * W::kKVBoxBytes, &tmV,
                      bVFull(sv), c * kBoxCols, (j0 + j) * BN, zk, keep);
        v_issued = j + 1;
      }
      // Never leave the CTA with copies in flight.
      for (int j = (k_issued > NK ? k_issued - NK : 0); j < k_issued; ++j)
        mbar_wait(bKFull(j % NK), (j / NK) & 1, wc, false);
      for (int j = (v_issued > NV ? v_issued - NV : 0); j < v_issued; ++j)
        mbar_wait(bVFull(j % NV), (j / NV) & 1, wc, false);
      mbar_wait(bQFull, 0, wc, false);
    }
  } else if (warp == kWideMmaWarp) {
    // ============================ MMA issuer ==============================
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = sdesc_sw128(sV, W::kKVBoxBytes, 1024);
    constexpr uint64_t kKVStep = static_cast<uint64_t>(W::kKVBytes >> 4);
    bool ok = __all_sync(kAll, mbar_wait(bQFull, 0, wc));
    // S(j) for j = 0, then per step: S(j+1), PV(j).
    for (int j = -1; ok && j < nblk; ++j) {
      const int jn = j + 1;                     // block of the next S
      if (jn < nblk) {
        const int s = jn % NK;
        if (!(ok = __all_sync(kAll, mbar_wait(bKFull(s), (jn / NK) & 1, wc))))
          break;
        wide_issue_qk<D>(tmem + static_cast<uint32_t>((jn & 1) * BN), dQ,
                         dK + static_cast<uint64_t>(s) * kKVStep, W::kIdescS);
        mma_commit_w(bSFull(jn & 1));
        mma_commit_w(bKEmpty(s));
      }
      if (j >= 0) {
        const int sv = j % NV;
        if (!(ok = __all_sync(kAll, mbar_wait(bVFull(sv), (j / NV) & 1, wc))))
          break;
        if (!(ok = __all_sync(kAll,
                              mbar_wait(bPFull(j & 1), (j >> 1) & 1, wc))))
          break;
        tc_fence_after();
        wide_issue_pv<D>(tmem + W::kColO,
                      tmem + static_cast<uint32_t>((j & 1) * BN),
                      dV + static_cast<uint64_t>(sv) * kKVStep, W::kIdescPV,
                      j > 0);
        mma_commit_w(bPVDone);
        mma_commit_w(bVEmpty(sv));
      }
    }
    mma_commit_w(bOFinal);
    mma_commit_w(bDrain);
    mbar_wait(bDrain, 0, wc, false);
  } else {
    // ============================ softmax warps ===========================
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    const bool neg_scale = c < 0.f;
    const int q_abs = row0 + (warp & 3) * 32 + lane;
    float m_ref = -INFINITY;   // reference max (log2 domain) of p and l
    float l_run = 0.f;         // sum of exp2(s*c - m_ref) over seen keys
    float w_run = 0.f;         // the same sum of the bf16-rounded values
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int u = j & 1;                      // S buffer of block j
      if (!(ok = __all_sync(kAll, mbar_wait(bSFull(u), (j >> 1) & 1, wc))))
        break;
      tc_fence_after();
      uint32_t sr[BN];
      const uint32_t s_addr =
          tmem + lane_off + static_cast<uint32_t>(u * BN);
      const int col0 = (j0 + j) * BN;
      const bool need_mask =
          (col0 + BN > p.Nkv) || (CAUSAL && col0 + BN - 1 > row0);
      float red[BN / 32];
      if (!need_mask && !neg_scale) {
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc)
          tmem_ld32_max(s_addr + cc * 32, sr + cc * 32, red[cc]);
      } else if (!need_mask) {
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc)
          tmem_ld32_min(s_addr + cc * 32, sr + cc * 32, red[cc]);
      } else {
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc) {
          tmem_ld32(s_addr + cc * 32, sr + cc * 32);
          red[cc] = 0.f;
        }
      }
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < BN / 32; ++cc) {
        reg_fence32(sr + cc * 32);
        reg_fence_f(red[cc]);
      }
#define S_(i) __uint_as_float(sr[(i)])
      // ---- row extreme over the visible keys of this block ----
      int n_vis = BN;
      if (need_mask) {
        int lim = p.Nkv - col0;
        if (CAUSAL) lim = min(lim, q_abs - col0 + 1);
        n_vis = max(0, min(BN, lim));
      }
      float ext;
      if (!need_mask) {
        ext = red[0];
#pragma unroll
        for (int cc = 1; cc < BN / 32; ++cc)
          ext = neg_scale ? fminf(ext, red[cc]) : fmaxf(ext, red[cc]);
      } else {
        // four independent chains of three-input extremes over the visible
        // keys (the others take the identity)
        const float idn = neg_scale ? INFINITY : -INFINITY;
        float e4[4] = {idn, idn, idn, idn};
#pragma unroll
        for (int i = 0; i < BN; i += 2) {
          const float v0 = (i < n_vis) ? S_(i) : idn;
          const float v1 = (i + 1 < n_vis) ? S_(i + 1) : idn;
          float& e = e4[(i >> 1) & 3];
          e = neg_scale ? fmin3(e, v0, v1) : fmax3(e, v0, v1);
        }
        ext = neg_scale ? fminf(fminf(e4[0], e4[1]), fminf(e4[2], e4[3]))
                        : fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]));
      }
      const float m_blk = (n_vis > 0) ? ext * c : -INFINITY;
      const bool move = m_blk > m_ref + kRescaleLog2 ||
                        (m_ref == -INFINITY && m_blk != -INFINITY);
      const float m_new = move ? m_blk : m_ref;
      const float alpha =
          (move && m_ref != -INFINITY) ? ex2_approx(m_ref - m_new) : 1.f;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;

      // the divisor of O also takes the rounding of this block's largest
      // weight (see top_rounding)
      w_run = w_run * alpha + (n_vis > 0 ? top_rounding(ext, c, m_use) : 0.f);

      // ---- P = exp2(s * c - m), packed to bf16, row sums ----
      uint32_t pp[BN / 2];
      const float rsum =
          need_mask ? exp_pack_row<BN, true>(sr, c, m_use, n_vis, pp)
                    : exp_pack_row<BN, false>(sr, c, m_use, BN, pp);
#undef S_
      l_run = l_run * alpha + rsum;
      w_run += rsum;
      m_ref = m_new;
      tmem_st32(tmem + lane_off + static_cast<uint32_t>(u * BN), pp);

      // ---- rescale O when the reference max moved.  PV(j-1) may still be
      // running (S(j) was issued before it), so wait for it first. ----
      if (j >= 1 && __any_sync(kAll, alpha != 1.f)) {
        if (!(ok = __all_sync(kAll,
                              mbar_wait(bPVDone, (j - 1) & 1, wc))))
          break;
        tc_fence_after();
        const uint32_t o_addr = tmem + lane_off + W::kColO;
#pragma unroll 1
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
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bPFull(u));
    }

    // ---- epilogue ----
    // The merge of split-KV partials may be scheduled from here on; it
    // waits for this whole grid before it reads them.
    if constexpr (SPLIT) grid_dep_launch();
    if (ok && nblk > 0) ok = __all_sync(kAll, mbar_wait(bOFinal, 0, wc));
    const int trow = (warp & 3) * 32 + lane;         // row within the tile
    const uint32_t o_addr = tmem + lane_off + W::kColO;
    if constexpr (SPLIT) {
      // Partial of one K/V range: unnormalised O (relative to m_ref), m and
      // l per row.  An empty range leaves m = -inf, l = 0.
      float* slot = p.work + ((static_cast<int64_t>(b) * p.Hq + hq) *
                                  static_cast<int64_t>(gridDim.x) +
                              tile) * splits * W::kSlotFloats +
                    static_cast<int64_t>(split) * W::kSlotFloats;
      if (ok && nblk > 0) {
        tc_fence_after();
        float4* orow = reinterpret_cast<float4*>(slot + trow * D);
#pragma unroll 1
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
      slot[kBM * D + trow] = nblk > 0 ? m_ref : -INFINITY;
      slot[kBM * D + kBM + trow] = nblk > 0 ? l_run : 0.f;
      slot[kBM * D + 2 * kBM + trow] = nblk > 0 ? w_run : 0.f;
    } else if (ok && nblk > 0) {
      tc_fence_after();
      const size_t row_idx =
          (static_cast<size_t>(b) * p.Hq + hq) * static_cast<size_t>(p.Nq) +
          static_cast<size_t>(q_abs);
      // Every MMA is complete and every K tile consumed: the K ring stages
      // the four warps' rows for TMA stores.
      const OutRows out{sK + static_cast<uint32_t>(warp & 3) * (32u * D * 2u),
                        &tmO, q_abs - lane, b * p.Hq + hq, p.Nq};
      store_final_row<D>(o_addr, m_ref, l_run, w_run, p.o + row_idx * D,
                         p.lse != nullptr ? p.lse + row_idx : nullptr,
                         q_abs < p.Nq, out);
    }
  }

  // ---- teardown: every role is done with TMEM and shared memory ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWideMmaWarp) tmem_dealloc(tmem, W::kTmemAlloc);
}

}  // namespace fa
