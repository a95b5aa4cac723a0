// fa_fwd_persist.cuh — the two-tile forward of fa_fwd_kernel.cuh run by
// persistent CTAs: one CTA per SM, each walking a list of whole tile pairs.
//
// Same method and per-block arithmetic as fa_fwd_kernel.cuh (softmax_block,
// the warp roles, TMEM columns and shared-memory rings).  With a causal mask
// the pairs of a head differ in length (pair t visits 2t + 2 key blocks), and
// one CTA per pair leaves the GPU with many short CTAs, each paying its own
// start-up (barrier set-up, TMEM allocation, the first Q, K and V from
// memory) and epilogue.  Here the grid has at most one CTA per SM and every
// CTA processes a list of pairs:
//
//   * Order: all pairs of the call sorted longest first (pair index
//     descending, then (batch, head)); CTA c of G takes items c, 2G-1-c,
//     2G+c, 4G-1-c, ... (a "snake" deal), which evens out the total length
//     per CTA without a run-time queue.
//   * Between pairs nothing is torn down: the K/V rings and the barrier
//     phases run on.  Q has two buffers where shared memory allows (head dim
//     64): the next pair's Q loads while the current pair runs.  With one
//     buffer (head dim 128) the next pair's Q is prefetched into L2 when the
//     current pair starts, and loaded once the current pair's last S has
//     been issued.
//   * Each tile has its own "O final" and "O empty" barriers: the MMA warp
//     commits tile x's O final after its last P*V, the tile's softmax warps
//     then write its rows while the other tile is still finishing, and the
//     next pair's first P*V into tile x waits for tile x's O empty.  The next
//     pair's first S MMAs do not wait for any epilogue (at head dim 128 P
//     lives in S's columns, whose last reader is the last P*V; at head dim 64
//     P has its own columns).
//   * Tile A of a causal pair has one block fewer than tile B.  With two Q
//     buffers, the next pair's first S for tile A is issued as soon as
//     tile A's last P of the current pair is consumed, so tile A starts the
//     next pair while tile B finishes this one (measured: causal B4 H16
//     N2048 D64 55.3 -> 53.2 us).
//   * Masking: only a tile's last block can hold hidden keys (its causal
//     diagonal, or the end of the keys).  Their scores are overwritten in
//     TMEM (hide_keys) and every block runs the same unmasked block code;
//     the host sends calls with a zero scale, for which no score has weight
//     0, to the one-pair-per-CTA kernels.
//
// Source of the method: as fa_fwd_kernel.cuh ("Hacker News Digest —
// gpu-computing", section "Алгоритм Flash Attention 2", and the online
// softmax of section "v1 — базовая версия", item 3); the work split keeps
// the pages' unit (a thread block owns row blocks of O and walks their
// key/value blocks; "flash attention v3 paper" search page, third snippet)
// and only changes which SM runs which unit, and when.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

// Warps: warpgroup 0 holds the MMA warp, the TMA warp and two idle warps,
// warpgroups 1 and 2 the softmax of tiles A and B.  Warpgroup 0 gives up
// registers and the softmax warpgroups take them: launched at
// kPersistRegsLaunch per thread (384 threads, the most that fits), then
// 128 x kPersistRegsLow + 256 x kPersistRegsHigh, the same total.  (At
// head dim 64 this removed the softmax's spills: causal B4 H16 N2048 63.5 ->
// 61.3 us; the same split in the one-pair-per-CTA kernel measured 1.8%
// slower on the 4096 x 8192 shape and is not used there.)
// Give up / take registers for the rest of the calling warpgroup's code:
// every warp of the warpgroup executes the same call, and the registers the
// incs take must not exceed what the decs gave back (the block's launch
// allocation is fixed).
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

constexpr int kPersistThreads = 384;
constexpr int kPersistSoftmaxWarp0 = 4;
constexpr int kPersistRegsLaunch = 168;
constexpr int kPersistRegsLow = 104;
constexpr int kPersistRegsHigh = 200;
static_assert(128 * kPersistRegsLow + 256 * kPersistRegsHigh ==
                  kPersistThreads * kPersistRegsLaunch,
              "register split");
static_assert(kPersistRegsLaunch * kPersistThreads <= 65536, "launch");

template <int D, bool QK8>
struct PersistCfg {
  using C = FwdCfg<D, QK8>;
  // Q buffers: two at head dim 64 (the next pair's Q loads during the
  // current pair), one at 128 (shared memory is full).
  static constexpr int kQBufs = (D == 64) ? 2 : 1;
  // barriers: Q full/empty per buffer, K and V full/empty per stage, S full
  // and P full per tile, O final and O empty per tile, drain, first half of
  // P per tile
  static constexpr int kNumBars =
      2 * kQBufs + 2 * C::kKStages + 2 * C::kVStages + 2 + 2 + 2 + 2 + 1 + 2;
  static constexpr int kBarBytes = 8 * kNumBars + 32;
  static constexpr int kSmemBytes =
      1024 + C::kQKTileBytes * (kTilesPerCta * kQBufs + C::kKStages) +
      C::kTileBytes * C::kVStages + kBarBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// Item (pair of the sorted list) that CTA c of G handles in its round r, or
// -1 when that round has none for it.  The list has fewer than 2^31 items
// (the host launches this kernel only then), so 32-bit arithmetic suffices.
__device__ __forceinline__ int persist_item(int total, int G, int c, int r) {
  const int i = r * G + ((r & 1) ? G - 1 - c : c);
  return i < total ? i : -1;
}

// Rounds of CTA c: items r with persist_item(...) >= 0 for r = 0 .. n-1.
__device__ __forceinline__ int persist_rounds(int total, int G, int c) {
  const int full = total / G;
  const int rem = total - full * G;
  const int pos = (full & 1) ? G - 1 - c : c;
  return full + (pos < rem ? 1 : 0);
}

struct PersistItem {
  int b, hq, pair;
};

// Item i of the list: pairs longest first (for a causal mask the pair with
// the highest index is the longest), then (batch, head).  i = -1 (no item)
// gives a harmless value that no caller uses.
__device__ __forceinline__ PersistItem persist_decode(const FwdParams& p,
                                                      int n_pairs, int i) {
  const unsigned bh_count = static_cast<unsigned>(p.B * p.Hq);
  const unsigned ui = static_cast<unsigned>(max(i, 0));
  const unsigned rank = ui / bh_count;
  const unsigned bh = ui - rank * bh_count;
  PersistItem it;
  it.pair = n_pairs - 1 - static_cast<int>(rank);
  it.b = static_cast<int>(bh / static_cast<unsigned>(p.Hq));
  it.hq = static_cast<int>(bh) - it.b * p.Hq;
  return it;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kPersistThreads, 1)
    fa_fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmO,
                          const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, false>;
  using PC = PersistCfg<D, false>;
  constexpr int NK = C::kKStages;
  constexpr int NV = C::kVStages;
  constexpr int NQ = PC::kQBufs;
  constexpr uint32_t kAll = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int n_pairs = (p.Nq + 2 * kBM - 1) / (2 * kBM);
  const int total = p.B * p.Hq * n_pairs;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int rounds = persist_rounds(total, G, cta);

  // Rows and K/V block counts of round r's pair.
  struct Unit {
    PersistItem it;
    int row0[2];
    int nblk[2];
    int n_pair;
  };
  auto unit = [&](int r) {
    Unit u;
    u.it = persist_decode(p, n_pairs, persist_item(total, G, cta, r));
    u.row0[0] = u.it.pair * (2 * kBM);
    u.row0[1] = u.row0[0] + kBM;
    u.nblk[0] = kv_blocks<CAUSAL>(u.row0[0], p.Nkv);
    u.nblk[1] = u.row0[1] < p.Nq ? kv_blocks<CAUSAL>(u.row0[1], p.Nkv) : 0;
    u.n_pair = max(u.nblk[0], u.nblk[1]);
    return u;
  };

  // ---- shared memory carve-up (1024-byte aligned for the swizzle atoms) --
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sQ = base;                    // [NQ][tile A, tile B]
  const uint32_t sK = sQ + NQ * kTilesPerCta * C::kQKTileBytes;
  const uint32_t sV = sK + NK * C::kQKTileBytes;
  const uint32_t sBar = sV + NV * C::kTileBytes;
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  auto bQFull = [&](int q) { return bar(q); };
  auto bQEmpty = [&](int q) { return bar(NQ + q); };
  constexpr int kK0 = 2 * NQ;
  auto bKFull = [&](int s) { return bar(kK0 + s); };
  auto bKEmpty = [&](int s) { return bar(kK0 + NK + s); };
  auto bVFull = [&](int s) { return bar(kK0 + 2 * NK + s); };
  auto bVEmpty = [&](int s) { return bar(kK0 + 2 * NK + NV + s); };
  constexpr int kB0 = kK0 + 2 * NK + 2 * NV;
  auto bSFull = [&](int x) { return bar(kB0 + x); };
  auto bPFull = [&](int x) { return bar(kB0 + 2 + x); };
  auto bOFinal = [&](int x) { return bar(kB0 + 4 + x); };
  auto bOEmpty = [&](int x) { return bar(kB0 + 6 + x); };
  const uint32_t bDrain = bar(kB0 + 8);
  // first half of tile x's P stored (see softmax_block); P*V runs in two
  // halves at head dim 64 (C3 53.2 -> 52.8 us), at 128 whole (the halves
  // measured 0.8% slower on the causal GQA N 8192 shape)
  constexpr bool kSplitP = D == 64;
  auto bPHalf = [&](int x) { return bar(kB0 + 9 + x); };
  static_assert(kB0 + 11 == PC::kNumBars, "barrier count");
  uint8_t* const misc = base_ptr + (sBar - base) + 8 * PC::kNumBars;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  WaitState* const wstate = reinterpret_cast<WaitState*>(misc + 8);

  if (threadIdx.x == 0) {
    for (int q = 0; q < NQ; ++q) {
      mbar_init(bQFull(q), 1);
      mbar_init(bQEmpty(q), 1);
    }
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
      mbar_init(bOFinal(x), 1);
      mbar_init(bOEmpty(x), 4);
    }
    mbar_init(bDrain, 1);
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

  // Warpgroup 0 (TMA, MMA and two idle warps) gives registers back first;
  // the softmax warpgroups' incs wait until they are free.
  if (warp < kPersistSoftmaxWarp0) {
  regs_dec<kPersistRegsLow>();
  if (warp == kLoadWarp) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      int k_issued = 0, v_issued = 0, q_loads = 0;
      int sk = 0, kph = 0, sv = 0, vph = 0;
      bool ok = true;
      Unit nxt = unit(0);
      for (int r = 0; ok && r < rounds; ++r) {
        const Unit u = nxt;
        if (r + 1 < rounds) nxt = unit(r + 1);
        const int zq = u.it.b * p.Hq + u.it.hq;
        const int zk = u.it.b * p.Hkv + u.it.hq / (p.Hq / p.Hkv);
        const int qb = r % NQ;
        const bool has_b = u.row0[1] < p.Nq;
        // Q of this pair, once the MMAs of the pair that last used this
        // buffer no longer read it
        if (r >= NQ && !(ok = mbar_wait(bQEmpty(qb), ((r / NQ) - 1) & 1, wc)))
          break;
        mbar_arrive_expect_tx(bQFull(qb), C::kQKTileBytes * (has_b ? 2 : 1));
        for (int x = 0; x < (has_b ? 2 : 1); ++x)
          for (int c = 0; c < C::kQKBoxes; ++c)
            tma_load_3d(sQ + (qb * kTilesPerCta + x) * C::kQKTileBytes +
                            c * kBoxBytes,
                        &tmQ, bQFull(qb), c * C::kQKBoxCols, u.row0[x], zq,
                        once);
        q_loads = r + 1;
        // With one Q buffer, the next pair's Q goes to L2 now, so its load
        // after this pair's last S is short.
        if (NQ == 1 && r + 1 < rounds) {
          const int zqn = nxt.it.b * p.Hq + nxt.it.hq;
          for (int x = 0; x < (nxt.row0[1] < p.Nq ? 2 : 1); ++x)
            for (int c = 0; c < C::kQKBoxes; ++c)
              tma_prefetch_l2_3d(&tmQ, c * C::kQKBoxCols, nxt.row0[x], zqn);
        }
        for (int j = 0; j < u.n_pair; ++j) {
          if (!(ok = mbar_wait(bKEmpty(sk), kph ^ 1, wc))) break;
          mbar_arrive_expect_tx(bKFull(sk), C::kQKTileBytes);
          for (int c = 0; c < C::kQKBoxes; ++c)
            tma_load_3d(sK + sk * C::kQKTileBytes + c * kBoxBytes, &tmK,
                        bKFull(sk), c * C::kQKBoxCols, j * kBN, zk, keep);
          ++k_issued;
          if (!(ok = mbar_wait(bVEmpty(sv), vph ^ 1, wc))) break;
          mbar_arrive_expect_tx(bVFull(sv), C::kTileBytes);
          for (int c = 0; c < C::kBoxes; ++c)
            tma_load_3d(sV + sv * C::kTileBytes + c * kBoxBytes, &tmV,
                        bVFull(sv), c * kBoxCols, j * kBN, zk, keep);
          ++v_issued;
          if (++sk == NK) {
            sk = 0;
            kph ^= 1;
          }
          if (++sv == NV) {
            sv = 0;
            vph ^= 1;
          }
        }
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the
      // last load issued into each stage of each ring and each Q buffer.
      for (int j = (k_issued > NK ? k_issued - NK : 0); j < k_issued; ++j)
        mbar_wait(bKFull(j % NK), (j / NK) & 1, wc, false);
      for (int j = (v_issued > NV ? v_issued - NV : 0); j < v_issued; ++j)
        mbar_wait(bVFull(j % NV), (j / NV) & 1, wc, false);
      for (int r = (q_loads > NQ ? q_loads - NQ : 0); r < q_loads; ++r)
        mbar_wait(bQFull(r % NQ), (r / NQ) & 1, wc, false);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ==============================
    // The whole warp runs this loop, converged and with warp-uniform values;
    // one elected lane issues each MMA and commit.
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = sdesc_sw128(sV, kBoxBytes, 1024);
    constexpr uint64_t kStep = static_cast<uint64_t>(C::kTileBytes >> 4);
    constexpr uint64_t kQKStep = static_cast<uint64_t>(C::kQKTileBytes >> 4);
    bool ok = true;
    int ks = 0, kph = 0;      // stage and phase of the next K block
    int vs = 0, vph = 0;      // stage and phase of the next V block
    uint32_t pph = 0;         // bit x: phase of tile x's next P
    // The next round's pair is worked out while this round's last P's are
    // awaited, off the path from the last P to the next S.
    Unit nxt = unit(0);
    bool next_a_early = false;  // the next round's S_A(0) is already issued
    for (int r = 0; ok && r < rounds; ++r) {
      const Unit u = nxt;
      const bool a_early = next_a_early;
      next_a_early = false;
      const int qb = r % NQ;
      if (!(ok = __all_sync(kAll, mbar_wait(bQFull(qb), (r / NQ) & 1, wc))))
        break;
      const uint64_t dQb =
          dQ + static_cast<uint64_t>(qb * kTilesPerCta) * kQKStep;
      for (int j = 0; ok && j <= u.n_pair; ++j) {
        if (j >= 1 &&
            !(ok = __all_sync(kAll, mbar_wait(bVFull(vs), vph, wc))))
          break;
        if (j < u.n_pair &&
            !(ok = __all_sync(kAll, mbar_wait(bKFull(ks), kph, wc))))
          break;
        const uint64_t dKs = dK + static_cast<uint64_t>(ks) * kQKStep;
        const uint64_t dVs = dV + static_cast<uint64_t>(vs) * kStep;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          // O_x += P_x(j-1) V_{j-1}
          if (j >= 1 && j - 1 < u.nblk[x]) {
            // the first P*V of a later pair overwrites O_x: the previous
            // pair's epilogue of tile x must have read it
            if (j == 1 && r > 0 &&
                !(ok = __all_sync(kAll,
                                  mbar_wait(bOEmpty(x), (r - 1) & 1, wc))))
              break;
            if constexpr (kSplitP) {
              // each half of the keys once its half of P is stored
              if (!(ok = __all_sync(
                        kAll, mbar_wait(bPHalf(x), (pph >> x) & 1u, wc))))
                break;
              tc_fence_after();
              issue_pv_half<D, 0>(tmem + C::col_o(x), tmem + C::col_p(x),
                                  dVs, C::kIdescPV, j > 1);
            }
            if (!(ok = __all_sync(kAll, mbar_wait(bPFull(x), (pph >> x) & 1u,
                                                  wc))))
              break;
            pph ^= 1u << x;
            tc_fence_after();
            if constexpr (kSplitP)
              issue_pv_half<D, 1>(tmem + C::col_o(x), tmem + C::col_p(x),
                                  dVs, C::kIdescPV, true);
            else
              issue_pv<D>(tmem + C::col_o(x), tmem + C::col_p(x), dVs,
                          C::kIdescPV, j > 1);
            if (j == u.nblk[x]) mma_commit_w(bOFinal(x));  // O_x complete
          }
          // S_x(j) = Q_x K_j^T
          if (j < u.nblk[x] && !(x == 0 && j == 0 && a_early)) {
            issue_qk<D, false>(tmem + C::col_s(x),
                               dQb + static_cast<uint64_t>(x) * kQKStep, dKs,
                               C::kIdescS);
            mma_commit_w(bSFull(x));
          }
        }
        if (!ok) break;
        // Q of this pair is read by no later MMA
        if (j == u.n_pair - 1) {
          mma_commit_w(bQEmpty(qb));
          if (r + 1 < rounds) nxt = unit(r + 1);
        }
        if (j < u.n_pair) {
          mma_commit_w(bKEmpty(ks));
          if (++ks == NK) {
            ks = 0;
            kph ^= 1;
          }
        }
        if (j >= 1) {
          mma_commit_w(bVEmpty(vs));
          if (++vs == NV) {
            vs = 0;
            vph ^= 1;
          }
        }
        // Tile A has one block fewer than tile B: once its scores of this
        // pair are done, the next pair's first S for it (its Q in the other
        // buffer, its K the next stage) is issued here, so tile A's softmax
        // starts the next pair while tile B finishes this one.  Needs the
        // second Q buffer; every wait here is on loads whose buffers were
        // released before this iteration.
        if (NQ > 1 && j == u.n_pair - 1 && u.nblk[0] < u.n_pair &&
            r + 1 < rounds) {
          const int qn = (r + 1) % NQ;
          if (!(ok = __all_sync(kAll, mbar_wait(bQFull(qn), ((r + 1) / NQ) & 1,
                                                wc))))
            break;
          if (!(ok = __all_sync(kAll, mbar_wait(bKFull(ks), kph, wc)))) break;
          issue_qk<D, false>(
              tmem + C::col_s(0),
              dQ + static_cast<uint64_t>(qn * kTilesPerCta) * kQKStep,
              dK + static_cast<uint64_t>(ks) * kQKStep, C::kIdescS);
          mma_commit_w(bSFull(0));
          next_a_early = true;
        }
      }
      if (!ok) break;
      // a tile without blocks in this pair still gets its O final, so its
      // softmax warps pass the epilogue in step
      for (int x = 0; x < 2; ++x)
        if (u.nblk[x] == 0) mma_commit_w(bOFinal(x));
    }
    // Every MMA this warp issued completes before the CTA tears down.
    mma_commit_w(bDrain);
    mbar_wait(bDrain, 0, wc, false);
  }
  }  // warpgroup 0
  else {
    regs_inc<kPersistRegsHigh>();
    // ============================ softmax warps ===========================
    const int x = (warp - kPersistSoftmaxWarp0) >> 2;   // tile A (0) or B (1)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    const bool neg_scale = c < 0.f;
    uint32_t sph = 0;          // phase of this tile's next S
    bool ok = true;
    // This round's rows, block count and (batch, head); the next round's
    // are worked out while this round's last P*V runs.
    int nx_row0, nx_nb;
    PersistItem nx_it;
    auto next_unit = [&](int r) {
      const Unit u = unit(r);
      nx_row0 = x ? u.row0[1] : u.row0[0];
      nx_nb = x ? u.nblk[1] : u.nblk[0];
      nx_it = u.it;
    };
    next_unit(0);
    for (int r = 0; r < rounds; ++r) {
      const int my_row0 = nx_row0, nb = nx_nb;
      const PersistItem it = nx_it;
      const int q_abs = my_row0 + (warp & 3) * 32 + lane;
      float m_ref = -INFINITY;   // reference max (log2 domain) of p and l
      float l_run = 0.f;         // sum of exp2(s*c - m_ref) over seen keys
      float w_run = 0.f;         // the divisor of O (see top_rounding)
      const uint32_t s_at = tmem + lane_off + C::col_s(x);
      const uint32_t p_at = tmem + lane_off + C::col_p(x);
      const uint32_t o_at = tmem + lane_off + C::col_o(x);
      // Only a tile's last block can hold hidden keys (the causal diagonal,
      // or the end of the keys).  Their scores are overwritten in TMEM
      // (hide_keys, which needs the nonzero scale the host guarantees), so
      // every block runs the same unmasked code.
      for (int j = 0; ok && j < nb; ++j) {
        if (!(ok = __all_sync(kAll, mbar_wait(bSFull(x), sph, wc)))) break;
        sph ^= 1u;
        tc_fence_after();
        const int col0 = j * kBN;
        if (j + 1 == nb && (col0 + kBN > p.Nkv ||
                            (CAUSAL && col0 + kBN - 1 > my_row0))) {
          int lim = p.Nkv - col0;
          if (CAUSAL) lim = min(lim, q_abs - col0 + 1);
          hide_keys(s_at, max(0, min(kBN, lim)),
                    neg_scale ? INFINITY : -INFINITY);
        }
        softmax_block<D, CAUSAL, true, kSplitP>(s_at, p_at, o_at, col0, my_row0,
                                             q_abs, p.Nkv, c, neg_scale,
                                             j >= 1, m_ref, l_run, w_run,
                                             bPHalf(x));
        __syncwarp();
        if (lane == 0) mbar_arrive(bPFull(x));
      }
      if (r + 1 < rounds) next_unit(r + 1);
      // ---- epilogue of tile x: every warp of the tile waits for its O,
      // also when the tile is absent from this pair, so its O-empty
      // arrival stays in step with the MMA warp's rounds ----
      if (ok) ok = __all_sync(kAll, mbar_wait(bOFinal(x), r & 1, wc));
      if (ok && nb > 0) {
        tc_fence_after();
        const size_t row_idx =
            (static_cast<size_t>(it.b) * p.Hq + it.hq) *
                static_cast<size_t>(p.Nq) +
            static_cast<size_t>(q_abs);
        // rows leave by direct stores: the K ring may still feed the other
        // tile or the next pair
        const OutRows out{0u, &tmO, my_row0 + (warp & 3) * 32,
                          it.b * p.Hq + it.hq, p.Nq};
        store_final_row<D>(tmem + lane_off + C::col_o(x), m_ref, l_run, w_run,
                           p.o + row_idx * D,
                           p.lse != nullptr ? p.lse + row_idx : nullptr,
                           q_abs < p.Nq, out);
      }
      // O_x of this pair has been read: the next pair may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bOEmpty(x));
      if (!ok) break;
    }
  }

  // ---- teardown: every role is done with TMEM and shared memory ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
