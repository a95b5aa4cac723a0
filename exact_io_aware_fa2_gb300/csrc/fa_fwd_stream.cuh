// fa_fwd_stream.cuh — the two-tile forward of fa_fwd_kernel.cuh with every
// SM given an equal share of the work ("stream" schedule), for shapes
// without a causal mask whose tile pairs do not fill whole waves of SMs.
//
// Same method and per-block arithmetic as fa_fwd_kernel.cuh (softmax_block,
// the same warp roles, TMEM columns and shared-memory rings).  Only the
// assignment of work differs.  With one pair of 128-row query tiles per CTA,
// P pairs on S SMs take ceil(P / S) pair-lengths of time, and every SM past
// P mod S idles for the last one (at 128 pairs on 152 SMs, 24 SMs idle the
// whole time).  Here the units are (pair, K/V block) items, numbered pair by
// pair (pair g = (batch, head, pair index), g-major), and CTA c takes the
// contiguous range [c L, (c + 1) L) of them.  A range covers the end of one
// pair, then whole pairs, then the start of another; each covered part of a
// pair is a "segment" of this CTA.
//
// A pair cut by range boundaries is completed by the CTA holding its last
// block (the "merger"); the CTAs holding its earlier blocks ("writers")
// each leave an fp32 partial: O unnormalised relative to their reference
// max m, with m and the row sum l.  The merger combines them with its own
// accumulator the way the online softmax combines two key ranges
// (M = max m_k, l = sum l_k 2^(m_k - M), O = sum O_k 2^(m_k - M) / l), in
// its epilogue, so no merge pass over HBM follows.  The pages describe this
// combination for split key ranges (FlashDecoding-style partition, "flash
// attention v3 paper" search page, second snippet); the even split of all
// work over the SMs is this library's schedule.
//
// Ordering: a CTA runs its segments from its last pair down to its first,
// so its writer segment (if any) comes first and its merger segment (if
// any) last, and a merger depends only on CTAs with lower grid indices,
// whose writer segments ran at their start.  The grid is launched
// cooperatively (at most one CTA per SM), so every CTA is resident from the
// start and every writer a merger waits for is running, whatever order the
// hardware starts CTAs in and whatever else shares the GPU.  Every wait is
// bounded and reports FA_ERR_TIMEOUT if it runs out.  A writer publishes its
// partial per softmax warp with a fence and a release store of the launch's
// epoch to a flag, once the next segment's first scores exist (its stores
// have drained by then); the merger's warp waits (bounded, acquire) for that
// value and clears the flag after reading, so a replay of the same launch
// (same epoch) waits again.  Partials are laid out column-chunk-major
// ([D/4][256 rows] float4) so a warp's 32 rows store and load as contiguous
// 512-byte runs.  In a CTA's last segment the finished rows are staged in
// the idle K ring and written by TMA stores, as in the plain kernel.
//
// Between segments the MMA warp releases Q (q_empty) once the segment's
// last S is issued, and waits for the epilogue to have read O (o_empty)
// before the next segment's first P*V overwrites it; the K/V rings run on
// across segments.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

enum SegKind : int { kSegWhole = 0, kSegWriter = 1, kSegMerger = 2 };

struct StreamSeg {
  int b, hq, pair;   // the tile pair
  int j0, n;         // its K/V blocks [j0, j0 + n) in this segment
  int first;         // block processed first; then first + 1, ... wrapping
                     // from j0 + n - 1 to j0
  int kind;          // SegKind
  int first_cta;     // CTA holding the pair's first block
};

// Segments of this CTA's range: [start, end) of the g-major item sequence.
// The host runs this schedule only for fewer than 2^31 items, so item
// indices and every quotient below fit 32-bit integers (whose divisions
// cost a fraction of 64-bit ones, on the path between segments).
struct StreamRange {
  int start, end;
  int n_seg;
};

__device__ __forceinline__ StreamRange stream_range(const FwdParams& p,
                                                    int n_pairs, int nbp,
                                                    int cta) {
  const int total = p.B * p.Hq * n_pairs * nbp;
  StreamRange r;
  r.start = cta * p.stream_len;
  r.end = min(r.start + p.stream_len, total);
  r.n_seg = r.start < r.end ? (r.end - 1) / nbp - r.start / nbp + 1 : 0;
  return r;
}

// Segment si (0 = the range's last pair, counting down).
//
// Block order within a segment: its blocks [j0, j0 + n) in order.  (Rotating
// each segment so that step t of every CTA visits block t mod nbp, as the
// one-pair-per-CTA grid does, was measured on GB300: the same time per
// block and per launch, but when the call's K/V exceed what L2 keeps it
// reads them about twice from DRAM, since a CTA whose run covers more than
// one pair's blocks meets the same block again a whole pair later: 218 MB
// against 138 MB read per launch for 25 heads of 2048 x 8192 at D 128,
// where Q, K and V are 118 MB.)
__device__ __forceinline__ StreamSeg stream_segment(const FwdParams& p,
                                                    const StreamRange& r,
                                                    int n_pairs, int nbp,
                                                    int si) {
  const unsigned unbp = static_cast<unsigned>(nbp);
  const int g = static_cast<int>(static_cast<unsigned>(r.end - 1) / unbp) -
                si;
  const int s = max(r.start, g * nbp) - g * nbp;
  const int e = min(r.end, (g + 1) * nbp) - g * nbp;
  StreamSeg sg;
  sg.j0 = s;
  sg.n = e - s;
  sg.first = s;
  sg.kind = e < nbp ? kSegWriter : (s > 0 ? kSegMerger : kSegWhole);
  sg.first_cta = static_cast<int>(static_cast<unsigned>(g * nbp) /
                                  static_cast<unsigned>(p.stream_len));
  const unsigned bh = static_cast<unsigned>(g) / static_cast<unsigned>(n_pairs);
  sg.pair = g - static_cast<int>(bh) * n_pairs;
  sg.b = static_cast<int>(bh / static_cast<unsigned>(p.Hq));
  sg.hq = static_cast<int>(bh) - sg.b * p.Hq;
  return sg;
}

// Scratch of a stream launch of G CTAs: G partial slots of
// stream_slot_floats() floats each (O as [D/4][256] float4, then m[256],
// l[256] (exact row sums) and w[256] (row sums of the bf16 weights)), then
// G * 8 64-bit flags (one per softmax warp of each CTA).
template <int D>
__host__ __device__ constexpr int64_t stream_slot_floats() {
  return static_cast<int64_t>(kTilesPerCta * kBM) * (D + 3);
}
constexpr int kStreamFlagsPerCta = 8;
template <int D>
__host__ __device__ constexpr int64_t stream_workspace_bytes(int64_t ctas) {
  return ctas * stream_slot_floats<D>() * 4 + ctas * kStreamFlagsPerCta * 8;
}

__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}
__device__ __forceinline__ float ld_l1(const float* ptr) { return *ptr; }
__device__ __forceinline__ float4 ld_l1(const float4* ptr) { return *ptr; }

// Publish this warp's stored partial: every lane's stores are ordered
// before the flag (fence, warp barrier, release by lane 0).
__device__ __forceinline__ void publish_partial(uint64_t* flag, uint64_t epoch,
                                                int lane) {
  __threadfence();
  __syncwarp();
  if (lane == 0) flag_release(flag, epoch);
}

// The merger's last step for one row: combine its own accumulator (TMEM at
// o_addr, reference max m_own, sums l_own and w_own) with the partials of
// CTAs k0 .. k1-1 for the same row (prow within the pair), then store the
// row (see OutRows) and its LSE as store_final_row does: O over the combined
// bf16-weight sum, the LSE from the combined exact sum.
template <int D>
__device__ __forceinline__ void merge_final_row(
    uint32_t o_addr, float m_own, float l_own, float w_own, const float* work,
    int k0, int k1, int prow, __nv_bfloat16* orow, float* lse_at,
    bool in_range, const OutRows& out) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  constexpr int64_t kSlot = stream_slot_floats<D>();
  constexpr int kRows = kTilesPerCta * kBM;
  // Start every load this row needs at once (into L1), so the loop below
  // waits for one L2 round trip rather than one per step.  Each CTA reads a
  // partial only after acquiring its flag, and no SM has read it before in
  // this launch.
  for (int k = k0; k < k1; ++k) {
    const float* slot = work + k * kSlot;
    prefetch_l1(slot + D * kRows + prow);
    prefetch_l1(slot + D * kRows + kRows + prow);
    prefetch_l1(slot + D * kRows + 2 * kRows + prow);
#pragma unroll
    for (int c4 = 0; c4 < D / 4; ++c4)
      prefetch_l1(reinterpret_cast<const float4*>(slot) + c4 * kRows + prow);
  }
  float M = m_own;
  for (int k = k0; k < k1; ++k)
    M = fmaxf(M, ld_l1(work + k * kSlot + D * kRows + prow));
  const float f_own = (m_own == -INFINITY) ? 0.f : ex2_approx(m_own - M);
  float l = l_own * f_own, wsum = w_own * f_own;
  for (int k = k0; k < k1; ++k) {
    const float* slot = work + k * kSlot;
    const float mk = ld_l1(slot + D * kRows + prow);
    if (mk != -INFINITY) {
      const float fk = ex2_approx(mk - M);
      l += ld_l1(slot + D * kRows + kRows + prow) * fk;
      wsum += ld_l1(slot + D * kRows + 2 * kRows + prow) * fk;
    }
  }
  const float inv_l = (wsum > 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t orr[32];
    tmem_ld32(o_addr + cc * 32, orr);
    tmem_ld_wait();
    reg_fence32(orr);
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(orr[i]) * f_own;
    for (int k = k0; k < k1; ++k) {
      const float* slot = work + k * kSlot;
      const float mk = ld_l1(slot + D * kRows + prow);
      const float wk = (mk == -INFINITY) ? 0.f : ex2_approx(mk - M);
      const float4* so = reinterpret_cast<const float4*>(slot);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = ld_l1(so + (cc * 8 + i) * kRows + prow);
        acc[4 * i] += wk * v.x;
        acc[4 * i + 1] += wk * v.y;
        acc[4 * i + 2] += wk * v.z;
        acc[4 * i + 3] += wk * v.w;
      }
    }
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = pack_bf16x2(acc[2 * i] * inv_l, acc[2 * i + 1] * inv_l);
    put_row_chunk<D>(out, lane, cc, packed, orow, in_range);
  }
  flush_rows<D>(out, lane);
  if (in_range && lse_at != nullptr) {
    const float lse2 = (l > 0.f) ? (M + log2f(l)) : -INFINITY;
    *lse_at = lse2 * 0.69314718055994530942f;
  }
}

template <int D, bool QK8>
struct StreamCfg {
  using C = FwdCfg<D, QK8>;
  // the two-tile kernel's barriers (its Q of tile B unused) plus q_empty
  // and o_empty
  static constexpr int kNumBars = C::kNumBars + 2;
  static constexpr int kSmemBytes = C::kSmemBytes + 16;
};

template <int D, bool QK8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_stream_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmO,
                         const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, QK8>;
  using SC = StreamCfg<D, QK8>;
  constexpr int NK = C::kKStages;
  constexpr int NV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int n_pairs = (p.Nq + 2 * kBM - 1) / (2 * kBM);
  const int nbp = (p.Nkv + kBN - 1) / kBN;          // K/V blocks per pair

  // This CTA's index and range of items sit in shared memory and are read
  // where used, which keeps them out of the registers of the block loops.
  __shared__ StreamRange range_s;
  __shared__ int cta_s;
  if (threadIdx.x == 0) {
    cta_s = static_cast<int>(blockIdx.x);
    range_s = stream_range(p, n_pairs, nbp, static_cast<int>(blockIdx.x));
  }
  __syncthreads();
  auto cta_index = [&]() -> int { return *static_cast<volatile int*>(&cta_s); };
  auto range = [&]() {
    const volatile StreamRange& r = range_s;
    return StreamRange{r.start, r.end, r.n_seg};
  };
  auto n_seg = [&]() -> int {
    return *static_cast<volatile int*>(&range_s.n_seg);
  };

  // ---- shared memory carve-up (as the two-tile kernel, two more barriers)
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sQ = base;
  const uint32_t sK = sQ + kTilesPerCta * C::kQKTileBytes;
  const uint32_t sV = sK + NK * C::kQKTileBytes;
  const uint32_t sBar = sV + NV * C::kTileBytes;
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  const uint32_t bQFull = bar(0);
  constexpr int kB0 = 1 + 2 * NK + 2 * NV;
  auto bKFull = [&](int s) { return bar(1 + s); };
  auto bKEmpty = [&](int s) { return bar(1 + NK + s); };
  auto bVFull = [&](int s) { return bar(1 + 2 * NK + s); };
  auto bVEmpty = [&](int s) { return bar(1 + 2 * NK + NV + s); };
  auto bSFull = [&](int x) { return bar(kB0 + x); };
  auto bPFull = [&](int x) { return bar(kB0 + 2 + x); };
  const uint32_t bOFinal = bar(kB0 + 4);
  const uint32_t bDrain = bar(kB0 + 5);
  const uint32_t bQEmpty = bar(kB0 + 6);
  const uint32_t bOEmpty = bar(kB0 + 7);
  // first half of tile x's P stored (see softmax_block)
  auto bPHalf = [&](int x) { return bar(kB0 + 8 + x); };
  static_assert(kB0 + 10 <= SC::kNumBars, "barrier count");
  uint8_t* const misc = base_ptr + (sBar - base) + 8 * SC::kNumBars;
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
    mbar_init(bQEmpty, 1);
    mbar_init(bOEmpty, 2 * 4);
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
      // r: this CTA's K/V blocks over all segments (ring position); the
      // stage and phase of each ring advance step by step
      int r = 0, k_issued = 0, v_issued = 0, q_loads = 0;
      int sk = 0, kph = 0, sv = 0, vph = 0;
      bool ok = true;
      for (int si = 0; ok && si < n_seg(); ++si) {
        const StreamSeg sg = stream_segment(p, range(), n_pairs, nbp, si);
        const int row0 = sg.pair * (2 * kBM);
        const bool has_b = row0 + kBM < p.Nq;
        const int zq = sg.b * p.Hq + sg.hq;
        const int zk = sg.b * p.Hkv + sg.hq / (p.Hq / p.Hkv);
        // Q of this segment once the MMAs no longer read the previous one
        if (si > 0 && !(ok = mbar_wait(bQEmpty, (si - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(bQFull, C::kQKTileBytes * (has_b ? 2 : 1));
        for (int x = 0; x < (has_b ? 2 : 1); ++x)
          for (int c = 0; c < C::kQKBoxes; ++c)
            tma_load_3d(sQ + x * C::kQKTileBytes + c * kBoxBytes, &tmQ,
                        bQFull, c * C::kQKBoxCols, row0 + x * kBM, zq, once);
        q_loads = si + 1;
        // The next segment's Q goes to L2 now: it loads into the one Q
        // buffer only once this segment's last S is issued, and the next
        // segment's first S waits for it.
        if (si + 1 < n_seg()) {
          const StreamSeg sn = stream_segment(p, range(), n_pairs, nbp, si + 1);
          const int row0n = sn.pair * (2 * kBM);
          const int zqn = sn.b * p.Hq + sn.hq;
          for (int x = 0; x < (row0n + kBM < p.Nq ? 2 : 1); ++x)
            for (int c = 0; c < C::kQKBoxes; ++c)
              tma_prefetch_l2_3d(&tmQ, c * C::kQKBoxCols, row0n + x * kBM, zqn);
        }
        int j = sg.first;                        // block index in the pair
        for (int i = 0; i < sg.n; ++i, ++r, j = (j + 1 == sg.j0 + sg.n)
                                                    ? sg.j0 : j + 1) {
          if (!(ok = mbar_wait(bKEmpty(sk), kph ^ 1, wc))) break;
          mbar_arrive_expect_tx(bKFull(sk), C::kQKTileBytes);
          for (int c = 0; c < C::kQKBoxes; ++c)
            tma_load_3d(sK + sk * C::kQKTileBytes + c * kBoxBytes, &tmK,
                        bKFull(sk), c * C::kQKBoxCols, j * kBN, zk, keep);
          k_issued = r + 1;
          if (!(ok = mbar_wait(bVEmpty(sv), vph ^ 1, wc))) break;
          mbar_arrive_expect_tx(bVFull(sv), C::kTileBytes);
          for (int c = 0; c < C::kBoxes; ++c)
            tma_load_3d(sV + sv * C::kTileBytes + c * kBoxBytes, &tmV,
                        bVFull(sv), c * kBoxCols, j * kBN, zk, keep);
          v_issued = r + 1;
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
      // last load issued into each stage of each ring, and for Q.
      for (int j = (k_issued > NK ? k_issued - NK : 0); j < k_issued; ++j)
        mbar_wait(bKFull(j % NK), (j / NK) & 1, wc, false);
      for (int j = (v_issued > NV ? v_issued - NV : 0); j < v_issued; ++j)
        mbar_wait(bVFull(j % NV), (j / NV) & 1, wc, false);
      if (q_loads > 0) mbar_wait(bQFull, (q_loads - 1) & 1, wc, false);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ==============================
    // Whole warp, converged, warp-uniform values; one elected lane issues.
    constexpr uint32_t kAll = 0xffffffffu;
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = sdesc_sw128(sV, kBoxBytes, 1024);
    constexpr uint64_t kStep = static_cast<uint64_t>(C::kTileBytes >> 4);
    constexpr uint64_t kQKStep = static_cast<uint64_t>(C::kQKTileBytes >> 4);
    bool ok = true;
    // Ring stages and phases run on across segments; they are advanced
    // step by step (no divisions in the issue loop).
    int ks = 0, kph = 0;      // stage and phase of the next K block
    int vs = 0, vph = 0;      // stage and phase of the next V block
    uint32_t pph = 0;         // bit x: phase of tile x's next P
    for (int si = 0; ok && si < n_seg(); ++si) {
      bool live_b;
      int n_blocks;
      {
        const StreamSeg sg = stream_segment(p, range(), n_pairs, nbp, si);
        live_b = sg.pair * (2 * kBM) + kBM < p.Nq;
        n_blocks = sg.n;
      }
      if (!(ok = __all_sync(kAll, mbar_wait(bQFull, si & 1, wc)))) break;
      for (int j = 0; ok && j <= n_blocks; ++j) {
        if (j >= 1 &&
            !(ok = __all_sync(kAll, mbar_wait(bVFull(vs), vph, wc))))
          break;
        if (j < n_blocks &&
            !(ok = __all_sync(kAll, mbar_wait(bKFull(ks), kph, wc))))
          break;
        // The first P*V of a later segment overwrites O: the previous
        // segment's epilogue must have read it.
        if (j == 1 && si > 0 &&
            !(ok = __all_sync(kAll, mbar_wait(bOEmpty, (si - 1) & 1, wc))))
          break;
        const uint64_t dKs = dK + static_cast<uint64_t>(ks) * kQKStep;
        const uint64_t dVs = dV + static_cast<uint64_t>(vs) * kStep;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (x == 1 && !live_b) continue;
          // O_x += P_x(j-1) V_{j-1}, each half of the keys once its half
          // of P is stored
          if (j >= 1) {
            if (!(ok = __all_sync(kAll, mbar_wait(bPHalf(x), (pph >> x) & 1u,
                                                  wc))))
              break;
            tc_fence_after();
            issue_pv_half<D, 0>(tmem + C::col_o(x), tmem + C::col_p(x), dVs,
                                C::kIdescPV, j > 1);
            if (!(ok = __all_sync(kAll, mbar_wait(bPFull(x), (pph >> x) & 1u,
                                                  wc))))
              break;
            pph ^= 1u << x;
            tc_fence_after();
            issue_pv_half<D, 1>(tmem + C::col_o(x), tmem + C::col_p(x), dVs,
                                C::kIdescPV, true);
          }
          // S_x(j) = Q_x K_j^T
          if (j < n_blocks) {
            issue_qk<D, QK8>(tmem + C::col_s(x),
                             dQ + static_cast<uint64_t>(x) * kQKStep, dKs,
                             C::kIdescS);
            mma_commit_w(bSFull(x));
          }
        }
        if (!ok) break;
        // Q of this segment is read by no later MMA: the next segment's Q
        // may load while this one's last softmax and P*V run.
        if (j == n_blocks - 1) mma_commit_w(bQEmpty);
        if (j < n_blocks) {
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
      }
      if (!ok) break;
      mma_commit_w(bOFinal);     // O of this segment: complete
    }
    mma_commit_w(bDrain);
    mbar_wait(bDrain, 0, wc, false);
  } else {
    // ============================ softmax warps ===========================
    const int role = warp - kSoftmaxWarp0;         // 0..7
    const int x = role >> 2;                       // tile A (0) or B (1)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_addr = tmem + lane_off + C::col_o(x);
    const float c = p.scale_log2;
    const bool neg_scale = c < 0.f;
    // row of this thread within a pair (the partial slots' row index)
    const int prow = x * kBM + (warp & 3) * 32 + lane;
    constexpr int64_t kSlot = stream_slot_floats<D>();
    // flag of this CTA's partial for this warp's rows, recomputed where
    // used (kept out of the softmax loop's registers)
    auto my_flag = [&]() {
      return reinterpret_cast<uint64_t*>(
                 p.work + static_cast<int64_t>(gridDim.x) * kSlot) +
             static_cast<int64_t>(cta_index()) * kStreamFlagsPerCta + role;
    };
    uint32_t sph = 0;          // phase of this tile's next S
    bool ok = true;
    bool publish = false;      // this warp's partial is stored, unpublished
    for (int si = 0; si < n_seg(); ++si) {
      // Only what the block loop needs stays live across it; the epilogue
      // recomputes the rest of the segment's description.
      int my_row0, nb, blk, blk_lo, blk_end;
      {
        const StreamSeg sg = stream_segment(p, range(), n_pairs, nbp, si);
        my_row0 = sg.pair * (2 * kBM) + x * kBM;
        nb = (x == 0 || my_row0 < p.Nq) ? sg.n : 0;
        blk = sg.first;                          // block index in the pair
        blk_lo = sg.j0;
        blk_end = sg.j0 + sg.n;
      }
      const int q_abs = my_row0 + (warp & 3) * 32 + lane;
      float m_ref = -INFINITY;
      float l_run = 0.f;
      float w_run = 0.f;
      if (publish) {
        // The previous segment's partial is stored: publish it once this
        // segment's first scores exist (Q load and S MMA later), when its
        // stores have drained and the fence before the flag is short.
        if (ok && nb > 0)
          ok = __all_sync(0xffffffffu, mbar_wait(bSFull(x), sph, wc));
        publish_partial(my_flag(), p.epoch, lane);
        publish = false;
      }
      for (int j = 0; ok && j < nb; ++j) {
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(bSFull(x), sph, wc))))
          break;
        sph ^= 1u;
        tc_fence_after();
        softmax_block<D, false, false, true>(
            tmem + lane_off + C::col_s(x), tmem + lane_off + C::col_p(x),
            o_addr, blk * kBN, my_row0, q_abs, p.Nkv, c, neg_scale, j >= 1,
            m_ref, l_run, w_run, bPHalf(x));
        __syncwarp();
        if (lane == 0) mbar_arrive(bPFull(x));
        blk = (blk + 1 == blk_end) ? blk_lo : blk + 1;
      }
      // Every softmax warp waits for the segment's end, also one whose tile
      // is absent from this pair: its o_empty arrival below must not run
      // ahead into a later segment's phase.
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bOFinal, si & 1, wc));
      if (ok && nb > 0) {
        tc_fence_after();
        const StreamSeg sg = stream_segment(p, range(), n_pairs, nbp, si);
        const size_t row_idx =
            (static_cast<size_t>(sg.b) * p.Hq + sg.hq) *
                static_cast<size_t>(p.Nq) +
            static_cast<size_t>(q_abs);
        __nv_bfloat16* const orow = p.o + row_idx * D;
        float* const lse_at = p.lse != nullptr ? p.lse + row_idx : nullptr;
        const bool in_range = q_abs < p.Nq;
        // In the CTA's last segment every MMA is complete and every K tile
        // consumed: the K ring stages the output rows for TMA stores.
        const OutRows out{
            si + 1 == n_seg() ? sK + static_cast<uint32_t>(role) * (32u * D * 2u)
                            : 0u,
            &tmO, my_row0 + (warp & 3) * 32, sg.b * p.Hq + sg.hq, p.Nq};
        if (sg.kind == kSegWhole) {
          store_final_row<D>(o_addr, m_ref, l_run, w_run, orow, lse_at,
                             in_range, out);
        } else if (sg.kind == kSegWriter) {
          float* const slot =
              p.work + static_cast<int64_t>(cta_index()) * kSlot;
          float4* const so = reinterpret_cast<float4*>(slot);
          constexpr int kRows = kTilesPerCta * kBM;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(o_addr + cc * 32, orr);
            tmem_ld_wait();
            reg_fence32(orr);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(so + (cc * 8 + i) * kRows + prow,
                     make_float4(__uint_as_float(orr[4 * i]),
                                 __uint_as_float(orr[4 * i + 1]),
                                 __uint_as_float(orr[4 * i + 2]),
                                 __uint_as_float(orr[4 * i + 3])));
          }
          __stcg(slot + D * kRows + prow, m_ref);
          __stcg(slot + D * kRows + kRows + prow, l_run);
          __stcg(slot + D * kRows + 2 * kRows + prow, w_run);
          // published during the next segment's first block, or below if
          // this is the CTA's last segment
          publish = si + 1 < n_seg();
          if (!publish) publish_partial(my_flag(), p.epoch, lane);
        } else {
          const int k1 = cta_index();
          uint64_t* const flags = my_flag() - static_cast<int64_t>(k1) *
                                                  kStreamFlagsPerCta;
          for (int k = sg.first_cta; ok && k < k1; ++k)
            ok = __all_sync(
                0xffffffffu,
                flag_wait(flags + static_cast<int64_t>(k) *
                                      kStreamFlagsPerCta,
                          p.epoch, wc));
          if (ok) {
            merge_final_row<D>(o_addr, m_ref, l_run, w_run, p.work,
                               sg.first_cta, k1, prow, orow, lse_at, in_range,
                               out);
            // Consumed: clear the flags so that a replay of this launch
            // waits for its own writers again.
            __syncwarp();
            if (lane == 0)
              for (int k = sg.first_cta; k < k1; ++k)
                flags[static_cast<int64_t>(k) * kStreamFlagsPerCta] = 0ull;
          }
        }
      }
      // O of this segment has been read: the next segment may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bOEmpty);
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
