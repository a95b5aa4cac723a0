// fa_fwd_kernel.cuh — exact attention forward on sm_103a (tcgen05 + TMA).
//
// Method: "Hacker News Digest — gpu-computing", section "Алгоритм Flash
// Attention 2" (loop over query tiles; for each key/value tile form
// S = Q K^T * scale, apply the online softmax in place, accumulate S @ V),
// with the running max / denominator of section "v1 — базовая версия",
// item 3, and the FA2 work split of the "flash attention v3 paper" search
// page, third snippet (one thread block owns one row block of O and walks
// all key/value blocks).  The division by the denominator is deferred to
// the epilogue (the same result as renormalising each tile, which the
// pages print).
//
// One CTA owns one 128-row query tile of one (batch, query head).  Warp
// roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t); reads S from
//              TMEM, masks, tracks the running max m and sum l (log2 domain,
//              scale folded into one FFMA), writes P = exp2(...) as bf16 into
//              TMEM, rescales the O accumulator in TMEM when m grows, and
//              finally writes O / l and LSE.
//   warp 4     TMA producer: Q once, then K_j and V_j into two rings of
//              NSTAGE shared-memory stages (128-byte swizzle).
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T (both operands in
//              shared memory, K-major) and O += P_j V_j (P from TMEM, V from
//              shared memory, MN-major), accumulators in TMEM.
//
// TMEM columns (512 allocated): S double buffer at 0 and 128, O at 256
// (D columns), P double buffer at 384 and 448 (64 columns of packed bf16x2
// each).  Nothing larger than one 128x128 score tile ever exists, and only
// on chip.
#pragma once

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBM = 128;          // query rows per tile (TMEM lanes)
constexpr int kBN = 128;          // keys per tile
constexpr int kBoxCols = 64;      // bf16 elements per 128-byte swizzle row
constexpr int kBoxBytes = kBM * kBoxCols * 2;   // one TMA box: 128 x 64 bf16
constexpr int kThreads = 192;

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384,
                   kColP1 = 448, kTmemCols = 512;

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kTileBytes = kBM * D * 2;       // 16 KiB or 32 KiB
  static constexpr int kBoxes = D / kBoxCols;          // TMA boxes per tile
  static constexpr int kStages = (D == 128) ? 3 : 4;   // K and V ring depth
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1 + 1 + 1;
  static constexpr int kBarBytes = 8 * kNumBars + 16;  // + tmem slot + abort
  static constexpr int kSmemBytes =
      1024 /*alignment slack*/ + kTileBytes * (1 + 2 * kStages) + kBarBytes;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int Nq, Nkv, Hq, Hkv;
  float scale_log2;   // scale * log2(e)
  int* status;        // device status word (bounded-wait timeouts)
  uint64_t wait_limit_ns;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV,
                  const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (batch b, query head hq, query tile t) ----
  const int n_qtiles = gridDim.x;
  const int t = CAUSAL ? (n_qtiles - 1 - static_cast<int>(blockIdx.x))
                       : static_cast<int>(blockIdx.x);
  const int hq = blockIdx.y;
  const int b = blockIdx.z;
  const int hk = hq / (p.Hq / p.Hkv);
  const int q_row0 = t * kBM;
  const int kv_end = CAUSAL ? min(p.Nkv, q_row0 + kBM) : p.Nkv;
  const int n_blocks = (kv_end + kBN - 1) / kBN;

  // ---- shared memory carve-up (1024-byte aligned for the swizzle atoms) --
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sQ = base;
  const uint32_t sK = sQ + C::kTileBytes;
  const uint32_t sV = sK + NS * C::kTileBytes;
  const uint32_t sBar = sV + NS * C::kTileBytes;
  auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  const uint32_t bQFull = bar(0);
  auto bKFull = [&](int s) { return bar(1 + s); };
  auto bKEmpty = [&](int s) { return bar(1 + NS + s); };
  auto bVFull = [&](int s) { return bar(1 + 2 * NS + s); };
  auto bVEmpty = [&](int s) { return bar(1 + 3 * NS + s); };
  auto bSFull = [&](int i) { return bar(1 + 4 * NS + i); };
  auto bSEmpty = [&](int i) { return bar(3 + 4 * NS + i); };
  const uint32_t bPFull = bar(5 + 4 * NS);
  const uint32_t bODone = bar(6 + 4 * NS);
  const uint32_t bDrain = bar(7 + 4 * NS);
  uint8_t* const misc = base_ptr + (sBar - base) + 8 * C::kNumBars;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile uint32_t* const abort = reinterpret_cast<uint32_t*>(misc + 4);

  if (threadIdx.x == 0) {
    mbar_init(bQFull, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKFull(s), 1);
      mbar_init(bKEmpty(s), 1);
      mbar_init(bVFull(s), 1);
      mbar_init(bVEmpty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bSFull(i), 1);
      mbar_init(bSEmpty(i), 4);
    }
    mbar_init(bPFull, 4);
    mbar_init(bODone, 1);
    mbar_init(bDrain, 1);
    *abort = 0u;
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort, p.status, p.wait_limit_ns};

  if (warp == 4) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      const int zq = b * p.Hq + hq;
      const int zk = b * p.Hkv + hk;
      mbar_arrive_expect_tx(bQFull, C::kTileBytes);
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_3d(sQ + c * kBoxBytes, &tmQ, bQFull, c * kBoxCols, q_row0,
                    zq, once);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_blocks; ++j) {
        const int s = j % NS;
        const uint32_t ph = ((j / NS) & 1) ^ 1;
        if (!mbar_wait(bKEmpty(s), ph, wc)) break;
        mbar_arrive_expect_tx(bKFull(s), C::kTileBytes);
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_3d(sK + s * C::kTileBytes + c * kBoxBytes, &tmK, bKFull(s),
                      c * kBoxCols, j * kBN, zk, keep);
        k_issued = j + 1;
        if (!mbar_wait(bVEmpty(s), ph, wc)) break;
        mbar_arrive_expect_tx(bVFull(s), C::kTileBytes);
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_3d(sV + s * C::kTileBytes + c * kBoxBytes, &tmV, bVFull(s),
                      c * kBoxCols, j * kBN, zk, keep);
        v_issued = j + 1;
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the
      // last load issued into each stage of each ring, and for Q.
      for (int j = (k_issued > NS ? k_issued - NS : 0); j < k_issued; ++j)
        mbar_wait(bKFull(j % NS), (j / NS) & 1, wc, false);
      for (int j = (v_issued > NS ? v_issued - NS : 0); j < v_issued; ++j)
        mbar_wait(bVFull(j % NS), (j / NS) & 1, wc, false);
      mbar_wait(bQFull, 0, wc, false);
    }
  } else if (warp == 5) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      bool ok = mbar_wait(bQFull, 0, wc);
      for (int j = 0; ok && j <= n_blocks; ++j) {
        if (j < n_blocks) {
          const int s = j % NS;
          const int sb = j & 1;
          if (!(ok = mbar_wait(bKFull(s), (j / NS) & 1, wc))) break;
          if (j >= 2 &&
              !(ok = mbar_wait(bSEmpty(sb), ((j >> 1) - 1) & 1, wc)))
            break;
          tc_fence_after();
          const uint32_t d_s = tmem + (sb ? kColS1 : kColS0);
          const uint32_t k_base = sK + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss(d_s, sdesc_sw128(sQ + off, 16, 1024),
                   sdesc_sw128(k_base + off, 16, 1024), C::kIdescS,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bSFull(sb));
          mma_commit(bKEmpty(s));
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int s = jj % NS;
          if (!(ok = mbar_wait(bPFull, jj & 1, wc))) break;
          if (!(ok = mbar_wait(bVFull(s), (jj / NS) & 1, wc))) break;
          tc_fence_after();
          const uint32_t a_p = tmem + ((jj & 1) ? kColP1 : kColP0);
          const uint32_t v_base = sV + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            mma_ts(tmem + kColO, a_p + kk * 8,
                   sdesc_sw128(v_base + kk * 2048, kBoxBytes, 1024),
                   C::kIdescPV, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bODone);
          mma_commit(bVEmpty(s));
        }
      }
      // Every MMA this thread issued completes before the CTA tears down.
      mma_commit(bDrain);
      mbar_wait(bDrain, 0, wc, false);
    }
  } else {
    // ============================ softmax warps ===========================
    const int row = threadIdx.x;                 // 0..127 == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c = p.scale_log2;
    const bool neg_scale = c < 0.f;
    const int q_abs = q_row0 + row;
    float m_run = -INFINITY;   // running max of scale*log2e*s
    float l_run = 0.f;         // running sum of exp2(.. - m_run)
    bool ok = true;
    for (int j = 0; j < n_blocks; ++j) {
      const int sb = j & 1;
      // Warp-uniform outcome: the tcgen05 loads below are .sync.aligned.
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bSFull(sb), (j >> 1) & 1, wc))))
        break;
      tc_fence_after();
      uint32_t sr[kBN];
      const uint32_t s_addr = tmem + lane_off + (sb ? kColS1 : kColS0);
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc) tmem_ld32(s_addr + cc * 32, sr + cc * 32);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc) reg_fence32(sr + cc * 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bSEmpty(sb));
#define S_(i) __uint_as_float(sr[(i)])

      // ---- row extreme over the visible keys of this block ----
      const int col0 = j * kBN;
      const bool need_mask =
          (col0 + kBN > p.Nkv) || (CAUSAL && col0 + kBN - 1 > q_row0);
      int n_vis = kBN;   // keys [col0, col0 + n_vis) are visible to this row
      if (need_mask) {
        int lim = p.Nkv - col0;
        if (CAUSAL) lim = min(lim, q_abs - col0 + 1);
        n_vis = max(0, min(kBN, lim));
      }
      float ext;
      if (!need_mask) {
        float a0 = S_(0), a1 = S_(1), a2 = S_(2), a3 = S_(3);
        if (!neg_scale) {
#pragma unroll
          for (int i = 4; i < kBN; i += 4) {
            a0 = fmaxf(a0, S_(i)); a1 = fmaxf(a1, S_(i + 1));
            a2 = fmaxf(a2, S_(i + 2)); a3 = fmaxf(a3, S_(i + 3));
          }
          ext = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        } else {
#pragma unroll
          for (int i = 4; i < kBN; i += 4) {
            a0 = fminf(a0, S_(i)); a1 = fminf(a1, S_(i + 1));
            a2 = fminf(a2, S_(i + 2)); a3 = fminf(a3, S_(i + 3));
          }
          ext = fminf(fminf(a0, a1), fminf(a2, a3));
        }
      } else {
        ext = neg_scale ? INFINITY : -INFINITY;
#pragma unroll
        for (int i = 0; i < kBN; ++i) {
          if (i < n_vis) ext = neg_scale ? fminf(ext, S_(i)) : fmaxf(ext, S_(i));
        }
      }
      const float m_blk = (n_vis > 0) ? ext * c : -INFINITY;
      const float m_new = fmaxf(m_run, m_blk);
      // exp2 base: finite whenever some key has been visible so far
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - m_use);

      // ---- P = exp2(s * c - m), row sum, pack to bf16 ----
      uint32_t pp[kBN / 2];
      float r0 = 0.f, r1 = 0.f;
      if (!need_mask) {
#pragma unroll
        for (int i = 0; i < kBN; i += 2) {
          const float e0 = ex2_approx(fmaf(S_(i), c, -m_use));
          const float e1 = ex2_approx(fmaf(S_(i + 1), c, -m_use));
          r0 += e0;
          r1 += e1;
          pp[i / 2] = pack_bf16x2(e0, e1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kBN; i += 2) {
          const float e0 = (i < n_vis) ? ex2_approx(fmaf(S_(i), c, -m_use)) : 0.f;
          const float e1 =
              (i + 1 < n_vis) ? ex2_approx(fmaf(S_(i + 1), c, -m_use)) : 0.f;
          r0 += e0;
          r1 += e1;
          pp[i / 2] = pack_bf16x2(e0, e1);
        }
      }
      l_run = l_run * alpha + (r0 + r1);
#undef S_

      // ---- O correction (needs PV_{j-1} complete) ----
      if (j >= 1) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bODone, (j - 1) & 1, wc))))
          break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t o_addr = tmem + lane_off + kColO;
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
      }
      const uint32_t p_addr = tmem + lane_off + (sb ? kColP1 : kColP0);
      tmem_st32(p_addr, pp);
      tmem_st32(p_addr + 32, pp + 32);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bPFull);
      m_run = m_new;
    }

    // ---- epilogue: O / l -> bf16, LSE ----
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(bODone, (n_blocks - 1) & 1, wc));
    if (ok) {
      tc_fence_after();
      const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const bool in_range = q_abs < p.Nq;
      const size_t row_idx =
          (static_cast<size_t>(b) * p.Hq + hq) * static_cast<size_t>(p.Nq) +
          static_cast<size_t>(q_abs);
      __nv_bfloat16* orow = p.o + row_idx * D;
      const uint32_t o_addr = tmem + lane_off + kColO;
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
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1],
                                packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
      if (in_range && p.lse != nullptr) {
        const float lse2 = (l_run > 0.f) ? (m_run + log2f(l_run)) : -INFINITY;
        p.lse[row_idx] = lse2 * 0.69314718055994530942f;
      }
    }
  }

  // ---- teardown: every role is done with TMEM and shared memory ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
