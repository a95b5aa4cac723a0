// fa_fwd_mx.cuh — the attention forward with Q and K in MXFP8: e4m3 values
// with one power-of-two scale (ue8m0) per 32 consecutive elements of a row,
// and S = Q K^T as a block-scaled tensor-core product.
//
// The low-precision direction of "Flash Attention на 5090 в CUDA C++"
// (introduction: MXFP8/NVFP4 MMA as the goal; closing "Что дальше" list) in
// its 8-bit form; the method is otherwise that of fa_fwd_kernel.cuh ("Hacker
// News Digest — gpu-computing", section "Алгоритм Flash Attention 2", with
// the online softmax of section "v1 — базовая версия", item 3).  P V stays
// bf16 (kind::f16).
//
// What the product computes: for a query row with e4m3 values q and scales
// 2^(eq_b - 127) per block b of 32 head-dim elements, and a key row with k
// and 2^(ek_b - 127) likewise,
//     S = sum_b 2^(eq_b - 127) 2^(ek_b - 127) sum_{d in b} q_d k_d,
// i.e. the dot product of the exactly dequantised rows, accumulated in fp32
// by tcgen05.mma.kind::mxf8f6f4.block_scale (one MMA of K = 32 per block).
//
// Schedule (one 128-row query tile per CTA, as fa_fwd_wide.cuh, here with
// 128-key blocks): the block-scaled product reads its scale factors from
// TMEM, and the two-tile kernel's TMEM is full at head dim 128.  TMEM (512
// columns): S buffers at 0 and 128, O at 256, the Q tile's scales at 384,
// a ring of three K-block scale groups at 416, 448 and 480.  P(j) (bf16x2,
// 64 columns) overwrites the first half of its own S buffer.  The MMA warp
// issues S(0) S(1) PV(0) S(2) PV(1) ...: S(j+1) runs while the softmax of
// block j does.
//
// Scale factors in TMEM: a group of four columns holds the scales of 128
// rows (query rows for Q, key rows for K).  Row r = r0 + 32 r1 (r0 < 32)
// sits in lane r0 of every lane quadrant, column r1 of the group, as one
// 32-bit word whose byte b is the ue8m0 scale of head-dim block b; the MMA
// of block b selects byte b through the scale-factor ids of its
// instruction descriptor.  (The same image as a 32-lane x 128-bit copy
// broadcast to the four quadrants.)  Each group starts on a column that is
// a multiple of 32.  The softmax warps (one TMEM lane quadrant each) write
// the groups with tcgen05.st: the Q tile's and the first two K blocks'
// before the loop, and K block j + 2's while they work on block j (S(j + 2)
// is issued only after P(j) is published, and the ring slot it reuses last
// served S(j - 1), complete before S(j) is).
#pragma once

#include "fa_fwd_kernel.cuh"
#include "fa_fwd_wide.cuh"

namespace fa {

constexpr int kMxThreads = 192;   // MMA warp, TMA warp, 4 softmax warps

struct MxCfg {
  static constexpr int D = 128;
  static constexpr int kBN = 128;                        // keys per block
  static constexpr int kQBytes = kBM * D;                // e4m3: 16 KiB
  static constexpr int kKBytes = kBN * D;                // e4m3: 16 KiB
  static constexpr int kVBytes = kBN * D * 2;            // bf16: 32 KiB
  static constexpr int kKStages = 4;
  static constexpr int kVStages = 3;
  // barriers: Q, K full/empty, V full/empty, S full x2, P full x2, PV
  // done, O final, drain, scales ready
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 4;
  static constexpr int kBarBytes = 8 * kNumBars + 32;
  static constexpr int kSmemBytes = 1024 + kQBytes + kKStages * kKBytes +
                                    kVStages * kVBytes + kBarBytes;
  static constexpr uint32_t kColO = 2 * kBN;             // 256
  static constexpr uint32_t kColSfq = kColO + D;         // 384 .. 387
  static constexpr uint32_t kColSfk = kColSfq + 32;      // 416, 448, 480
  static constexpr uint32_t kSfkStride = 32;
  static constexpr int kSfkSlots = 3;
  static_assert(kColSfq % 32 == 0 && kColSfk % 32 == 0 &&
                    kColSfk + (kSfkSlots - 1) * kSfkStride + 4 <= 512,
                "scale-factor groups: 32-aligned, inside the allocation");
  static constexpr uint32_t kTmemAlloc = 512;
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
  // the K ring holds the four softmax warps' staged output rows
  static_assert(4 * 32 * D * 2 <= kKStages * kKBytes, "output staging");
};

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale with e4m3
// A and B (format code 0 in bits 7-9 and 10-12), both K-major, N >> 3 in
// bits 17-22, ue8m0 scale factors (bit 23), M >> 4 in bits 24-28, and the
// scale-factor ids of B (bits 4-5) and A (bits 29-30): the byte of each
// 32-bit scale word this MMA uses.  The accumulator is fp32.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N,
                                                     uint32_t sf_id) {
  return (sf_id << 4) | ((static_cast<uint32_t>(N) >> 3) << 17) | (1u << 23) |
         ((static_cast<uint32_t>(M) >> 4) << 24) | (sf_id << 29);
}

// D[tmem] (+)= (A[smem] with scales sfa) * (B[smem] with scales sfb)^T,
// block-scaled 8-bit operands, issued by one elected lane of the warp.
template <int ACC>
__device__ __forceinline__ void mma_mx_w(uint32_t d_tmem, uint64_t a_desc,
                                         uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem,
                                         uint32_t sfb_tmem) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "n"(ACC)
      : "memory");
}

// Registers -> TMEM: this warp's 32 lanes, four consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
      : "memory");
}

// S = Q K^T for one 128-key block: four block-scaled MMAs of 128x128x32,
// one per 32-element head-dim block b (32 bytes along the 128-byte swizzle
// row; scale byte b).
__device__ __forceinline__ void mx_issue_qk(uint32_t d_tmem, uint64_t dq,
                                            uint64_t dk, uint32_t sfq,
                                            uint32_t sfk) {
  mma_mx_w<0>(d_tmem, dq, dk, idesc_mx_e4m3(kBM, MxCfg::kBN, 0), sfq, sfk);
#pragma unroll
  for (int b = 1; b < MxCfg::D / 32; ++b) {
    const uint64_t off = static_cast<uint64_t>((b * 32) >> 4);
    mma_mx_w<1>(d_tmem, dq + off, dk + off,
                idesc_mx_e4m3(kBM, MxCfg::kBN, static_cast<uint32_t>(b)), sfq,
                sfk);
  }
}

// Parameters beyond FwdParams: the scale tensors, ue8m0 bytes [B, H, N, 4]
// (four per row: head-dim blocks 0..3), read as one 32-bit word per row.
struct MxScales {
  const uint32_t* q_sf;   // [B, Hq, Nq]
  const uint32_t* k_sf;   // [B, Hkv, Nkv]
};

template <bool CAUSAL>
__global__ void __launch_bounds__(kMxThreads, 1)
    fa_fwd_mx_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ FwdParams p,
                     const __grid_constant__ MxScales sf) {
  using M = MxCfg;
  constexpr int D = M::D;
  constexpr int BN = M::kBN;
  constexpr int NK = M::kKStages;
  constexpr int NV = M::kVStages;
  constexpr uint32_t kAll = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (batch b, query head hq, 128-row tile) ----
  int tile = CAUSAL ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                    : static_cast<int>(blockIdx.x);
  int hq = blockIdx.y;
  int b = blockIdx.z;
  // K (e4m3) and V (bf16) of a KV head
  if constexpr (CAUSAL) causal_grid_item(p, 3ll * p.Nkv * 128, tile, hq, b);
  const int hk = hq / (p.Hq / p.Hkv);
  const int row0 = tile * kBM;
  const int kv_end = CAUSAL ? min(p.Nkv, row0 + kBM) : p.Nkv;
  const int nblk = (kv_end + BN - 1) / BN;

  // ---- shared memory (1024-byte aligned for the swizzle atoms) ----
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sQ = base;
  const uint32_t sK = sQ + M::kQBytes;
  const uint32_t sV = sK + NK * M::kKBytes;
  const uint32_t sBar = sV + NV * M::kVBytes;
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
  const uint32_t bSfReady = bar(kB0 + 7);
  static_assert(kB0 + 8 == M::kNumBars, "barrier count");
  uint8_t* const misc = base_ptr + (sBar - base) + 8 * M::kNumBars;
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
    mbar_init(bSfReady, 4);
    wstate->abort = 0u;
    wstate->status = p.status;
    wstate->limit_ns = p.wait_limit_ns;
    mbar_init_fence();
  }
  if (warp == kWideMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), M::kTmemAlloc);
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
      mbar_arrive_expect_tx(bQFull, M::kQBytes);
      tma_load_3d(sQ, &tmQ, bQFull, 0, row0, zq, once);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int sk = j % NK, sv = j % NV;
        if (!mbar_wait(bKEmpty(sk), ((j / NK) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bKFull(sk), M::kKBytes);
        tma_load_3d(sK + sk * M::kKBytes, &tmK, bKFull(sk), 0, j * BN, zk,
                    keep);
        k_issued = j + 1;
        if (!mbar_wait(bVEmpty(sv), ((j / NV) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bVFull(sv), M::kVBytes);
        for (int c = 0; c < D / kBoxCols; ++c)
          tma_load_3d(sV + sv * M::kVBytes + c * kBoxBytes, &tmV, bVFull(sv),
                      c * kBoxCols, j * BN, zk, keep);
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
    const uint64_t dV = sdesc_sw128(sV, kBoxBytes, 1024);
    constexpr uint64_t kKStep = static_cast<uint64_t>(M::kKBytes >> 4);
    constexpr uint64_t kVStep = static_cast<uint64_t>(M::kVBytes >> 4);
    bool ok = __all_sync(kAll, mbar_wait(bQFull, 0, wc)) &&
              __all_sync(kAll, mbar_wait(bSfReady, 0, wc));
    tc_fence_after();
    // S(j) for j = 0, then per step: S(j+1), PV(j).
    for (int j = -1; ok && j < nblk; ++j) {
      const int jn = j + 1;                     // block of the next S
      if (jn < nblk) {
        const int s = jn % NK;
        if (!(ok = __all_sync(kAll, mbar_wait(bKFull(s), (jn / NK) & 1, wc))))
          break;
        mx_issue_qk(tmem + static_cast<uint32_t>((jn & 1) * BN), dQ,
                    dK + static_cast<uint64_t>(s) * kKStep,
                    tmem + M::kColSfq,
                    tmem + M::kColSfk +
                        static_cast<uint32_t>(jn % M::kSfkSlots) *
                            M::kSfkStride);
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
        issue_pv<D>(tmem + M::kColO, tmem + static_cast<uint32_t>((j & 1) * BN),
                    dV + static_cast<uint64_t>(sv) * kVStep, M::kIdescPV,
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
    const int quad = warp & 3;                  // TMEM lane quadrant
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float c = p.scale_log2;
    const bool neg_scale = c < 0.f;
    const int q_abs = row0 + quad * 32 + lane;
    // Scale words of a group (see the header): this lane holds rows
    // lane + 32 c, c = 0..3, of the query tile or of a key block (0 past the
    // end of the sequence: those rows are masked or never stored).
    const uint32_t* q_sf_head =
        sf.q_sf + (static_cast<int64_t>(b) * p.Hq + hq) * p.Nq;
    const uint32_t* k_sf_head =
        sf.k_sf + (static_cast<int64_t>(b) * p.Hkv + hk) * p.Nkv;
    auto k_scale_words = [&](int j, uint32_t (&w)[4]) {
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int key = j * BN + c4 * 32 + lane;
        w[c4] = key < p.Nkv ? __ldg(k_sf_head + key) : 0u;
      }
    };
    auto k_group = [&](int j) {
      return tmem + lane_off + M::kColSfk +
             static_cast<uint32_t>(j % M::kSfkSlots) * M::kSfkStride;
    };
    {
      uint32_t w[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int row = row0 + c4 * 32 + lane;
        w[c4] = row < p.Nq ? __ldg(q_sf_head + row) : 0u;
      }
      tmem_st4(tmem + lane_off + M::kColSfq, w);
      for (int j = 0; j < 2 && j < nblk; ++j) {
        k_scale_words(j, w);
        tmem_st4(k_group(j), w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bSfReady);
    }
    float m_ref = -INFINITY;   // reference max (log2 domain) of p and l
    float l_run = 0.f;         // sum of exp2(s*c - m_ref) over seen keys
    float w_run = 0.f;         // the divisor of O (see top_rounding)
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int u = j & 1;                      // S buffer of block j
      // the scales of block j + 2, loaded now, stored before P(j) is
      // published (S(j + 2) is issued only after that)
      uint32_t kw_next[4] = {0u, 0u, 0u, 0u};
      if (j + 2 < nblk) k_scale_words(j + 2, kw_next);
      if (!(ok = __all_sync(kAll, mbar_wait(bSFull(u), (j >> 1) & 1, wc))))
        break;
      tc_fence_after();
      uint32_t sr[BN];
      const uint32_t s_addr = tmem + lane_off + static_cast<uint32_t>(u * BN);
      const int col0 = j * BN;
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
      // ---- row extreme over the visible keys of this block ----
      int n_vis = BN;
      if (need_mask) {
        int lim = p.Nkv - col0;
        if (CAUSAL) lim = min(lim, q_abs - col0 + 1);
        n_vis = max(0, min(BN, lim));
      }
      float ext;
      if (!need_mask) {
        ext = neg_scale ? fminf(fminf(red[0], red[1]), fminf(red[2], red[3]))
                        : fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      } else {
        const float idn = neg_scale ? INFINITY : -INFINITY;
        float e4[4] = {idn, idn, idn, idn};
#pragma unroll
        for (int i = 0; i < BN; i += 2) {
          const float v0 = (i < n_vis) ? __uint_as_float(sr[i]) : idn;
          const float v1 = (i + 1 < n_vis) ? __uint_as_float(sr[i + 1]) : idn;
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
      w_run = w_run * alpha + (n_vis > 0 ? top_rounding(ext, c, m_use) : 0.f);

      // ---- P = exp2(s * c - m), packed to bf16, row sums ----
      uint32_t pp[BN / 2];
      const float rsum =
          need_mask ? exp_pack_row<BN, true>(sr, c, m_use, n_vis, pp)
                    : exp_pack_row<BN, false>(sr, c, m_use, BN, pp);
      l_run = l_run * alpha + rsum;
      w_run += rsum;
      m_ref = m_new;
      tmem_st32(s_addr, pp);
      tmem_st32(s_addr + 32, pp + 32);
      if (j + 2 < nblk) tmem_st4(k_group(j + 2), kw_next);

      // ---- rescale O when the reference max moved.  PV(j-1) may still be
      // running (S(j) was issued before it), so wait for it first. ----
      if (j >= 1 && __any_sync(kAll, alpha != 1.f)) {
        if (!(ok = __all_sync(kAll, mbar_wait(bPVDone, (j - 1) & 1, wc))))
          break;
        tc_fence_after();
        rescale_o<D>(tmem + lane_off + M::kColO, alpha);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bPFull(u));
    }

    // ---- epilogue ----
    if (ok && nblk > 0) ok = __all_sync(kAll, mbar_wait(bOFinal, 0, wc));
    if (ok && nblk > 0) {
      tc_fence_after();
      const size_t row_idx =
          (static_cast<size_t>(b) * p.Hq + hq) * static_cast<size_t>(p.Nq) +
          static_cast<size_t>(q_abs);
      // Every MMA is complete and every K tile consumed: the K ring stages
      // the four warps' rows for TMA stores.
      const OutRows out{sK + static_cast<uint32_t>(quad) * (32u * D * 2u), &tmO,
                        q_abs - lane, b * p.Hq + hq, p.Nq};
      store_final_row<D>(tmem + lane_off + M::kColO, m_ref, l_run, w_run,
                         p.o + row_idx * D,
                         p.lse != nullptr ? p.lse + row_idx : nullptr,
                         q_abs < p.Nq, out);
    }
  }

  // ---- teardown: every role is done with TMEM and shared memory ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWideMmaWarp) tmem_dealloc(tmem, M::kTmemAlloc);
}

}  // namespace fa
