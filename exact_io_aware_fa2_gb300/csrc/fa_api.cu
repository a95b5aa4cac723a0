// fa_api.cu — host side of the C ABI declared in include/fa.h: argument
// validation, TMA tensor-map encoding, kernel selection and launch.
//
// The operation and its sources are described in include/fa.h.  This file
// holds no arithmetic of the method; it only prepares the launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_fwd_kernel.cuh"
#include "fa_fwd_mx.cuh"
#include "fa_fwd_persist.cuh"
#include "fa_fwd_stream.cuh"
#include "fa_fwd_wide.cuh"

namespace fa {
// Device-side status word (one per device), written by bounded waits that
// ran out and read back / cleared by fa_last_device_error().
__device__ int g_fa_status = 0;
}  // namespace fa

namespace {

constexpr int kMaxDevices = 64;
// Wall-clock limit of every wait inside the attention kernel.  Real waits
// last microseconds; this only turns a broken launch into an error code.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType,
                                   cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

template <int D, bool CAUSAL, bool QK8 = false>
cudaError_t opt_in_smem() {
  constexpr int kSmem = fa::FwdCfg<D, QK8>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(
      fa::fa_fwd_kernel<D, CAUSAL, false, QK8>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, CAUSAL, true, QK8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmem);
}

template <int D, bool QK8 = false>
cudaError_t opt_in_smem_stream() {
  return cudaFuncSetAttribute(fa::fa_fwd_stream_kernel<D, QK8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa::StreamCfg<D, QK8>::kSmemBytes);
}

template <int D>
cudaError_t opt_in_smem_persist() {
  return cudaFuncSetAttribute(fa::fa_fwd_persist_kernel<D, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa::PersistCfg<D, false>::kSmemBytes);
}

cudaError_t opt_in_smem_mx() {
  cudaError_t e = cudaFuncSetAttribute(
      fa::fa_fwd_mx_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      fa::MxCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa::fa_fwd_mx_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa::MxCfg::kSmemBytes);
}

template <int D, bool CAUSAL>
cudaError_t opt_in_smem_wide() {
  cudaError_t e = cudaFuncSetAttribute(
      fa::fa_fwd_wide_kernel<D, CAUSAL, false>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, fa::WideCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa::fa_fwd_wide_kernel<D, CAUSAL, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa::WideCfg<D>::kSmemBytes);
}

// Head dims with a kernel: 64 and 128 (two query tiles per CTA, split-KV
// capable) and 192 and 256 (one query tile per CTA, fa_fwd_wide.cuh).
bool supported_head_dim(int D) {
  return D == 64 || D == 128 || D == 192 || D == 256;
}
// Shapes whose split-KV form runs the one-tile kernel (fa_fwd_wide.cuh):
// head dims 192 and 256 (every schedule), and causal head dim 64 (its
// one-tile split is finer than the two-tile one; unsplit, causal shapes run
// the persistent two-tile kernel).
bool one_tile(int D, int causal) {
  return D == 192 || D == 256 || (D == 64 && causal);
}

int* g_status_word[kMaxDevices];
int g_sm_count[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];

// Split-KV scratch for fa_fwd_noalloc: a fixed array in device memory, part
// of the loaded module, so that entry point never allocates.  Each device
// that loads the library holds it until the process exits.  In host code
// the name only stands for the symbol; its device address comes from
// cudaGetSymbolAddress, taken once per device in device_ready.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices];   // nullptr if the lookup failed

// Freed split-KV / stream scratch the pool keeps reserved for later calls.
// Every shape needs at most about 30 MB on a 152-SM GB300 (the need grows
// with the SM count, not the sequence lengths), so this keeps one call's
// scratch; anything above it returns to the device at the next
// synchronisation.
constexpr uint64_t kPoolKeepBytes = 64ull << 20;

// Per-device readiness: compute capability 10.3, the kernels' shared memory
// opt-in and the device address of the status word, done once per device
// with that device current.
int device_ready(int** word_out, int* dev_out = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  static std::once_flag flags[kMaxDevices];
  static int status[kMaxDevices];
  std::call_once(flags[dev], [dev] {
    status[dev] = FA_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor,
                               dev) != cudaSuccess) {
      status[dev] = FA_ERR_CUDA;
      cudaGetLastError();
      return;
    }
    if (major != 10 || minor != 3) {
      status[dev] = FA_ERR_UNSUPPORTED;
      return;
    }
    if (opt_in_smem<64, false>() != cudaSuccess ||
        opt_in_smem<64, true>() != cudaSuccess ||
        opt_in_smem<128, false>() != cudaSuccess ||
        opt_in_smem<128, true>() != cudaSuccess ||
        opt_in_smem<128, false, true>() != cudaSuccess ||
        opt_in_smem<128, true, true>() != cudaSuccess ||
        opt_in_smem_stream<64>() != cudaSuccess ||
        opt_in_smem_stream<128>() != cudaSuccess ||
        opt_in_smem_stream<128, true>() != cudaSuccess ||
        opt_in_smem_persist<64>() != cudaSuccess ||
        opt_in_smem_mx() != cudaSuccess ||
        opt_in_smem_persist<128>() != cudaSuccess ||
        opt_in_smem_wide<64, false>() != cudaSuccess ||
        opt_in_smem_wide<64, true>() != cudaSuccess ||
        opt_in_smem_wide<192, false>() != cudaSuccess ||
        opt_in_smem_wide<192, true>() != cudaSuccess ||
        opt_in_smem_wide<256, false>() != cudaSuccess ||
        opt_in_smem_wide<256, true>() != cudaSuccess) {
      status[dev] = FA_ERR_CUDA;
      cudaGetLastError();
      return;
    }
    void* word = nullptr;
    if (cudaGetSymbolAddress(&word, fa::g_fa_status) != cudaSuccess) {
      status[dev] = FA_ERR_CUDA;
      cudaGetLastError();   // leave no pending error for the next launch
      return;
    }
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) == cudaSuccess)
      g_noalloc_ptr[dev] = scratch;
    else
      cudaGetLastError();   // only fa_fwd_noalloc fails then
    g_status_word[dev] = static_cast<int*>(word);
    if (cudaDeviceGetAttribute(&g_sm_count[dev],
                               cudaDevAttrMultiProcessorCount,
                               dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    // Stream-ordered pool for fa_fwd's split-KV scratch (fa_fwd_ws takes
    // the caller's memory instead); up to kPoolKeepBytes of freed blocks
    // stay reserved for the next call.
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    uint64_t keep = kPoolKeepBytes;
    if (cudaMemPoolCreate(&g_pool[dev], &props) != cudaSuccess ||
        cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold,
                                &keep) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    status[dev] = FA_OK;
  });
  if (status[dev] == FA_OK && word_out != nullptr) *word_out = g_status_word[dev];
  if (status[dev] == FA_OK && dev_out != nullptr) *dev_out = dev;
  return status[dev];
}

// Split-KV: when the pairs of query tiles fill fewer than half the SMs, cut
// each pair's K/V range into contiguous pieces (at least kMinSplitBlocks
// blocks each, at most kMaxSplits pieces).  The count minimises the
// estimated time: waves of CTAs x (blocks per piece + kSplitOverheadBlocks,
// a piece's fixed cost for its Q load, set-up and fp32 partial write, in
// units of one K/V block), the smaller count on a tie.  The one-tile kernel's
// 64-key blocks are short against its fixed cost per piece: fitted to GB300
// timings at head dims 192 and 256 (one wave of 2 to 4 pieces against 2 to
// 3 waves of 7 to 9: 64 heads of 1024 x 8192 at D 192 62.5 vs 79.8 us,
// 16 heads of 256 x 16384 at D 256 90.6 vs 100.8; 2 heads of 4096 x 32768
// at D 256 266.1 vs 250.8 the other way), about 15 blocks.
constexpr int kMinSplitBlocks = 4;
constexpr int kMaxSplits = 64;
constexpr int kSplitOverheadBlocks = 3;
constexpr int kSplitOverheadBlocksOneTile = 15;

// Query rows per CTA and keys per K/V block of the kernel a head dim runs
// (the two-tile kernel: 256 and 128; the wide-head kernel: 128 and 64).
int unit_rows(int D, int causal) {
  return one_tile(D, causal) ? fa::kBM : fa::kBM * fa::kTilesPerCta;
}
int block_keys(int D, int causal) {
  return one_tile(D, causal) ? 64 : fa::kBN;
}

int plan_splits(int B, int Hq, int Nq, int Nkv, int D, int causal, int sms) {
  const int rows_u = unit_rows(D, causal), keys_b = block_keys(D, causal);
  const long long units = (Nq + rows_u - 1) / rows_u;
  const long long ctas = units * Hq * B;
  if (ctas * 2 > sms) return 1;
  long long longest = (Nkv + keys_b - 1) / keys_b;       // K/V blocks
  if (causal) {
    const int rows = Nq < Nkv ? Nq : Nkv;
    longest = (rows + keys_b - 1) / keys_b;
  }
  long long cap = longest / kMinSplitBlocks;
  if (cap > kMaxSplits) cap = kMaxSplits;
  if (cap > 65535 / B) cap = 65535 / B;                  // grid.z limit
  long long best_s = 1, best_cost = -1;
  for (long long s = 1; s <= cap; ++s) {
    const long long waves = (ctas * s + sms - 1) / sms;
    const long long cost =
        waves * ((longest + s - 1) / s +
                 (keys_b == fa::kBN ? kSplitOverheadBlocks
                                    : kSplitOverheadBlocksOneTile));
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = s;
    }
  }
  return static_cast<int>(best_s);
}

// Stream schedule (fa_fwd_stream.cuh; two-tile kernel, no causal mask):
// when whole tile pairs leave SMs idle in their last wave, give every CTA
// an equal contiguous share of all (pair, K/V block) items instead.  Costs
// in units of one K/V block of one pair on the two-tile kernel, fitted by
// least squares to GB300 timings of both schedules on 21 shapes per head
// dim (80 to 256 pairs of 4096 to 32768 keys):
//   plain  = waves x (blocks per pair + wave_overhead) + plain_overhead
//   stream = block_factor x blocks per CTA + stream_overhead
//            + segment_cost x (segments per CTA - 1)
// The stream kernel's blocks take about as long as the plain kernel's; its
// partial writes, merges and segment switches cost about 6 blocks more
// than the plain kernel's start-up and epilogue.  Stream runs when its
// estimate is the smaller one and a CTA's share is at least half a pair (a
// merger then combines at most two partials); on the 42 shapes the choice
// is within 0.6% of the faster schedule.  Measured, stream against plain
// at D = 128: 80 pairs 70.6 vs 98.3 us, 112 pairs 87.0 vs 98.3, 128 pairs
// 96.3 vs 98.3, 144 pairs 106.5 vs 100.4 (plain), 256 pairs 177.1 vs 192.5;
// at D = 64 and 128 pairs 84.1 vs 90.1.
struct StreamCost {
  double wave_overhead, plain_overhead, block_factor, stream_overhead,
      segment_cost;
};
constexpr StreamCost kStreamCostD128{4.06, 4.52, 1.024, 14.39, 2.08};
constexpr StreamCost kStreamCostD64{1.46, 6.50, 0.988, 12.35, 1.48};

// Schedule forced by fa_set_schedule (FA_SCHEDULE_AUTO: the estimate).
std::atomic<int> g_forced_schedule{FA_SCHEDULE_AUTO};

struct Plan {
  int splits;        // split-KV pieces per unit of query rows (1: none)
  int stream_len;    // K/V blocks per CTA of the stream schedule (0: off)
  int stream_ctas;   // CTAs of the stream schedule
  int persist_ctas;  // CTAs of the persistent schedule (0: off)
};

// Persistent schedule (fa_fwd_persist.cuh): causal shapes at head dims 64
// and 128 that do not split, bf16 inputs, whose K and V together fit in
// kPersistKVBytes.  One CTA per SM (at most one per pair) walks a list of
// whole tile pairs sorted longest first over all heads, so at any moment
// every head's K/V is in use; past L2's reach that re-reads K/V from DRAM
// (measured on the 16-head 32768-key shape: 2.14 GB read per launch against
// 0.40 GB with one CTA per pair, which walks the heads in order), and such
// shapes keep one CTA per pair.  Measured same-GPU against one CTA per pair:
// causal B4 H16 N2048 D64 63.5 vs 69.2 us, causal GQA B2 Hq32/Hkv8 N8192
// D128 727 vs 753 us; B1 H16 N32768 D128 2885 vs 2832 us.
constexpr int64_t kPersistKVBytes = 96ll << 20;

bool persist_ok(int B, int Hkv, int Nkv, int D, int causal, bool qk8) {
  const int64_t kv_bytes = 4ll * B * Hkv * Nkv * D;     // K and V, bf16
  return causal && (D == 64 || D == 128) && !qk8 &&
         kv_bytes <= kPersistKVBytes;
}

Plan plan_forward(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                  int causal, int sms, bool qk8 = false) {
  const int forced = g_forced_schedule.load(std::memory_order_relaxed);
  if (forced == FA_SCHEDULE_PLAIN) return Plan{1, 0, 0, 0};
  const bool stream_ok = !causal && !one_tile(D, causal);
  Plan pl{1, 0, 0, 0};
  if (forced != FA_SCHEDULE_STREAM || !stream_ok)
    pl.splits = plan_splits(B, Hq, Nq, Nkv, D, causal, sms);
  if (pl.splits == 1 && persist_ok(B, Hkv, Nkv, D, causal, qk8)) {
    const int64_t pairs = static_cast<int64_t>(B) * Hq *
                          ((Nq + 2 * fa::kBM - 1) / (2 * fa::kBM));
    // (the kernel numbers its list of pairs with 32-bit integers)
    if (pairs < (int64_t{1} << 31)) {
      pl.persist_ctas = static_cast<int>(pairs < sms ? pairs : sms);
      return pl;
    }
  }
  if (!stream_ok) return pl;
  const int64_t pairs = static_cast<int64_t>(B) * Hq *
                        ((Nq + 2 * fa::kBM - 1) / (2 * fa::kBM));
  bool from_split = false;
  if (pl.splits > 1) {
    // A split whose pieces need more than one wave of CTAs loses to the
    // stream schedule, which gives every SM one equal share (measured on
    // GB300, split against stream: 64 pairs x 16384 keys in 7 pieces, 448
    // CTAs, 135.7 vs 111.6 us at D = 128 and 100.6 vs 90.2 at D = 64; 32
    // pairs x 32768 keys in 9 pieces 209.4 vs 193.5; within one wave the
    // split wins, e.g. 16 pairs x 16384 keys in 4 pieces 66.0 vs 72.2).
    if (pairs * pl.splits <= sms) return pl;
    pl.splits = 1;
    from_split = true;
  }
  const int64_t nbp = (Nkv + fa::kBN - 1) / fa::kBN;
  const int64_t total = pairs * nbp;
  // (the kernel numbers its items with 32-bit integers)
  if (total >= (int64_t{1} << 31)) return pl;
  const int64_t L = (total + sms - 1) / sms;
  if (forced != FA_SCHEDULE_STREAM && !from_split) {
    const StreamCost& k = D == 64 ? kStreamCostD64 : kStreamCostD128;
    const int64_t waves = (pairs + sms - 1) / sms;
    const double plain =
        static_cast<double>(waves) * (static_cast<double>(nbp) +
                                      k.wave_overhead) +
        k.plain_overhead;
    const int64_t segments = (L - 1 + nbp - 1) / nbp + 1;   // at most
    const double stream = k.block_factor * static_cast<double>(L) +
                          k.stream_overhead +
                          k.segment_cost * static_cast<double>(segments - 1);
    if (2 * L < nbp || stream > plain) return pl;
  }
  pl.stream_len = static_cast<int>(L);
  pl.stream_ctas = static_cast<int>((total + L - 1) / L);
  return pl;
}

// The shape the kernel runs.  Without a causal mask every query row of a
// GQA group reads the same K/V, and the group's heads are adjacent in the
// [B, Hq, Nq, D] layout (as are their O rows and LSE entries), so the group
// runs as one head of (Hq / Hkv) * Nq rows: no padded query tile per head
// and one pass over K/V per group.  With the mask a row's visible keys
// depend on its index within its own head, so causal shapes run as given.
struct RunShape {
  int Hq, Nq;
};

RunShape run_shape(int Hq, int Hkv, int Nq, int causal) {
  const long long packed = static_cast<long long>(Hq / Hkv) * Nq;
  if (causal || Hq == Hkv || packed > (1ll << 30)) return {Hq, Nq};
  return {Hkv, static_cast<int>(packed)};
}

// Scratch: for split-KV one fp32 slot of unit_rows(D) * (D + 3) words per
// (batch, head, unit of query rows, K/V range); for the stream schedule one
// slot per CTA plus its flags.
int64_t workspace_bytes(int B, int Hq, int Nq, int D, int causal,
                        const Plan& pl) {
  if (pl.stream_len > 0)
    return D == 64 ? fa::stream_workspace_bytes<64>(pl.stream_ctas)
                   : fa::stream_workspace_bytes<128>(pl.stream_ctas);
  const int splits = pl.splits;
  if (splits <= 1) return 0;
  const int64_t rows_u = unit_rows(D, causal);
  const int64_t units = (Nq + rows_u - 1) / rows_u;
  const int64_t slot = rows_u * (D + 3);
  return static_cast<int64_t>(B) * Hq * units * splits * slot * 4;
}

// Tensor maps are cached per (pointer, [BH, N, D] extent, box, element
// type): a map holds only an address, extents, strides and the box, so an
// entry stays valid for any later tensor at that address with that shape.
// A small least-recently-used table, shared by all threads and devices.
struct MapKey {
  const void* ptr;
  long long BH;
  int N, D, box_rows, e4m3;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && BH == o.BH && N == o.N && D == o.D &&
           box_rows == o.box_rows && e4m3 == o.e4m3;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  uint64_t last_use;   // 0: empty
};
constexpr int kMapCacheEntries = 64;
MapEntry g_map_cache[kMapCacheEntries];
uint64_t g_map_clock = 0;
std::mutex g_map_mu;
std::atomic<size_t> g_map_encodes{0};

// Looks the key up; on a miss calls `encode` to fill a free or the least
// recently used entry.  Returns FA_OK or the encoder's error.
template <typename Encode>
int cached_map(CUtensorMap* out, const MapKey& key, Encode encode) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry* victim = &g_map_cache[0];
  for (MapEntry& e : g_map_cache) {
    if (e.last_use != 0 && e.key == key) {
      e.last_use = ++g_map_clock;
      *out = e.map;
      return FA_OK;
    }
    if (e.last_use < victim->last_use) victim = &e;
  }
  const int st = encode(&victim->map);
  g_map_encodes.fetch_add(1, std::memory_order_relaxed);
  if (st != FA_OK) {
    victim->last_use = 0;
    return st;
  }
  victim->key = key;
  victim->last_use = ++g_map_clock;
  *out = victim->map;
  return FA_OK;
}

// Tensor map of a contiguous bf16 [BH, N, D] tensor, read in boxes of 64
// head-dim elements (one 128-byte swizzle row) by `box_rows` sequence rows,
// with the 128-byte swizzle.  Rows past N are zero-filled by the TMA unit.
int encode_bhnd_uncached(CUtensorMap* map, const void* ptr, long long BH,
                         int N, int D, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(N) * D * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(fa::kBoxCols),
                       static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int encode_bhnd(CUtensorMap* map, const void* ptr, long long BH, int N,
                int D, int box_rows = fa::kBM) {
  return cached_map(map, MapKey{ptr, BH, N, D, box_rows, 0},
                    [&](CUtensorMap* m) {
                      return encode_bhnd_uncached(m, ptr, BH, N, D, box_rows);
                    });
}

// The same for a one-byte (e4m3) [BH, N, D] tensor: boxes of 128 head-dim
// elements (one 128-byte swizzle row) by 128 sequence rows.
int encode_bhnd_e4m3_uncached(CUtensorMap* map, const void* ptr, long long BH,
                              int N, int D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D),
                           static_cast<cuuint64_t>(N) * D};
  cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(fa::kBM), 1};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                   const_cast<void*>(ptr), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int encode_bhnd_e4m3(CUtensorMap* map, const void* ptr, long long BH, int N,
                     int D) {
  return cached_map(map, MapKey{ptr, BH, N, D, fa::kBM, 1},
                    [&](CUtensorMap* m) {
                      return encode_bhnd_e4m3_uncached(m, ptr, BH, N, D);
                    });
}

// fa_merge_kernel over units of ROWS query rows.
template <int D, int ROWS>
int launch_merge(const fa::FwdParams& p, int B, int Hq, int Nq,
                 cudaStream_t stream) {
  using M = fa::MergeCfg<D>;
  const int units = (Nq + ROWS - 1) / ROWS;
  // Programmatic serialization: the merge grid is scheduled once every
  // forward CTA has reached its epilogue, and waits (griddepcontrol.wait)
  // for the forward grid to complete before reading the partials.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * (ROWS / M::kRowsPerBlock), Hq, B);
  cfg.blockDim = dim3(M::kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fa::fa_merge_kernel<D, ROWS>, p) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool CAUSAL, bool QK8 = false>
int launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
           const CUtensorMap& o, const fa::FwdParams& p, int B, int Hq,
           int Nq, cudaStream_t stream) {
  constexpr int kSmem = fa::FwdCfg<D, QK8>::kSmemBytes;
  const int rows_per_cta = fa::kBM * fa::kTilesPerCta;
  const int pairs = (Nq + rows_per_cta - 1) / rows_per_cta;
  if constexpr (!CAUSAL) {
    if (p.stream_len > 0) {
      const int64_t total = static_cast<int64_t>(B) * Hq * pairs *
                            ((p.Nkv + fa::kBN - 1) / fa::kBN);
      const dim3 sgrid(static_cast<unsigned>(
          (total + p.stream_len - 1) / p.stream_len));
      // cooperative: every CTA resident at once, since mergers wait for
      // writers of lower grid index (at most one CTA per SM)
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = sgrid;
      cfg.blockDim = dim3(fa::kThreads);
      cfg.dynamicSmemBytes = fa::StreamCfg<D, QK8>::kSmemBytes;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, fa::fa_fwd_stream_kernel<D, QK8>, q, k, v,
                             o, p) != cudaSuccess)
        return FA_ERR_CUDA;
      return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
  }
  dim3 grid(pairs, Hq, B * p.kv_splits);
  if (p.kv_splits > 1)
    fa::fa_fwd_kernel<D, CAUSAL, true, QK8>
        <<<grid, fa::kThreads, kSmem, stream>>>(q, k, v, o, p);
  else
    fa::fa_fwd_kernel<D, CAUSAL, false, QK8>
        <<<grid, fa::kThreads, kSmem, stream>>>(q, k, v, o, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (p.kv_splits > 1) return launch_merge<D, fa::kBM * fa::kTilesPerCta>(
                                p, B, Hq, Nq, stream);
  return FA_OK;
}

template <int D>
int launch_persist(const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const CUtensorMap& o,
                   const fa::FwdParams& p, int ctas, cudaStream_t stream) {
  // The kernel's register split redistributes the launch allocation: the
  // build must have given it kPersistRegsLaunch registers per thread.
  static const bool regs_ok = [] {
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, fa::fa_fwd_persist_kernel<D, true>) ==
               cudaSuccess &&
           a.numRegs == fa::kPersistRegsLaunch;
  }();
  if (!regs_ok) return FA_ERR_CUDA;
  if (p.scale_log2 == 0.f) return FA_ERR_INVALID_VALUE;  // see run_forward
  fa::fa_fwd_persist_kernel<D, true>
      <<<ctas, fa::kPersistThreads, fa::PersistCfg<D, false>::kSmemBytes,
         stream>>>(q, k, v, o, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool CAUSAL>
int launch_wide(const CUtensorMap& q, const CUtensorMap& k,
                const CUtensorMap& v, const CUtensorMap& o,
                const fa::FwdParams& p, int B, int Hq, int Nq,
                cudaStream_t stream) {
  dim3 grid((Nq + fa::kBM - 1) / fa::kBM, Hq, B * p.kv_splits);
  if (p.kv_splits > 1)
    fa::fa_fwd_wide_kernel<D, CAUSAL, true>
        <<<grid, fa::kWideThreads, fa::WideCfg<D>::kSmemBytes, stream>>>(
            q, k, v, o, p);
  else
    fa::fa_fwd_wide_kernel<D, CAUSAL, false>
        <<<grid, fa::kWideThreads, fa::WideCfg<D>::kSmemBytes, stream>>>(
            q, k, v, o, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (p.kv_splits > 1)
    return launch_merge<D, fa::kBM>(p, B, Hq, Nq, stream);
  return FA_OK;
}

// Value under which one launch's stream-schedule CTAs publish their
// partials: distinct for every call of the process, never 0 (the value a
// merger leaves behind), and starting from a clock-derived 64-bit value so
// that scratch memory left by other work is unlikely to hold it.
uint64_t next_epoch() {
  static std::atomic<uint64_t> counter{
      static_cast<uint64_t>(
          std::chrono::steady_clock::now().time_since_epoch().count()) *
      0x9E3779B97F4A7C15ull};
  uint64_t e = counter.fetch_add(1, std::memory_order_relaxed);
  if (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed);
  return e;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

__global__ void probe_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ fa::WaitState ws;
  if (threadIdx.x == 0) {
    fa::mbar_init(fa::smem_addr(&bar_mem), 1);
    ws.abort = 0;
    ws.status = status;
    ws.limit_ns = limit_ns;
    fa::mbar_init_fence();
    // Nothing arrives on this barrier: the wait must run out.
    const fa::WaitCtx wc{fa::smem_addr(&ws)};
    fa::mbar_wait(fa::smem_addr(&bar_mem), 0, wc);
  }
  __syncwarp();
}

// A global-memory flag nothing ever sets, for fa_probe_flag_wait.
__device__ uint64_t g_probe_flag = 0;

__global__ void probe_flag_kernel(int* status, uint64_t limit_ns) {
  __shared__ fa::WaitState ws;
  if (threadIdx.x == 0) {
    ws.abort = 0;
    ws.status = status;
    ws.limit_ns = limit_ns;
  }
  __syncwarp();
  // The value 1 is never published: the wait must run out.
  const fa::WaitCtx wc{fa::smem_addr(&ws)};
  fa::flag_wait(&g_probe_flag, 1ull, wc);
  __syncwarp();
}

int check_args(const void* q, const void* k, const void* v, const void* o,
               const float* lse, int B, int Hq, int Hkv, int Nq, int Nkv,
               int D, float scale) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr)
    return FA_ERR_INVALID_VALUE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || D < 1)
    return FA_ERR_INVALID_VALUE;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_VALUE;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_VALUE;
  if (B > 65535 || Hq > 65535) return FA_ERR_INVALID_VALUE;  // grid limits
  if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || (lse != nullptr && !aligned(lse, 4)))
    return FA_ERR_MISALIGNED;
  return FA_OK;
}

// Shared body of fa_fwd and fa_fwd_ws.  Scratch: from the device pool when
// `pool_scratch`, else the caller's `workspace` (`ws_bytes` long).
// `qk8`: q and k are e4m3 with descale factors q_descale and k_descale
// (D = 128 only); the scores are then (q k^T) * q_descale * k_descale.
int run_forward(const void* q, const void* k, const void* v, void* o,
                float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                float scale, int causal, void* workspace, size_t ws_bytes,
                bool pool_scratch, cudaStream_t s, bool qk8 = false,
                float q_descale = 1.f, float k_descale = 1.f) {
  int st = check_args(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale);
  if (st != FA_OK) return st;
  if (qk8) {
    if (!std::isfinite(q_descale) || !std::isfinite(k_descale) ||
        !(q_descale > 0.f) || !(k_descale > 0.f))
      return FA_ERR_INVALID_VALUE;
    if (D != 128) return FA_ERR_UNSUPPORTED;
  }
  int* word = nullptr;
  int dev = 0;
  if ((st = device_ready(&word, &dev)) != FA_OK) return st;

  const RunShape rs = run_shape(Hq, Hkv, Nq, causal);
  Hq = rs.Hq;
  Nq = rs.Nq;
  fa::FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nkv = Nkv;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale_log2 = static_cast<float>(
      static_cast<double>(scale) * 1.4426950408889634074 *
      (qk8 ? static_cast<double>(q_descale) * k_descale : 1.0));
  p.status = word;
  p.wait_limit_ns = kWaitLimitNs;
  Plan pl = plan_forward(B, Hq, Hkv, Nq, Nkv, D, causal, g_sm_count[dev], qk8);
  // The persistent kernel hides masked keys through their scores, which
  // needs a nonzero scale: a zero scale runs the one-pair-per-CTA kernels.
  if (pl.persist_ctas > 0 && p.scale_log2 == 0.f) pl.persist_ctas = 0;
  p.kv_splits = pl.splits;
  p.work = nullptr;
  p.B = B;
  p.stream_len = pl.stream_len;
  p.epoch = next_epoch();
  const int64_t need = workspace_bytes(B, Hq, Nq, D, causal, pl);
  void* owned = nullptr;
  if (need > 0) {
    if (pool_scratch) {
      if (cudaMallocFromPoolAsync(&owned, static_cast<size_t>(need),
                                  g_pool[dev], s) != cudaSuccess)
        return FA_ERR_CUDA;
      p.work = static_cast<float*>(owned);
    } else {
      if (workspace == nullptr || ws_bytes < static_cast<size_t>(need))
        return FA_ERR_INVALID_VALUE;
      if (!aligned(workspace, 16)) return FA_ERR_MISALIGNED;
      p.work = static_cast<float*>(workspace);
    }
  }

  CUtensorMap tq, tk, tv, to;
  const bool wide = one_tile(D, causal) && pl.persist_ctas == 0;
  const int kv_rows = wide ? fa::WideCfg<256>::kBN : fa::kBN;
  const bool qk_ok =
      qk8 ? (encode_bhnd_e4m3(&tq, q, static_cast<long long>(B) * Hq, Nq,
                              D) == FA_OK &&
             encode_bhnd_e4m3(&tk, k, static_cast<long long>(B) * Hkv, Nkv,
                              D) == FA_OK)
          : (encode_bhnd(&tq, q, static_cast<long long>(B) * Hq, Nq, D) ==
                 FA_OK &&
             encode_bhnd(&tk, k, static_cast<long long>(B) * Hkv, Nkv, D,
                         kv_rows) == FA_OK);
  // O: written by the kernels' TMA stores in boxes of 32 rows
  if ((st = qk_ok ? FA_OK : FA_ERR_CUDA) ||
      (st = encode_bhnd(&tv, v, static_cast<long long>(B) * Hkv, Nkv, D,
                        kv_rows)) ||
      (st = encode_bhnd(&to, o, static_cast<long long>(B) * Hq, Nq, D, 32))) {
    if (owned != nullptr) cudaFreeAsync(owned, s);
    return st;
  }
  if (pl.persist_ctas > 0)
    st = D == 64 ? launch_persist<64>(tq, tk, tv, to, p, pl.persist_ctas, s)
                 : launch_persist<128>(tq, tk, tv, to, p, pl.persist_ctas, s);
  else if (qk8)
    st = causal ? launch<128, true, true>(tq, tk, tv, to, p, B, Hq, Nq, s)
                : launch<128, false, true>(tq, tk, tv, to, p, B, Hq, Nq, s);
  else if (D == 256)
    st = causal ? launch_wide<256, true>(tq, tk, tv, to, p, B, Hq, Nq, s)
                : launch_wide<256, false>(tq, tk, tv, to, p, B, Hq, Nq, s);
  else if (D == 192)
    st = causal ? launch_wide<192, true>(tq, tk, tv, to, p, B, Hq, Nq, s)
                : launch_wide<192, false>(tq, tk, tv, to, p, B, Hq, Nq, s);
  else if (D == 64 && wide)
    st = causal ? launch_wide<64, true>(tq, tk, tv, to, p, B, Hq, Nq, s)
                : launch_wide<64, false>(tq, tk, tv, to, p, B, Hq, Nq, s);
  else if (D == 64)
    st = causal ? launch<64, true>(tq, tk, tv, to, p, B, Hq, Nq, s)
                : launch<64, false>(tq, tk, tv, to, p, B, Hq, Nq, s);
  else
    st = causal ? launch<128, true>(tq, tk, tv, to, p, B, Hq, Nq, s)
                : launch<128, false>(tq, tk, tv, to, p, B, Hq, Nq, s);
  if (owned != nullptr && cudaFreeAsync(owned, s) != cudaSuccess &&
      st == FA_OK)
    st = FA_ERR_CUDA;
  return st;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int Hq, int Hkv, int Nq, int Nkv, int D, float scale,
           int causal, void* stream) {
  return run_forward(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale, causal,
                     nullptr, 0, true, static_cast<cudaStream_t>(stream));
}

int fa_fwd_ws(const void* q, const void* k, const void* v, void* o,
              float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
              float scale, int causal, void* workspace,
              size_t workspace_bytes_, void* stream) {
  return run_forward(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale, causal,
                     workspace, workspace_bytes_, false,
                     static_cast<cudaStream_t>(stream));
}

int fa_fwd_qk8(const void* q8, const void* k8, const void* v, void* o,
               float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
               float scale, float q_descale, float k_descale, int causal,
               void* stream) {
  return run_forward(q8, k8, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale, causal,
                     nullptr, 0, true, static_cast<cudaStream_t>(stream),
                     true, q_descale, k_descale);
}

int fa_fwd_mxfp8(const void* q8, const void* k8, const void* v,
                 const void* q_scale, const void* k_scale, void* o,
                 float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                 float scale, int causal, void* stream) {
  int st = check_args(q8, k8, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale);
  if (st != FA_OK) return st;
  if (q_scale == nullptr || k_scale == nullptr) return FA_ERR_INVALID_VALUE;
  if (D != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned(q_scale, 4) || !aligned(k_scale, 4)) return FA_ERR_MISALIGNED;
  int* word = nullptr;
  int dev = 0;
  if ((st = device_ready(&word, &dev)) != FA_OK) return st;
  fa::FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nkv = Nkv;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) *
                                    1.4426950408889634074);
  p.status = word;
  p.wait_limit_ns = kWaitLimitNs;
  p.kv_splits = 1;
  p.work = nullptr;
  p.B = B;
  p.stream_len = 0;
  p.epoch = next_epoch();
  fa::MxScales sf;
  sf.q_sf = static_cast<const uint32_t*>(q_scale);
  sf.k_sf = static_cast<const uint32_t*>(k_scale);
  CUtensorMap tq, tk, tv, to;
  if ((st = encode_bhnd_e4m3(&tq, q8, static_cast<long long>(B) * Hq, Nq,
                             D)) ||
      (st = encode_bhnd_e4m3(&tk, k8, static_cast<long long>(B) * Hkv, Nkv,
                             D)) ||
      (st = encode_bhnd(&tv, v, static_cast<long long>(B) * Hkv, Nkv, D,
                        fa::kBN)) ||
      (st = encode_bhnd(&to, o, static_cast<long long>(B) * Hq, Nq, D, 32)))
    return st;
  const dim3 grid((Nq + fa::kBM - 1) / fa::kBM, Hq, B);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (causal)
    fa::fa_fwd_mx_kernel<true>
        <<<grid, fa::kMxThreads, fa::MxCfg::kSmemBytes, s>>>(tq, tk, tv, to,
                                                             p, sf);
  else
    fa::fa_fwd_mx_kernel<false>
        <<<grid, fa::kMxThreads, fa::MxCfg::kSmemBytes, s>>>(tq, tk, tv, to,
                                                             p, sf);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                          int causal, size_t* bytes) {
  if (bytes == nullptr) return FA_ERR_INVALID_VALUE;
  *bytes = 0;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || D < 1 ||
      Hq % Hkv != 0 || B > 65535 || Hq > 65535)
    return FA_ERR_INVALID_VALUE;
  if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  const int st = device_ready(nullptr, &dev);
  if (st != FA_OK) return st;
  const RunShape rs = run_shape(Hq, Hkv, Nq, causal);
  *bytes = static_cast<size_t>(workspace_bytes(
      B, rs.Hq, rs.Nq, D, causal,
      plan_forward(B, rs.Hq, Hkv, rs.Nq, Nkv, D, causal, g_sm_count[dev])));
  return FA_OK;
}

int fa_set_schedule(int kind) {
  if (kind != FA_SCHEDULE_AUTO && kind != FA_SCHEDULE_PLAIN &&
      kind != FA_SCHEDULE_STREAM)
    return FA_ERR_INVALID_VALUE;
  g_forced_schedule.store(kind, std::memory_order_relaxed);
  return FA_OK;
}

int fa_fwd_schedule_for(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                        int causal, int sms, int* kind, int* ctas,
                        int* pieces, int* blocks_per_cta,
                        size_t* workspace) {
  if (kind == nullptr || ctas == nullptr || pieces == nullptr ||
      blocks_per_cta == nullptr || workspace == nullptr || sms < 1)
    return FA_ERR_INVALID_VALUE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || D < 1 ||
      Hq % Hkv != 0 || B > 65535 || Hq > 65535)
    return FA_ERR_INVALID_VALUE;
  if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
  const RunShape rs = run_shape(Hq, Hkv, Nq, causal);
  const Plan pl = plan_forward(B, rs.Hq, Hkv, rs.Nq, Nkv, D, causal, sms);
  const int64_t rows_u = unit_rows(D, causal);
  const int64_t units = (rs.Nq + rows_u - 1) / rows_u;
  *kind = pl.stream_len > 0     ? FA_SCHEDULE_STREAM
          : pl.persist_ctas > 0 ? FA_SCHEDULE_PERSIST
          : pl.splits > 1       ? FA_SCHEDULE_SPLIT_KV
                                : FA_SCHEDULE_PLAIN;
  *ctas = pl.stream_len > 0     ? pl.stream_ctas
          : pl.persist_ctas > 0 ? pl.persist_ctas
                                : static_cast<int>(units * rs.Hq * B *
                                                   pl.splits);
  *pieces = pl.splits;
  *blocks_per_cta = pl.stream_len;
  *workspace = static_cast<size_t>(workspace_bytes(B, rs.Hq, rs.Nq, D,
                                                   causal, pl));
  return FA_OK;
}

int fa_fwd_schedule(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                    int causal, int* kind, int* ctas, int* pieces,
                    int* blocks_per_cta) {
  if (kind == nullptr || ctas == nullptr || pieces == nullptr ||
      blocks_per_cta == nullptr)
    return FA_ERR_INVALID_VALUE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || D < 1 ||
      Hq % Hkv != 0 || B > 65535 || Hq > 65535)
    return FA_ERR_INVALID_VALUE;
  if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  const int st = device_ready(nullptr, &dev);
  if (st != FA_OK) return st;
  size_t ws = 0;
  return fa_fwd_schedule_for(B, Hq, Hkv, Nq, Nkv, D, causal, g_sm_count[dev],
                             kind, ctas, pieces, blocks_per_cta, &ws);
}

}  // extern "C"

namespace {

// fa_fwd_host: per-device side streams (host-to-device and device-to-host
// copies) and events, created once; a mutex per device keeps concurrent
// callers' enqueue sequences from interleaving on them.  Chunk count
// measured on GB300 for the 4096 x 8192 x 8-head shape (copy-in 205 us,
// forward 97 us, copy-out 45 us when run alone): 1 chunk 362 us per call,
// 2 chunks 329, 4 chunks 312, 8 chunks 362 (one-head chunks take 39 us each
// on their own, so compute becomes the bottleneck).
constexpr int kHostChunks = 4;
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, d2h_done = nullptr;
  cudaEvent_t in[kHostChunks] = {}, done[kHostChunks] = {};
};
HostPipe g_host_pipe[kMaxDevices];

int host_pipe_init(HostPipe& hp) {
  if (hp.ready) return FA_OK;
  const unsigned fl = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) !=
          cudaSuccess ||
      cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) !=
          cudaSuccess ||
      cudaEventCreateWithFlags(&hp.start, fl) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp.d2h_done, fl) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int c = 0; c < kHostChunks; ++c)
    if (cudaEventCreateWithFlags(&hp.in[c], fl) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.done[c], fl) != cudaSuccess)
      return FA_ERR_CUDA;
  hp.ready = true;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                void* o_host, float* lse_host, void* q_dev, void* k_dev,
                void* v_dev, void* o_dev, float* lse_dev, int B, int Hq,
                int Hkv, int Nq, int Nkv, int D, float scale, int causal,
                void* stream) {
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr ||
      o_host == nullptr || (lse_host == nullptr) != (lse_dev == nullptr))
    return FA_ERR_INVALID_VALUE;
  int st = check_args(q_dev, k_dev, v_dev, o_dev, lse_dev, B, Hq, Hkv, Nq,
                      Nkv, D, scale);
  if (st != FA_OK) return st;
  int dev = 0;
  if ((st = device_ready(nullptr, &dev)) != FA_OK) return st;
  HostPipe& hp = g_host_pipe[dev];
  std::lock_guard<std::mutex> lock(hp.mu);
  if ((st = host_pipe_init(hp)) != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // Chunks of consecutive (batch, kv head) groups: each group's Q, K, V, O
  // and LSE rows are contiguous in the [B, H, N, D] layout, so a chunk is a
  // forward of its own with B = groups, Hq = Hq / Hkv, Hkv = 1.
  const int64_t groups = static_cast<int64_t>(B) * Hkv;
  const int G = Hq / Hkv;
  // At most kHostChunks chunks, more only when a chunk's group count would
  // pass the grid's batch limit (each chunk runs with B = its groups); the
  // chunks then take the events round-robin (each event is waited on before
  // it is recorded again).
  const int64_t min_chunks = (groups + 65534) / 65535;
  const int n_chunks = static_cast<int>(
      min_chunks > kHostChunks ? min_chunks
                               : (groups < kHostChunks ? groups : kHostChunks));
  const int64_t q_group = static_cast<int64_t>(G) * Nq * D * 2;   // bytes
  const int64_t kv_group = static_cast<int64_t>(Nkv) * D * 2;
  const int64_t lse_group = static_cast<int64_t>(G) * Nq * 4;
  auto cptr = [](const void* p, int64_t off) {
    return static_cast<const char*>(p) + off;
  };
  auto mptr = [](void* p, int64_t off) { return static_cast<char*>(p) + off; };
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };

  // The copies start after the caller's earlier work on `stream`.
  if (!ok(cudaEventRecord(hp.start, s)) ||
      !ok(cudaStreamWaitEvent(hp.h2d, hp.start, 0)) ||
      !ok(cudaStreamWaitEvent(hp.d2h, hp.start, 0)))
    return FA_ERR_CUDA;
  // From here on, whatever happens, `stream` is made to wait for both side
  // streams, so synchronising it covers every copy this call enqueued.
  auto join = [&](int status) {
    const bool j = ok(cudaEventRecord(hp.in[0], hp.h2d)) &&
                   ok(cudaStreamWaitEvent(s, hp.in[0], 0)) &&
                   ok(cudaEventRecord(hp.d2h_done, hp.d2h)) &&
                   ok(cudaStreamWaitEvent(s, hp.d2h_done, 0));
    return status != FA_OK ? status : (j ? FA_OK : FA_ERR_CUDA);
  };
  for (int c = 0; c < n_chunks; ++c) {
    const int64_t g0 = groups * c / n_chunks, g1 = groups * (c + 1) / n_chunks;
    const int64_t ng = g1 - g0;
    // in: K and V first (every query row of the chunk needs them), then Q
    const auto h2d = cudaMemcpyHostToDevice;
    if (!ok(cudaMemcpyAsync(mptr(k_dev, g0 * kv_group),
                            cptr(k_host, g0 * kv_group), ng * kv_group, h2d,
                            hp.h2d)) ||
        !ok(cudaMemcpyAsync(mptr(v_dev, g0 * kv_group),
                            cptr(v_host, g0 * kv_group), ng * kv_group, h2d,
                            hp.h2d)) ||
        !ok(cudaMemcpyAsync(mptr(q_dev, g0 * q_group),
                            cptr(q_host, g0 * q_group), ng * q_group, h2d,
                            hp.h2d)) ||
        !ok(cudaEventRecord(hp.in[c % kHostChunks], hp.h2d)) ||
        !ok(cudaStreamWaitEvent(s, hp.in[c % kHostChunks], 0)))
      return join(FA_ERR_CUDA);
    // compute on the caller's stream
    st = run_forward(cptr(q_dev, g0 * q_group), cptr(k_dev, g0 * kv_group),
                     cptr(v_dev, g0 * kv_group), mptr(o_dev, g0 * q_group),
                     lse_dev != nullptr ? reinterpret_cast<float*>(
                                              mptr(lse_dev, g0 * lse_group))
                                        : nullptr,
                     static_cast<int>(ng), G, 1, Nq, Nkv, D, scale, causal,
                     nullptr, 0, true, s);
    if (st != FA_OK) return join(st);
    // out: this chunk's O and LSE while later chunks copy in and compute
    if (!ok(cudaEventRecord(hp.done[c % kHostChunks], s)) ||
        !ok(cudaStreamWaitEvent(hp.d2h, hp.done[c % kHostChunks], 0)) ||
        !ok(cudaMemcpyAsync(mptr(o_host, g0 * q_group),
                            cptr(o_dev, g0 * q_group), ng * q_group,
                            cudaMemcpyDeviceToHost, hp.d2h)))
      return join(FA_ERR_CUDA);
    if (lse_host != nullptr &&
        !ok(cudaMemcpyAsync(mptr(lse_host, g0 * lse_group),
                            cptr(lse_dev, g0 * lse_group), ng * lse_group,
                            cudaMemcpyDeviceToHost, hp.d2h)))
      return join(FA_ERR_CUDA);
  }
  // The caller's stream completes after the last copy out.
  return join(FA_OK);
}

int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                   float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                   float scale, int causal, void* stream) {
  size_t need = 0;
  int st = fa_fwd_workspace_size(B, Hq, Hkv, Nq, Nkv, D, causal, &need);
  if (st != FA_OK) return st;
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_INVALID_VALUE;
  void* scratch = nullptr;
  if (need > 0) {
    int dev = 0;
    if ((st = device_ready(nullptr, &dev)) != FA_OK) return st;
    scratch = g_noalloc_ptr[dev];
    if (scratch == nullptr) return FA_ERR_CUDA;
  }
  return fa_fwd_ws(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale, causal,
                   scratch, need, stream);
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_VALUE: return "FA_ERR_INVALID_VALUE";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_last_device_error(void) {
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_fa_status, sizeof(int)) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(int)) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return word;
}

int fa_probe_bounded_wait(long long timeout_ns, void* stream) {
  if (timeout_ns < 1 || timeout_ns > 1000000000ll) return FA_ERR_INVALID_VALUE;
  int* word = nullptr;
  int st = device_ready(&word);
  if (st != FA_OK) return st;
  probe_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      word, static_cast<uint64_t>(timeout_ns));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_probe_flag_wait(long long timeout_ns, void* stream) {
  if (timeout_ns < 1 || timeout_ns > 1000000000ll) return FA_ERR_INVALID_VALUE;
  int* word = nullptr;
  int st = device_ready(&word);
  if (st != FA_OK) return st;
  probe_flag_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      word, static_cast<uint64_t>(timeout_ns));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_version(void) { return 100; }

size_t fa_tensor_map_encodes(void) {
  return g_map_encodes.load(std::memory_order_relaxed);
}

}  // extern "C"
