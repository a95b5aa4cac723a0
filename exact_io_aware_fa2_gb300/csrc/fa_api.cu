// fa_api.cu — host side of the C ABI declared in include/fa.h: argument
// validation, TMA tensor-map encoding, kernel selection and launch.
//
// The operation and its sources are described in include/fa.h.  This file
// holds no arithmetic of the method; it only prepares the launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_fwd_kernel.cuh"

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

template <int D, bool CAUSAL>
cudaError_t opt_in_smem() {
  return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, CAUSAL>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa::FwdCfg<D>::kSmemBytes);
}

int* g_status_word[kMaxDevices];

// Per-device readiness: compute capability 10.3, the kernels' shared memory
// opt-in and the device address of the status word, done once per device
// with that device current.
int device_ready(int** word_out) {
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
      return;
    }
    if (major != 10 || minor != 3) {
      status[dev] = FA_ERR_UNSUPPORTED;
      return;
    }
    if (opt_in_smem<64, false>() != cudaSuccess ||
        opt_in_smem<64, true>() != cudaSuccess ||
        opt_in_smem<128, false>() != cudaSuccess ||
        opt_in_smem<128, true>() != cudaSuccess) {
      status[dev] = FA_ERR_CUDA;
      return;
    }
    void* word = nullptr;
    if (cudaGetSymbolAddress(&word, fa::g_fa_status) != cudaSuccess) {
      status[dev] = FA_ERR_CUDA;
      return;
    }
    g_status_word[dev] = static_cast<int*>(word);
    status[dev] = FA_OK;
  });
  if (status[dev] == FA_OK && word_out != nullptr) *word_out = g_status_word[dev];
  return status[dev];
}

// Tensor map of a contiguous bf16 [BH, N, D] tensor, read in 64 x 128 boxes
// (64 head-dim elements = one 128-byte swizzle row, 128 sequence rows) with
// the 128-byte swizzle.  Rows past N are zero-filled by the TMA unit.
int encode_bhnd(CUtensorMap* map, const void* ptr, long long BH, int N,
                int D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(N) * D * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(fa::kBoxCols),
                       static_cast<cuuint32_t>(fa::kBM), 1};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool CAUSAL>
int launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
           const fa::FwdParams& p, int B, int Hq, int Nq,
           cudaStream_t stream) {
  const int rows_per_cta = fa::kBM * fa::kTilesPerCta;
  dim3 grid((Nq + rows_per_cta - 1) / rows_per_cta, Hq, B);
  fa::fa_fwd_kernel<D, CAUSAL>
      <<<grid, fa::kThreads, fa::FwdCfg<D>::kSmemBytes, stream>>>(q, k, v, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

__global__ void probe_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(fa::smem_addr(&bar_mem), 1);
    abort_flag = 0;
    fa::mbar_init_fence();
    // Nothing arrives on this barrier: the wait must run out.
    const fa::WaitCtx wc{&abort_flag, status, limit_ns};
    fa::mbar_wait(fa::smem_addr(&bar_mem), 0, wc);
  }
  __syncwarp();
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int Hq, int Hkv, int Nq, int Nkv, int D, float scale,
           int causal, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr)
    return FA_ERR_INVALID_VALUE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || D < 1)
    return FA_ERR_INVALID_VALUE;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_VALUE;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_VALUE;
  if (B > 65535 || Hq > 65535) return FA_ERR_INVALID_VALUE;  // grid limits
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || (lse != nullptr && !aligned(lse, 4)))
    return FA_ERR_MISALIGNED;

  int* word = nullptr;
  int st = device_ready(&word);
  if (st != FA_OK) return st;

  CUtensorMap tq, tk, tv;
  if ((st = encode_bhnd(&tq, q, static_cast<long long>(B) * Hq, Nq, D)) ||
      (st = encode_bhnd(&tk, k, static_cast<long long>(B) * Hkv, Nkv, D)) ||
      (st = encode_bhnd(&tv, v, static_cast<long long>(B) * Hkv, Nkv, D)))
    return st;

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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 64)
    return causal ? launch<64, true>(tq, tk, tv, p, B, Hq, Nq, s)
                  : launch<64, false>(tq, tk, tv, p, B, Hq, Nq, s);
  return causal ? launch<128, true>(tq, tk, tv, p, B, Hq, Nq, s)
                : launch<128, false>(tq, tk, tv, p, B, Hq, Nq, s);
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

int fa_version(void) { return 100; }

}  // extern "C"
