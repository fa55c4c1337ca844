// tq_noalloc.cu -- tq_gemm_noalloc: the prefill GEMM for callers that cannot
// allocate device memory.
//
// tq_gemm needs a workspace (the rotated activations in fp16 plus a status
// word) that the caller allocates.  Some callers cannot call cudaMalloc at
// all -- code running inside a fixed memory pool or arena, plugins that get
// their buffers from a host framework and are not allowed to allocate on
// their own, or code paths that must not reach the allocator at all.  For
// them this entry point takes its workspace from a fixed array that lives in
// the library's own device memory.  The caller still passes the inputs and
// the output.
//
// The array is a file-scope __device__ object of kScratchBytes, so every GPU
// that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, not a device address; its device
// address is looked up with cudaGetSymbolAddress, with the device current, on
// every call (a host-side query that allocates nothing; looking it up each
// time keeps a stale address from outliving a reset of the device).  The
// first call on a device also loads the library's module there (set-up).
//
// The GEMM records a bounded wait that ran out in the status word at the
// start of the array; tq_device_fault reads that word on every device where
// this entry point has been used.
#include <atomic>

#include "tq_internal.h"

namespace tq {

namespace {

// 256-byte status word area + fp16 rotated activations for M * K <= 2^24.
constexpr size_t kScratchBytes = 256 + ((size_t)1 << 24) * 2;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<int> g_used[kMaxDevices];  // tq_gemm_noalloc has launched on this device

// Device address of g_scratch on the current device (nullptr on failure).
void* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return p;
}

}  // namespace

// Reads the status word of the scratch array on the current device when this
// entry point has run there; returns kFaultTimeout-style bit 1 when a bounded
// wait of the GEMM ran out, and clears that bit.  Called after a device-wide
// synchronisation.
unsigned int take_fault_noalloc() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (g_used[dev].load(std::memory_order_acquire) == 0) return 0;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_scratch, sizeof(w)) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (!(w & 2u)) return 0;
  w &= ~2u;
  (void)cudaMemcpyToSymbol(g_scratch, &w, sizeof(w));
  return 2u;
}

}  // namespace tq

using namespace tq;

extern "C" TQ_API tq_status tq_gemm_noalloc(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales,
                                             int64_t lds, int64_t N, int64_t K, const void* x, int64_t ldx, int64_t M,
                                             float* y, int64_t ldy, tq_stream stream) {
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return TQ_ERR_INVALID_ARG;
  if (N < 0 || M < 0) return TQ_ERR_INVALID_ARG;
  if (K <= 0 || K % 128 != 0) return TQ_ERR_SHAPE;
  if (N == 0 || M == 0) return TQ_OK;
  if (fmt != TQ_PACK_2BIT) return TQ_ERR_UNSUPPORTED;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
  if (ldc < K / 4 || lds < K / 128 || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  // the rotated activations must fit the fixed scratch array
  if (M > (int64_t)((kScratchBytes - 256) / 2) / K) return TQ_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(codes) & 15u) || ldc % 16 || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(x) & 15u) || (ldx * 2) % 16 || (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  unsigned char* ws = static_cast<unsigned char*>(scratch_on_current_device());
  if (ws == nullptr) return TQ_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) g_used[dev].store(1, std::memory_order_release);
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* flag = reinterpret_cast<uint32_t*>(ws);
  uint16_t* xrot = reinterpret_cast<uint16_t*>(ws + 256);
  // the array keeps the previous call's contents: clear the status word
  if (cudaMemsetAsync(flag, 0, sizeof(uint32_t), s) != cudaSuccess) return TQ_ERR_CUDA;
  cudaError_t e = launch_fwht128(x, TQ_BF16, ldx, xrot, TQ_F16, K, M, K, true, flag, s);
  // no room for the partial tiles of a K-split last wave: whole tiles only
  if (e == cudaSuccess) e = launch_gemm(codes, ldc, scales, lds, N, K, xrot, M, y, ldy, flag, nullptr, 0, s);
  if (e == cudaSuccess) return TQ_OK;
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    return TQ_ERR_UNSUPPORTED;
  }
  return TQ_ERR_CUDA;
}
