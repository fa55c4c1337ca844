// tq_api.cu -- the C ABI of libtq: host-side validation, then one launch (or
// two for tq_gemm) on the caller's stream.  No entry point allocates memory,
// throws, aborts or synchronises (except tq_gemm_check_range, which must).
#include <atomic>
#include <cstring>

#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_smem[kMaxDevices];

int cached_attr(std::atomic<int>* cache, cudaDeviceAttr attr, int fallback) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fallback;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v <= 0) return fallback;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

int dtype_size(int t) { return t == TQ_F32 ? 4 : 2; }

bool k_ok(int64_t K) { return K > 0 && K % 128 == 0; }

tq_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TQ_OK;
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();  // clear a sticky launch-config error, if any
    return TQ_ERR_UNSUPPORTED;
  }
  return TQ_ERR_CUDA;
}

int64_t ld3_min(int64_t K) { return ((K + 4) / 5 + 15) / 16 * 16; }

}  // namespace

int device_sm_count() { return cached_attr(g_sms, cudaDevAttrMultiProcessorCount, 148); }
int device_max_smem_optin() { return cached_attr(g_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, 227 * 1024); }

}  // namespace tq

using namespace tq;

extern "C" {

const char* tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG: null pointer, bad enum or negative size";
    case TQ_ERR_SHAPE: return "TQ_ERR_SHAPE: K must be a positive multiple of 128; M or a leading dimension out of range";
    case TQ_ERR_ALIGN: return "TQ_ERR_ALIGN: pointer or row start not 16-byte aligned";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED: format/dtype/shape combination not provided";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA: a CUDA call failed";
    case TQ_ERR_RANGE: return "TQ_ERR_RANGE: a rotated activation overflowed fp16";
    case TQ_ERR_TIMEOUT: return "TQ_ERR_TIMEOUT: a kernel gave up a bounded wait; its outputs are not meaningful";
    default: return "unknown tq_status";
  }
}

int tq_version(void) { return 100; }

int64_t tq_packed_ld(int64_t K, int fmt) {
  if (K <= 0) return -1;
  if (fmt == TQ_PACK_2BIT) return K % 4 == 0 ? K / 4 : -1;
  if (fmt == TQ_PACK_BASE3) return ld3_min(K);
  return -1;
}

tq_status tq_fwht128(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows, int64_t K,
                     tq_stream stream) {
  if (xt != TQ_F32 && xt != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (yt != TQ_F32 && yt != TQ_BF16 && yt != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (rows < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K)) return TQ_ERR_SHAPE;
  if (rows == 0) return TQ_OK;
  if (x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
  if (ldx < K || ldy < K) return TQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(y) || (ldx * dtype_size(xt)) % 16 || (ldy * dtype_size(yt)) % 16)
    return TQ_ERR_ALIGN;
  if (x == y && (xt != yt || ldx != ldy)) return TQ_ERR_INVALID_ARG;
  return from_cuda(launch_fwht128(x, xt, ldx, y, yt, ldy, rows, K, false, nullptr, (cudaStream_t)stream));
}

tq_status tq_quantize_pack(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt, uint8_t* codes2,
                           int64_t ld2, uint8_t* codes3, int64_t ld3, uint16_t* scales, int64_t lds,
                           tq_stream stream) {
  if (wt != TQ_F32 && wt != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3 && fmt != TQ_PACK_BOTH) return TQ_ERR_INVALID_ARG;
  if (N < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K)) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  const bool do2 = (fmt & TQ_PACK_2BIT) != 0, do3 = (fmt & TQ_PACK_BASE3) != 0;
  if (W == nullptr || scales == nullptr || (do2 && codes2 == nullptr) || (do3 && codes3 == nullptr))
    return TQ_ERR_INVALID_ARG;
  if (ldw < K || lds < K / 128 || (do2 && ld2 < K / 4) || (do3 && ld3 < ld3_min(K))) return TQ_ERR_SHAPE;
  if (!aligned16(W) || (ldw * dtype_size(wt)) % 16 || !aligned2(scales)) return TQ_ERR_ALIGN;
  return from_cuda(launch_quantize_pack(W, wt, N, K, ldw, fmt, do2 ? codes2 : nullptr, ld2, do3 ? codes3 : nullptr,
                                        ld3, scales, lds, (cudaStream_t)stream));
}

namespace {
// Validation shared by tq_gemv_ex and tq_gemv_rotate_next (x is bf16, or the
// fp32 rotated x with TQ_GEMV_X_ROTATED).
tq_status gemv_check(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                     int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, unsigned int flags) {
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return TQ_ERR_INVALID_ARG;
  if (flags & ~(unsigned int)(TQ_GEMV_WEIGHTS_READY | TQ_GEMV_X_ROTATED | TQ_GEMV_TEST_STALL))
    return TQ_ERR_INVALID_ARG;
  if (N < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K) || M < 1 || M > 16) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
  if (ldc < tq_packed_ld(K, fmt) || lds < K / 128 || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  const bool xrot = (flags & TQ_GEMV_X_ROTATED) != 0;
  const bool x_ok = xrot ? (reinterpret_cast<uintptr_t>(x) & 3u) == 0 : (aligned16(x) && (ldx * 2) % 16 == 0);
  if (!aligned16(codes) || ldc % 16 || !aligned2(scales) || !x_ok || (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  return TQ_OK;
}
}  // namespace

tq_status tq_gemv_ex(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                     int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, unsigned int flags,
                     tq_stream stream) {
  const tq_status st = gemv_check(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, flags);
  if (st != TQ_OK || N == 0) return st;
  if (flags & TQ_GEMV_X_ROTATED) {  // the tensor-memory kernel reads the fp32 x'
    if (tq::gemv_tc_launches(N, K, M, fmt) == 0) return TQ_ERR_UNSUPPORTED;
    const GemvChain ch{static_cast<const float*>(x), ldx, nullptr, 0};
    return from_cuda(launch_gemv_tc(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy,
                                    (flags & TQ_GEMV_WEIGHTS_READY) != 0, (cudaStream_t)stream,
                                    (flags & TQ_GEMV_TEST_STALL) != 0, nullptr, &ch));
  }
  if (flags & TQ_GEMV_TEST_STALL) {  // only the tensor-memory kernel has waits to stall
    if (tq::gemv_tc_launches(N, K, M, fmt) == 0) return TQ_ERR_UNSUPPORTED;
    return from_cuda(launch_gemv_tc(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy,
                                    (flags & TQ_GEMV_WEIGHTS_READY) != 0, (cudaStream_t)stream, true));
  }
  return from_cuda(launch_gemv(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy,
                               (flags & TQ_GEMV_WEIGHTS_READY) != 0, (cudaStream_t)stream));
}

tq_status tq_gemv_rotate_next(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds,
                              int64_t N, int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                              unsigned int flags, float* xnext, int64_t ldxn, tq_stream stream) {
  const tq_status st = gemv_check(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, flags);
  if (st != TQ_OK) return st;
  if (N % 128 != 0) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  if (xnext == nullptr) return TQ_ERR_INVALID_ARG;
  if (ldxn < N) return TQ_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(xnext) & 3u) return TQ_ERR_ALIGN;
  const bool xrot = (flags & TQ_GEMV_X_ROTATED) != 0;
  const uintptr_t xn0 = reinterpret_cast<uintptr_t>(xnext), xn1 = xn0 + (uintptr_t)((M - 1) * ldxn + N) * 4;
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(y), y1 = y0 + (uintptr_t)((M - 1) * ldy + N) * 4;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), x1 = x0 + (uintptr_t)((M - 1) * ldx + K) * (xrot ? 4 : 2);
  if ((xn0 < y1 && y0 < xn1) || (xn0 < x1 && x0 < xn1)) return TQ_ERR_INVALID_ARG;
  if (tq::gemv_tc_launches(N, K, M, fmt, true) == 0) return TQ_ERR_UNSUPPORTED;
  const GemvChain ch{xrot ? static_cast<const float*>(x) : nullptr, ldx, xnext, ldxn};
  return from_cuda(launch_gemv_tc(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy,
                                  (flags & TQ_GEMV_WEIGHTS_READY) != 0, (cudaStream_t)stream,
                                  (flags & TQ_GEMV_TEST_STALL) != 0, nullptr, &ch));
}

tq_status tq_gemv(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                  int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, tq_stream stream) {
  return tq_gemv_ex(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, 0u, stream);
}

int tq_gemv_path(int64_t N, int64_t K, int64_t M, int fmt) {
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return -(int)TQ_ERR_INVALID_ARG;
  if (N < 0) return -(int)TQ_ERR_INVALID_ARG;
  if (!k_ok(K) || M < 1 || M > 16) return -(int)TQ_ERR_SHAPE;
  if (tq::gemv_tc_launches(N, K, M, fmt) > 0) return TQ_GEMV_TENSOR_MEMORY;
  return TQ_GEMV_MMA_SYNC;
}

tq_status tq_gemv_plan(int64_t N, int64_t K, int64_t M, int fmt, int chained, int* ctas_per_cluster, int* clusters,
                       int* launches) {
  if (ctas_per_cluster == nullptr || clusters == nullptr || launches == nullptr) return TQ_ERR_INVALID_ARG;
  const int path = tq_gemv_path(N, K, M, fmt);
  if (path < 0) return (tq_status)(-path);
  if (chained && N % 128 != 0) return TQ_ERR_SHAPE;
  const int l = tq::gemv_tc_launches(N, K, M, fmt, chained != 0);
  if (l < 1) return TQ_ERR_UNSUPPORTED;
  if (!tq::plan_gemv_tc(N, K, M / l, fmt, ctas_per_cluster, clusters, chained != 0)) return TQ_ERR_UNSUPPORTED;
  *launches = l;
  return TQ_OK;
}

namespace {
// start of the split-partial area of a tq_gemm workspace (256-byte aligned)
size_t gemm_split_offset(int64_t M, int64_t K) { return (256 + (size_t)M * (size_t)K * 2 + 255) / 256 * 256; }
}  // namespace

size_t tq_gemm_workspace_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  // status word, rotated activations (fp16), then the partial tiles of a K-split last wave
  return gemm_split_offset(M, K) + tq::kGemmSplitBytes;
}

tq_status tq_gemm(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                  int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, void* workspace,
                  size_t ws_bytes, tq_stream stream) {
  return tq_gemm_ex(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, workspace, ws_bytes, 0u, stream);
}

tq_status tq_gemm_ex(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                     int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, void* workspace,
                     size_t ws_bytes, unsigned int flags, tq_stream stream) {
  if (flags & ~(unsigned int)(TQ_GEMM_REUSE_ROTATED | TQ_GEMM_TEST_STALL)) return TQ_ERR_INVALID_ARG;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return TQ_ERR_INVALID_ARG;
  if (N < 0 || M < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K)) return TQ_ERR_SHAPE;
  if (N == 0 || M == 0) return TQ_OK;
  if (fmt != TQ_PACK_2BIT) return TQ_ERR_UNSUPPORTED;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr || workspace == nullptr)
    return TQ_ERR_INVALID_ARG;
  if (ldc < K / 4 || lds < K / 128 || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  if (ws_bytes < tq_gemm_workspace_bytes(M, K)) return TQ_ERR_SHAPE;
  if (!aligned16(codes) || ldc % 16 || !aligned2(scales) || !aligned16(x) || (ldx * 2) % 16 ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* flag = static_cast<uint32_t*>(workspace);
  uint16_t* xrot = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(workspace) + 256);
  if (!(flags & TQ_GEMM_REUSE_ROTATED)) {  // else x' (and its status) are the previous call's
    cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
    e = launch_fwht128(x, TQ_BF16, ldx, xrot, TQ_F16, K, M, K, true, flag, s);
    if (e != cudaSuccess) return from_cuda(e);
  }
  unsigned char* split = static_cast<unsigned char*>(workspace) + gemm_split_offset(M, K);
  return from_cuda(launch_gemm(codes, ldc, scales, lds, N, K, xrot, M, y, ldy, flag, split,
                               ws_bytes - gemm_split_offset(M, K), s, (flags & TQ_GEMM_TEST_STALL) != 0));
}

tq_status tq_gemm_rotate_next(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds,
                              int64_t N, int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                              void* workspace, size_t ws_bytes, unsigned int flags, void* next_ws,
                              size_t next_ws_bytes, tq_stream stream) {
  if (flags & ~(unsigned int)(TQ_GEMM_REUSE_ROTATED | TQ_GEMM_TEST_STALL)) return TQ_ERR_INVALID_ARG;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return TQ_ERR_INVALID_ARG;
  if (N < 0 || M < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K) || N % 128 != 0) return TQ_ERR_SHAPE;
  if (N == 0 || M == 0) return TQ_OK;
  if (fmt != TQ_PACK_2BIT) return TQ_ERR_UNSUPPORTED;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr || workspace == nullptr ||
      next_ws == nullptr)
    return TQ_ERR_INVALID_ARG;
  if (ldc < K / 4 || lds < K / 128 || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  if (ws_bytes < tq_gemm_workspace_bytes(M, K) || next_ws_bytes < tq_gemm_workspace_bytes(M, N)) return TQ_ERR_SHAPE;
  if (!aligned16(codes) || ldc % 16 || !aligned2(scales) || !aligned16(x) || (ldx * 2) % 16 ||
      !aligned16(workspace) || !aligned16(next_ws) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(workspace), b0 = reinterpret_cast<uintptr_t>(next_ws);
  if (a0 < b0 + next_ws_bytes && b0 < a0 + ws_bytes) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* flag = static_cast<uint32_t*>(workspace);
  uint16_t* xrot = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(workspace) + 256);
  uint32_t* flag_next = static_cast<uint32_t*>(next_ws);
  uint16_t* xnext = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(next_ws) + 256);
  cudaError_t e = cudaMemsetAsync(flag_next, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return TQ_ERR_CUDA;
  if (!(flags & TQ_GEMM_REUSE_ROTATED)) {
    e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
    e = launch_fwht128(x, TQ_BF16, ldx, xrot, TQ_F16, K, M, K, true, flag, s);
    if (e != cudaSuccess) return from_cuda(e);
  }
  unsigned char* split = static_cast<unsigned char*>(workspace) + gemm_split_offset(M, K);
  return from_cuda(launch_gemm(codes, ldc, scales, lds, N, K, xrot, M, y, ldy, flag, split,
                               ws_bytes - gemm_split_offset(M, K), s, (flags & TQ_GEMM_TEST_STALL) != 0, 128,
                               xnext, flag_next));
}

tq_status tq_gemm_check_range(const void* workspace, tq_stream stream) {
  if (workspace == nullptr) return TQ_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return TQ_ERR_ALIGN;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TQ_ERR_CUDA;
  uint32_t flag = 0;
  if (cudaMemcpy(&flag, workspace, sizeof(flag), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ERR_CUDA;
  if (flag & 2u) return TQ_ERR_TIMEOUT;
  return (flag & 1u) ? TQ_ERR_RANGE : TQ_OK;
}

}  // extern "C"

namespace {

// A checked layout: returns TQ_OK and fills the fields, or the status a call
// with it returns.
struct Lay {
  int block = 128, group = 128, residual = 0;
  bool plain() const { return block == 128 && group == 128 && residual == 0; }
  int64_t keff(int64_t K) const { return residual ? 2 * K : K; }
  int64_t geff(int64_t K) const { return (residual ? 2 : 1) * (K / group); }
};

tq_status read_layout(const tq_layout* lay, Lay* out) {
  Lay L;
  if (lay != nullptr) {
    if (lay->block != 64 && lay->block != 128 && lay->block != 256) return TQ_ERR_INVALID_ARG;
    if (lay->group != 128 && lay->group != 256) return TQ_ERR_INVALID_ARG;
    if (lay->flags & ~(uint32_t)TQ_LAYOUT_RESIDUAL) return TQ_ERR_INVALID_ARG;
    L.block = lay->block;
    L.group = lay->group;
    L.residual = (lay->flags & TQ_LAYOUT_RESIDUAL) ? 1 : 0;
  }
  *out = L;
  return TQ_OK;
}

bool k_fits(int64_t K, const Lay& L) { return k_ok(K) && K % L.block == 0 && K % L.group == 0; }

}  // namespace

extern "C" {

int64_t tq_layout_codes_ld(int64_t K, int fmt, const tq_layout* lay) {
  Lay L;
  if (read_layout(lay, &L) != TQ_OK || !k_fits(K, L)) return -1;
  return tq_packed_ld(L.keff(K), fmt);
}

int64_t tq_layout_scales_ld(int64_t K, const tq_layout* lay) {
  Lay L;
  if (read_layout(lay, &L) != TQ_OK || !k_fits(K, L)) return -1;
  return L.geff(K);
}

tq_status tq_fwht(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows, int64_t K,
                  int block, tq_stream stream) {
  if (block != 64 && block != 128 && block != 256) return TQ_ERR_INVALID_ARG;
  if (block == 128) return tq_fwht128(x, xt, ldx, y, yt, ldy, rows, K, stream);
  if (xt != TQ_F32 && xt != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (yt != TQ_F32 && yt != TQ_BF16 && yt != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (rows < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K) || K % block) return TQ_ERR_SHAPE;
  if (rows == 0) return TQ_OK;
  if (x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
  if (ldx < K || ldy < K) return TQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(y) || (ldx * dtype_size(xt)) % 16 || (ldy * dtype_size(yt)) % 16)
    return TQ_ERR_ALIGN;
  if (x == y && (xt != yt || ldx != ldy)) return TQ_ERR_INVALID_ARG;
  return from_cuda(launch_fwht(x, xt, ldx, y, yt, ldy, rows, K, block, false, nullptr, (cudaStream_t)stream));
}

tq_status tq_quantize_pack_layout(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt,
                                  uint8_t* codes2, int64_t ld2, uint8_t* codes3, int64_t ld3, uint16_t* scales,
                                  int64_t lds, const tq_layout* lay, tq_stream stream) {
  Lay L;
  const tq_status st = read_layout(lay, &L);
  if (st != TQ_OK) return st;
  if (L.plain()) return tq_quantize_pack(W, wt, N, K, ldw, fmt, codes2, ld2, codes3, ld3, scales, lds, stream);
  if (wt != TQ_F32 && wt != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3 && fmt != TQ_PACK_BOTH) return TQ_ERR_INVALID_ARG;
  if (N < 0) return TQ_ERR_INVALID_ARG;
  if (!k_fits(K, L)) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  const bool do2 = (fmt & TQ_PACK_2BIT) != 0, do3 = (fmt & TQ_PACK_BASE3) != 0;
  if (W == nullptr || scales == nullptr || (do2 && codes2 == nullptr) || (do3 && codes3 == nullptr))
    return TQ_ERR_INVALID_ARG;
  const int64_t Ke = L.keff(K);
  if (ldw < K || lds < L.geff(K) || (do2 && ld2 < Ke / 4) || (do3 && ld3 < ld3_min(Ke))) return TQ_ERR_SHAPE;
  if (!aligned16(W) || (ldw * dtype_size(wt)) % 16 || !aligned2(scales)) return TQ_ERR_ALIGN;
  return from_cuda(launch_quantize_layout(W, wt, N, K, ldw, L.block, L.group, L.residual, do2 ? codes2 : nullptr,
                                          ld2, do3 ? codes3 : nullptr, ld3, scales, lds, (cudaStream_t)stream));
}

tq_status tq_gemv_layout(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                         int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                         const tq_layout* lay, unsigned int flags, tq_stream stream) {
  Lay L;
  const tq_status st = read_layout(lay, &L);
  if (st != TQ_OK) return st;
  if (L.plain()) return tq_gemv_ex(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, flags, stream);
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return TQ_ERR_INVALID_ARG;
  if (flags & ~(unsigned int)(TQ_GEMV_WEIGHTS_READY | TQ_GEMV_TEST_STALL)) return TQ_ERR_INVALID_ARG;
  if (N < 0) return TQ_ERR_INVALID_ARG;
  if (!k_fits(K, L) || M < 1 || M > 16) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
  const int64_t Ke = L.keff(K);
  if (ldc < tq_packed_ld(Ke, fmt) || lds < L.geff(K) || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  if (!aligned16(codes) || ldc % 16 || !aligned2(scales) || !aligned16(x) || (ldx * 2) % 16 ||
      (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  if (tq::gemv_tc_launches(N, Ke, M, fmt) == 0) return TQ_ERR_UNSUPPORTED;
  const GemvLayout gl{L.block, L.group, L.residual};
  return from_cuda(launch_gemv_tc(codes, ldc, fmt, scales, lds, N, Ke, x, ldx, M, y, ldy,
                                  (flags & TQ_GEMV_WEIGHTS_READY) != 0, (cudaStream_t)stream,
                                  (flags & TQ_GEMV_TEST_STALL) != 0, &gl));
}

size_t tq_gemm_workspace_bytes_layout(int64_t M, int64_t K, const tq_layout* lay) {
  Lay L;
  if (read_layout(lay, &L) != TQ_OK || M < 0 || K < 0) return 0;
  return tq_gemm_workspace_bytes(M, L.keff(K));
}

tq_status tq_gemm_layout(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                         int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, void* workspace,
                         size_t ws_bytes, const tq_layout* lay, unsigned int flags, tq_stream stream) {
  Lay L;
  const tq_status st = read_layout(lay, &L);
  if (st != TQ_OK) return st;
  if (L.plain())
    return tq_gemm_ex(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, workspace, ws_bytes, flags, stream);
  if (flags & ~(unsigned int)(TQ_GEMM_REUSE_ROTATED | TQ_GEMM_TEST_STALL)) return TQ_ERR_INVALID_ARG;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return TQ_ERR_INVALID_ARG;
  if (N < 0 || M < 0) return TQ_ERR_INVALID_ARG;
  if (!k_fits(K, L)) return TQ_ERR_SHAPE;
  if (N == 0 || M == 0) return TQ_OK;
  if (fmt != TQ_PACK_2BIT) return TQ_ERR_UNSUPPORTED;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr || workspace == nullptr)
    return TQ_ERR_INVALID_ARG;
  const int64_t Ke = L.keff(K);
  if (ldc < Ke / 4 || lds < L.geff(K) || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  if (ws_bytes < tq_gemm_workspace_bytes(M, Ke)) return TQ_ERR_SHAPE;
  if (!aligned16(codes) || ldc % 16 || !aligned2(scales) || !aligned16(x) || (ldx * 2) % 16 ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* flag = static_cast<uint32_t*>(workspace);
  uint16_t* xrot = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(workspace) + 256);
  if (!(flags & TQ_GEMM_REUSE_ROTATED)) {
    cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
    e = launch_fwht(x, TQ_BF16, ldx, xrot, TQ_F16, Ke, M, K, L.block, true, flag, s);
    // the residual pass meets x itself: converted and laid out the same way
    if (e == cudaSuccess && L.residual) e = launch_fwht(x, TQ_BF16, ldx, xrot + K, TQ_F16, Ke, M, K, 0, true, flag, s);
    if (e != cudaSuccess) return from_cuda(e);
  }
  unsigned char* split = static_cast<unsigned char*>(workspace) + gemm_split_offset(M, Ke);
  return from_cuda(launch_gemm(codes, ldc, scales, lds, N, Ke, xrot, M, y, ldy, flag, split,
                               ws_bytes - gemm_split_offset(M, Ke), s, (flags & TQ_GEMM_TEST_STALL) != 0, L.group));
}

int64_t tq_sparse24_ld(int64_t K) { return k_ok(K) ? 24 * (K / 128) : -1; }

tq_status tq_quantize_pack_sparse24(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, uint8_t* codes,
                                    int64_t ldc, uint16_t* scales, int64_t lds, tq_stream stream) {
  if (wt != TQ_F32 && wt != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (N < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K)) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  if (W == nullptr || codes == nullptr || scales == nullptr) return TQ_ERR_INVALID_ARG;
  if (ldw < K || ldc < tq_sparse24_ld(K) || lds < K / 128) return TQ_ERR_SHAPE;
  if (!aligned16(W) || (ldw * dtype_size(wt)) % 16 || (reinterpret_cast<uintptr_t>(codes) & 3u) || ldc % 4 ||
      !aligned2(scales))
    return TQ_ERR_ALIGN;
  return from_cuda(launch_quantize_sparse24(W, wt, N, K, ldw, codes, ldc, scales, lds, (cudaStream_t)stream));
}

size_t tq_gemv_sparse24_workspace_bytes(int64_t N, int64_t K, int64_t M) {
  if (N < 0 || !k_ok(K) || M < 1 || M > 16) return 0;
  return sparse24_gemv_workspace(N, K, M);
}

tq_status tq_gemv_sparse24(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N,
                           int64_t K, const uint16_t* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                           void* workspace, size_t ws_bytes, tq_stream stream) {
  if (N < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K) || M < 1 || M > 16) return TQ_ERR_SHAPE;
  if (N == 0) return TQ_OK;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr || workspace == nullptr)
    return TQ_ERR_INVALID_ARG;
  if (ldc < tq_sparse24_ld(K) || lds < K / 128 || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  if (ws_bytes < sparse24_gemv_workspace(N, K, M)) return TQ_ERR_SHAPE;
  if (!aligned16(x) || (ldx * 2) % 16 || !aligned2(scales) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(y) & 3u) || (reinterpret_cast<uintptr_t>(codes) & 3u) || ldc % 4)
    return TQ_ERR_ALIGN;
  // the tensor-memory kernel when the codes suit its copies (16-byte aligned
  // rows; an even number of groups per row, at least four), else the
  // zero-skipping kernel on the CUDA cores
  if (aligned16(codes) && ldc % 16 == 0 && tq_gemv_sparse24_path(N, K, M) == TQ_GEMV_TENSOR_MEMORY)
    return from_cuda(launch_gemv_tc(codes, ldc, kFmtSparse24, scales, lds, N, K, x, ldx, M, y, ldy, false,
                                    (cudaStream_t)stream));
  return from_cuda(launch_gemv_sparse24(codes, ldc, scales, lds, N, K, x, ldx, M, y, ldy, workspace,
                                        (cudaStream_t)stream));
}

int tq_gemv_sparse24_path(int64_t N, int64_t K, int64_t M) {
  if (N < 0) return -TQ_ERR_INVALID_ARG;
  if (!k_ok(K) || M < 1 || M > 16) return -TQ_ERR_SHAPE;
  return tq::gemv_tc_launches(N, K, M, kFmtSparse24) > 0 ? TQ_GEMV_TENSOR_MEMORY : TQ_GEMV_CUDA_CORES;
}

tq_status tq_gemm_sparse24(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N,
                           int64_t K, const uint16_t* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                           void* workspace, size_t ws_bytes, tq_stream stream) {
  if (N < 0 || M < 0) return TQ_ERR_INVALID_ARG;
  if (!k_ok(K)) return TQ_ERR_SHAPE;
  if (N == 0 || M == 0) return TQ_OK;
  if (codes == nullptr || scales == nullptr || x == nullptr || y == nullptr || workspace == nullptr)
    return TQ_ERR_INVALID_ARG;
  if (ldc < tq_sparse24_ld(K) || lds < K / 128 || ldx < K || ldy < N) return TQ_ERR_SHAPE;
  if (ws_bytes < tq_gemm_workspace_bytes(M, K)) return TQ_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(codes) & 7u) || ldc % 8 || !aligned2(scales) || !aligned16(x) || (ldx * 2) % 16 ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return TQ_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* flag = static_cast<uint32_t*>(workspace);
  uint16_t* xrot = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(workspace) + 256);
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return TQ_ERR_CUDA;
  e = launch_fwht128(x, TQ_BF16, ldx, xrot, TQ_F16, K, M, K, true, flag, s);
  if (e != cudaSuccess) return from_cuda(e);
  unsigned char* split = static_cast<unsigned char*>(workspace) + gemm_split_offset(M, K);
  return from_cuda(launch_gemm(codes, ldc, scales, lds, N, K, xrot, M, y, ldy, flag, split,
                               ws_bytes - gemm_split_offset(M, K), s, false, 128, nullptr, nullptr, true));
}

tq_status tq_device_fault(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
  const unsigned int f = take_fault_gemv() | take_fault_quant() | take_fault_noalloc();
  if (f & 2u) return TQ_ERR_TIMEOUT;
  return (f & 4u) ? TQ_ERR_RANGE : TQ_OK;
}

}  // extern "C"
