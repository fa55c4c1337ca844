// tq_internal.h -- declarations shared by the libtq translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/tq.h"
#include "tq_device.cuh"

namespace tq {

// Device properties of the current device, cached per device (read-only
// after the first query).
int device_sm_count();
int device_max_smem_optin();

// Block FWHT-128 of `rows` rows of x into y.  perm16: the GEMM pre-pass form
// (bf16 -> fp16 in the GEMM's k order inside each 16-element chunk), which
// ORs 1 into *flag when an output overflows fp16; the other forms ignore flag.
cudaError_t launch_fwht128(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows,
                           int64_t K, bool perm16, uint32_t* flag, cudaStream_t s);

// Block FWHT of size `block` (64, 128 or 256; K a multiple of it), same
// forms as launch_fwht128.  block == 0: no rotation, the GEMM pre-pass form
// only (bf16 -> fp16 permuted, overflow flagged) -- the residual half of the
// activations of a residual layout.
cudaError_t launch_fwht(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows, int64_t K,
                        int block, bool perm16, uint32_t* flag, cudaStream_t s);

cudaError_t launch_quantize_pack(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt,
                                 uint8_t* codes2, int64_t ld2, uint8_t* codes3, int64_t ld3, uint16_t* scales,
                                 int64_t lds, cudaStream_t s);

// Quantise + pack under a layout variant (block 64/128/256, group 128/256,
// residual pass): one CTA per row, the row's trits (K, or 2K with the
// residual pass) in shared memory; cudaErrorNotSupported when they do not fit.
size_t quantize_layout_smem(int64_t K, int residual);
cudaError_t launch_quantize_layout(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int block, int group,
                                   int residual, uint8_t* codes2, int64_t ld2, uint8_t* codes3, int64_t ld3,
                                   uint16_t* scales, int64_t lds, cudaStream_t s);

// prefetch: codes and scales may be read before the preceding kernel on the
// stream has finished (they were complete before it started).
cudaError_t launch_gemv(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                        int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, bool prefetch,
                        cudaStream_t s);

// 2-bit or base-3 codes, M = 1..16, on tcgen05 fp8 MMAs with the weights in
// tensor memory; cudaErrorNotSupported when the shape does not suit it (the
// caller then uses launch_gemv's mma.sync kernel).  gemv_tc_launches: 1 when
// one launch takes all M rows of x, 2 when it takes two launches of half the
// rows each, 0 when the shape does not suit it.
// all_rows: the chained form (GemvChain::xnext), where rank 0 of each cluster
// holds the partial sums of every row of its tiles.
// fmt: TQ_PACK_2BIT, TQ_PACK_BASE3, or kFmtSparse24 (the 2:4-sparse codes:
// 24 bytes per group; K / 128 even and at least 4, codes 16-byte aligned,
// ldc a multiple of 16; method's layout only, no chain, no stall test).
constexpr int kFmtSparse24 = 0x24;
bool plan_gemv_tc(int64_t N, int64_t K, int64_t M, int fmt, int* kcl, int* clusters, bool all_rows = false);
int gemv_tc_launches(int64_t N, int64_t K, int64_t M, int fmt, bool all_rows = false);
// A layout variant of the method (block size, scale group, residual pass);
// nullptr means block 128, group 128, no residual pass.
struct GemvLayout {
  int block;     // 64, 128 or 256
  int group;     // 128 or 256
  int residual;  // codes and scales hold a residual pass after the first
};

// Chained decode: xr (if set) is x already rotated, fp32 [M][ldxr], read
// instead of x; xnext (if set) receives FWHT-128(y) in fp32 [M][ldxn] (N a
// multiple of 128).  Method's layout only.
struct GemvChain {
  const float* xr;
  int64_t ldxr;
  float* xnext;
  int64_t ldxn;
};

// test_stall: failure-path test (CTA 0 withholds a copy; waits bounded by
// milliseconds), see TQ_GEMV_TEST_STALL.  lay: K counts the codes of both
// passes of a residual layout (twice the activations' K).
cudaError_t launch_gemv_tc(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds,
                           int64_t N, int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                           bool prefetch, cudaStream_t s, bool test_stall = false,
                           const GemvLayout* lay = nullptr, const GemvChain* chain = nullptr);

// Returns cudaErrorNotSupported when the shape needs more shared memory than
// one CTA can have.
// split_ws (may be null): room for the fp32 partial tiles of a K-split last
// wave (up to kMaxSplitUnits tiles of 256 x 256), split_bytes long.
constexpr int64_t kMaxSplitUnits = 160;  // one segment per SM on up to 160 SMs
constexpr size_t kGemmSplitBytes = (size_t)kMaxSplitUnits * 256 * 256 * sizeof(float);  // 40 MiB
// test_stall: failure-path test (CTA 0 withholds a copy; waits bounded by
// milliseconds), see TQ_GEMM_TEST_STALL.  group: weights per scale (128 or
// 256).  K counts every code column (both passes of a residual layout).
// xnext: also write FWHT-128(y) as the next GEMM's fp16 x' ([M][N], N a
// multiple of 128) and OR its fp16 overflow into *flag_next (the K split of a
// short last wave is then not used).  sparse24: codes are the 2:4-sparse
// format (24 bytes per group of 128; group 128, no xnext).
cudaError_t launch_gemm(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N, int64_t K,
                        const uint16_t* xrot, int64_t M, float* y, int64_t ldy, uint32_t* flag, void* split_ws,
                        size_t split_bytes, cudaStream_t s, bool test_stall = false, int group = 128,
                        uint16_t* xnext = nullptr, uint32_t* flag_next = nullptr, bool sparse24 = false);

// 2:4-sparse ternary format (24 code bytes per group of 128).  The GEMV takes
// a workspace of sparse24_gemv_workspace(N, K, M) bytes: the fp32 rotated x,
// then (when K is split into several slices) the slices' partial sums.
void sparse24_plan(int64_t N, int64_t K, int64_t M, int* groups_per_slice, int* slices);
size_t sparse24_gemv_workspace(int64_t N, int64_t K, int64_t M);
cudaError_t launch_quantize_sparse24(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, uint8_t* codes,
                                     int64_t ldc, uint16_t* scales, int64_t lds, cudaStream_t s);
cudaError_t launch_gemv_sparse24(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N,
                                 int64_t K, const uint16_t* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                                 void* ws, cudaStream_t s);

// Reads and clears the device status word of the GEMV kernels (non-zero:
// a bounded wait ran out).
unsigned int take_fault_gemv();
unsigned int take_fault_quant();
// Same for the status word of tq_gemm_noalloc's scratch array (its timeout
// bit only; the word is left as it is otherwise).
unsigned int take_fault_noalloc();

}  // namespace tq
