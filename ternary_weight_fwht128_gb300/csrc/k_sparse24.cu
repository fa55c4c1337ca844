// k_sparse24.cu -- the 2:4-sparse ternary format (mhpq.cn/news/1159370
// sec. 1.2: structured 2:4 sparsity, two of every four weights kept at
// regular positions, then the kept weights ternarised; sec. 1.1: the absmean
// rule).  Readings of the steps the page leaves open: the pattern is chosen on
// the rotated weights w' per quad of four consecutive k, keeping the two
// largest |w'| (a tie goes to the lower index); the scale is fp16_RN of the
// mean |w'| of the 64 kept weights of the group (halving tree over them in k
// order, times 2^-6); t = clamp(rint(w' / scale), -1, 1) on the kept weights,
// 0 on the pruned ones.
//
// Storage, one tensor for mask and trits together (24 bytes per group of 128,
// 1.5 bits per weight plus 0.125 of fp16 scale): quad j of a group has
// pattern p (kept i0 < i1 in the order (0,1) (0,2) (0,3) (1,2) (1,3) (2,3))
// and code c = 9 p + 3 (t[i0] + 1) + (t[i1] + 1) < 54; the low nibble of c
// is nibble j % 2 of byte j / 2 (bytes 0..15), its two high bits sit at bits
// 2 (j % 4) of byte 16 + j / 4 (bytes 16..23).  Codes 54..63 are not written
// by the quantiser; the GEMV reads them as a quad of zeros.
//
// k_quantize_sparse24: one CTA per row, a warp per group at a time; the
// staged FWHT-128, the selection, the 64-value halving tree and the division
// follow the definition step by step, so codes and scales are bit-exact with
// it.  Lane l owns quad l; the code bytes are assembled with OR shuffles.
//
// k_gemv_sparse24: decode with the pruned weights skipped.  A pre-pass
// rotates x into an fp32 workspace; a CTA owns one slice of the K groups and
// a share of the 32-row blocks (as many CTAs as fit on the SMs at once), with
// the slice of x' staged in shared memory transposed as [m][group][position
// in quad][quad] (groups padded to 129 floats).  A warp takes eight groups of
// a row at a time, four lanes per group: lane (g, q) reads one 32-bit word of
// low nibbles and one 16-bit word of high bits (its eight codes) and the
// group's scale, and looks each code up in two 64-entry tables (the two
// activation offsets; the two trits as fp32 high halves).  The eight groups
// fall on different banks, so the two kept activations of each quad are read
// without conflicts whatever the pattern.  Each kept weight is one FMA with
// its trit as an fp32 -1, 0 or 1 (exact products); a lane scales its eight
// quads' sum by the group's fp16 scale and accumulates in fp32; the lanes are
// added by a fixed xor tree and the K slices by a second kernel in slice
// order, so results do not change from call to call.
#include <algorithm>

#include "tq_internal.h"

namespace tq {

namespace {

// ------------------------------------------------------------------ quantise
constexpr int kQWarps = 8;

struct SQParams {
  const void* W;
  int wt;
  int64_t N, K, ldw;
  uint8_t* codes;
  int64_t ldc;
  uint16_t* scales;
  int64_t lds;
};

// pattern index of the kept positions i0 < i1
__device__ __forceinline__ int pattern24(int i0, int i1) { return i0 == 0 ? i1 - 1 : (i0 == 1 ? i1 + 1 : 5); }

// o beats i: larger magnitude, or equal magnitude and lower index
__device__ __forceinline__ bool beats(const float* a, int o, int i) { return a[o] > a[i] || (a[o] == a[i] && o < i); }

__global__ void __launch_bounds__(32 * kQWarps) k_quantize_sparse24(const SQParams p) {
  __shared__ float sv[kQWarps][128];
  __shared__ float ss[kQWarps][64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = blockIdx.x, G = p.K / 128;
  float* v = sv[warp];
  float* s = ss[warp];
  pdl_wait();
  for (int64_t g = warp; g < G; g += kQWarps) {
    if (p.wt == TQ_F32) {
      const float* w = static_cast<const float*>(p.W) + n * p.ldw + 128 * g;
      for (int i = lane; i < 128; i += 32) v[i] = w[i];
    } else {
      const uint16_t* w = static_cast<const uint16_t*>(p.W) + n * p.ldw + 128 * g;
      for (int i = lane; i < 128; i += 32) v[i] = __uint_as_float((uint32_t)w[i] << 16);
    }
    __syncwarp();
    fwht_warp(v, 128, kInvSqrt128, lane);
    // quad `lane`: the best position under "beats", then the best of the rest
    float w[4], a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = v[4 * lane + i];
      a[i] = fabsf(w[i]);
    }
    int b0 = 0;
#pragma unroll
    for (int i = 1; i < 4; ++i)
      if (beats(a, i, b0)) b0 = i;
    int b1 = b0 == 0 ? 1 : 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i != b0 && i != b1 && beats(a, i, b1)) b1 = i;
    const int i0 = b0 < b1 ? b0 : b1, i1 = b0 < b1 ? b1 : b0;
    // the 64 kept magnitudes in k order: quad l holds kept[2l], kept[2l + 1]
    s[2 * lane] = a[i0];
    s[2 * lane + 1] = a[i1];
    __syncwarp();
    for (int h = 32; h >= 1; h >>= 1) {
      if (lane < h) s[lane] = __fadd_rn(s[lane], s[lane + h]);
      __syncwarp();
    }
    const uint16_t sb = __half_as_ushort(__float2half_rn(__fmul_rn(s[0], 0.015625f)));
    const float sc = __half2float(__ushort_as_half(sb));
    const int t0 = ternarise(w[i0], sc), t1 = ternarise(w[i1], sc);
    const uint32_t c = (uint32_t)(9 * pattern24(i0, i1) + 3 * (t0 + 1) + (t1 + 1));
    // low nibbles: word q (bytes 4q ..) holds codes 8q .. 8q + 7; high bits:
    // word q (bytes 16 + 4q ..) holds codes 16q .. 16q + 15
    uint32_t lo = (c & 15u) << (4 * (lane & 7));
    uint32_t hi = (c >> 4) << (2 * (lane & 15));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) lo |= __shfl_xor_sync(0xffffffffu, lo, o);
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) hi |= __shfl_xor_sync(0xffffffffu, hi, o);
    uint8_t* gp = p.codes + n * p.ldc + 24 * g;
    if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(gp + (lane >> 1)) = lo;
    if ((lane & 15) == 0) *reinterpret_cast<uint32_t*>(gp + 16 + (lane >> 2)) = hi;
    if (lane == 0) p.scales[n * p.lds + g] = sb;
    __syncwarp();  // v and s are refilled for the next group
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------- GEMV
constexpr int kGWarps = 8;
constexpr int kGRowsPerWarp = 4;
constexpr int kGRows = kGWarps * kGRowsPerWarp;  // rows per CTA
constexpr int kSliceBytes = 96 * 1024;            // x' of one K slice in shared memory

struct SGParams {
  const uint8_t* codes;
  int64_t ldc;
  const uint16_t* scales;
  int64_t lds;
  int64_t N, K;
  const float* xr;  // FWHT-128 of x, fp32 [M][K]
  int M, gs, nsl;   // rows of x, groups per slice, slices
  float* y;
  int64_t ldy;
  float* part;  // [nsl][M][N] when nsl > 1
};

// x' of one group in shared memory: [position in quad i][quad j] (i * 32 + j),
// groups kXStride floats apart (one float of padding: the eight groups a warp
// reads at once then fall on different banks)
constexpr int kXStride = 129;

// The two tables of a code c < 54 (pattern p = c / 9, trits t0, t1 at the
// kept positions i0 < i1): offsets 32 i0 | (32 i1) << 16 of the two
// activations (x' is stored [position][quad]); and the high halves of t0 and
// t1 as fp32 (0xbf80 for -1, 0 for 0, 0x3f80 for 1; the low halves of these
// values are zero), t0's in bits 16..31 and t1's in bits 0..15.  Codes 54..63
// give trits 0 (offsets 0).
__device__ __forceinline__ void code_tables(uint32_t c, uint32_t& off, uint32_t& tr) {
  if (c >= 54) {
    off = 0u;
    tr = 0u;
    return;
  }
  const uint32_t pt = c / 9, v = c - 9 * pt, f0 = v / 3, f1 = v % 3;
  const uint32_t i0 = pt < 3 ? 0u : (pt < 5 ? 1u : 2u);
  const uint32_t i1 = pt < 3 ? pt + 1 : (pt < 5 ? pt - 1 : 3u);
  auto hi16 = [](uint32_t f) { return f == 0u ? 0xbf80u : (f == 1u ? 0u : 0x3f80u); };
  off = (32u * i0) | ((32u * i1) << 16);
  tr = (hi16(f0) << 16) | hi16(f1);
}

template <int MB>
__global__ void __launch_bounds__(32 * kGWarps) k_gemv_sparse24(const SGParams p) {
  extern __shared__ float xs[];  // [M][gs][kXStride]
  __shared__ uint32_t tab_off[64], tab_tr[64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = p.K / 128, g0 = (int64_t)blockIdx.y * p.gs;
  const int gn = (int)((G - g0) < p.gs ? (G - g0) : p.gs);
  const int M = p.M;
  if (threadIdx.x < 64) code_tables(threadIdx.x, tab_off[threadIdx.x], tab_tr[threadIdx.x]);
  pdl_wait();
  // the slice of x': xs[(m gs + gl) kXStride + 32 i + j] = x'[m][128 (g0 + gl) + 4 j + i]
  const int nx = M * gn * 128;
  for (int idx = threadIdx.x; idx < nx; idx += 32 * kGWarps) {
    const int m = idx / (gn * 128), r = idx - m * gn * 128, gl = r >> 7, k = r & 127;
    xs[(m * p.gs + gl) * kXStride + (k & 3) * 32 + (k >> 2)] = p.xr[(int64_t)m * p.K + 128 * (g0 + gl) + k];
  }
  __syncthreads();
  // lane (gq, q) = (lane / 4, lane % 4) takes quads 8q .. 8q + 7 of group gb + gq
  const int gq = lane >> 2, q = lane & 3;
  // the CTA keeps its slice of x' and takes row blocks blockIdx.x, + gridDim.x, ..
  const int64_t nrb = (p.N + kGRows - 1) / kGRows;
  for (int64_t rb = blockIdx.x; rb < nrb; rb += gridDim.x) {
    for (int rr = 0; rr < kGRowsPerWarp; ++rr) {
    const int64_t n = rb * kGRows + warp * kGRowsPerWarp + rr;
    if (n >= p.N) break;
    const uint8_t* crow = p.codes + n * p.ldc + 24 * g0;
    const uint16_t* srow = p.scales + n * p.lds + g0;
    float acc[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) acc[m] = 0.0f;
    for (int gb = 0; gb < gn; gb += 8) {
      const int gl = gb + gq;
      const bool on = gl < gn;
      const int gc = on ? gl : gn - 1;  // a lane past the slice reads group gn - 1 and adds zeros
      const uint8_t* gp = crow + 24 * gc;
      // past the slice: all codes 63, whose table entries are zero
      const uint32_t lo = on ? ld_in_u32(gp + 4 * q) : 0xffffffffu, hi = on ? ld_in_u16(gp + 16 + 2 * q) : 0xffffu;
      const float sc = __half2float(__ushort_as_half(ld_in_u16(srow + gc)));
      float part[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) part[m] = 0.0f;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const uint32_t c = ((lo >> (4 * jj)) & 15u) | (((hi >> (2 * jj)) & 3u) << 4);
        const uint32_t off = tab_off[c], tr = tab_tr[c];
        const float* xq = xs + gc * kXStride + 8 * q + jj;
        const uint32_t o0 = off & 0xffffu, o1 = off >> 16;
        const float t0 = __uint_as_float(tr & 0xffff0000u), t1 = __uint_as_float(tr << 16);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            const float* xm = xq + m * p.gs * kXStride;
            part[m] = fmaf(t1, xm[o1], fmaf(t0, xm[o0], part[m]));
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[m] = fmaf(sc, part[m], acc[m]);
    }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < M) {
          if (p.nsl == 1)
            p.y[m * p.ldy + n] = acc[m];
          else
            p.part[((int64_t)blockIdx.y * M + m) * p.N + n] = acc[m];
        }
      }
    }
    }
  }
  pdl_launch_dependents();
}

// y[m][n] = sum over the slices, in slice order
__global__ void __launch_bounds__(256) k_sparse24_reduce(const float* part, int nsl, int64_t N, int M, float* y,
                                                         int64_t ldy) {
  pdl_wait();
  const int64_t total = (int64_t)M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / N, n = i - m * N;
    float s = part[i];
    for (int q = 1; q < nsl; ++q) s += part[(int64_t)q * total + i];
    y[m * ldy + n] = s;
  }
  pdl_launch_dependents();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int MB>
cudaError_t set_smem_once(int bytes) {
  static std::atomic<int> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_gemv_sparse24<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int cur = done[dev].load(std::memory_order_acquire);
  while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes)) {
  }
  return cudaSuccess;
}

template <int MB>
cudaError_t launch_gemv_mb(const SGParams& p, int64_t row_blocks, cudaStream_t s) {
  const int smem = p.M * p.gs * kXStride * (int)sizeof(float);
  cudaError_t e = set_smem_once<MB>(smem);
  if (e != cudaSuccess) return e;
  // as many CTAs as fit on the SMs at once (over all slices), each taking
  // row blocks in turn after staging its slice of x' once
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_gemv_sparse24<MB>, 32 * kGWarps, (size_t)smem);
  if (e != cudaSuccess) return e;
  const int64_t per_slice = std::max<int64_t>(1, (int64_t)std::max(occ, 1) * device_sm_count() / p.nsl);
  const int64_t grid_x = std::min<int64_t>(row_blocks, per_slice);
  return launch_pdl(k_gemv_sparse24<MB>, dim3((unsigned)grid_x, (unsigned)p.nsl), dim3(32 * kGWarps),
                    (size_t)smem, s, p);
}

}  // namespace

// K slices: at least enough for each slice of x' to fit kSliceBytes, and,
// for a short N, enough that the grid has about 512 CTAs (keeping at least
// 8 groups per slice); a slice holds a multiple of 8 groups when it fits
// (a warp takes 8 groups at a time).  The same on every device.
void sparse24_plan(int64_t N, int64_t K, int64_t M, int* gs, int* nsl) {
  const int64_t G = K / 128, row_blocks = (N + kGRows - 1) / kGRows;
  const int64_t cap = kSliceBytes / (M * kXStride * (int64_t)sizeof(float));  // groups of x' per slice
  int64_t ns = (G + cap - 1) / cap;
  const int64_t want = std::min<int64_t>((512 + row_blocks - 1) / std::max<int64_t>(row_blocks, 1), G / 8);
  ns = std::max<int64_t>(std::max<int64_t>(ns, want), 1);
  int64_t g = (G + ns - 1) / ns;
  if ((g + 7) / 8 * 8 <= cap) g = (g + 7) / 8 * 8;
  *gs = (int)g;
  *nsl = (int)((G + g - 1) / g);
}

size_t sparse24_gemv_workspace(int64_t N, int64_t K, int64_t M) {
  int gs = 0, nsl = 0;
  sparse24_plan(N, K, M, &gs, &nsl);
  const size_t xr = (size_t)M * (size_t)K * sizeof(float);
  const size_t part = nsl > 1 ? (size_t)nsl * (size_t)M * (size_t)N * sizeof(float) : 0;
  return (xr + 255) / 256 * 256 + part;
}

cudaError_t launch_quantize_sparse24(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, uint8_t* codes,
                                     int64_t ldc, uint16_t* scales, int64_t lds, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (N > 0x7fffffffll) return cudaErrorNotSupported;
  SQParams p{W, wt, N, K, ldw, codes, ldc, scales, lds};
  return launch_pdl(k_quantize_sparse24, dim3((unsigned)N), dim3(32 * kQWarps), 0, s, p);
}

cudaError_t launch_gemv_sparse24(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N,
                                 int64_t K, const uint16_t* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                                 void* ws, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  int gs = 0, nsl = 0;
  sparse24_plan(N, K, M, &gs, &nsl);
  const int64_t row_blocks = (N + kGRows - 1) / kGRows;
  if (row_blocks > 0x7fffffffll || nsl > 65535) return cudaErrorNotSupported;
  float* xr = static_cast<float*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) +
                                         ((size_t)M * (size_t)K * sizeof(float) + 255) / 256 * 256);
  cudaError_t e = launch_fwht128(x, TQ_BF16, ldx, xr, TQ_F32, K, M, K, false, nullptr, s);
  if (e != cudaSuccess) return e;
  SGParams p{codes, ldc, scales, lds, N, K, xr, (int)M, gs, nsl, y, ldy, part};
  if (M <= 1)
    e = launch_gemv_mb<1>(p, row_blocks, s);
  else if (M <= 2)
    e = launch_gemv_mb<2>(p, row_blocks, s);
  else if (M <= 4)
    e = launch_gemv_mb<4>(p, row_blocks, s);
  else if (M <= 8)
    e = launch_gemv_mb<8>(p, row_blocks, s);
  else
    e = launch_gemv_mb<16>(p, row_blocks, s);
  if (e != cudaSuccess || nsl == 1) return e;
  const int64_t total = M * N;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)device_sm_count() * 8);
  return launch_pdl(k_sparse24_reduce, dim3((unsigned)blocks), dim3(256), 0, s, (const float*)part, nsl, N,
                    (int)M, y, ldy);
}

}  // namespace tq
