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
// k_quantize_sparse24: an 8-lane group per 128-weight group, lane q holding
// weights 16q .. 16q + 15 (quads 4q .. 4q + 3) in registers: the staged
// FWHT-128 (stages h = 1 .. 8 in the lane, h = 16 .. 64 as shuffles), the
// selection, the 64-value halving tree and the ternarisation give codes and
// scales bit-exact with the definition.
//
// k_gemv_sparse24: decode with the pruned weights skipped, on the CUDA cores
// (the shapes and code layouts the tensor-memory kernel does not take: an
// odd number of groups per row, fewer than four, unaligned codes).  A pre-pass
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
#include <atomic>

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

// One quad: the two positions of largest |w'| (a tie to the lower index),
// its pattern index (kept positions (0,1) (0,2) (0,3) (1,2) (1,3) (2,3) ->
// 0..5) and the kept values in position order.  Position o beats i > o when
// |w_o| >= |w_i|; that is a strict total order, so the positions that beat at
// least two others are exactly the two largest.
__device__ __forceinline__ int select24(const float* w, float& k0, float& k1) {
  const float a0 = fabsf(w[0]), a1 = fabsf(w[1]), a2 = fabsf(w[2]), a3 = fabsf(w[3]);
  const int g01 = a0 >= a1, g02 = a0 >= a2, g03 = a0 >= a3;
  const int g12 = a1 >= a2, g13 = a1 >= a3, g23 = a2 >= a3;
  const bool keep0 = g01 + g02 + g03 >= 2, keep1 = (1 - g01) + g12 + g13 >= 2;
  const bool keep2 = (2 - g02 - g12) + g23 >= 2, keep3 = 3 - g03 - g13 - g23 >= 2;
  const int i0 = keep0 ? 0 : (keep1 ? 1 : 2);
  const int i1 = keep3 ? 3 : (keep2 ? 2 : 1);
  k0 = keep0 ? w[0] : (keep1 ? w[1] : w[2]);
  k1 = keep3 ? w[3] : (keep2 ? w[2] : w[1]);
  return i0 == 0 ? i1 - 1 : (i0 == 1 ? i1 + 1 : 5);
}

__global__ void __launch_bounds__(32 * kQWarps, 4) k_quantize_sparse24(const SQParams p) {
  const int lane = threadIdx.x & 31, q = lane & 7;
  const int64_t G = p.K / 128, units = p.N * G;
  const int64_t wid = ((int64_t)blockIdx.x * (32 * kQWarps) + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * (32 * kQWarps)) >> 5;
  pdl_wait();
  // a warp takes four consecutive units (row-major groups) at a time; the
  // 8-lane group j = lane / 8 takes unit 4 i + j, lane q of it holding
  // weights 16q .. 16q + 15 (quads 4q .. 4q + 3)
  // (the host keeps the unit count below 2^31: 32-bit row / group split)
  for (int64_t u0 = 4 * wid; u0 < units; u0 += 4 * nw) {
    const int64_t u = u0 + (lane >> 3);
    const bool live = u < units;
    const uint32_t n32 = live ? (uint32_t)u / (uint32_t)G : 0u;
    const int64_t n = n32, g = live ? (int64_t)((uint32_t)u - n32 * (uint32_t)G) : 0;
    float v[16];
    if (p.wt == TQ_F32) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.W) + n * p.ldw + 128 * g + 16 * q);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = live ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.W) + n * p.ldw + 128 * g + 16 * q);
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      bf16x8_to_f32(live ? src[0] : z, v);
      bf16x8_to_f32(live ? src[1] : z, v + 8);
    }
    fwht128_x16(v, lane);  // the staged FWHT-128 and the normalisation
    float k[8];
    int pat[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) pat[r] = select24(v + 4 * r, k[2 * r], k[2 * r + 1]);
    // the 64 kept magnitudes in k order (lane q: kept[8q .. 8q + 7]) by the
    // halving tree s[i] += s[i + h], h = 32 .. 1: h = 32, 16, 8 pair lane q
    // with q + 4, q + 2, q + 1 (both lanes form the same IEEE sums), h = 4, 2,
    // 1 stay in the lane
    uint64_t t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = f2_pack(fabsf(k[2 * i]), fabsf(k[2 * i + 1]));
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float lo, hi;
        f2_unpack(t[i], lo, hi);
        t[i] = f2_add(t[i], f2_pack(__shfl_xor_sync(kFull, lo, m), __shfl_xor_sync(kFull, hi, m)));
      }
    }
    t[0] = f2_add(t[0], t[2]);  // h = 4
    t[1] = f2_add(t[1], t[3]);
    t[0] = f2_add(t[0], t[1]);  // h = 2
    float s0, s1;
    f2_unpack(t[0], s0, s1);
    const float ssum = __shfl_sync(kFull, __fadd_rn(s0, s1), lane & 24);  // h = 1, from lane q = 0
    const uint16_t sb = __half_as_ushort(__float2half_rn(__fmul_rn(ssum, 0.015625f)));
    const float sc = __half2float(__ushort_as_half(sb));
    // t = sign(w') [|w'| > s/2] for a finite s > 0, 0 for s = 0, inf or NaN:
    // the same values as clamp(rint(w' / s), -1, 1) with IEEE division and
    // ties to even (the quotient rounds above 1/2 exactly when |w'| > s/2)
    const float thr = (sc != 0.0f) ? __fmul_rn(sc, 0.5f) : __int_as_float(0x7f800000);
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t0 = (int)(k[2 * r] > thr) - (int)(k[2 * r] < -thr);
      const int t1 = (int)(k[2 * r + 1] > thr) - (int)(k[2 * r + 1] < -thr);
      const uint32_t c = (uint32_t)(9 * pat[r] + 3 * (t0 + 1) + (t1 + 1));
      lo |= (c & 15u) << (4 * r);  // codes 4q .. 4q + 3: low nibbles in bytes 2q, 2q + 1
      hi |= (c >> 4) << (2 * r);   // high bits in byte 16 + q
    }
    if (live) {
      uint8_t* gp = p.codes + n * p.ldc + 24 * g;
      *reinterpret_cast<uint16_t*>(gp + 2 * q) = (uint16_t)lo;
      gp[16 + q] = (uint8_t)hi;
      if (q == 0) p.scales[n * p.lds + g] = sb;
    }
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

// CTAs of k_gemv_sparse24<MB> resident per SM with `kb` KB of dynamic shared
// memory, queried once per device and size (a host query, kept off the
// per-call path)
template <int MB>
cudaError_t occupancy_of(int kb, int* occ) {
  constexpr int kMaxKb = kSliceBytes / 1024 + 1;
  static std::atomic<int> cache[64][kMaxKb + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || kb < 0 || kb > kMaxKb)
    return cudaErrorInvalidValue;
  int v = cache[dev][kb].load(std::memory_order_relaxed);
  if (v == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_gemv_sparse24<MB>, 32 * kGWarps,
                                                                  (size_t)kb * 1024);
    if (e != cudaSuccess) return e;
    if (v < 1) v = 1;
    cache[dev][kb].store(v, std::memory_order_relaxed);
  }
  *occ = v;
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
  e = occupancy_of<MB>((smem + 1023) / 1024, &occ);
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
  // the kernel splits its unit index into row and group in 32 bits
  if (N * (K / 128) + 4 * 32 * kQWarps * (int64_t)device_sm_count() * 4 >= (int64_t(1) << 31))
    return cudaErrorNotSupported;
  SQParams p{W, wt, N, K, ldw, codes, ldc, scales, lds};
  // four groups per warp at a time; four CTAs of eight warps per SM
  const int64_t units = N * (K / 128);
  const int64_t grid = std::min<int64_t>((units + 4 * kQWarps - 1) / (4 * kQWarps), (int64_t)device_sm_count() * 4);
  return launch_pdl(k_quantize_sparse24, dim3((unsigned)grid), dim3(32 * kQWarps), 0, s, p);
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
