// k_quant.cu -- offline quantise + pack (tq_quantize_pack).
//
// Per (row n, group g) of 128 weights, one warp:
//   1. loads the group (lane l: elements 4l..4l+3),
//   2. rotates it with the staged FWHT-128 in fp32 (tq_device.cuh),
//   3. sums |w'| in the halving-tree order h = 64, 32, ..., 1: h >= 4 pairs
//      lane l with lane l ^ (h/4) through shuffles, h = 2, 1 stay in-lane
//      (IEEE addition commutes, so every lane ends with the same bits),
//   4. mean = sum * 2^-7, scale = fp16_RN(mean) (absmean, mhpq.cn/news/1159370
//      sec. 1.1; one fp16 scale per 128, sec. 1.3),
//   5. t = sign(w') * [|w'| > s/2] for a finite s > 0, t = 0 when s == 0.
//      This equals clamp(rint(w'/s), -1, 1) with IEEE division and ties to
//      even: the quotient rounds above 0.5 exactly when |w'| > (s/2)(1 + 2^-24),
//      and no fp32 value lies strictly between s/2 and that bound.  For
//      s = +inf both forms give 0.
//   6. packs: 2-bit codes straight from registers (lane l owns byte 32g + l);
//      base-3 bytes after the trits of five consecutive groups (640 trits =
//      128 bytes, so segments of five groups never share a byte) are staged
//      in shared memory.
// A CTA of five warps handles kSeg segments (row, five groups) per iteration,
// issuing every load of the iteration before any arithmetic so that enough
// bytes are in flight for this bandwidth-bound pass.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kWarps = 5;
constexpr int kThreads = 32 * kWarps;
constexpr int kSeg = 4;  // segments per CTA iteration

template <int WT>
__device__ __forceinline__ void load_group(const void* W, int64_t off, float v[4]) {
  if constexpr (WT == TQ_F32) {
    const uint4 w = ldg_nc_u4(static_cast<const float*>(W) + off);
    v[0] = __uint_as_float(w.x);
    v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z);
    v[3] = __uint_as_float(w.w);
  } else {
    bf16x4_to_f32(ldg_nc_u2(static_cast<const uint16_t*>(W) + off), v);
  }
}

template <int WT, bool DO2, bool DO3>
__global__ void __launch_bounds__(kThreads) k_quantize_pack(const void* __restrict__ W, int64_t N, int64_t K,
                                                            int64_t ldw, uint8_t* __restrict__ codes2, int64_t ld2,
                                                            uint8_t* __restrict__ codes3, int64_t ld3,
                                                            uint16_t* __restrict__ scales, int64_t lds) {
  __shared__ int8_t trits[kSeg][640];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t G = K / 128;
  const int64_t nseg = (G + 4) / 5;
  const int64_t total = N * nseg;
  const int64_t nbytes3 = (K + 4) / 5;
  const int64_t ld3min = (nbytes3 + 15) / 16 * 16;

  for (int64_t s0 = (int64_t)blockIdx.x * kSeg; s0 < total; s0 += (int64_t)gridDim.x * kSeg) {
    float v[kSeg][4];
    int64_t row[kSeg], grp[kSeg];
#pragma unroll
    for (int u = 0; u < kSeg; ++u) {
      const int64_t sid = s0 + u;
      row[u] = -1;
      grp[u] = -1;
      if (sid < total) {
        row[u] = sid / nseg;
        const int64_t g = (sid - row[u] * nseg) * 5 + warp;
        if (g < G) {
          grp[u] = g;
          load_group<WT>(W, row[u] * ldw + g * 128 + 4 * lane, v[u]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kSeg; ++u) {
      if (grp[u] < 0) continue;  // warp-uniform
      fwht128_lane(v[u], lane);
      float a[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) a[j] = fabsf(v[u][j]);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {  // h = 64, 32, 16, 8, 4
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = __fadd_rn(a[j], __shfl_xor_sync(kFull, a[j], m));
      }
      a[0] = __fadd_rn(a[0], a[2]);  // h = 2
      a[1] = __fadd_rn(a[1], a[3]);
      a[0] = __fadd_rn(a[0], a[1]);  // h = 1
      const float mean = __fmul_rn(a[0], 0.0078125f);
      const __half sh = __float2half_rn(mean);
      const float sc = __half2float(sh);
      const float half_s = sc * 0.5f;  // exact
      int t[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = v[u][j];
        t[j] = (sc != 0.0f && fabsf(w) > half_s) ? (w > 0.0f ? 1 : -1) : 0;
      }
      const int64_t n = row[u], g = grp[u];
      if constexpr (DO2) {
        const uint32_t byte = (uint32_t)(t[0] + 1) | ((uint32_t)(t[1] + 1) << 2) | ((uint32_t)(t[2] + 1) << 4) |
                              ((uint32_t)(t[3] + 1) << 6);
        codes2[n * ld2 + g * 32 + lane] = (uint8_t)byte;
      }
      if constexpr (DO3) {
        char4 c4 = make_char4((signed char)t[0], (signed char)t[1], (signed char)t[2], (signed char)t[3]);
        *reinterpret_cast<char4*>(&trits[u][warp * 128 + 4 * lane]) = c4;
      }
      if (lane == 0) scales[n * lds + g] = __half_as_ushort(sh);
    }
    if constexpr (DO3) {
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kSeg; ++u) {
        const int64_t sid = s0 + u;
        if (sid >= total) break;  // CTA-uniform
        const int64_t n = sid / nseg, seg = sid - n * nseg;
        const int64_t k0 = seg * 640;
        const int64_t seg_trits = (K - k0) < 640 ? (K - k0) : 640;
        const int64_t b0 = seg * 128;
        // bytes of this segment, plus the zero padding after the last one
        const int64_t bend = (seg == nseg - 1) ? ld3min : b0 + 128;
        for (int64_t b = b0 + threadIdx.x; b < bend; b += kThreads) {
          const int64_t lb = b - b0;
          uint32_t val = 0;
          if (b < nbytes3) {
            uint32_t p = 1;
#pragma unroll
            for (int i = 0; i < 5; ++i) {
              const int64_t lk = 5 * lb + i;
              const uint32_t d = lk < seg_trits ? (uint32_t)(trits[u][lk] + 1) : 1u;
              val += d * p;
              p *= 3;
            }
          }
          codes3[n * ld3 + b] = (uint8_t)val;
        }
      }
      __syncthreads();
    }
  }
}

template <int WT, bool DO2, bool DO3>
cudaError_t launch_t(const void* W, int64_t N, int64_t K, int64_t ldw, uint8_t* c2, int64_t ld2, uint8_t* c3,
                     int64_t ld3, uint16_t* sc, int64_t lds, cudaStream_t s) {
  const int64_t G = K / 128;
  const int64_t total = N * ((G + 4) / 5);
  const int64_t want = (total + kSeg - 1) / kSeg;
  const int64_t cap = (int64_t)device_sm_count() * 12;  // 12 CTAs x 160 threads per SM
  const int64_t grid = want < cap ? want : cap;
  k_quantize_pack<WT, DO2, DO3><<<(unsigned)grid, kThreads, 0, s>>>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds);
  return cudaGetLastError();
}

template <int WT>
cudaError_t launch_w(const void* W, int64_t N, int64_t K, int64_t ldw, int fmt, uint8_t* c2, int64_t ld2,
                     uint8_t* c3, int64_t ld3, uint16_t* sc, int64_t lds, cudaStream_t s) {
  if (fmt == TQ_PACK_2BIT) return launch_t<WT, true, false>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, s);
  if (fmt == TQ_PACK_BASE3) return launch_t<WT, false, true>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, s);
  return launch_t<WT, true, true>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, s);
}

}  // namespace

cudaError_t launch_quantize_pack(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt, uint8_t* codes2,
                                 int64_t ld2, uint8_t* codes3, int64_t ld3, uint16_t* scales, int64_t lds,
                                 cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (wt == TQ_F32) return launch_w<TQ_F32>(W, N, K, ldw, fmt, codes2, ld2, codes3, ld3, scales, lds, s);
  return launch_w<TQ_BF16>(W, N, K, ldw, fmt, codes2, ld2, codes3, ld3, scales, lds, s);
}

}  // namespace tq
