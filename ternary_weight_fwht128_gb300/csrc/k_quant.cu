// k_quant.cu -- offline quantise + pack (tq_quantize_pack).
//
// Per (row n, group g) of 128 weights, one half-warp:
//   1. loads the group with 16-byte loads (lane p: elements 8p .. 8p+7),
//   2. rotates it with the staged FWHT-128 in fp32 (fwht128_x8),
//   3. sums |w'| in the halving-tree order h = 64, 32, ..., 1: h >= 8 pairs
//      lane p with lane p ^ (h/8) through shuffles, h = 4, 2, 1 stay in-lane
//      (IEEE addition commutes, so every lane ends with the same bits),
//   4. mean = sum * 2^-7, scale = fp16_RN(mean) (absmean, mhpq.cn/news/1159370
//      sec. 1.1; one fp16 scale per 128 weights, sec. 1.3),
//   5. t = sign(w') * [|w'| > s/2] for a finite s > 0, t = 0 when s == 0.
//      This equals clamp(rint(w'/s), -1, 1) with IEEE division and ties to
//      even: the quotient rounds above 0.5 exactly when |w'| > (s/2)(1 + 2^-24),
//      and no fp32 value lies strictly between s/2 and that bound.  For
//      s = +inf both forms give 0.
//   6. packs: 2-bit codes straight from registers (lane p owns bytes 2p,
//      2p + 1 of the group); base-3 bytes from the trits of ten consecutive
//      groups (1280 trits = 256 bytes, so such units never share a byte),
//      staged in shared memory.
//
// This pass reads 2 or 4 bytes per weight and is bound by HBM.  A CTA of five
// warps handles units of (row, ten groups); every warp keeps kDepth units of
// 16-byte loads in flight in registers.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kWarps = 5;
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 4;

template <int WT>
struct Raw {
  uint4 w[WT == TQ_F32 ? 2 : 1];
};

template <int WT, bool DO2, bool DO3>
__global__ void __launch_bounds__(kThreads, 4) k_quantize_pack(const void* __restrict__ W, int64_t N, int64_t K,
                                                            int64_t ldw, uint8_t* __restrict__ codes2, int64_t ld2,
                                                            uint8_t* __restrict__ codes3, int64_t ld3,
                                                            uint16_t* __restrict__ scales, int64_t lds) {
  constexpr int esize = WT == TQ_F32 ? 4 : 2;
  __shared__ __align__(16) int8_t trits[2][1280];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int p = lane & 15, half = lane >> 4;
  const int64_t G = K / 128;
  const int64_t ndec = (G + 9) / 10;
  const int64_t total = N * ndec;
  const int64_t nbytes3 = (K + 4) / 5;
  const int64_t ld3min = (nbytes3 + 15) / 16 * 16;
  const int64_t mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int gw = 2 * warp + half;  // this half-warp's group inside a unit

  pdl_wait();

  // Units of this CTA: u = blockIdx.x + i * gridDim.x, i = 0, 1, ...  Two
  // iterators (loads run kDepth units ahead of the arithmetic) walk them with
  // a constant stride, advancing (row n, unit-in-row d) without division.
  const int64_t dn = (int64_t)gridDim.x / ndec, dd = (int64_t)gridDim.x - dn * ndec;
  struct It {
    int64_t n, d;
  };
  auto advance = [&](It& it) {
    it.d += dd;
    it.n += dn;
    if (it.d >= ndec) {
      it.d -= ndec;
      it.n += 1;
    }
  };
  It li{(int64_t)blockIdx.x / ndec, (int64_t)blockIdx.x % ndec};
  It ci = li;
  auto load = [&](Raw<WT>& r) {
    const int64_t g = li.d * 10 + gw;
    r.w[0] = make_uint4(0, 0, 0, 0);
    if constexpr (WT == TQ_F32) r.w[1] = r.w[0];
    if (g < G) {
      const unsigned char* src = static_cast<const unsigned char*>(W) + ((li.n * ldw) + g * 128 + 8 * p) * esize;
      r.w[0] = ldg_nc_u4(src);
      if constexpr (WT == TQ_F32) r.w[1] = ldg_nc_u4(src + 16);
    }
    advance(li);
  };

  Raw<WT> buf[kDepth];
#pragma unroll
  for (int s = 0; s < kDepth; ++s)
    if (s < mine) load(buf[s]);

  for (int64_t ib = 0; ib < mine; ib += kDepth) {
#pragma unroll
    for (int s = 0; s < kDepth; ++s) {
      const int64_t i = ib + s;
      if (i >= mine) break;  // CTA-uniform
      const Raw<WT> cur = buf[s];
      if (i + kDepth < mine) load(buf[s]);
      const int64_t n = ci.n, d = ci.d;
      advance(ci);
      const int64_t g = d * 10 + gw;
      int8_t* tr = trits[i & 1];
      // A half-warp whose group lies past the row end still runs the
      // arithmetic (its shuffles stay inside the half-warp) and discards it.
      {
        float v[8];
        if constexpr (WT == TQ_F32) {
          v[0] = __uint_as_float(cur.w[0].x);
          v[1] = __uint_as_float(cur.w[0].y);
          v[2] = __uint_as_float(cur.w[0].z);
          v[3] = __uint_as_float(cur.w[0].w);
          v[4] = __uint_as_float(cur.w[1].x);
          v[5] = __uint_as_float(cur.w[1].y);
          v[6] = __uint_as_float(cur.w[1].z);
          v[7] = __uint_as_float(cur.w[1].w);
        } else {
          bf16x8_to_f32(cur.w[0], v);
        }
        fwht128_x8(v, lane);
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = fabsf(v[j]);
#pragma unroll
        for (int m = 8; m >= 1; m >>= 1) {  // h = 64, 32, 16, 8
#pragma unroll
          for (int j = 0; j < 8; ++j) a[j] = __fadd_rn(a[j], __shfl_xor_sync(kFull, a[j], m));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = __fadd_rn(a[j], a[j + 4]);  // h = 4
        a[0] = __fadd_rn(a[0], a[2]);                                  // h = 2
        a[1] = __fadd_rn(a[1], a[3]);
        a[0] = __fadd_rn(a[0], a[1]);  // h = 1
        const float mean = __fmul_rn(a[0], 0.0078125f);
        const __half sh = __float2half_rn(mean);
        const float sc = __half2float(sh);
        const float half_s = sc * 0.5f;  // exact
        uint32_t codes = 0;
        uint32_t tw[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float w = v[j];
          const int t = (sc != 0.0f && fabsf(w) > half_s) ? (w > 0.0f ? 1 : -1) : 0;
          codes |= (uint32_t)(t + 1) << (2 * j);
          tw[j >> 2] |= ((uint32_t)t & 0xffu) << (8 * (j & 3));
        }
        if (g < G) {
          if constexpr (DO2) *reinterpret_cast<uint16_t*>(codes2 + n * ld2 + g * 32 + 2 * p) = (uint16_t)codes;
          if constexpr (DO3) *reinterpret_cast<uint2*>(&tr[gw * 128 + 8 * p]) = make_uint2(tw[0], tw[1]);
          if (p == 0) scales[n * lds + g] = __half_as_ushort(sh);
        }
      }
      if constexpr (DO3) {
        // ten groups' trits -> 256 base-3 bytes (plus the zero padding after
        // the row's last byte); trits[] is double-buffered, so one barrier per
        // unit suffices.
        __syncwarp();
        __syncthreads();
        const int64_t k0 = d * 1280;
        const int64_t unit_trits = (K - k0) < 1280 ? (K - k0) : 1280;
        const int64_t b0 = d * 256;
        const int64_t bend = (d == ndec - 1) ? ld3min : b0 + 256;
        for (int64_t b = b0 + threadIdx.x; b < bend; b += kThreads) {
          const int64_t lb = b - b0;
          uint32_t val = 0;
          if (b < nbytes3) {
            uint32_t pw = 1;
#pragma unroll
            for (int q = 0; q < 5; ++q) {
              const int64_t lk = 5 * lb + q;
              const uint32_t dg = lk < unit_trits ? (uint32_t)(tr[lk] + 1) : 1u;
              val += dg * pw;
              pw *= 3;
            }
          }
          codes3[n * ld3 + b] = (uint8_t)val;
        }
      }
    }
  }
  pdl_launch_dependents();
}

template <int WT, bool DO2, bool DO3>
cudaError_t launch_t(const void* W, int64_t N, int64_t K, int64_t ldw, uint8_t* c2, int64_t ld2, uint8_t* c3,
                     int64_t ld3, uint16_t* sc, int64_t lds, cudaStream_t s) {
  const int64_t G = K / 128;
  const int64_t total = N * ((G + 9) / 10);
  // exactly the resident CTAs: units are dealt out statically, so a CTA
  // waiting for a second wave would leave the tail to few SMs
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quantize_pack<WT, DO2, DO3>, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  const int64_t grid = total < cap ? total : cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_quantize_pack<WT, DO2, DO3>, W, N, K, ldw, c2, ld2, c3, ld3, sc, lds);
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

// No wait in this kernel can stall (no producer/consumer barriers).
unsigned int take_fault_quant() { return 0; }

}  // namespace tq
