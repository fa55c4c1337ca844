// k_fwht.cu -- block FWHT-128 of activation rows (tq_fwht128, and the
// rotation pre-pass of tq_gemm).
//
// A half-warp rotates one 128-block (row r, group g): lane p holds elements
// 8p .. 8p+7, loaded with one 16-byte load (bf16) or two (fp32), so a warp
// moves two blocks per load instruction.  Each warp keeps kUnroll block pairs
// in flight before it computes; with four CTAs of eight warps per SM that is
// 64-128 KB in flight per SM, which is what this bandwidth-bound pass needs.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int XT>
struct Raw {
  uint4 w[XT == TQ_F32 ? 2 : 1];
};

template <int XT>
__device__ __forceinline__ void unpack8(const Raw<XT>& r, float v[8]) {
  if constexpr (XT == TQ_F32) {
    v[0] = __uint_as_float(r.w[0].x);
    v[1] = __uint_as_float(r.w[0].y);
    v[2] = __uint_as_float(r.w[0].z);
    v[3] = __uint_as_float(r.w[0].w);
    v[4] = __uint_as_float(r.w[1].x);
    v[5] = __uint_as_float(r.w[1].y);
    v[6] = __uint_as_float(r.w[1].z);
    v[7] = __uint_as_float(r.w[1].w);
  } else {
    bf16x8_to_f32(r.w[0], v);
  }
}

// PERM16: inside every 16-element chunk store element order 0,8,1,9,...,7,15
// (the order in which the tensor-core GEMM unpacks its weight codes, see
// k_gemm.cu).  Lane p holds elements 8(p&1) .. 8(p&1)+7 of chunk p/2; the two
// lanes of a chunk swap four values so each writes 8 interleaved slots.
// With PERM16 (the GEMM pre-pass), fp16 overflow is recorded in *flag.
template <int YT, bool PERM16>
__device__ __forceinline__ void store8(void* y, int64_t off, int p, const float v[8], uint32_t* flag, bool valid) {
  if constexpr (YT == TQ_F32) {
    if (!valid) return;
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + off + 8 * p);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else if constexpr (YT == TQ_BF16) {
    if (!valid) return;
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + off + 8 * p) =
        make_uint4(pack_bf162(v[0], v[1]), pack_bf162(v[2], v[3]), pack_bf162(v[4], v[5]), pack_bf162(v[6], v[7]));
  } else {
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = pack_half2(v[2 * j], v[2 * j + 1]);
    if (PERM16 && flag != nullptr && valid) {
      // round-to-nearest-even gives an fp16 infinity exactly from |v| >= 65520
      // (the midpoint between 65504 and 2^16 rounds to the even 2^16); NaN
      // is not an overflow, and fmaxf passes over it
      const float amax = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                               fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
      if (amax >= 65520.0f) atomicOr(flag, 1u);
    }
    uint16_t* yp = static_cast<uint16_t*>(y) + off;
    if constexpr (PERM16) {
      // even lane (elements a0..a7 of the chunk) writes slots 0..7 =
      // a0 b0 a1 b1 a2 b2 a3 b3; odd lane (b0..b7) writes slots 8..15 =
      // a4 b4 .. a7 b7.  Odd sends b0..b3, even sends a4..a7.
      const bool odd = p & 1;
      const uint32_t s0 = odd ? h[0] : h[2], s1 = odd ? h[1] : h[3];
      const uint32_t r0 = __shfl_xor_sync(kFull, s0, 1), r1 = __shfl_xor_sync(kFull, s1, 1);
      const uint32_t a01 = odd ? r0 : h[0], a23 = odd ? r1 : h[1];  // a(0..3) or a(4..7)
      const uint32_t b01 = odd ? h[2] : r0, b23 = odd ? h[3] : r1;  // b(0..3) or b(4..7)
      uint4 o;
      o.x = __byte_perm(a01, b01, 0x5410);  // a_lo b_lo
      o.y = __byte_perm(a01, b01, 0x7632);  // a_hi b_hi
      o.z = __byte_perm(a23, b23, 0x5410);
      o.w = __byte_perm(a23, b23, 0x7632);
      if (valid) *reinterpret_cast<uint4*>(yp + 16 * (p >> 1) + 8 * (p & 1)) = o;
    } else {
      if (valid) *reinterpret_cast<uint4*>(yp + 8 * p) = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

template <int XT, int YT, bool PERM16>
__global__ void __launch_bounds__(kThreads, 4) k_fwht128(const void* __restrict__ x, int64_t ldx, void* y,
                                                         int64_t ldy, int64_t rows, int64_t G, uint32_t* flag) {
  constexpr int esize = XT == TQ_F32 ? 4 : 2;
  const int lane = threadIdx.x & 31, p = lane & 15, half = lane >> 4;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t nblk = rows * G;
  pdl_wait();
  // Warp-iteration u covers block pair b0 + u * nwarps, i.e. blocks
  // 2 * (b0 + u * nwarps) + {0, 1}.  Each lane walks its block sequence with
  // a constant stride of 2 * nwarps blocks, advancing (row, group) and the
  // element offsets incrementally (no division inside the loop).
  const int64_t step = 2 * nwarps, dr = step / G, dg = step - (step / G) * G;
  const int64_t b_first = 2 * warp + half;
  int64_t g = b_first % G, r = b_first / G;
  int64_t xo = r * ldx + g * 128, yo = r * ldy + g * 128;
  const int64_t xadv = dr * ldx + dg * 128, yadv = dr * ldy + dg * 128;
  const int64_t xwrap = ldx - G * 128, ywrap = ldy - G * 128;
  for (int64_t b0 = warp; 2 * b0 < nblk; b0 += nwarps * kUnroll) {
    Raw<XT> raw[kUnroll];
    int64_t yof[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      ok[u] = r < rows;
      yof[u] = yo;
      raw[u].w[0] = make_uint4(0, 0, 0, 0);
      if constexpr (XT == TQ_F32) raw[u].w[1] = raw[u].w[0];
      if (ok[u]) {
        const unsigned char* src = static_cast<const unsigned char*>(x) + (xo + 8 * p) * esize;
        raw[u].w[0] = ldg_nc_u4(src);
        if constexpr (XT == TQ_F32) raw[u].w[1] = ldg_nc_u4(src + 16);
      }
      g += dg;
      r += dr;
      xo += xadv;
      yo += yadv;
      if (g >= G) {
        g -= G;
        r += 1;
        xo += xwrap;
        yo += ywrap;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (2 * (b0 + (int64_t)u * nwarps) >= nblk) break;  // warp-uniform
      float v[8];
      unpack8<XT>(raw[u], v);
      fwht128_x8(v, lane);
      store8<YT, PERM16>(y, yof[u], p, v, flag, ok[u]);
    }
  }
  pdl_launch_dependents();
}

template <int XT, int YT, bool PERM16>
cudaError_t launch_t(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t rows, int64_t G, uint32_t* flag,
                     cudaStream_t s) {
  const int64_t nblk = rows * G;
  const int sms = device_sm_count();
  const int64_t want = (nblk + 2 * (kThreads / 32) - 1) / (2 * (kThreads / 32));
  const int64_t cap = (int64_t)sms * 4;  // 4 resident CTAs of 256 threads per SM
  int64_t grid = want < cap ? want : cap;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_fwht128<XT, YT, PERM16>, x, ldx, y, ldy, rows, G, flag);
}

}  // namespace

cudaError_t launch_fwht128(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows,
                           int64_t K, bool perm16, uint32_t* flag, cudaStream_t s) {
  const int64_t G = K / 128;
  if (rows == 0 || G == 0) return cudaSuccess;
  if (perm16) return launch_t<TQ_BF16, TQ_F16, true>(x, ldx, y, ldy, rows, G, flag, s);
  flag = nullptr;  // overflow is recorded by the pre-pass form only
  if (xt == TQ_F32) {
    if (yt == TQ_F32) return launch_t<TQ_F32, TQ_F32, false>(x, ldx, y, ldy, rows, G, flag, s);
    if (yt == TQ_BF16) return launch_t<TQ_F32, TQ_BF16, false>(x, ldx, y, ldy, rows, G, flag, s);
    return launch_t<TQ_F32, TQ_F16, false>(x, ldx, y, ldy, rows, G, flag, s);
  }
  if (yt == TQ_F32) return launch_t<TQ_BF16, TQ_F32, false>(x, ldx, y, ldy, rows, G, flag, s);
  if (yt == TQ_BF16) return launch_t<TQ_BF16, TQ_BF16, false>(x, ldx, y, ldy, rows, G, flag, s);
  return launch_t<TQ_BF16, TQ_F16, false>(x, ldx, y, ldy, rows, G, flag, s);
}

}  // namespace tq
