// k_fwht.cu -- block FWHT of activation rows (tq_fwht128 / tq_fwht, and the
// rotation pre-pass of tq_gemm), block sizes 64, 128 and 256.
//
// Block 128 (k_fwht128_x16): an 8-lane group rotates one 128-block, lane p
// holding elements 16p .. 16p+15 (two 16-byte loads for bf16), so four of the
// seven butterfly stages stay in registers and three cross lanes.  Blocks 64
// and 256 and the copy form (k_fwht128): a half-warp per 128-block, lane p
// holding elements 8p .. 8p+7, loaded with one 16-byte load (bf16) or two
// (fp32), so a warp moves two blocks per load instruction.  Each warp keeps
// enough loads in flight before it computes that, with four CTAs of eight
// warps per SM, 64-128 KB are in flight per SM, which is what this
// bandwidth-bound pass needs.
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

// The other block sizes on the same lane layout (lane p of a half-warp holds
// elements 8p .. 8p + 7 of a 128-block; the two half-warps hold consecutive
// 128-blocks of one row): 64 runs the stages h = 1 .. 32 (the last
// cross-lane stage, lanes l ^ 8, would join the two 64-blocks of the half)
// and multiplies by 1/8; 256 runs h = 1 .. 64 in each half and then h = 128
// across the halves (lanes l ^ 16), and multiplies by 1/16.  The stages run
// in the order h = 1, 2, 4, ..., the lower element of a pair keeping a + b,
// so the result equals the staged fp32 definition bit for bit, as for 128.
template <int BLK>
__device__ __forceinline__ void fwht_blk_x8(float v[8], int lane) {
  static_assert(BLK == 64 || BLK == 256, "block size");
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float a = v[j], b = v[j + 1];
    v[j] = a + b;
    v[j + 1] = a - b;
  }
  uint64_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = f2_pack(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int hp = 1; hp < 4; hp <<= 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if ((i & hp) == 0) {
        const uint64_t a = q[i], b = q[i + hp];
        q[i] = f2_add(a, b);
        q[i + hp] = f2_sub(a, b);
      }
    }
  }
  constexpr int kLast = BLK == 64 ? 8 : 32;  // cross-lane stages m = 1 .. kLast / 2
#pragma unroll
  for (int m = 1; m < kLast; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;
    const uint64_t sg = f2_pack(sgn, sgn);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      f2_unpack(q[i], lo, hi);
      const float olo = __shfl_xor_sync(kFull, lo, m), ohi = __shfl_xor_sync(kFull, hi, m);
      q[i] = f2_fma(sg, q[i], f2_pack(olo, ohi));
    }
  }
  const float c = BLK == 64 ? 0.125f : 0.0625f;
  const uint64_t sc = f2_pack(c, c);
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(q[i], sc), v[2 * i], v[2 * i + 1]);
}

// BLK: 64, 128 or 256, or 0 for no rotation (the residual half of the
// pre-pass of a residual layout copies x, converted and permuted the same way).
template <int XT, int YT, bool PERM16, int BLK>
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
        raw[u].w[0] = ld_in_u4(src);
        if constexpr (XT == TQ_F32) raw[u].w[1] = ld_in_u4(src + 16);
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
      if constexpr (BLK == 128) {
        fwht128_x8(v, lane);
      } else if constexpr (BLK != 0) {
        fwht_blk_x8<BLK>(v, lane);
      }
      store8<YT, PERM16>(y, yof[u], p, v, flag, ok[u]);
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Block size 128 with 16 elements per lane: an 8-lane group rotates one
// 128-block (lane p = lane % 8 holds elements 16p .. 16p + 15; a warp holds four
// blocks).  Stages h = 1, 2, 4, 8 run in the lane's registers (h = 1 on single
// values, then packed f32x2 pairs), h = 16, 32, 64 across lanes l ^ 1, 2, 4 --
// three shuffle stages instead of four, on half as many lanes per block -- then
// one multiply by c; every operation as in the staged definition, so the result
// is bit-identical to it.  A lane also holds a whole 16-element chunk, so the
// GEMM pre-pass order (0,8,1,9,...,7,15) is a permutation of its own registers.
template <int XT>
struct Raw16 {
  uint4 w[XT == TQ_F32 ? 4 : 2];
};

template <int YT, bool PERM16>
__device__ __forceinline__ void store16(void* y, int64_t off, const float v[16], uint32_t* flag, bool valid) {
  if (!valid) return;
  if constexpr (YT == TQ_F32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else if constexpr (YT == TQ_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + off);
    dst[0] = make_uint4(pack_bf162(v[0], v[1]), pack_bf162(v[2], v[3]), pack_bf162(v[4], v[5]), pack_bf162(v[6], v[7]));
    dst[1] = make_uint4(pack_bf162(v[8], v[9]), pack_bf162(v[10], v[11]), pack_bf162(v[12], v[13]),
                        pack_bf162(v[14], v[15]));
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + off);
    if constexpr (PERM16) {
      if (flag != nullptr) {  // fp16 infinity exactly from |v| >= 65520 (round to nearest even)
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        if (amax >= 65520.0f) atomicOr(flag, 1u);
      }
      // slots 2i, 2i + 1 hold elements i and 8 + i
      dst[0] = make_uint4(pack_half2(v[0], v[8]), pack_half2(v[1], v[9]), pack_half2(v[2], v[10]),
                          pack_half2(v[3], v[11]));
      dst[1] = make_uint4(pack_half2(v[4], v[12]), pack_half2(v[5], v[13]), pack_half2(v[6], v[14]),
                          pack_half2(v[7], v[15]));
    } else {
      dst[0] = make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]), pack_half2(v[6], v[7]));
      dst[1] = make_uint4(pack_half2(v[8], v[9]), pack_half2(v[10], v[11]), pack_half2(v[12], v[13]),
                          pack_half2(v[14], v[15]));
    }
  }
}

// Loads in flight per lane: 32 bytes each (bf16) -- two keep as many bytes in
// flight per SM as four of the 8-element form; one for fp32 (64 bytes).
template <int XT>
constexpr int kUnroll16 = XT == TQ_F32 ? 1 : 2;

template <int XT, int YT, bool PERM16>
__global__ void __launch_bounds__(kThreads, 4) k_fwht128_x16(const void* __restrict__ x, int64_t ldx, void* y,
                                                             int64_t ldy, int64_t rows, int64_t G, uint32_t* flag) {
  constexpr int esize = XT == TQ_F32 ? 4 : 2;
  const int lane = threadIdx.x & 31, p = lane & 7, grp = lane >> 3;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t nblk = rows * G;
  pdl_wait();
  // Warp-iteration u covers blocks 4 (warp + u nwarps) + {0 .. 3}; each lane
  // walks its block sequence with a constant stride of 4 nwarps blocks,
  // advancing (row, group) and the offsets incrementally (no division).
  const int64_t step = 4 * nwarps, dr = step / G, dg = step - (step / G) * G;
  const int64_t b_first = 4 * warp + grp;
  int64_t g = b_first % G, r = b_first / G;
  int64_t xo = r * ldx + g * 128 + 16 * p, yo = r * ldy + g * 128 + 16 * p;
  const int64_t xadv = dr * ldx + dg * 128, yadv = dr * ldy + dg * 128;
  const int64_t xwrap = ldx - G * 128, ywrap = ldy - G * 128;
  for (int64_t b0 = warp; 4 * b0 < nblk; b0 += nwarps * kUnroll16<XT>) {
    Raw16<XT> raw[kUnroll16<XT>];
    int64_t yof[kUnroll16<XT>];
    bool ok[kUnroll16<XT>];
#pragma unroll
    for (int u = 0; u < kUnroll16<XT>; ++u) {
      ok[u] = r < rows;
      yof[u] = yo;
#pragma unroll
      for (int i = 0; i < (XT == TQ_F32 ? 4 : 2); ++i) raw[u].w[i] = make_uint4(0, 0, 0, 0);
      if (ok[u]) {
        const unsigned char* src = static_cast<const unsigned char*>(x) + xo * esize;
#pragma unroll
        for (int i = 0; i < (XT == TQ_F32 ? 4 : 2); ++i) raw[u].w[i] = ld_in_u4(src + 16 * i);
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
    for (int u = 0; u < kUnroll16<XT>; ++u) {
      if (4 * (b0 + (int64_t)u * nwarps) >= nblk) break;  // warp-uniform
      float v[16];
      if constexpr (XT == TQ_F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[4 * i] = __uint_as_float(raw[u].w[i].x);
          v[4 * i + 1] = __uint_as_float(raw[u].w[i].y);
          v[4 * i + 2] = __uint_as_float(raw[u].w[i].z);
          v[4 * i + 3] = __uint_as_float(raw[u].w[i].w);
        }
      } else {
        bf16x8_to_f32(raw[u].w[0], v);
        bf16x8_to_f32(raw[u].w[1], v + 8);
      }
      fwht128_x16(v, lane);
      store16<YT, PERM16>(y, yof[u], v, flag, ok[u]);
    }
  }
  pdl_launch_dependents();
}

template <int XT, int YT, bool PERM16>
cudaError_t launch_x16(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t rows, int64_t G, uint32_t* flag,
                       cudaStream_t s) {
  const int64_t nblk = rows * G;
  const int sms = device_sm_count();
  const int64_t want = (nblk + 4 * (kThreads / 32) - 1) / (4 * (kThreads / 32));
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
  return cudaLaunchKernelEx(&cfg, k_fwht128_x16<XT, YT, PERM16>, x, ldx, y, ldy, rows, G, flag);
}

template <int XT, int YT, bool PERM16, int BLK = 128>
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
  return cudaLaunchKernelEx(&cfg, k_fwht128<XT, YT, PERM16, BLK>, x, ldx, y, ldy, rows, G, flag);
}

}  // namespace

cudaError_t launch_fwht128(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows,
                           int64_t K, bool perm16, uint32_t* flag, cudaStream_t s) {
  const int64_t G = K / 128;
  if (rows == 0 || G == 0) return cudaSuccess;
  if (perm16)  // the GEMM pre-pass form: from bf16 x, or from an fp32 y (x' of a split tile's output)
    return xt == TQ_F32 ? launch_x16<TQ_F32, TQ_F16, true>(x, ldx, y, ldy, rows, G, flag, s)
                        : launch_x16<TQ_BF16, TQ_F16, true>(x, ldx, y, ldy, rows, G, flag, s);
  flag = nullptr;  // overflow is recorded by the pre-pass form only
  if (xt == TQ_F32) {
    if (yt == TQ_F32) return launch_x16<TQ_F32, TQ_F32, false>(x, ldx, y, ldy, rows, G, flag, s);
    if (yt == TQ_BF16) return launch_x16<TQ_F32, TQ_BF16, false>(x, ldx, y, ldy, rows, G, flag, s);
    return launch_x16<TQ_F32, TQ_F16, false>(x, ldx, y, ldy, rows, G, flag, s);
  }
  if (yt == TQ_F32) return launch_x16<TQ_BF16, TQ_F32, false>(x, ldx, y, ldy, rows, G, flag, s);
  if (yt == TQ_BF16) return launch_x16<TQ_BF16, TQ_BF16, false>(x, ldx, y, ldy, rows, G, flag, s);
  return launch_x16<TQ_BF16, TQ_F16, false>(x, ldx, y, ldy, rows, G, flag, s);
}

namespace {
template <int BLK>
cudaError_t launch_blk(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows, int64_t G,
                       bool perm16, uint32_t* flag, cudaStream_t s) {
  if (perm16) return launch_t<TQ_BF16, TQ_F16, true, BLK>(x, ldx, y, ldy, rows, G, flag, s);
  flag = nullptr;
  if (xt == TQ_F32) {
    if (yt == TQ_F32) return launch_t<TQ_F32, TQ_F32, false, BLK>(x, ldx, y, ldy, rows, G, flag, s);
    if (yt == TQ_BF16) return launch_t<TQ_F32, TQ_BF16, false, BLK>(x, ldx, y, ldy, rows, G, flag, s);
    return launch_t<TQ_F32, TQ_F16, false, BLK>(x, ldx, y, ldy, rows, G, flag, s);
  }
  if (yt == TQ_F32) return launch_t<TQ_BF16, TQ_F32, false, BLK>(x, ldx, y, ldy, rows, G, flag, s);
  if (yt == TQ_BF16) return launch_t<TQ_BF16, TQ_BF16, false, BLK>(x, ldx, y, ldy, rows, G, flag, s);
  return launch_t<TQ_BF16, TQ_F16, false, BLK>(x, ldx, y, ldy, rows, G, flag, s);
}
}  // namespace

cudaError_t launch_fwht(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows, int64_t K,
                        int block, bool perm16, uint32_t* flag, cudaStream_t s) {
  const int64_t G = K / 128;
  if (rows == 0 || G == 0) return cudaSuccess;
  switch (block) {
    case 128: return launch_fwht128(x, xt, ldx, y, yt, ldy, rows, K, perm16, flag, s);
    case 64: return launch_blk<64>(x, xt, ldx, y, yt, ldy, rows, G, perm16, flag, s);
    case 256: return launch_blk<256>(x, xt, ldx, y, yt, ldy, rows, G, perm16, flag, s);
    case 0: return launch_t<TQ_BF16, TQ_F16, true, 0>(x, ldx, y, ldy, rows, G, perm16 ? flag : nullptr, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace tq
