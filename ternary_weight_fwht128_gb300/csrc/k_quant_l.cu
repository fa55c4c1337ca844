// k_quant_l.cu -- offline quantise + pack under a layout variant
// (tq_quantize_pack_layout): FWHT block size 64, 128 or 256 (dpshk.com/news/
// 5289456 sec. 2.1, xxqk.cn/news/652513 sec. 2.2), one fp16 scale per 128 or
// 256 weights (mhpq.cn/news/1159370 sec. 1.4), and optionally the residual
// two-pass ternarisation (xxqk.cn/news/652513 sec. 3, residual calibrator):
// the residual r = w' - s1 t1 is rotated once more by the same block
// transform and ternarised with a scale of its own.
//
// One CTA per weight row, eight warps.  A warp takes 256 consecutive weights
// of its row at a time, lane l holding weights 8 l .. 8 l + 7 in registers
// (blocks and groups of 128 and 256 weights both tile the span; at block and
// group <= 128 each half-warp holds one 128-weight unit).  The transform runs
// stages h = 1, 2, 4 inside the lane and h = 8 .. block / 2 as shuffles with
// lane l ^ (h / 8) (the lower index of a pair keeps a + b), then one multiply
// by RN_fp32(1/sqrt(block)); the absmean sum is the halving tree
// s[i] += s[i + h] for h = group / 2 .. 1 -- levels h >= 8 between lanes,
// where both lanes of a pair form the sum (an IEEE sum does not depend on the
// order of its operands, so they hold the same bits), levels 4, 2, 1 inside
// the lane; the scale is fp16 round-to-nearest; and t = sign(w') [|w'| > s/2]
// for a finite s > 0, else 0 -- the same trits as clamp(rint(w' / s), -1, 1)
// with IEEE division and ties to even (the rule of the method-layout kernel in
// k_quant.cu).  Each step follows the definition's order, so codes and scales
// are bit-exact with it.  The trits of the whole row (both passes: Keff = K or
// 2K) are kept in shared memory; once the row is done, its 2-bit bytes (code
// t + 1 at bits 2 (k % 4)) and base-3 bytes (five digits t + 1 per byte,
// lowest k least significant, digit 1 past Keff, zero bytes up to the 16-byte
// padded length) are written from there.  This is the general path; the
// method's own layout (128, 128, no residual) keeps the fused lane-pair
// kernel of k_quant.cu.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSpan = 256;  // weights a warp takes at a time (8 per lane)
constexpr int kTritTail = 32;  // zero bytes after the row's trits (word reads of the base-3 packing)

struct LParams {
  const void* W;
  int wt;
  int64_t N, K, ldw;
  int block, group, residual;
  uint8_t* codes2;
  int64_t ld2;
  uint8_t* codes3;
  int64_t ld3;
  uint16_t* scales;
  int64_t lds;
};

// Block transform of the lane's 8 weights (elements 8 lane .. 8 lane + 7 of
// the span): stages h = 1, 2, 4 in the lane, h = 8 .. block / 2 with lane
// l ^ (h / 8), then * c; from h = 2 on in f32x2 pairs (elements 2i, 2i + 1),
// each half rounded as the scalar operation.  A cross-lane step is
// fma(+-1, own, other): other + own in the lower lane, other - own in the
// upper, one rounding each as the add or subtract it stands for.
__device__ __forceinline__ void fwht_lanes(float v[8], int block, float c, int lane) {
#pragma unroll
  for (int j = 0; j < 8; j += 2) {  // h = 1
    const float a = v[j], b = v[j + 1];
    v[j] = __fadd_rn(a, b);
    v[j + 1] = __fsub_rn(a, b);
  }
  uint64_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = f2_pack(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int hp = 1; hp < 4; hp <<= 1) {  // h = 2, 4 on pairs
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i & hp) continue;
      const uint64_t a = q[i], b = q[i + hp];
      q[i] = f2_add(a, b);
      q[i + hp] = f2_sub(a, b);
    }
  }
  for (int m = 1; 8 * m < block; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;  // the upper lane holds elements i + h
    const uint64_t sg = f2_pack(sgn, sgn);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      f2_unpack(q[i], lo, hi);
      const float olo = __shfl_xor_sync(kFull, lo, m), ohi = __shfl_xor_sync(kFull, hi, m);
      q[i] = f2_fma(sg, q[i], f2_pack(olo, ohi));
    }
  }
  const uint64_t c2 = f2_pack(c, c);
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(q[i], c2), v[2 * i], v[2 * i + 1]);
}

// fp16 scale of the group of g values this lane's 8 belong to: halving-tree
// sum of |v| in fp32 (levels h = g / 2 .. 8 with lane l ^ (h / 8), both lanes
// forming the sum; levels 4, 2, 1 in the lane), times 1/g (exact).  Every
// lane of the group returns it.
__device__ __forceinline__ uint16_t group_scale_lanes(const float v[8], int g) {
  uint64_t s2[4];  // |v| of elements 2i, 2i + 1 as f32x2 pairs
#pragma unroll
  for (int i = 0; i < 4; ++i) s2[i] = f2_pack(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
  for (int m = g / 16; m >= 1; m >>= 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      f2_unpack(s2[i], lo, hi);
      s2[i] = f2_add(s2[i], f2_pack(__shfl_xor_sync(kFull, lo, m), __shfl_xor_sync(kFull, hi, m)));
    }
  }
  s2[0] = f2_add(s2[0], s2[2]);  // level 4: sums 0, 1 and (below) 2, 3
  s2[1] = f2_add(s2[1], s2[3]);
  s2[0] = f2_add(s2[0], s2[1]);  // level 2: sums 0, 1
  float s0, s1;
  f2_unpack(s2[0], s0, s1);
  float s[1] = {__fadd_rn(s0, s1)};  // level 1
  const float mean = __fmul_rn(s[0], 1.0f / (float)g);
  return __half_as_ushort(__float2half_rn(mean));
}

// Trits of the lane's 8 values under scale bits sb: t = [w > s/2] - [w < -s/2]
// for a finite s > 0, else 0 (see the file comment); packed as int8 bytes.
__device__ __forceinline__ uint2 ternarise8(const float v[8], uint16_t sb, int t[8]) {
  const float sc = __half2float(__ushort_as_half(sb));
  const float thr = (sc != 0.0f) ? sc * 0.5f : __int_as_float(0x7f800000);  // sc * 0.5 is exact
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    t[j] = (v[j] > thr ? 1 : 0) - (v[j] < -thr ? 1 : 0);
    w[j >> 2] |= (uint32_t)(uint8_t)(int8_t)t[j] << (8 * (j & 3));
  }
  return make_uint2(w[0], w[1]);
}

__global__ void __launch_bounds__(kThreads) k_quantize_layout(const LParams p) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int64_t Keff = p.residual ? 2 * p.K : p.K;
  int8_t* trits = reinterpret_cast<int8_t*>(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the tail past the row's trits reads as t = 0 in the base-3 packing
  if (threadIdx.x < kTritTail) trits[Keff + threadIdx.x] = 0;
  const int64_t n = blockIdx.x;
  const int lgg = p.group == 256 ? 8 : 7;  // group 128 or 256: shifts, not 64-bit divisions
  const int64_t G = p.K >> lgg;
  const float cb = p.block == 64 ? 0.125f : (p.block == 256 ? 0.0625f : kInvSqrt128);
  pdl_wait();
  for (int64_t k0 = (int64_t)warp * kSpan; k0 < p.K; k0 += (int64_t)kWarps * kSpan) {
    // K is a multiple of 128: a half-warp is wholly inside the row or past it
    // (then it computes on zeros and stores nothing; the shuffles need it)
    const int64_t kl = k0 + 8 * lane;
    const bool live = kl < p.K;
    float v[8];
    if (p.wt == TQ_F32) {
      const float* w = static_cast<const float*>(p.W) + n * p.ldw + kl;
      const uint4 a = live ? ld_in_u4(w) : make_uint4(0, 0, 0, 0), b = live ? ld_in_u4(w + 4) : make_uint4(0, 0, 0, 0);
      v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
      v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    } else {
      const uint16_t* w = static_cast<const uint16_t*>(p.W) + n * p.ldw + kl;
      bf16x8_to_f32(live ? ld_in_u4(w) : make_uint4(0, 0, 0, 0), v);
    }
    const bool first = live && (kl & (p.group - 1)) == 0;  // the lane that stores its group's scale
    fwht_lanes(v, p.block, cb, lane);
    const uint16_t sb = group_scale_lanes(v, p.group);
    if (first) p.scales[n * p.lds + (kl >> lgg)] = sb;
    int t[8];
    const uint2 tw = ternarise8(v, sb, t);
    if (live) *reinterpret_cast<uint2*>(trits + kl) = tw;
    if (!p.residual) continue;
    // residual r = w' - s t (a zero trit leaves w' itself, whatever the scale)
    const float sc = __half2float(__ushort_as_half(sb));
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = t[j] == 0 ? v[j] : __fsub_rn(v[j], __fmul_rn(sc, (float)t[j]));
    fwht_lanes(v, p.block, cb, lane);
    const uint16_t sb2 = group_scale_lanes(v, p.group);
    if (first) p.scales[n * p.lds + G + (kl >> lgg)] = sb2;
    const uint2 tw2 = ternarise8(v, sb2, t);
    if (live) *reinterpret_cast<uint2*>(trits + p.K + kl) = tw2;
  }
  __syncthreads();
  if (p.codes2 != nullptr) {
    // 16 trits a thread: one 16-byte read, t + 1 per byte (no carries), and
    // the four 2-bit fields of each byte word gathered by two shift-ors
    uint8_t* row = p.codes2 + n * p.ld2;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.codes2) | (uintptr_t)p.ld2) & 3u) == 0;
    const int nw = (int)(Keff / 16);
    for (int j = threadIdx.x; j < nw; j += kThreads) {
      const uint4 tb = *reinterpret_cast<const uint4*>(trits + 16 * j);
      const uint32_t q[4] = {tb.x, tb.y, tb.z, tb.w};
      uint32_t w = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = __vadd4(q[i], 0x01010101u);  // codes 0..2, one per byte
        const uint32_t y = c | (c >> 6);                 // codes 0, 1 at bits 0..3; 2, 3 at 16..19
        w |= ((y & 0xfu) | ((y >> 12) & 0xf0u)) << (8 * i);
      }
      if (vec) {
        *reinterpret_cast<uint32_t*>(row + 4 * j) = w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) row[4 * j + i] = (uint8_t)(w >> (8 * i));
      }
    }
  }
  if (p.codes3 != nullptr) {
    // four bytes a thread: 20 trits in five word reads (past Keff the zeroed
    // tail reads as t = 0, digit 1), each byte sum (t + 1) 3^i by Horner's rule;
    // bytes past ceil(Keff / 5) up to the padded length are zero
    uint8_t* row = p.codes3 + n * p.ld3;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.codes3) | (uintptr_t)p.ld3) & 3u) == 0;
    const int nb = (int)((Keff + 4) / 5), padded = (nb + 15) / 16 * 16;
    for (int j = threadIdx.x; j < padded / 4; j += kThreads) {
      uint32_t w = 0;
      if (4 * j < nb) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(trits + 20 * j);
        uint32_t c[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) c[i] = __vadd4(src[i], 0x01010101u);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (4 * j + b >= nb) continue;
          uint32_t v = 0;
#pragma unroll
          for (int i = 4; i >= 0; --i) {
            const int e = 5 * b + i;  // code e of the 20
            v = 3u * v + ((c[e >> 2] >> (8 * (e & 3))) & 0xffu);
          }
          w |= v << (8 * b);
        }
      }
      if (vec) {
        *reinterpret_cast<uint32_t*>(row + 4 * j) = w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) row[4 * j + i] = (uint8_t)(w >> (8 * i));
      }
    }
  }
  pdl_launch_dependents();
}

}  // namespace

size_t quantize_layout_smem(int64_t K, int residual) {
  const int64_t Keff = residual ? 2 * K : K;
  return (size_t)((Keff + kTritTail + 15) / 16 * 16);  // the row's trits and a zero tail
}

cudaError_t launch_quantize_layout(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int block, int group,
                                   int residual, uint8_t* codes2, int64_t ld2, uint8_t* codes3, int64_t ld3,
                                   uint16_t* scales, int64_t lds, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const size_t smem = quantize_layout_smem(K, residual);
  if ((int64_t)smem > (int64_t)device_max_smem_optin() || N > 0x7fffffffll) return cudaErrorNotSupported;
  static std::atomic<int> smem_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev].load(std::memory_order_acquire) < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_layout, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int cur = smem_set[dev].load(std::memory_order_acquire);
    while (cur < (int)smem && !smem_set[dev].compare_exchange_weak(cur, (int)smem)) {
    }
  }
  LParams p{W, wt, N, K, ldw, block, group, residual, codes2, ld2, codes3, ld3, scales, lds};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)N);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_quantize_layout, p);
}

}  // namespace tq
