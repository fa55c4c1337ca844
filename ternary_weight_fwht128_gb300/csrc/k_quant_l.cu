// k_quant_l.cu -- offline quantise + pack under a layout variant
// (tq_quantize_pack_layout): FWHT block size 64, 128 or 256 (dpshk.com/news/
// 5289456 sec. 2.1, xxqk.cn/news/652513 sec. 2.2), one fp16 scale per 128 or
// 256 weights (mhpq.cn/news/1159370 sec. 1.4), and optionally the residual
// two-pass ternarisation (xxqk.cn/news/652513 sec. 3, residual calibrator):
// the residual r = w' - s1 t1 is rotated once more by the same block
// transform and ternarised with a scale of its own.
//
// One CTA per weight row, eight warps.  A warp takes a unit of
// u = max(block, group) weights at a time, staged in its own shared memory:
// every butterfly stage of the transform runs in parallel over the unit's
// pairs (h = 1, 2, ..., block / 2, lower index keeps a + b, then one multiply
// by RN_fp32(1/sqrt(block))), the absmean sum is the halving tree
// s[i] += s[i + h] for h = group / 2 .. 1, the scale is fp16 round-to-nearest,
// and t = clamp(rint(w' / s)) with IEEE division -- each step in the order of
// the definition, so codes and scales are bit-exact with it.  The trits of the
// whole row (both passes: Keff = K or 2K) are kept in shared memory; once the
// row is done, its 2-bit bytes (code t + 1 at bits 2 (k % 4)) and base-3 bytes
// (five digits t + 1 per byte, lowest k least significant, digit 1 past Keff,
// zero bytes up to the 16-byte padded length) are written from there.  This
// is the general path; the method's own layout (128, 128, no residual) keeps
// the fused lane-pair kernel of k_quant.cu.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnitMax = 256;
constexpr int kWarpFloats = 3 * kUnitMax;  // w', r and the sum tree

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

// fp16 scale of g values: halving-tree sum of |v| in fp32, times 1/g (exact).
__device__ __forceinline__ uint16_t group_scale(const float* v, float* s, int g, int lane) {
  for (int i = lane; i < g; i += 32) s[i] = fabsf(v[i]);
  __syncwarp();
  for (int h = g / 2; h >= 1; h >>= 1) {
    for (int i = lane; i < h; i += 32) s[i] = __fadd_rn(s[i], s[i + h]);
    __syncwarp();
  }
  const float mean = __fmul_rn(s[0], 1.0f / (float)g);
  __syncwarp();
  return __half_as_ushort(__float2half_rn(mean));
}

__global__ void __launch_bounds__(kThreads) k_quantize_layout(const LParams p) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int64_t Keff = p.residual ? 2 * p.K : p.K;
  const int64_t tbytes = (Keff + 15) / 16 * 16;
  int8_t* trits = reinterpret_cast<int8_t*>(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* v = reinterpret_cast<float*>(sm + tbytes) + warp * kWarpFloats;
  float* r = v + kUnitMax;
  float* s = r + kUnitMax;
  const int u = p.block > p.group ? p.block : p.group;
  const int64_t n = blockIdx.x;
  const int64_t G = p.K / p.group;
  const float cb = p.block == 64 ? 0.125f : (p.block == 256 ? 0.0625f : kInvSqrt128);
  pdl_wait();
  for (int64_t k0 = (int64_t)warp * u; k0 < p.K; k0 += (int64_t)kWarps * u) {
    if (p.wt == TQ_F32) {
      const float* w = static_cast<const float*>(p.W) + n * p.ldw + k0;
      for (int i = lane; i < u; i += 32) v[i] = w[i];
    } else {
      const uint16_t* w = static_cast<const uint16_t*>(p.W) + n * p.ldw + k0;
      for (int i = lane; i < u; i += 32) v[i] = __uint_as_float((uint32_t)w[i] << 16);
    }
    __syncwarp();
    for (int b = 0; b < u; b += p.block) fwht_warp(v + b, p.block, cb, lane);
    for (int g = 0; g < u; g += p.group) {
      const uint16_t sb = group_scale(v + g, s, p.group, lane);
      if (lane == 0) p.scales[n * p.lds + (k0 + g) / p.group] = sb;
      const float sc = __half2float(__ushort_as_half(sb));
      for (int i = lane; i < p.group; i += 32) {
        const float w = v[g + i];
        const int t = ternarise(w, sc);
        trits[k0 + g + i] = (int8_t)t;
        // a zero trit dequantises to 0 whatever the scale (which may be inf)
        r[g + i] = t == 0 ? w : __fsub_rn(w, __fmul_rn(sc, (float)t));
      }
      __syncwarp();
    }
    if (!p.residual) continue;
    for (int b = 0; b < u; b += p.block) fwht_warp(r + b, p.block, cb, lane);
    for (int g = 0; g < u; g += p.group) {
      const uint16_t sb = group_scale(r + g, s, p.group, lane);
      if (lane == 0) p.scales[n * p.lds + G + (k0 + g) / p.group] = sb;
      const float sc = __half2float(__ushort_as_half(sb));
      for (int i = lane; i < p.group; i += 32) trits[p.K + k0 + g + i] = (int8_t)ternarise(r[g + i], sc);
      __syncwarp();
    }
  }
  __syncthreads();
  if (p.codes2 != nullptr) {
    uint8_t* row = p.codes2 + n * p.ld2;
    for (int64_t j = threadIdx.x; j < Keff / 4; j += kThreads) {
      uint32_t b = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) b |= (uint32_t)(trits[4 * j + i] + 1) << (2 * i);
      row[j] = (uint8_t)b;
    }
  }
  if (p.codes3 != nullptr) {
    uint8_t* row = p.codes3 + n * p.ld3;
    const int64_t nb = (Keff + 4) / 5, padded = (nb + 15) / 16 * 16;
    for (int64_t j = threadIdx.x; j < padded; j += kThreads) {
      uint32_t b = 0;
      if (j < nb) {
        uint32_t pw = 1;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          const int64_t k = 5 * j + i;
          b += (k < Keff ? (uint32_t)(trits[k] + 1) : 1u) * pw;
          pw *= 3;
        }
      }
      row[j] = (uint8_t)b;
    }
  }
  pdl_launch_dependents();
}

}  // namespace

size_t quantize_layout_smem(int64_t K, int residual) {
  const int64_t Keff = residual ? 2 * K : K;
  return (size_t)((Keff + 15) / 16 * 16) + (size_t)kWarps * kWarpFloats * sizeof(float);
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
