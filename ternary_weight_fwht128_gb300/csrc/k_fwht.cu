// k_fwht.cu -- block FWHT-128 of activation rows (tq_fwht128, and the
// rotation pre-pass of tq_gemm).
//
// One warp rotates one 128-block (row r, group g) at a time; every lane loads
// four consecutive elements (16 B for fp32, 8 B for bf16), so a warp moves
// 256-512 contiguous bytes per block.  Each warp keeps kUnroll blocks' loads
// in flight before it computes, which is what keeps HBM busy in this purely
// bandwidth-bound pass.  The grid is a whole number of waves over the SMs.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int XT>
__device__ __forceinline__ void load4(const void* x, int64_t off, float v[4]) {
  if constexpr (XT == TQ_F32) {
    const uint4 w = ldg_nc_u4(static_cast<const float*>(x) + off);
    v[0] = __uint_as_float(w.x);
    v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z);
    v[3] = __uint_as_float(w.w);
  } else {
    bf16x4_to_f32(ldg_nc_u2(static_cast<const uint16_t*>(x) + off), v);
  }
}

// PERM16: inside every 16-element chunk store element order
// 0,8,1,9,...,7,15 (the order in which the tensor-core GEMM unpacks its
// weight codes, see k_gemm.cu).  FLAG: record fp16 overflow in *flag.
template <int YT, bool PERM16>
__device__ __forceinline__ void store4(void* y, int64_t row_off, int lane, const float v[4], uint32_t* flag) {
  if constexpr (YT == TQ_F32) {
    float4 o = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(static_cast<float*>(y) + row_off + 4 * lane) = o;
  } else if constexpr (YT == TQ_BF16) {
    uint2 o = make_uint2(pack_bf162(v[0], v[1]), pack_bf162(v[2], v[3]));
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + row_off + 4 * lane) = o;
  } else {
    __half h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __float2half_rn(v[j]);
    if (flag != nullptr) {
      bool bad = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) bad |= __hisinf(h[j]) != 0;
      if (bad) atomicOr(flag, 1u);
    }
    uint16_t* yp = static_cast<uint16_t*>(y) + row_off;
    if constexpr (PERM16) {
      // element p of the 16-chunk goes to slot 2p (p < 8) or 2(p-8)+1
      const int chunk = lane >> 2;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = 4 * (lane & 3) + j;
        const int slot = p < 8 ? 2 * p : 2 * (p - 8) + 1;
        yp[16 * chunk + slot] = __half_as_ushort(h[j]);
      }
    } else {
      uint2 o;
      o.x = (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
      o.y = (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16);
      *reinterpret_cast<uint2*>(yp + 4 * lane) = o;
    }
  }
}

template <int XT, int YT, bool PERM16>
__global__ void __launch_bounds__(kThreads) k_fwht128(const void* __restrict__ x, int64_t ldx, void* y,
                                                      int64_t ldy, int64_t rows, int64_t G, uint32_t* flag) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t nblk = rows * G;
  for (int64_t b0 = warp; b0 < nblk; b0 += nwarps * kUnroll) {
    float v[kUnroll][4];
    int64_t yo[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t b = b0 + (int64_t)u * nwarps;
      yo[u] = -1;
      if (b < nblk) {
        const int64_t r = b / G, g = b - r * G;
        load4<XT>(x, r * ldx + g * 128 + 4 * lane, v[u]);
        yo[u] = r * ldy + g * 128;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (yo[u] < 0) continue;  // warp-uniform
      fwht128_lane(v[u], lane);
      store4<YT, PERM16>(y, yo[u], lane, v[u], flag);
    }
  }
}

template <int XT, int YT, bool PERM16>
cudaError_t launch_t(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t rows, int64_t G, uint32_t* flag,
                     cudaStream_t s) {
  const int64_t nblk = rows * G;
  const int sms = device_sm_count();
  const int64_t want = (nblk + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)sms * 8;  // 8 CTAs of 256 threads per SM = full occupancy
  int64_t grid = want < cap ? want : cap;
  if (grid < 1) grid = 1;
  k_fwht128<XT, YT, PERM16><<<(unsigned)grid, kThreads, 0, s>>>(x, ldx, y, ldy, rows, G, flag);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwht128(const void* x, int xt, int64_t ldx, void* y, int yt, int64_t ldy, int64_t rows,
                           int64_t K, bool perm16, uint32_t* flag, cudaStream_t s) {
  const int64_t G = K / 128;
  if (rows == 0 || G == 0) return cudaSuccess;
  if (perm16) return launch_t<TQ_BF16, TQ_F16, true>(x, ldx, y, ldy, rows, G, flag, s);
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
