// k_gemv.cu -- decode GEMV / skinny GEMM (tq_gemv), M = 1..16.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} t[n][k] * x'[m][k],  x' = FWHT-128(x)
//
// Decode is bound by the HBM stream of packed weights (mhpq.cn/news/1159370
// sec. 4.2), so the kernel reads the codes exactly once, in 16-byte loads
// with enough of them in flight, and spends few instructions per weight:
//
// * Work split.  A thread-block cluster of kCl CTAs owns a range of 16-row
//   tiles; CTA rank r of the cluster owns the r-th slice of the K groups.
//   Each CTA rotates only its own slice of x (no CTA repeats another's
//   transform) and keeps it in shared memory as fp16; the kCl partial sums of
//   every output are added through distributed shared memory at the end
//   (fixed order, no global atomics, no workspace).  Inside a CTA, (tile,
//   group pair) units are dealt to the warps in contiguous ranges.
// * Loads.  Lane (gid, tq) reads 8 bytes (32 codes) of each of the unit's two
//   groups, for row gid and for row gid + 8; a warp instruction therefore
//   moves 8 rows x 32 contiguous bytes (whole sectors).  Each warp keeps
//   kDepth units in flight in registers (64 KB per SM), which is what HBM
//   needs to run near its peak.
// * Inner product on tensor cores (mma.sync m16n8k16, fp16 x fp16 -> fp32):
//   A = 16 weight rows x 16 k as fp16 trits, B = 16 k x 8 activation columns.
//   The four lanes of a quad feed one MMA from a single group (its scale is
//   applied afterwards): lane tq's 32 codes fill its four k-slots of each of
//   the group's eight MMAs.  Which physical k sits in which MMA slot does not
//   change the dot product as long as A and B agree, so x' is stored in
//   shared memory already permuted to match.
// * Trit decode: code c (= t + 1) sits at bits 2j..2j+1 of a 16-bit half;
//   OR-ing the exponent of 2^(10-2j) over it gives the fp16 value
//   2^(10-2j) + c, and subtracting 2^(10-2j) + 1 leaves t exactly (one LOP3
//   and one HADD2 per two weights).
// * Scales: each group's MMA result is scaled by its fp16 scale and added to
//   fp32 row totals, so the group structure of the sum is kept exactly.
#include <atomic>
#include <type_traits>

#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kCl = 2;       // CTAs per cluster (split of K)
constexpr int kWarps = 16;   // warps per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 4;    // units of codes in flight per warp

struct Unit {
  uint2 a0, a1, b0, b1;        // 32 codes of groups g, g + 1 for rows gid (a) and gid + 8 (b)
  uint32_t sa, sb;             // fp16 scales of the two groups (low = first)
};

// Base-3 codes: the lane's 32 trits of a group start at trit 128 g + 32 tq,
// inside byte b0 = k0 / 5 at digit r0 = k0 % 5; they span at most 8 bytes,
// which lie in the 16-byte window starting at a8 = b0 & ~7 (two 8-byte loads).
struct Unit3 {
  uint2 w[8];                  // windows: (group 0, group 1) x (row gid, row gid + 8) x (lo, hi)
  uint32_t sa, sb;
};

// 32 trits -> the 2-bit code words of the same 32 k (code = digit = t + 1):
// every byte goes through a 256-entry table (five 2-bit codes per byte).
__device__ __forceinline__ uint2 trits_to_codes(uint2 lo, uint2 hi, int o, int r0, const uint16_t* lut) {
  const uint64_t L = ((uint64_t)lo.y << 32) | lo.x, H = ((uint64_t)hi.y << 32) | hi.x;
  const uint64_t v = o ? ((L >> (8 * o)) | (H << (64 - 8 * o))) : L;  // bytes b0 .. b0 + 7
  uint64_t a0 = 0, a1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) a0 |= (uint64_t)lut[(v >> (8 * i)) & 255u] << (10 * i);      // trits 0..19
#pragma unroll
  for (int i = 3; i < 8; ++i) a1 |= (uint64_t)lut[(v >> (8 * i)) & 255u] << (10 * (i - 3));  // trits 15..39
  return make_uint2((uint32_t)(a0 >> (2 * r0)), (uint32_t)(a1 >> (2 * (r0 + 1))));
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Trits of codes j (low half) and j + 8 (high half) of a 16-code word as an
// fp16x2 register.  w10 = w >> 10 (codes 5..7 and 13..15 at bits 0..5).
template <int J>
__device__ __forceinline__ uint32_t trit_pair(uint32_t w, uint32_t w10) {
  constexpr int jj = J < 5 ? J : J - 5;
  constexpr uint32_t mask = 0x00030003u << (2 * jj);
  constexpr uint32_t magic = (uint32_t)(25 - 2 * jj) << 10;  // fp16 exponent field of 2^(10-2jj)
  constexpr uint32_t magic2 = magic | (magic << 16);
  constexpr uint32_t bias = magic | (1u << (2 * jj));        // 2^(10-2jj) + 1
  constexpr uint32_t bias2 = bias | (bias << 16);
  const uint32_t src = J < 5 ? w : w10;
  return hsub2_bits((src & mask) | magic2, bias2);
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(const float* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

struct Params {
  const uint8_t* codes;
  int64_t ldc;
  const uint16_t* scales;
  int64_t lds;
  int64_t N, K;
  const uint16_t* x;  // bf16
  int64_t ldx;
  int M;
  float* y;
  int64_t ldy;
  int clusters;      // tile ranges: cluster c owns [c*T/clusters, (c+1)*T/clusters)
  int chunk_groups;  // K groups whose rotated activations are in shared memory at once
  int xs_bytes;      // shared bytes for those activations (permuted x', then per-group sums)
  int sum_off;       // byte offset of the per-group sums of x' inside that region
  int ms;            // activation rows stored per (group, quad): 1 for M == 1, else M
  int prefetch;      // codes and scales are ready before the preceding kernel ends
};

// Rotated activations in shared memory (fp16).  Lane tq of a quad holds the
// codes of k = 128 g + 32 tq + 0..31.  Entry (gl, tq, m, i) = 4 fp16 at byte
// offset gl*XG + tq*XQ + m*64 + i*8, XQ = ms*64 + 16 (pad), XG = 4*XQ, holds
// x'[m][128 g + 32 tq + {0, 8, 16, 24} + i]: the activations MMA i multiplies
// with the lane's codes.
__host__ __device__ constexpr int xs_quad_bytes(int ms) { return ms * 64 + 16; }
__host__ __device__ constexpr int xs_group_bytes(int ms) { return 4 * xs_quad_bytes(ms); }

template <int MB>
__device__ __forceinline__ void group_mma(uint32_t wa0, uint32_t wa1, uint32_t wb0, uint32_t wb1, uint32_t xq,
                                          int dm1, float c0v[4], float c1v[4]) {
  const uint32_t a_lo10 = wa0 >> 10, a_hi10 = wa1 >> 10;
  const uint32_t b_lo10 = wb0 >> 10, b_hi10 = wb1 >> 10;
#define TQ_MMA_ONE(I, B0, B1)                                                              \
  {                                                                                        \
    const uint32_t a0 = trit_pair<I>(wa0, a_lo10), a2 = trit_pair<I>(wa1, a_hi10);         \
    const uint32_t a1 = trit_pair<I>(wb0, b_lo10), a3 = trit_pair<I>(wb1, b_hi10);         \
    mma16816(c0v, a0, a1, a2, a3, B0, B1);                                                 \
    if (MB == 16) {                                                                        \
      const uint2 bc = lds_u2(xq + dm1 + (I)*8);                                           \
      mma16816(c1v, a0, a1, a2, a3, bc.x, bc.y);                                           \
    }                                                                                      \
  }
#define TQ_MMA_PAIR(I)                   \
  {                                      \
    const uint4 bq = lds_u4(xq + (I)*8); \
    TQ_MMA_ONE(I, bq.x, bq.y)            \
    TQ_MMA_ONE((I) + 1, bq.z, bq.w)      \
  }
  TQ_MMA_PAIR(0)
  TQ_MMA_PAIR(2)
  TQ_MMA_PAIR(4)
  TQ_MMA_PAIR(6)
#undef TQ_MMA_PAIR
#undef TQ_MMA_ONE
}

// Codes j and j + 8 of a 16-code word, masked in place: as fp16 subnormals
// they are exactly c * 2^(2jj - 24) (c = t + 1 in {0, 1, 2}).  One LOP3 per
// two weights and no fp16 arithmetic; the tensor cores take fp16 subnormals
// exactly and the products c * x' are exact in fp32.
template <int J>
__device__ __forceinline__ uint32_t code_pair_sub(uint32_t w, uint32_t w10) {
  constexpr int jj = J < 5 ? J : J - 5;
  constexpr uint32_t mask = 0x00030003u << (2 * jj);
  return (J < 5 ? w : w10) & mask;
}

// One group with the subnormal decode (M <= 8): MMA i lands in the
// accumulator of its bit position jj (codes 0..4 and 5..7 share positions
// 0..2), so accumulator jj holds 2^(2jj - 24) * (sum of c x' over its slots).
// Returns, per C fragment entry, 2^-24 * sum_k c_k x'_k = sum_jj 4^-jj acc_jj
// (powers of two: the weights are exact).
__device__ __forceinline__ void group_sub(uint32_t wa0, uint32_t wa1, uint32_t wb0, uint32_t wb1, uint32_t xq,
                                          float v[4]) {
  const uint32_t a_lo10 = wa0 >> 10, a_hi10 = wa1 >> 10;
  const uint32_t b_lo10 = wb0 >> 10, b_hi10 = wb1 >> 10;
  float c[5][4];
#pragma unroll
  for (int q = 0; q < 5; ++q) c[q][0] = c[q][1] = c[q][2] = c[q][3] = 0.0f;
#define TQ_SUB_ONE(I, B0, B1)                                                              \
  {                                                                                        \
    const uint32_t a0 = code_pair_sub<I>(wa0, a_lo10), a2 = code_pair_sub<I>(wa1, a_hi10); \
    const uint32_t a1 = code_pair_sub<I>(wb0, b_lo10), a3 = code_pair_sub<I>(wb1, b_hi10); \
    mma16816(c[(I) < 5 ? (I) : (I)-5], a0, a1, a2, a3, B0, B1);                            \
  }
#define TQ_SUB_PAIR(I)                   \
  {                                      \
    const uint4 bq = lds_u4(xq + (I)*8); \
    TQ_SUB_ONE(I, bq.x, bq.y)            \
    TQ_SUB_ONE((I) + 1, bq.z, bq.w)      \
  }
  TQ_SUB_PAIR(0)
  TQ_SUB_PAIR(2)
  TQ_SUB_PAIR(4)
  TQ_SUB_PAIR(6)
#undef TQ_SUB_PAIR
#undef TQ_SUB_ONE
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float t = fmaf(0.25f, c[1][e], c[0][e]);
    t = fmaf(0.0625f, c[2][e], t);
    t = fmaf(0.015625f, c[3][e], t);
    v[e] = fmaf(0.00390625f, c[4][e], t);
  }
}

template <int MB>
__device__ __forceinline__ void scale_add(float acc[8], const float c0v[4], const float c1v[4], float sa, float sb) {
  acc[0] = fmaf(sa, c0v[0], acc[0]);
  acc[1] = fmaf(sa, c0v[1], acc[1]);
  acc[2] = fmaf(sb, c0v[2], acc[2]);
  acc[3] = fmaf(sb, c0v[3], acc[3]);
  if (MB == 16) {
    acc[4] = fmaf(sa, c1v[0], acc[4]);
    acc[5] = fmaf(sa, c1v[1], acc[5]);
    acc[6] = fmaf(sb, c1v[2], acc[6]);
    acc[7] = fmaf(sb, c1v[3], acc[7]);
  }
}

// Per-(group, activation row) sums of the fp16-rounded x', used by the
// subnormal decode: sum_k t_k x'_k = sum_k c_k x'_k - sum_k x'_k.  Stride 1
// (M == 1) or 8 floats per group.
__host__ __device__ constexpr int xsum_stride(int mb) { return mb == 1 ? 1 : 8; }

// Shared memory: [x' chunk][x' group sums][partial y]
template <int MB, int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_gemv(const Params p) {
  constexpr bool B3 = FMT == TQ_PACK_BASE3;
  __shared__ uint16_t lut3[256];  // base-3 byte -> five 2-bit codes
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* xs = smem;
  float* xsum = reinterpret_cast<float*>(smem + p.sum_off);
  float* ypart = reinterpret_cast<float*>(smem + p.xs_bytes);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tq = lane & 3;
  const int M = p.M;
  const uint32_t rank = cluster_rank();
  const int64_t cluster = blockIdx.x / kCl;
  const int64_t G = p.K / 128;
  const int64_t g0 = G * rank / kCl, g1 = G * (rank + 1) / kCl;
  const int64_t ntiles_all = (p.N + 15) / 16;
  const int64_t t0 = ntiles_all * cluster / p.clusters;
  const int ntiles = (int)(ntiles_all * (cluster + 1) / p.clusters - t0);
  const int nchunks = (int)((g1 - g0 + p.chunk_groups - 1) / p.chunk_groups);
  const int ms = p.ms;
  const int mB0 = MB == 1 ? 0 : (gid < M ? gid : M - 1);  // B column of this lane
  const int mB1 = (8 + gid) < M ? 8 + gid : M - 1;        // second MMA (M > 8)
  const int dm1 = (mB1 - mB0) * 64;
  const uint32_t xs_base = smem_u32(xs);

  for (int i = threadIdx.x; i < ntiles * 16 * M; i += kThreads) ypart[i] = 0.0f;
  if (B3) {
    for (int b = threadIdx.x; b < 256; b += kThreads) {
      uint32_t v = 0x155u, q = (uint32_t)b;  // bytes >= 243 never occur; read as all zero trits
      if (b < 243) {
        v = 0;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          v |= (q % 3u) << (2 * i);
          q /= 3u;
        }
      }
      lut3[b] = (uint16_t)v;
    }
  }
  // Inputs may come from the preceding kernel on the stream: x always waits
  // for it; codes and scales too unless the caller declared them ready, in
  // which case the first units of codes are in flight while it finishes.
  if (!p.prefetch) {
    pdl_wait();
    pdl_launch_dependents();
  }

  for (int c = 0; c < nchunks; ++c) {
    const int64_t cg0 = g0 + (int64_t)c * p.chunk_groups;
    const int ng = (int)((g1 - cg0) < p.chunk_groups ? (g1 - cg0) : p.chunk_groups);
    const int npairs = (ng + 1) >> 1;
    const int U = ntiles * npairs;
    const int u0 = (int)((int64_t)U * warp / kWarps), u1 = (int)((int64_t)U * (warp + 1) / kWarps);

    // loader iterator: unit (lt, lp); pointers at pair 0 of tile lt
    int lt = npairs ? u0 / npairs : 0, lp = u0 - lt * npairs;
    const uint8_t *pa = nullptr, *pb = nullptr;
    const uint16_t *qa = nullptr, *qb = nullptr;
    auto set_tile = [&]() {
      int64_t ra = (t0 + lt) * 16 + gid, rb = ra + 8;
      if (ra >= p.N) ra = p.N - 1;
      if (rb >= p.N) rb = p.N - 1;
      pa = p.codes + ra * p.ldc + (B3 ? 0 : cg0 * 32 + tq * 8);
      pb = p.codes + rb * p.ldc + (B3 ? 0 : cg0 * 32 + tq * 8);
      qa = p.scales + ra * p.lds + cg0;
      qb = p.scales + rb * p.lds + cg0;
    };
    set_tile();
    auto load_unit3 = [&](Unit3& d) {
      const bool two = 2 * lp + 1 < ng;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int64_t k0 = (cg0 + 2 * lp + q) * 128 + 32 * tq;
        const int64_t a8 = (k0 / 5) & ~(int64_t)7;
        const bool has = q == 0 || two, hi = a8 + 16 <= p.ldc;
        d.w[4 * q + 0] = has ? ld_in_u2(pa + a8) : make_uint2(0, 0);
        d.w[4 * q + 1] = (has && hi) ? ld_in_u2(pa + a8 + 8) : make_uint2(0, 0);
        d.w[4 * q + 2] = has ? ld_in_u2(pb + a8) : make_uint2(0, 0);
        d.w[4 * q + 3] = (has && hi) ? ld_in_u2(pb + a8 + 8) : make_uint2(0, 0);
      }
      d.sa = (uint32_t)ld_in_u16(qa + 2 * lp) | (two ? ((uint32_t)ld_in_u16(qa + 2 * lp + 1) << 16) : 0u);
      d.sb = (uint32_t)ld_in_u16(qb + 2 * lp) | (two ? ((uint32_t)ld_in_u16(qb + 2 * lp + 1) << 16) : 0u);
      if (++lp == npairs) {
        lp = 0;
        ++lt;
        set_tile();
      }
    };
    auto load_unit = [&](Unit& d) {
      const bool two = 2 * lp + 1 < ng;  // the unit's second group exists
      const int o = lp * 64;
      d.a0 = ld_in_u2(pa + o);
      d.b0 = ld_in_u2(pb + o);
      if (two) {
        d.a1 = ld_in_u2(pa + o + 32);
        d.b1 = ld_in_u2(pb + o + 32);
      } else {
        d.a1 = make_uint2(0, 0);
        d.b1 = d.a1;
      }
      d.sa = (uint32_t)ld_in_u16(qa + 2 * lp) | (two ? ((uint32_t)ld_in_u16(qa + 2 * lp + 1) << 16) : 0u);
      d.sb = (uint32_t)ld_in_u16(qb + 2 * lp) | (two ? ((uint32_t)ld_in_u16(qb + 2 * lp + 1) << 16) : 0u);
      if (++lp == npairs) {
        lp = 0;
        ++lt;
        set_tile();
      }
    };

    using Raw = typename std::conditional<B3, Unit3, Unit>::type;
    constexpr int D = B3 ? 2 : kDepth;  // units in flight (base-3 units hold twice the registers)
    Raw buf[D];
    auto load_raw = [&](Raw& d) {
      if constexpr (B3)
        load_unit3(d);
      else
        load_unit(d);
    };
#pragma unroll
    for (int s = 0; s < D; ++s)
      if (u0 + s < u1) load_raw(buf[s]);
    if (c == 0 && p.prefetch) {
      pdl_wait();
      pdl_launch_dependents();
    }

    // rotate this chunk of x (all M rows) into the permuted fp16 layout
    __syncwarp();  // warps reach block barriers whole
    if (c > 0) __syncthreads();  // previous chunk's activations no longer read
    for (int b = warp; b < ng * M; b += kWarps) {
      const int m = b / ng, gl = b - m * ng;
      float v[4];
      bf16x4_to_f32(ld_in_u2(p.x + (int64_t)m * p.ldx + (cg0 + gl) * 128 + 4 * lane), v);
      fwht128_lane(v, lane);
      float hsum = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 4 * lane + j;  // element of the group
        const int q = e >> 5, o = e & 31, h = ((o >> 4) << 1) | ((o >> 3) & 1), i = o & 7;
        uint16_t* dst =
            reinterpret_cast<uint16_t*>(xs + gl * xs_group_bytes(ms) + q * xs_quad_bytes(ms) + m * 64 + i * 8) + h;
        const __half hv = __float2half_rn(v[j]);
        *dst = __half_as_ushort(hv);
        hsum += __half2float(hv);
      }
      if (MB != 16) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) hsum += __shfl_xor_sync(kFull, hsum, off);
        if (lane == 0) xsum[gl * xsum_stride(MB) + m] = hsum;
      }
    }
    __syncwarp();
    __syncthreads();

    // compute iterator
    int ct = npairs ? u0 / npairs : 0, cp = u0 - ct * npairs;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

    for (int ub = u0; ub < u1; ub += D) {
#pragma unroll
      for (int s = 0; s < D; ++s) {
        if (ub + s < u1) {
          Unit cur;
          if constexpr (B3) {
            const Unit3 raw = buf[s];
            if (ub + s + D < u1) load_raw(buf[s]);
            uint2 cw[4];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int64_t k0 = (cg0 + 2 * cp + q) * 128 + 32 * tq;
              const int64_t b0 = k0 / 5;
              const int r0 = (int)(k0 - 5 * b0), o = (int)(b0 & 7);
              cw[2 * q] = trits_to_codes(raw.w[4 * q], raw.w[4 * q + 1], o, r0, lut3);
              cw[2 * q + 1] = trits_to_codes(raw.w[4 * q + 2], raw.w[4 * q + 3], o, r0, lut3);
            }
            cur.a0 = cw[0];
            cur.b0 = cw[1];
            cur.a1 = cw[2];
            cur.b1 = cw[3];
            cur.sa = raw.sa;
            cur.sb = raw.sb;
          } else {
            cur = buf[s];
            if (ub + s + D < u1) load_raw(buf[s]);
          }
          const int gl = 2 * cp;
          const uint32_t xq = xs_base + (uint32_t)(gl * xs_group_bytes(ms) + tq * xs_quad_bytes(ms) + mB0 * 64);
          if constexpr (MB == 16) {
            {
              float c0v[4] = {0.f, 0.f, 0.f, 0.f}, c1v[4] = {0.f, 0.f, 0.f, 0.f};
              group_mma<MB>(cur.a0.x, cur.a0.y, cur.b0.x, cur.b0.y, xq, dm1, c0v, c1v);
              scale_add<MB>(acc, c0v, c1v, __half2float(__ushort_as_half((uint16_t)(cur.sa & 0xffffu))),
                            __half2float(__ushort_as_half((uint16_t)(cur.sb & 0xffffu))));
            }
            if (gl + 1 < ng) {
              float c0v[4] = {0.f, 0.f, 0.f, 0.f}, c1v[4] = {0.f, 0.f, 0.f, 0.f};
              group_mma<MB>(cur.a1.x, cur.a1.y, cur.b1.x, cur.b1.y, xq + xs_group_bytes(ms), dm1, c0v, c1v);
              scale_add<MB>(acc, c0v, c1v, __half2float(__ushort_as_half((uint16_t)(cur.sa >> 16))),
                            __half2float(__ushort_as_half((uint16_t)(cur.sb >> 16))));
            }
          } else {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              if (q == 1 && gl + 1 >= ng) break;
              float v[4];
              group_sub(q ? cur.a1.x : cur.a0.x, q ? cur.a1.y : cur.a0.y, q ? cur.b1.x : cur.b0.x,
                        q ? cur.b1.y : cur.b0.y, xq + q * xs_group_bytes(ms), v);
              const float sa = __half2float(__ushort_as_half((uint16_t)(q ? cur.sa >> 16 : cur.sa & 0xffffu)));
              const float sb = __half2float(__ushort_as_half((uint16_t)(q ? cur.sb >> 16 : cur.sb & 0xffffu)));
              const float* sg = xsum + (gl + q) * xsum_stride(MB);
              // columns 2 tq and 2 tq + 1 of the C fragment (all equal when M == 1)
              const float x0 = MB == 1 ? sg[0] : sg[2 * tq], x1 = MB == 1 ? sg[0] : sg[2 * tq + 1];
              // s * (sum c x' - sum x'), with sum c x' = 2^24 v
              acc[0] = fmaf(-sa, x0, fmaf(sa * 16777216.0f, v[0], acc[0]));
              acc[1] = fmaf(-sa, x1, fmaf(sa * 16777216.0f, v[1], acc[1]));
              acc[2] = fmaf(-sb, x0, fmaf(sb * 16777216.0f, v[2], acc[2]));
              acc[3] = fmaf(-sb, x1, fmaf(sb * 16777216.0f, v[3], acc[3]));
            }
          }
          // leaving the tile (or the range): add the row totals into the CTA's partial outputs
          const bool last = (ub + s + 1 == u1);
          if (++cp == npairs || last) {
            const int64_t ra = (t0 + ct) * 16 + gid;
#pragma unroll
            for (int half = 0; half < (MB == 16 ? 2 : 1); ++half) {
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int m = 8 * half + 2 * tq + cc;
                const bool use_m = MB == 1 ? (tq == 0 && cc == 0) : (m < M);
                if (use_m) {
                  if (ra < p.N) atomicAdd(&ypart[(ct * 16 + gid) * M + m], acc[4 * half + cc]);
                  if (ra + 8 < p.N) atomicAdd(&ypart[(ct * 16 + gid + 8) * M + m], acc[4 * half + 2 + cc]);
                }
                acc[4 * half + cc] = 0.0f;
                acc[4 * half + 2 + cc] = 0.0f;
              }
            }
            if (cp == npairs) {
              cp = 0;
              ++ct;
            }
          }
        }
      }
    }
  }
  // ---- reduce the kCl partial sums through distributed shared memory
  __syncwarp();
  __syncthreads();
  cluster_sync();
  const int nout = ntiles * 16 * M;
  const int r0 = nout * (int)rank / kCl, r1 = nout * ((int)rank + 1) / kCl;
  for (int i = r0 + threadIdx.x; i < r1; i += kThreads) {
    const int row = i / M, m = i - row * M;
    const int64_t n = t0 * 16 + row;
    if (n >= p.N) continue;
    float sum = 0.0f;
#pragma unroll
    for (int q = 0; q < kCl; ++q) sum += ld_dsmem_f32(ypart + i, (uint32_t)q);
    p.y[(int64_t)m * p.ldy + n] = sum;
  }
  cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
}

template <int MB, int FMT>
cudaError_t launch_mb(const Params& p0, cudaStream_t s) {
  Params p = p0;
  const int64_t G = p.K / 128;
  const int64_t ng_max = (G + kCl - 1) / kCl;
  const int64_t ntiles_all = (p.N + 15) / 16;
  const int64_t max_smem = device_max_smem_optin();
  const int sms = device_sm_count();
  p.ms = MB == 1 ? 1 : p.M;
  // one CTA per SM: as many clusters as fit, each owning a balanced tile range
  int64_t clusters = sms / kCl;
  if (clusters > ntiles_all) clusters = ntiles_all;
  int64_t tpc = (ntiles_all + clusters - 1) / clusters;
  // partial sums take tpc*16*M floats; keep them to a quarter of shared memory
  while (tpc * 16 * p.M * 4 > max_smem / 4 && clusters < ntiles_all) {
    clusters *= 2;
    if (clusters > ntiles_all) clusters = ntiles_all;
    tpc = (ntiles_all + clusters - 1) / clusters;
  }
  const int64_t per_group = xs_group_bytes(p.ms) + 4 * xsum_stride(MB);
  int64_t chunk = (max_smem - tpc * 16 * p.M * 4) / per_group;
  if (chunk > ng_max) chunk = ng_max;
  if (chunk < 1) return cudaErrorNotSupported;
  const int64_t steps = (ng_max + chunk - 1) / chunk;  // walk the slice in near-equal chunks
  chunk = (ng_max + steps - 1) / steps;
  p.clusters = (int)clusters;
  p.chunk_groups = (int)chunk;
  p.xs_bytes = (int)(chunk * per_group);
  p.sum_off = (int)(chunk * xs_group_bytes(p.ms));
  const int smem = (int)(p.xs_bytes + tpc * 16 * p.M * 4);
  // raise the kernel's shared-memory limit only when a launch needs more
  static std::atomic<int> smem_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev].load(std::memory_order_acquire) < smem) {
    cudaError_t e = cudaFuncSetAttribute(k_gemv<MB, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int cur = smem_set[dev].load(std::memory_order_acquire);
    while (cur < smem && !smem_set[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * kCl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_gemv<MB, FMT>, p);
}

}  // namespace

cudaError_t launch_gemv(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                        int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, bool prefetch,
                        cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3) return cudaErrorNotSupported;
  Params p{};
  p.codes = codes;
  p.ldc = ldc;
  p.scales = scales;
  p.lds = lds;
  p.N = N;
  p.K = K;
  p.x = static_cast<const uint16_t*>(x);
  p.ldx = ldx;
  p.M = (int)M;
  p.y = y;
  p.ldy = ldy;
  p.prefetch = prefetch ? 1 : 0;
  {
    const cudaError_t e = launch_gemv_tc(codes, ldc, fmt, scales, lds, N, K, x, ldx, M, y, ldy, prefetch, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (fmt == TQ_PACK_BASE3) {
    if (M == 1) return launch_mb<1, TQ_PACK_BASE3>(p, s);
    if (M <= 8) return launch_mb<8, TQ_PACK_BASE3>(p, s);
    return launch_mb<16, TQ_PACK_BASE3>(p, s);
  }
  if (M == 1) return launch_mb<1, TQ_PACK_2BIT>(p, s);
  if (M <= 8) return launch_mb<8, TQ_PACK_2BIT>(p, s);
  return launch_mb<16, TQ_PACK_2BIT>(p, s);
}


}  // namespace tq
