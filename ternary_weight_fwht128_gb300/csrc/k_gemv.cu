// k_gemv.cu -- decode GEMV / skinny GEMM (tq_gemv), M = 1..16.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} t[n][k] * x'[m][k],  x' = FWHT-128(x)
//
// Decode is bound by the HBM stream of packed weights (mhpq.cn/news/1159370
// sec. 4.2), so the kernel is built around reading the codes once, with many
// bytes in flight and few instructions per weight:
//
// * Work split.  A thread-block cluster of kCl CTAs owns a range of 16-row
//   tiles; CTA rank r of the cluster owns the r-th slice of the K groups.
//   Each CTA rotates only its own slice of x (no CTA repeats another's
//   transform) and keeps it in shared memory as fp16; the kCl partial sums of
//   every output are added through distributed shared memory at the end
//   (fixed order, no global atomics, no workspace).
// * Weight stream.  One producer warp copies "stages" (16 rows x up to
//   kStageGroups groups of codes) from global into a ring of kSlots shared
//   buffers with cp.async.bulk, completing on mbarriers; about 100 KB are in
//   flight per SM, which is what HBM needs to run near its peak.  Sixteen
//   consumer warps take the stages round-robin.
// * Inner product on tensor cores (mma.sync m16n8k16, fp16 x fp16 -> fp32):
//   A = 16 weight rows x 16 k as fp16 trits, B = 16 k x 8 activation columns.
//   Lane (gid, tq) reads 8 bytes (32 codes) of row gid and of row gid + 8 per
//   group; those codes feed the lane's four k-slots of each of the group's
//   eight MMAs.  The dot product does not depend on which physical k sits in
//   which slot as long as A and B agree, so x' is stored already permuted.
// * Trit decode: code c (= t + 1) sits at bits 2j..2j+1 of a 16-bit half;
//   OR-ing the exponent of 2^(10-2j) over it gives the fp16 value
//   2^(10-2j) + c, and subtracting 2^(10-2j) + 1 leaves t exactly (one LOP3
//   and one HADD2 per two weights).
// * Scales: each group's MMA result is scaled by its fp16 scale and added to
//   fp32 row totals, so the group structure of the sum is kept exactly.
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kCl = 2;            // CTAs per cluster (split of K)
constexpr int kConsumers = 16;    // consumer warps per CTA
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kStageGroups = 8;   // groups per stage and row (256 bytes)
constexpr int kPitch = kStageGroups * 32 + 32;  // padded row: 2 wavefronts per 64-bit lane read
constexpr int kStageBytes = 16 * kPitch;
constexpr int kSlots = 24;
static_assert(2 * kSlots * 8 + 16 <= 1024, "barrier area");

__device__ unsigned int g_fault;  // set when a bounded wait ran out

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
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
  asm volatile(
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
  int xs_bytes;      // shared bytes for those activations
  int ms;            // activation rows stored per (group, quad): 1 for M == 1, else M
};

// Rotated activations in shared memory (fp16), per chunk-local group gl:
//   entry (gl, tq, m, i) = 4 fp16 at byte offset
//     gl*XG + tq*XQ + m*64 + i*8,  XQ = ms*64 + 16 (pad), XG = 4*XQ
//   holding x'[m][128 g + 32 tq + {0, 8, 16, 24} + i] -- the four activations
//   lane quad tq multiplies with the codes feeding MMA i.
__host__ __device__ constexpr int xs_quad_bytes(int ms) { return ms * 64 + 16; }
__host__ __device__ constexpr int xs_group_bytes(int ms) { return 4 * xs_quad_bytes(ms); }

// Shared memory: [barriers][stage ring][x' chunk][partial y]
template <int MB>
__global__ void __launch_bounds__(kThreads, 1) k_gemv(const Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kSlots;
  volatile int* abort = reinterpret_cast<volatile int*>(empty + kSlots);
  unsigned char* ring = smem + 1024;
  unsigned char* xs = ring + kSlots * kStageBytes;
  float* ypart = reinterpret_cast<float*>(xs + p.xs_bytes);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = p.M;
  const uint32_t rank = cluster_rank();
  const int64_t cluster = blockIdx.x / kCl;
  const int64_t G = p.K / 128;
  const int64_t g0 = G * rank / kCl, g1 = G * (rank + 1) / kCl;
  const int64_t ntiles_all = (p.N + 15) / 16;
  const int64_t t0 = ntiles_all * cluster / p.clusters;
  const int ntiles = (int)(ntiles_all * (cluster + 1) / p.clusters - t0);
  const int nchunks = (int)((g1 - g0 + p.chunk_groups - 1) / p.chunk_groups);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < ntiles * 16 * M; i += kThreads) ypart[i] = 0.0f;
  __syncthreads();
  // Inputs (codes, scales, x) may come from the preceding kernel on the stream.
  pdl_wait();

  // Stage numbering: chunk-major, then tile, then group block inside the chunk.
  auto chunk_range = [&](int c, int64_t& cg0, int& ng, int& nsub) {
    cg0 = g0 + (int64_t)c * p.chunk_groups;
    const int64_t rest = g1 - cg0;
    ng = (int)(rest < p.chunk_groups ? rest : p.chunk_groups);
    nsub = (ng + kStageGroups - 1) / kStageGroups;
  };

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int s = 0;
    for (int c = 0; c < nchunks && ok; ++c) {
      int64_t cg0;
      int ng, nsub;
      chunk_range(c, cg0, ng, nsub);
      for (int tl = 0; tl < ntiles && ok; ++tl) {
        int64_t row = (t0 + tl) * 16 + (lane & 15);
        if (row >= p.N) row = p.N - 1;
        for (int sb = 0; sb < nsub; ++sb, ++s) {
          const int slot = s % kSlots, use = s / kSlots;
          if (use > 0 && !mbar_wait_abortable(&empty[slot], (use - 1) & 1, abort)) {
            ok = false;
            break;
          }
          const int gs = sb * kStageGroups;
          const int ngs = (ng - gs) < kStageGroups ? (ng - gs) : kStageGroups;
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], 16u * 32u * ngs);
          __syncwarp();
          if (lane < 16)
            bulk_g2s(ring + slot * kStageBytes + lane * kPitch, p.codes + row * p.ldc + (cg0 + gs) * 32,
                     32u * ngs, &full[slot]);
        }
      }
    }
    if (!ok) {
      // A consumer stopped (timeout).  Copies already issued must land before
      // this CTA's shared memory is released, so wait (bounded) for the last
      // kSlots stages: their full barriers complete once their bytes arrive.
      if (lane == 0) atomicOr(&g_fault, 1u);
      for (int q = (s > kSlots ? s - kSlots : 0); q < s; ++q) (void)mbar_wait(&full[q % kSlots], (q / kSlots) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gid = lane >> 2, tq = lane & 3;
    const int mB0 = MB == 1 ? 0 : (gid < M ? gid : M - 1);
    const int mB1 = (8 + gid) < M ? 8 + gid : M - 1;
    const int ms = p.ms;
    const uint32_t xs_base = smem_u32(xs);
    const uint32_t ring_base = smem_u32(ring);
    int s_base = 0;  // first stage number of the current chunk
    bool ok = true;

    for (int c = 0; c < nchunks; ++c) {
      int64_t cg0;
      int ng, nsub;
      chunk_range(c, cg0, ng, nsub);
      // rotate this chunk of x (all M rows) into the permuted fp16 layout
      if (c > 0) named_sync(1, 32 * kConsumers);  // previous chunk's activations no longer read
      for (int b = warp; b < ng * M; b += kConsumers) {
        const int m = b / ng, gl = b - m * ng;
        float v[4];
        bf16x4_to_f32(ldg_nc_u2(p.x + (int64_t)m * p.ldx + (cg0 + gl) * 128 + 4 * lane), v);
        fwht128_lane(v, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 4 * lane + j;  // element of the group
          const int q = e >> 5, o = e & 31, h = ((o >> 4) << 1) | ((o >> 3) & 1), i = o & 7;
          uint16_t* dst =
              reinterpret_cast<uint16_t*>(xs + gl * xs_group_bytes(ms) + q * xs_quad_bytes(ms) + m * 64 + i * 8) + h;
          *dst = __half_as_ushort(__float2half_rn(v[j]));
        }
      }
      named_sync(1, 32 * kConsumers);

      const int nst = ntiles * nsub;
      for (int st = warp; st < nst && ok; st += kConsumers) {
        const int s = s_base + st;
        const int slot = s % kSlots, use = s / kSlots;
        const int tl = st / nsub, sb = st - tl * nsub;
        const int gs = sb * kStageGroups;
        const int ngs = (ng - gs) < kStageGroups ? (ng - gs) : kStageGroups;
        const int64_t ra = (t0 + tl) * 16 + gid, rb = ra + 8;
        const int64_t rac = ra < p.N ? ra : p.N - 1, rbc = rb < p.N ? rb : p.N - 1;
        const uint16_t* spa = p.scales + rac * p.lds + cg0 + gs;
        const uint16_t* spb = p.scales + rbc * p.lds + cg0 + gs;
        if (!mbar_wait_abortable(&full[slot], use & 1, abort)) {
          if (lane == 0) atomicOr(&g_fault, 1u);
          ok = false;
          break;
        }
        const uint32_t ca = ring_base + slot * kStageBytes + gid * kPitch + tq * 8;
        const uint32_t cb = ca + 8 * kPitch;
        uint32_t xq = xs_base + (uint32_t)(gs * xs_group_bytes(ms) + tq * xs_quad_bytes(ms) + mB0 * 64);
        float acc[MB == 16 ? 8 : 4];
#pragma unroll
        for (int i = 0; i < (MB == 16 ? 8 : 4); ++i) acc[i] = 0.0f;
        for (int gl = 0; gl < ngs; ++gl, xq += xs_group_bytes(ms)) {
          const uint2 wa = lds_u2(ca + gl * 32), wb = lds_u2(cb + gl * 32);
          const float sa = __half2float(__ushort_as_half(__ldg(spa + gl)));
          const float sb2 = __half2float(__ushort_as_half(__ldg(spb + gl)));
          const uint32_t a_lo10 = wa.x >> 10, a_hi10 = wa.y >> 10;
          const uint32_t b_lo10 = wb.x >> 10, b_hi10 = wb.y >> 10;
          float c0v[4] = {0.f, 0.f, 0.f, 0.f};
          float c1v[4] = {0.f, 0.f, 0.f, 0.f};
#define TQ_MMA_ONE(I, B0, B1)                                                                   \
  {                                                                                             \
    const uint32_t a0 = trit_pair<I>(wa.x, a_lo10), a2 = trit_pair<I>(wa.y, a_hi10);            \
    const uint32_t a1 = trit_pair<I>(wb.x, b_lo10), a3 = trit_pair<I>(wb.y, b_hi10);            \
    mma16816(c0v, a0, a1, a2, a3, B0, B1);                                                      \
    if (MB == 16) {                                                                             \
      const uint2 bc = lds_u2(xq + (mB1 - mB0) * 64 + (I)*8);                                   \
      mma16816(c1v, a0, a1, a2, a3, bc.x, bc.y);                                                \
    }                                                                                           \
  }
#define TQ_MMA_PAIR(I)                       \
  {                                          \
    const uint4 bq = lds_u4(xq + (I)*8);     \
    TQ_MMA_ONE(I, bq.x, bq.y)                \
    TQ_MMA_ONE((I) + 1, bq.z, bq.w)          \
  }
          TQ_MMA_PAIR(0)
          TQ_MMA_PAIR(2)
          TQ_MMA_PAIR(4)
          TQ_MMA_PAIR(6)
#undef TQ_MMA_PAIR
#undef TQ_MMA_ONE
          acc[0] = fmaf(sa, c0v[0], acc[0]);
          acc[1] = fmaf(sa, c0v[1], acc[1]);
          acc[2] = fmaf(sb2, c0v[2], acc[2]);
          acc[3] = fmaf(sb2, c0v[3], acc[3]);
          if (MB == 16) {
            acc[4] = fmaf(sa, c1v[0], acc[4]);
            acc[5] = fmaf(sa, c1v[1], acc[5]);
            acc[6] = fmaf(sb2, c1v[2], acc[6]);
            acc[7] = fmaf(sb2, c1v[3], acc[7]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        // add this stage's partial sums into the CTA's partial outputs
#pragma unroll
        for (int half = 0; half < (MB == 16 ? 2 : 1); ++half) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int m = 8 * half + 2 * tq + cc;
            const bool use_m = MB == 1 ? (tq == 0 && cc == 0) : (m < M);
            if (use_m) {
              if (ra < p.N) atomicAdd(&ypart[(tl * 16 + gid) * M + m], acc[4 * half + cc]);
              if (rb < p.N) atomicAdd(&ypart[(tl * 16 + gid + 8) * M + m], acc[4 * half + 2 + cc]);
            }
          }
        }
      }
      s_base += ntiles * nsub;
      // after a timeout the warp skips its remaining stages but still takes
      // part in every named barrier, so no warp is left waiting there
    }
  }
  pdl_launch_dependents();

  // ---- reduce the kCl partial sums through distributed shared memory
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

template <int MB>
cudaError_t launch_mb(const Params& p0, cudaStream_t s) {
  Params p = p0;
  const int64_t G = p.K / 128;
  const int64_t ng_max = (G + kCl - 1) / kCl;
  const int64_t ntiles_all = (p.N + 15) / 16;
  const int64_t max_smem = device_max_smem_optin();
  const int sms = device_sm_count();
  p.ms = MB == 1 ? 1 : p.M;
  const int64_t fixed = 1024 + (int64_t)kSlots * kStageBytes;
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
  const int64_t per_group = xs_group_bytes(p.ms);
  int64_t chunk = (max_smem - fixed - tpc * 16 * p.M * 4) / per_group;
  if (chunk > ng_max) chunk = ng_max;
  if (chunk < 1) return cudaErrorNotSupported;
  const int64_t steps = (ng_max + chunk - 1) / chunk;  // walk the slice in near-equal chunks
  chunk = (ng_max + steps - 1) / steps;
  p.clusters = (int)clusters;
  p.chunk_groups = (int)chunk;
  p.xs_bytes = (int)(chunk * per_group);
  const int smem = (int)(fixed + p.xs_bytes + tpc * 16 * p.M * 4);
  cudaError_t e = cudaFuncSetAttribute(k_gemv<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
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
  return cudaLaunchKernelEx(&cfg, k_gemv<MB>, p);
}

}  // namespace

cudaError_t launch_gemv(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds, int64_t N,
                        int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (fmt != TQ_PACK_2BIT) return cudaErrorNotSupported;
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
  if (M == 1) return launch_mb<1>(p, s);
  if (M <= 8) return launch_mb<8>(p, s);
  return launch_mb<16>(p, s);
}

unsigned int take_fault_gemv() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_fault, sizeof(v)) != cudaSuccess) return 0;
  if (v) (void)cudaMemcpyToSymbol(g_fault, &z, sizeof(z));
  return v;
}

}  // namespace tq
