// k_gemv_tc.cu -- decode GEMV (tq_gemv, M = 1, 2-bit codes) on tcgen05 tensor
// cores with the weight operand in tensor memory.
//
//   y[n] = sum_g s[n][g] * sum_{k in g} t[n][k] * x'[k],  x' = FWHT-128(x)
//
// Decode streams every packed weight once and should run at the HBM rate
// (mhpq.cn/news/1159370 sec. 4.2).  On this GPU the limit of a GEMV over
// 2-bit codes is the instruction count of the unpacking, so the inner product
// uses the operand form that needs the fewest instructions per weight:
//
// * Weights as fp8 subnormals.  tcgen05.mma kind::f8f6f4 takes e4m3 operands,
//   one byte per element.  A 2-bit code c = t + 1 sits at bits 2j .. 2j+1 of
//   its byte; masking a 32-bit word of codes with 0x03030303 leaves four
//   bytes whose e4m3 values are c * 2^-9 (j = 0), masking with 0x0C0C0C0C
//   leaves 4c * 2^-9 (j = 1), and the same masks on the word shifted right by
//   4 give j = 2 and 3: one LOP3 unpacks four weights.  The e4m3 products and
//   their fp32 sums are exact, and sum_k t x = sum_k c x - sum_k x.
// * Weights in tensor memory.  Lane r of tensor memory holds weight row r of
//   a 128-row tile; each thread unpacks its own row into 32 columns per group
//   (tcgen05.st), and the MMA reads A from there, so the unpacked bytes never
//   pass through shared memory (whose bandwidth would not cover them).
// * Activations as three e4m3 pieces (the B operand, N = 16 columns, three
//   used).  Per group of 128 the rotated activations are scaled by a power
//   of two 2^E with max |x' 2^E| in [128, 256), and each scaled value v is
//   written as p1 + p2 + p3, p1 = e4m3(v), p2 = e4m3(v - p1),
//   p3 = e4m3(v - p1 - p2) (nearest even; the residuals are exact in fp32):
//   within max(2^-12 |v|, 2^-8) of v, finer than an fp16 rounding of x' for
//   all but the smallest elements.  Values that meet the 4c weights are
//   stored divided by 4 (exact).
// * Groups.  Each group's four MMAs (K = 32 each) write their own 16-column
//   accumulator, so C[row][p] = 2^-9 sum_k c_k a_k piece_p(k) for one group;
//   the thread of that row adds the pieces and the correction term
//   -2^-9 sum_k a_k (p1 + p2 + p3)(k), and multiplies by s[row][g] 2^(9 - E)
//   in fp32 -- the scale is applied to each group's inner product.
//
// Work split: a cluster of kcl CTAs owns a range of 128-row tiles; CTA rank r
// owns the r-th slice of the K groups and rotates only that slice of x.  A
// CTA walks (tile, two-group) decode stages with four warp roles that hand
// buffers to one another through mbarriers, so each runs ahead on its own:
//   warp 16      (one lane) TMA-loads 128 x 128-byte code tiles (four groups,
//                128-byte swizzle) into a ring of kRing slots; each slot feeds
//                two decode stages of two groups;
//   warps 0-15   two teams of eight take the even and the odd decode stages
//                (the two halves of each slot); warp w unpacks group
//                (w / 4) % 2 of its stage for rows 32 (w % 4) .. +31 into one
//                of kAbuf A buffers in tensor memory;
//   warps 17-18  warp 17 allocates tensor memory; warp 17 + t issues the
//                sixteen MMAs of each stage of team t into accumulator
//                buffer t;
//   warps 19-22  read the accumulators of their 32 rows and apply the scales.
// Ranks 1 .. kcl-1 push each finished row sum into rank 0's shared memory
// (st.async, counted on an mbarrier there) and exit; rank 0 adds the kcl
// partial sums in a fixed order and writes y.  Every wait is bounded in time;
// a wait that runs out sets the library's GEMV status word and the CTA winds
// down (pending copies and MMAs are waited for, tensor memory is freed, the
// cluster barrier is still met).
#include <cuda.h>
#include <cuda_fp8.h>

#include <atomic>

#include "tq_internal.h"

namespace tq {

__device__ unsigned int g_gemv_fault;  // bit 1: a bounded wait ran out

namespace {

constexpr int kDecWarps = 16;                 // two teams of 8: even and odd decode stages
constexpr int kTeamWarps = 8;
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;                  // warps 17, 18 issue the MMAs of team 0, 1
constexpr int kEpiWarp0 = 19;                 // warps 19-22: epilogue
constexpr int kThreads = 32 * 23;             // + 4 epilogue warps (19-22)
constexpr int kRing = 4;                      // code slots in flight (four groups each)
constexpr int kAbuf = 3;                      // weight (A) buffers in tensor memory, one stage each
constexpr int kDbuf = 2;                      // accumulator buffers: buffer t belongs to team t's stages
constexpr int kSlotBytes = 128 * 128;         // 128 rows x 128 bytes (four groups): one stage
// B of one MMA: two core matrices (8 rows x 16 bytes: k 0-15 and k 16-31)
// 144 bytes apart (16 bytes of padding spread the prologue's stores over all
// banks); rows 8..15 come from a shared zero block.
constexpr int kBLbo = 144;
constexpr int kMmaBBytes = 2 * kBLbo;         // 288
constexpr int kGroupBBytes = 4 * kMmaBBytes;  // B of one group: 4 MMAs
constexpr int kZeroBytes = kMmaBBytes;        // B rows 8..15 of every MMA
constexpr int kTmemCols = 512;                // one CTA per SM
constexpr uint32_t kAcol = 0;                 // A buffer b: columns 128 b .. 128 b + 127 (4 groups x 32)
constexpr uint32_t kDcol = 128 * kAbuf;       // D buffer b: columns kDcol + 64 b .. + 63 (4 groups x 16)
static_assert(kDcol + 64 * kDbuf <= kTmemCols, "tensor memory budget");
constexpr uint32_t kFaultTimeout = 2u;

// kind::f8f6f4: fp32 accumulator, A = B = e4m3, both K-major, N = 16, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

struct Ctl {
  uint64_t full[kRing];   // TMA -> decoders
  uint64_t empty[kRing];  // decoders -> TMA
  uint64_t a_full[kAbuf]; // decoders -> MMA
  uint64_t a_free[kAbuf]; // MMA -> decoders
  uint64_t d_full[kDbuf]; // MMA -> epilogue
  uint64_t d_free[kDbuf]; // epilogue -> MMA
  uint64_t red_bar;       // rank 0: the other ranks' partial outputs have landed
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const uint16_t* scales;
  int64_t lds;
  int64_t N, K;
  const uint16_t* x;  // bf16
  float* y;
  int kcl;         // CTAs per cluster (K split)
  int clusters;    // tile ranges: cluster c owns [c*T/clusters, (c+1)*T/clusters)
  int groups_cap;  // groups per CTA the shared layout holds (multiple of 4)
  int tiles_cap;   // tiles per cluster the partial outputs hold
  int prefetch;    // codes and scales are ready before the preceding kernel ends
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: 8-row x 16-byte core
// matrices; lbo = distance between core matrices along K, sbo = along N.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  return d;
}

__device__ __forceinline__ void mma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t r[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float v[4]) {
  uint32_t r0, r1, r2, r3;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  v[0] = __uint_as_float(r0);
  v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2);
  v[3] = __uint_as_float(r3);
}

__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  return remote;
}

// 4-byte store into another CTA's shared memory that counts as 4 bytes of
// transaction on that CTA's mbarrier.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote_addr), "f"(v),
               "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ uint16_t ldg_nc_u16(const uint16_t* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// FWHT-128 with lane 4i + j holding elements 16i + j + 4b (b = 0..3): stages
// h = 1, 2 pair lanes l ^ 1, l ^ 2; h = 4, 8 stay in the lane (b ^ 1, b ^ 2);
// h = 16, 32, 64 pair lanes l ^ 4, l ^ 8, l ^ 16.  The stages run in the
// order h = 1, 2, 4, ..., 64 with the lower index keeping a + b, then * c,
// so the result equals the staged fp32 definition bit for bit.
__device__ __forceinline__ void fwht128_strided(float v[4], int lane) {
  auto shfl_stage = [&](int m) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float o = __shfl_xor_sync(kFull, v[b], m);
      v[b] = __fmaf_rn(sgn, v[b], o);  // lower lane: o + v; upper lane: o - v
    }
  };
  shfl_stage(1);
  shfl_stage(2);
  {
    const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[2] = a0 - a2;
    v[1] = a1 + a3;
    v[3] = a1 - a3;
  }
  shfl_stage(4);
  shfl_stage(8);
  shfl_stage(16);
#pragma unroll
  for (int b = 0; b < 4; ++b) v[b] = __fmul_rn(v[b], kInvSqrt128);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Two fp32 -> two e4m3 (nearest even, finite), and their values back in fp32.
__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi, float& rlo, float& rhi) {
  const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3);
  rlo = __half2float(__ushort_as_half(h.x));
  rhi = __half2float(__ushort_as_half(h.y));
  return (uint32_t)q;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl) {
  if (mbar_wait_abortable(bar, parity, &ctl->abort)) return true;
  atomicOr(&g_gemv_fault, kFaultTimeout);
  return false;
}

// Shared memory (1024-aligned): [code ring][B: groups_cap x kGroupBBytes][zeros kZeroBytes]
// [ztab: groups_cap x {Zt, pw}][partial y: kcl slots x tiles_cap x 128][Ctl]
__global__ void __launch_bounds__(kThreads, 1) k_gemv_tc(const __grid_constant__ CUtensorMap cmap, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = smem;
  unsigned char* bsm = ring + kRing * kSlotBytes;
  unsigned char* zero = bsm + p.groups_cap * kGroupBBytes;
  float2* ztab = reinterpret_cast<float2*>(zero + kZeroBytes);
  float* ypart = reinterpret_cast<float*>(ztab + p.groups_cap);
  Ctl* ctl = reinterpret_cast<Ctl*>(ypart + p.kcl * p.tiles_cap * 128);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int64_t cluster = blockIdx.x / p.kcl;
  const int64_t G = p.K / 128;
  const int64_t g0 = G * rank / p.kcl, g1 = G * (rank + 1) / p.kcl;
  const int ng = (int)(g1 - g0), nch = (ng + 3) >> 2, nlc = nch;  // four-group stages per tile
  const int64_t T = (p.N + 127) / 128;
  const int64_t t0 = T * cluster / p.clusters;
  const int ntiles = (int)(T * (cluster + 1) / p.clusters - t0);
  const int S = ntiles * nch;  // stages (ring loads) of this CTA
  const int L = S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], kTeamWarps);
    }
    for (int i = 0; i < kAbuf; ++i) {
      mbar_init(&ctl->a_full[i], kTeamWarps);
      mbar_init(&ctl->a_free[i], 1);
    }
    for (int i = 0; i < kDbuf; ++i) {
      mbar_init(&ctl->d_full[i], 1);
      mbar_init(&ctl->d_free[i], 4);
    }
    mbar_init(&ctl->red_bar, 1);
    // rank 0 receives every other rank's partial outputs: ntiles x 128 floats each
    if (rank == 0 && p.kcl > 1) mbar_arrive_expect_tx(&ctl->red_bar, (uint32_t)((p.kcl - 1) * ntiles * 128 * 4));
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // zero B (unused rows and groups), the zero block, ztab and the partial outputs
  {
    uint4* z4 = reinterpret_cast<uint4*>(bsm);
    const int n16 = (p.groups_cap * kGroupBBytes + kZeroBytes) / 16;
    for (int i = threadIdx.x; i < n16; i += kThreads) z4[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < p.groups_cap; i += kThreads) ztab[i] = make_float2(0.0f, 0.0f);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  // Rank 0's reduction barrier is armed: the other ranks may push once they
  // pass the matching wait (epilogue warps before their first push, every
  // other warp before it exits -- each thread waits exactly once).
  cluster_arrive();

  // Inputs may come from the preceding kernel on the stream: x always waits
  // for it; codes and scales too unless the caller declared them ready, in
  // which case the ring fills while that kernel finishes.
  int issued_loads = 0;
  auto fill_ring = [&]() {
    for (; issued_loads < L && issued_loads < kRing; ++issued_loads) {
      const int l = issued_loads, tile = l / nlc, lc = l - tile * nlc;
      mbar_arrive_expect_tx(&ctl->full[l], kSlotBytes);
      tma_load_2d(smem_u32(ring + l * kSlotBytes), &cmap, (int)((g0 + 4 * lc) * 32), (int)((t0 + tile) * 128),
                  &ctl->full[l]);
    }
  };
  if (p.prefetch && warp == kTmaWarp && lane == 0) fill_ring();
  pdl_wait();
  pdl_launch_dependents();
  if (!p.prefetch && warp == kTmaWarp && lane == 0) fill_ring();  // while the others rotate x

  // ---- rotate this CTA's slice of x and split it into three e4m3 pieces.
  // Lane 4i + j holds elements k = 16i + j + 4b (b = 0..3) of its group: these
  // are the four B bytes that meet one code class j of one code word i, so
  // the lane writes each piece as one 32-bit word.
  for (int gl = warp; gl < ng; gl += kThreads / 32) {
    const int i8 = lane >> 2, jc = lane & 3;
    const uint16_t* xg = p.x + (g0 + gl) * 128 + 16 * i8 + jc;
    float v[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) v[b] = __uint_as_float((uint32_t)ldg_nc_u16(xg + 4 * b) << 16);
    fwht128_strided(v, lane);
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    int E = amax > 0.0f ? 134 - (int)((__float_as_uint(amax) >> 23) & 0xffu) : 0;  // max |x' 2^E| in [128, 256)
    E = E < -100 ? -100 : (E > 100 ? 100 : E);
    const float up = __uint_as_float((uint32_t)(127 + E) << 23);
    const float pw = __uint_as_float((uint32_t)(127 + 9 - E) << 23);
    // odd classes j meet the 4c weights: their values are stored divided by 4
    const float cls = (jc & 1) ? 0.25f : 1.0f, acls = (jc & 1) ? 4.0f : 1.0f;
    float u[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) u[b] = v[b] * up * cls;
    float zs = 0.0f;
    // MMA m = i / 2 of the group; k'' = 16 (i % 2) + 4 j + b inside it, at byte
    // (k'' / 16) * kBLbo + piece * 16 + k'' % 16 of the MMA's B
    uint32_t* dst = reinterpret_cast<uint32_t*>(bsm + gl * kGroupBBytes + (i8 >> 1) * kMmaBBytes + (i8 & 1) * kBLbo +
                                                4 * jc);
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      float r0, r1, r2, r3;
      const uint32_t lo = to_e4m3x2(u[0], u[1], r0, r1), hi = to_e4m3x2(u[2], u[3], r2, r3);
      dst[q * 4] = (lo & 0xffffu) | (hi << 16);
      zs += (r0 + r1) + (r2 + r3);
      u[0] -= r0;
      u[1] -= r1;
      u[2] -= r2;
      u[3] -= r3;
    }
    zs = warp_sum(zs * acls);
    if (lane == 0) ztab[gl] = make_float2(zs * -0.001953125f, pw);  // -2^-9 sum
  }
  fence_async_smem();  // B written by ordinary stores, read by the tensor cores
  __syncthreads();

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int l = issued_loads, slot = l % kRing, use = l / kRing, tile = l / (nlc > 0 ? nlc : 1), lc = l - tile * nlc;
      for (; l < L; ++l) {
        if (!wait_or_abort(&ctl->empty[slot], (use - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&ctl->full[slot], kSlotBytes);
        tma_load_2d(smem_u32(ring + slot * kSlotBytes), &cmap, (int)((g0 + 4 * lc) * 32), (int)((t0 + tile) * 128),
                    &ctl->full[slot]);
        if (++slot == kRing) { slot = 0; ++use; }
        if (++lc == nlc) { lc = 0; ++tile; }
      }
      // loads issued but possibly never consumed: let them land before exit
      for (int q = (l > kRing ? l - kRing : 0); q < l; ++q) (void)mbar_wait(&ctl->full[q % kRing], (q / kRing) & 1);
    }
  } else if (warp < kDecWarps) {
    // ------------------------------------------------------------ decoders
    // team (warp / 8) takes the stages of its parity, so two stages are
    // unpacked at once; warp w unpacks groups 2 ((w / 4) % 2) .. +1 of the
    // stage for rows 32 (w % 4) .. +31
    const int team = warp >> 3, quad = warp & 3, gh = (warp >> 2) & 1;
    const int r = quad * 32 + lane;  // row inside the tile = tensor-memory lane
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
    const uint32_t rx = (uint32_t)(r & 7), rbase = (uint32_t)(r * 128);
    const uint32_t ring_u32 = smem_u32(ring);
    uint32_t off[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) off[q] = rbase + ((((uint32_t)(4 * gh + q)) ^ rx) << 4);
    for (int s = team; s < S; s += 2) {
      const int slot = s % kRing, use = s / kRing, ab = s % kAbuf, ause = s / kAbuf;
      bool ok = wait_or_abort(&ctl->full[slot], use & 1, ctl);
      uint4 c[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) c[q] = ok ? lds_u4(ring_u32 + slot * kSlotBytes + off[q]) : make_uint4(0, 0, 0, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[slot]);
      if (ause > 0) ok = wait_or_abort(&ctl->a_free[ab], (ause - 1) & 1, ctl) && ok;
      if (!__all_sync(kFull, ok)) break;  // the tensor-memory stores below are warp-collective
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w[8] = {c[2 * h].x, c[2 * h].y, c[2 * h].z, c[2 * h].w,
                               c[2 * h + 1].x, c[2 * h + 1].y, c[2 * h + 1].z, c[2 * h + 1].w};
        uint32_t a[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t w4 = w[i] >> 4;
          a[4 * i + 0] = w[i] & 0x03030303u;
          a[4 * i + 1] = w[i] & 0x0C0C0C0Cu;
          a[4 * i + 2] = w4 & 0x03030303u;
          a[4 * i + 3] = w4 & 0x0C0C0C0Cu;
        }
        tmem_st32(tmem + lane_addr + kAcol + (uint32_t)(ab * 128 + (2 * gh + h) * 32), a);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->a_full[ab]);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ MMA issue
    // The whole warp walks the stages (its loop state stays warp-uniform);
    // lane 0 waits; one elected lane issues the MMAs and the commits.
    const uint32_t bsm_u32 = smem_u32(bsm), zero_u32 = smem_u32(zero);
    // B descriptor of MMA m of local group gl: start = bsm + kGroupBBytes gl +
    // kMmaBBytes m, sbo = zero - start; consecutive MMAs step start up and sbo
    // down by kMmaBBytes
    const uint64_t desc_g0 = smem_desc_plain(bsm_u32, kBLbo, zero_u32 - bsm_u32);
    constexpr uint64_t kStepM = (uint64_t)(kMmaBBytes >> 4) - ((uint64_t)(kMmaBBytes >> 4) << 32);
    constexpr uint64_t kStepG = (uint64_t)(kGroupBBytes >> 4) - ((uint64_t)(kGroupBBytes >> 4) << 32);
    // warp kMmaWarp + t takes the stages of parity t (team t), accumulating
    // into D buffer t
    const int t = warp - kMmaWarp;
    int s = t, ch = t % (nch > 0 ? nch : 1), duse = 0;  // ch: stage inside the tile
    for (; s < S; s += 2) {
      const int ab = s % kAbuf, ause = s / kAbuf;
      // only lane 0 waits; one elected lane issues the tensor-core work
      bool ok = true;
      if (lane == 0) {
        ok = wait_or_abort(&ctl->a_full[ab], ause & 1, ctl);
        if (ok && duse > 0) ok = wait_or_abort(&ctl->d_free[t], (duse - 1) & 1, ctl);
      }
      if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t d0 = tmem + kDcol + (uint32_t)(t * 64), a0 = tmem + kAcol + (uint32_t)(ab * 128);
        uint64_t bd = desc_g0 + (uint64_t)(4 * ch) * kStepG;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            mma_f8_tmem_a(d0 + h * 16, a0 + h * 32 + m * 8, bd, m > 0 ? 1u : 0u);
            bd += kStepM;
          }
        }
        mma_commit(&ctl->a_free[ab]);
        mma_commit(&ctl->d_full[t]);
      }
      __syncwarp();
      ++duse;
      ch += 2;
      while (ch >= nch) ch -= nch;
    }
    // every MMA this warp issued must be complete before tensor memory is freed
    if (s - 2 >= 0 && lane == 0) (void)mbar_wait(&ctl->d_full[t], ((s - 2) >> 1) & 1);
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // warps 19..22 reach tensor-memory lanes 32 (warp % 4) ..
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    float acc = 0.0f;
    int tile = 0, ch = 0, db = 0, duse = 0;
    // scales of the stage's four groups for this row (groups past the slice: 0)
    auto ld_scales = [&](int tl, int c, uint32_t sc[2]) {
      sc[0] = sc[1] = 0u;
      const int64_t n = (t0 + tl) * 128 + r;
      if (tl >= ntiles || n >= p.N) return;
      const uint16_t* q = p.scales + n * p.lds + g0 + 4 * c;
#pragma unroll
      for (int h = 0; h < 4; ++h)
        if (4 * c + h < ng) sc[h >> 1] |= (uint32_t)__ldg(q + h) << (16 * (h & 1));
    };
    uint32_t sc[2];
    ld_scales(0, 0, sc);
    cluster_wait();
    const uint32_t push_base = rank == 0 ? 0u : map_rank(ypart + rank * p.tiles_cap * 128 + r, 0);
    const uint32_t push_bar = rank == 0 ? 0u : map_rank(&ctl->red_bar, 0);
    for (int s = 0; s < S; ++s) {
      // scales of the next stage, loaded one stage ahead
      const int ntl = (ch + 1 == nch) ? tile + 1 : tile, nc = (ch + 1 == nch) ? 0 : ch + 1;
      uint32_t sc_next[2];
      ld_scales(ntl, nc, sc_next);
      const bool ok = wait_or_abort(&ctl->d_full[db], duse & 1, ctl);
      if (!__all_sync(kFull, ok)) break;  // the tensor-memory loads below are warp-collective
      tc_fence_after();
      float d[4][4];
#pragma unroll
      for (int h = 0; h < 4; ++h) tmem_ld4(tmem + lane_addr + kDcol + (uint32_t)(db * 64 + h * 16), d[h]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->d_free[db]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 z = ztab[4 * ch + h];  // zero for a group past the slice
        const float sh = __half2float(__ushort_as_half((uint16_t)(sc[h >> 1] >> (16 * (h & 1)))));
        acc = fmaf(sh * z.y, (d[h][0] + d[h][1]) + d[h][2] + z.x, acc);
      }
      if (ch + 1 == nch) {  // this row of the tile is complete: into rank 0's slot of this rank
        if (rank == 0)
          ypart[tile * 128 + r] = acc;
        else
          st_async_f32(push_base + (uint32_t)(tile * 128 * 4), acc, push_bar);
        acc = 0.0f;
      }
      sc[0] = sc_next[0];
      sc[1] = sc_next[1];
      tile = ntl;
      ch = nc;
      if (++db == kDbuf) { db = 0; ++duse; }
    }
  }

  // ---- rank 0 adds the kcl partial sums (fixed order) once the others' have landed
  tc_fence_before();
  __syncthreads();
  if (warp < kEpiWarp0) cluster_wait();
  if (rank == 0) {
    bool ok = true;
    if (p.kcl > 1) {
      ok = mbar_wait(&ctl->red_bar, 0);
      if (!ok && threadIdx.x == 0) atomicOr(&g_gemv_fault, kFaultTimeout);
    }
    if (ok && !ctl->abort) {
      for (int i = threadIdx.x; i < ntiles * 128; i += kThreads) {
        const int64_t n = t0 * 128 + i;
        if (n >= p.N) continue;
        float sum = ypart[i];
        for (int q = 1; q < p.kcl; ++q) sum += ypart[q * p.tiles_cap * 128 + i];
        p.y[n] = sum;
      }
    }
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f != nullptr) return f;
  void* q = nullptr;
  cudaDriverEntryPointQueryResult r;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) != cudaSuccess ||
      r != cudaDriverEntryPointSuccess)
    return nullptr;
  f = reinterpret_cast<EncodeTiledFn>(q);
  fn.store(f, std::memory_order_release);
  return f;
}

size_t smem_bytes(int groups_cap, int tiles_cap, int kcl) {
  return 1024 + (size_t)kRing * kSlotBytes + (size_t)groups_cap * kGroupBBytes + kZeroBytes +
         (size_t)groups_cap * sizeof(float2) + (size_t)kcl * tiles_cap * 128 * sizeof(float) + sizeof(Ctl);
}

// Clusters of kcl CTAs that can be resident at once (a cluster lives on one
// GPC, so large clusters do not tile all SMs); queried once per device.
int max_active_clusters(int kcl) {
  static std::atomic<int> cache[64][4];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int slot = kcl == 1 ? 0 : kcl == 2 ? 1 : kcl == 4 ? 2 : 3;
  int v = cache[dev][slot].load(std::memory_order_acquire);
  if (v > 0) return v;
  const int smem = device_max_smem_optin();
  if (cudaFuncSetAttribute(k_gemv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(device_sm_count() * kcl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)kcl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&v, k_gemv_tc, &cfg) != cudaSuccess || v < 1) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev][slot].store(v, std::memory_order_release);
  return v;
}

}  // namespace

unsigned int take_fault_gemv() {
  unsigned int f = 0, z = 0;
  if (cudaMemcpyFromSymbol(&f, g_gemv_fault, sizeof(f)) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (f != 0) (void)cudaMemcpyToSymbol(g_gemv_fault, &z, sizeof(z));
  return f;
}

// Work split: kcl in {1, 2, 4, 8} CTAs per cluster share a tile range and
// split its K groups; at most as many clusters as can be resident at once
// (one wave).  The choice minimises the stages of the busiest CTA (a stage
// is four groups of one 128-row tile); ties go to fewer CTAs.  Returns false
// when this kernel does not suit the shape.
bool plan_gemv_tc(int64_t N, int64_t K, int* kcl_out, int* clusters_out) {
  if (N <= 0 || K <= 0 || K % 128 != 0) return false;
  const int64_t G = K / 128, T = (N + 127) / 128;
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  const int64_t smem_max = device_max_smem_optin();
  int64_t best = 0, best_kcl = 0, best_c = 0;
  for (int64_t kcl = 1; kcl <= 8; kcl *= 2) {
    if (kcl > G) break;
    int64_t c = max_active_clusters((int)kcl);
    if (c > sms / kcl) c = sms / kcl;
    if (c > T) c = T;
    if (c < 1) continue;
    const int64_t gcap = 4 * (((G + kcl - 1) / kcl + 3) / 4);
    const int64_t tcap = (T + c - 1) / c;
    if ((int64_t)smem_bytes((int)gcap, (int)tcap, (int)kcl) > smem_max) continue;
    const int64_t cost = tcap * (gcap / 4);
    if (best_kcl == 0 || cost < best || (cost == best && c * kcl < best_c * best_kcl)) {
      best = cost;
      best_kcl = kcl;
      best_c = c;
    }
  }
  if (best_kcl == 0) return false;
  *kcl_out = (int)best_kcl;
  *clusters_out = (int)best_c;
  return true;
}

cudaError_t launch_gemv_tc(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N,
                           int64_t K, const void* x, float* y, bool prefetch, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int64_t G = K / 128, T = (N + 127) / 128;
  int kcl_i = 0, c_i = 0;
  if (!plan_gemv_tc(N, K, &kcl_i, &c_i)) return cudaErrorNotSupported;
  const int64_t best_kcl = kcl_i, best_c = c_i;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)(K / 4), (cuuint64_t)N};
  const cuuint64_t gstride[1] = {(cuuint64_t)ldc};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p{};
  p.scales = scales;
  p.lds = lds;
  p.N = N;
  p.K = K;
  p.x = static_cast<const uint16_t*>(x);
  p.y = y;
  p.kcl = (int)best_kcl;
  p.clusters = (int)best_c;
  p.groups_cap = (int)(4 * (((G + best_kcl - 1) / best_kcl + 3) / 4));
  p.tiles_cap = (int)((T + best_c - 1) / best_c);
  p.prefetch = prefetch ? 1 : 0;
  const size_t smem = smem_bytes(p.groups_cap, p.tiles_cap, p.kcl);
  // raise the kernel's shared-memory limit only when a launch needs more
  static std::atomic<int> smem_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev].load(std::memory_order_acquire) < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(k_gemv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int cur = smem_set[dev].load(std::memory_order_acquire);
    while (cur < (int)smem && !smem_set[dev].compare_exchange_weak(cur, (int)smem)) {
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(best_c * best_kcl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)best_kcl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_gemv_tc, map, p);
}

}  // namespace tq
