// k_gemv_tc.cu -- decode GEMV / skinny GEMM (tq_gemv, 2-bit or base-3 codes,
// M = 1..16) on tcgen05 tensor cores with the weight operand in tensor memory.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} t[n][k] * x'[m][k],  x' = FWHT-128(x)
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
//   pass through shared memory (whose bandwidth would not cover them).  The
//   weights are unpacked once whatever M is.
// * Activations as three e4m3 pieces (the B operand, N = 16 columns).  Per
//   group of 128 and row m of x the rotated activations are scaled by a
//   power of two 2^E with max |x' 2^E| in [128, 256), and each scaled value
//   v is written as p1 + p2 + p3, p1 = e4m3(v), p2 = e4m3(v - p1),
//   p3 = e4m3(v - p1 - p2) (nearest even; the residuals are exact in fp32):
//   within max(2^-12 |v|, 2^-8) of v, finer than an fp16 rounding of x' for
//   all but the smallest elements.  Values that meet the 4c weights are
//   stored divided by 4 (exact).  The 3M pieces go to the 16 B columns in
//   kP passes per 32-wide K step, each pass one MMA accumulating into the
//   same 16 accumulator columns: M <= 5 (one pass, column 3m + piece),
//   M <= 8 (two passes; columns m and 8 + m), M <= 16 (three passes, one
//   piece each, column m).  For M <= 2 only B rows 0..7 are stored; rows
//   8..15 come from a shared zero block.
// * Groups.  Each group's MMAs write their own 16 accumulator columns, so
//   the thread of row n reads one group's inner products with x'[m] (after
//   adding the columns that share an m), adds the correction term
//   -2^-9 sum_k (p1 + p2 + p3)(k) and multiplies by s[n][g] 2^(9 - E) in fp32
//   -- the scale is applied to each group's inner product.
//
// Base-3 codes (five trits per byte, byte = sum_i d_i 3^i, d = t + 1;
// mhpq.cn/news/1159370 sec. 3.1, tighter packing) take the same pipeline with
// stages of five groups (640 trits = 128 bytes per row, so a stage starts on
// a byte).  Digits come out of a 32-bit word of four code bytes with integer
// arithmetic on two 16-bit lanes: p_k = floor(b / 3^k) from
// floor(v / 3) = (85 v + 80) >> 8 (exact for v <= 242), the high bytes of
// the lanes gathered by one byte permute, and digit i of every byte is
// p_i - 3 p_(i+1) in one multiply-add on the whole word (no carry or borrow
// crosses a byte).  Digit word i of code word q (digit i of its four bytes)
// goes to tensor-memory column 5 q + i of the stage, so a group of 128 trits
// no longer fills whole columns of its own: its MMAs run over a window of
// 8-column K steps that covers its trits (5 or 6 steps), and the activations
// of that group sit at the matching places of a B block of its own, zero
// elsewhere, so the trits of the neighbouring groups that share the window
// add nothing.  Digits are e4m3 bytes d * 2^-9 (no 4c class), and
// sum_k t x = sum_k d x - sum_k x as before.
//
// The 2:4-sparse codes (tq_gemv_sparse24) take the 2-bit pipeline with a
// table-driven unpack into natural-order columns (see the SP instance below).
//
// Work split: a cluster of kcl CTAs owns a range of 128-row tiles; CTA rank r
// owns the r-th slice of the K groups and rotates only that slice of x.  A
// CTA walks (tile, four-group) stages with four warp roles that hand buffers
// to one another through mbarriers, so each runs ahead on its own:
//   warp 16      (one lane) TMA-loads 128 x 128-byte code tiles (four groups,
//                128-byte swizzle) into a ring of kRing slots, one per stage;
//   warps 0-15   two teams of eight take the even and the odd stages; warp w
//                unpacks groups 2 ((w / 4) % 2) .. +1 of its stage for rows
//                32 (w % 4) .. +31 into one of kAbuf A buffers in tensor
//                memory;
//   warps 17-18  warp 17 allocates tensor memory; warp 17 + t issues the
//                MMAs of each stage of team t into accumulator buffer t;
//   warps 19-22  read the accumulators of their 32 rows and apply the scales.
// The partial sums of the K slices are reduced across the cluster by rows:
// rank q owns rows R q .. R q + R - 1 of every tile (R = ceil(128 / kcl); the
// last rank owns what is left), the others push their
// partial sums of those rows into its shared memory (st.async, counted on an
// mbarrier there), and rank q adds the kcl partials in rank order and writes
// y.  Every wait is bounded in time; a wait that runs out sets the library's
// GEMV status word and the CTA winds down (pending copies and MMAs are
// waited for, tensor memory is freed, the cluster barrier is still met).
#include <cuda.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "tq_internal.h"

namespace tq {

__device__ unsigned int g_gemv_fault;  // bit 1: a bounded wait ran out; bit 2: activations out of range

namespace {

constexpr int kDecWarps = 16;                 // two teams of 8: even and odd decode stages
constexpr int kTeamWarps = 8;
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;                  // warps 17, 18 issue the MMAs of team 0, 1
constexpr int kEpiWarp0 = 19;                 // warps 19-22: epilogue
constexpr int kThreads = 32 * 23;             // + 4 epilogue warps (19-22)
// code slots in flight (one stage each); an even count, so that slot
// s % kRing always belongs to team s % 2
constexpr int kRing = 4;
constexpr int kDbuf = 2;                      // accumulator buffers: buffer t belongs to team t's stages
constexpr int kSlotBytes = 128 * 128;         // 128 rows x 128 bytes of codes: one stage
constexpr int kZeroBytes = 288;               // B rows 8..15 of the 8-row layout (two core matrices 144 apart)
constexpr int kTmemCols = 512;                // one CTA per SM
constexpr int kAbufMax = 3;
constexpr uint32_t kFaultTimeout = 2u;
constexpr uint32_t kFaultRange = 4u;  // a group's rotated activations outside what the e4m3 pieces represent

// Per code format: groups per stage (kGS), weight (A) buffers in tensor
// memory (kAbuf, one stage each), A columns per stage (kACols) and K steps
// of 32 per group in the B layout (kSteps).  2-bit: four groups of 32
// columns; base-3: five groups in 160 columns, each group's MMAs over a
// window of up to six K steps.  A buffer b of a stage: columns b kACols ..;
// D buffer b: kDcol + b kDCols .. (16 accumulator columns per group).
template <bool B3> struct Fmt;
template <> struct Fmt<false> { static constexpr int kGS = 4, kAbuf = 3, kACols = 128, kSteps = 4; };
template <> struct Fmt<true> { static constexpr int kGS = 5, kAbuf = 2, kACols = 160, kSteps = 6; };
template <bool B3>
struct FmtGeo : Fmt<B3> {
  using F = Fmt<B3>;
  // stages between two uses of one A buffer by one team (buffers alternate
  // between the teams when their count is odd)
  static constexpr int kAPeriod = (F::kAbuf % 2) ? 2 * F::kAbuf : F::kAbuf;
  static constexpr uint32_t kDCols = 16 * F::kGS;
  static constexpr uint32_t kDcol = (uint32_t)(F::kACols * F::kAbuf);
  static_assert(kDcol + kDCols * kDbuf <= kTmemCols, "tensor memory budget");
  static_assert(F::kAbuf <= kAbufMax, "barrier arrays");
};

// Base-3 group windows: group h of a stage (trits 128 h .. 128 h + 127, in
// bytes 25.6 h ..) starts at A column kWin0[h] (a multiple of 8) and spans
// kWinN[h] K steps of 8 columns.
constexpr int win0(int h) { return h == 0 ? 0 : h == 1 ? 24 : h == 2 ? 56 : h == 3 ? 88 : 120; }
constexpr int winn(int h) { return (h == 0 || h == 4) ? 5 : 6; }

// kind::f8f6f4: fp32 accumulator, A = B = e4m3, both K-major, N = 16, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// B layouts by how many rows of x they hold (kMM): kP MMA passes per 32-wide
// K step, kRows B rows stored per pass (8: rows 8..15 are read from the zero
// block).  One pass of one K step (a "unit") holds kRows / 8 core matrices
// (8 rows x 16 bytes) for k 0..15 and the same for k 16..31 at kLbo; the 16
// bytes of padding after each make the prologue's stores conflict-free
// (kLbo / 4 = 4 and kUnit / 4 = 8 banks, mod 32).  A group's units are
// stored pass-major: unit (pass, K step i) at (4 pass + i) kUnit.
template <int V> struct Lay;
template <> struct Lay<1> { static constexpr int kP = 1, kRows = 8, kMM = 2; };
template <> struct Lay<2> { static constexpr int kP = 1, kRows = 16, kMM = 5; };
template <> struct Lay<3> { static constexpr int kP = 2, kRows = 16, kMM = 8; };
template <> struct Lay<4> { static constexpr int kP = 3, kRows = 16, kMM = 16; };

template <int V, bool B3>
struct Geo {
  static constexpr int kP = Lay<V>::kP, kRows = Lay<V>::kRows, kMM = Lay<V>::kMM;
  static constexpr int kGS = Fmt<B3>::kGS, kSteps = Fmt<B3>::kSteps;
  static constexpr int kLbo = 16 * kRows + 16;
  static constexpr int kUnit = 2 * kLbo;
  static constexpr int kGroupB = kSteps * kP * kUnit;
  static constexpr int kZs = (kMM + 1) & ~1;       // ztab entries per group (even: read in pairs)
  static constexpr int kCw = kRows == 8 ? 8 : 16;  // accumulator columns read per group
  static constexpr int kGw = kMM > 5 ? 1 : 2;      // groups read per tensor-memory wait
  static constexpr int kScAhead = kMM > 5 ? 3 : 4; // stages the epilogue loads scales ahead
  static_assert(kLbo % 128 == 16 && kUnit % 128 == 32, "bank-spreading padding");
  static_assert(3 * kMM <= kP * (kRows == 8 ? 8 : 16), "pieces fit the B columns");
};

// B column (pass, row) that carries piece q (0..2) of row m of x.  The
// epilogue adds the accumulator columns of one m: 3m .. 3m + 2 (one pass),
// m and 8 + m (two passes), m (three passes).
template <int V>
__device__ __forceinline__ void piece_slot(int m, int q, int& pass, int& row) {
  if constexpr (Lay<V>::kP == 1) {
    pass = 0;
    row = 3 * m + q;
  } else if constexpr (Lay<V>::kP == 2) {
    pass = q >> 1;
    row = q == 1 ? 8 + m : m;
  } else {
    pass = q;
    row = m;
  }
}

int variant_of(int64_t M) { return M <= 2 ? 1 : M <= 5 ? 2 : M <= 8 ? 3 : 4; }

// Largest cluster (K split) the planner uses: 16, a non-portable size (the
// kernels opt in before such a launch), taken only when no cluster of at most
// 8 -- the portable limit -- fits the activations of one launch
constexpr int kMaxPortable = 8, kMaxCluster = 16;

// Rows of a 128-row tile each cluster rank reduces (the last rank: the rest)
__host__ __device__ constexpr int rows_per_rank(int kcl) { return (128 + kcl - 1) / kcl; }

// A buffer b holds the stages s with s % kAbuf == b, so its stages alternate
// between the teams (and MMA warps).  Its barriers are kept per team, which
// gives every barrier one sequential producer and one sequential consumer and
// so keeps each waiter within one phase of the barrier (a parity wait cannot
// pass on an older phase):
//   a_full[b][t]  team t's decode of a stage in b -> MMA warp t;
//   a_free[b][t]  the reads of b by the MMA warp of the stage before -> team t,
//                 which writes b next.
// With three buffers (2-bit) a buffer alternates between the teams (every
// 6th stage is team t's in buffer b); with two (base-3) buffer t is team t's.
struct Ctl {
  uint64_t full[kRing];      // TMA -> decoders (slot s % kRing: always team s % 2)
  uint64_t empty[kRing];     // decoders -> TMA
  uint64_t a_full[kAbufMax][2]; // decoders -> MMA
  uint64_t a_free[kAbufMax][2]; // MMA -> decoders
  uint64_t d_full[kDbuf]; // MMA -> epilogue
  uint64_t d_free[kDbuf]; // epilogue -> MMA
  uint64_t red_bar;       // this rank's rows: the other ranks' partial sums have landed
  unsigned long long wait_ns;  // limit of every bounded wait of this launch
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const uint16_t* scales;
  int64_t lds;
  int64_t N, K;
  const uint16_t* x;  // bf16, M rows of ldx
  int64_t ldx;
  float* y;           // M rows of ldy
  int64_t ldy;
  int M;
  int kcl;         // CTAs per cluster (K split)
  int clusters;    // tile ranges: cluster c owns [c*T/clusters, (c+1)*T/clusters)
  int groups_cap;  // groups per CTA the shared layout holds (multiple of 4)
  int tiles_cap;   // tiles per cluster the partial sums hold
  int prefetch;    // codes and scales are ready before the preceding kernel ends
  // Failure-path test: CTA stall_cta (-1: none) never issues the copy of its
  // first stage of codes, so its waits run out; wait_ns bounds every wait.
  int stall_cta;
  unsigned long long wait_ns;
  // Layout variants: FWHT block size (64, 128 or 256), log2 of the scale
  // group over 128 (0 or 1), and the number of 128-groups of K that meet
  // rotated activations (K / 128 without a residual pass; with one, K counts
  // the codes of both passes and groups from g_rot on meet x unrotated).
  int blk;
  int lgs;
  int64_t g_rot;
  // Chained decode (compiled into the LAYOUT instance only).  xr: x already
  // rotated (fp32 x' of M rows of ldxr), read instead of x and not rotated
  // again.  xnext: also write FWHT-128(y) in fp32 (M rows of ldxn; N a
  // multiple of 128) -- rank 0 of each cluster then reduces all 128 rows of
  // its tiles, so that it holds whole groups.
  const float* xr;
  int64_t ldxr;
  float* xnext;
  int64_t ldxn;
  int64_t ypart_floats;  // partial sums in shared memory (floats)
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

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t r[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tcgen05.ld of 8 / 16 consecutive columns of this warp's 32 lanes; the
// registers are valid after tmem_ld_wait on them.
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Waits for this thread's tensor-memory loads; the registers pass through an
// empty asm after the wait so that no use of them is scheduled before it.
template <int G, int N>
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&a)[G][N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(a[g][i]));
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


// FWHT-128 with lane 4i + j holding elements 16i + j + 4b (b = 0..3): stages
// h = 1, 2 pair lanes l ^ 1, l ^ 2; h = 4, 8 stay in the lane (b ^ 1, b ^ 2);
// h = 16, 32, 64 pair lanes l ^ 4, l ^ 8, l ^ 16.  The stages run in the
// order h = 1, 2, 4, ..., 64 with the lower index keeping a + b, then * c,
// so the result equals the staged fp32 definition bit for bit.
template <bool kH64 = true>
__device__ __forceinline__ void fwht128_strided_stages(float v[4], int lane) {
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
  if constexpr (kH64) shfl_stage(16);
}

__device__ __forceinline__ void fwht128_strided(float v[4], int lane) {
  fwht128_strided_stages(v, lane);
#pragma unroll
  for (int b = 0; b < 4; ++b) v[b] = __fmul_rn(v[b], kInvSqrt128);
}

// The layout variants on the same lane layout (fp32, staged order, bit for
// bit the definition): 64-blocks stop before the stage h = 64 (lanes l ^ 16)
// and multiply by 1/8; a 256-block also rotates the other 128-group of its
// block (partner, same lanes), then runs the stage h = 128 between the two
// (the lower group keeps a + b) and multiplies by 1/16.
__device__ __forceinline__ void rotate_group(float v[4], int lane, int blk, const uint16_t* partner, bool upper) {
  if (blk == 128) {
    fwht128_strided(v, lane);
  } else if (blk == 64) {
    fwht128_strided_stages<false>(v, lane);
#pragma unroll
    for (int b = 0; b < 4; ++b) v[b] = __fmul_rn(v[b], 0.125f);
  } else {
    float o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) o[b] = __uint_as_float((uint32_t)ld_in_u16(partner + 4 * b) << 16);
    fwht128_strided_stages(v, lane);
    fwht128_strided_stages(o, lane);
#pragma unroll
    for (int b = 0; b < 4; ++b) v[b] = __fmul_rn(upper ? __fsub_rn(o[b], v[b]) : __fadd_rn(v[b], o[b]), 0.0625f);
  }
}

// The five base-3 digits of the four code bytes of w (byte b = sum_i d_i 3^i,
// b <= 242): d[i] holds digit i of byte j in its byte j.  p_k = floor(b / 3^k)
// comes from p_(k-1) with floor(v / 3) = (85 v + 80) >> 8 (exact for
// v <= 242) on two 16-bit lanes per word (bytes 0, 2 and 1, 3), whose high
// bytes one byte permute gathers; then digit i = p_i - 3 p_(i+1) for the
// whole word at once (3 p_(i+1) <= p_i <= 242 in every byte: no carry or
// borrow crosses a byte).
__device__ __forceinline__ void trits5(uint32_t w, uint32_t d[5]) {
  uint32_t lo = w & 0x00ff00ffu, hi = __byte_perm(w, 0u, 0x4341u);
  uint32_t p[5];
  p[0] = w;
#pragma unroll
  for (int k = 1; k < 5; ++k) {
    const uint32_t vl = lo * 85u + 0x00500050u, vh = hi * 85u + 0x00500050u;
    p[k] = __byte_perm(vl, vh, 0x7351u);
    if (k < 4) {
      lo = __byte_perm(vl, 0u, 0x4341u);
      hi = __byte_perm(vh, 0u, 0x4341u);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = p[i] - 3u * p[i + 1];
  d[4] = p[4];
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
  if (mbar_wait_abortable(bar, parity, &ctl->abort, ctl->wait_ns)) return true;
  atomicOr(&g_gemv_fault, kFaultTimeout);
  return false;
}

// The 2:4-sparse codes (SP): a group of 128 weights is 24 code bytes (16
// bytes of low nibbles, 8 of high bit pairs; one 6-bit code per quad of four
// consecutive k: pattern and two trits), a stage of four groups 96 bytes per
// row, copied without swizzle.  Each code becomes one 32-bit tensor-memory
// column -- the quad's four weights as e4m3 bytes c * 2^-9, c = t + 1 (1 for
// the pruned positions and for the codes 54..63 the quantiser never writes)
// -- through a 64-entry table replicated for every lane (lane l reads copy l,
// so the 32 lookups of a warp fall on 32 banks).  The columns then hold k in
// natural order, and the prologue writes x' bytes in natural order too (no
// odd-class scaling).
constexpr int kSpTabBytes = 64 * 32 * 4;

__host__ __device__ constexpr uint32_t sp24_word(uint32_t c) {
  if (c >= 54) return 0x01010101u;
  const uint32_t p = c / 9, r = c % 9;
  const uint32_t i0 = p < 3 ? 0u : (p < 5 ? 1u : 2u);
  const uint32_t i1 = p == 0 ? 1u : (p == 1 ? 2u : (p == 2 ? 3u : (p == 3 ? 2u : 3u)));
  uint32_t w = 0x01010101u;
  w = (w & ~(0xffu << (8 * i0))) | ((r / 3) << (8 * i0));
  w = (w & ~(0xffu << (8 * i1))) | ((r % 3) << (8 * i1));
  return w;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Shared memory (1024-aligned): [code ring][B: groups_cap x kGroupB][zeros kZeroBytes]
// [ztab: groups_cap x kZs x {pw Zt, pw}][partial sums: tiles_cap x kcl x M x R]
// [SP: code table, kSpTabBytes][Ctl]
// LAYOUT: the layout variants' parameters (blk, lgs, g_rot) and the chained
// decode (xr, xnext) are read; without it the kernel is compiled for the
// method's own layout only.
template <int V, bool B3, bool LAYOUT, bool SP = false>
__global__ void __launch_bounds__(kThreads, 1) k_gemv_tc(const __grid_constant__ CUtensorMap cmap, const Params p) {
  static_assert(!SP || (!B3 && !LAYOUT), "2:4 codes: the method's own layout only");
  using Gm = Geo<V, B3>;
  using Fg = FmtGeo<B3>;
  constexpr int kGS = Fg::kGS, kAbuf = Fg::kAbuf, kAPeriod = Fg::kAPeriod;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = smem;
  unsigned char* bsm = ring + kRing * kSlotBytes;
  unsigned char* zero = bsm + p.groups_cap * Gm::kGroupB;
  float2* ztab = reinterpret_cast<float2*>(zero + kZeroBytes);
  float* ypart = reinterpret_cast<float*>(ztab + p.groups_cap * Gm::kZs);
  uint32_t* sptab = reinterpret_cast<uint32_t*>(ypart + p.ypart_floats);
  Ctl* ctl = reinterpret_cast<Ctl*>(reinterpret_cast<unsigned char*>(sptab) + (SP ? kSpTabBytes : 0));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  // kcl is 1 .. 8; the slices use 32-bit division (the host keeps G kcl
  // below 2^31; 64-bit division is a long instruction sequence)
  const uint32_t kcl = (uint32_t)p.kcl;
  const int64_t cluster = blockIdx.x / kcl;
  const int64_t G = p.K / 128;
  // K slice of this rank: whole groups (2-bit), whole five-group stages (base-3,
  // so that a slice starts on a code byte); nch stages per tile
  int64_t g0, g1;
  if constexpr (B3) {
    const int64_t nst = (G + 4) / 5;
    g0 = 5 * (int64_t)((uint32_t)nst * rank / kcl);
    g1 = std::min<int64_t>(5 * (int64_t)((uint32_t)nst * (rank + 1) / kcl), G);
  } else if constexpr (SP) {
    // slices of whole group pairs (G is even), so that every stage's copy
    // starts on a multiple of 48 code bytes (the copy engine needs 16); a
    // short last stage reads the next slice's codes, which meet zero x'
    // pieces and zero scales
    g0 = 2 * (int64_t)((uint32_t)(G / 2) * rank / kcl);
    g1 = 2 * (int64_t)((uint32_t)(G / 2) * (rank + 1) / kcl);
  } else {
    g0 = (int64_t)((uint32_t)G * rank / kcl);
    g1 = (int64_t)((uint32_t)G * (rank + 1) / kcl);
  }
  const int ng = (int)(g1 - g0), nch = (ng + kGS - 1) / kGS;
  // bytes one stage's copy delivers: 128 rows x 128 code bytes (96 for 2:4 codes)
  constexpr uint32_t kStageTx = SP ? 128u * 96u : (uint32_t)kSlotBytes;
  // TMA x (bytes) of stage lc of the slice
  auto stage_x = [&](int lc) -> int {
    return B3 ? (int)((g0 / 5 + lc) * 128) : (int)((g0 + 4 * lc) * (SP ? 24 : 32));
  };
  const int64_t T = (p.N + 127) / 128;
  int64_t t0, t1;
  {
    // the first T % clusters clusters take one tile more: CTAs of a GEMV
    // launched behind another start in index order as SMs free up, so the
    // last to start (on the SMs the previous GEMV held longest) get less work
    // (32-bit: the planner keeps T below 2^31)
    const int64_t base = (uint32_t)T / (uint32_t)p.clusters, extra = T - base * p.clusters;
    t0 = cluster * base + (cluster < extra ? cluster : extra);
    t1 = t0 + base + (cluster < extra ? 1 : 0);
  }
  const int ntiles = (int)(t1 - t0);
  const int S = ntiles * nch;  // stages (ring loads) of this CTA
  const int M = p.M;
  // rank q reduces rows R q .. R q + Rq - 1 of every tile (R = ceil(128 /
  // kcl), Rq = R but for the last rank, which takes what is left); with xnext
  // rank 0 reduces all of them (R = 128: the other ranks own none).  R is
  // also the stride of the partial sums in shared memory.
  const bool all_rows = LAYOUT && p.xnext != nullptr;
  const int R = all_rows ? 128 : rows_per_rank(p.kcl);
  const int Rq = all_rows ? (rank == 0 ? 128 : 0) : min(R, 128 - (int)rank * R);

  int issued_loads = 0;
  auto fill_ring = [&]() {
    for (; issued_loads < S && issued_loads < kRing; ++issued_loads) {
      const int l = issued_loads, tile = l / nch, lc = l - tile * nch;
      if (l == 0 && (int)blockIdx.x == p.stall_cta) continue;  // failure-path test: never arrives
      mbar_arrive_expect_tx(&ctl->full[l], kStageTx);
      tma_load_2d(smem_u32(ring + l * kSlotBytes), &cmap, stage_x(lc), (int)((t0 + tile) * 128), &ctl->full[l]);
    }
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], kTeamWarps);
    }
    for (int i = 0; i < kAbuf; ++i) {
      for (int t = 0; t < 2; ++t) {
        mbar_init(&ctl->a_full[i][t], kTeamWarps);
        mbar_init(&ctl->a_free[i][t], 1);
      }
    }
    for (int i = 0; i < kDbuf; ++i) {
      mbar_init(&ctl->d_full[i], 1);
      mbar_init(&ctl->d_free[i], 4);
    }
    mbar_init(&ctl->red_bar, 1);
    // every other rank sends its partial sums of this rank's rows: ntiles x M x R floats each
    if (p.kcl > 1)
      mbar_arrive_expect_tx(&ctl->red_bar, (uint32_t)((p.kcl - 1) * ntiles * M * Rq * 4));
    ctl->abort = 0;
    ctl->wait_ns = p.wait_ns;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // zero B (unused rows and groups), the zero block and ztab
  {
    uint4* z4 = reinterpret_cast<uint4*>(bsm);
    const int n16 = (p.groups_cap * Gm::kGroupB + kZeroBytes) / 16;
    for (int i = threadIdx.x; i < n16; i += kThreads) z4[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < p.groups_cap * Gm::kZs; i += kThreads) ztab[i] = make_float2(0.0f, 0.0f);
    if constexpr (SP)
      for (int i = threadIdx.x; i < kSpTabBytes / 4; i += kThreads) sptab[i] = sp24_word((uint32_t)(i >> 5));
  }
  tc_fence_before();
  __syncwarp();  // a warp reaches the block barrier whole (lanes may have diverged)
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  // This CTA's reduction barrier is armed: the other ranks may push once they
  // pass the matching wait (epilogue warps before their first push, every
  // other warp before it exits -- each thread waits exactly once).
  cluster_arrive();

  // Inputs may come from the preceding kernel on the stream: x always waits
  // for it; codes and scales too unless the caller declared them ready, in
  // which case the ring fills while that kernel finishes.  The TMA warp fills
  // the ring while the other warps rotate x; block-wide barriers must not be
  // reached by part of a warp, hence the __syncwarp.
  if (p.prefetch && warp == kTmaWarp && lane == 0) fill_ring();
  pdl_wait();
  pdl_launch_dependents();
  if (!p.prefetch && warp == kTmaWarp && lane == 0) fill_ring();
  if (warp == kTmaWarp) __syncwarp();

  // ---- rotate this CTA's slice of each row of x and split it into three
  // e4m3 pieces.  Lane 4i + j holds elements k = 16i + j + 4b (b = 0..3) of
  // its group: these are the four B bytes that meet one code class j of one
  // code word i, so the lane writes each piece as one 32-bit word.
  const int pwarp = warp < kTmaWarp ? warp : warp - 1;  // rotation warps: all but the TMA warp
  for (int it = pwarp; it < ng * M && warp != kTmaWarp; it += kThreads / 32 - 1) {
    const int gl = it / M, m = it - gl * M;
    const int i8 = lane >> 2, jc = lane & 3;
    float v[4];
    if constexpr (LAYOUT) {
      if (p.xr != nullptr) {  // x' given (the method's layout only): read, no rotation
        const float* xg = p.xr + m * p.ldxr + (g0 + gl) * 128 + 16 * i8 + jc;
#pragma unroll
        for (int b = 0; b < 4; ++b) v[b] = ld_in_f32(xg + 4 * b);
      } else {
      // a residual layout's second half of the codes meets x itself
      const int64_t gg = g0 + gl;
      const bool rot = gg < p.g_rot;
      const int64_t xc = rot ? gg : gg - p.g_rot;
      const uint16_t* xrow = p.x + m * p.ldx + 16 * i8 + jc;
      const uint16_t* xg = xrow + xc * 128;
#pragma unroll
      for (int b = 0; b < 4; ++b) v[b] = __uint_as_float((uint32_t)ld_in_u16(xg + 4 * b) << 16);
      if (rot) rotate_group(v, lane, p.blk, xrow + (xc ^ 1) * 128, (xc & 1) != 0);
      }
    } else {
      const uint16_t* xg = p.x + m * p.ldx + (g0 + gl) * 128 + 16 * i8 + jc;
#pragma unroll
      for (int b = 0; b < 4; ++b) v[b] = __uint_as_float((uint32_t)ld_in_u16(xg + 4 * b) << 16);
      fwht128_strided(v, lane);
    }
    // the group's max |x'| in one warp reduction: non-negative fp32 values
    // order like their bit patterns
    const float amax = __uint_as_float(__reduce_max_sync(
        kFull, __float_as_uint(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))))));
    int E = amax > 0.0f ? 134 - (int)((__float_as_uint(amax) >> 23) & 0xffu) : 0;  // max |x' 2^E| in [128, 256)
    // |x'| >= 2^108 (or infinite) or 0 < max |x'| < 2^-93 in a group: the
    // pieces under the clamped scale would saturate or flush -- recorded
    if (E < -100 || E > 100) {
      if (lane == 0) atomicOr(&g_gemv_fault, kFaultRange);
      E = E < -100 ? -100 : 100;
    }
    const float up = __uint_as_float((uint32_t)(127 + E) << 23);
    const float pw = __uint_as_float((uint32_t)(127 + 9 - E) << 23);
    // 2-bit: odd classes j meet the 4c weights, so their values are stored
    // divided by 4; base-3 digits are all plain d * 2^-9
    const float cls = (!B3 && !SP && (jc & 1)) ? 0.25f : 1.0f, acls = (!B3 && !SP && (jc & 1)) ? 4.0f : 1.0f;
    float u[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) u[b] = v[b] * up * cls;
    float zs = 0.0f;
    unsigned char* gbase = bsm + gl * Gm::kGroupB;
    // 2-bit: K step i / 2 of the group; k'' = 16 (i % 2) + 4 j + b inside it,
    // at byte (k'' / 16) kLbo + 16 row + k'' % 16 of the unit of the piece's
    // pass.  Base-3: element e of group h of its stage is trit 128 h + e, in
    // code byte j = trit / 5 (digit trit % 5), which sits in byte j % 4 of
    // A column 5 (j / 4) + digit; its place in the group's window of K steps
    // is kappa = 4 (column - window start) + j % 4.
    // 2:4 codes: natural order, k'' = 16 (i % 2) + j + 4 b
    unsigned char* gdst = gbase + (i8 >> 1) * Gm::kUnit + (i8 & 1) * Gm::kLbo + (SP ? jc : 4 * jc);
    int boff[4];
    if constexpr (B3) {
      const int h = (int)((g0 + gl) % 5);
      const int w0 = win0(h);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int tr = 128 * h + 16 * i8 + jc + 4 * b, j = tr / 5, dg = tr - 5 * j;
        const int kap = 4 * (5 * (j >> 2) + dg - w0) + (j & 3);
        boff[b] = (kap >> 5) * Gm::kUnit + ((kap >> 4) & 1) * Gm::kLbo + (kap & 15);
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      float r0, r1, r2, r3;
      const uint32_t lo = to_e4m3x2(u[0], u[1], r0, r1), hi = to_e4m3x2(u[2], u[3], r2, r3);
      int pass, row;
      piece_slot<V>(m, q, pass, row);
      const uint32_t word = (lo & 0xffffu) | (hi << 16);
      if constexpr (B3) {
        unsigned char* rdst = gbase + pass * Gm::kSteps * Gm::kUnit + (row >> 3) * 128 + (row & 7) * 16;
#pragma unroll
        for (int b = 0; b < 4; ++b) rdst[boff[b]] = (unsigned char)(word >> (8 * b));
      } else if constexpr (SP) {
        unsigned char* rdst = gdst + pass * 4 * Gm::kUnit + (row >> 3) * 128 + (row & 7) * 16;
#pragma unroll
        for (int b = 0; b < 4; ++b) rdst[4 * b] = (unsigned char)(word >> (8 * b));
      } else {
        *reinterpret_cast<uint32_t*>(gdst + pass * 4 * Gm::kUnit + (row >> 3) * 128 + (row & 7) * 16) = word;
      }
      zs += (r0 + r1) + (r2 + r3);
      u[0] -= r0;
      u[1] -= r1;
      u[2] -= r2;
      u[3] -= r3;
    }
    zs = warp_sum(zs * acls);
    if (lane == 0) ztab[gl * Gm::kZs + m] = make_float2(pw * (zs * -0.001953125f), pw);  // pw * (-2^-9 sum), pw
  }
  fence_async_smem();  // B written by ordinary stores, read by the tensor cores
  __syncwarp();  // a warp reaches the block barrier whole (lanes may have diverged)
  __syncthreads();

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int l = issued_loads, slot = l % kRing, use = l / kRing, tile = l / (nch > 0 ? nch : 1), lc = l - tile * nch;
      for (; l < S; ++l) {
        if (!wait_or_abort(&ctl->empty[slot], (use - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&ctl->full[slot], kStageTx);
        tma_load_2d(smem_u32(ring + slot * kSlotBytes), &cmap, stage_x(lc), (int)((t0 + tile) * 128),
                    &ctl->full[slot]);
        if (++slot == kRing) { slot = 0; ++use; }
        if (++lc == nch) { lc = 0; ++tile; }
      }
      // loads issued but possibly never consumed: let them land before exit
      for (int q = (l > kRing ? l - kRing : 0); q < l; ++q)
        (void)mbar_wait(&ctl->full[q % kRing], (q / kRing) & 1, ctl->wait_ns);
    }
    __syncwarp();
  } else if (warp < kDecWarps) {
    // ------------------------------------------------------------ decoders
    // team (warp / 8) takes the stages of its parity, so two stages are
    // unpacked at once; warp w unpacks half (w / 4) % 2 of the stage's code
    // bytes (2-bit: groups 2 ((w / 4) % 2) .. +1) for rows 32 (w % 4) .. +31
    const int team = warp >> 3, quad = warp & 3, gh = (warp >> 2) & 1;
    const int r = quad * 32 + lane;  // row inside the tile = tensor-memory lane
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
    const uint32_t rx = (uint32_t)(r & 7), rbase = (uint32_t)(r * 128);
    const uint32_t ring_u32 = smem_u32(ring);
    uint32_t off[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) off[q] = rbase + ((((uint32_t)(4 * gh + q)) ^ rx) << 4);
    if constexpr (SP) {  // rows of 96 bytes, no swizzle: this half's two groups are bytes 48 gh .. + 47
#pragma unroll
      for (int q = 0; q < 4; ++q) off[q] = (uint32_t)(r * 96 + 48 * gh + 16 * (q < 3 ? q : 2));
    }
    const uint32_t tab_lane = smem_u32(sptab) + 4u * (uint32_t)lane;  // this lane's copy of the code table
    int slot = team, use = 0;  // ring slot of stage s and its use count (s % kRing, s / kRing)
    for (int s = team; s < S; s += 2) {
      // A buffer ab last held stage s - kAbuf, whose MMAs are the
      // ((s - kAbuf) / kAPeriod)-th completion a_free[ab][team] counts
      const int ab = s % kAbuf;
      bool ok = wait_or_abort(&ctl->full[slot], use & 1, ctl);
      uint4 c[4];
#pragma unroll
      for (int q = 0; q < (SP ? 3 : 4); ++q) c[q] = ok ? lds_u4(ring_u32 + slot * kSlotBytes + off[q]) : make_uint4(0, 0, 0, 0);
      // The slot is released only after the tensor-memory stores below have
      // consumed c: the refill is a TMA (async-proxy) write, which is not
      // ordered after shared-memory loads whose values have not returned yet,
      // so an earlier release let the next stage's codes reach some lanes.
      if (s >= kAbuf) ok = wait_or_abort(&ctl->a_free[ab][team], ((s - kAbuf) / kAPeriod) & 1, ctl) && ok;
      if (!__all_sync(kFull, ok)) break;  // the tensor-memory stores below are warp-collective
      // order the stores below after the MMAs that read this buffer (observed
      // through the barrier): without this fence they may overtake those reads
      tc_fence_after();
      const uint32_t acol = tmem + lane_addr + (uint32_t)(ab * Fg::kACols);
      if constexpr (B3) {
        // 16 code words: word q of this half -> columns 80 gh + 5 q .. + 4
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t w[8] = {c[2 * h].x, c[2 * h].y, c[2 * h].z, c[2 * h].w,
                                 c[2 * h + 1].x, c[2 * h + 1].y, c[2 * h + 1].z, c[2 * h + 1].w};
          uint32_t a[40];
#pragma unroll
          for (int i = 0; i < 8; ++i) trits5(w[i], &a[5 * i]);
          const uint32_t col = acol + (uint32_t)(80 * gh + 40 * h);
          tmem_st32(col, a);
          tmem_st8(col + 32, a + 32);
        }
      } else if constexpr (SP) {
        // group h of this half: low-nibble words nw (8 codes each) and
        // high-bit words hw (16 codes each); code j -> column 32 (2 gh + h) + j
        const uint32_t nw[2][4] = {{c[0].x, c[0].y, c[0].z, c[0].w}, {c[1].z, c[1].w, c[2].x, c[2].y}};
        const uint32_t hw[2][2] = {{c[1].x, c[1].y}, {c[2].z, c[2].w}};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t code = ((nw[h][j >> 3] >> (4 * (j & 7))) & 15u) | (((hw[h][j >> 4] >> (2 * (j & 15))) & 3u) << 4);
            a[j] = lds_u32(tab_lane + (code << 7));
          }
          tmem_st32(acol + (uint32_t)((2 * gh + h) * 32), a);
        }
      } else {
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
          tmem_st32(acol + (uint32_t)((2 * gh + h) * 32), a);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->empty[slot]);
        mbar_arrive(&ctl->a_full[ab][team]);
      }
      slot += 2;
      if (slot >= kRing) { slot -= kRing; ++use; }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ MMA issue
    // The whole warp walks the stages (its loop state stays warp-uniform);
    // lane 0 waits; one elected lane issues the MMAs and the commits.
    const uint32_t bsm_u32 = smem_u32(bsm), zero_u32 = smem_u32(zero);
    // B descriptor of unit (pass, K step i) of local group gl: start = bsm +
    // kGroupB gl + kUnit (4 pass + i).  In the 8-row layout the stride to the
    // next 8 rows points at the zero block, so moving the start up by d moves
    // that stride down by d; in the 16-row layout it is 128.
    constexpr bool k8 = Gm::kRows == 8;
    const uint64_t desc_g0 = smem_desc_plain(bsm_u32, Gm::kLbo, k8 ? zero_u32 - bsm_u32 : 128u);
    constexpr uint64_t kStepU = (uint64_t)(Gm::kUnit >> 4) - (k8 ? ((uint64_t)(Gm::kUnit >> 4) << 32) : 0);
    constexpr uint64_t kStepG = (uint64_t)(Gm::kGroupB >> 4) - (k8 ? ((uint64_t)(Gm::kGroupB >> 4) << 32) : 0);
    // warp kMmaWarp + t takes the stages of parity t (team t), accumulating
    // into D buffer t
    const int t = warp - kMmaWarp;
    int s = t, ch = t % (nch > 0 ? nch : 1), duse = 0;  // ch: stage inside the tile
    for (; s < S; s += 2) {
      // stage s is the (s / kAPeriod)-th that a_full[ab][t] counts
      const int ab = s % kAbuf;
      // only lane 0 waits; one elected lane issues the tensor-core work
      bool ok = true;
      if (lane == 0) {
        ok = wait_or_abort(&ctl->a_full[ab][t], (s / kAPeriod) & 1, ctl);
        if (ok && duse > 0) ok = wait_or_abort(&ctl->d_free[t], (duse - 1) & 1, ctl);
      }
      if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t d0 = tmem + Fg::kDcol + (uint32_t)t * Fg::kDCols, a0 = tmem + (uint32_t)(ab * Fg::kACols);
        uint64_t bg = desc_g0 + (uint64_t)(kGS * ch) * kStepG;
#pragma unroll
        for (int h = 0; h < kGS; ++h) {
          // 2-bit: the group's own 32 columns; base-3: its window of K steps
          constexpr int kNs = Gm::kSteps;
          const int ns = B3 ? winn(h) : 4;
          const uint32_t ah = a0 + (uint32_t)(B3 ? win0(h) : 32 * h);
#pragma unroll
          for (int pass = 0; pass < Gm::kP; ++pass) {
#pragma unroll
            for (int i = 0; i < kNs; ++i)
              if (i < ns)
                mma_f8_tmem_a(d0 + h * 16, ah + i * 8, bg + (uint64_t)(kNs * pass + i) * kStepU,
                              (pass | i) != 0 ? 1u : 0u);
          }
          bg += kStepG;
        }
        // the team that writes buffer ab next (stage s + kAbuf)
        mma_commit(&ctl->a_free[ab][(kAbuf & 1) ? t ^ 1 : t]);
        mma_commit(&ctl->d_full[t]);
      }
      __syncwarp();
      ++duse;
      ch += 2;
      while (ch >= nch) ch -= nch;
    }
    // every MMA this warp issued must be complete before tensor memory is freed
    if (s - 2 >= 0 && lane == 0) (void)mbar_wait(&ctl->d_full[t], ((s - 2) >> 1) & 1, ctl->wait_ns);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int kMM = Gm::kMM, kCw = Gm::kCw;
    const int quad = warp & 3;  // warps 19..22 reach tensor-memory lanes 32 (warp % 4) ..
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    float acc[kMM];
#pragma unroll
    for (int m = 0; m < kMM; ++m) acc[m] = 0.0f;
    int tile = 0, ch = 0, db = 0, duse = 0;
    // Raw fp16 scales of the stage's kGS groups for this row (groups past
    // the slice: 0).  Each stays in its own register until it is used, so
    // the loads remain in flight meanwhile.
    auto ld_scales = [&](int tl, int c, uint32_t (&sc)[kGS]) {
#pragma unroll
      for (int h = 0; h < kGS; ++h) sc[h] = 0u;
      const int64_t n = (t0 + tl) * 128 + r;
      if (tl >= ntiles || n >= p.N) return;
      if constexpr (LAYOUT) {
        const uint16_t* q = p.scales + n * p.lds;
        const int64_t gc = g0 + kGS * c;  // a scale per 2^lgs groups of 128
#pragma unroll
        for (int h = 0; h < kGS; ++h)
          if (kGS * c + h < ng) sc[h] = ld_in_u16(q + ((gc + h) >> p.lgs));
      } else {
        const uint16_t* q = p.scales + n * p.lds + g0 + kGS * c;
#pragma unroll
        for (int h = 0; h < kGS; ++h)
          if (kGS * c + h < ng) sc[h] = ld_in_u16(q + h);
      }
    };
    // The scales are loaded kAhead stages before they are used (a DRAM miss
    // takes longer than a stage).  The stage loop is unrolled by kAhead so
    // that slot j of the ring is always the same registers: a slot is read
    // (converted) at the start of its stage, then reloaded for the stage
    // kAhead later; (ltl, lc) is the next stage to load.
    constexpr int kAhead = Gm::kScAhead;
    uint32_t scq[kAhead][kGS];
    int ltl = 0, lc = 0;
#pragma unroll
    for (int i = 0; i < kAhead; ++i) {
      ld_scales(ltl, lc, scq[i]);
      if (++lc == nch) { lc = 0; ++ltl; }
    }
    cluster_wait();
    // this row's partial sums go to the rank that reduces it
    const uint32_t owner = (uint32_t)(r / R);
    const int rr = r - (int)owner * R;
    const bool local = owner == rank;
    const uint32_t push_base = local ? 0u : map_rank(ypart, owner);
    const uint32_t push_bar = local ? 0u : map_rank(&ctl->red_bar, owner);
    const float4* ztab4 = reinterpret_cast<const float4*>(ztab);
    // one stage; false when a wait gave up
    auto stage = [&](uint32_t (&slot)[kGS]) -> bool {
      float sh[kGS];
#pragma unroll
      for (int h = 0; h < kGS; ++h) sh[h] = __half2float(__ushort_as_half((uint16_t)slot[h]));
      ld_scales(ltl, lc, slot);
      if (++lc == nch) { lc = 0; ++ltl; }
      const int ntl = (ch + 1 == nch) ? tile + 1 : tile, nc = (ch + 1 == nch) ? 0 : ch + 1;
      const bool ok = wait_or_abort(&ctl->d_full[db], duse & 1, ctl);
      if (!__all_sync(kFull, ok)) return false;  // the tensor-memory loads below are warp-collective
      tc_fence_after();
      // kGw groups per tensor-memory wait (fewer registers for the wide layouts)
      constexpr int kHp = (kGS + Gm::kGw - 1) / Gm::kGw;
#pragma unroll
      for (int hp = 0; hp < kHp; ++hp) {
        uint32_t d[Gm::kGw][kCw];
        const uint32_t dcol = tmem + lane_addr + Fg::kDcol + (uint32_t)db * Fg::kDCols + (uint32_t)(hp * 16 * Gm::kGw);
#pragma unroll
        for (int u = 0; u < Gm::kGw; ++u) {
          if (Gm::kGw * hp + u < kGS) {
            tmem_ld(dcol + 16 * u, d[u]);
          } else {
#pragma unroll
            for (int i = 0; i < kCw; ++i) d[u][i] = 0u;
          }
        }
        tmem_ld_wait(d);
        if (hp == kHp - 1) {  // the whole accumulator buffer has been read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->d_free[db]);
        }
#pragma unroll
        for (int u = 0; u < Gm::kGw; ++u) {
          const int h = Gm::kGw * hp + u;
          if (h >= kGS) continue;
          float vs[kMM];
#pragma unroll
          for (int m = 0; m < kMM; ++m) {
            if constexpr (Gm::kP == 1)
              vs[m] = (__uint_as_float(d[u][3 * m]) + __uint_as_float(d[u][3 * m + 1])) + __uint_as_float(d[u][3 * m + 2]);
            else if constexpr (Gm::kP == 2)
              vs[m] = __uint_as_float(d[u][m]) + __uint_as_float(d[u][m + 8]);
            else
              vs[m] = __uint_as_float(d[u][m]);
          }
          // {pw Zt, pw} of (group, m) and (group, m + 1); zero past the slice and for m >= M
          const float4* z = ztab4 + (((kGS * ch + h) * Gm::kZs) >> 1);
#pragma unroll
          for (int m = 0; m < kMM; m += 2) {
            if (m < M) {
              const float4 zz = z[m >> 1];
              acc[m] = fmaf(sh[h], fmaf(zz.y, vs[m], zz.x), acc[m]);
              if (m + 1 < kMM) acc[m + 1] = fmaf(sh[h], fmaf(zz.w, vs[m + 1], zz.z), acc[m + 1]);
            }
          }
        }
      }
      if (ch + 1 == nch) {  // this row of the tile is complete: to the rank that reduces it
        const int base = (tile * p.kcl + (int)rank) * M * R + rr;
        if (local) {
#pragma unroll
          for (int m = 0; m < kMM; ++m)
            if (m < M) ypart[base + m * R] = acc[m];
        } else {
#pragma unroll
          for (int m = 0; m < kMM; ++m)
            if (m < M) st_async_f32(push_base + (uint32_t)((base + m * R) * 4), acc[m], push_bar);
        }
#pragma unroll
        for (int m = 0; m < kMM; ++m) acc[m] = 0.0f;
      }
      tile = ntl;
      ch = nc;
      if (++db == kDbuf) { db = 0; ++duse; }
      return true;
    };
    bool go = true;
    for (int s0 = 0; go && s0 < S; s0 += kAhead) {
#pragma unroll
      for (int j = 0; j < kAhead; ++j)
        if (go && s0 + j < S) go = stage(scq[j]);
    }
  }

  // ---- each rank adds the kcl partial sums of its rows (in rank order) once
  // the others' have landed
  tc_fence_before();
  __syncwarp();  // a warp reaches the block barrier whole (lanes may have diverged)
  __syncthreads();
  if (warp < kEpiWarp0) cluster_wait();
  bool ok = true;
  if (p.kcl > 1) {
    ok = mbar_wait(&ctl->red_bar, 0, ctl->wait_ns);
    if (ok) mbar_acquire_cluster(&ctl->red_bar, 0);
    if (!ok && threadIdx.x == 0) atomicOr(&g_gemv_fault, kFaultTimeout);
  }
  if (ok && !ctl->abort && all_rows) {
    // rank 0: y of every row, then FWHT-128 of each (tile, row of x) group as
    // the next layer's x'; warp w takes groups w, w + 23, ..  Lane 4i + j
    // holds rows 16i + j + 4b of the tile (the transform's lane layout).
    if (rank == 0) {
      for (int it = warp; it < ntiles * M; it += kThreads / 32) {
        const int tl = it / M, m = it - tl * M;
        const int64_t n0 = (t0 + tl) * 128;
        float v[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int rr = 16 * (lane >> 2) + (lane & 3) + 4 * b;
          const float* src = ypart + (tl * p.kcl * M + m) * 128 + rr;
          float sum = src[0];
          for (int q = 1; q < p.kcl; ++q) sum += src[q * M * 128];
          p.y[m * p.ldy + n0 + rr] = sum;
          v[b] = sum;
        }
        fwht128_strided(v, lane);
#pragma unroll
        for (int b = 0; b < 4; ++b) p.xnext[m * p.ldxn + n0 + 16 * (lane >> 2) + (lane & 3) + 4 * b] = v[b];
      }
    }
  } else if (ok && !ctl->abort) {
    const int total = ntiles * M * Rq;
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int j = i / Rq, rr = i - j * Rq, tl = j / M, m = j - tl * M;
      const int64_t n = (t0 + tl) * 128 + (int64_t)rank * R + rr;
      if (n >= p.N) continue;
      const float* src = ypart + (tl * p.kcl * M + m) * R + rr;
      float sum = src[0];
      for (int q = 1; q < p.kcl; ++q) sum += src[q * M * R];
      p.y[m * p.ldy + n] = sum;
    }
  }
  if (warp == kMmaWarp) {
    __syncwarp();  // the reduction loop above may leave the warp diverged
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

// Partial-sum floats per (tile, row of x) in a rank's shared memory: the kcl
// ranks' sums of its R rows, or of all 128 when rank 0 reduces every row
// (chained decode)
int64_t ypart_cols(int64_t kcl, bool all_rows) { return kcl * (all_rows ? 128 : rows_per_rank((int)kcl)); }
// The partial-sum area in floats, whole 128-byte blocks (what follows it, the
// control block's mbarriers and the 2:4 code table, stays aligned)
int64_t ypart_floats_of(int64_t tiles_cap, int64_t M, int64_t ycols) { return (tiles_cap * M * ycols + 31) / 32 * 32; }

template <int V, bool B3>
size_t smem_bytes_v(int64_t groups_cap, int64_t tiles_cap, int64_t M, int64_t ycols) {
  return 1024 + (size_t)kRing * kSlotBytes + (size_t)groups_cap * Geo<V, B3>::kGroupB + kZeroBytes +
         (size_t)groups_cap * Geo<V, B3>::kZs * sizeof(float2) +
         (size_t)ypart_floats_of(tiles_cap, M, ycols) * sizeof(float) + sizeof(Ctl);
}

template <bool B3>
size_t smem_bytes_f(int64_t groups_cap, int64_t tiles_cap, int64_t M, int64_t ycols) {
  switch (variant_of(M)) {
    case 1: return smem_bytes_v<1, B3>(groups_cap, tiles_cap, M, ycols);
    case 2: return smem_bytes_v<2, B3>(groups_cap, tiles_cap, M, ycols);
    case 3: return smem_bytes_v<3, B3>(groups_cap, tiles_cap, M, ycols);
    default: return smem_bytes_v<4, B3>(groups_cap, tiles_cap, M, ycols);
  }
}

size_t smem_bytes(bool b3, int64_t groups_cap, int64_t tiles_cap, int64_t M, int64_t ycols, bool sp = false) {
  return (b3 ? smem_bytes_f<true>(groups_cap, tiles_cap, M, ycols)
             : smem_bytes_f<false>(groups_cap, tiles_cap, M, ycols)) +
         (sp ? (size_t)kSpTabBytes : 0);
}

// Groups per CTA the shared layout holds: the largest K slice a rank gets,
// in whole stages (2-bit: slices of whole groups; base-3: of five-group
// stages).
int64_t groups_cap_of(bool b3, int64_t G, int64_t kcl, bool sp = false) {
  if (b3) return 5 * (((G + 4) / 5 + kcl - 1) / kcl);
  if (sp) return 4 * ((2 * ((G / 2 + kcl - 1) / kcl) + 3) / 4);  // slices of group pairs
  return 4 * (((G + kcl - 1) / kcl + 3) / 4);
}

// Clusters of kcl CTAs that can be resident at once (a cluster lives on one
// GPC, so large clusters do not tile all SMs); queried once per device.  The
// layouts share block size and shared-memory limit, so one query serves all.
int max_active_clusters(int kcl) {
  static std::atomic<int> cache[64][kMaxCluster + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || kcl < 1 || kcl > kMaxCluster) return 0;
  const int slot = kcl;
  int v = cache[dev][slot].load(std::memory_order_acquire);
  if (v > 0) return v;
  const int smem = device_max_smem_optin();
  if (cudaFuncSetAttribute(k_gemv_tc<1, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  if (kcl > kMaxPortable &&
      cudaFuncSetAttribute(k_gemv_tc<1, false, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
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
  if (cudaOccupancyMaxActiveClusters(&v, k_gemv_tc<1, false, false>, &cfg) != cudaSuccess || v < 1) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev][slot].store(v, std::memory_order_release);
  return v;
}

template <int V, bool B3, bool LAYOUT, bool SP = false>
cudaError_t launch_v(const CUtensorMap& map, const Params& p, size_t smem, cudaStream_t s) {
  // raise the kernel's shared-memory limit only when a launch needs more
  static std::atomic<int> smem_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev].load(std::memory_order_acquire) < (int)smem) {
    cudaError_t e =
        cudaFuncSetAttribute(k_gemv_tc<V, B3, LAYOUT, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int cur = smem_set[dev].load(std::memory_order_acquire);
    while (cur < (int)smem && !smem_set[dev].compare_exchange_weak(cur, (int)smem)) {
    }
  }
  if (p.kcl > kMaxPortable) {  // a non-portable cluster size: opt in once per device
    static std::atomic<bool> np_set[64];
    if (!np_set[dev].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(k_gemv_tc<V, B3, LAYOUT, SP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      np_set[dev].store(true, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.clusters * p.kcl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)p.kcl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_gemv_tc<V, B3, LAYOUT, SP>, map, p);
}

// Cost model of the busiest CTA, in units of 1/24 stage: a stage streams
// 16 KB of codes (about 0.4 us per SM at the HBM rate), and rotating and
// splitting one (group, row of x) in the prologue costs about 1/24 of that.
constexpr int64_t kItemsPerStage = 24;

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

// Work split for M rows of x: kcl in 1 .. 8 CTAs per cluster share a
// tile range and split its K groups; at most as many clusters as can be
// resident at once (one wave).  The choice minimises the cost model of the
// busiest CTA (its stages -- 128 code bytes of one 128-row tile -- and its
// prologue items) over kcl = 1, 2, 4, 8, ties going to fewer CTAs.  A
// cluster of 3, 6 or 7 (46, 23, 15 resident on 152 SMs) replaces that choice
// only when it costs at least 10 % less and gives the busiest CTA at most one
// tile more, since the model leaves out what these cost beyond their stages.
// Measured: 5120x5120 (M = 1 .. 4) and 5120x27648 (M = 1) gain from clusters
// of 6 (5120x5120 also from 3, less); 2048x2048 at M = 1 lost with 6 at a
// 4 % lower modelled cost.  Clusters of 5 are left out: they lost wherever
// measured (5120x5120 in the decode step, 27648x5120 at M = 2 .. 16), below
// the power-of-two plans they replaced.  When no cluster of at most 8 fits the
// activations in shared memory, a cluster of 16 (non-portable; 7 resident)
// gives each CTA a sixteenth of K, so that one launch still takes all rows of
// x (5120x27648 at M = 16 instead of two launches).  Returns false when no
// split fits in shared memory.
bool plan_gemv_tc(int64_t N, int64_t K, int64_t M, int fmt, int* kcl_out, int* clusters_out, bool all_rows) {
  if (N <= 0 || K <= 0 || K % 128 != 0 || M < 1 || M > 16) return false;
  if (fmt != TQ_PACK_2BIT && fmt != TQ_PACK_BASE3 && fmt != kFmtSparse24) return false;
  const bool b3 = fmt == TQ_PACK_BASE3, sp = fmt == kFmtSparse24;
  const int64_t G = K / 128, T = (N + 127) / 128;
  if (sp && (G % 2 != 0 || G < 4)) return false;  // 2:4 rows: whole 16-byte pitches, at least one full stage
  const int64_t gs = b3 ? 5 : 4;
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  const int64_t smem_max = device_max_smem_optin();
  int64_t best = 0, best_kcl = 0, best_c = 0, best_t = 0, best_p = 0;
  if (G * kMaxCluster >= (int64_t(1) << 31) || T >= (int64_t(1) << 31)) return false;  // the kernel's 32-bit slice and tile arithmetic
  const int64_t most = b3 ? (G + gs - 1) / gs : (sp ? G / 2 : G);  // a group (2-bit), pair (2:4) or stage (base-3) per rank
  // the last entry, 16, is tried only when none of the others fits
  static constexpr int kOrder[] = {1, 2, 4, 8, 3, 6, 7, 16};
  constexpr int kOrders = (int)(sizeof(kOrder) / sizeof(kOrder[0]));
  for (int i = 0; i < kOrders; ++i) {
    const int64_t kcl = kOrder[i];
    const bool pow2 = i < 4 || i == kOrders - 1;
    if (kcl > most) continue;
    // 3, 6 and 7 refine a plan of the first four; 16 is the last resort
    if (i == kOrders - 1 ? best_kcl != 0 : (!pow2 && best_kcl == 0)) continue;
    int64_t c = max_active_clusters((int)kcl);
    if (c > sms / kcl) c = sms / kcl;
    if (c > T) c = T;
    if (c < 1) continue;
    const int64_t gcap = groups_cap_of(b3, G, kcl, sp);
    const int64_t gslice = b3 ? std::min(gcap, G) : (G + kcl - 1) / kcl;
    const int64_t tcap = (T + c - 1) / c;
    if ((int64_t)smem_bytes(b3, gcap, tcap, M, ypart_cols(kcl, all_rows), sp) > smem_max) continue;
    const int64_t cost = tcap * (gcap / gs) * kItemsPerStage + gslice * M;
    const bool better = best_kcl == 0 || cost < best || (cost == best && c * kcl < best_c * best_kcl);
    if (better && (pow2 || (10 * cost <= 9 * best_p && tcap <= best_t + 1))) {
      best = cost;
      best_kcl = kcl;
      best_c = c;
      if (pow2) {  // the refinement is measured against the first four's plan
        best_t = tcap;
        best_p = cost;
      }
    }
  }
  if (best_kcl == 0) return false;
  *kcl_out = (int)best_kcl;
  *clusters_out = (int)best_c;
  return true;
}

// Launches that take M rows of x: the rows are split into the fewest
// launches of at most m_fit rows each, m_fit the most rows one launch's
// shared-memory layout holds (the B layout grows with M), at most
// kMaxLaunches launches; 0 when the shape does not suit the kernel.
constexpr int kMaxLaunches = 4;
int gemv_tc_launches(int64_t N, int64_t K, int64_t M, int fmt, bool all_rows) {
  int kcl = 0, c = 0;
  for (int64_t m = M; m >= 1; --m) {
    if (!plan_gemv_tc(N, K, m, fmt, &kcl, &c, all_rows)) continue;
    const int64_t l = (M + m - 1) / m;
    return l <= kMaxLaunches ? (int)l : 0;
  }
  return 0;
}

cudaError_t launch_gemv_tc(const uint8_t* codes, int64_t ldc, int fmt, const uint16_t* scales, int64_t lds,
                           int64_t N, int64_t K, const void* x, int64_t ldx, int64_t M, float* y, int64_t ldy,
                           bool prefetch, cudaStream_t s, bool test_stall, const GemvLayout* lay,
                           const GemvChain* chain) {
  if (N == 0) return cudaSuccess;
  const bool b3 = fmt == TQ_PACK_BASE3, sp = fmt == kFmtSparse24;
  if (sp && (lay != nullptr || chain != nullptr || test_stall)) return cudaErrorNotSupported;
  const int64_t G = K / 128, T = (N + 127) / 128;
  const bool all_rows = chain != nullptr && chain->xnext != nullptr;
  if (all_rows && N % 128 != 0) return cudaErrorNotSupported;
  int kcl = 0, clusters = 0;
  if (!plan_gemv_tc(N, K, M, fmt, &kcl, &clusters, all_rows)) {
    // several launches, the rows of x split as evenly as possible
    const int l = gemv_tc_launches(N, K, M, fmt, all_rows);
    if (l < 2) return cudaErrorNotSupported;
    int64_t m0 = 0;
    for (int i = 0; i < l; ++i) {
      const int64_t mi = (M - m0) / (l - i);
      GemvChain ci{};
      if (chain != nullptr) {
        ci = *chain;
        if (ci.xr != nullptr) ci.xr += m0 * ci.ldxr;
        if (ci.xnext != nullptr) ci.xnext += m0 * ci.ldxn;
      }
      const uint16_t* xi = chain != nullptr && chain->xr != nullptr ? static_cast<const uint16_t*>(x)
                                                                     : static_cast<const uint16_t*>(x) + m0 * ldx;
      cudaError_t e = launch_gemv_tc(codes, ldc, fmt, scales, lds, N, K, xi, ldx, mi, y + m0 * ldy, ldy, prefetch, s,
                                     test_stall && i == 0, lay, chain != nullptr ? &ci : nullptr);
      if (e != cudaSuccess) return e;
      m0 += mi;
    }
    return cudaSuccess;
  }
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap map;
  // 2-bit rows hold K / 4 code bytes; base-3 rows ceil(K / 5) rounded up to
  // 16 (zero padding); 2:4 rows 24 bytes per group, copied 96 bytes (a
  // stage) per row without swizzle.  Boxes past the row read zeros, which
  // meet zero activations.
  const int64_t row_bytes = b3 ? ((K + 4) / 5 + 15) / 16 * 16 : (sp ? 24 * G : K / 4);
  const cuuint64_t gdim[2] = {(cuuint64_t)row_bytes, (cuuint64_t)N};
  const cuuint64_t gstride[1] = {(cuuint64_t)ldc};
  const cuuint32_t box[2] = {sp ? 96u : 128u, 128};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, sp ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p{};
  p.scales = scales;
  p.lds = lds;
  p.N = N;
  p.K = K;
  p.x = static_cast<const uint16_t*>(x);
  p.ldx = ldx;
  p.y = y;
  p.ldy = ldy;
  p.M = (int)M;
  p.kcl = kcl;
  p.clusters = clusters;
  p.groups_cap = (int)groups_cap_of(b3, G, kcl, sp);
  p.tiles_cap = (int)((T + clusters - 1) / clusters);
  p.prefetch = prefetch ? 1 : 0;
  p.stall_cta = test_stall ? 0 : -1;
  p.wait_ns = test_stall ? kTestWaitLimitNs : kWaitLimitNs;
  p.blk = lay != nullptr ? lay->block : 128;
  p.lgs = (lay != nullptr && lay->group == 256) ? 1 : 0;
  p.g_rot = (lay != nullptr && lay->residual) ? G / 2 : G;
  if (chain != nullptr) {
    p.xr = chain->xr;
    p.ldxr = chain->ldxr;
    p.xnext = chain->xnext;
    p.ldxn = chain->ldxn;
  }
  p.ypart_floats = ypart_floats_of(p.tiles_cap, M, ypart_cols(kcl, all_rows));
  const int64_t smem_max = device_max_smem_optin();
  // More than half an SM's shared memory, so no two CTAs share an SM whatever
  // the register count: each allocates all of tensor memory, and a second
  // one would block in tcgen05.alloc while its cluster peers wait for it.
  const size_t smem =
      std::max(smem_bytes(b3, p.groups_cap, p.tiles_cap, M, ypart_cols(kcl, all_rows), sp), (size_t)(smem_max / 2 + 1024));
  const bool lv = (lay != nullptr && (lay->block != 128 || lay->group != 128 || lay->residual)) ||
                  (chain != nullptr && (chain->xr != nullptr || chain->xnext != nullptr));
  const int v = variant_of(M);
  if (sp)
    return v == 1 ? launch_v<1, false, false, true>(map, p, smem, s)
           : v == 2 ? launch_v<2, false, false, true>(map, p, smem, s)
           : v == 3 ? launch_v<3, false, false, true>(map, p, smem, s) : launch_v<4, false, false, true>(map, p, smem, s);
  if (lv) {
    if (b3) return v == 1 ? launch_v<1, true, true>(map, p, smem, s) : v == 2 ? launch_v<2, true, true>(map, p, smem, s)
                 : v == 3 ? launch_v<3, true, true>(map, p, smem, s) : launch_v<4, true, true>(map, p, smem, s);
    return v == 1 ? launch_v<1, false, true>(map, p, smem, s) : v == 2 ? launch_v<2, false, true>(map, p, smem, s)
           : v == 3 ? launch_v<3, false, true>(map, p, smem, s) : launch_v<4, false, true>(map, p, smem, s);
  }
  if (b3) return v == 1 ? launch_v<1, true, false>(map, p, smem, s) : v == 2 ? launch_v<2, true, false>(map, p, smem, s)
               : v == 3 ? launch_v<3, true, false>(map, p, smem, s) : launch_v<4, true, false>(map, p, smem, s);
  return v == 1 ? launch_v<1, false, false>(map, p, smem, s) : v == 2 ? launch_v<2, false, false>(map, p, smem, s)
         : v == 3 ? launch_v<3, false, false>(map, p, smem, s) : launch_v<4, false, false>(map, p, smem, s);
}

}  // namespace tq
