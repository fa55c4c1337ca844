// k_gemm.cu -- prefill GEMM (tq_gemm) on the 5th-generation tensor cores.
//
//   y[m][n] = sum_k x'[m][k] * (t[n][k] * s[n][k/128]),  fp32 accumulation
//
// Prefill (M = 2048 tokens) is the one dense contraction of the path, so it
// runs on tcgen05 MMA with accumulators in tensor memory.  The operands are
// fp16: x' comes from the rotation pre-pass (fp16, with an overflow flag) and
// the weight operand is t * s, which is exact in fp16 because s is an fp16
// number and t is -1, 0 or +1.  Folding the per-group scale into the operand
// applies it exactly where the group structure needs it, so one K-long
// accumulation covers all groups (equivalent to scaling each group's partial
// sum in an epilogue, without per-group accumulator traffic).
//
// One CTA computes a 256 (tokens) x bn (weight rows) tile, K in stages of 64;
// bn (a multiple of 16, at most 256) and the K split of a short last wave
// come from a cost model of the busiest SM (gemm_plan):
//   warp 8     (one lane) TMA-loads the 256 x 64 fp16 tile of x' (128-byte
//              swizzle, K-major) into the stage ring;
//   warps 0-7  decode the bn x 64 weight tile from 2-bit codes straight into
//              the same swizzled K-major layout (lane = weight row), then,
//              after the last stage, drain tensor memory to y: 32 x 32 fp32
//              blocks staged in the freed stage ring (128-byte swizzle) and
//              written by TMA stores, so y leaves as whole 128-byte lines and
//              the CTA does not wait for the writes to land;
//   warp 9     allocates tensor memory and (one lane) issues the MMAs: per
//              stage 2 (token halves) x 4 (K steps of 16) tcgen05.mma of
//              128 x bn x 16 into two fp32 accumulators (256 columns apart).
// When the tiles leave a last wave of few tiles (2048 x 5120 in 256-row tiles:
// 160 tiles on 152 SMs), those tiles are split along K instead (up to one
// segment per SM): each K segment runs as a CTA of its own and writes its
// fp32 partial tile to the workspace, and k_gemm_fixup adds the segments of
// every output in segment order and writes y (deterministic; no atomics, no
// CTA waits for another).
// Stages are handed over with mbarriers (TMA bytes, decoder arrivals, MMA
// completion via tcgen05.commit).  Every wait is bounded in time; a wait that
// runs out records bit 1 of the status word and the CTA winds down.
//
// The k order inside each 16-element chunk is 0,8,1,9,...,7,15 on both
// operands: the decoder produces (c_j, c_{j+8}) fp16 pairs from one 32-bit
// word of codes without shuffling, and the pre-pass stores x' in that order.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "tq_internal.h"

namespace tq {

namespace {

constexpr int BM = 256;  // tokens per CTA (two 128-row MMA tiles)
constexpr int BN = 256;  // most weight rows per CTA (MMA N); a launch uses bn <= BN
constexpr int BK = 64;   // k per stage: 128 bytes of fp16 = one swizzle row
constexpr int kStages = 3;
constexpr int kDecoders = 8;  // warps
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 32 * 10;
constexpr int kAStage = BM * BK * 2;  // 32 KB
constexpr int kBStage = BN * BK * 2;  // 32 KB
constexpr int kTmemCols = 512;
constexpr int kOutBox = 32;                         // output block: 32 rows x 32 fp32 (128-byte rows)
constexpr int kOutBlock = kOutBox * kOutBox * 4;    // 4 KB
constexpr int kOutSlots = 4;                        // staged blocks in flight per warp
constexpr uint32_t kFaultTimeout = 2u;  // status word bit

struct SmemCtl {
  uint64_t full_a[kStages];
  uint64_t full_b[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  unsigned long long wait_ns;  // limit of every bounded wait of this launch
  uint32_t tmem_base;
  int abort;
  uint8_t sp_tab[64];  // 2:4 codes: code -> the 2-bit code byte of its quad
};

// ---------------------------------------------------------------- PTX helpers

// Bulk tensor store of a staged shared-memory block, and the waits on the
// issuing thread's bulk groups (.read: the source may be reused).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset 1024), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);            // start address
  d |= (uint64_t)1 << 16;                              // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                    // stride byte offset
  d |= (uint64_t)1 << 46;                              // version
  d |= (uint64_t)2 << 61;                              // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N = bn, M = 128.
constexpr uint32_t idesc_f16(int bn) { return (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(128 >> 4) << 24); }

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%"
      "20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// (c_j, c_{j+8}) of a 16-code word -> fp16x2 (t_j * s, t_{j+8} * s), exact:
// OR the exponent of 2^(10-2jj) over the code bits, subtract 2^(10-2jj) + 1
// (gives t), multiply by s (exact: t is -1, 0 or +1).
template <int J>
__device__ __forceinline__ uint32_t ts_pair(uint32_t w, uint32_t w10, uint32_t s2) {
  constexpr int jj = J < 5 ? J : J - 5;
  constexpr uint32_t mask = 0x00030003u << (2 * jj);
  constexpr uint32_t magic = (uint32_t)(25 - 2 * jj) << 10;
  constexpr uint32_t magic2 = magic | (magic << 16);
  constexpr uint32_t bias = magic | (1u << (2 * jj));
  constexpr uint32_t bias2 = bias | (bias << 16);
  const uint32_t src = J < 5 ? w : w10;
  return hmul2_bits(hsub2_bits((src & mask) | magic2, bias2), s2);
}

struct Params {
  const uint8_t* codes;
  int64_t ldc;
  const uint16_t* scales;
  int64_t lds;
  int64_t N, K, M;
  float* y;
  int64_t ldy;
  uint32_t* flag;
  int n_tiles_m;
  int n_main;      // blocks below n_main compute whole tiles 0 .. n_main - 1
  int splits;      // K segments of each later tile (blocks n_main + u: tile n_main + u / splits)
  float* part;     // their partial tiles, [unit][BM][bn] fp32
  int bn;          // weight rows per tile (multiple of 16, <= BN)
  uint32_t idesc;  // idesc_f16(bn)
  int vec_store;  // y 16-byte aligned and ldy % 4 == 0: rows can take 16-byte stores
  int tma_y;      // ymap describes y (M x N fp32, row pitch ldy): blocks leave by TMA store
  int tma_part;   // pmap describes the partial tiles ([unit * BM + row][bn] fp32)
  // Failure-path test: CTA stall_cta (-1: none) never issues the copy of its
  // first x' stage, so its waits run out; wait_ns bounds every wait.
  int stall_cta;
  unsigned long long wait_ns;
  int lgs;  // one scale per 128 << lgs weights (layout variants: groups of 256)
  // Fused producer of the next layer's x': when xnext is set (whole tiles of
  // whole 128-column groups, no K split), the epilogue also writes
  // FWHT-128(y) rounded to fp16, in the GEMM's k order inside each 16-chunk,
  // to xnext ([M][ldxn]) and ORs fp16 overflow into *flag_next.
  uint16_t* xnext;
  int64_t ldxn;
  uint32_t* flag_next;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, SmemCtl* ctl, uint32_t* flag) {
  if (mbar_wait_abortable(bar, parity, &ctl->abort, ctl->wait_ns)) return true;
  atomicOr(flag, kFaultTimeout);
  return false;
}

// The 2-bit code byte of a quad of the 2:4 format's code c (9 p + 3 (t0 + 1)
// + (t1 + 1), kept positions of pattern p in the order (0,1) (0,2) (0,3)
// (1,2) (1,3) (2,3)): t + 1 at bits 2i for every position i, 1 (t = 0) at
// the pruned ones; codes 54..63 give a quad of zeros.
__device__ __forceinline__ uint32_t sp24_code_byte(uint32_t c) {
  if (c >= 54) return 0x55u;
  const uint32_t pt = c / 9, v = c - 9 * pt;
  const uint32_t i0 = pt < 3 ? 0u : (pt < 5 ? 1u : 2u);
  const uint32_t i1 = pt < 3 ? pt + 1 : (pt < 5 ? pt - 1 : 3u);
  uint32_t b = 0x55u;
  b = (b & ~(3u << (2 * i0))) | ((v / 3) << (2 * i0));
  b = (b & ~(3u << (2 * i1))) | ((v % 3) << (2 * i1));
  return b;
}

// EXT: the layout variants' scale groups (lgs) and the fused producer of the
// next layer's x' (xnext) are compiled in; without it the kernel is the
// method's plain GEMM.  SP: the weights are 2:4-sparse codes (24 bytes per
// group of 128: low nibbles, then high bit pairs); a stage's 16 codes are
// turned into the four 2-bit code words of its 64 weights through a 64-entry
// table and then decoded as usual.
template <bool EXT, bool SP = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
              const __grid_constant__ CUtensorMap pmap, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment (of the shared-window address) for the swizzled tiles
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* a_ring = smem;
  unsigned char* b_ring = smem + kStages * kAStage;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(b_ring + kStages * kBStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk_all = (int)(p.K / BK);
  // whole tile, or K segment [s0, s1) of a split tile (unit >= 0)
  int tile = (int)blockIdx.x, s0 = 0, s1 = nk_all, unit = -1;
  if (tile >= p.n_main) {
    unit = tile - p.n_main;
    tile = p.n_main + unit / p.splits;
    const int seg = unit % p.splits;
    s0 = nk_all * seg / p.splits;
    s1 = nk_all * (seg + 1) / p.splits;
  }
  const int tile_m = tile % p.n_tiles_m, tile_n = tile / p.n_tiles_m;
  const int bn = p.bn;
  const int64_t m0 = (int64_t)tile_m * BM, n0 = (int64_t)tile_n * bn;
  const int nk = s1 - s0;  // stages of this CTA

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->full_a[i], 1);
      mbar_init(&ctl->full_b[i], kDecoders);
      mbar_init(&ctl->empty[i], 1);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort = 0;
    if constexpr (SP) {
      for (int c = 0; c < 64; ++c) ctl->sp_tab[c] = (uint8_t)sp24_code_byte((uint32_t)c);
    }
    ctl->wait_ns = p.wait_ns;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();  // a warp reaches the block barrier whole (lanes may have diverged)
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_wait();  // x' and the status word come from the pre-pass

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- TMA (x')
    if (lane == 0) {
      int s = 0;
      for (; s < nk; ++s) {
        const int slot = s % kStages, use = s / kStages;
        if (use > 0 && !wait_or_abort(&ctl->empty[slot], (use - 1) & 1, ctl, p.flag)) break;
        if (s == 0 && (int)blockIdx.x == p.stall_cta) continue;  // failure-path test: never arrives
        mbar_arrive_expect_tx(&ctl->full_a[slot], kAStage);
        tma_load_2d(smem_u32(a_ring + slot * kAStage), &xmap, (s0 + s) * BK, (int)m0, &ctl->full_a[slot]);
      }
      // loads issued but possibly not consumed: let them land before exit
      for (int q = (s > kStages ? s - kStages : 0); q < s; ++q)
        (void)mbar_wait(&ctl->full_a[q % kStages], (q / kStages) & 1, ctl->wait_ns);
    }
    __syncwarp();  // block-wide barriers must not be reached by part of a warp
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      for (int s = 0; s < nk; ++s) {
        const int slot = s % kStages, par = (s / kStages) & 1;
        if (!wait_or_abort(&ctl->full_a[slot], par, ctl, p.flag)) break;
        if (!wait_or_abort(&ctl->full_b[slot], par, ctl, p.flag)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(a_ring + slot * kAStage), b0 = smem_u32(b_ring + slot * kBStage);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            mma_f16(tmem + h * BN, smem_desc_sw128(a0 + h * (kAStage / 2) + kk * 32), smem_desc_sw128(b0 + kk * 32),
                    p.idesc, (s > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&ctl->empty[slot]);  // stage free once these MMAs have read it
      }
      mma_commit(&ctl->done);  // accumulators complete (or, after an abort, all issued MMAs done)
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- decoders
    const int r = warp * 32 + lane;  // weight row inside the tile (rows >= bn only arrive)
    const bool in_tile = r < bn;
    int64_t n = n0 + r;
    const bool row_ok = in_tile && n < p.N;
    if (!row_ok) n = p.N - 1;
    const uint8_t* crow = p.codes + n * p.ldc;
    const uint16_t* srow = p.scales + n * p.lds;
    const uint32_t row_off = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
    const int rx = r & 7;
    // codes and scales run two stages ahead of the decode, so their latency
    // hides behind two stages of MMA
    auto ld_codes = [&](int st) {
      if (!(in_tile && st < nk)) return make_uint4(0, 0, 0, 0);
      if constexpr (SP) {
        // stage half hf of group g: low nibbles at bytes 8 hf .., high bits at 16 + 4 hf ..
        const int64_t kk = (int64_t)(s0 + st) * BK;
        const uint8_t* gp = crow + 24 * (kk >> 7);
        const int hf = (int)((kk >> 6) & 1);
        const uint2 lo = ld_in_u2(gp + 8 * hf);
        return make_uint4(lo.x, lo.y, ld_in_u32(gp + 16 + 4 * hf), 0u);
      } else {
        return ld_in_u4(crow + (s0 + st) * (BK / 4));
      }
    };
    auto ld_scale = [&](int st) {
      const int lgs = EXT ? p.lgs : 0;
      return (row_ok && st < nk) ? ld_in_u16(srow + (((s0 + st) * BK) >> (7 + lgs))) : (uint16_t)0;
    };
    uint4 cur = ld_codes(0), nx1 = ld_codes(1);
    uint16_t scur = ld_scale(0), snx1 = ld_scale(1);
    for (int s = 0; s < nk; ++s) {
      const int slot = s % kStages, use = s / kStages;
      const uint4 nx2 = ld_codes(s + 2);
      const uint16_t snx2 = ld_scale(s + 2);
      const uint16_t sbits = scur;
      if (use > 0 && !wait_or_abort(&ctl->empty[slot], (use - 1) & 1, ctl, p.flag)) break;
      const uint32_t s2 = (uint32_t)sbits | ((uint32_t)sbits << 16);
      unsigned char* dst = b_ring + slot * kBStage + row_off;
      uint32_t w[4] = {cur.x, cur.y, cur.z, cur.w};
      if constexpr (SP) {
        // quad j of the stage (j = 0..15): low nibble j of (x, y), high bits j of z
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t b = 0;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * q + jj;
            const uint32_t c = (((j < 8 ? cur.x : cur.y) >> (4 * (j & 7))) & 15u) | (((cur.z >> (2 * j)) & 3u) << 4);
            b |= (uint32_t)ctl->sp_tab[c] << (8 * jj);
          }
          w[q] = b;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 16 codes -> two 16-byte chunks (rows past the tile: none)
        if (!in_tile) break;
        const uint32_t wq = w[q], w10 = wq >> 10;
        const uint4 lo = make_uint4(ts_pair<0>(wq, w10, s2), ts_pair<1>(wq, w10, s2), ts_pair<2>(wq, w10, s2),
                                    ts_pair<3>(wq, w10, s2));
        const uint4 hi = make_uint4(ts_pair<4>(wq, w10, s2), ts_pair<5>(wq, w10, s2), ts_pair<6>(wq, w10, s2),
                                    ts_pair<7>(wq, w10, s2));
        *reinterpret_cast<uint4*>(dst + (((2 * q) ^ rx) << 4)) = lo;
        *reinterpret_cast<uint4*>(dst + (((2 * q + 1) ^ rx) << 4)) = hi;
      }
      fence_async_smem();  // generic-proxy writes -> visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->full_b[slot]);
      cur = nx1;
      nx1 = nx2;
      scur = snx1;
      snx1 = snx2;
    }
    // ---------------------------------------------------------------- epilogue
    (void)wait_or_abort(&ctl->done, 0, ctl, p.flag);
    tc_fence_after();
    const int quad = warp & 3, half = warp >> 2;  // TMEM lanes 32*quad.., accumulator half
    const int row = half * 128 + quad * 32 + lane;
    const int64_t m = m0 + row;
    // a K segment writes its whole partial tile; a whole tile writes y
    const bool m_ok = unit >= 0 || m < p.M;
    float* yrow = unit >= 0 ? p.part + ((int64_t)unit * BM + row) * bn : p.y + (m < p.M ? m : 0) * p.ldy + n0;
    const bool vec = unit >= 0 || p.vec_store;
    const int ncols = unit >= 0 ? bn : (int)((p.N - n0) < bn ? (p.N - n0) : bn);
    // TMA path: this warp's 32 rows leave as 32 x 32 blocks staged in its own
    // 16 KB of the (now idle) stage ring; a block is written only where all 32
    // of its columns belong to this tile (TMA clips rows >= M and columns >= N)
    const bool tma = unit >= 0 ? p.tma_part != 0 : p.tma_y != 0;
    const CUtensorMap* omap = unit >= 0 ? &pmap : &ymap;
    const int64_t oy64 = unit >= 0 ? (int64_t)unit * BM + half * 128 + quad * 32 : m0 + half * 128 + quad * 32;
    const bool rows_any = unit >= 0 || oy64 < p.M;  // warp-uniform
    const int ox = unit >= 0 ? 0 : (int)n0, oy = (int)oy64;
    unsigned char* stage = smem + warp * (kOutSlots * kOutBlock);
    int issued = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      __syncwarp();  // tcgen05.ld is warp-collective; the stores below diverge
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * BN + c0), v);
      const bool aborted = __any_sync(0xffffffffu, ctl->abort != 0);
      if (aborted) continue;
      if (tma && c0 + kOutBox <= bn) {
        if (!rows_any) continue;
        unsigned char* buf = stage + (issued % kOutSlots) * kOutBlock;
        if (issued >= kOutSlots) {  // the block staged kOutSlots ago has been read
          if (lane == 0) bulk_wait_read<kOutSlots - 1>();
          __syncwarp();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)  // row = lane, 16-byte chunk i at position i ^ (row % 8)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((i ^ (lane & 7)) << 4)) =
              make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
                         __float_as_uint(v[4 * i + 3]));
        fence_async_smem();  // generic-proxy writes -> visible to the bulk copy
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(omap, ox + c0, oy, smem_u32(buf));
          bulk_commit();
        }
        ++issued;
      } else if (m_ok) {
        if (vec && c0 + 32 <= ncols) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(yrow + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)  // constant indices keep v in registers
            if (c0 + i < ncols) yrow[c0 + i] = v[i];
        }
      }
    }
    // ---- the next layer's rotated activations: FWHT-128 of each 128-column
    // group of this thread's row of y, all in registers (the row of a
    // tensor-memory lane is one thread's), in the staged order of the
    // definition (h = 1 .. 64, lower element a + b, then * c), fp16 RN
    if (EXT && p.xnext != nullptr && unit < 0) {
      const bool row_ok = m < p.M;
#pragma unroll 1
      for (int j = 0; j < bn / 128 && n0 + 128 * j < p.N; ++j) {  // warp-uniform bounds
        float w[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __syncwarp();
          tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * BN + 128 * j + 32 * q), w + 32 * q);
        }
        if (__any_sync(0xffffffffu, ctl->abort != 0)) break;
#pragma unroll
        for (int h = 1; h < 128; h *= 2) {
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            if ((i & h) == 0) {
              const float a = w[i], b = w[i + h];
              w[i] = __fadd_rn(a, b);
              w[i + h] = __fsub_rn(a, b);
            }
          }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          w[i] = __fmul_rn(w[i], kInvSqrt128);
          amax = fmaxf(amax, fabsf(w[i]));
        }
        if (!row_ok) continue;
        // |v| >= 65520 rounds to an fp16 infinity (round to nearest even)
        if (amax >= 65520.0f) atomicOr(p.flag_next, 1u);
        uint16_t* dst = p.xnext + m * p.ldxn + n0 + 128 * j;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-chunk c: slots hold elements 0, 8, 1, 9, ..., 7, 15
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = pack_half2(w[16 * c + i], w[16 * c + 8 + i]);
          reinterpret_cast<uint4*>(dst + 16 * c)[0] = make_uint4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<uint4*>(dst + 16 * c)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
    }
    // staged blocks must be read out before the CTA's shared memory is released
    if (lane == 0 && issued > 0) bulk_wait_read<0>();
    __syncwarp();
  }
  tc_fence_before();
  __syncwarp();  // a warp reaches the block barrier whole (lanes may have diverged)
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
  pdl_launch_dependents();
}

// y of the split tiles: output (tile, row, 4 columns) per thread, the sum of
// its splits partials in segment order.
__global__ void __launch_bounds__(256) k_gemm_fixup(const float* __restrict__ part, int n_main, int n_split_tiles,
                                                   int splits, int n_tiles_m, int bn, int64_t M, int64_t N,
                                                   float* __restrict__ y, int64_t ldy) {
  pdl_wait();
  // 32-bit index arithmetic: the split tiles are at most one wave (a few
  // million outputs of 4 columns)
  const uint32_t c4 = (uint32_t)bn / 4, per_tile = (uint32_t)BM * c4;
  const uint32_t total = (uint32_t)n_split_tiles * per_tile;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const uint32_t lt = i / per_tile, rem = i - lt * per_tile;
    const uint32_t row = rem / c4, c = 4 * (rem - row * c4);
    const uint32_t tile = (uint32_t)n_main + lt, tn = tile / (uint32_t)n_tiles_m;
    const int64_t m = (int64_t)(tile - tn * (uint32_t)n_tiles_m) * BM + row, n = (int64_t)tn * bn + c;
    if (m >= M || n >= N) continue;
    const float* src = part + ((int64_t)lt * splits * BM + row) * bn + c;
    const int64_t seg = (int64_t)BM * bn;
    float4 acc = *reinterpret_cast<const float4*>(src);
    for (int q0 = 1; q0 < splits; q0 += 8) {  // loads of 8 segments in flight, added in segment order
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (q0 + j < splits) v[j] = *reinterpret_cast<const float4*>(src + (q0 + j) * seg);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (q0 + j < splits) {
          acc.x += v[j].x;
          acc.y += v[j].y;
          acc.z += v[j].z;
          acc.w += v[j].w;
        }
      }
    }
    float* dst = y + m * ldy + n;
    dst[0] = acc.x;
    if (n + 1 < N) dst[1] = acc.y;
    if (n + 2 < N) dst[2] = acc.z;
    if (n + 3 < N) dst[3] = acc.w;
  }
  pdl_launch_dependents();
}

// cuTensorMapEncodeTiled from the CUDA driver, looked up once (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    tried = true;
  }
  return fn;
}

}  // namespace

constexpr size_t kGemmSmem = (size_t)kStages * (kAStage + kBStage) + sizeof(SmemCtl) + 1024;

// The launch shape: weight rows per tile (bn, a multiple of 16 in [64, 256])
// and the K split of a short last wave.  Cost model of the busiest SM, in
// 1/352 of one 64-k stage of a 256-row tile: a stage of a bn-row tile costs
// bn + 96 (the 96 stand for what a stage costs whatever bn is -- streaming
// the 256 x 64 x' tile, the hand-overs; fitted to the 27B shapes) and a tile
// adds kFillStages stages' worth of pipeline fill and output drain.  A last
// wave of L <= SMs / 2 tiles can instead run as L x S K segments (S <= SMs /
// L, at most kMaxSplitUnits units and what the workspace holds), costing
// ceil(nk / S) + kFillStages stages plus the fix-up: a launch (2.5 stages'
// worth) and reading the L x S partial tiles (a 256 x 256 partial tile: 1/32
// of a stage's worth).  A narrower tile replaces a wider one only when it is
// more than 1 % cheaper.
struct GemmPlan {
  int bn, n_main, splits;
  int64_t tiles;
};

constexpr int64_t kFillStages = 4;

static GemmPlan gemm_plan(int64_t N, int64_t M, int64_t K, size_t split_bytes, bool whole_groups = false) {
  const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 1;
  const int64_t tm = (M + BM - 1) / BM, nk = K / BK;
  GemmPlan best{BN, 0, 0, 0};
  int64_t best_cost = -1;
  // whole_groups: tiles of whole 128-column groups (bn 256 or 128)
  for (int bn = BN; bn >= 64; bn -= whole_groups ? 128 : 16) {
    const int64_t tiles = tm * ((N + bn - 1) / bn), w = bn + 96, c = (nk + kFillStages) * w;
    const int64_t full = tiles / sms, L = tiles - full * sms;
    int64_t cost = (full + (L > 0 ? 1 : 0)) * c, n_main = tiles, S = 0;
    if (full >= 1 && L > 0 && 2 * L <= sms) {
      int64_t sp_max = sms / L;
      if (sp_max > nk) sp_max = nk;
      if (sp_max > kMaxSplitUnits / L) sp_max = kMaxSplitUnits / L;
      for (int64_t sp = 2; sp <= sp_max; ++sp) {
        if ((size_t)(L * sp * BM * bn) * sizeof(float) > split_bytes) break;
        const int64_t split_cost = full * c + ((nk + sp - 1) / sp + kFillStages) * w + 880 + 11 * L * sp * bn / 256;
        if (split_cost < cost) {
          cost = split_cost;
          n_main = tiles - L;
          S = sp;
        }
      }
    }
    if (best_cost < 0 || cost * 100 < best_cost * 99) {
      best_cost = cost;
      best = GemmPlan{bn, (int)n_main, (int)S, tiles};
    }
  }
  return best;
}

cudaError_t launch_gemm(const uint8_t* codes, int64_t ldc, const uint16_t* scales, int64_t lds, int64_t N, int64_t K,
                        const uint16_t* xrot, int64_t M, float* y, int64_t ldy, uint32_t* flag, void* split_ws,
                        size_t split_bytes, cudaStream_t s, bool test_stall, int group, uint16_t* xnext,
                        uint32_t* flag_next, bool sparse24) {
  if (N == 0 || M == 0) return cudaSuccess;
  if ((int64_t)device_max_smem_optin() < (int64_t)kGemmSmem) return cudaErrorNotSupported;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {BK, BM};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(xrot), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p{};
  p.codes = codes;
  p.ldc = ldc;
  p.scales = scales;
  p.lds = lds;
  p.N = N;
  p.K = K;
  p.M = M;
  p.y = y;
  p.ldy = ldy;
  p.flag = flag;
  p.stall_cta = test_stall ? 0 : -1;
  p.wait_ns = test_stall ? kTestWaitLimitNs : kWaitLimitNs;
  p.lgs = group == 256 ? 1 : 0;
  p.n_tiles_m = (int)((M + BM - 1) / BM);
  // With xnext, split tiles get their x' from the finished y (a pre-pass form
  // of the transform over their columns after the fix-up), which reads y with
  // 16-byte loads: no K split unless y allows them.
  const bool y_vec16 = (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && ldy % 4 == 0;
  const size_t split_ok = (split_ws != nullptr && (xnext == nullptr || y_vec16)) ? split_bytes : 0;
  const GemmPlan g = gemm_plan(N, M, K, split_ok, xnext != nullptr);
  if (xnext != nullptr && (N % 128 != 0 || g.bn % 128 != 0)) return cudaErrorNotSupported;
  p.xnext = xnext;
  p.ldxn = N;
  p.flag_next = flag_next;
  p.bn = g.bn;
  p.idesc = idesc_f16(p.bn);
  p.vec_store = ((reinterpret_cast<uintptr_t>(y) & 15u) == 0 && ldy % 4 == 0) ? 1 : 0;
  p.n_main = g.n_main;
  p.splits = g.splits > 0 ? g.splits : 1;
  p.part = static_cast<float*>(split_ws);
  const int64_t n_split_tiles = g.tiles - g.n_main;
  const int64_t tiles = g.n_main + n_split_tiles * g.splits;  // CTAs
  // output maps: 32 x 32 fp32 boxes, 128-byte swizzle (the staging layout);
  // where one cannot be made the kernel stores from registers instead
  auto out_map = [&](CUtensorMap* m, void* base, int64_t cols, int64_t rows, int64_t pitch) {
    const cuuint64_t od[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t os[1] = {(cuuint64_t)pitch * 4};
    const cuuint32_t ob[2] = {kOutBox, kOutBox};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, od, os, ob, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  CUtensorMap ymap = map, pmap = map;
  p.tma_y = (p.vec_store && M < (int64_t)1 << 31 && N < (int64_t)1 << 31 && out_map(&ymap, y, N, M, ldy)) ? 1 : 0;
  p.tma_part = (n_split_tiles > 0 && out_map(&pmap, split_ws, p.bn, n_split_tiles * g.splits * BM, p.bn)) ? 1 : 0;
  static std::atomic<bool> smem_set[64];  // the kernel's shared-memory limit, raised once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_gemm_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_gemm_tc<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e != cudaSuccess) return e;
    smem_set[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const bool ext = p.lgs != 0 || p.xnext != nullptr;
  if (sparse24 && ext) return cudaErrorNotSupported;
  cudaError_t e = sparse24 ? cudaLaunchKernelEx(&cfg, k_gemm_tc<false, true>, map, ymap, pmap, p)
                  : ext    ? cudaLaunchKernelEx(&cfg, k_gemm_tc<true>, map, ymap, pmap, p)
                           : cudaLaunchKernelEx(&cfg, k_gemm_tc<false>, map, ymap, pmap, p);
  if (e != cudaSuccess || n_split_tiles == 0) return e;
  // y of the split tiles: the partials added in segment order
  const int64_t work = n_split_tiles * BM * (p.bn / 4);
  const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 1;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 4 * sms) blocks = 4 * sms;
  cudaLaunchConfig_t fc = {};
  fc.gridDim = dim3((unsigned)blocks);
  fc.blockDim = dim3(256);
  fc.stream = s;
  fc.attrs = at;
  fc.numAttrs = 1;  // programmatic serialisation: waits for the GEMM in pdl_wait
  e = cudaLaunchKernelEx(&fc, k_gemm_fixup, static_cast<const float*>(split_ws), g.n_main, (int)n_split_tiles,
                         g.splits, p.n_tiles_m, p.bn, M, N, y, ldy);
  if (e != cudaSuccess || xnext == nullptr) return e;
  // x' of the split tiles: FWHT-128 of their finished y, in the GEMM pre-pass
  // form (fp16, 16-chunk order, overflow into *flag_next) -- one launch per
  // run of split tiles that share a column block (tile = tile_m + tile_n * n_tiles_m)
  for (int64_t t = g.n_main; t < g.tiles;) {
    const int64_t tn = t / p.n_tiles_m, tm0 = t % p.n_tiles_m;
    int64_t t1 = t;
    while (t1 < g.tiles && t1 / p.n_tiles_m == tn) ++t1;
    const int64_t tm1 = (t1 - 1) % p.n_tiles_m;
    const int64_t m0 = tm0 * BM, m1 = std::min<int64_t>(M, (tm1 + 1) * BM);
    const int64_t nc0 = tn * p.bn, ncols = std::min<int64_t>(N - nc0, p.bn);
    e = launch_fwht128(y + m0 * ldy + nc0, TQ_F32, ldy, xnext + m0 * N + nc0, TQ_F16, N, m1 - m0, ncols, true,
                       flag_next, s);
    if (e != cudaSuccess) return e;
    t = t1;
  }
  return cudaSuccess;
}

}  // namespace tq
