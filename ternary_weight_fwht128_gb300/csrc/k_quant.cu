// k_quant.cu -- offline quantise + pack (tq_quantize_pack).
//
// Per (row n, group g) of 128 weights, one lane pair; lane h (0, 1) of the
// pair holds elements 64h .. 64h + 63 of the group in registers:
//   1. 16-byte loads (8 for bf16, 16 for fp32);
//   2. the staged FWHT-128 in fp32: stages h = 1 .. 32 inside the lane, stage
//      64 across the pair (one shuffle per element), then * c -- from stage 2
//      on in f32x2 pairs;
//   3. sum |w'| in the halving-tree order h = 64, 32, ..., 1.  Level 64
//      adds each element to the partner lane's (one shuffle per element);
//      both lanes form every sum, which gives both the same bits since an
//      IEEE sum does not depend on the order of its two operands; levels
//      32 .. 1 run inside the lane.  The tree is the oracle's bit for bit;
//   4. mean = sum * 2^-7, scale = fp16_RN(mean) (absmean, mhpq.cn/news/1159370
//      sec. 1.1; one fp16 scale per 128 weights, sec. 1.3);
//   5. t = sign(w') * [|w'| > s/2] for a finite s > 0, t = 0 when s == 0.
//      This equals clamp(rint(w'/s), -1, 1) with IEEE division and ties to
//      even: the quotient rounds above 0.5 exactly when |w'| > (s/2)(1 + 2^-24),
//      and no fp32 value lies strictly between s/2 and that bound.  For
//      s = +inf both forms give 0.
//   6. packs: the lane's 64 codes c = t + 1 form four 32-bit words that are
//      its 16 bytes of the 2-bit layout (one store).  The same words are the
//      base-3 digits: a warp takes three units of five groups (640 trits =
//      128 bytes each, so units never share a byte; lanes 30, 31 idle), puts
//      its code words in shared memory, and each lane forms 12 of the warp's
//      384 base-3 bytes (three 32-bit words) from 10-bit windows of them.
//
// The pass reads 2 or 4 bytes per weight and should be bound by HBM: each warp
// copies the next unit triple's weights into shared memory (cp.async, no
// registers held) while it works on the current one.
#include <atomic>

#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

template <int WT>
struct Raw {
  uint4 w[WT == TQ_F32 ? 16 : 8];  // this lane's 64 weights
};

// Staging of the weights: per warp and buffer, 32 lanes x (the lane's 64
// weights + 16 bytes, so that lanes 16-byte reads spread over all banks).
template <int WT>
constexpr int kLaneStage = (WT == TQ_F32 ? 256 : 128) + 16;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int WT, bool DO2, bool DO3>
__global__ void __launch_bounds__(kThreads, 3) k_quantize_pack(const void* __restrict__ W, int64_t N, int64_t K,
                                                            int64_t ldw, uint8_t* __restrict__ codes2, int64_t ld2,
                                                            uint8_t* __restrict__ codes3, int64_t ld3,
                                                            uint16_t* __restrict__ scales, int64_t lds, int vec2,
                                                            int vec3) {
  constexpr int esize = WT == TQ_F32 ? 4 : 2;
  __shared__ __align__(16) uint32_t cw[kWarps][32 * 4 + 4];  // code words of the warp's lanes (+ one spare word)
  // base-3 byte of every 10-bit window of five 2-bit codes c0 + 3 c1 + ... + 81 c4
  // (windows holding a code 3 never occur)
  __shared__ uint8_t b3[1024];
  // weights of two triples (dynamic: 72 KB for fp32 weights)
  extern __shared__ __align__(16) unsigned char qstage[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto stage_at = [&](int buf) { return qstage + ((size_t)buf * kWarps + warp) * (32 * kLaneStage<WT>); };
  const int h = lane & 1;            // half of the group
  const int ul = lane / 10;          // unit of the triple (3: idle lanes 30, 31)
  const int kq = (lane % 10) >> 1;   // group inside the unit
  const int64_t G = K / 128;
  const int64_t nu = (G + 4) / 5;    // units per row
  const int64_t nunits = N * nu;
  const int64_t niters = (nunits + 2) / 3;
  const int64_t nbytes3 = (K + 4) / 5;
  const int64_t ld3min = (nbytes3 + 15) / 16 * 16;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  uint32_t* const wbuf = cw[warp];

  if constexpr (DO3) {
    for (int i = threadIdx.x; i < 1024; i += kThreads)
      b3[i] = (uint8_t)((i & 3) + 3 * ((i >> 2) & 3) + 9 * ((i >> 4) & 3) + 27 * ((i >> 6) & 3) + 81 * ((i >> 8) & 3));
    __syncwarp();
    __syncthreads();
  }
  pdl_wait();

  // rows and units-in-row of the three units of triple `it`: one 32-bit
  // division (the host keeps the unit count below 2^31), done once per
  // triple -- the loop hands the triple it loads on to its processing
  struct Tri {
    uint32_t n[3], u[3];
  };
  auto triple = [&](int64_t it) {
    Tri t;
    const uint32_t U0 = (uint32_t)(3 * it), row = U0 / (uint32_t)nu;
    t.n[0] = row;
    t.u[0] = U0 - row * (uint32_t)nu;
#pragma unroll
    for (int q = 1; q < 3; ++q) {
      t.n[q] = t.n[q - 1];
      t.u[q] = t.u[q - 1] + 1;
      if (t.u[q] == nu) {
        t.u[q] = 0;
        ++t.n[q];
      }
    }
    return t;
  };
  // group of this lane in triple `it`: row n, group g (valid: inside the matrix)
  auto locate = [&](int64_t it, const Tri& t, int64_t& n, int64_t& g) -> bool {
    const int q = ul < 3 ? ul : 0;
    const uint32_t n32 = q == 0 ? t.n[0] : (q == 1 ? t.n[1] : t.n[2]);
    const uint32_t g32 = 5u * (q == 0 ? t.u[0] : (q == 1 ? t.u[1] : t.u[2])) + (uint32_t)kq;
    n = n32;
    g = g32;
    return ul < 3 && (uint32_t)(3 * it) + (uint32_t)ul < (uint32_t)nunits && g32 < (uint32_t)G;
  };
  // starts the copy of triple `it`'s weights into staging buffer `buf`
  auto load = [&](int buf, int64_t it, const Tri& tri) {
    int64_t n, g;
    if (it < niters && locate(it, tri, n, g)) {
      const unsigned char* src = static_cast<const unsigned char*>(W) + (n * ldw + g * 128 + 64 * h) * esize;
      const uint32_t dst = smem_u32(stage_at(buf) + lane * kLaneStage<WT>);
#pragma unroll
      for (int i = 0; i < (WT == TQ_F32 ? 16 : 8); ++i) cp_async16(dst + 16 * i, src + 16 * i);
    }
    cp_async_commit();
  };
  auto fetch = [&](Raw<WT>& r, int buf, bool ok) {
    const uint4* src = reinterpret_cast<const uint4*>(stage_at(buf) + lane * kLaneStage<WT>);
#pragma unroll
    for (int i = 0; i < (WT == TQ_F32 ? 16 : 8); ++i) r.w[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
  };

  auto process = [&](int buf, int64_t it, const Tri& tri) {
    int64_t n, g;
    const bool ok = locate(it, tri, n, g);
    Raw<WT> r;
    fetch(r, buf, ok);
    float v[64];
#pragma unroll
    for (int i = 0; i < (WT == TQ_F32 ? 16 : 8); ++i) {
      if constexpr (WT == TQ_F32) {
        v[4 * i + 0] = __uint_as_float(r.w[i].x);
        v[4 * i + 1] = __uint_as_float(r.w[i].y);
        v[4 * i + 2] = __uint_as_float(r.w[i].z);
        v[4 * i + 3] = __uint_as_float(r.w[i].w);
      } else {
        bf16x8_to_f32(r.w[i], &v[8 * i]);
      }
    }
    // ---- FWHT-128: stages 1 .. 32 in the lane, 64 across the pair, then * c.
    // Elements 2i and 2i + 1 travel as one f32x2 pair from stage 2 on (each
    // half rounds as the scalar operation, so the stages are unchanged).
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
      const float a = v[j], b = v[j + 1];
      v[j] = __fadd_rn(a, b);
      v[j + 1] = __fsub_rn(a, b);
    }
    {
      uint64_t q[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) q[i] = f2_pack(v[2 * i], v[2 * i + 1]);
#pragma unroll
      for (int hp = 1; hp < 32; hp <<= 1) {  // element stride 2 hp = 2 .. 32
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i & hp) continue;
          const uint64_t a = q[i], b = q[i + hp];
          q[i] = f2_add(a, b);
          q[i + hp] = f2_sub(a, b);
        }
      }
      // lower half: own + other; upper half: other - own
      const float sgn = h ? -1.0f : 1.0f;
      const uint64_t sg = f2_pack(sgn, sgn), c2 = f2_pack(kInvSqrt128, kInvSqrt128);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float lo, hi;
        f2_unpack(q[i], lo, hi);
        const float olo = __shfl_xor_sync(kFull, lo, 1), ohi = __shfl_xor_sync(kFull, hi, 1);
        f2_unpack(f2_mul(f2_fma(sg, q[i], f2_pack(olo, ohi)), c2), v[2 * i], v[2 * i + 1]);
      }
    }
    // ---- sum |w'|: halving tree h = 64 .. 1.  Both lanes of the pair form
    // every sum (an IEEE sum does not depend on the order of its two
    // operands, so the lanes hold the same bits): h = 64 pairs each element
    // with the partner lane's, h = 32 .. 1 run inside the lane, from h = 32
    // on in f32x2 pairs (sums 2i, 2i + 1).
    uint64_t t16[16];  // the 32 sums of level h = 32
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a[2], b[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 2 * i + e;
        a[e] = __fadd_rn(fabsf(v[j]), fabsf(__shfl_xor_sync(kFull, v[j], 1)));            // level 64, sum j
        b[e] = __fadd_rn(fabsf(v[32 + j]), fabsf(__shfl_xor_sync(kFull, v[32 + j], 1)));  // level 64, sum 32 + j
      }
      t16[i] = f2_add(f2_pack(a[0], a[1]), f2_pack(b[0], b[1]));
    }
#pragma unroll
    for (int hp = 8; hp >= 1; hp >>= 1) {  // levels 16, 8, 4, 2
#pragma unroll
      for (int i = 0; i < hp; ++i) t16[i] = f2_add(t16[i], t16[i + hp]);
    }
    float s0, s1;
    f2_unpack(t16[0], s0, s1);
    const float sum = __fadd_rn(s0, s1);  // level 1
    const float mean = __fmul_rn(sum, 0.0078125f);
    const __half sh = __float2half_rn(mean);
    const float sc = __half2float(sh);
    const float half_s = sc * 0.5f;  // exact
    // ---- ternarise: code c = t + 1 at bits 2 (j % 16) of word j / 16.
    // c = [w > thr] + [not (w < -thr)] with thr = s/2 for a finite s > 0 and
    // +inf otherwise: 2 above s/2, 0 below -s/2, 1 in between, at +-s/2
    // exactly, for NaN and for every weight of a zero, infinite or NaN scale
    // -- the compare rule above.
    const float thr = (sc != 0.0f) ? half_s : __int_as_float(0x7f800000);
    uint32_t cwd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      // c 4^j as two conditional adds of 4^j (the fields never carry: c <= 2)
      const uint32_t bit = 1u << (2 * (j & 15));
      cwd[j >> 4] += (v[j] > thr ? bit : 0u) + (!(v[j] < -thr) ? bit : 0u);
    }
    if (ok) {
      if constexpr (DO2) {
        uint8_t* dst = codes2 + n * ld2 + g * 32 + 16 * h;
        if (vec2) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(cwd[0], cwd[1], cwd[2], cwd[3]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) dst[i] = (uint8_t)(cwd[i >> 2] >> (8 * (i & 3)));
        }
      }
      if (h == 0) scales[n * lds + g] = __half_as_ushort(sh);
    }
    if constexpr (DO3) {
      // ---- base-3: trit T of unit q of the triple is bits 2T .. 2T + 1 of
      // the unit's 1280-bit run in wbuf (lanes 10q .. 10q + 9, 128 bits each);
      // groups past the matrix read as code 1 (t = 0).
      __syncwarp();  // the previous triple's reads of wbuf are done
      if (ok) {
        reinterpret_cast<uint4*>(wbuf)[lane] = make_uint4(cwd[0], cwd[1], cwd[2], cwd[3]);
      } else {
        reinterpret_cast<uint4*>(wbuf)[lane] = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
      }
      __syncwarp();
      // Each lane forms three 32-bit words of the triple's 384 bytes (bytes
      // 12 lane .. 12 lane + 11): a word never straddles two units (128 bytes
      // each), and its four bytes take their 10-bit windows from three
      // consecutive code words.
      const uint32_t U0 = (uint32_t)(3 * it);
#pragma unroll
      for (int m4 = 0; m4 < 3; ++m4) {
        const int B = 12 * lane + 4 * m4;  // first byte of the word, of the triple's 384
        const int q = B >> 7, b = B & 127;
        if (U0 + (uint32_t)q >= (uint32_t)nunits) continue;
        const uint32_t un = q == 0 ? tri.n[0] : (q == 1 ? tri.n[1] : tri.n[2]);
        const uint32_t uu = q == 0 ? tri.u[0] : (q == 1 ? tri.u[1] : tri.u[2]);
        const uint32_t pos = uu * 128u + (uint32_t)b;  // byte of the row (a multiple of 4)
        if (pos >= (uint32_t)ld3min) continue;          // past the row's zero padding (ld3min % 16 == 0)
        const int bit0 = 1280 * q + 10 * b;
        const uint32_t w0 = wbuf[bit0 >> 5], w1 = wbuf[(bit0 >> 5) + 1], w2 = wbuf[(bit0 >> 5) + 2];
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (pos + k < (uint32_t)nbytes3) {
            const int sh = (bit0 & 31) + 10 * k;  // 0 .. 61
            const uint32_t win = sh < 32 ? __funnelshift_r(w0, w1, sh) : __funnelshift_r(w1, w2, sh - 32);
            word |= (uint32_t)b3[win & 0x3ffu] << (8 * k);
          }
        }
        uint8_t* dst = codes3 + (int64_t)un * ld3 + pos;
        if (vec3) {
          *reinterpret_cast<uint32_t*>(dst) = word;
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = (uint8_t)(word >> (8 * k));
        }
      }
    }
  };

  int64_t it = (int64_t)blockIdx.x * kWarps + warp;
  int buf = 0;
  Tri cur = triple(it);
  load(buf, it, cur);
  for (; it < niters; it += stride) {
    const Tri next = triple(it + stride);
    load(buf ^ 1, it + stride, next);  // the next triple streams in meanwhile
    cp_async_wait<1>();                // this lane's copies of triple `it` have landed
    process(buf, it, cur);
    __syncwarp();                      // every lane has read `buf` before it is refilled
    buf ^= 1;
    cur = next;
  }
  cp_async_wait<0>();
  pdl_launch_dependents();
}

template <int WT, bool DO2, bool DO3>
cudaError_t launch_t(const void* W, int64_t N, int64_t K, int64_t ldw, uint8_t* c2, int64_t ld2, uint8_t* c3,
                     int64_t ld3, uint16_t* sc, int64_t lds, cudaStream_t s) {
  const int64_t G = K / 128;
  const int64_t niters = (N * ((G + 4) / 5) + 2) / 3;  // unit triples, one per warp iteration
  // the kernel's unit index is 32-bit (about 2.8 TB of bf16 weights; never reached in memory)
  if (3 * niters >= (int64_t(1) << 31) - (int64_t(1) << 24)) return cudaErrorInvalidValue;
  // exactly the resident CTAs: triples are dealt out statically, so a CTA
  // waiting for a second wave would leave the tail to few SMs
  const size_t smem = (size_t)2 * kWarps * 32 * kLaneStage<WT>;
  static std::atomic<bool> smem_set[64];  // the kernel's dynamic shared-memory limit, raised once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_pack<WT, DO2, DO3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    smem_set[dev].store(true, std::memory_order_release);
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quantize_pack<WT, DO2, DO3>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  const int64_t want = (niters + kWarps - 1) / kWarps;
  const int64_t grid = want < cap ? want : cap;
  const int vec2 = (c2 != nullptr && (reinterpret_cast<uintptr_t>(c2) & 15u) == 0 && ld2 % 16 == 0) ? 1 : 0;
  const int vec3 = (c3 != nullptr && (reinterpret_cast<uintptr_t>(c3) & 3u) == 0 && ld3 % 4 == 0) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_quantize_pack<WT, DO2, DO3>, W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, vec2,
                            vec3);
}

template <int WT>
cudaError_t launch_w(const void* W, int64_t N, int64_t K, int64_t ldw, int fmt, uint8_t* c2, int64_t ld2,
                     uint8_t* c3, int64_t ld3, uint16_t* sc, int64_t lds, cudaStream_t s) {
  if (fmt == TQ_PACK_2BIT) return launch_t<WT, true, false>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, s);
  if (fmt == TQ_PACK_BASE3) return launch_t<WT, false, true>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, s);
  return launch_t<WT, true, true>(W, N, K, ldw, c2, ld2, c3, ld3, sc, lds, s);
}

}  // namespace

cudaError_t launch_quantize_pack(const void* W, int wt, int64_t N, int64_t K, int64_t ldw, int fmt, uint8_t* codes2,
                                 int64_t ld2, uint8_t* codes3, int64_t ld3, uint16_t* scales, int64_t lds,
                                 cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (wt == TQ_F32) return launch_w<TQ_F32>(W, N, K, ldw, fmt, codes2, ld2, codes3, ld3, scales, lds, s);
  return launch_w<TQ_BF16>(W, N, K, ldw, fmt, codes2, ld2, codes3, ld3, scales, lds, s);
}

// No wait in this kernel can stall (no producer/consumer barriers).
unsigned int take_fault_quant() { return 0; }

}  // namespace tq
