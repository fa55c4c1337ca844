// tq_device.cuh -- device building blocks shared by the libtq kernels.
//
// FWHT-128 on one warp: lane l holds elements 4l .. 4l+3 of a 128-block.
// Butterfly stage h pairs element i with i ^ h (xxqk.cn/news/652513 sec. 2,
// log2(n) rounds of (a + b, a - b)); stages h = 1, 2 stay inside a lane and
// stages h = 4 .. 64 pair lane l with lane l ^ (h / 4) through shuffles.
// The lower element of a pair keeps a + b, the upper one a - b, so the fp32
// result equals the staged definition bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

constexpr unsigned kFull = 0xffffffffu;
// RN_fp32(1/sqrt(128)) -- the normalisation of the 128-point transform.
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

__device__ __forceinline__ void fwht128_lane(float v[4], int lane) {
  // h = 1: (0,1), (2,3);  h = 2: (0,2), (1,3)
  const float a0 = v[0] + v[1], a1 = v[0] - v[1];
  const float a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
  // h = 4 .. 64.  fma(-1, mine, other) is exactly other - mine.
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float o = __shfl_xor_sync(kFull, v[j], m);
      v[j] = __fmaf_rn(sgn, v[j], o);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = __fmul_rn(v[j], kInvSqrt128);
}

// Two fp32 lanes in one 64-bit register pair, and the paired (f32x2)
// arithmetic on them: each half is rounded as the scalar operation would be.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// FWHT-128 on half a warp: lane l holds elements 8p .. 8p+7 (p = l & 15) of
// the block of its half-warp (l >> 4), so one warp rotates two blocks.
// Stages h = 1, 2, 4 stay inside a lane; stages h = 8 .. 64 pair lane l with
// lane l ^ (h / 8), never crossing the half-warp.  Bit-identical to the
// staged definition, like fwht128_lane.  Elements 2i and 2i + 1 travel as one
// f32x2 pair, so every stage but h = 1 takes one paired instruction per two
// elements.
__device__ __forceinline__ void fwht128_x8(float v[8], int lane) {
  // h = 1: inside each pair
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float a = v[j], b = v[j + 1];
    v[j] = a + b;
    v[j + 1] = a - b;
  }
  uint64_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = f2_pack(v[2 * i], v[2 * i + 1]);
  // h = 2, 4: pair i with pair i ^ (h / 2)
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
  // h = 8 .. 64 across lanes: the upper lane of a butterfly keeps o - v, the
  // lower v + o (one fma with a +-1 multiplier, exact like the add)
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
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
  const uint64_t sc = f2_pack(kInvSqrt128, kInvSqrt128);
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(q[i], sc), v[2 * i], v[2 * i + 1]);
}

// FWHT-128 on an 8-lane group: lane p (= lane & 7) holds elements
// 16p .. 16p+15 of the block; stages h = 1 .. 8 in registers (2 .. 8 on
// f32x2 pairs), h = 16, 32, 64 across lanes, then the normalisation.
__device__ __forceinline__ void fwht128_x16(float v[16], int lane) {
#pragma unroll
  for (int j = 0; j < 16; j += 2) {  // h = 1
    const float a = v[j], b = v[j + 1];
    v[j] = a + b;
    v[j + 1] = a - b;
  }
  uint64_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = f2_pack(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int hp = 1; hp < 8; hp <<= 1) {  // h = 2, 4, 8 on pairs
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & hp) == 0) {
        const uint64_t a = q[i], b = q[i + hp];
        q[i] = f2_add(a, b);
        q[i + hp] = f2_sub(a, b);
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {  // h = 16, 32, 64: lower lane a + b, upper lane a - b
    const float sgn = (lane & m) ? -1.0f : 1.0f;
    const uint64_t sg = f2_pack(sgn, sgn);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float lo, hi;
      f2_unpack(q[i], lo, hi);
      const float olo = __shfl_xor_sync(kFull, lo, m), ohi = __shfl_xor_sync(kFull, hi, m);
      q[i] = f2_fma(sg, q[i], f2_pack(olo, ohi));
    }
  }
  const uint64_t sc = f2_pack(kInvSqrt128, kInvSqrt128);
#pragma unroll
  for (int i = 0; i < 8; ++i) f2_unpack(f2_mul(q[i], sc), v[2 * i], v[2 * i + 1]);
}

// Eight consecutive bf16 (as a 128-bit word) -> fp32.
__device__ __forceinline__ void bf16x8_to_f32(uint4 w, float v[8]) {
  v[0] = __uint_as_float(w.x << 16);
  v[1] = __uint_as_float(w.x & 0xffff0000u);
  v[2] = __uint_as_float(w.y << 16);
  v[3] = __uint_as_float(w.y & 0xffff0000u);
  v[4] = __uint_as_float(w.z << 16);
  v[5] = __uint_as_float(w.z & 0xffff0000u);
  v[6] = __uint_as_float(w.w << 16);
  v[7] = __uint_as_float(w.w & 0xffff0000u);
}

// Four consecutive bf16 (as a 64-bit word) -> fp32.
__device__ __forceinline__ void bf16x4_to_f32(uint2 w, float v[4]) {
  v[0] = __uint_as_float(w.x << 16);
  v[1] = __uint_as_float(w.x & 0xffff0000u);
  v[2] = __uint_as_float(w.y << 16);
  v[3] = __uint_as_float(w.y & 0xffff0000u);
}

// Loads of kernel inputs.  Every kernel here may start before the kernel that
// precedes it on the stream has finished (programmatic dependent launch) and
// waits for it with griddepcontrol.wait before it reads anything that kernel
// may have written.  Ordinary loads after that wait see those writes.  The
// non-coherent path (ld.global.nc) is not used: it assumes the data is
// read-only for the whole lifetime of the kernel, which a kernel that starts
// early cannot promise.  These are plain C++ loads rather than volatile inline
// assembly, so that the compiler may batch and schedule them, yet it cannot
// move them above the wait (an asm statement with a memory clobber).
__device__ __forceinline__ uint8_t ld_in_u8(const void* p) { return *reinterpret_cast<const uint8_t*>(p); }
__device__ __forceinline__ uint16_t ld_in_u16(const void* p) { return *reinterpret_cast<const uint16_t*>(p); }
__device__ __forceinline__ uint32_t ld_in_u32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ float ld_in_f32(const void* p) { return *reinterpret_cast<const float*>(p); }
__device__ __forceinline__ uint2 ld_in_u2(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 ld_in_u4(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// Staged transform of n values in shared memory by one warp: butterfly
// stages h = 1, 2, .., n / 2 (the lower index of a pair keeps a + b), then one
// multiply by c -- the order of the definition, so the result is bit-exact
// with it.
__device__ __forceinline__ void fwht_warp(float* v, int n, float c, int lane) {
  for (int h = 1; h < n; h <<= 1) {
    for (int q = lane; q < n / 2; q += 32) {
      const int i = (q / h) * 2 * h + (q % h);  // lower index of pair q
      const float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    }
    __syncwarp();
  }
  for (int i = lane; i < n; i += 32) v[i] = __fmul_rn(v[i], c);
  __syncwarp();
}

// t = clamp(rint(w / sc), -1, 1) with IEEE division and round half to even;
// 0 when the scale is 0.
__device__ __forceinline__ int ternarise(float w, float sc) {
  if (sc == 0.0f) return 0;
  const float q = rintf(__fdiv_rn(w, sc));  // round half to even
  return q > 1.0f ? 1 : (q < -1.0f ? -1 : (int)q);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace tq

// ---------------------------------------------------------------------------
// Asynchronous bulk copies into shared memory, completed on mbarriers.
//
// Every wait is bounded by a wall-clock limit (kWaitLimitNs): a wait that
// runs out returns false and the caller records a fault and winds down
// instead of spinning forever.
namespace tq {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete yet sleeps in
// the barrier until the phase completes or about `ns` nanoseconds pass, so
// waiting warps take no issue slots from the warps they wait for.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

constexpr uint32_t kSleepNs = 10000;  // longest sleep between checks of the limits

// Waits for the phase with the given parity to complete; false once
// limit_ns have passed without it.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kSleepNs)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// As mbar_wait, but also gives up as soon as *abort becomes non-zero, and
// sets *abort itself when its own limit runs out, so that one stalled wait
// releases every other waiter of the CTA within microseconds.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                    unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kSleepNs)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// A completed phase observed again with cluster-scope acquire: data that other
// CTAs of the cluster wrote with st.async (signalling this barrier) is then
// ordered before this thread's later reads.  Only for a phase already seen
// complete (it returns at once).
__device__ __forceinline__ void mbar_acquire_cluster(uint64_t* bar, uint32_t parity) {
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%0], %1;\n}\n" ::"r"(
          smem_u32(bar)),
      "r"(parity)
      : "memory");
}

// Bounded-wait limit of a launch that tests the failure path (a stalled copy
// is then noticed within milliseconds instead of seconds).
constexpr unsigned long long kTestWaitLimitNs = 20000000ull;  // 20 ms

// One contiguous global -> shared copy; dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier over `threads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace tq
