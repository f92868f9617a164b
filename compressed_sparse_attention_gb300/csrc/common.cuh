// Shared device helpers of the CSA2 kernels: inline PTX for tcgen05 / TMEM,
// mbarriers and cp.async, shared-memory matrix descriptors, bf16 / e4m3
// packing, RoPE angles and the device error word. sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kHeads = 64;    // attention heads sharing one KV row
constexpr int kDim = 512;     // head dim = stored KV row width
constexpr int kIdxDim = 128;  // indexer dim
constexpr int kMaxPairs = 32; // rope_dim / 2 upper bound

// RoPE frequencies f_i of the rotated pairs (double precision angles).
struct RopeParams {
  int32_t pairs;  // rope_dim / 2; 0 disables rotation
  double freq[kMaxPairs];
};

__device__ __forceinline__ void set_flag(uint32_t* flags, uint32_t bit) {
  if (flags) atomicOr(flags, bit);
}

// cos / sin of pos * f_i. The angle is formed in double precision and reduced
// to [-pi, pi] by Cody-Waite reduction with a two-term 2*pi (high part + the
// rounding remainder), both products fused; the reduced angle then goes to
// single-precision sincosf. The reduction error is ~1e-16 * |angle / 2pi|
// radians, so the result is the correctly rotated float to about 1e-7 even at
// positions near 2^20, at a few double operations instead of a double sincos.
__device__ __forceinline__ void rope_cs(const RopeParams& rp, int i, int64_t pos, float& c, float& s) {
  constexpr double kTwoPiHi = 6.283185307179586232;     // nearest double to 2*pi
  constexpr double kTwoPiLo = 2.4492935982947064e-16;   // 2*pi - kTwoPiHi
  constexpr double kInvTwoPi = 0.15915494309189533577;
  const double a = (double)pos * rp.freq[i];
  const double k = rint(a * kInvTwoPi);
  double r = fma(-k, kTwoPiHi, a);
  r = fma(-k, kTwoPiLo, r);
  sincosf((float)r, &s, &c);
}

// ---------------------------------------------------------------- bf16 packing

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// f16x2 bits of two floats (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t h2_bits(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// two e4m3 codes (low byte first) -> f16x2 (low half first), exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)(two & 0xFFFFu)));
  return r;
}
// two e4m3 codes (low byte first) -> two floats, exact
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  __half2_raw h;
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  h.x = (unsigned short)(r & 0xFFFFu);
  h.y = (unsigned short)(r >> 16);
  return __half22float2(__half2(h));
}

// value of a ue8m0 scale byte: 2^(E-127)
__device__ __forceinline__ float ue8m0_value(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// ue8m0 byte of a block: least k with amax <= 448 * 2^k, E = k + 127 in [0, 254]
__device__ __forceinline__ uint32_t fp8_scale_byte(float amax) {
  if (!(amax > 0.0f)) return 0u;
  int ex;
  float fr = frexpf(amax, &ex);  // amax = fr * 2^ex, fr in [0.5, 1)
  int k = (fr <= 0.875f) ? ex - 9 : ex - 8;  // 448 = 0.875 * 2^9
  int e = k + 127;
  return (uint32_t)(e < 0 ? 0 : (e > 254 ? 254 : e));
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// ---------------------------------------------------------------- fp4 (E2M1)
// E2M1 code of x for a block scale s: the nearest of s * {0, 0.5, 1, 1.5, 2,
// 3, 4, 6}, ties to the even code (mantissa bit 0), saturating at 6 s; the
// sign bit follows x (also for -0). Each midpoint m * s has at most 7
// significant bits (m <= 3 bits, s an e4m3 value or a power of two), so the
// comparisons are exact and no division rounds.
__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
  const float ax = fabsf(x);
  uint32_t c = 0u;
  c += (ax > 0.25f * s) ? 1u : 0u;   // tie -> 0
  c += (ax >= 0.75f * s) ? 1u : 0u;  // tie -> 1.0
  c += (ax > 1.25f * s) ? 1u : 0u;   // tie -> 1.0
  c += (ax >= 1.75f * s) ? 1u : 0u;  // tie -> 2.0
  c += (ax > 2.5f * s) ? 1u : 0u;    // tie -> 2.0
  c += (ax >= 3.5f * s) ? 1u : 0u;   // tie -> 4.0
  c += (ax > 5.0f * s) ? 1u : 0u;    // tie -> 4.0
  return c | ((__float_as_uint(x) >> 28) & 8u);
}
// two E2M1 codes (low nibble first) -> two floats, each 2^-14 times its value:
// the code's exponent and mantissa bits dropped into fp16's low exponent and
// top mantissa bits give exactly that (subnormal codes included)
__device__ __forceinline__ float2 e2m1x2_to_float2_scaled(uint32_t two) {
  const uint32_t lo = two & 0xFu, hi = (two >> 4) & 0xFu;
  const uint32_t h = ((lo & 7u) << 9) | ((lo & 8u) << 12) | (((hi & 7u) << 9) << 16) | (((hi & 8u) << 12) << 16);
  __half2_raw r;
  r.x = (unsigned short)(h & 0xFFFFu);
  r.y = (unsigned short)(h >> 16);
  return __half22float2(__half2(r));
}
constexpr float kE2M1Unscale = 16384.0f;  // 2^14
// eight E2M1 codes (the nibbles n0 .. n7 of w, n0 lowest) -> four f16x2
// words holding their exact values, o[i] = (n(2i), n(2i+1)), low half first:
// one hardware conversion per byte (two codes)
__device__ __forceinline__ void e2m1x8_to_f16x2x4_cvt(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n.reg .b8 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
// e4m3 byte of the fp4 block scale: e4m3(max(amax, 6 * 2^-9) / 6), the
// quotient formed in double (exact enough that its rounding to e4m3 equals
// that of the real quotient) and rounded by CUDA's own conversion
__device__ __forceinline__ uint8_t fp4_scale_e4m3(float amax) {
  const double r = (double)fmaxf(amax, 6.0f * 0x1p-9f) / 6.0;
  return (uint8_t)__nv_cvt_double_to_fp8(r, __NV_SATFINITE, __NV_E4M3);
}
// value of an e4m3 byte
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  return e4m3x2_to_float2((uint16_t)(b & 0xFFu)).x;
}
// ue8m0 byte of the MXFP4 block scale 2^round(log2(max(amax, 6 * 2^-126) / 6)):
// with r = f * 2^k (f in [0.5, 1)), round(log2 r) = k - 1 if f < 2^-1/2, else k
__device__ __forceinline__ uint32_t mxfp4_scale_byte(float amax) {
  const double r = (double)fmaxf(amax, 6.0f * 0x1p-126f) / 6.0;
  int k;
  const double f = frexp(r, &k);
  const int e = (f < 0.70710678118654752440) ? k - 1 : k;
  const int b = e + 127;
  return (uint32_t)(b < 0 ? 0 : (b > 254 ? 254 : b));
}

// order-preserving 32-bit key of a score; -0.0 maps with +0.0
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------- smem / proxies

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte cp.async into shared memory; src_bytes 0 zero-fills
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most n (0..3) of this thread's committed groups are pending
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
  }
}

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ldg_stream4(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Test for the completion of the phase with parity `phase`. The thread is
// suspended until the phase completes or the hint (1 ms) elapses, instead of
// polling: waiting threads then take neither issue slots nor shared-memory
// bandwidth from the warps and the tensor cores still working.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(phase), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait on an mbarrier phase: gives up after ~limit_ns of wall time,
// records CSA2_FLAG_WAIT_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase, uint32_t* flags,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, phase)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      set_flag(flags, CSA2_FLAG_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- tcgen05 / TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive (once) on an mbarrier when all prior tcgen05.mma of this thread complete
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, K-major (0) or
// MN-major (1) operands, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int a_mn_major, int b_mn_major) {
  return (1u << 4)                         // D format: f32
         | (1u << 7)                       // A format: bf16
         | (1u << 10)                      // B format: bf16
         | ((uint32_t)a_mn_major << 15)    // A major
         | ((uint32_t)b_mn_major << 16)    // B major
         | ((uint32_t)(n >> 3) << 17)      // N >> 3
         | ((uint32_t)(m >> 4) << 24);     // M >> 4
}

// Shared-memory matrix descriptor, 128-byte swizzle. The tile base must be
// 1024-byte aligned; start may be offset inside a 128-byte row (K steps).
//   K-major: rows of 128 B, 8-row core groups `sbo` apart.
//   MN-major: 64-element (128 B) MN blocks `lbo` apart, 8-row K groups `sbo` apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// The descriptor of the operand `off` bytes past the one `d` describes (same
// strides and swizzle). The start-address field holds (address >> 4) in the
// low 14 bits; shared-memory addresses stay below 2^18, so the add never
// carries out of the field.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); }

// 32 lanes x 32 bit, 32 consecutive columns -> 32 registers per thread
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- warp-level mma.sync (indexer)

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while
// the previous kernel of its stream still runs: it must wait here before it
// reads anything that kernel writes. Without such a launch this returns at
// once. The trigger lets this kernel's dependents start before it ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- small utils

__device__ __forceinline__ int find_segment(const int64_t* off, int n, int64_t x) {
  // largest b in [0, n) with off[b] <= x (off non-decreasing, off[0] = 0)
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace csa2
