// Shared device helpers and cache geometry for the rotated INT2 KV cache kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "oscar_kv.h"

namespace oscar {

constexpr int kGroup = OSCAR_KV_GROUP;
constexpr int kNcapRound = 64;

// Geometry of one layer of the cache (host computed, passed by value).
struct Geom {
  int B, Hq, Hkv, D, G, Dg, S, W, cap;
  int64_t ncap;
  uint64_t sink_bytes, ring_bytes, codes_bytes, sz_bytes, role_bytes, layer_bytes;
  int vb;                 // V kept BF16 at every position (K-only INT2)
  int lm;                 // INT2 codes index the Lloyd-Max levels (fills the padding before v_role_bytes)
  uint64_t v_role_bytes;  // V role: role_bytes, or with vb [B][Hkv][cap][D] bf16
};

__host__ __device__ inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// Division of 32-bit unsigned integers by a divisor d (1 <= d <= 2^31) fixed
// for a launch, as a multiply-high, an add and a shift: with l = ceil(log2 d)
// and m = floor(2^32 (2^l - d) / d) + 1, floor(x / d) = (mulhi(x, m) + x) >> l
// for every 32-bit x (Granlund and Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994, section 4).
struct FastDiv {
  uint32_t mul, shift;
};
inline FastDiv fastdiv_make(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  FastDiv f;
  f.shift = l;
  f.mul = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  return f;
}
__device__ __forceinline__ uint32_t fastdiv(uint32_t x, const FastDiv& f) {
  return uint32_t((uint64_t(__umulhi(x, f.mul)) + x) >> f.shift);
}

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void status_or(int32_t* st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Precision of two-bit codes as fp16 subnormal operands: a half whose only
// bits are a code at mantissa bit 2k has the exact value code * 4^k * 2^-24,
// and the tensor cores multiply subnormal inputs exactly, but they align the
// products of one MMA by the operands' exponent fields, and a subnormal's
// field says 2^-14 whatever its leading bit: a code at bit 2k keeps about
// 15 + 2k significant bits of the accumulation window instead of ~25
// (measured on GB300: ~2e-5 relative error on sums of k = 0 codes, ~2e-6 from
// k = 1 up).  So codes are unpacked to mantissa bits 4..9 only (k = 2, 3, 4),
// for K (QK^T, where one MMA mixes the k of two registers) and V (P.V, where
// each output row takes one register index) alike: register p holds the codes
// at bits 2p and 16 + 2p (the word's low and high half) moved to mantissa bit
// 2 kq(p):
//   p = 0, 1: the word shifted left by 4 (k = 2, 3);
//   p = 2, 3, 4: the word itself (k = 2, 3, 4);
//   p = 5, 6, 7: the word shifted right by 6 (k = 2, 3, 4).
// The masks keep bits 4..9 of each half, so bits a shift carries across the
// halves are never kept.  Two shifts and eight ANDs per 16 codes; the factor
// 4^kq(p) * 2^-24 is constant per register index, so the caller folds it into
// the other operand.
__device__ __forceinline__ constexpr int unpack_kq(int p) { return p < 2 ? p + 2 : (p < 5 ? p : p - 3); }

__device__ __forceinline__ void unpack16(uint32_t w, uint32_t (&r)[8]) {
  const uint32_t wl = w << 4, wr = w >> 6;
  r[0] = wl & 0x00300030u;
  r[1] = wl & 0x00C000C0u;
  r[2] = w & 0x00300030u;
  r[3] = w & 0x00C000C0u;
  r[4] = w & 0x03000300u;
  r[5] = wr & 0x00300030u;
  r[6] = wr & 0x00C000C0u;
  r[7] = wr & 0x03000300u;
}

// log2 of the value unpack16 gives a code of register p, per unit of code
__device__ __forceinline__ constexpr int unpack_exp(int p) { return 2 * unpack_kq(p) - 24; }

// Lloyd-Max levels: level(c) = (0, rho, rho + 1, 2 rho + 1)[c] with rho = 1.16
// (LM_RATIO as printed, rounded to float32).  Writing c = c0 + 2 c1,
// level(c) = rho * c + (1 - rho) * c1 = rho * c + kLmHi * (2 c1): the decode
// multiplies the code sum by rho and adds kLmHi times the same sum over the
// codes' high bits (unpack16_hi).  The codec's span and level midpoints are
// float32, each the single rounding of an exact value (so any evaluation of
// these constant expressions at float or higher precision gives the same bits):
//   span = 2 rho + 1 (exact), m0 = rho / 2 (exact), m1 = rho + 1/2 (exact),
//   m2 = span - m0 = the float32 nearest to 3 rho / 2 + 1;
// kLmHi = (1 - rho) / 2 is exact as well (Sterbenz).
constexpr float kLmRho = 1.16f;
constexpr float kLmSpan = 2.0f * kLmRho + 1.0f;      // the group's range in level units
constexpr float kLmHi = (1.0f - kLmRho) * 0.5f;
constexpr float kLmMid0 = kLmRho * 0.5f;
constexpr float kLmMid1 = kLmRho + 0.5f;
constexpr float kLmMid2 = kLmSpan - kLmMid0;

// nearest Lloyd-Max level of y = (x - zero) / unit; on a midpoint the lower one
__device__ __forceinline__ int lm_code(float y) { return (y > kLmMid0) + (y > kLmMid1) + (y > kLmMid2); }

// As unpack16, keeping only the high bit of each code: register p holds
// 2 * c1 * 4^kq(p) * 2^-24 where unpack16 holds c * 4^kq(p) * 2^-24.
__device__ __forceinline__ void unpack16_hi(uint32_t w, uint32_t (&r)[8]) {
  const uint32_t wl = w << 4, wr = w >> 6;
  r[0] = wl & 0x00200020u;
  r[1] = wl & 0x00800080u;
  r[2] = w & 0x00200020u;
  r[3] = w & 0x00800080u;
  r[4] = w & 0x02000200u;
  r[5] = wr & 0x00200020u;
  r[6] = wr & 0x00800080u;
  r[7] = wr & 0x02000200u;
}


__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// min / max that return NaN when either input is NaN
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
// three-operand forms (one instruction on sm_100 and later)
__device__ __forceinline__ float fmin3_nan(float a, float b, float c) {
  float d;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (r0 - z, r1 - z) * inv as one packed subtract and one packed multiply; each
// element is rounded as __fmul_rn(__fsub_rn(r, z), inv) rounds it.  zz and ii
// hold z and inv in both halves.
__device__ __forceinline__ void sub_mul_x2(float r0, float r1, uint64_t zz, uint64_t ii, float& y0, float& y1) {
  uint64_t x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(r0), "f"(r1));
  asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(zz));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(ii));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(x));
}
__device__ __forceinline__ uint64_t splat_x2(float x) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(x));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1 / sqrt(128), rounded to float32
constexpr float kInvSqrt128 = 0.0883883476483184405f;

// In-quant Hadamard of one 128-channel group held by a warp: lane l holds
// channels l + 32 e in x[e] (e = 0..3); on return x[e] holds output channel
// l + 32 e of y = x H / sqrt(128), H[i][k] = (-1)^popcount(i & k) (Sylvester
// order).  Fast Walsh-Hadamard transform: one butterfly (a, c) -> (a + c,
// a - c) per channel-index bit, bits 5 and 6 inside the lane, bits 0-4 across
// lanes; then one multiplication by 1/sqrt(128).
__device__ __forceinline__ void hadamard128_warp(float (&x)[4], int lane) {
  const float s0 = x[0] + x[1], d0 = x[0] - x[1], s1 = x[2] + x[3], d1 = x[2] - x[3];
  x[0] = s0 + s1;
  x[2] = s0 - s1;
  x[1] = d0 + d1;
  x[3] = d0 - d1;
#pragma unroll
  for (int bit = 1; bit < 32; bit <<= 1) {
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], bit);
      x[e] = upper ? o - x[e] : x[e] + o;
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] *= kInvSqrt128;
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

__device__ __forceinline__ uint32_t pack_bf162(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// (hi, lo) split of a float into two fp16 values packed as one f16x2: hi in
// the low half, the rounding residue in the high half.
__device__ __forceinline__ uint32_t split_f16(float x) {
  const __half h = __float2half_rn(x);
  const __half l = __float2half_rn(x - __half2float(h));
  return pack_half2(h, l);
}

__device__ __forceinline__ uint32_t split_bf16(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  return pack_bf162(h, l);
}

// Three-way bf16 split: x ~ p[0] + p[1] + p[2] (bf16 bit patterns), ~24 bits.
__device__ __forceinline__ void split3_bf16(float x, uint32_t (&p)[3]) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
  p[0] = __bfloat16_as_ushort(h);
  p[1] = __bfloat16_as_ushort(m);
  p[2] = __bfloat16_as_ushort(l);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk copy (TMA engine, non-tensor form)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
      "p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or hint_ns nanoseconds pass, instead of spinning on issue slots
// the other warps of its SM sub-partition could use.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, "
      "p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity`: gives up after limit_ns of wall time (~2 s
// by default; checked at least every 20 us) and reports false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load of box (x, y) into shared memory, completing on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace oscar
