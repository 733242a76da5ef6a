// Per-element arithmetic of the Sage Q/K quantisation, shared by the prepare
// kernels (8 lanes per 128-channel row) and by the attention kernel's
// quantise-on-load of Q (one thread per row), so that both produce the same
// codes bit for bit.  Follows the aiter pull request "gfx1201_sage_prepare /
// gfx1201_sage_attention" (commit message of gfx1201_sage_prepare; Technical
// Details): INT8 codes with one scale per 32-row block, softmax_scale * log2 e
// folded into Q's scales, after an optional RMSNorm and rotate-half RoPE of Q
// and K with PyTorch's eager BF16 rounding points.
//
// Instruction selection keeps the instruction count low while every result
// stays that of the rounded operation it implements: BF16 roundings of binary32
// values go in pairs (cvt.rn.bf16x2.f32); a BF16 x BF16 product or BF16 + BF16
// sum that eager arithmetic rounds from binary32 is one mul/add.rn.bf16x2 (the
// same value, see bf2_mul); block maxima of |BF16| values are taken on packed
// pairs (max.bf16x2); and the code clamp(rne(v * inv), -127, 127) is formed as
// v * inv + 1.5 * 2^23, whose addition rounds to the integer and leaves it in
// the low mantissa bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace sa {
namespace qk {

// A BF16 pair packed in 32 bits (channel 2w low, 2w + 1 high) as two floats.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two floats rounded to BF16 (nearest even) by one paired conversion, packed.
__device__ __forceinline__ uint32_t bf2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Products and sums of two BF16 values, rounded once to BF16 (mul/add.rn.bf16x2).
// Eager BF16 arithmetic computes them in binary32 and rounds that to BF16; the two
// agree for all finite operands.  A product of two 8-bit significands is exact in
// binary32 down to 2^-149, and below that it lies under the smallest BF16 rounding
// midpoint (2^-134) either way.  A sum is exact in binary32 unless the exponents
// differ by more than 15, and then the smaller term is far below half a BF16 ulp
// of the larger, so both roundings return the larger.
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Per-half maximum of two BF16 pairs (max.bf16x2).
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf2_abs(uint32_t a) { return a & 0x7fff7fffu; }

// ------------------------------------------------------------------ RMSNorm
// Sum of squares of 16 channels (8 packed pairs) in channel order, from 0.
__device__ __forceinline__ float sumsq16(const uint32_t* w) {
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // unpacked by byte permutes rather than the shifts of bf_lo / bf_hi, so that callers
    // which scale the same words afterwards recompute the floats instead of holding them
    const float lo = __uint_as_float(__byte_perm(w[i], 0u, 0x1044));
    const float hi = __uint_as_float(__byte_perm(w[i], 0u, 0x3244));
    acc = __fadd_rn(acc, __fmul_rn(lo, lo));
    acc = __fadd_rn(acc, __fmul_rn(hi, hi));
  }
  return acc;
}
// The row's sum of squares from the partials P_0..P_7 of its eight 16-channel
// groups: ((P0 + P4) + (P2 + P6)) + ((P1 + P5) + (P3 + P7)), the order an XOR
// butterfly over eight lanes at distances 4, 2, 1 gives every lane.
__device__ __forceinline__ float sumsq_combine(const float (&P)[8]) {
  return __fadd_rn(__fadd_rn(__fadd_rn(P[0], P[4]), __fadd_rn(P[2], P[6])),
                   __fadd_rn(__fadd_rn(P[1], P[5]), __fadd_rn(P[3], P[7])));
}
// r = 1 / sqrt(mean of squares + eps), the square root and the reciprocal each rounded once.
__device__ __forceinline__ float rms_factor(float sumsq, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(sumsq, 1.0f / 128.0f), eps)));
}
// bf16(bf16(x * r) * w) for a channel pair.
__device__ __forceinline__ uint32_t rms_apply(uint32_t x, float r, uint32_t w) {
  return bf2_mul(bf2_bits(__fmul_rn(bf_lo(x), r), __fmul_rn(bf_hi(x), r)), w);
}

// ------------------------------------------------------------------ RoPE
// Rotate-half: bf16(bf16(x * cos) + bf16(rot * sin)), rot = -partner on the first half of
// the rotated channels and +partner on the second.  round(-u) = -round(u) under
// nearest-even rounding, so the rounded partner * sin pair has its signs flipped instead.
__device__ __forceinline__ uint32_t rope_first_half(uint32_t x, uint32_t partner, uint32_t c, uint32_t s) {
  return bf2_add(bf2_mul(x, c), bf2_mul(partner, s) ^ 0x80008000u);
}
__device__ __forceinline__ uint32_t rope_second_half(uint32_t x, uint32_t partner, uint32_t c, uint32_t s) {
  return bf2_add(bf2_mul(x, c), bf2_mul(partner, s));
}

// ------------------------------------------------------------------ codes
// 1.5 * 2^23: for |v| < 2^22, v + kRoundMagic is rounded to an integer (nearest even) by the
// addition itself, and that integer n is stored in the low mantissa bits: bits = 0x4B400000 + n.
constexpr float kRoundMagic = 12582912.0f;

// 127 / a for the block's largest |x| = a (0 for an all-zero block).
__device__ __forceinline__ float code_factor(float a) { return (a > 0.0f) ? __fdiv_rn(127.0f, a) : 0.0f; }
// The block's scale a / 127, times mult (Q: softmax_scale * log2 e; K: 1).
__device__ __forceinline__ float block_scale(float a, float mult, bool is_q) {
  if (!(a > 0.0f)) return 0.0f;
  const float sc = __fdiv_rn(a, 127.0f);
  return is_q ? __fmul_rn(sc, mult) : sc;
}
// rne(v * inv) + kRoundMagic, with v * inv clamped to [-127, 127] first (the same integer
// as clamping after rounding).  With a finite inv the clamp never binds: |v| <= a, so
// |v * inv| <= 127 (1 + 2^-24) before rounding, which rounds to 127.  Only when 127 / a
// overflows (a whole block below 3.7e-37) is it needed; kClamp selects it.
template <bool kClamp>
__device__ __forceinline__ float code_magic(float v, float inv) {
  float t = __fmul_rn(v, inv);
  if (kClamp) t = fminf(fmaxf(t, -127.0f), 127.0f);
  return __fadd_rn(t, kRoundMagic);
}
// Two codes (as their kRoundMagic sums) -> the FP16 pair of the codes, exact (|code| <= 127).
__device__ __forceinline__ uint32_t codes_fp16x2(float y0, float y1) {
  const __half2 hv = __floats2half2_rn(__fsub_rn(y0, kRoundMagic), __fsub_rn(y1, kRoundMagic));
  return *reinterpret_cast<const uint32_t*>(&hv);
}
// Four codes (as their kRoundMagic sums) -> four INT8 bytes, element 0 lowest: a code's
// two's-complement byte is the low byte of its sum.
__device__ __forceinline__ uint32_t codes_int8x4(float y0, float y1, float y2, float y3) {
  const uint32_t lo = __byte_perm(__float_as_uint(y0), __float_as_uint(y1), 0x0040);
  const uint32_t hi = __byte_perm(__float_as_uint(y2), __float_as_uint(y3), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

}  // namespace qk
}  // namespace sa
