// qmv_decode.cuh -- code decode and the exact block dot shared by every
// CUDA-core kernel (and by the unpack check kernel).
//
// Decode ("Gemma4 raw-Metal loop on A19", section "What moved the needle":
// int2 codes, 16 per 32-bit word, decoding to {-2,-1,0,1}; int4 and int8 use
// the same offset-binary fields).  Two fields that sit at the same offset in
// the two 16-bit halves of a word are decoded together: a LOP3 masks them in
// place and ORs in the fp16 exponent of 1024, giving the half2
// (1024 + u_a * 2^j, 1024 + u_b * 2^j) exactly (the field stays inside the
// 10-bit mantissa), and one HFMA2 rescales by 2^-j and removes 1024*2^-j plus
// the offset 2^(bits-1).  Every intermediate is an integer-valued fp16 and the
// fused multiply-add's exact result is representable, so v = u - 2^(bits-1)
// comes out exact.  Fields above bit 9 of a half are first brought down by
// one shift of the whole word.  This is the magic-exponent int->float
// conversion (a public technique), about one instruction per code.
//
// Block dot: p = sum over 32 consecutive codes of y_k * v_k, serially in k,
// each step one fp32 fused multiply-add whose product is exact (an 11-bit
// fp16 times an integer of at most 8 bits), so each step equals one rounded
// fp32 add -- the oracle's code order.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace qmv {

template <int BITS> struct Fmt {
  static constexpr int CPW = 32 / BITS;              // codes per 32-bit word
  static constexpr int P = CPW / 2;                  // half2 pairs per word
  static constexpr int ITEM_U4 = (BITS == 8) ? 2 : 1;  // 16-byte loads per item
  static constexpr int WORDS = ITEM_U4 * 4;          // words per item
  static constexpr int CODES = WORDS * CPW;          // codes per item: 64 / 32 / 32
  static constexpr int BLOCKS = CODES / 32;          // 32-code blocks per item: 2 / 1 / 1
  static constexpr int WPB = 32 / CPW;               // words per block: 2 / 4 / 8
};

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = u;
  return h;
}

__device__ __forceinline__ __half2 h2c(uint16_t lo, uint16_t hi) {
  return u32_as_h2((uint32_t)lo | ((uint32_t)hi << 16));
}

// fp16 bit patterns of the decode constants
#define QMV_H_ONE 0x3C00u       // 1.0
#define QMV_H_Q   0x3400u       // 0.25
#define QMV_H_S16 0x2C00u       // 1/16
#define QMV_H_S64 0x2400u       // 1/64
#define QMV_H_S256 0x1C00u      // 1/256
#define QMV_MAGIC 0x64006400u   // half2(1024, 1024)

__device__ __forceinline__ __half2 affine(uint32_t t, uint16_t scale, uint16_t offs) {
  return __hfma2(u32_as_h2(t), h2c(scale, scale), h2c(offs, offs));
}

// vp[i] holds (v_i, v_{i+P}) of the word's codes 0 .. CPW-1.
template <int BITS> __device__ __forceinline__ void decode_word(uint32_t w, __half2 (&vp)[Fmt<BITS>::P]);

template <> __device__ __forceinline__ void decode_word<2>(uint32_t w, __half2 (&vp)[8]) {
  const uint32_t w5 = w >> 10;
  // offsets -(1024*4^-j + 2): -1026, -258, -66, -18, -6 as fp16 bits
  vp[0] = affine((w & 0x00030003u) | QMV_MAGIC, QMV_H_ONE, 0xE402u);
  vp[1] = affine((w & 0x000C000Cu) | QMV_MAGIC, QMV_H_Q, 0xDC08u);
  vp[2] = affine((w & 0x00300030u) | QMV_MAGIC, QMV_H_S16, 0xD420u);
  vp[3] = affine((w & 0x00C000C0u) | QMV_MAGIC, QMV_H_S64, 0xCC80u);
  vp[4] = affine((w & 0x03000300u) | QMV_MAGIC, QMV_H_S256, 0xC600u);
  vp[5] = affine((w5 & 0x00030003u) | QMV_MAGIC, QMV_H_ONE, 0xE402u);
  vp[6] = affine((w5 & 0x000C000Cu) | QMV_MAGIC, QMV_H_Q, 0xDC08u);
  vp[7] = affine((w5 & 0x00300030u) | QMV_MAGIC, QMV_H_S16, 0xD420u);
}

template <> __device__ __forceinline__ void decode_word<4>(uint32_t w, __half2 (&vp)[4]) {
  const uint32_t w8 = w >> 8;
  // offsets -(1024 + 8) = -1032 and -(64 + 8) = -72
  vp[0] = affine((w & 0x000F000Fu) | QMV_MAGIC, QMV_H_ONE, 0xE408u);
  vp[1] = affine((w & 0x00F000F0u) | QMV_MAGIC, QMV_H_S16, 0xD480u);
  vp[2] = affine((w8 & 0x000F000Fu) | QMV_MAGIC, QMV_H_ONE, 0xE408u);
  vp[3] = affine((w8 & 0x00F000F0u) | QMV_MAGIC, QMV_H_S16, 0xD480u);
}

template <> __device__ __forceinline__ void decode_word<8>(uint32_t w, __half2 (&vp)[2]) {
  // offset -(1024 + 128) = -1152
  vp[0] = affine((w & 0x00FF00FFu) | QMV_MAGIC, QMV_H_ONE, 0xE480u);
  vp[1] = affine(((w >> 8) & 0x00FF00FFu) | QMV_MAGIC, QMV_H_ONE, 0xE480u);
}

// code j (0 .. CPW-1) of a decoded word
template <int BITS>
__device__ __forceinline__ __half code_of(const __half2 (&vp)[Fmt<BITS>::P], int j) {
  constexpr int P = Fmt<BITS>::P;
  return (j < P) ? __low2half(vp[j % P]) : __high2half(vp[j % P]);
}

// d = c + a*b with one rounding; a, b fp16, c and d fp32 (the product of two
// fp16 values is exact in fp32, so this equals the rounded fp32 add).
__device__ __forceinline__ float fma_hh(__half a, __half b, float c) {
#if defined(QMV_NO_MIXED_FMA)
  return __fmaf_rn(__half2float(a), __half2float(b), c);
#else
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;"
      : "=f"(d)
      : "h"(__half_as_ushort(a)), "h"(__half_as_ushort(b)), "f"(c));
  return d;
#endif
}

// y_k of a slice held as consecutive half2 pairs
__device__ __forceinline__ __half y_of(const __half2* ys, int k) {
  return (k & 1) ? __high2half(ys[k >> 1]) : __low2half(ys[k >> 1]);
}

// Serial exact dot of one 32-code block: words w[0 .. WPB-1], activations
// y_k = yk(k) for k = 0 .. 31 of the block.
template <int BITS, typename YF>
__device__ __forceinline__ float block_dot(const uint32_t* w, YF yk) {
  constexpr int CPW = Fmt<BITS>::CPW;
  constexpr int WPB = Fmt<BITS>::WPB;
  float p = 0.0f;
#pragma unroll
  for (int wi = 0; wi < WPB; ++wi) {
    __half2 vp[Fmt<BITS>::P];
    decode_word<BITS>(w[wi], vp);
#pragma unroll
    for (int j = 0; j < CPW; ++j) p = fma_hh(yk(wi * CPW + j), code_of<BITS>(vp, j), p);
  }
  return p;
}


// ---- exact fp32 decode on paired lanes (used by the M = 1 pipeline and the
// ---- M-column tiles) -------------------------------------------------------
//
// A b-bit field u at bit offset o < 16 - b of a 32-bit word becomes the fp32
// value 2^23 + u*2^o with one LOP3 ((w & (mask << o)) | 0x4B000000, exact:
// the field lies in the mantissa).  Subtracting 2^23 + 2^(b-1)*2^o gives
// v*2^o exactly (v = u - 2^(b-1)).  Two such values, one from each of the two
// 32-code blocks of a 64-code item, share one paired fp32 instruction; the
// activation is pre-scaled by 2^-o so that (y*2^-o)*(v*2^o) = y*v exactly and
// one paired FMA advances both blocks' serial sums by their exact products.

typedef unsigned long long u64;

__device__ __forceinline__ u64 pk(float a, float b) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(u64 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
// d = a*b + c on two fp32 lanes, each lane rounded once
__device__ __forceinline__ u64 ffma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// v' = ((a & m) | 0x4B000000, (b & m) | 0x4B000000) - off on two fp32 lanes.
// With m = (2^bits - 1) << o the magic float is 2^23 + u*2^o exactly, and
// off = 2^23 + 2^(bits-1)*2^o, so v' = (u - 2^(bits-1)) * 2^o = v * 2^o
// exactly.  Both LOP3s write the halves of one register pair that the paired
// add reads.
__device__ __forceinline__ u64 decode2(uint32_t a, uint32_t b, uint32_t m, u64 off) {
  u64 v;
  asm("{\n\t.reg .b32 t0, t1;\n\t.reg .b64 t;\n\t"
      "lop3.b32 t0, %1, %3, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 t1, %2, %3, 0x4B000000, 0xEA;\n\t"
      "mov.b64 t, {t0, t1};\n\t"
      "sub.rn.f32x2 %0, t, %4;\n\t}"
      : "=l"(v)
      : "r"(a), "r"(b), "r"(m), "l"(off));
  return v;
}

// ---- fast mode: the folded-offset form ------------------------------------
//
// With v = u - 2^(b-1), a block's dot is sum_k y_k*u_k - 2^(b-1)*S where
// S = sum_k y_k, so the offset can be taken out of the per-code work.  A field
// at bit offset o (o + b <= 16) masked in place, (w & (mask << o)), read as
// fp32 bits is the subnormal u * 2^o * 2^-149 exactly.  With the activation
// pre-scaled to y' = y * 2^(FOLD_E - o) one paired FMA adds y*u*2^-40 (an
// exact product, |y'| < 2^125 for every finite fp16 y, and every nonzero
// product is a normal number) to a running sum: one mask per code and one
// paired FMA per two codes, no subtraction.  The two lanes of the paired FMA
// take two adjacent words of a block (words 2p and 2p+1, which sit in one
// 64-bit register pair, so one 64-bit AND masks both fields in place): lane 0
// sums the block's even words and lane 1 its odd words, each serially in code
// order, and P = P_even + P_odd.  The block result is fma(P, 2^40,
// -2^(b-1)*S) (P*2^40 is exact), then scaled as in the exact form.  The sums
// differ from the exact form's serial order only by rounding, so this is the
// fast mode's arithmetic.  S is formed in the same order as P (S_even and
// S_odd serially, then added): P*2^40 is then exactly 2^(b-1)*S when every
// code of the block is zero (u = 2^(b-1)), which gives exactly 0, and every
// kernel that uses the form agrees bit for bit.
constexpr int FOLD_E = 109;

// block result from the running sum P (units of 2^-40) and bS = 2^(b-1)*S
__device__ __forceinline__ float fold_block(float P, float bS) {
  return __fmaf_rn(P, 1099511627776.0f /* 2^40 */, -bS);
}

}  // namespace qmv
