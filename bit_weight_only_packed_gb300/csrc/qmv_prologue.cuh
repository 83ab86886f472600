// qmv_prologue.cuh -- device helpers shared by the CUDA-core kernels: 16-byte
// loads, fp16 element access, and the residual-add + RMSNorm steps ("Gemma4
// raw-Metal loop on A19", section "What moved the needle": the residual add
// and RMSNorm folded into the matvec prologue).  Every step is one IEEE fp32
// operation with round-to-nearest, in the order the oracle uses.
#pragma once
#include "qmv_internal.cuh"

namespace qmv {

__device__ __forceinline__ uint4 ldg16(const uint4* p) { return __ldg(p); }

__device__ __forceinline__ uint4 lds16(const __half* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ __half h_of(const uint4& v, int e) {
  const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
  return __ushort_as_half((e & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xFFFFu));
}

// inv = 1 / sqrt(ss / K + eps), each step one IEEE fp32 operation
__device__ __forceinline__ float rms_inv(float ss, int K, float eps) {
  const float mean = __fdiv_rn(ss, (float)K);
  const float t = __fadd_rn(mean, eps);
  const float rt = __fsqrt_rn(t);
  return __fdiv_rn(1.0f, rt);
}

__device__ __forceinline__ __half add_h(__half x, __half r) {
  return __float2half_rn(__fadd_rn(__half2float(x), __half2float(r)));
}

__device__ __forceinline__ __half norm_h(__half h, float inv, __half g) {
  return __float2half_rn(__fmul_rn(__fmul_rn(__half2float(h), inv), __half2float(g)));
}

// Block sum of squares of h = fp16(x + r) over the 32 codes at k0, serial in
// k; optionally stores h.  Squares of fp16 values are exact in fp32, so the
// fused multiply-add equals the rounded add of the square.
__device__ __forceinline__ float block_sumsq(const __half* x, const __half* r, int k0,
                                             __half* h_store) {
  float blk = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + k0 + 8 * q));
    const uint4 rv = __ldg(reinterpret_cast<const uint4*>(r + k0 + 8 * q));
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const __half h = add_h(h_of(xv, e), h_of(rv, e));
      if (h_store) h_store[k0 + 8 * q + e] = h;
      const float hf = __half2float(h);
      blk = __fmaf_rn(hf, hf, blk);
    }
  }
  return blk;
}


}  // namespace qmv
