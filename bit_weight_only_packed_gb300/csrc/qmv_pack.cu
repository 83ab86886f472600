// qmv_pack.cu -- the packer (signed int8 codes -> packed words) and the
// unpack check kernel (packed words -> int8 codes through the same decode
// routine the matvec kernels use).
//
// Layout ("Gemma4 raw-Metal loop on A19", section "What moved the needle":
// sixteen int2 codes per 32-bit word): code k of a row sits in word
// floor(k*bits/32) at bit offset bits*(k mod (32/bits)), field u = v + 2^(bits-1).
// Because every row holds a whole number of words, word w of the matrix holds
// the 32/bits consecutive codes starting at w*(32/bits) of the row-major code
// array, so both kernels are flat over words.
#include "qmv_internal.cuh"

namespace qmv {

template <int BITS>
__global__ void __launch_bounds__(256) pack_kernel(const int8_t* __restrict__ in,
                                                  uint32_t* __restrict__ out, int64_t nwords) {
  constexpr int CPW = 32 / BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  constexpr int BIAS = 1 << (BITS - 1);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < nwords; w += stride) {
    const int8_t* src = in + w * CPW;
    int8_t c[CPW];
    if (CPW == 16) {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      memcpy(c, &v, 16);
    } else if (CPW == 8) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      memcpy(c, &v, 8);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
      memcpy(c, &v, 4);
    }
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < CPW; ++j) word |= ((uint32_t)(c[j] + BIAS) & MASK) << (BITS * j);
    out[w] = word;
  }
}

template <int BITS>
__global__ void __launch_bounds__(256) unpack_kernel(const uint32_t* __restrict__ in,
                                                    int8_t* __restrict__ out, int64_t nwords) {
  constexpr int CPW = 32 / BITS;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < nwords; w += stride) {
    __half2 vp[Fmt<BITS>::P];
    decode_word<BITS>(in[w], vp);
    int8_t c[CPW];
#pragma unroll
    for (int j = 0; j < CPW; ++j) c[j] = (int8_t)__half2int_rz(code_of<BITS>(vp, j));
    int8_t* dst = out + w * CPW;
    if (CPW == 16) {
      uint4 v;
      memcpy(&v, c, 16);
      *reinterpret_cast<uint4*>(dst) = v;
    } else if (CPW == 8) {
      uint2 v;
      memcpy(&v, c, 8);
      *reinterpret_cast<uint2*>(dst) = v;
    } else {
      uint32_t v;
      memcpy(&v, c, 4);
      *reinterpret_cast<uint32_t*>(dst) = v;
    }
  }
}

static int flat_grid(int64_t nwords) {
  const int64_t blocks = (nwords + 255) / 256;
  const int cap = 152 * 16;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

cudaError_t launch_pack(int bits, const int8_t* in, uint32_t* out, int64_t nwords, cudaStream_t s) {
  if (nwords == 0) return cudaSuccess;
  const int g = flat_grid(nwords);
  switch (bits) {
    case 2: pack_kernel<2><<<g, 256, 0, s>>>(in, out, nwords); break;
    case 4: pack_kernel<4><<<g, 256, 0, s>>>(in, out, nwords); break;
    default: pack_kernel<8><<<g, 256, 0, s>>>(in, out, nwords); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_unpack(int bits, const uint32_t* in, int8_t* out, int64_t nwords, cudaStream_t s) {
  if (nwords == 0) return cudaSuccess;
  const int g = flat_grid(nwords);
  switch (bits) {
    case 2: unpack_kernel<2><<<g, 256, 0, s>>>(in, out, nwords); break;
    case 4: unpack_kernel<4><<<g, 256, 0, s>>>(in, out, nwords); break;
    default: unpack_kernel<8><<<g, 256, 0, s>>>(in, out, nwords); break;
  }
  return cudaGetLastError();
}

}  // namespace qmv
