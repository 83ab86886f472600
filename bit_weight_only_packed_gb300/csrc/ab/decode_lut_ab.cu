// decode_lut_ab.cu -- measurement harness for the int2 decode choice (not
// part of libqmv: build.py compiles only csrc/*.cu).
//
// "Gemma4 raw-Metal loop on A19", section "What moved the needle": on the A19
// the arithmetic 2-bit unpack was ALU-bound and a constant-memory table of
// byte -> 4 values was the lever.  This harness asks the same question on
// GB300: the same streaming matvec over the int2 lm_head shape (262144 x
// 2048, group-32 fp16 scales), identical except for how the 2-bit fields
// become fp32 operands of the paired FMA:
//   MASK  the library's folded form: one 64-bit AND per field pair, the
//         fields read as fp32 subnormals, activations pre-scaled per offset
//   LUT   byte -> 4 fp32 values from a shared-memory table (one copy)
//   LUTR  the same table in 8 copies (lane & 7 picks one)
//   CLUT  the table in constant memory
// Each warp takes one row per iteration (lane l: 64 codes, two 32-code
// blocks), sums the blocks in fp32, scales them and reduces across lanes.
// It prints, per variant, the median, p10 and p90 of 9 interleaved timed
// launches and the largest relative difference from MASK.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo \
//        -o /tmp/decode_lut_ab bit_weight_only_packed_gb300/csrc/ab/decode_lut_ab.cu
//   /tmp/decode_lut_ab
#include <cstdio>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

typedef unsigned long long u64;
__device__ __forceinline__ u64 pk(float a, float b) { return ((u64)__float_as_uint(b) << 32) | __float_as_uint(a); }
__device__ __forceinline__ void upk(u64 v, float& a, float& b) { a = __uint_as_float((uint32_t)v); b = __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ u64 ffma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__constant__ float4 c_lut[256];

enum { MASK = 0, LUT = 1, LUTR = 2, CLUT = 3 };

// y table in shared memory: MASK: per item (64 codes) 32 steps of (even word, odd word) pairs pre-scaled
// by 2^(109 - o); LUT forms: per item 32 pairs of consecutive codes (plain y).
template <int DEC>
__global__ void __launch_bounds__(256) gemv_dec(const uint4* __restrict__ codes, const __half* __restrict__ scales,
                                                 const __half* __restrict__ x, float* __restrict__ y, int N) {
  constexpr int K = 2048, C = K / 64;          // 32 items per row (one per lane)
  __shared__ __align__(16) u64 ytab[C * 34];    // item stride 34 pairs: a warp's lanes (items) spread over all banks
  __shared__ __align__(16) float ysum[K / 32];
  __shared__ __align__(16) float4 lut[256 * 8];  // LUTR uses 8 copies; LUT the first
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 256 * 8; i += blockDim.x) {
    const int b = i & 255;
    lut[i] = make_float4((float)(b & 3), (float)((b >> 2) & 3), (float)((b >> 4) & 3), (float)((b >> 6) & 3));
  }
  // activation table
  for (int k = tid; k < K; k += blockDim.x) {
    const float f = __half2float(x[k]);
    const int c = k >> 6, kk = k & 63, blk = kk >> 5, k32 = kk & 31, j = k32 & 15, wi = k32 >> 4;
    float* t = reinterpret_cast<float*>(ytab);
    if (DEC == MASK) {
      const int o = 2 * (j & 7);
      t[2 * (34 * c + 16 * blk + j) + wi] = f * __int_as_float((127 + 109 - o) << 23);
    } else {
      t[2 * (34 * c) + kk] = f;   // consecutive codes: pair p = codes 2p, 2p+1
    }
  }
  for (int b = tid; b < K / 32; b += blockDim.x) {
    float s = 0.f;
    for (int k = 0; k < 32; ++k) s += __half2float(x[32 * b + k]);
    ysum[b] = 2.0f * s;
  }
  __syncthreads();
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + warp; row < N; row += nw) {
    const uint4 w = __ldg(codes + (size_t)row * (K / 64) + lane);   // words 4l .. 4l+3
    const __half2 sc = *reinterpret_cast<const __half2*>(scales + (size_t)row * (K / 32) + 2 * lane);
    float blk_sum[2];
    if (DEC == MASK) {
      const u64 p0 = ((u64)w.y << 32) | w.x, p1 = ((u64)w.w << 32) | w.z;   // block 0: words 0,1; block 1: 2,3
      const u64 h0 = p0 >> 16, h1 = p1 >> 16;
      u64 a0 = 0, a1 = 0;
      const u64* yc = ytab + 34 * lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t m = 3u << (2 * (j & 7));
        const u64 mm = ((u64)m << 32) | m;
        a0 = ffma2(yc[j], ((j < 8) ? p0 : h0) & mm, a0);
        a1 = ffma2(yc[16 + j], ((j < 8) ? p1 : h1) & mm, a1);
      }
      float e0, o0, e1, o1;
      upk(a0, e0, o0);
      upk(a1, e1, o1);
      blk_sum[0] = __fmaf_rn(e0 + o0, 1099511627776.0f, -ysum[2 * lane]);       // * 2^40
      blk_sum[1] = __fmaf_rn(e1 + o1, 1099511627776.0f, -ysum[2 * lane + 1]);
    } else {
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      const u64* yc = ytab + 34 * lane;
      u64 acc[2] = {0, 0};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t byte = (ws[q] >> (8 * b)) & 0xFFu;
          float4 u;
          if (DEC == LUT) u = lut[byte];
          else if (DEC == LUTR) u = lut[(lane & 7) * 256 + byte];
          else u = c_lut[byte];
          const int p = 8 * q + 2 * b;     // code pairs (16q+4b, +1), (+2, +3) -> pairs p, p+1 of the item
          acc[q >> 1] = ffma2(yc[p], pk(u.x, u.y), acc[q >> 1]);
          acc[q >> 1] = ffma2(yc[p + 1], pk(u.z, u.w), acc[q >> 1]);
        }
      }
      float e0, o0, e1, o1;
      upk(acc[0], e0, o0);
      upk(acc[1], e1, o1);
      blk_sum[0] = (e0 + o0) - ysum[2 * lane];
      blk_sum[1] = (e1 + o1) - ysum[2 * lane + 1];
    }
    float v = blk_sum[0] * __low2float(sc) + blk_sum[1] * __high2float(sc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0) y[row] = v;
  }
}

int main() {
  const int N = 262144, K = 2048;
  const size_t cb = (size_t)N * K / 4, sb = (size_t)N * (K / 32) * 2;
  uint4* codes; __half* scales; __half* x; float* y[4];
  cudaMalloc(&codes, cb); cudaMalloc(&scales, sb); cudaMalloc(&x, K * 2);
  for (int d = 0; d < 4; ++d) cudaMalloc(&y[d], N * 4);
  // deterministic pseudo-random codes, scales ~0.0125, x ~ small values
  {
    uint32_t* h = (uint32_t*)malloc(cb);
    uint64_t s = 0x9E3779B97F4A7C15ull;
    for (size_t i = 0; i < cb / 4; ++i) { s = s * 6364136223846793005ull + 1442695040888963407ull; h[i] = (uint32_t)(s >> 32); }
    cudaMemcpy(codes, h, cb, cudaMemcpyHostToDevice); free(h);
    __half* hs = (__half*)malloc(sb);
    for (size_t i = 0; i < sb / 2; ++i) hs[i] = __float2half(0.005f + 0.015f * (float)((i * 2654435761u) % 1000) / 1000.f);
    cudaMemcpy(scales, hs, sb, cudaMemcpyHostToDevice); free(hs);
    __half hx[2048];
    for (int k = 0; k < K; ++k) hx[k] = __float2half(((k * 7919) % 2001 - 1000) / 700.0f);
    cudaMemcpy(x, hx, K * 2, cudaMemcpyHostToDevice);
  }
  float4 hl[256];
  for (int b = 0; b < 256; ++b) hl[b] = make_float4(b & 3, (b >> 2) & 3, (b >> 4) & 3, (b >> 6) & 3);
  cudaMemcpyToSymbol(c_lut, hl, sizeof(hl));
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const char* names[4] = {"MASK (library folded form)", "LUT  (smem, one copy)", "LUTR (smem, 8 bank copies)", "CLUT (constant memory)"};
  void (*kern[4])(const uint4*, const __half*, const __half*, float*, int) = {gemv_dec<MASK>, gemv_dec<LUT>, gemv_dec<LUTR>, gemv_dec<CLUT>};
  int occ[4];
  for (int d = 0; d < 4; ++d) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[d], kern[d], 256, 0);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  float ms[4][9];
  const int only = getenv("DEC_ONLY") ? atoi(getenv("DEC_ONLY")) : -1;
  for (int rep = 0; rep < 9; ++rep)
    for (int d = 0; d < 4; ++d) {
      if (only >= 0 && d != only) continue;
      const int grid = sms * occ[d];
      kern[d]<<<grid, 256>>>(codes, scales, x, y[d], N);   // warm / interleaved
      cudaEventRecord(e0);
      kern[d]<<<grid, 256>>>(codes, scales, x, y[d], N);
      cudaEventRecord(e1);
      cudaEventSynchronize(e1);
      cudaEventElapsedTime(&ms[d][rep], e0, e1);
    }
  float* hy[4];
  for (int d = 0; d < 4; ++d) { hy[d] = (float*)malloc(N * 4); cudaMemcpy(hy[d], y[d], N * 4, cudaMemcpyDeviceToHost); }
  for (int d = 0; d < 4; ++d) {
    if (only >= 0 && d != only) continue;
    float v[9]; for (int r = 0; r < 9; ++r) v[r] = ms[d][r];
    for (int i = 0; i < 9; ++i) for (int j = i + 1; j < 9; ++j) if (v[j] < v[i]) { float t = v[i]; v[i] = v[j]; v[j] = t; }
    double maxd = 0;
    for (int i = 0; i < N; ++i) { double dd = fabs((double)hy[d][i] - hy[0][i]) / (1.0 + fabs((double)hy[0][i])); if (dd > maxd) maxd = dd; }
    printf("%-28s occ %d  median %8.2f us  p10 %8.2f  p90 %8.2f  %7.1f GB/s  max|y-mask|/(1+|mask|) %.2e\n", names[d], occ[d],
           v[4] * 1e3, v[1] * 1e3, v[7] * 1e3, (cb + sb) / (v[4] * 1e-3) / 1e9, maxd);
  }
  cudaError_t e = cudaDeviceSynchronize();
  printf("status %s\n", cudaGetErrorString(e));
  return e != cudaSuccess;
}
