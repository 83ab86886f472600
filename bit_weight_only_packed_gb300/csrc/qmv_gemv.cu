// qmv_gemv.cu -- CUDA-core matvec kernels (M = 1, and M-column tiles up to 32).
//
// What they compute ("Gemma4 raw-Metal loop on A19", section "What moved the
// needle"; "raw-metal-loop-playbook", prefill-regimes table): for each output
// scalar, every 32-code block is summed serially in k in fp32 (exact
// products), scaled (group 32) and folded into the accumulator serially over
// the blocks -- the order is a property of the output scalar alone, so the
// M = 1 kernel, every column of an M-tile and the oracle agree bit for bit.
//
// How the work is laid out on the GPU:
//   * Weights are streamed once with 16-byte coalesced loads (32 bytes per
//     thread for int8).  A thread's "item" is one load unit of one row, which
//     always covers whole 32-code blocks (int2: 64 codes = 2 blocks;
//     int4: 32 codes; int8: 32 codes in two 16-byte loads).
//   * The serial fold over a row's blocks is split from the block sums:
//     threads write each block's scaled sum to shared memory, then one thread
//     per row folds them in block order.  The dots run fully parallel; only
//     the K/32 adds of the fold are serial.
//   * M = 1 (gemv_m1): consecutive threads take consecutive items of a row
//     (coalesced).  A thread keeps the same item index for every row it
//     visits, so its slice of the activation vector stays in registers for
//     the whole kernel.  Each CTA owns a contiguous range of rows (balanced
//     over a persistent grid sized from the occupancy), walks it in passes of
//     RP*U rows with the next pass's loads in flight while the current pass
//     is decoded, and double-buffers the fold buffer so one barrier per pass
//     suffices.  With the fused prologue every CTA first forms
//     h = fp16(x + r), the blocked sum of squares, inv, and y in shared
//     memory (CTA 0 also writes h out).
//   * M-column tiles (gemm_small): a CTA owns 32 rows (one per lane) and
//     walks K in slabs; in each slab warp w takes item w of all 32 rows,
//     decodes it once and runs the block dots for all MT columns, reading the
//     activations from shared memory as broadcasts.  Fold threads own fixed
//     (row, column) pairs and keep their accumulators in registers across
//     slabs.
#include "qmv_prologue.cuh"

namespace qmv {

constexpr int M1_MAXT = 672;   // largest CTA of gemv_m1 (C*RP, a multiple of 32)

// CTAs of up to 256 threads keep 4 passes in flight; larger CTAs (long or
// odd K) keep 2, so that two register sets still fit without spills.
template <int MAXT> struct M1Lim { static constexpr int UM = (MAXT > 256) ? 2 : 4; };

// ============================================================== M = 1 ====

template <int BITS, int UM> struct PassRegs {
  uint4 q[UM][Fmt<BITS>::ITEM_U4];
  uint32_t s[UM];
};

template <int BITS, bool PERROW, int UM>
__device__ __forceinline__ void m1_load(PassRegs<BITS, UM>& R, const GemvArgs& a, int64_t rb, int ro,
                                        int c, int RP, int U, int64_t r_end) {
  using F = Fmt<BITS>;
#pragma unroll
  for (int j = 0; j < UM; ++j) {
    const int64_t row = rb + ro + (int64_t)j * RP;
    if (j < U && row < r_end) {
      const uint4* src = a.codes + row * a.row_u4 + (int64_t)c * F::ITEM_U4;
#pragma unroll
      for (int u = 0; u < F::ITEM_U4; ++u) R.q[j][u] = ldg16(src + u);
      if (!PERROW) {
        const __half* sp = a.scales + row * a.G + (int64_t)c * F::BLOCKS;
        if (F::BLOCKS == 2)
          R.s[j] = __ldg(reinterpret_cast<const unsigned int*>(sp));
        else
          R.s[j] = (uint32_t)__half_as_ushort(__ldg(sp));
      }
    }
  }
}

template <int BITS, bool PERROW, int UM>
__device__ __forceinline__ void m1_compute(const PassRegs<BITS, UM>& R, const __half2 (&ys)[Fmt<BITS>::CODES / 2],
                                           float* tb, int64_t rb, int ro, int c, int RP, int U,
                                           int64_t r_end, int GS) {
  using F = Fmt<BITS>;
#pragma unroll
  for (int j = 0; j < UM; ++j) {
    const int64_t row = rb + ro + (int64_t)j * RP;
    if (j < U && row < r_end) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&R.q[j][0]);
      float* dst = tb + (j * RP + ro) * GS + c * F::BLOCKS;
#pragma unroll
      for (int bb = 0; bb < F::BLOCKS; ++bb) {
        const float p = block_dot<BITS>(w + bb * F::WPB,
                                        [&](int k) { return y_of(ys, bb * 32 + k); });
        if (PERROW) {
          dst[bb] = p;
        } else {
          const uint16_t sb = (uint16_t)(R.s[j] >> (16 * bb));
          dst[bb] = __fmul_rn(p, __half2float(__ushort_as_half(sb)));
        }
      }
    }
  }
}

template <bool PERROW>
__device__ __forceinline__ void m1_fold(const GemvArgs& a, const float* tb, int64_t rb, int PR,
                                        int64_t r_end, int NB, int GS) {
  for (int lr = threadIdx.x; lr < PR; lr += blockDim.x) {
    const int64_t row = rb + lr;
    if (row >= r_end) break;
    const float* tr = tb + lr * GS;
    float acc;
    if (!PERROW) {
      acc = 0.0f;
#pragma unroll 8
      for (int b = 0; b < NB; ++b) acc = __fadd_rn(acc, tr[b]);
    } else {
      float q = tr[0];
#pragma unroll 8
      for (int b = 1; b < NB; ++b) q = __fadd_rn(q, tr[b]);
      acc = __fadd_rn(0.0f, __fmul_rn(q, __half2float(a.scales[row])));
    }
    if (a.y_f16)
      reinterpret_cast<__half*>(a.y)[row] = __float2half_rn(acc);
    else
      reinterpret_cast<float*>(a.y)[row] = acc;
  }
}

// shared-memory layout of gemv_m1 (floats): [tbuf: 2*PR*GS rounded to 4]
// [fused: y K halves][fused: block sums NB][inv 1] (each part 16-byte aligned)
__host__ __device__ inline int m1_tbuf_floats(int PR, int NB) { return ((2 * PR * (NB + 1)) + 3) & ~3; }

template <int BITS, bool PERROW, bool FUSED, int MAXT>
__global__ void __launch_bounds__(MAXT) gemv_m1_kernel(GemvArgs a, int C, int RP, int U) {
  using F = Fmt<BITS>;
  constexpr int UM = M1Lim<MAXT>::UM;
  const int t = threadIdx.x;
  const int T = blockDim.x;
  const int c = t % C;
  const int ro = t / C;
  const int K = a.K;
  const int NB = K / 32;
  const int GS = NB + 1;
  const int PR = RP * U;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* tbuf = reinterpret_cast<float*>(smem_raw);
  const int tfl = m1_tbuf_floats(RP * UM, NB);

  const int64_t r_begin = (int64_t)blockIdx.x * a.N / gridDim.x;
  const int64_t r_end = (int64_t)(blockIdx.x + 1) * a.N / gridDim.x;

  __half2 ys[F::CODES / 2];
  if (FUSED) {
    __half* hy = reinterpret_cast<__half*>(tbuf + tfl);
    float* bsum = reinterpret_cast<float*>(hy + ((K + 7) & ~7));
    float* inv_sh = bsum + ((NB + 3) & ~3);
    __half* h_out = (blockIdx.x == 0) ? a.h_out : nullptr;
    for (int b = t; b < NB; b += T) bsum[b] = block_sumsq(a.x, a.r, b * 32, hy);
    __syncthreads();
    if (t == 0) {
      float ss = 0.0f;
      for (int b = 0; b < NB; ++b) ss = __fadd_rn(ss, bsum[b]);
      *inv_sh = rms_inv(ss, K, a.eps);
    }
    __syncthreads();
    const float inv = *inv_sh;
    for (int k = t; k < K; k += T) {
      const __half h = hy[k];
      if (h_out) h_out[k] = h;
      hy[k] = norm_h(h, inv, a.gamma[k]);
    }
    __syncthreads();
#pragma unroll
    for (int v = 0; v < F::CODES / 8; ++v) {
      const uint4 q = lds16(hy + c * F::CODES + 8 * v);
      ys[4 * v + 0] = u32_as_h2(q.x);
      ys[4 * v + 1] = u32_as_h2(q.y);
      ys[4 * v + 2] = u32_as_h2(q.z);
      ys[4 * v + 3] = u32_as_h2(q.w);
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + c * F::CODES);
#pragma unroll
    for (int v = 0; v < F::CODES / 8; ++v) {
      const uint4 q = __ldg(src + v);
      ys[4 * v + 0] = u32_as_h2(q.x);
      ys[4 * v + 1] = u32_as_h2(q.y);
      ys[4 * v + 2] = u32_as_h2(q.z);
      ys[4 * v + 3] = u32_as_h2(q.w);
    }
  }

  PassRegs<BITS, UM> A, B;
  int64_t rb = r_begin;
  int buf = 0;
  if (rb < r_end) m1_load<BITS, PERROW, UM>(A, a, rb, ro, c, RP, U, r_end);
  while (rb < r_end) {
    const int64_t rn = rb + PR;
    if (rn < r_end) m1_load<BITS, PERROW, UM>(B, a, rn, ro, c, RP, U, r_end);
    m1_compute<BITS, PERROW, UM>(A, ys, tbuf + buf * PR * GS, rb, ro, c, RP, U, r_end, GS);
    __syncthreads();
    m1_fold<PERROW>(a, tbuf + buf * PR * GS, rb, PR, r_end, NB, GS);
    buf ^= 1;
    rb = rn;
    if (rb >= r_end) break;
    const int64_t rn2 = rb + PR;
    if (rn2 < r_end) m1_load<BITS, PERROW, UM>(A, a, rn2, ro, c, RP, U, r_end);
    m1_compute<BITS, PERROW, UM>(B, ys, tbuf + buf * PR * GS, rb, ro, c, RP, U, r_end, GS);
    __syncthreads();
    m1_fold<PERROW>(a, tbuf + buf * PR * GS, rb, PR, r_end, NB, GS);
    buf ^= 1;
    rb = rn2;
  }
}

// ======================================================= M-column tiles ====

constexpr int SM_WARPS = 8;

template <int BITS, int MT> struct SmallCfg {
  static constexpr int SLAB = SM_WARPS * Fmt<BITS>::CODES;   // codes per slab
  static constexpr int SB = SLAB / 32;                       // blocks per slab
  static constexpr int PAIRS = 32 * MT;
  static constexpr int PPT = (PAIRS + 255) / 256;
  static constexpr int YS_HALVES = MT * SLAB;
  static constexpr int TB_FLOATS = SB * MT * 32;
};

// smem: [ys MT*SLAB halves][tb SB*MT*32 floats][inv MT floats][bsum MT*NB floats (fused)]
template <int BITS, int MT>
__host__ __device__ inline size_t small_smem_bytes(int NB, bool fused) {
  using S = SmallCfg<BITS, MT>;
  size_t b = (size_t)S::YS_HALVES * 2 + (size_t)S::TB_FLOATS * 4 + (size_t)((MT + 3) & ~3) * 4;
  if (fused) b += (size_t)MT * NB * 4;
  return b;
}

template <int BITS, int MT>
__global__ void __launch_bounds__(256) gemm_small_kernel(GemvArgs a) {
  using F = Fmt<BITS>;
  using S = SmallCfg<BITS, MT>;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int K = a.K, NB = K / 32, M = a.M;
  const int64_t row0 = (int64_t)blockIdx.x * 32;
  const int64_t row = row0 + lane;
  const bool row_ok = row < a.N;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __half* ys = reinterpret_cast<__half*>(smem_raw);
  float* tb = reinterpret_cast<float*>(ys + S::YS_HALVES);
  float* inv = tb + S::TB_FLOATS;
  float* bsum = inv + ((MT + 3) & ~3);

  if (a.fused) {
    for (int e = t; e < M * NB; e += 256) {
      const int m = e / NB, b = e % NB;
      bsum[m * NB + b] = block_sumsq(a.x + (int64_t)m * K, a.r + (int64_t)m * K, b * 32, nullptr);
    }
    __syncthreads();
    if (t < M) {
      float ss = 0.0f;
      for (int b = 0; b < NB; ++b) ss = __fadd_rn(ss, bsum[t * NB + b]);
      inv[t] = rms_inv(ss, K, a.eps);
    }
    __syncthreads();
  }

  float acc[S::PPT];
#pragma unroll
  for (int i = 0; i < S::PPT; ++i) acc[i] = 0.0f;

  for (int s0 = 0; s0 < K; s0 += S::SLAB) {
    const int slab = min(S::SLAB, K - s0);
    const int v8 = slab / 8;
    // stage the activations of this slab for all MT columns (zeros past M)
    for (int e = t; e < MT * v8; e += 256) {
      const int m = e / v8, kk = 8 * (e % v8);
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (m < M) {
        const int64_t off = (int64_t)m * K + s0 + kk;
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + off));
        if (a.fused) {
          const uint4 rv = __ldg(reinterpret_cast<const uint4*>(a.r + off));
          const uint4 gv = __ldg(reinterpret_cast<const uint4*>(a.gamma + s0 + kk));
          const float iv = inv[m];
          uint16_t hh[8], yy[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const __half h = add_h(h_of(xv, q), h_of(rv, q));
            hh[q] = __half_as_ushort(h);
            yy[q] = __half_as_ushort(norm_h(h, iv, h_of(gv, q)));
          }
          if (a.h_out && blockIdx.x == 0) {
            uint4 hv;
            memcpy(&hv, hh, 16);
            *reinterpret_cast<uint4*>(a.h_out + off) = hv;
          }
          memcpy(&out, yy, 16);
        } else {
          out = xv;
        }
      }
      *reinterpret_cast<uint4*>(ys + m * S::SLAB + kk) = out;
    }
    __syncthreads();

    // block sums of item `warp` of this slab for the 32 rows, all columns
    if (warp * F::CODES < slab) {
      const int item = s0 / F::CODES + warp;
      uint4 q[F::ITEM_U4];
      uint32_t sc = 0;
      if (row_ok) {
        const uint4* src = a.codes + row * a.row_u4 + (int64_t)item * F::ITEM_U4;
#pragma unroll
        for (int u = 0; u < F::ITEM_U4; ++u) q[u] = ldg16(src + u);
        if (!a.perrow) {
          const __half* sp = a.scales + row * a.G + (int64_t)item * F::BLOCKS;
          if (F::BLOCKS == 2)
            sc = __ldg(reinterpret_cast<const unsigned int*>(sp));
          else
            sc = (uint32_t)__half_as_ushort(__ldg(sp));
        }
      } else {
#pragma unroll
        for (int u = 0; u < F::ITEM_U4; ++u) q[u] = make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t* w = reinterpret_cast<const uint32_t*>(q);
      __half2 vp[F::WORDS][F::P];
#pragma unroll
      for (int wi = 0; wi < F::WORDS; ++wi) decode_word<BITS>(w[wi], vp[wi]);
#pragma unroll
      for (int bb = 0; bb < F::BLOCKS; ++bb) {
        const float s = __half2float(__ushort_as_half((uint16_t)(sc >> (16 * bb))));
        float* dst = tb + ((warp * F::BLOCKS + bb) * MT) * 32 + lane;
#pragma unroll 1
        for (int m = 0; m < MT; ++m) {
          const __half* yrow = ys + m * S::SLAB + warp * F::CODES + bb * 32;
          float p = 0.0f;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const uint4 yv = lds16(yrow + 8 * c8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int k = bb * 32 + c8 * 8 + e;             // code index inside the item
              const int wi = k / F::CPW, j = k % F::CPW;
              p = fma_hh(h_of(yv, e), code_of<BITS>(vp[wi], j), p);
            }
          }
          dst[m * 32] = a.perrow ? p : __fmul_rn(p, s);
        }
      }
    }
    __syncthreads();

    // fold this slab's blocks, in order, into the (row, column) accumulators
    const int sbe = slab / 32;
#pragma unroll
    for (int i = 0; i < S::PPT; ++i) {
      const int pq = t + 256 * i;
      if (pq < S::PAIRS) {
        const int prow = pq & 31, pm = pq >> 5;
        float v = acc[i];
        for (int b = 0; b < sbe; ++b) v = __fadd_rn(v, tb[(b * MT + pm) * 32 + prow]);
        acc[i] = v;
      }
    }
  }

#pragma unroll
  for (int i = 0; i < S::PPT; ++i) {
    const int pq = t + 256 * i;
    if (pq < S::PAIRS) {
      const int prow = pq & 31, pm = pq >> 5;
      const int64_t r = row0 + prow;
      if (r < a.N && pm < M) {
        float v = acc[i];
        if (a.perrow) v = __fadd_rn(0.0f, __fmul_rn(v, __half2float(a.scales[r])));
        const int64_t o = (int64_t)pm * a.N + r;
        if (a.y_f16)
          reinterpret_cast<__half*>(a.y)[o] = __float2half_rn(v);
        else
          reinterpret_cast<float*>(a.y)[o] = v;
      }
    }
  }
}


// ============================================================ launchers ====

template <int BITS, bool PERROW, bool FUSED, int MAXT>
static int run_m1_t(const GemvArgs& a, int C, int RP, cudaStream_t s, cudaError_t* err) {
  constexpr int UM = M1Lim<MAXT>::UM;
  const int T = C * RP;
  const int NB = a.K / 32;
  size_t smem = (size_t)m1_tbuf_floats(RP * UM, NB) * 4;
  if (FUSED) smem += (size_t)((a.K + 7) & ~7) * 2 + (size_t)(((NB + 3) & ~3) + 4) * 4;
  const DevInfo& d = dev_info();
  if (smem > (size_t)d.max_smem_optin) return QMV_ERR_UNSUPPORTED;
  auto kern = gemv_m1_kernel<BITS, PERROW, FUSED, MAXT>;
  static thread_local KernCache cache;
  int occ = 0;
  cudaError_t e = prep_kernel(kern, cache, T, smem, &occ);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  if (occ < 1) return QMV_ERR_UNSUPPORTED;
  int64_t grid = (int64_t)d.sms * occ;
  const int64_t need = ((int64_t)a.N + RP - 1) / RP;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  const int64_t rows_per_cta = ((int64_t)a.N + grid - 1) / grid;
  int U = (int)((rows_per_cta + RP - 1) / RP);
  if (U > UM) U = UM;
  if (U < 1) U = 1;
  kern<<<(unsigned)grid, T, smem, s>>>(a, C, RP, U);
  e = cudaGetLastError();
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

template <int BITS, bool PERROW, bool FUSED>
static int run_m1(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  const int C = a.K / Fmt<BITS>::CODES;
  int RP = 1;
  while ((C * RP) % 32 != 0) ++RP;
  while (C * RP * 2 <= 256) RP *= 2;
  const int T = C * RP;
  if (T > M1_MAXT) return QMV_ERR_UNSUPPORTED;
  if (T <= 256) return run_m1_t<BITS, PERROW, FUSED, 256>(a, C, RP, s, err);
  return run_m1_t<BITS, PERROW, FUSED, M1_MAXT>(a, C, RP, s, err);
}

int launch_gemv_m1(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err) {
  const bool pr = a.perrow != 0, fu = a.fused != 0;
#define QMV_M1(B)                                                   \
  if (pr) return fu ? run_m1<B, true, true>(a, s, err) : run_m1<B, true, false>(a, s, err); \
  return fu ? run_m1<B, false, true>(a, s, err) : run_m1<B, false, false>(a, s, err);
  switch (bits) {
    case 2: { QMV_M1(2) }
    case 4: { QMV_M1(4) }
    default: { QMV_M1(8) }
  }
#undef QMV_M1
}

template <int BITS, int MT>
static int run_small(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  const int NB = a.K / 32;
  const size_t smem = small_smem_bytes<BITS, MT>(NB, a.fused != 0);
  const DevInfo& d = dev_info();
  if (smem > (size_t)d.max_smem_optin) return QMV_ERR_UNSUPPORTED;
  auto kern = gemm_small_kernel<BITS, MT>;
  static thread_local KernCache cache;
  cudaError_t e = prep_kernel(kern, cache, 256, smem, nullptr);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  const int64_t grid = ((int64_t)a.N + 31) / 32;
  kern<<<(unsigned)grid, 256, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

template <int BITS>
static int small_bits(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  if (a.K % 64 == 0) {
    const int rc = launch_tile(a, BITS, s, err);
    if (rc != QMV_ERR_UNSUPPORTED) return rc;
  }
  if (a.M <= 4) return run_small<BITS, 4>(a, s, err);
  if (a.M <= 8) return run_small<BITS, 8>(a, s, err);
  if (a.M <= 16) return run_small<BITS, 16>(a, s, err);
  return run_small<BITS, 32>(a, s, err);
}
int launch_gemm_small(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err) {
  if (a.M < 1 || a.M > 32) return QMV_ERR_INVALID_ARG;
  switch (bits) {
    case 2: return small_bits<2>(a, s, err);
    case 4: return small_bits<4>(a, s, err);
    default: return small_bits<8>(a, s, err);
  }
}

}  // namespace qmv
