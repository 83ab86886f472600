// qmv_tc.cu -- tensor-core tiles for M >= 33 token columns (fast mode, int2).
//
// "raw-metal-loop-playbook", prefill-regimes table: chunks of 64/128 tokens
// go to the matrix units; the accumulation order then is the hardware's, not
// the M = 1 code order (checked against the oracle by tolerance).
//
// Y^T[n][m] = sum_k W[n][k] * X[m][k] with W[n][k] = v[n][k] * s[n][g(k)].
// For int2, v in {-2,-1,0,1}, so v * s is exact in fp16 and the weight tile
// can be fed to a kind::f16 MMA without any rounding of the weights; the
// fp32 accumulator lives in tensor memory.
//
// One CTA computes a 128-row x MT-token tile (MT = 64 or 128) over a K range
// (split-K when there are fewer row tiles than SMs; partial tiles are added
// into y with fp32 reductions).  Warps 0..3 stream the packed codes and the
// activations, decode the weights into fp16 and write both operands into a
// ring of shared-memory stages in the 128-byte-swizzled K-major layout; warp
// 4 allocates the accumulator in tensor memory and issues tcgen05.mma (M=128,
// N=MT, K=16; four per 64-wide K slab) from one thread, releasing each stage
// with tcgen05.commit on the stage's mbarrier.  The epilogue reads the
// accumulator back with tcgen05.ld (warp w owns TMEM lanes 32w..32w+31, i.e.
// weight rows 32w..32w+31 of the tile).
//
// Inside every 16-code word the k order in shared memory is permuted the
// same way for both operands (position 2i holds code i, position 2i+1 holds
// code i+8): a dot product does not depend on the order of its terms, and
// this order is the one in which the half2 decode yields the codes.
#include "qmv_internal.cuh"

namespace qmv {

// This file's device error word (device variables are per translation unit).
__device__ int g_tc_error = 0;

namespace {

constexpr uint32_t TC_SPIN = 1u << 22;
constexpr int ERR_TC_TIMEOUT = 16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void tc_mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void tc_mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool tc_mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __noinline__ bool tc_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < TC_SPIN; ++i) {
    if (tc_mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (i > 16) __nanosleep(100);
  }
  *abort_flag = 1;
  atomicCAS(&g_tc_error, 0, ERR_TC_TIMEOUT);
  return false;
}

// 64-bit shared-memory matrix descriptor: K-major operand, 128-byte swizzle,
// rows of 128 bytes stacked in 1024-byte groups of 8 (SBO = 1024 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
  d |= (uint64_t)(16u >> 4) << 16;                   // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset
  d |= (uint64_t)1 << 46;                            // descriptor version
  d |= (uint64_t)2 << 61;                            // 128-byte swizzle
  return d;
}

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
}

}  // namespace

struct TcArgs {
  const uint32_t* codes;   // int2 words [N][K/16]
  const __half* scales;    // [N][G]
  const __half* x;         // [M][K]
  float* y;                // [M][N] fp32 (reduced into when split > 1)
  __half* y16;             // [M][N] fp16 output (only without split)
  int N, K, G, M, perrow;
  int slabs_per_split;     // 64-wide K slabs per CTA
  int split;               // gridDim.y
};

template <int MT, int NST>
__global__ void __launch_bounds__(160, 1) tc_gemm_kernel(TcArgs a) {
  constexpr int A_BYTES = 128 * 128;              // 128 rows x 64 fp16
  constexpr int B_BYTES = MT * 128;               // MT tokens x 64 fp16
  constexpr int STAGE = A_BYTES + B_BYTES;
  constexpr uint32_t IDESC = (1u << 4)               // D = f32
                             | ((uint32_t)(MT >> 3) << 17)  // N
                             | ((uint32_t)(128 >> 4) << 24);  // M
  extern __shared__ unsigned char tc_smem_raw[];
  // 1024-byte aligned tiles (the swizzle pattern is keyed to address bits 7..9)
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  unsigned char* tiles = tc_smem_raw + pad;
  unsigned char* ctrl = tiles + NST * STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + NST;
  uint64_t* done = empty + NST;
  volatile int* abort_f = reinterpret_cast<volatile int*>(done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * 128;
  const int slab0 = blockIdx.y * a.slabs_per_split;
  const int nslab_total = a.K / 64;
  const int nslab = min(a.slabs_per_split, nslab_total - slab0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      tc_mbar_init(&full[s], 128);
      tc_mbar_init(&empty[s], 1);
    }
    tc_mbar_init(done, 1);
    *abort_f = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"((uint32_t)MT)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      for (int i = 0; i < nslab; ++i) {
        const int s = i % NST;
        if (!tc_wait(&full[s], (i / NST) & 1, abort_f)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t abase = smem_u32(tiles + s * STAGE);
        const uint32_t bbase = abase + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_desc(abase + 32 * kk);
          const uint64_t bd = sw128_desc(bbase + 32 * kk);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\t"
              "setp.ne.u32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(IDESC), "r"(acc)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_u32(&empty[s]))
            : "memory");
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_u32(done))
          : "memory");
    }
  } else {
    // -------------------------------------- producers (128 threads) ------
    const int tid = threadIdx.x;     // weight row of the tile; token for B
    const int64_t row = n0 + tid;
    const bool row_ok = row < a.N;
    const int wpr = a.K / 16;        // words per row
    for (int i = 0; i < nslab; ++i) {
      const int s = i % NST;
      const int slab = slab0 + i;
      // operands for this slab (loaded before waiting for the stage)
      uint4 cw = make_uint4(0u, 0u, 0u, 0u);
      uint32_t sc2 = 0u;
      if (row_ok) {
        cw = __ldg(reinterpret_cast<const uint4*>(a.codes + row * wpr + slab * 4));
        if (a.perrow) {
          const uint32_t sh = (uint32_t)__half_as_ushort(__ldg(a.scales + row));
          sc2 = sh | (sh << 16);
        } else {
          sc2 = __ldg(reinterpret_cast<const unsigned int*>(a.scales + row * a.G + slab * 2));
        }
      }
      uint4 xv[8];
      const bool tok_ok = tid < MT && tid < a.M;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        xv[c] = tok_ok ? __ldg(reinterpret_cast<const uint4*>(a.x + (int64_t)tid * a.K + slab * 64 + 8 * c))
                       : make_uint4(0u, 0u, 0u, 0u);
      if (i >= NST && !tc_wait(&empty[s], ((i / NST) - 1) & 1, abort_f)) break;
      unsigned char* A = tiles + s * STAGE;
      unsigned char* B = A + A_BYTES;
      // A: 4 words = 64 codes; word wi covers k = 16 wi .. 16 wi + 15 (two chunks)
      const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const __half2 s2 = u32_as_h2((blk == 0) ? ((sc2 & 0xFFFFu) | (sc2 << 16))
                                                : ((sc2 >> 16) | (sc2 & 0xFFFF0000u)));
#pragma unroll
        for (int wj = 0; wj < 2; ++wj) {
          const int wi = 2 * blk + wj;
          __half2 vp[8];
          decode_word<2>(words[wi], vp);
          uint32_t o[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const __half2 w2 = __hmul2(vp[p], s2);       // exact: v in {-2..1}
            o[p] = *reinterpret_cast<const uint32_t*>(&w2);
          }
          *reinterpret_cast<uint4*>(A + sw128_off(tid, 2 * wi)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(A + sw128_off(tid, 2 * wi + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      // B: token tid, same permutation inside each 16-element word
      if (tid < MT) {
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          const uint4 lo = xv[2 * wi], hi = xv[2 * wi + 1];   // x_0..7, x_8..15 of the word
          const uint32_t L[4] = {lo.x, lo.y, lo.z, lo.w}, H[4] = {hi.x, hi.y, hi.z, hi.w};
          uint32_t o[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o[2 * j] = __byte_perm(L[j], H[j], 0x5410);      // (x_2j, x_8+2j)
            o[2 * j + 1] = __byte_perm(L[j], H[j], 0x7632);  // (x_2j+1, x_9+2j)
          }
          *reinterpret_cast<uint4*>(B + sw128_off(tid, 2 * wi)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(B + sw128_off(tid, 2 * wi + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_mbar_arrive(&full[s]);
    }

    // --------------------------------------------------------- epilogue --
    if (tc_wait(done, 0, abort_f)) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int r = 32 * warp + lane;
      const int64_t n = n0 + r;
#pragma unroll 1
      for (int c0 = 0; c0 < MT; c0 += 16) {
        uint32_t v[16];
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
            "%11, %12, %13, %14, %15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
              "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(taddr)
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (n < a.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = c0 + j;
            if (m < a.M) {
              const float f = __uint_as_float(v[j]);
              const int64_t o = (int64_t)m * a.N + n;
              if (a.split > 1)
                atomicAdd(a.y + o, f);
              else if (a.y16)
                a.y16[o] = __float2half_rn(f);
              else
                a.y[o] = f;
            }
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 4) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)MT)
                 : "memory");
  }
}

template <int MT, int NST>
static int run_tc(const TcArgs& a0, int tiles, cudaStream_t s, cudaError_t* err) {
  constexpr int STAGE = 128 * 128 + MT * 128;
  const size_t smem = 1024 + (size_t)NST * STAGE + 256;
  static thread_local int set_dev = -1;
  auto kern = tc_gemm_kernel<MT, NST>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  if (set_dev != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
    set_dev = dev;
  }
  TcArgs a = a0;
  const int nslab = a.K / 64;
  const int sms = dev_info().sms;
  int split = 1;
  if (a.y16 == nullptr) {
    while (tiles * split * 2 <= sms && nslab / (split * 2) >= 8) split *= 2;
  }
  a.split = split;
  a.slabs_per_split = (nslab + split - 1) / split;
  if (split > 1) {
    e = cudaMemsetAsync(a.y, 0, (size_t)a.M * a.N * sizeof(float), s);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  }
  kern<<<dim3(tiles, split), 160, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

int read_tc_error(int clear, int* out) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_tc_error, &z, sizeof(int));
    if (e != cudaSuccess) return (int)e;
  }
  *out = v;
  return 0;
}

// M in 33 .. 128 token columns, int2 weights; y fp32 or fp16.
int launch_tc_gemm(const GemvArgs& g, int bits, cudaStream_t s, cudaError_t* err) {
  if (bits != 2 || g.fused || g.M < 1 || g.M > 128 || g.K % 64 != 0) return QMV_ERR_UNSUPPORTED;
  TcArgs a;
  a.codes = reinterpret_cast<const uint32_t*>(g.codes);
  a.scales = g.scales;
  a.x = g.x;
  a.y = g.y_f16 ? nullptr : reinterpret_cast<float*>(g.y);
  a.y16 = g.y_f16 ? reinterpret_cast<__half*>(g.y) : nullptr;
  a.N = g.N;
  a.K = g.K;
  a.G = g.G;
  a.M = g.M;
  a.perrow = g.perrow;
  a.split = 1;
  a.slabs_per_split = g.K / 64;
  const int tiles = (g.N + 127) / 128;
  if (g.M <= 64) return run_tc<64, 4>(a, tiles, s, err);
  return run_tc<128, 3>(a, tiles, s, err);
}

}  // namespace qmv
