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
// (split-K when there are fewer row tiles than SMs: with two splits and fp32
// output the partial tiles are added into the zeroed y with fp32 atomics,
// which is order-independent for two terms (0 + a + b == 0 + b + a); otherwise
// each split stores its partial tile to a stream-ordered fp32 scratch and a
// second kernel adds the splits in split order, so the result never depends
// on CTA timing).  A pipeline stage carries KSUB 64-code slabs (4 for MT =
// 64, 2 for MT = 128): one hand-off between the roles per 64*KSUB codes.
// The 16 decode warps form groups that take stages in turn, so several
// stages' decodes are in flight at once: four groups of four warps at
// MT = 128, two groups of eight at MT = 64 (a group's parity wait for the
// reuse of an A stage needs groups <= A stages).
// Roles:
//   warp 16 (one thread): TMA of the packed codes (64-byte swizzle) and
//     scales of the tile, 4 K-slabs (256 codes) at a time, into a ring of
//     raw stages.
//   warp 18 (one thread): TMA of the activation sub-tiles of each stage's
//     slabs straight into the MMA operand stage, with a 128-byte-swizzle
//     tensor map (the K-major layout the MMA reads).
//   warps 0..15: decode.  Thread t of a group takes row t % 128 of every
//     slab of its stage, both 32-code blocks with four-warp groups, block
//     (t / 128) % 2 with eight-warp groups: it turns them into fp16 weights
//     w = v*s (half2 magic decode, re-paired into natural k order) and stores
//     them straight into tensor memory, the MMA's A operand (row = lane of
//     its warp's lane quarter, two weights a column), so the weights never
//     pass through shared memory.  At the end they are the epilogue:
//     tcgen05.ld of their TMEM lane quarter, a quarter of the tile's columns
//     each.
//   warp 17 (one thread): allocates tensor memory (the accumulator and the
//     A stages) and issues tcgen05.mma (A from tensor memory, B from shared
//     memory; M=128, N=MT, K=16; four per slab), releasing each stage with
//     tcgen05.commit on its mbarrier.
// Every wait is bounded; a wait that runs out records an error code in this
// file's device error word and the CTA winds down.
#include <cuda.h>

#include "qmv_internal.cuh"

namespace qmv {

// This file's device error word (device variables are per translation unit).
__device__ int g_tc_error = 0;

namespace {

constexpr uint32_t TC_SPIN = 1u << 22;
constexpr int ERR_TC_TIMEOUT = 16;
constexpr int RS = 4;          // K slabs per raw stage (256 codes)
constexpr int TC_TMEM_COLS = 512;   // tensor-memory columns a CTA allocates (accumulator + A stages)
constexpr int NDEC = 16;       // decode (and epilogue) warps
constexpr int W_RAW = NDEC, W_MMA = NDEC + 1, W_B = NDEC + 2;   // role warps
constexpr int TC_THREADS = 32 * (NDEC + 3);
constexpr int RAW_CODES = 128 * RS * 16;   // bytes of codes per raw stage
constexpr int RAW_SC = 128 * RS * 4;       // bytes of scales per raw stage
constexpr int RAW_BYTES = RAW_CODES + RAW_SC;
static_assert(RS * 16 == 64, "a row of a raw stage's codes is one 64-byte swizzle span");
static_assert(RAW_BYTES % 1024 == 0, "raw stages keep the swizzle's alignment");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void tc_mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void tc_mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void tc_mbar_arrive_tx(uint64_t* b, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(tx)
               : "memory");
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
// bounded wait that ignores the abort flag (lets issued copies land)
__device__ __noinline__ void tc_drain(uint64_t* b, uint32_t parity) {
  for (uint32_t i = 0; i < TC_SPIN; ++i) {
    if (tc_mbar_try(b, parity)) return;
    __nanosleep(100);
  }
  atomicCAS(&g_tc_error, 0, ERR_TC_TIMEOUT);
}

// A 2-D tensor copy global -> shared with an L2 cache policy (from
// createpolicy): the streamed
// weights are marked evict-first and the activation tiles, which every row
// tile re-reads, evict-last, so the weight stream does not push the
// activations out of L2.
__device__ __forceinline__ void tc_tma2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
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

// Raw-ring depth (raw stages of RS slabs) of the two tile shapes.
constexpr int TC_RS_M64 = 3, TC_RS_M128 = 3;

// How K is split across CTAs: split K to balance the waves; the time is
// about ceil(tiles * split / SMs) CTA-slots of 1/split of the work each; the
// smallest such time wins (at least 8 slabs per split), the smaller split on
// a tie.  A split that needs the scratch and the reduction kernel (fp16
// output, or more than two splits) must save a third of the time: the
// partial tiles' round trip costs about 15 us on a 28672 x 4096 M = 128 tile
// set (two splits, fp16: 94 us against 79 us for fp32 atomics).  Each split
// takes whole raw stages, so every box starts on a 16-byte boundary.  Two
// splits with fp32 output add into the zeroed output with atomics.
struct TcSplit {
  int split, slabs_per_split;
  bool atomics;
};
static TcSplit tc_split(int tiles, int K, bool y16, int RS) {
  const int nslab = K / 64;
  const int sms = dev_info().sms;
  int split = 1;
  double best = 1e30;
  for (int sp = 1; sp <= 8 && nslab / sp >= 8; ++sp) {
    double t = (double)((tiles * sp + sms - 1) / sms) / sp;
    const bool scratch = sp > 1 && (sp > 2 || y16);
    if (scratch) t *= 1.5;
    if (t < best - 1e-9) {
      best = t;
      split = sp;
    }
  }
  int sps = (((nslab + split - 1) / split) + RS - 1) / RS * RS;
  while (split > 1 && (split - 1) * sps >= nslab) --split;
  return TcSplit{split, sps, split == 2 && !y16};
}

struct TcArgs {
  const __half* scales;    // [N][G] (one scale per row when perrow)
  float* y;                // [M][N] fp32 output (or null)
  __half* y16;             // [M][N] fp16 output (or null)
  float* part;             // [split][M][N] fp32 partial tiles (split > 1, unless atomics)
  int N, K, G, M, perrow;
  int slabs_per_split;     // 64-wide K slabs per CTA
  int split;               // gridDim.y
};

// KSUB 64-code slabs per pipeline stage: each stage holds KSUB weight
// sub-tiles (128 rows x 64 fp16 each) and KSUB activation sub-tiles (MT x 64
// fp16 each), so the roles hand a stage over once per 64*KSUB codes.
template <int MT, int NST, int NRAW, int KSUB, int GW>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(TcArgs a, const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_scales, const __grid_constant__ CUtensorMap tm_x) {
  // the decoded weights (the MMA's A operand, 128 rows x 64 fp16 a slab) go
  // to tensor memory: 32 columns a slab after the MT accumulator columns;
  // only the activations (B) are staged in shared memory
  constexpr int B_SUB = MT * 128;                 // MT tokens x 64 fp16
  constexpr int B_BYTES = KSUB * B_SUB;
  constexpr int STAGE = B_BYTES;
  constexpr uint32_t A_COL = MT;                  // first tensor-memory column of the A stages
  static_assert(MT + NST * KSUB * 32 <= TC_TMEM_COLS, "A stages fit tensor memory");
  static_assert(RS % KSUB == 0, "a stage's slabs come from one raw stage");
  // decode warps are at most NST - 1 stages apart; the raw stages they read
  // must then differ by less than two trips round the raw ring, or a parity
  // wait could match an older phase
  static_assert((NST - 1) * KSUB / RS + 1 < 2 * NRAW, "raw ring too shallow for the decode spread");
  // a decode group's wait for the MMAs of stage i - NST (A stage reuse) is a
  // parity wait, which tells a phase only from the one before it: the
  // group's previous wait (stage i - NGRP - NST) must already imply the
  // completion of stage i - 2 * NST, i.e. NGRP <= NST
  static_assert(GW == 4 || GW == 8, "decode groups of 4 warps (both blocks a thread) or 8 (one)");
  constexpr int NGRP = NDEC / GW;   // decode groups, each taking every NGRP-th stage
  static_assert(NGRP <= NST, "more decode groups than A stages: the A-stage parity waits could alias");
  // likewise a decode warp's raw-stage wait: when it waits for raw stage j
  // it has seen the MMAs of stage i - NST complete, so every raw stage up to
  // (i - NST) * KSUB / RS has landed; raw stage j - NRAW (the previous phase
  // of the same buffer) must be among them
  static_assert(NST * KSUB <= NRAW * RS, "raw ring too shallow for the A ring: raw parity waits could alias");
  constexpr uint32_t IDESC = (1u << 4)               // D = f32
                             | ((uint32_t)(MT >> 3) << 17)  // N
                             | ((uint32_t)(128 >> 4) << 24);  // M
  extern __shared__ unsigned char tc_smem_raw[];
  // 1024-byte aligned tiles (the swizzle pattern is keyed to address bits 7..9)
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  unsigned char* tiles = tc_smem_raw + pad;
  unsigned char* rawbuf = tiles + NST * STAGE;             // NRAW x RAW_BYTES
  unsigned char* ctrl = rawbuf + NRAW * RAW_BYTES;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* b_full = a_full + NST;
  uint64_t* empty = b_full + NST;
  uint64_t* raw_full = empty + NST;
  uint64_t* raw_empty = raw_full + NRAW;
  uint64_t* done = raw_empty + NRAW;
  volatile int* abort_f = reinterpret_cast<volatile int*>(done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * 128;
  const int slab0 = blockIdx.y * a.slabs_per_split;
  const int nslab = min(a.slabs_per_split, a.K / 64 - slab0);   // a multiple of RS
  const int nstage = nslab / KSUB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      tc_mbar_init(&a_full[s], NDEC / NGRP);
      tc_mbar_init(&b_full[s], 1);
      tc_mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < NRAW; ++r) {
      tc_mbar_init(&raw_full[r], 1);
      // the decode groups whose stages read a raw stage each arrive once
      tc_mbar_init(&raw_empty[r], (NDEC / NGRP) * (RS / KSUB < NGRP ? RS / KSUB : NGRP));
    }
    tc_mbar_init(done, 1);
    *abort_f = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"((uint32_t)TC_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == W_RAW) {
    // ------------------------------------------- TMA: packed codes/scales --
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nslab; i += RS) {
        const int j = i / RS, rr = j % NRAW;
        if (j >= NRAW && !tc_wait(&raw_empty[rr], ((j / NRAW) - 1) & 1, abort_f)) break;
        unsigned char* rb = rawbuf + rr * RAW_BYTES;
        tc_mbar_arrive_tx(&raw_full[rr], a.perrow ? RAW_CODES : RAW_BYTES);
        tc_tma2d_hint(rb, &tm_codes, (slab0 + i) * 4, n0, &raw_full[rr], pol);
        if (!a.perrow) tc_tma2d_hint(rb + RAW_CODES, &tm_scales, (slab0 + i) * 2, n0, &raw_full[rr], pol);
        ++issued;
      }
      for (int j = (issued > NRAW ? issued - NRAW : 0); j < issued; ++j)
        tc_drain(&raw_full[j % NRAW], (j / NRAW) & 1);
    }
  } else if (warp == W_B) {
    // --------------------------------------------- TMA: activation tiles --
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      int issued = 0;
      for (int i = 0; i < nstage; ++i) {
        const int s = i % NST;
        if (i >= NST && !tc_wait(&empty[s], ((i / NST) - 1) & 1, abort_f)) break;
        tc_mbar_arrive_tx(&b_full[s], B_BYTES);
#pragma unroll
        for (int u = 0; u < KSUB; ++u)
          tc_tma2d_hint(tiles + s * STAGE + u * B_SUB, &tm_x, (slab0 + i * KSUB + u) * 64, 0, &b_full[s], pol);
        ++issued;
      }
      for (int i = (issued > NST ? issued - NST : 0); i < issued; ++i)
        tc_drain(&b_full[i % NST], (i / NST) & 1);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      for (int i = 0; i < nstage; ++i) {
        const int s = i % NST;
        if (!tc_wait(&a_full[s], (i / NST) & 1, abort_f)) break;
        if (!tc_wait(&b_full[s], (i / NST) & 1, abort_f)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t bbase = smem_u32(tiles + s * STAGE);
        const uint32_t acol = tmem + A_COL + (uint32_t)(s * KSUB * 32);
#pragma unroll
        for (int kk = 0; kk < 4 * KSUB; ++kk) {
          // A: 8 tensor-memory columns (16 fp16 a row) per K = 16 step
          const uint32_t at = acol + (uint32_t)(kk * 8);
          const uint64_t bd = sw128_desc(bbase + (kk >> 2) * B_SUB + 32 * (kk & 3));
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\t"
              "setp.ne.u32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
              "r"(at), "l"(bd), "r"(IDESC), "r"(acc)
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
    // ------------------------ decode (NGRP groups of GW warps, by stage) --
    // group g decodes stages g, g + NGRP, ...: the groups' stages are in
    // flight at once, each group's chain (raw wait, decode, tensor-memory
    // store, its completion, the hand-off) overlapping the others'.  With
    // 8-warp groups a thread decodes one 32-code block of its row of a slab,
    // with 4-warp groups both.
    const int grp = warp / GW;
    const int row = threadIdx.x & 127;        // weight row of the tile
    const int blk = GW == 8 ? (threadIdx.x >> 7) & 1 : 0;   // first 32-code block of the slab
    constexpr int NB = GW == 8 ? 1 : 2;       // blocks a thread decodes
    int waited = -1;                          // the last raw stage this thread waited for
    const uint32_t prs = a.perrow && n0 + row < a.N
                             ? (uint32_t)__half_as_ushort(__ldg(a.scales + n0 + row))
                             : 0u;
    for (int i = grp; i < nstage; i += NGRP) {
      const int s = i % NST;
      // every wait's outcome is made warp-uniform: the warp-wide tensor-memory
      // stores below must be reached by all of its lanes or by none
      if (__any_sync(0xFFFFFFFFu, i >= NST && !tc_wait(&empty[s], ((i / NST) - 1) & 1, abort_f))) break;
      // the MMAs that read this A stage have completed (their commit)
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      bool ok = true;
#pragma unroll 1
      for (int u = 0; u < KSUB; ++u) {
        const int sl = i * KSUB + u;   // slab
        const int j = sl / RS, rr = j % NRAW, sub = sl % RS;
        if (j != waited) {
          if (__any_sync(0xFFFFFFFFu, !tc_wait(&raw_full[rr], (j / NRAW) & 1, abort_f))) {
            ok = false;
            break;
          }
          waited = j;
        }
        const unsigned char* rb = rawbuf + rr * RAW_BYTES;
        // the codes arrive 64-byte swizzled (offset bits 4..5 XOR bits 7..8):
        // a thread's 8 (one block) or 16 bytes (both) of its 64-byte row
        const uint32_t co = (uint32_t)(row * (RS * 16) + sub * 16 + blk * 8);
        const unsigned char* cp = rb + (co ^ (((co >> 7) & 3u) << 4));
        uint32_t words[2 * NB], sbb;
        if constexpr (NB == 1) {
          const uint2 cw = *reinterpret_cast<const uint2*>(cp);
          words[0] = cw.x;
          words[1] = cw.y;
          sbb = a.perrow ? prs
                         : *reinterpret_cast<const uint16_t*>(rb + RAW_CODES + row * (RS * 4) + sub * 4 + blk * 2);
        } else {
          const uint4 cw = *reinterpret_cast<const uint4*>(cp);
          words[0] = cw.x;
          words[1] = cw.y;
          words[2] = cw.z;
          words[3] = cw.w;
          // block 0's scale in the low half, block 1's in the high half
          sbb = a.perrow ? (prs | (prs << 16))
                         : *reinterpret_cast<const uint32_t*>(rb + RAW_CODES + row * (RS * 4) + sub * 4);
        }
        uint32_t o[16 * NB];   // the blocks' weights in k order, two fp16 a word
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const uint32_t sb = (sbb >> (16 * b)) & 0xFFFFu;
          const __half2 s2 = u32_as_h2(sb | (sb << 16));
#pragma unroll
          for (int wj = 0; wj < 2; ++wj) {
            __half2 vp[8];
            decode_word<2>(words[2 * b + wj], vp);   // vp[i] = (v_i, v_{i+8})
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              // natural order: (v_2q, v_2q+1) and (v_8+2q, v_9+2q)
              const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&vp[2 * q]);
              const uint32_t a1 = *reinterpret_cast<const uint32_t*>(&vp[2 * q + 1]);
              const __half2 lo = __hmul2(u32_as_h2(__byte_perm(a0, a1, 0x5410)), s2);   // exact
              const __half2 hi = __hmul2(u32_as_h2(__byte_perm(a0, a1, 0x7632)), s2);
              o[16 * b + 8 * wj + q] = *reinterpret_cast<const uint32_t*>(&lo);
              o[16 * b + 8 * wj + 4 + q] = *reinterpret_cast<const uint32_t*>(&hi);
            }
          }
        }
        // row `row` is tensor-memory lane `row` (this warp's lane quarter);
        // a block's 16 words go to its 16 columns of the slab
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + A_COL +
                               (uint32_t)((s * KSUB + u) * 32 + blk * 16);
        if constexpr (NB == 1) {
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
              "%13, %14, %15, %16};" ::"r"(taddr),
              "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7]), "r"(o[8]),
              "r"(o[9]), "r"(o[10]), "r"(o[11]), "r"(o[12]), "r"(o[13]), "r"(o[14]), "r"(o[15])
              : "memory");
        } else {
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
              "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
              "%32};" ::"r"(taddr),
              "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7]), "r"(o[8]),
              "r"(o[9]), "r"(o[10]), "r"(o[11]), "r"(o[12]), "r"(o[13]), "r"(o[14]), "r"(o[15]), "r"(o[16]),
              "r"(o[17]), "r"(o[18]), "r"(o[19]), "r"(o[20]), "r"(o[21]), "r"(o[22]), "r"(o[23]), "r"(o[24]),
              "r"(o[25]), "r"(o[26]), "r"(o[27]), "r"(o[28]), "r"(o[29]), "r"(o[30]), "r"(o[31])
              : "memory");
        }
      }
      if (!ok) break;
      // the stores are complete before the MMA thread may read them
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        tc_mbar_arrive(&a_full[s]);
        // this group is done with a raw stage when its next stage reads another
        const int j = (i * KSUB) / RS;
        if (i + NGRP >= nstage || ((i + NGRP) * KSUB) / RS != j) tc_mbar_arrive(&raw_empty[j % NRAW]);
      }
    }

    // --------------------------------------------------------- epilogue --
    // warp w reads TMEM lanes 32*(w%4) .. +31 (its lane quarter), columns of
    // its half of the tile's tokens
    if (nstage > 0 && __all_sync(0xFFFFFFFFu, tc_wait(done, 0, abort_f))) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int q4 = warp & 3;
      const int r = 32 * q4 + lane;
      const int64_t n = (int64_t)n0 + r;
      const int cbeg = (warp >> 2) * (MT / (NDEC / 4)), cend = cbeg + MT / (NDEC / 4);
#pragma unroll 1
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        uint32_t v[16];
        const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)c0;
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
          for (int q = 0; q < 16; ++q) {
            const int m = c0 + q;
            if (m < a.M) {
              const float f = __uint_as_float(v[q]);
              const int64_t o = (int64_t)m * a.N + n;
              if (a.part)
                a.part[(int64_t)blockIdx.y * a.M * a.N + o] = f;
              else if (a.split > 1)
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
  if (warp == W_MMA) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"((uint32_t)TC_TMEM_COLS)
                 : "memory");
  }
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

// ------------------------------------------------------------- launcher --

typedef CUresult (*TcEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                               const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                               const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static TcEncodeFn tc_encode_fn() {
  static TcEncodeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (TcEncodeFn) nullptr;
    return (TcEncodeFn)f;
  }();
  return fn;
}

// Split-K reduction: y[i] = sum of the splits' partials in split order (fp32
// adds), stored as fp32 or as the RNE fp16 of that sum.
__global__ void tc_reduce_kernel(const float* __restrict__ part, int split, int64_t total, float* y,
                                 __half* y16) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  float v = part[i];
  for (int sp = 1; sp < split; ++sp) v = __fadd_rn(v, part[(int64_t)sp * total + i]);
  if (y16)
    y16[i] = __float2half_rn(v);
  else
    y[i] = v;
}

// A 2-D tensor map (also used by the M-column pipeline tiles).
bool enc2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  TcEncodeFn enc = tc_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MT, int NST, int NRAW, int KSUB, int GW>
static int run_tc(const TcArgs& a0, const GemvArgs& g, int tiles, cudaStream_t s, cudaError_t* err) {
  constexpr int STAGE = KSUB * MT * 128;
  // at least 116 KB, so that one CTA runs per SM: each allocates all the
  // tensor-memory columns it uses (accumulator + A stages, 512)
  size_t smem = 1024 + (size_t)NST * STAGE + (size_t)NRAW * RAW_BYTES + 256;
  if (smem < 116 * 1024) smem = 116 * 1024;
  static thread_local int set_dev = -1;
  auto kern = tc_gemm_kernel<MT, NST, NRAW, KSUB, GW>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  if (set_dev != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
    set_dev = dev;
  }
  // tensor maps: codes as UINT32 [N][K/16] (box 4*RS x 128), scales as UINT16
  // [N][K/32] (box 2*RS x 128), activations as FP16 [M][K] (box 64 x MT,
  // 128-byte swizzle = the MMA's K-major operand layout).  Rows past N or M
  // and columns past K are zero-filled.
  CUtensorMap tmc, tms, tmx;
  if (!enc2d(&tmc, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.codes, (uint64_t)g.K / 16, (uint64_t)g.N,
             (uint64_t)g.K / 4, 4 * RS, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return QMV_ERR_UNSUPPORTED;
  if (g.perrow) {
    tms = tmc;   // unused
  } else if (!enc2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.scales, (uint64_t)g.G, (uint64_t)g.N,
                    (uint64_t)g.G * 2, 2 * RS, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    return QMV_ERR_UNSUPPORTED;
  }
  if (!enc2d(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.x, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.K * 2,
             64, MT, CU_TENSOR_MAP_SWIZZLE_128B))
    return QMV_ERR_UNSUPPORTED;
  TcArgs a = a0;
  const TcSplit sp = tc_split(tiles, a.K, a.y16 != nullptr, RS);
  a.split = sp.split;
  a.slabs_per_split = sp.slabs_per_split;
  a.part = nullptr;
  const int64_t total = (int64_t)a.M * a.N;
  if (sp.atomics) {
    e = cudaMemsetAsync(a.y, 0, (size_t)total * sizeof(float), s);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  } else if (sp.split > 1) {
    // the partial tiles go to the caller's workspace (checked by the ABI)
    if (!g.ws || g.ws_bytes < (size_t)sp.split * total * sizeof(float)) return QMV_ERR_WORKSPACE;
    a.part = reinterpret_cast<float*>(g.ws);
  }
  kern<<<dim3(tiles, sp.split), TC_THREADS, smem, s>>>(a, tmc, tms, tmx);
  e = cudaGetLastError();
  if (a.part && e == cudaSuccess) {
    tc_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(a.part, sp.split, total, a.y, a.y16);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

// Scratch of a launch of up to 128 columns: split-K partial tiles in fp32
// when the chosen split needs the reduction kernel.
size_t tc_workspace_bytes(int M, int N, int K, bool y_f16) {
  if (M < 1 || K % 256 != 0) return 0;
  const int m = M < 128 ? M : 128;
  const int tiles = (N + 127) / 128;
  const TcSplit sp = tc_split(tiles, K, y_f16, RS);
  if (sp.split <= 1 || sp.atomics) return 0;
  return (size_t)sp.split * (size_t)m * (size_t)N * sizeof(float);
}

// M in 1 .. 128 token columns, int2 weights; y fp32 or fp16.
int launch_tc_gemm(const GemvArgs& g, int bits, cudaStream_t s, cudaError_t* err) {
  if (bits != 2 || g.fused || g.M < 1 || g.M > 128 || g.K % 256 != 0) return QMV_ERR_UNSUPPORTED;
  TcArgs a;
  a.scales = g.scales;
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
  // stages of several 64-code slabs (smaller stages measured slower): four
  // slabs for M <= 64, two for M = 128.  Only the activation tiles sit in
  // shared memory (32 KB a stage), the decoded weights in tensor memory, so
  // there are three stages at M <= 64 and six at M = 128 (the tensor-memory
  // columns' limit), and three raw stages of codes and scales
  if (g.M <= 64) return run_tc<64, 3, TC_RS_M64, 4, 8>(a, g, tiles, s, err);
  return run_tc<128, 6, TC_RS_M128, 2, 4>(a, g, tiles, s, err);
}

}  // namespace qmv
