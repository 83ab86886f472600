// qmv_tma.cu -- the M = 1 matvec as a warp-specialised pipeline (GB300).
//
// What it computes is exactly what the CUDA-core kernels compute (and the
// oracle): per output row, each 32-code block summed serially in k in fp32
// with exact products, scaled (group 32), and folded serially over blocks
// ("Gemma4 raw-Metal loop on A19", section "What moved the needle": int2 at
// 16 codes per word, exact products, fp32 in code order; the residual-add +
// RMSNorm fold into the matvec prologue).
//
// How:
//   * Rows are processed in groups of R rows.  A group's codes (and its
//     group-32 scales) are contiguous in memory, so one producer thread moves
//     each group into a ring of NS shared-memory stages with two
//     cp.async.bulk copies completing on the stage's "full" mbarrier.  The
//     producer runs ahead of the math by up to NS groups (tens of KB in
//     flight per SM) and starts before the prologue, since weights do not
//     depend on the activations.
//   * Compute warps: thread t owns one 64-code item (two 32-code blocks) of
//     RP rows in parallel, U rows after another, and keeps that item's 64
//     activations in registers as fp32 pairs (y_k, y_{32+k}).  A code field
//     is turned into fp32 exactly by one LOP3: (w & (mask << o)) | 0x4B000000
//     = 2^23 + u*2^o (every field is first brought below bit 16: the low and
//     high halves of a word use the same o).  One packed sub.rn.f32x2 maps
//     the pair (block 0, block 1) to v*2^o exactly, and one fma.rn.f32x2 with
//     the activations pre-scaled by 2^-o advances both blocks' serial sums
//     (y*2^-o times v*2^o is y*v exactly).  About 2 instructions per code.
//   * Block sums (scaled) go to a double-buffered fold buffer; a dedicated
//     fold warp adds them serially per row (one lane per row) and writes y,
//     so the compute warps never wait at a CTA-wide barrier.
//   * Every mbarrier wait is bounded; on timeout the kernel records an error
//     code in the device error word, stops issuing, lets its own copies land
//     and returns.
#include <cuda.h>

#include "qmv_internal.cuh"

namespace qmv {

__device__ int g_qmv_error = 0;

namespace {

constexpr int NS = 4;                      // ring stages (a power of two)
constexpr uint32_t SPIN_LIMIT = 1u << 22;  // tries per bounded wait (a backstop to the time limit)
constexpr int ERR_TIMEOUT_FULL = 1, ERR_TIMEOUT_EMPTY = 2, ERR_TIMEOUT_TFULL = 3,
              ERR_TIMEOUT_TEMPTY = 4, ERR_SMEM_ALIGN = 5;


__device__ __forceinline__ uint32_t sa(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(tx)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the warp sleeps in hardware until the
// phase completes (it wakes at once then) or the hint elapses
__device__ __forceinline__ bool mbar_try_hint(uint64_t* b, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint32_t WAIT_HINT_NS = 20000;            // one suspended try
constexpr uint64_t WAIT_LIMIT_NS = 500000000ull;    // give up after 0.5 s

// Bounded wait.  Returns false (after setting the CTA's abort flag and the
// device error word) if the phase does not complete within WAIT_LIMIT_NS (or
// SPIN_LIMIT tries), or soon after another warp of the CTA has aborted.
__device__ __noinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                       int code) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (mbar_try_hint(b, parity, WAIT_HINT_NS)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > WAIT_LIMIT_NS) break;
  }
  *abort_flag = 1;
  atomicCAS(&g_qmv_error, 0, code);
  return false;
}

// The common case inline (one try_wait, which itself suspends the warp for a
// while), the bounded loop out of line.
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                               int code) {
  return mbar_try(b, parity) || mbar_wait(b, parity, abort_flag, code);
}

// Bounded wait that ignores the abort flag (used to let copies land).
__device__ __noinline__ void mbar_drain(uint64_t* b, uint32_t parity) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (mbar_try_hint(b, parity, WAIT_HINT_NS)) return;
    if (global_ns() - t0 > WAIT_LIMIT_NS) break;
  }
  atomicCAS(&g_qmv_error, 0, ERR_TIMEOUT_FULL);
}

// 2-D tiled tensor copy global -> shared (box given by the tensor map),
// completing on `bar`.  x is the innermost coordinate (in elements).
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          sa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(sa(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The activation table: per 64-code item c, 32 steps of fp32 pairs at
// y2f[2*(YS*c + step) + lane].  The item stride YS = 34 pairs (272 bytes)
// keeps 16-byte loads of two consecutive steps aligned and spreads the
// threads of a warp (consecutive items) over all banks; within an item the
// steps are immediate offsets.
constexpr int YS = 34;

// Store 8 consecutive fp16 activations starting at element e0 (a multiple of
// 8; element 64*c + 32*h + k) into the table.  Exact form: y * 2^-o(k), step
// k holds (block 0, block 1) code k.  Folded form: y * 2^(FOLD_E - o(k)),
// step 16*blk + CPW*p + j holds (code j of word 2p, of word 2p+1) of block
// blk.
template <int BITS, bool EXACT>
__device__ __forceinline__ void store_y8(float* y2f, int e0, const uint32_t (&h8)[4]) {
  constexpr int CPW = 32 / BITS, HALF = CPW / 2;
  const int c = e0 >> 6, h = (e0 >> 5) & 1, k0 = e0 & 31;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int k = k0 + e;
    const int j = k % CPW, o = BITS * (j % HALF);
    const __half2 v = u32_as_h2(h8[e >> 1]);
    const float f = (e & 1) ? __high2float(v) : __low2float(v);
    if (EXACT) {
      y2f[2 * (YS * c + k) + h] = __fmul_rn(f, pow2f(-o));
    } else {
      const int wi = k / CPW, step = 16 * h + CPW * (wi >> 1) + j;
      y2f[2 * (YS * c + step) + (wi & 1)] = __fmul_rn(f, pow2f(FOLD_E - o));
    }
  }
}

// Both blocks of one 64-code item, for U rows at once.  w[u][0 .. 2*WPB-1]:
// words of block 0 then block 1.  yc: the item's activation pairs
// (y'_k, y'_{32+k}), two steps per 16-byte load; one pair serves all U rows.  y'_k = y_k * 2^-o(k) where o(k)
// is the bit offset the code k is decoded at, so y'_k * (v_k * 2^o(k)) =
// y_k * v_k exactly (powers of two; no underflow for fp16 inputs).  acc[u] =
// (p0, p1) are the two blocks' serial sums.  Fields in the high 16-bit half
// of a word are first shifted down by 16, so every field is masked below
// bit 16.  (Exact form; the folded form is block_dots_fold.)
template <int BITS, int U>
__device__ __forceinline__ void item_dots(const uint32_t (&w)[U][64 * BITS / 32],
                                          const u64* __restrict__ yc, u64 (&acc)[U]) {
  constexpr int CPW = 32 / BITS;   // codes per word
  constexpr int HALF = CPW / 2;    // codes per 16-bit half
  constexpr int WPB = 32 / CPW;    // words per block
  constexpr uint32_t MASK = (1u << BITS) - 1u;
#pragma unroll
  for (int wi = 0; wi < WPB; ++wi) {
    uint32_t h0[U], h1[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      h0[u] = w[u][wi] >> 16;
      h1[u] = w[u][WPB + wi] >> 16;
    }
#pragma unroll
    for (int j = 0; j < CPW; ++j) {
      const int o = BITS * (j % HALF);
      const float offf = pow2f(23) + (float)(1 << (BITS - 1 + o));
      const u64 off = pk(offf, offf);
      const ulonglong2 y2 = *reinterpret_cast<const ulonglong2*>(yc + wi * CPW + (j & ~1));
      const u64 y = (j & 1) ? y2.y : y2.x;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t a = (j < HALF) ? w[u][wi] : h0[u];
        const uint32_t b = (j < HALF) ? w[u][WPB + wi] : h1[u];
        const u64 v = decode2(a, b, MASK << o, off);
        acc[u] = ffma2(y, v, acc[u]);
      }
    }
  }
}

// Folded form, both 32-code blocks of a 64-code item for U rows: wp[u][q]
// are the item's words as 64-bit pairs (words 2q, 2q+1), so a pair's two
// fields at one offset are masked by one 64-bit AND straight into the
// register pair the paired FMA reads.  Lane 0 of acc[u][blk] sums block
// blk's even words, lane 1 its odd words, each serially in code order; the
// two blocks' chains are interleaved for independent work.  The high 16-bit
// fields come from the pair shifted right by 16 as a whole: what crosses from
// the odd word into the even word's upper half is masked off.
template <int BITS, int U>
__device__ __forceinline__ void item_dots_fold(const u64 (&wp)[U][BITS], const u64* __restrict__ yc,
                                               u64 (&acc)[U][2]) {
  constexpr int CPW = 32 / BITS, HALF = CPW / 2;
  constexpr int NP = 16 / CPW;                 // word pairs per block
  constexpr uint32_t MASK = (1u << BITS) - 1u;
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    u64 lo[U][2], hi[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        lo[u][blk] = wp[u][blk * NP + p];
        hi[u][blk] = lo[u][blk] >> 16;
      }
#pragma unroll
    for (int j = 0; j < CPW; ++j) {
      const uint32_t m = MASK << (BITS * (j % HALF));
      const u64 mm = ((u64)m << 32) | m;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const ulonglong2 y2 =
            *reinterpret_cast<const ulonglong2*>(yc + 16 * blk + CPW * p + (j & ~1));
        const u64 y = (j & 1) ? y2.y : y2.x;
#pragma unroll
        for (int u = 0; u < U; ++u)
          acc[u][blk] = ffma2(y, ((j < HALF) ? lo[u][blk] : hi[u][blk]) & mm, acc[u][blk]);
      }
    }
  }
}

}  // namespace

// Launch plan (host computes it; the kernel reads it).
//
// Rows are processed in groups of R, and each group in NSEG segments of KS
// codes (KS = K when K <= 2048, else the largest multiple of 256 up to 2048
// that divides K).  A pipeline stage holds one (group, segment): R rows x KS
// codes plus their group-32 scales.  The fold warp keeps one accumulator per
// row across the segments of a group, so the fold stays serial over all K/32
// blocks of the row while 32 rows are folded side by side.
struct TmaPlan {
  int C;             // 64-code items per row (table layout)
  int Cs;            // 64-code items per segment
  int KS, NSEG;      // codes per segment, segments per row
  int RP;            // rows in parallel (Cs*RP <= Tc)
  int R;             // rows per group = RP*U (<= 32: one fold lane per row)
  int Tc;            // compute threads (multiple of 32)
  int row_bytes;     // code bytes per row
  int seg_bytes;     // code bytes per row per segment
  int seg_sc;        // scale bytes per row per segment (0 with one scale per row)
  int sc_off;        // offset of the scales inside a stage (128-byte aligned)
  int stage_bytes;   // whole stage, a multiple of 128 bytes
  int ngroups;       // ceil(N / R)
  int y_off, ysum_off, stage_off, tbuf_off;   // shared-memory offsets (bytes)
};

__host__ __device__ inline int tma_round16(int x) { return (x + 15) & ~15; }

template <int BITS, bool PERROW, bool FUSED, bool EXACT, int U, int MAXT>
__global__ void __launch_bounds__(MAXT, (MAXT <= 320) ? 2 : 1)
    gemv_tma_kernel(GemvArgs a, TmaPlan P, const __grid_constant__ CUtensorMap tm_codes,
                    const __grid_constant__ CUtensorMap tm_scales) {
  constexpr int IW = 64 * BITS / 32;   // words per item
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  uint64_t* empty = full + NS;
  uint64_t* tfull = empty + NS;
  uint64_t* tempty = tfull + 2;
  volatile int* abort_f = reinterpret_cast<volatile int*>(sm + 96);
  float* inv_sh = reinterpret_cast<float*>(sm + 100);
  float* y2f = reinterpret_cast<float*>(sm + P.y_off);   // pairs [k][item] as fp32
  float* ysum = reinterpret_cast<float*>(sm + P.ysum_off); // folded form: 2^(b-1) * S per block
  unsigned char* stages = sm + P.stage_off;
  float* tbuf = reinterpret_cast<float*>(sm + P.tbuf_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, NB = K / 32, R = P.R;
  const int NBS = P.KS / 32;             // blocks per segment
  const int GS = NBS + 1;                // fold-buffer row stride
  const int my_groups = (blockIdx.x < (unsigned)P.ngroups)
                            ? (P.ngroups - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                            : 0;
  const int my_stages = my_groups * P.NSEG;

  // Programmatic dependent launch (a no-op when the launch did not ask for
  // it): let the next kernel in the stream be scheduled as soon as SMs free
  // up; its weight copies then overlap this kernel's tail.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // tensor copies need 128-byte aligned destinations: the dynamic shared
  // memory window starts aligned when there is no static shared memory
  if ((sa(sm) & 127u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(&g_qmv_error, 0, ERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    // consumers arrive once per warp (lane 0, after __syncwarp orders the
    // lanes' shared-memory accesses before its release)
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], P.Tc / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], P.Tc / 32);
      mbar_init(&tempty[b], 1);
    }
    *abort_f = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ------------------------------------------------------------ producer --
  if (warp == 0) {
    int issued = 0;
    int seg = 0;
    int64_t g = blockIdx.x;
    for (int i = 0; i < my_stages; ++i) {
      const int s = i & (NS - 1);
      if (i >= NS && !mbar_wait_fast(&empty[s], ((i / NS) - 1) & 1, abort_f, ERR_TIMEOUT_EMPTY)) break;
      if (*abort_f) break;
      const int64_t r0 = g * R;
      const int rows = (int)min((int64_t)R, (int64_t)a.N - r0);
      // one box of R rows x one segment: rows past N are zero-filled, the
      // transaction count is always the whole box
      unsigned char* st = stages + (size_t)s * P.stage_bytes;
      if (lane == 0) {
        const uint32_t tx = (uint32_t)R * P.seg_bytes + (PERROW ? 0u : (uint32_t)R * P.seg_sc);
        mbar_arrive_tx(&full[s], tx);
        tma_2d(st, &tm_codes, seg * (P.seg_bytes / 8), (int)r0, &full[s]);
        if (!PERROW) tma_2d(st + P.sc_off, &tm_scales, seg * (P.KS / 32), (int)r0, &full[s]);
      }
      ++issued;
      if (++seg == P.NSEG) {
        seg = 0;
        g += gridDim.x;
      }
    }
    // let every copy this warp issued land before the CTA can exit
    if (lane == 0)
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        mbar_drain(&full[j % NS], (j / NS) & 1);
    return;
  }

  // ------------------------------------------- prologue (warps 1 .. end) --
  // Activations, residual and gamma may come from the previous kernel, and
  // the outputs may still be read by it: wait for it to complete (no-op
  // without a programmatic launch).  The producer above never waits: packed
  // weights are not written by the kernels a matvec overlaps.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tt = threadIdx.x - 32;        // 0 .. 32 + Tc - 1
  const int nt = 32 + P.Tc;
  if (FUSED) {
    float* bsum = tbuf;                   // the fold buffer is free until the main loop
    __half* h_out = (blockIdx.x == 0) ? a.h_out : nullptr;
    for (int b = tt; b < NB; b += nt) {
      float blk = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + 32 * b + 8 * q));
        const uint4 rv = __ldg(reinterpret_cast<const uint4*>(a.r + 32 * b + 8 * q));
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, rs[4] = {rv.x, rv.y, rv.z, rv.w};
        uint32_t hs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 xx = u32_as_h2(xs[e]), rr = u32_as_h2(rs[e]);
          const __half lo = __float2half_rn(__fadd_rn(__low2float(xx), __low2float(rr)));
          const __half hi = __float2half_rn(__fadd_rn(__high2float(xx), __high2float(rr)));
          const float fl = __half2float(lo), fh = __half2float(hi);
          blk = __fmaf_rn(fl, fl, blk);
          blk = __fmaf_rn(fh, fh, blk);
          hs[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        if (h_out)
          *reinterpret_cast<uint4*>(h_out + 32 * b + 8 * q) = make_uint4(hs[0], hs[1], hs[2], hs[3]);
      }
      bsum[b] = blk;
    }
    named_bar(1, nt);
    if (tt == 0) {
      float ss = 0.0f;
      for (int b = 0; b < NB; ++b) ss = __fadd_rn(ss, bsum[b]);
      const float mean = __fdiv_rn(ss, (float)K);
      *inv_sh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
    }
    named_bar(1, nt);
    const float inv = *inv_sh;
    for (int v8 = tt; v8 < K / 8; v8 += nt) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + 8 * v8));
      const uint4 rv = __ldg(reinterpret_cast<const uint4*>(a.r + 8 * v8));
      const uint4 gv = __ldg(reinterpret_cast<const uint4*>(a.gamma + 8 * v8));
      const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, rs[4] = {rv.x, rv.y, rv.z, rv.w},
                     gs[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t ys[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 xx = u32_as_h2(xs[e]), rr = u32_as_h2(rs[e]), gg = u32_as_h2(gs[e]);
        const float hl = __half2float(__float2half_rn(__fadd_rn(__low2float(xx), __low2float(rr))));
        const float hh = __half2float(__float2half_rn(__fadd_rn(__high2float(xx), __high2float(rr))));
        const __half yl = __float2half_rn(__fmul_rn(__fmul_rn(hl, inv), __low2float(gg)));
        const __half yh = __float2half_rn(__fmul_rn(__fmul_rn(hh, inv), __high2float(gg)));
        ys[e] = (uint32_t)__half_as_ushort(yl) | ((uint32_t)__half_as_ushort(yh) << 16);
      }
      store_y8<BITS, EXACT>(y2f, 8 * v8, ys);
    }
  } else {
    for (int v8 = tt; v8 < K / 8; v8 += nt) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + 8 * v8));
      const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
      store_y8<BITS, EXACT>(y2f, 8 * v8, xs);
    }
  }
  if (!EXACT) {
    // block sums of the activations in the order of the dots (even and odd
    // words serially, then added), read back from the scaled pairs
    // (y' * 2^(o - FOLD_E) = y exactly), times the offset 2^(b-1)
    named_bar(1, nt);
    constexpr int CPW = 32 / BITS, HALF = CPW / 2;
    for (int b = tt; b < NB; b += nt) {
      const float* src = y2f + 2 * (YS * (b >> 1) + 16 * (b & 1));
      float S0 = 0.0f, S1 = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float sc = pow2f(BITS * ((t % CPW) % HALF) - FOLD_E);
        S0 = __fmaf_rn(src[2 * t], sc, S0);
        S1 = __fmaf_rn(src[2 * t + 1], sc, S1);
      }
      ysum[b] = __fmul_rn(__fadd_rn(S0, S1), (float)(1 << (BITS - 1)));
    }
  }
  named_bar(1, nt);

  // ---------------------------------------------------------- fold warp --
  if (warp == 1) {
    float acc = 0.0f;   // this lane's row: group-32 accumulator, or the per-row block sum
    int seg = 0;
    int64_t g = blockIdx.x;
    for (int i = 0; i < my_stages; ++i) {
      const int tb = i & 1;
      if (!mbar_wait_fast(&tfull[tb], (i >> 1) & 1, abort_f, ERR_TIMEOUT_TFULL)) break;
      const int64_t r0 = g * R;
      const int rows = (int)min((int64_t)R, (int64_t)a.N - r0);
      if (lane < rows) {
        const float* tr = tbuf + (size_t)(tb * R + lane) * GS;
        if (!PERROW) {
          if (seg == 0) acc = 0.0f;
#pragma unroll 8
          for (int b = 0; b < NBS; ++b) acc = __fadd_rn(acc, tr[b]);
        } else {
          int b0 = 0;
          if (seg == 0) {
            acc = tr[0];
            b0 = 1;
          }
#pragma unroll 8
          for (int b = b0; b < NBS; ++b) acc = __fadd_rn(acc, tr[b]);
        }
        if (seg == P.NSEG - 1) {
          float out = acc;
          if (PERROW) out = __fadd_rn(0.0f, __fmul_rn(acc, __half2float(a.scales[r0 + lane])));
          if (a.y_f16)
            reinterpret_cast<__half*>(a.y)[r0 + lane] = __float2half_rn(out);
          else
            reinterpret_cast<float*>(a.y)[r0 + lane] = out;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[tb]);
      if (++seg == P.NSEG) {
        seg = 0;
        g += gridDim.x;
      }
    }
    return;
  }

  // ------------------------------------------------------- compute warps --
  const int tc = threadIdx.x - 64;
  const bool active = tc < P.Cs * P.RP;
  const int c = active ? tc % P.Cs : 0;
  const int rp = active ? tc / P.Cs : 0;
  const u64* y2s = reinterpret_cast<const u64*>(y2f);

  int seg = 0;
  int64_t g = blockIdx.x;
  for (int i = 0; i < my_stages; ++i) {
    const int s = i & (NS - 1);
    const int tb = i & 1;
    if (!mbar_wait_fast(&full[s], (i / NS) & 1, abort_f, ERR_TIMEOUT_FULL)) break;
    if (i >= 2 && !mbar_wait_fast(&tempty[tb], ((i >> 1) - 1) & 1, abort_f, ERR_TIMEOUT_TEMPTY)) break;
    const int64_t r0 = g * R;
    const int rows = (int)min((int64_t)R, (int64_t)a.N - r0);
    if (active && !EXACT) {
      // folded form: rows past N in the box are zero-filled, so every row of
      // the group is computed (the fold warp stores only real rows)
      const unsigned char* st = stages + (size_t)s * P.stage_bytes;
      u64 wp[U][IW / 2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = rp * U + u;
        const ulonglong2* src =
            reinterpret_cast<const ulonglong2*>(st + (size_t)r * P.seg_bytes + (size_t)c * (IW * 4));
#pragma unroll
        for (int q = 0; q < IW / 4; ++q) {
          const ulonglong2 v = src[q];
          wp[u][2 * q] = v.x;
          wp[u][2 * q + 1] = v.y;
        }
      }
      const __half* scs = reinterpret_cast<const __half*>(st + P.sc_off);
      const float2 bS = *reinterpret_cast<const float2*>(ysum + 2 * (seg * P.Cs + c));
      u64 acc[U][2];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u][0] = acc[u][1] = 0ull;
      item_dots_fold<BITS, U>(wp, y2s + YS * (seg * P.Cs + c), acc);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = rp * U + u;
        float2 sc = make_float2(1.0f, 1.0f);
        if (!PERROW) sc = __half22float2(*reinterpret_cast<const __half2*>(scs + (size_t)r * NBS + 2 * c));
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          float pe, po;
          upk(acc[u][blk], pe, po);
          float pb = fold_block(__fadd_rn(pe, po), blk ? bS.y : bS.x);
          if (!PERROW) pb = __fmul_rn(pb, blk ? sc.y : sc.x);
          tbuf[(size_t)(tb * R + r) * GS + 2 * c + blk] = pb;
        }
      }
    } else if (active) {
      const unsigned char* st = stages + (size_t)s * P.stage_bytes;
      uint32_t w[U][IW];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = rp * U + u;
        if (r < rows) {
          const uint4* src = reinterpret_cast<const uint4*>(st + (size_t)r * P.seg_bytes + (size_t)c * (IW * 4));
#pragma unroll
          for (int q = 0; q < IW / 4; ++q) {
            const uint4 v = src[q];
            w[u][4 * q + 0] = v.x;
            w[u][4 * q + 1] = v.y;
            w[u][4 * q + 2] = v.z;
            w[u][4 * q + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int q = 0; q < IW; ++q) w[u][q] = 0x00000000u;
        }
      }
      u64 acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = 0ull;
      item_dots<BITS, U>(w, y2s + YS * (seg * P.Cs + c), acc);
      const __half* scs = reinterpret_cast<const __half*>(st + P.sc_off);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = rp * U + u;
        if (r < rows) {
          float p0, p1;
          upk(acc[u], p0, p1);
          float* dst = tbuf + (size_t)(tb * R + r) * GS + 2 * c;
          if (PERROW) {
            dst[0] = p0;
            dst[1] = p1;
          } else {
            const __half2 s2 = *reinterpret_cast<const __half2*>(scs + (size_t)r * NBS + 2 * c);
            dst[0] = __fmul_rn(p0, __low2float(s2));
            dst[1] = __fmul_rn(p1, __high2float(s2));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[s]);
      mbar_arrive(&tfull[tb]);
    }
    if (++seg == P.NSEG) {
      seg = 0;
      g += gridDim.x;
    }
  }
}

// ------------------------------------------------------------- launcher --

// Codes per segment: the whole row up to 2048, else the largest multiple of
// 256 up to 2048 that divides K.
static int tma_segment(int K) {
  if (K <= 2048) return K;
  for (int d = 8; d >= 1; --d)
    if ((K / 256) % d == 0) return 256 * d;
  return 256;
}

// Plan for about `tc_target` compute threads and U rows per thread
// (RP*U <= 32 rows per group: one fold lane per row).
static bool tma_plan(int N, int K, int bits, bool perrow, int tc_target, int U, TmaPlan* P) {
  if (K % 256 != 0) return false;
  const int KS = tma_segment(K);
  const int Cs = KS / 64;
  int RP = tc_target / Cs;
  if (RP < 1) RP = 1;
  if (RP > 32 / U) RP = 32 / U;
  const int Tc = ((Cs * RP + 31) / 32) * 32;
  if (Tc > 512) return false;
  if (RP * U > 32) return false;
  P->C = K / 64;
  P->Cs = Cs;
  P->KS = KS;
  P->NSEG = K / KS;
  P->RP = RP;
  P->R = RP * U;
  P->Tc = Tc;
  P->row_bytes = K * bits / 8;
  P->seg_bytes = KS * bits / 8;
  P->seg_sc = perrow ? 0 : (KS / 32) * 2;
  P->sc_off = (P->R * P->seg_bytes + 127) & ~127;
  P->stage_bytes = (P->sc_off + P->R * P->seg_sc + 127) & ~127;
  P->ngroups = (int)(((int64_t)N + P->R - 1) / P->R);
  P->y_off = 128;
  P->ysum_off = P->y_off + (K / 64) * YS * 8;
  P->stage_off = (P->ysum_off + (K / 32) * 4 + 127) & ~127;
  P->tbuf_off = tma_round16(P->stage_off + NS * P->stage_bytes);
  return true;
}

// ------------------------------------------------------- tensor maps ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return (EncodeTiledFn)f;
  }();
  return fn;
}

// Tensor maps of a pack for a plan: codes as UINT64 [N][row_bytes/8] with a
// box of (segment bytes / 8) x R, scales as UINT16 [N][K/32] with a box of
// (K_seg / 32) x R.  Cached per thread (a few entries).
static bool tensor_maps(const GemvArgs& a, int bits, const TmaPlan& P, CUtensorMap* tc, CUtensorMap* ts) {
  struct Entry { const void* codes; const void* scales; int N, K, bits, R, KS; CUtensorMap c, s; };
  static thread_local Entry cache[8];
  static thread_local int valid = 0, next = 0;
  for (int i = 0; i < valid; ++i) {
    const Entry& e = cache[i];
    if (e.codes == a.codes && e.scales == a.scales && e.N == a.N && e.K == a.K && e.bits == bits &&
        e.R == P.R && e.KS == P.KS) {
      *tc = e.c;
      *ts = e.s;
      return true;
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  Entry e;
  e.codes = a.codes;
  e.scales = a.scales;
  e.N = a.N;
  e.K = a.K;
  e.bits = bits;
  e.R = P.R;
  e.KS = P.KS;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)(P.row_bytes / 8), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)P.row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(P.seg_bytes / 8), (cuuint32_t)P.R};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&e.c, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, (void*)a.codes, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  if (a.perrow) {
    e.s = e.c;   // unused
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 32), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 32) * 2};
    const cuuint32_t box[2] = {(cuuint32_t)(P.KS / 32), (cuuint32_t)P.R};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&e.s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void*)a.scales, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  cache[next] = e;
  next = (next + 1) % 8;
  if (valid < 8) ++valid;
  *tc = e.c;
  *ts = e.s;
  return true;
}

// The fold buffer (2 x R rows x (KS/32 + 1) floats) also holds the fused
// prologue's K/32 block sums before the main loop starts.
static size_t tma_smem(const TmaPlan& P, int K) {
  const int fold = 2 * P.R * (P.KS / 32 + 1) * 4;
  const int bsum = (K / 32) * 4;
  return (size_t)P.tbuf_off + (size_t)tma_round16(fold > bsum ? fold : bsum);
}

template <int BITS, bool PERROW, bool FUSED, bool EXACT, int U, int MAXT>
static int run_tma(const GemvArgs& a, const TmaPlan& P, cudaStream_t s, cudaError_t* err,
                   int* occ_only = nullptr) {
  static thread_local int cached_dev = -1;
  static thread_local size_t smem_set = 0;
  static thread_local int occ_cache = 0;
  static thread_local size_t occ_smem = 0;
  static thread_local int occ_threads = 0;
  auto kern = gemv_tma_kernel<BITS, PERROW, FUSED, EXACT, U, MAXT>;
  const size_t smem = tma_smem(P, a.K);
  const DevInfo& d = dev_info();
  if (smem > (size_t)d.max_smem_optin) return QMV_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  if (dev != cached_dev) { cached_dev = dev; smem_set = 0; occ_smem = 0; occ_threads = 0; }
  if (smem > smem_set) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
    smem_set = smem;
  }
  const int threads = 64 + P.Tc;
  if (occ_smem != smem || occ_threads != threads) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_cache, kern, threads, smem);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
    occ_smem = smem;
    occ_threads = threads;
  }
  if (occ_only) {
    *occ_only = occ_cache;
    return QMV_OK;
  }
  if (occ_cache < 1) return QMV_ERR_UNSUPPORTED;
  int grid = d.sms * occ_cache;
  if (grid > P.ngroups) grid = P.ngroups;
  CUtensorMap tmc, tms;
  if (!tensor_maps(a, BITS, P, &tmc, &tms)) return QMV_ERR_UNSUPPORTED;
  if (pdl_enabled()) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, P, tmc, tms);
    if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  } else {
    kern<<<grid, threads, smem, s>>>(a, P, tmc, tms);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

// CTAs of up to 256 compute threads (320 in all) take 4 or 2 rows per
// thread (2 for int8); larger ones (long K) 2.  These are the plans
// tma_bits generates.
template <int BITS, bool PERROW, bool FUSED, bool EXACT>
static int tma_u(const GemvArgs& a, const TmaPlan& P, cudaStream_t s, cudaError_t* err,
                 int* occ_only) {
  const int U = P.R / P.RP;
  if (P.Tc > 256) {
    if (U != 2) return QMV_ERR_UNSUPPORTED;
    return run_tma<BITS, PERROW, FUSED, EXACT, 2, 576>(a, P, s, err, occ_only);
  }
  if (U == 2) return run_tma<BITS, PERROW, FUSED, EXACT, 2, 320>(a, P, s, err, occ_only);
  if constexpr (BITS != 8)
    if (U == 4) return run_tma<BITS, PERROW, FUSED, EXACT, 4, 320>(a, P, s, err, occ_only);
  return QMV_ERR_UNSUPPORTED;
}

template <int BITS, bool EXACT>
static int tma_mode(const GemvArgs& a, const TmaPlan& P, cudaStream_t s, cudaError_t* err,
                    int* occ_only) {
  if (a.perrow)
    return a.fused ? tma_u<BITS, true, true, EXACT>(a, P, s, err, occ_only)
                   : tma_u<BITS, true, false, EXACT>(a, P, s, err, occ_only);
  return a.fused ? tma_u<BITS, false, true, EXACT>(a, P, s, err, occ_only)
                 : tma_u<BITS, false, false, EXACT>(a, P, s, err, occ_only);
}

template <int BITS>
static int tma_dispatch(const GemvArgs& a, const TmaPlan& P, cudaStream_t s, cudaError_t* err,
                        int* occ_only) {
  return a.folded ? tma_mode<BITS, false>(a, P, s, err, occ_only)
                  : tma_mode<BITS, true>(a, P, s, err, occ_only);
}

// Choose the plan with the most resident compute warps per SM (occupancy
// from the runtime for the exact kernel, block size and shared memory); on a
// tie, the larger row group.  Candidates: ~256 or ~512 compute threads, and
// 4 or 2 rows per thread (2 for int8 and for the 512-thread CTAs), with at
// least 3 row groups per CTA slot when N allows it (load balance).  The
// choice is cached per shape.
template <int BITS>
static int tma_bits(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  struct Key { int N, K, perrow, fused, folded, dev; };
  struct Entry { Key k; TmaPlan p; bool ok; };
  static thread_local Entry cache[16];
  static thread_local int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  const Key key{a.N, a.K, a.perrow, a.fused, a.folded, dev};
  for (int i = 0; i < 16; ++i) {
    const Key& k = cache[i].k;
    if (cache[i].ok && k.N == key.N && k.K == key.K && k.perrow == key.perrow &&
        k.fused == key.fused && k.folded == key.folded && k.dev == key.dev)
      return tma_dispatch<BITS>(a, cache[i].p, s, err, nullptr);
  }
  static const int tc_force = [] {
    const char* e = getenv("QMV_TC");
    const int v = e ? atoi(e) : 0;
    return (v >= 128 && v <= 512) ? v : 0;
  }();
  const int sms = dev_info().sms;
  TmaPlan best;
  int best_score = -1;
  for (int tc : {256, 512}) {
    if (tc_force && tc != tc_force) continue;
    for (int U : {4, 2}) {
      if (BITS == 8 && U > 2) continue;
      if (tc > 256 && U > 2) continue;
      TmaPlan P;
      if (!tma_plan(a.N, a.K, BITS, a.perrow != 0, tc, U, &P)) continue;
      if (tma_smem(P, a.K) > (size_t)dev_info().max_smem_optin) continue;
      int occ = 0;
      if (tma_dispatch<BITS>(a, P, s, err, &occ) != QMV_OK || occ < 1) continue;
      int score = occ * (P.Tc / 32) * 64 + P.R;
      if ((int64_t)P.ngroups < 3LL * occ * sms && U > 2) score -= 64 * 64;   // balance
      if (score > best_score) {
        best_score = score;
        best = P;
      }
    }
  }
  if (best_score < 0) return QMV_ERR_UNSUPPORTED;
  cache[next] = Entry{key, best, true};
  next = (next + 1) % 16;
  return tma_dispatch<BITS>(a, best, s, err, nullptr);
}

// Whether some plan of the pipeline fits this K (shared memory), i.e. whether
// launch_gemv_tma can run the shape at all.
bool tma_fits(int K, int bits, bool perrow) {
  for (int tc : {256, 512})
    for (int U : {4, 2}) {
      if (bits == 8 && U > 2) continue;
      if (tc > 256 && U > 2) continue;
      TmaPlan P;
      if (tma_plan(1, K, bits, perrow, tc, U, &P) && tma_smem(P, K) <= (size_t)dev_info().max_smem_optin)
        return true;
    }
  return false;
}

int launch_gemv_tma(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err) {
  switch (bits) {
    case 2: return tma_bits<2>(a, s, err);
    case 4: return tma_bits<4>(a, s, err);
    default: return tma_bits<8>(a, s, err);
  }
}

int read_tc_error(int clear, int* out);

int read_device_error(int clear, int* out) {
  int t = 0;
  const int et = read_tc_error(clear, &t);
  if (et != 0) return et;
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qmv_error, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_qmv_error, &z, sizeof(int));
    if (e != cudaSuccess) return (int)e;
  }
  *out = v ? v : t;
  return 0;
}

}  // namespace qmv
