// qmv_pipe.cuh -- building blocks of the M = 1 bulk-copy pipeline, shared by
// the single-matvec kernel (qmv_tma.cu) and the persistent chain kernel
// (qmv_chain.cu): bounded mbarrier waits, tensor copies, the activation
// table, the per-stage dots in the exact and folded forms, and the fold.
//
// What they compute is the oracle's definition ("Gemma4 raw-Metal loop on
// A19", section "What moved the needle": int2 at 16 codes per word, exact
// products, fp32 in code order; the residual-add + RMSNorm fold into the
// matvec prologue): per output row, each 32-code block summed in fp32,
// scaled (group 32) and folded serially over the blocks.
#pragma once
#include <cuda.h>

#include "qmv_internal.cuh"

namespace qmv {
namespace pipe {

constexpr int NS = 4;                      // ring stages (a power of two)
constexpr uint32_t SPIN_LIMIT = 1u << 22;  // tries per bounded wait (a backstop to the time limit)
constexpr int ERR_TIMEOUT_FULL = 1, ERR_TIMEOUT_EMPTY = 2, ERR_TIMEOUT_TFULL = 3,
              ERR_TIMEOUT_TEMPTY = 4, ERR_SMEM_ALIGN = 5, ERR_BAD_EXPERT = 8;


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
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                              int code, int* err) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (mbar_try_hint(b, parity, WAIT_HINT_NS)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > WAIT_LIMIT_NS) break;
  }
  *abort_flag = 1;
  atomicCAS(err, 0, code);
  return false;
}

// The common case inline (one try_wait, which itself suspends the warp for a
// while), the bounded loop out of line.
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                               int code, int* err) {
  return mbar_try(b, parity) || mbar_wait(b, parity, abort_flag, code, err);
}

// Bounded wait that ignores the abort flag (used to let copies land).
__device__ __forceinline__ void mbar_drain(uint64_t* b, uint32_t parity, int* err) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (mbar_try_hint(b, parity, WAIT_HINT_NS)) return;
    if (global_ns() - t0 > WAIT_LIMIT_NS) break;
  }
  atomicCAS(err, 0, ERR_TIMEOUT_FULL);
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
  int ids_off;       // expert gather: the selected experts' ids (shared memory)
};

constexpr int GATHER_MAX = 256;   // selected experts per expert-gather call at most

// Where row group g of a matvec sits: the first output row (log0), the first
// row of the pack it reads (phys0), the rows it really has, and whether its
// expert id is valid.  Without expert gather the two are the same.  With it,
// each selected expert's rows form ceil(rows/R) groups; an invalid id reads
// past the end of the pack (the copies zero-fill) and its outputs are zeroed.
struct GroupRows {
  int64_t log0, phys0;
  int rows;
  bool ok;
};

__host__ __device__ __forceinline__ GroupRows group_rows(const GemvArgs& a, int R, int64_t g,
                                                         const int* ids) {
  GroupRows gr;
  if (!a.gather_rows) {
    gr.log0 = gr.phys0 = g * R;
    gr.rows = (int)((int64_t)a.N - g * R < R ? (int64_t)a.N - g * R : R);
    gr.ok = true;
    return gr;
  }
  const int gpe = (a.gather_rows + R - 1) / R;
  const int64_t j = g / gpe;
  const int lr0 = (int)(g % gpe) * R;
  const int e = ids[j];
  gr.ok = e >= 0 && e < a.gather_E;
  gr.log0 = j * a.gather_rows + lr0;
  gr.rows = (a.gather_rows - lr0 < R) ? a.gather_rows - lr0 : R;
  gr.phys0 = gr.ok ? (int64_t)e * a.gather_rows + lr0 : (int64_t)a.N;
  return gr;
}

__host__ __device__ inline int tma_round16(int x) { return (x + 15) & ~15; }

// ------------------------------------------------------ op-level pieces --

// Codes per segment: the whole row up to ks_max (2048 or 4096), else the
// largest multiple of 256 up to ks_max that divides K.
inline int tma_segment(int K, int ks_max = 2048) {
  if (K <= ks_max) return K;
  for (int d = ks_max / 256; d >= 1; --d)
    if ((K / 256) % d == 0) return 256 * d;
  return 256;
}

// fp16 element k (0..31) of a block held as 16 words (element 2e in the low
// half of word e), as fp32
__device__ __forceinline__ float blk_elem(const uint32_t (&y)[16], int k) {
  const __half2 v = u32_as_h2(y[k >> 1]);
  return (k & 1) ? __high2float(v) : __low2float(v);
}

// One 32-code block b of the activation table from its 32 fp16 activations;
// the folded form also gets the block's activation sum in the order of the
// dots (even and odd words serially, then added) times 2^(b-1).
template <int BITS, bool EXACT>
__device__ __forceinline__ void table_block(float* y2f, float* ysum, int b, const uint32_t (&y)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t y8[4] = {y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]};
    store_y8<BITS, EXACT>(y2f, 32 * b + 8 * q, y8);
  }
  if (!EXACT) {
    constexpr int CPW = 32 / BITS;
    float S0 = 0.0f, S1 = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int k0 = CPW * 2 * (t / CPW) + t % CPW;   // code of the even word; the odd word's is k0 + CPW
      S0 = __fadd_rn(S0, blk_elem(y, k0));
      S1 = __fadd_rn(S1, blk_elem(y, k0 + CPW));
    }
    ysum[b] = __fmul_rn(__fadd_rn(S0, S1), (float)(1 << (BITS - 1)));
  }
}

__device__ __forceinline__ void load_blk(const __half* p, uint32_t (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p + 8 * q));
    v[4 * q] = u.x;
    v[4 * q + 1] = u.y;
    v[4 * q + 2] = u.z;
    v[4 * q + 3] = u.w;
  }
}

// h = fp16(x + r) of one block, and its serial sum of squares
__device__ __forceinline__ float residual_blk(const uint32_t (&x)[16], const uint32_t (&r)[16],
                                              uint32_t (&h)[16]) {
  float blk = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const __half2 xx = u32_as_h2(x[e]), rr = u32_as_h2(r[e]);
    const __half lo = __float2half_rn(__fadd_rn(__low2float(xx), __low2float(rr)));
    const __half hi = __float2half_rn(__fadd_rn(__high2float(xx), __high2float(rr)));
    const float fl = __half2float(lo), fh = __half2float(hi);
    blk = __fmaf_rn(fl, fl, blk);
    blk = __fmaf_rn(fh, fh, blk);
    h[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
  return blk;
}

// The activation table of one matvec (threads tt = 0 .. nt-1 of the CTA, which
// synchronise on named barrier bar_id), one thread per 32-code block: y (the
// fused prologue's normalised h = fp16(x + r), or x) into the pair table y2f,
// and for the folded form the per-block activation sums into ysum.  With the
// fused prologue, bsum holds K/32 floats of scratch and h_out (nullable)
// receives h.  One round of global loads: x and r of a thread's block are
// loaded together (gamma prefetched into L1 meanwhile), and the block's h
// stays in registers.
// The fused prologue with eight elements a thread, for K <= 8 * nt (whole
// warps: tt = 0 .. nt-1 in warp order).  Every thread runs the same short
// straight-line path once: a launch's prologue runs cold, at several cycles
// per instruction, so its length, not its arithmetic, sets its time.  Lanes
// 4j .. 4j+3 hold the four octets of one 32-code block; the block's serial
// chains (its sum of squares over elements 0..31, and the folded form's two
// activation sums) pass through them in element order by shuffles, so every
// sum is formed in the same order as with one thread per block.
template <int BITS, bool EXACT>
__device__ __forceinline__ void build_table_octets(const GemvArgs& a, float* y2f, float* ysum, float* bsum,
                                                   float* inv_sh, __half* h_out, int tt, int nt, int bar_id) {
  constexpr int CPW = 32 / BITS;
  const int K = a.K, NB = K / 32;
  const int lane = tt & 31, base = lane & ~3, oq = lane & 3;
  const bool live = 8 * tt < K;   // a block's four octets are all live or all not
  const int e0 = live ? 8 * tt : 0;
  const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + e0));
  const uint4 rv = __ldg(reinterpret_cast<const uint4*>(a.r + e0));
  const uint4 gv = __ldg(reinterpret_cast<const uint4*>(a.gamma + e0));
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  uint32_t hw[4];
  float hf[8];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const __half2 xx = u32_as_h2(xw[w]), rr = u32_as_h2(rw[w]);
    const __half lo = __float2half_rn(__fadd_rn(__low2float(xx), __low2float(rr)));
    const __half hi = __float2half_rn(__fadd_rn(__high2float(xx), __high2float(rr)));
    hf[2 * w] = __half2float(lo);
    hf[2 * w + 1] = __half2float(hi);
    hw[w] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
  float run = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (oq == k) {
#pragma unroll
      for (int e = 0; e < 8; ++e) run = __fmaf_rn(hf[e], hf[e], run);
    }
    run = __shfl_sync(0xffffffffu, run, base | k);
  }
  if (live) {
    if (oq == 3) bsum[tt >> 2] = run;
    if (h_out) *reinterpret_cast<uint4*>(h_out + e0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  }
  named_bar(bar_id, nt);
  if (tt == 0) {
    // serial over the blocks, 16-byte loads issued ahead of the adds
    float ss = 0.0f;
    const float4* b4 = reinterpret_cast<const float4*>(bsum);
#pragma unroll 4
    for (int q = 0; q < NB / 4; ++q) {
      const float4 v = b4[q];
      ss = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(ss, v.x), v.y), v.z), v.w);
    }
    const float mean = __fdiv_rn(ss, (float)K);
    *inv_sh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
  }
  named_bar(bar_id, nt);
  const float inv = *inv_sh;
  uint32_t y[4];
  float yf[8];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const __half2 hh = u32_as_h2(hw[w]), gg = u32_as_h2(gw[w]);
    const __half yl = __float2half_rn(__fmul_rn(__fmul_rn(__low2float(hh), inv), __low2float(gg)));
    const __half yh = __float2half_rn(__fmul_rn(__fmul_rn(__high2float(hh), inv), __high2float(gg)));
    yf[2 * w] = __half2float(yl);
    yf[2 * w + 1] = __half2float(yh);
    y[w] = (uint32_t)__half_as_ushort(yl) | ((uint32_t)__half_as_ushort(yh) << 16);
  }
  if (live) store_y8<BITS, EXACT>(y2f, e0, y);
  if (!EXACT) {
    // the block's two activation sums (elements with (k / CPW) even, odd),
    // each serially in k, through the block's octets in order
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (oq == k) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (((8 * k + e) / CPW) & 1)
            s1 = __fadd_rn(s1, yf[e]);
          else
            s0 = __fadd_rn(s0, yf[e]);
        }
      }
      s0 = __shfl_sync(0xffffffffu, s0, base | k);
      s1 = __shfl_sync(0xffffffffu, s1, base | k);
    }
    if (live && oq == 3) ysum[tt >> 2] = __fmul_rn(__fadd_rn(s0, s1), (float)(1 << (BITS - 1)));
  }
}

template <int BITS, bool FUSED, bool EXACT>
__device__ __forceinline__ void build_table(const GemvArgs& a, float* y2f, float* ysum, float* bsum,
                                            float* inv_sh, __half* h_out, int tt, int nt, int bar_id) {
  const int K = a.K, NB = K / 32;
  if (FUSED && K <= 8 * nt) {
    build_table_octets<BITS, EXACT>(a, y2f, ysum, bsum, inv_sh, h_out, tt, nt, bar_id);
    return;
  }
  if (FUSED) {
    // pass 1: h and the block sums of squares (the block's h stays in
    // registers when every thread has at most one block; its gamma is
    // prefetched into L1 for pass 2)
    const bool one = NB <= nt;
    uint32_t h0[16], g0[16];
    for (int b = tt; b < NB; b += nt) {
      uint32_t x[16], r[16];
      load_blk(a.x + 32 * b, x);
      load_blk(a.r + 32 * b, r);
      if (one)
        load_blk(a.gamma + 32 * b, g0);
      else
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a.gamma + 32 * b));
      bsum[b] = residual_blk(x, r, h0);
      if (h_out) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(h_out + 32 * b + 8 * q) =
              make_uint4(h0[4 * q], h0[4 * q + 1], h0[4 * q + 2], h0[4 * q + 3]);
      }
    }
    named_bar(bar_id, nt);
    if (tt == 0) {
      // serial over the blocks, 16-byte loads issued ahead of the adds
      float ss = 0.0f;
      const float4* b4 = reinterpret_cast<const float4*>(bsum);
#pragma unroll 4
      for (int q = 0; q < NB / 4; ++q) {
        const float4 v = b4[q];
        ss = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(ss, v.x), v.y), v.z), v.w);
      }
      const float mean = __fdiv_rn(ss, (float)K);
      *inv_sh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
    }
    named_bar(bar_id, nt);
    const float inv = *inv_sh;
    for (int b = tt; b < NB; b += nt) {
      if (!one) {
        uint32_t x[16], r[16];
        load_blk(a.x + 32 * b, x);
        load_blk(a.r + 32 * b, r);
        residual_blk(x, r, h0);
      }
      uint32_t y[16];
      if (!one) load_blk(a.gamma + 32 * b, g0);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const __half2 hh = u32_as_h2(h0[e]), gg = u32_as_h2(g0[e]);
        const __half yl = __float2half_rn(__fmul_rn(__fmul_rn(__low2float(hh), inv), __low2float(gg)));
        const __half yh = __float2half_rn(__fmul_rn(__fmul_rn(__high2float(hh), inv), __high2float(gg)));
        y[e] = (uint32_t)__half_as_ushort(yl) | ((uint32_t)__half_as_ushort(yh) << 16);
      }
      table_block<BITS, EXACT>(y2f, ysum, b, y);
    }
  } else {
    for (int b = tt; b < NB; b += nt) {
      uint32_t x[16];
      load_blk(a.x + 32 * b, x);
      table_block<BITS, EXACT>(y2f, ysum, b, x);
    }
  }
}

// One compute thread's share of one stage (R rows x one K segment in `st`):
// item c of the segment for rows rp*U .. rp*U+U-1, block results (scaled by
// the group-32 scale) into the fold buffer rows tbr (stride GS).
template <int BITS, bool PERROW, bool EXACT, int U>
__device__ __forceinline__ void compute_stage(const unsigned char* st, const TmaPlan& P, int c, int rp,
                                              int seg, int rows, const u64* y2s, const float* ysum,
                                              float* tbr, int GS) {
  constexpr int IW = 64 * BITS / 32;   // words per item
  const int NBS = P.KS / 32;
  const __half* scs = reinterpret_cast<const __half*>(st + P.sc_off);
  const int ci = seg * P.Cs + c;       // item index in the row
  if (!EXACT) {
    // folded form: rows past N in the box are zero-filled, so every row of
    // the group is computed (the fold warp stores only real rows)
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
    const float2 bS = *reinterpret_cast<const float2*>(ysum + 2 * ci);
    u64 acc[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u][0] = acc[u][1] = 0ull;
    item_dots_fold<BITS, U>(wp, y2s + YS * ci, acc);
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
        tbr[(size_t)r * GS + 2 * c + blk] = pb;
      }
    }
  } else {
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
    item_dots<BITS, U>(w, y2s + YS * ci, acc);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = rp * U + u;
      if (r < rows) {
        float p0, p1;
        upk(acc[u], p0, p1);
        float* dst = tbr + (size_t)r * GS + 2 * c;
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
}

// Argmax key of output row n with value v: the value's bits made
// order-preserving as an unsigned number (after -0 -> +0) in the high word,
// ~n in the low word, so the largest key is the largest value and, among
// equal values, the lowest row (first-max tie-break).  NaN gets 0 (never
// wins; every other value's key is nonzero).
__device__ __forceinline__ unsigned long long amax_key(float v, int64_t n) {
  if (v != v) return 0ull;
  const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
}

// The fold warp's argmax epilogue, after its last stage: the warp's best key
// goes into the workspace key with one atomic max; the CTA that arrives last
// on the workspace counter writes the index and value and clears both words.
__device__ __forceinline__ void amax_finish(const GemvArgs& a, unsigned long long best, int lane) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
    best = o > best ? o : best;
  }
  if (lane != 0) return;
  unsigned long long* key = a.amax_ws;
  unsigned int* count = reinterpret_cast<unsigned int*>(a.amax_ws + 1);
  if (best) atomicMax(key, best);
  __threadfence();
  if (atomicAdd(count, 1u) == gridDim.x - 1) {
    __threadfence();
    const unsigned long long k = atomicExch(key, 0ull);
    atomicExch(count, 0u);
    int idx = -1;
    float val = __uint_as_float(0x7FC00000u);
    if (k) {
      idx = (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
      const uint32_t ord = (uint32_t)(k >> 32);
      val = __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
    }
    *a.amax_index = idx;
    if (a.amax_value) *a.amax_value = val;
  }
}

// The fold warp's share of one stage: lane = row of the group; acc carries
// the row's accumulator across the segments; the last segment stores y (when
// a.y is set) and, with the argmax epilogue, updates the lane's best key.
__device__ __forceinline__ void fold_stage(const GemvArgs& a, const TmaPlan& P, const float* tbr, int GS,
                                           int lane, const GroupRows& gr, int seg, float& acc,
                                           unsigned long long* best = nullptr) {
  const int NBS = P.KS / 32;
  const int64_t r0 = gr.log0;
  if (lane < gr.rows) {
    // the row's block results, serially (16-byte loads issued ahead of the
    // dependent adds; rows are GS floats apart, GS a multiple of 4)
    const float4* tr = reinterpret_cast<const float4*>(tbr + (size_t)lane * GS);
    if (seg == 0) acc = 0.0f;
#pragma unroll 4
    for (int q = 0; q < NBS / 4; ++q) {
      const float4 v = tr[q];
      // one scale per row: the row's first block starts the sum as is
      acc = (a.perrow && seg == 0 && q == 0) ? v.x : __fadd_rn(acc, v.x);
      acc = __fadd_rn(acc, v.y);
      acc = __fadd_rn(acc, v.z);
      acc = __fadd_rn(acc, v.w);
    }
    if (seg == P.NSEG - 1) {
      float out = acc;
      if (a.perrow && gr.ok) out = __fadd_rn(0.0f, __fmul_rn(acc, __half2float(a.scales[gr.phys0 + lane])));
      if (!gr.ok) out = 0.0f;
      if (a.y) {
        if (a.y_f16)
          reinterpret_cast<__half*>(a.y)[r0 + lane] = __float2half_rn(out);
        else
          reinterpret_cast<float*>(a.y)[r0 + lane] = out;
      }
      if (best) {
        const unsigned long long k = amax_key(out, r0 + lane);
        if (k > *best) *best = k;
      }
    }
  }
}

}  // namespace pipe

// Tensor maps of a pack for a plan (qmv_tma.cu): codes as UINT64
// [N][row_bytes/8] with a box of (segment bytes / 8) x R, scales as UINT16
// [N][K/32] with a box of (K_seg / 32) x R.  Host only.
bool encode_pack_maps(const GemvArgs& a, const pipe::TmaPlan& P, CUtensorMap* tc, CUtensorMap* ts);
// A 2-D tensor map: `rows` rows of `inner` elements, `row_bytes` apart, a box
// of box_inner x box_rows, zero fill past the edges (qmv_tc.cu).  Host only.
bool enc2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
           uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw);

}  // namespace qmv
